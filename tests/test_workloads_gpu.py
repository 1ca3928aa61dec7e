"""Parity at the workload sizes, in the launch configuration the benchmark times.

The oracle computes sampled rows (all N columns) of each full-size problem; the
integer decisions (padding rows of the contiguous layout, masked rows) are checked
bit-exactly over the whole output.
"""
from __future__ import annotations

import functools

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import (SENTINEL, assert_parity, bf16_bits, bf16_f64, dev, run_contiguous, run_dense, run_k_grouped,
                      run_masked, run_wgrad, sentinel_like)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_gemm_nt_gb300 as L
    L.load_library()
    return L


@functools.lru_cache(maxsize=1)
def _workload(name):
    return W.make_workload(name)


def _rows(n, k, seed):
    rng = np.random.default_rng(seed)
    r = set(rng.choice(n, size=min(k, n), replace=False).tolist())
    r.update({0, n - 1, min(127, n - 1), min(128, n - 1)})
    return np.array(sorted(r))


@pytest.mark.parametrize("name", [n for n in W.WORKLOAD_ORDER if W.WORKLOADS[n]["kind"] == "dense"])
def test_dense_workload(lib, name):
    p = W.make_workload(name)
    d = run_dense(lib, p)
    rows = np.arange(p.M) if p.M <= 128 else _rows(p.M, 96, 1)
    if p.M >= 512:
        # and one whole 256-row pair tile (rows 256..511: both CTAs of a pair, every column)
        rows = np.unique(np.concatenate([rows, np.arange(256, 512)]))
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, p.M, p.N, p.K, rows=rows)
    assert_parity(bf16_f64(d)[rows], ref, name)
    assert lib.dg_get_device_status() == 0


def test_contiguous_workload(lib):
    name = "contiguous_g8_t32768_n4096_k7168"
    p = W.make_workload(name)
    d = run_contiguous(lib, p)
    bits = bf16_bits(d)
    pad = p.m_indices < 0
    assert (bits[pad] == SENTINEL).all()
    assert not (bits[~pad] == SENTINEL).all(axis=1).any()
    # sampled rows, including each expert's first and last valid row
    starts = [int(np.nonzero(p.m_indices == g)[0][0]) for g in range(p.G) if (p.m_indices == g).any()]
    ends = [int(np.nonzero(p.m_indices == g)[0][-1]) for g in range(p.G) if (p.m_indices == g).any()]
    rows = np.unique(np.concatenate([_rows(p.M_total, 96, 2), starts, ends]))
    rows = rows[p.m_indices[rows] >= 0]
    ref, valid = O.m_grouped_fp8_gemm_nt_contiguous(p.a, p.sfa, p.b, p.sfb, p.m_indices, p.M_total, p.N, p.K,
                                                    p.G, rows=rows)
    assert valid.all()
    assert_parity(bf16_f64(d)[rows], ref, name)
    assert lib.dg_get_device_status() == 0


def test_masked_workload(lib):
    name = "masked_g32_m256_n7168_k2048"
    p = W.make_workload(name)
    d = run_masked(lib, p)
    bits = bf16_bits(d)
    valid = np.arange(p.max_m)[None, :] < p.masked_m[:, None]
    assert (bits[~valid] == SENTINEL).all()
    groups = list(range(p.G))                   # every group, all of its valid rows
    ref, v = O.m_grouped_fp8_gemm_nt_masked(p.a, p.sfa, p.b, p.sfb, p.masked_m, p.G, p.max_m, p.N, p.K,
                                            groups=groups)
    got = bf16_f64(d)[groups]
    for g in groups:
        if v[g].any():
            assert_parity(got[g][v[g]], ref[g][v[g]], f"{name} group {g}")
    assert lib.dg_get_device_status() == 0


def test_wgrad_workload(lib):
    name = "wgrad_7168x4096x4096_c"
    p = W.make_workload(name)
    d = run_wgrad(lib, p).cpu().numpy().astype(np.float64)
    rows = _rows(p.M, 64, 4)
    ref = O.wgrad_gemm_fp8_fp8_fp32_nt(p.a, p.sfa, p.b, p.sfb, p.c, p.M, p.N, p.K, rows=rows)
    assert_parity(d[rows], ref, name)
    assert np.isfinite(d).all()
    assert lib.dg_get_device_status() == 0


def test_k_grouped_workload(lib):
    name = "k_grouped_wgrad_g4_m4096_n7168_t16384"
    p = W.make_workload(name)
    d = run_k_grouped(lib, p)
    rows = _rows(p.M, 32, 5)
    groups = list(range(p.G))                   # every expert
    ref = O.k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(p.a, p.sfa, p.b, p.sfb, p.c, p.ks, p.M, p.N, groups=groups, rows=rows)
    got = d[groups].cpu().numpy().astype(np.float64)[:, rows]
    for i, g in enumerate(groups):
        assert_parity(got[i], ref[i], f"{name} expert {g}")
    assert torch.isfinite(d).all()
    assert lib.dg_get_device_status() == 0


def test_layout_workload(lib):
    name = "dense_nn_4096x7168x2048"
    p = W.make_workload(name)
    assert p.layout == "nn"
    b_kn = dev(np.ascontiguousarray(p.b.T))
    d = sentinel_like((p.M, p.N))
    lib.dg_fp8_gemm_nn(dev(p.a), dev(p.sfa), b_kn, dev(p.sfb), None, d)
    torch.cuda.synchronize()
    rows = _rows(p.M, 64, 6)
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, None, p.M, p.N, p.K, rows=rows)
    assert_parity(bf16_f64(d)[rows], ref, name)
    assert lib.dg_get_device_status() == 0


def test_fp4_dense_workload(lib):
    name = "fp4_dense_decode_128x7168x16384_c"
    p = W.make_workload(name)
    d = run_dense(lib, p)
    ref = O.fp8_fp4_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, p.M, p.N, p.K)
    assert_parity(bf16_f64(d), ref, name)
    assert lib.dg_get_device_status() == 0


def test_fp4_masked_workload(lib):
    name = "fp4_masked_g32_m256_n7168_k2048"
    p = W.make_workload(name)
    d = run_masked(lib, p)
    bits = bf16_bits(d)
    valid = np.arange(p.max_m)[None, :] < p.masked_m[:, None]
    assert (bits[~valid] == SENTINEL).all()
    groups = list(range(p.G))                   # every group, all of its valid rows
    ref, v = O.m_grouped_fp8_fp4_gemm_nt_masked(p.a, p.sfa, p.b, p.sfb, p.masked_m, p.G, p.max_m, p.N, p.K,
                                                groups=groups)
    got = bf16_f64(d)[groups]
    for g in groups:
        if v[g].any():
            assert_parity(got[g][v[g]], ref[g][v[g]], f"{name} group {g}")
    assert lib.dg_get_device_status() == 0


def test_fp4_contiguous_workload(lib):
    name = "fp4_contiguous_g8_t32768_n4096_k7168"
    p = _workload(name)
    d = run_contiguous(lib, p)
    bits = bf16_bits(d)
    pad = p.m_indices < 0
    assert (bits[pad] == SENTINEL).all()
    starts = [int(np.nonzero(p.m_indices == g)[0][0]) for g in range(p.G) if (p.m_indices == g).any()]
    ends = [int(np.nonzero(p.m_indices == g)[0][-1]) for g in range(p.G) if (p.m_indices == g).any()]
    rows = np.unique(np.concatenate([_rows(p.M_total, 64, 5), starts, ends]))
    rows = rows[p.m_indices[rows] >= 0]
    ref, valid = O.m_grouped_fp8_fp4_gemm_nt_contiguous(p.a, p.sfa, p.b, p.sfb, p.m_indices, p.M_total, p.N, p.K,
                                                        p.G, rows=rows)
    assert valid.all()
    assert_parity(bf16_f64(d)[rows], ref, name)
    assert lib.dg_get_device_status() == 0


def test_contiguous_pair_fresh_streams(lib):
    # Batches of back-to-back launches, each batch on a new stream (a new, freshly zeroed
    # workspace for the preparation kernel's pair list). A CTA that read a stale pair count
    # (an L1 line from before the preparation kernel wrote it) once left its cluster partner
    # waiting: 9 of 60 such batches of this workload timed out on GB300 before the kernels
    # read their inputs at L2.
    p = _workload("fp4_contiguous_g8_t32768_n4096_k7168")
    a, sfa, b, sfb, idx = dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb), dev(p.m_indices)
    d = sentinel_like((p.M_total, p.N))
    for batch in range(24):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for _ in range(25):
                lib.dg_m_grouped_fp8_fp4_gemm_nt_contiguous(a, sfa, b, sfb, d, idx)
        torch.cuda.synchronize()
        assert lib.dg_get_device_status() == 0, f"batch {batch}"
