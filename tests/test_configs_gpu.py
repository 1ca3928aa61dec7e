"""Every tile configuration (BN = 128, 192, 256; DG_FORCE_BN overrides the heuristic)
against the oracle, on all three forms, with ragged edges."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import SENTINEL, assert_parity, bf16_bits, bf16_f64, run_contiguous, run_dense, run_masked

pytestmark = pytest.mark.gpu

BNS = [128, 192, 256]


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_gemm_nt_gb300 as L
    L.load_library()
    return L


@pytest.mark.parametrize("bn", BNS)
def test_dense_tile_mode(lib, bn, monkeypatch):
    monkeypatch.setenv("DG_FORCE_BN", str(bn))
    # 2048 x 1552 has more 128 x 128 tiles than SMs, so the forced width is used
    p = W.make_dense(2048, 1552, 384, seed=60 + bn, with_c=True)
    d = run_dense(lib, p)
    rows = np.unique(np.concatenate([np.arange(0, 2048, 7), [2047]]))
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, p.M, p.N, p.K, rows=rows)
    assert_parity(bf16_f64(d)[rows], ref, f"dense bn={bn}")
    assert lib.dg_get_device_status() == 0


@pytest.mark.parametrize("bn", BNS)
def test_contiguous(lib, bn, monkeypatch):
    monkeypatch.setenv("DG_FORCE_BN", str(bn))
    p = W.make_contiguous(G=3, tokens=500, N=400, K=640, seed=70 + bn, counts=[200, 1, 299])
    d = run_contiguous(lib, p)
    ref, valid = O.m_grouped_fp8_gemm_nt_contiguous(p.a, p.sfa, p.b, p.sfb, p.m_indices, p.M_total, p.N, p.K, p.G)
    assert (bf16_bits(d)[~valid] == SENTINEL).all()
    assert_parity(bf16_f64(d)[valid], ref[valid], f"contiguous bn={bn}")
    assert lib.dg_get_device_status() == 0


@pytest.mark.parametrize("bn", BNS)
def test_masked(lib, bn, monkeypatch):
    monkeypatch.setenv("DG_FORCE_BN", str(bn))
    p = W.make_masked(G=3, max_m=192, N=464, K=512, seed=80 + bn, masked_m=[192, 0, 77])
    d = run_masked(lib, p)
    ref, valid = O.m_grouped_fp8_gemm_nt_masked(p.a, p.sfa, p.b, p.sfb, p.masked_m, p.G, p.max_m, p.N, p.K)
    assert (bf16_bits(d)[~valid] == SENTINEL).all()
    assert_parity(bf16_f64(d)[valid], ref[valid], f"masked bn={bn}")
    assert lib.dg_get_device_status() == 0
