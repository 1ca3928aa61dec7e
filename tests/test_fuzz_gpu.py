"""Seeded random shapes through every dispatch path of the three forms of the operation
(README "Normal dense GEMMs", "Grouped GEMMs (contiguous layout)", "Grouped GEMMs (masked
layout)"): ragged M, N a multiple of 16, K a multiple of 128, sizes that land on tile mode,
stream-K, split-K over CTA pairs and the CTA-pair kernel. Every case is compared with the
oracle over all of its output (padding and masked rows, and rows past M, must stay
untouched)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import SENTINEL, assert_parity, bf16_bits, bf16_f64, dev, run_contiguous, run_masked, sentinel_like

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_gemm_nt_gb300 as L
    L.load_library()
    return L


def _dense_shapes(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        M = int(rng.choice([int(rng.integers(1, 129)), int(rng.integers(129, 1200))]))
        N = 16 * int(rng.integers(1, 240))
        K = 128 * int(rng.integers(1, 40))
        if M * N * K <= 1_500_000_000:     # the oracle in FP64 stays within seconds
            out.append((M, N, K, bool(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("M,N,K,with_c", _dense_shapes(24, 2026))
def test_fuzz_dense(lib, M, N, K, with_c):
    p = W.make_dense(M, N, K, seed=M * 7 + N * 3 + K, with_c=with_c)
    c = dev(p.c.view(np.int16), torch.bfloat16) if p.c is not None else None
    full = sentinel_like((M + 4, N))
    d = full[:M]
    lib.dg_fp8_gemm_nt(dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb), c, d)
    torch.cuda.synchronize()
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
    assert_parity(bf16_f64(d), ref, f"dense {M}x{N}x{K} c={with_c}")
    assert (bf16_bits(full[M:]) == SENTINEL).all()
    assert lib.dg_get_device_status() == 0


def _grouped_shapes(n, seed):
    rng = np.random.default_rng(seed)
    return [(int(rng.integers(1, 7)), int(rng.integers(1, 700)), 16 * int(rng.integers(1, 80)),
             128 * int(rng.integers(1, 12)), int(rng.integers(0, 1 << 30))) for _ in range(n)]


@pytest.mark.parametrize("G,tokens,N,K,seed", _grouped_shapes(12, 2027))
def test_fuzz_contiguous(lib, G, tokens, N, K, seed):
    p = W.make_contiguous(G=G, tokens=tokens, N=N, K=K, seed=seed)
    d = run_contiguous(lib, p)
    bits = bf16_bits(d)
    ref, valid = O.m_grouped_fp8_gemm_nt_contiguous(p.a, p.sfa, p.b, p.sfb, p.m_indices, p.M_total, p.N, p.K, p.G)
    assert (bits[~valid] == SENTINEL).all()
    if valid.any():
        assert_parity(bf16_f64(d)[valid], ref[valid], f"contiguous G={G} tokens={tokens} N={N} K={K}")
    assert lib.dg_get_device_status() == 0


@pytest.mark.parametrize("G,max_m,N,K,seed", [(g, 1 + t % 300, n, k, s) for g, t, n, k, s in _grouped_shapes(12, 2028)])
def test_fuzz_masked(lib, G, max_m, N, K, seed):
    p = W.make_masked(G=G, max_m=max_m, N=N, K=K, seed=seed)
    d = run_masked(lib, p)
    bits = bf16_bits(d)
    ref, valid = O.m_grouped_fp8_gemm_nt_masked(p.a, p.sfa, p.b, p.sfb, p.masked_m, p.G, p.max_m, p.N, p.K)
    assert (bits[~valid] == SENTINEL).all()
    if valid.any():
        assert_parity(bf16_f64(d)[valid], ref[valid], f"masked G={G} max_m={max_m} N={N} K={K}")
    assert lib.dg_get_device_status() == 0
