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


# ---- the other forms: FP8 x FP4, FP32-output weight gradients, the NN / TN / TT layouts

@pytest.mark.parametrize("M,N,K,with_c", [(m, n, k, c) for m, n, k, c in _dense_shapes(10, 2029)])
def test_fuzz_fp4_dense(lib, M, N, K, with_c):
    p = W.make_dense_fp4(M, N, K, seed=M + 11 * N + K, with_c=with_c)
    c = dev(p.c.view(np.int16), torch.bfloat16) if p.c is not None else None
    full = sentinel_like((M + 4, N))
    d = full[:M]
    lib.dg_fp8_fp4_gemm_nt(dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb), c, d)
    torch.cuda.synchronize()
    ref = O.fp8_fp4_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
    assert_parity(bf16_f64(d), ref, f"fp4 dense {M}x{N}x{K}")
    assert (bf16_bits(full[M:]) == SENTINEL).all()
    assert lib.dg_get_device_status() == 0


@pytest.mark.parametrize("G,tokens,N,K,seed", _grouped_shapes(6, 2030))
def test_fuzz_fp4_contiguous_and_masked(lib, G, tokens, N, K, seed):
    p = W.make_contiguous(G=G, tokens=tokens, N=N, K=K, seed=seed, b_format="e2m1")
    d = run_contiguous(lib, p)
    ref, valid = O.m_grouped_fp8_fp4_gemm_nt_contiguous(p.a, p.sfa, p.b, p.sfb, p.m_indices, p.M_total, p.N, p.K,
                                                        p.G)
    assert (bf16_bits(d)[~valid] == SENTINEL).all()
    if valid.any():
        assert_parity(bf16_f64(d)[valid], ref[valid], f"fp4 contiguous G={G} N={N} K={K}")
    q = W.make_masked(G=G, max_m=1 + tokens % 256, N=N, K=K, seed=seed + 1, b_format="e2m1")
    dq = run_masked(lib, q)
    refq, vq = O.m_grouped_fp8_fp4_gemm_nt_masked(q.a, q.sfa, q.b, q.sfb, q.masked_m, q.G, q.max_m, q.N, q.K)
    assert (bf16_bits(dq)[~vq] == SENTINEL).all()
    if vq.any():
        assert_parity(bf16_f64(dq)[vq], refq[vq], f"fp4 masked G={G} N={N} K={K}")
    assert lib.dg_get_device_status() == 0


@pytest.mark.parametrize("M,N,K,with_c", _dense_shapes(8, 2031))
def test_fuzz_wgrad(lib, M, N, K, with_c):
    p = W.make_wgrad(M, N, K, seed=M + 5 * N + K, with_c=with_c)
    c = dev(p.c) if p.c is not None else None
    d = torch.full((M, N), float("nan"), dtype=torch.float32).cuda()
    lib.dg_wgrad_gemm_fp8_fp8_fp32_nt(dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb), c, d)
    torch.cuda.synchronize()
    ref = O.wgrad_gemm_fp8_fp8_fp32_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
    assert_parity(d.cpu().numpy().astype(np.float64), ref, f"wgrad {M}x{N}x{K}")
    assert lib.dg_get_device_status() == 0


@pytest.mark.parametrize("G,M,N,tokens,seed", [(1 + g % 5, 16 * (1 + t % 40), n, 64 + t, s)
                                               for g, t, n, _, s in _grouped_shapes(6, 2032)])
def test_fuzz_k_grouped(lib, G, M, N, tokens, seed):
    p = W.make_k_grouped(G=G, M=M, N=N, tokens=tokens, seed=seed)
    c = dev(p.c) if p.c is not None else None
    d = torch.full((p.G, M, N), float("nan"), dtype=torch.float32).cuda()
    lib.dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb), c, d,
                                                dev(np.asarray(p.ks, np.int32)))
    torch.cuda.synchronize()
    ref = O.k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(p.a, p.sfa, p.b, p.sfb, p.c, p.ks, M, N)
    got = d.cpu().numpy().astype(np.float64)
    for g in range(p.G):
        assert_parity(got[g], ref[g], f"k-grouped G={G} M={M} N={N} expert {g}")
    assert lib.dg_get_device_status() == 0


@pytest.mark.parametrize("layout", ["nn", "tn", "tt"])
@pytest.mark.parametrize("M,N,K,with_c", [(16 * (1 + m % 70), n, k, c) for m, n, k, c in _dense_shapes(4, 2033)])
def test_fuzz_layouts(lib, layout, M, N, K, with_c):
    p = W.make_dense(M, N, K, seed=M + N + 3 * K, with_c=with_c)
    a = p.a if layout[0] == "n" else np.ascontiguousarray(p.a.T)
    b = p.b if layout[1] == "t" else np.ascontiguousarray(p.b.T)
    c = dev(p.c.view(np.int16), torch.bfloat16) if p.c is not None else None
    d = sentinel_like((M, N))
    getattr(lib, f"dg_fp8_gemm_{layout}")(dev(a), dev(p.sfa), dev(b), dev(p.sfb), c, d)
    torch.cuda.synchronize()
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
    assert_parity(bf16_f64(d), ref, f"{layout} {M}x{N}x{K}")
    assert lib.dg_get_device_status() == 0
