"""Every form of the library captured into a CUDA graph (README "Grouped GEMMs (masked
layout)": the masked form exists so that decoding can run in graphs; the library keeps every
form capturable): one eager call on the capturing stream first (it sizes the stream's
workspace), then a capture, then two replays, each bit-identical to the eager result."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_gemm_nt_gb300 as L
    L.load_library()
    return L


def _bits(t):
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16).cpu().numpy().copy()


def _dense(L, M, N, K, with_c, fp4=False):
    p = W.make_dense_fp4(M, N, K, seed=M + N + K, with_c=with_c) if fp4 else \
        W.make_dense(M, N, K, seed=M + N + K, with_c=with_c)
    ops = (dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb))
    c = dev(p.c.view(np.int16), torch.bfloat16) if p.c is not None else None
    d = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fn = L.dg_fp8_fp4_gemm_nt if fp4 else L.dg_fp8_gemm_nt
    return d, lambda s: fn(*ops, c, d, stream=s)


def _contiguous(L):
    p = W.make_contiguous(G=4, tokens=2000, N=1024, K=1024, seed=61)
    ops = (dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb))
    idx = dev(p.m_indices)
    d = torch.zeros((p.M_total, p.N), dtype=torch.bfloat16, device="cuda")
    return d, lambda s: L.dg_m_grouped_fp8_gemm_nt_contiguous(*ops, d, idx, stream=s)


def _masked(L):
    p = W.make_masked(G=8, max_m=256, N=1024, K=1024, seed=62)
    ops = (dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb))
    mm = dev(p.masked_m)
    d = torch.zeros((p.G, p.max_m, p.N), dtype=torch.bfloat16, device="cuda")
    return d, lambda s: L.dg_m_grouped_fp8_gemm_nt_masked(*ops, d, mm, stream=s)


def _wgrad(L):
    p = W.make_wgrad(1024, 2048, 1024, seed=63, with_c=True)
    ops = (dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb))
    c = dev(p.c)
    d = torch.empty((p.M, p.N), dtype=torch.float32, device="cuda")
    return d, lambda s: L.dg_wgrad_gemm_fp8_fp8_fp32_nt(*ops, c, d, stream=s)


def _k_grouped(L):
    p = W.make_k_grouped(G=3, M=512, N=768, tokens=1500, seed=64)
    ops = (dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb))
    c = dev(p.c)
    ks = dev(np.asarray(p.ks, np.int32))
    d = torch.empty((p.G, p.M, p.N), dtype=torch.float32, device="cuda")
    return d, lambda s: L.dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(*ops, c, d, ks, stream=s)


CASES = {
    "dense_tile": lambda L: _dense(L, 512, 1024, 1024, True),
    "dense_stream_k": lambda L: _dense(L, 200, 384, 4096, True),
    "dense_split_k_pairs": lambda L: _dense(L, 128, 7168, 4096, True),
    "dense_cta_pairs": lambda L: _dense(L, 2048, 4096, 1024, False),
    "fp4_dense": lambda L: _dense(L, 1024, 2048, 1024, False, fp4=True),
    "contiguous": _contiguous,
    "masked": _masked,
    "wgrad": _wgrad,
    "k_grouped": _k_grouped,
}


@pytest.mark.parametrize("name", list(CASES))
def test_form_replays_bit_identically(lib, name):
    d, call = CASES[name](lib)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call(s)                                  # eager: sizes the stream's workspace
    torch.cuda.synchronize()
    want = _bits(d)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call(s)
    torch.cuda.synchronize()
    for _ in range(2):
        d.fill_(float("nan") if d.dtype == torch.float32 else 0.0)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(_bits(d), want), name
    assert lib.dg_get_device_status() == 0
