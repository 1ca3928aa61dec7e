"""dg_fp8_gemm_nt_no_alloc: the dense GEMM for callers that cannot allocate device memory
when they run it (servers with a footprint fixed at start-up, custom allocators that own
all device memory, code under a memory budget or that cannot afford the implicit
synchronisation of cudaMalloc). Its scratch is a fixed device array inside the library,
so its output must match the regular entry point's, call after call; problems larger
than the array must be refused; its bounded waits must report through the caller's
status word; and its calls must not change the device's free memory.

Collected last on purpose (file name), and written to pass both alone and after the
other GPU tests."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import SENTINEL, bf16_f64, dev, sentinel_like

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_gemm_nt_gb300 as lib
    lib.load_library()
    return lib


def _operands(p: W.Dense):
    c = dev(p.c.view(np.int16), torch.bfloat16) if p.c is not None else None
    return dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb), c


def _no_alloc_call(L, a, sfa, b, sfb, c, d, status, M, N, K):
    """Straight through the C ABI (ctypes), no Python-side checks."""
    raw = L.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    return raw.dg_fp8_gemm_nt_no_alloc(a.data_ptr(), sfa.data_ptr(), b.data_ptr(), sfb.data_ptr(),
                                       None if c is None else c.data_ptr(), d.data_ptr(), status.data_ptr(),
                                       M, N, K, stream)


@pytest.mark.parametrize("M,N,K,with_c", [
    (128, 7168, 16384, True),     # the decode shape
    (200, 384, 4096, True),
    (64, 1024, 2048, False),
    # fewer CTAs than tiles (kgroups / 4 < tiles): whole tiles per CTA, several segments each
    (128, 1024, 128, True),       # 8 tiles of one K-group on 2 CTAs
    (128, 128, 128, False),       # a single CTA
    (1024, 1024, 256, True),      # 64 tiles on 32 CTAs
    (200, 384, 256, False),       # ragged M, 6 tiles on 3 CTAs
])
def test_no_alloc_matches_regular_entry_point_twice(L, M, N, K, with_c):
    p = W.make_dense(M, N, K, seed=1200 + M + N + K, with_c=with_c)
    a, sfa, b, sfb, c = _operands(p)
    d_ref = sentinel_like((M, N))
    L.dg_fp8_gemm_nt(a, sfa, b, sfb, c, d_ref)
    torch.cuda.synchronize()
    ref = bf16_f64(d_ref)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):                      # the second call reuses the scratch as left by the first
        d = sentinel_like((M, N))
        assert _no_alloc_call(L, a, sfa, b, sfb, c, d, status, M, N, K) == 0
        torch.cuda.synchronize()
        rep = O.parity_report(bf16_f64(d), ref)
        assert rep["ok"], f"call {call}: {rep}"
        assert int(status.item()) == 0


def test_no_alloc_against_oracle(L):
    p = W.make_dense(128, 1024, 8192, seed=77, with_c=True)
    a, sfa, b, sfb, c = _operands(p)
    d = sentinel_like((p.M, p.N))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _no_alloc_call(L, a, sfa, b, sfb, c, d, status, p.M, p.N, p.K) == 0
    torch.cuda.synchronize()
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, p.M, p.N, p.K)
    rep = O.parity_report(bf16_f64(d), ref)
    assert rep["ok"], rep
    assert int(status.item()) == 0


def test_no_alloc_refuses_problems_larger_than_its_scratch(L):
    M, N, K = 4096, 4096, 512                 # needs far more than the 16 MiB scratch
    a = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    b = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    sfa = torch.zeros((1, M), dtype=torch.int32, device="cuda")
    sfb = torch.zeros((1, N // 128), dtype=torch.int32, device="cuda")
    d = sentinel_like((M, N))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _no_alloc_call(L, a, sfa, b, sfb, None, d, status, M, N, K) == 1   # DG_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (d.view(torch.int16).cpu().numpy().view(np.uint16) == SENTINEL).all()   # nothing launched


def test_no_alloc_small_problems_against_oracle(L):
    # the fewer-CTAs-than-tiles partition, checked against the oracle directly, rows past M untouched
    for (M, N, K) in [(128, 1024, 128), (1024, 1024, 256), (200, 384, 256)]:
        p = W.make_dense(M, N, K, seed=90 + M + N + K, with_c=True)
        a, sfa, b, sfb, c = _operands(p)
        d_full = sentinel_like((M + 8, N))
        d = d_full[:M]
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _no_alloc_call(L, a, sfa, b, sfb, c, d, status, M, N, K) == 0
        torch.cuda.synchronize()
        ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
        rep = O.parity_report(bf16_f64(d), ref)
        assert rep["ok"], (M, N, K, rep)
        assert (d_full[M:].view(torch.int16).cpu().numpy().view(np.uint16) == SENTINEL).all()
        assert int(status.item()) == 0


def test_no_alloc_timeout_reaches_callers_status_word(L):
    # the producer issues nothing, the bounded waits run out: the caller's word gets the timeout
    # bit, the context stays usable and the next call (fault switched off) is correct
    p = W.make_dense(128, 2048, 4096, seed=31, with_c=False)
    a, sfa, b, sfb, c = _operands(p)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = sentinel_like((p.M, p.N))
    L.dg_set_debug(1, 20_000_000)
    try:
        assert _no_alloc_call(L, a, sfa, b, sfb, c, d, status, p.M, p.N, p.K) == 0
        torch.cuda.synchronize()
    finally:
        L.dg_set_debug(0, 0)
    assert int(status.item()) == 1 << 5          # 1 << DG_ERR_TIMEOUT
    status.zero_()
    d = sentinel_like((p.M, p.N))
    assert _no_alloc_call(L, a, sfa, b, sfb, c, d, status, p.M, p.N, p.K) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, None, p.M, p.N, p.K)
    rep = O.parity_report(bf16_f64(d), ref)
    assert rep["ok"], rep


def test_no_alloc_calls_leave_free_device_memory_unchanged(L):
    p = W.make_dense(128, 7168, 16384, seed=32, with_c=True)
    a, sfa, b, sfb, c = _operands(p)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [sentinel_like((p.M, p.N)) for _ in range(3)]
    assert _no_alloc_call(L, a, sfa, b, sfb, c, outs[0], status, p.M, p.N, p.K) == 0   # set-up call
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for d in outs[1:]:
        assert _no_alloc_call(L, a, sfa, b, sfb, c, d, status, p.M, p.N, p.K) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert int(status.item()) == 0
    first = outs[0].view(torch.int16).cpu()
    for d in outs[1:]:
        assert torch.equal(d.view(torch.int16).cpu(), first)   # deterministic partition and order
