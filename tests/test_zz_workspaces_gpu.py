"""The per-stream workspaces on the GPU: a CUDA graph replayed after the workspace cache has
turned over, and host threads that share the cache.

Runs last in the session: the workspace captured here stays allocated until the process
exits. The policy itself is checked on the host by tests/test_workspace_cache.py.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import bf16_bits, dev, sentinel_like

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_gemm_nt_gb300 as L
    L.load_library()
    return L


def _operands(seed):
    # fewer 128 x 128 tiles than SMs: the stream-K path, which uses its stream's workspace on
    # every call and sums its partials in a fixed order (the same bits on every stream)
    p = W.make_dense(256, 384, 1152, seed=seed)
    return p, (dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb))


def test_graph_replays_after_the_workspace_cache_turned_over(lib):
    p, (a, sfa, b, sfb) = _operands(57)
    lib.dg_get_device_status()
    s = torch.cuda.Stream()
    d = sentinel_like((p.M, p.N))
    with torch.cuda.stream(s):
        lib.dg_fp8_gemm_nt(a, sfa, b, sfb, None, d)      # the stream's workspace, before capture
    torch.cuda.synchronize()
    want = bf16_bits(d)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        lib.dg_fp8_gemm_nt(a, sfa, b, sfb, None, d)
    # more streams than the cache keeps: the workspaces no graph uses are released and
    # rebuilt, the captured one is kept
    others = []
    for t in [torch.cuda.Stream() for _ in range(24)]:
        e = sentinel_like((p.M, p.N))
        with torch.cuda.stream(t):
            lib.dg_fp8_gemm_nt(a, sfa, b, sfb, None, e)
        others.append(e)
    torch.cuda.synchronize()
    for i, e in enumerate(others):
        assert np.array_equal(bf16_bits(e), want), f"stream {i}"
    d.zero_()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(d), want)
    assert lib.dg_get_device_status() == 0


def test_host_threads_share_the_workspace_cache(lib):
    # four host threads, six streams each (24 streams: more than the cache keeps), so
    # workspaces are released while other threads are between their lookup and their launch
    p, (a, sfa, b, sfb) = _operands(58)
    lib.dg_get_device_status()
    ref = sentinel_like((p.M, p.N))
    lib.dg_fp8_gemm_nt(a, sfa, b, sfb, None, ref)
    torch.cuda.synchronize()
    want = bf16_bits(ref)

    def worker(_):
        streams = [torch.cuda.Stream() for _ in range(6)]
        outs = []
        for i in range(18):
            s = streams[i % len(streams)]
            with torch.cuda.stream(s):
                d = torch.empty((p.M, p.N), dtype=torch.bfloat16, device="cuda")
                lib.dg_fp8_gemm_nt(a, sfa, b, sfb, None, d)
            outs.append(d)
        for s in streams:
            s.synchronize()
        return [bf16_bits(d) for d in outs]

    with ThreadPoolExecutor(max_workers=4) as ex:
        results = list(ex.map(worker, range(4)))
    for t, outs in enumerate(results):
        for i, bits in enumerate(outs):
            assert np.array_equal(bits, want), f"thread {t}, call {i}"
    assert lib.dg_get_device_status() == 0


def test_reserved_workspace_calls_allocate_nothing(lib):
    # a warm-up call sizes the stream's workspace, dg_reserve_workspace(0) pins it; later calls on
    # that stream (while other streams come and go) leave the device's free memory unchanged
    p, (a, sfa, b, sfb) = _operands(59)
    s = torch.cuda.Stream()
    d = sentinel_like((p.M, p.N))
    with torch.cuda.stream(s):
        lib.dg_fp8_gemm_nt(a, sfa, b, sfb, None, d)
        lib.dg_reserve_workspace(0, stream=s)
    torch.cuda.synchronize()
    size = lib.dg_get_workspace_size(stream=s)
    assert size > 0
    want = bf16_bits(d)
    outs = [sentinel_like((p.M, p.N)) for _ in range(8)]
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    with torch.cuda.stream(s):
        for e in outs:
            lib.dg_fp8_gemm_nt(a, sfa, b, sfb, None, e)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    for e in outs:
        assert np.array_equal(bf16_bits(e), want)
    # other streams churn through the cache; the reserved workspace is never evicted
    for t in [torch.cuda.Stream() for _ in range(20)]:
        with torch.cuda.stream(t):
            lib.dg_fp8_gemm_nt(a, sfa, b, sfb, None, sentinel_like((p.M, p.N)))
    torch.cuda.synchronize()
    assert lib.dg_get_workspace_size(stream=s) == size
    lib.dg_release_workspace(stream=s)
    assert lib.dg_get_workspace_size(stream=s) == 0
    assert lib.dg_get_device_status() == 0


def test_reserve_up_front_then_first_call_allocates_nothing(lib):
    p, (a, sfa, b, sfb) = _operands(60)
    s = torch.cuda.Stream()
    lib.dg_reserve_workspace(64 << 20, stream=s)        # well above what this shape needs
    assert lib.dg_get_workspace_size(stream=s) >= 64 << 20
    d = sentinel_like((p.M, p.N))
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    with torch.cuda.stream(s):
        lib.dg_fp8_gemm_nt(a, sfa, b, sfb, None, d)      # the stream's first GEMM call
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    ref = sentinel_like((p.M, p.N))
    lib.dg_fp8_gemm_nt(a, sfa, b, sfb, None, ref)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(d), bf16_bits(ref))
    lib.dg_release_workspace(stream=s)
    assert lib.dg_get_device_status() == 0
