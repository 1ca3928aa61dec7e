"""Stream-K (split over K across SMs) parity and determinism, and the bounded-wait
failure path: a kernel whose producer never issues a load must end with
DG_ERR_TIMEOUT in the device status word and leave the context usable."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import assert_parity, bf16_bits, bf16_f64, run_dense

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_gemm_nt_gb300 as L
    L.load_library()
    return L


@pytest.fixture(autouse=True)
def _stream_k_only(monkeypatch):
    # shapes that would take the split-K cluster path (tests/test_split_gpu.py) stay on stream-K here
    monkeypatch.setenv("DG_SPLIT", "0")


# shapes with fewer 128 x 128 tiles than SMs, so the K-groups are shared among CTAs
SK_SHAPES = [
    (128, 1024, 8192, False),     # 8 tiles, 64 K-groups each: many contributors per tile
    (200, 384, 4096, True),       # ragged M, 6 tiles, with C
    (64, 7168, 16384, True),      # the decode shape with half the rows
    (128, 256, 2304, False),      # 2 tiles, K-groups not a multiple of 4 per CTA
    (1, 128, 1152, True),         # one row
]


@pytest.mark.parametrize("M,N,K,with_c", SK_SHAPES)
def test_stream_k_parity(lib, M, N, K, with_c):
    lib.dg_get_device_status()
    p = W.make_dense(M, N, K, seed=500 + M + N + K, with_c=with_c)
    d = run_dense(lib, p)
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
    assert_parity(bf16_f64(d), ref, f"stream-K {M}x{N}x{K}")
    assert lib.dg_get_device_status() == 0


def test_stream_k_is_deterministic(lib):
    p = W.make_dense(128, 1024, 8192, seed=9, with_c=True)
    first = bf16_bits(run_dense(lib, p))
    for _ in range(3):
        assert np.array_equal(bf16_bits(run_dense(lib, p)), first)


def test_stream_k_small_sm_cap(lib):
    # capping the SM count changes the partition; results stay within tolerance
    p = W.make_dense(128, 512, 4096, seed=10)
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, None, p.M, p.N, p.K)
    try:
        for sms in (5, 17, 64):
            lib.dg_set_num_sms(sms)
            assert lib.dg_get_num_sms() == sms
            assert_parity(bf16_f64(run_dense(lib, p)), ref, f"sms={sms}")
    finally:
        lib.dg_set_num_sms(0)
    assert lib.dg_get_device_status() == 0


@pytest.mark.parametrize("shape", [(256, 256, 512), (128, 2048, 4096)])
def test_timeout_is_reported_and_context_survives(lib, shape):
    M, N, K = shape
    p = W.make_dense(M, N, K, seed=3)
    lib.dg_get_device_status()
    lib.dg_set_debug(1, 20_000_000)          # producer issues nothing; waits give up after 20 ms
    try:
        run_dense(lib, p)
        assert lib.dg_get_device_status() == 5   # DG_ERR_TIMEOUT
    finally:
        lib.dg_set_debug(0, 0)
    # the same call works afterwards
    d = run_dense(lib, p)
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, None, M, N, K)
    assert_parity(bf16_f64(d), ref, "after timeout")
    assert lib.dg_get_device_status() == 0


@pytest.mark.parametrize("sk_bn", [128, 192, 256])
@pytest.mark.parametrize("M,N,K", [(128, 2048, 8192), (96, 7168, 4096)])
def test_stream_k_tile_widths(lib, sk_bn, M, N, K, monkeypatch):
    monkeypatch.setenv("DG_SK_BN", str(sk_bn))
    p = W.make_dense(M, N, K, seed=700 + sk_bn + M, with_c=True)
    d = run_dense(lib, p)
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
    assert_parity(bf16_f64(d), ref, f"stream-K bn={sk_bn}")
    assert lib.dg_get_device_status() == 0


@pytest.mark.parametrize("kg", ["1", "2"])
@pytest.mark.parametrize("M,N,K", [(128, 1024, 1152), (100, 640, 2944), (128, 7168, 16384)])
def test_stream_k_kgroups_per_stage(lib, kg, M, N, K, monkeypatch):
    # one or two K-groups per pipeline stage; odd K-group counts leave a half-filled last stage
    monkeypatch.setenv("DG_KG", kg)
    p = W.make_dense(M, N, K, seed=800 + M + N + K, with_c=True)
    d = run_dense(lib, p)
    rows = np.arange(M) if M * N * K < 2 ** 31 else np.arange(0, M, 5)
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K, rows=rows)
    assert_parity(bf16_f64(d)[rows], ref, f"stream-K kg={kg}")
    assert lib.dg_get_device_status() == 0
