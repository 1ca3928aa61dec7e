"""Weight-gradient GEMM with FP32 output (D = C + A @ B.T, C may be D itself) against the
FP64 oracle: stream-K shapes (few tiles) and tile-mode shapes for every tile width,
accumulation in place, and the exact cases (C only, identity operands)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import assert_parity, dev, run_wgrad

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_gemm_nt_gb300 as L
    L.load_library()
    return L


@pytest.fixture(autouse=True)
def _clean(lib):
    lib.dg_get_device_status()
    yield
    assert lib.dg_get_device_status() == 0


@pytest.mark.parametrize("M,N,K,with_c,bn", [
    (128, 256, 512, False, None),      # stream-K
    (300, 400, 640, True, None),       # stream-K, ragged M and N
    (2048, 1536, 512, True, None),     # tile mode
    (2048, 1536, 384, True, "128"),
    (2048, 1536, 1152, False, "192"),
    (1000, 2304, 256, True, "256"),    # ragged M
])
def test_wgrad_parity(lib, monkeypatch, M, N, K, with_c, bn):
    if bn is not None:
        monkeypatch.setenv("DG_FORCE_BN", bn)
    p = W.make_wgrad(M, N, K, seed=800 + M + N + K, with_c=with_c)
    d = run_wgrad(lib, p).cpu().numpy().astype(np.float64)
    ref = O.wgrad_gemm_fp8_fp8_fp32_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
    rep = assert_parity(d, ref, f"wgrad {M}x{N}x{K}")
    # the FP32 output keeps what the BF16 form rounds away: the error stays far inside the bar
    print(f"wgrad {M}x{N}x{K}: max |d - ref| / rms(ref) = {rep['max_err'] / rep['rms']:.3e}")
    # measured on GB300: 6e-7 .. 1e-6 (FP32 accumulation); the bound leaves a factor of ten
    assert rep["max_err"] <= 1e-5 * rep["rms"], rep


def test_wgrad_accumulates_in_place(lib):
    p = W.make_wgrad(2048, 1536, 512, seed=31, with_c=True)
    c0 = p.c.astype(np.float64)
    d = dev(p.c)
    args = (dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb))
    for _ in range(2):
        lib.dg_wgrad_gemm_fp8_fp8_fp32_nt(*args, d, d)
    torch.cuda.synchronize()
    prod = O.wgrad_gemm_fp8_fp8_fp32_nt(p.a, p.sfa, p.b, p.sfb, None, p.M, p.N, p.K)
    assert_parity(d.cpu().numpy().astype(np.float64), c0 + 2.0 * prod, "two accumulations")


def test_wgrad_c_only_bit_exact(lib):
    p = W.make_wgrad(256, 512, 256, seed=32, with_c=True)
    p.a[:] = 0
    d = run_wgrad(lib, p).cpu().numpy()
    assert np.array_equal(d, p.c)


def test_wgrad_identity_exact(lib):
    # A = [I | 0] with unit scales: D[i, n] = B[n, i] exactly (E4M3 values are exact in FP32)
    M, N, K = 128, 384, 256
    rng = np.random.default_rng(33)
    a = np.zeros((M, K), np.uint8)
    a[np.arange(M), np.arange(M)] = 0x38
    b = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    b[(b & 0x7F) == 0x7F] = 0x30
    p = W.Wgrad(a, W.pack_sf(np.full((M, 2), 127, np.uint8)), b, W.pack_sf(np.full((3, 2), 127, np.uint8)),
                None, M, N, K)
    d = run_wgrad(lib, p).cpu().numpy().astype(np.float64)
    assert np.array_equal(d, O.decode_e4m3(b[:, :M]).T)


@pytest.mark.parametrize("pair_bn", [256, 240, 192])
@pytest.mark.parametrize("M,N,K,with_c", [
    (512, 496, 640, True),     # N = 2 x 240 + 16: the 240-wide tile's 16-column FP32 box lies past N
    (384, 768, 1152, False),   # an odd number of 128-row blocks
])
def test_wgrad_pair(lib, monkeypatch, pair_bn, M, N, K, with_c):
    # the CTA-pair kernel with its FP32 epilogue (the SM cap makes these shapes tile-mode)
    monkeypatch.setenv("DG_PAIR_BN", str(pair_bn))
    lib.dg_set_num_sms(8)
    try:
        p = W.make_wgrad(M, N, K, seed=850 + M + N + K + pair_bn, with_c=with_c)
        d = run_wgrad(lib, p).cpu().numpy().astype(np.float64)
    finally:
        lib.dg_set_num_sms(0)
    ref = O.wgrad_gemm_fp8_fp8_fp32_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
    rep = assert_parity(d, ref, f"wgrad pair {pair_bn} {M}x{N}x{K}")
    assert rep["max_err"] <= 1e-5 * rep["rms"], rep
