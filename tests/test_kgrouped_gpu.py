"""K-grouped weight-gradient GEMM (MoE experts, each owning a K-slice; FP32 output per
expert) against the FP64 oracle: several expert-size mixes including empty experts, every
tile width, accumulation in place, empty experts with and without C, and malformed slice
sizes reported through the device status word."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import assert_parity, dev, run_k_grouped

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


def _ref(p, c=None):
    return O.k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(p.a, p.sfa, p.b, p.sfb, p.c if c is None else c, p.ks, p.M, p.N)


@pytest.mark.parametrize("ks,M,N,with_c,bn", [
    ([256, 0, 384], 256, 384, True, None),
    ([128, 512, 0, 640], 300, 272, False, None),      # ragged M and N, an empty expert
    ([384, 128], 512, 512, True, "128"),
    ([256, 768, 128], 384, 640, True, "192"),
    ([1152], 128, 256, False, "256"),                 # one expert, K-groups not a multiple of 4
])
def test_k_grouped_parity(lib, monkeypatch, ks, M, N, with_c, bn):
    if bn is not None:
        monkeypatch.setenv("DG_FORCE_BN", bn)
    p = W.make_k_grouped(G=len(ks), M=M, N=N, tokens=0, seed=900 + M + N, with_c=with_c, ks=np.array(ks))
    d = run_k_grouped(lib, p).cpu().numpy().astype(np.float64)
    ref = _ref(p)
    for g in range(p.G):
        rep = assert_parity(d[g], ref[g], f"expert {g} ks={ks}")
        assert rep["max_err"] <= 1e-5 * max(rep["rms"], 1e-30), rep
    assert lib.dg_get_device_status() == 0


def test_k_grouped_empty_expert_writes_c_or_zero(lib):
    p = W.make_k_grouped(G=3, M=256, N=256, tokens=0, seed=5, with_c=True, ks=np.array([0, 256, 0]))
    d = run_k_grouped(lib, p).cpu().numpy()
    assert np.array_equal(d[0], p.c[0]) and np.array_equal(d[2], p.c[2])
    q = W.make_k_grouped(G=2, M=128, N=128, tokens=0, seed=6, with_c=False, ks=np.array([128, 0]))
    d = run_k_grouped(lib, q).cpu().numpy()
    assert (d[1] == 0).all()
    assert lib.dg_get_device_status() == 0


def test_k_grouped_accumulates_in_place(lib):
    p = W.make_k_grouped(G=3, M=256, N=384, tokens=0, seed=7, with_c=True, ks=np.array([256, 128, 384]))
    c0 = p.c.astype(np.float64)
    d = dev(p.c)
    args = (dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb))
    ks = dev(np.asarray(p.ks, np.int32))
    for _ in range(2):
        lib.dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(*args, d, d, ks)
    torch.cuda.synchronize()
    prod = O.k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(p.a, p.sfa, p.b, p.sfb, None, p.ks, p.M, p.N)
    got = d.cpu().numpy().astype(np.float64)
    for g in range(p.G):
        assert_parity(got[g], c0[g] + 2.0 * prod[g], f"expert {g}")
    assert lib.dg_get_device_status() == 0


def test_k_grouped_no_tokens_at_all(lib):
    M, N, G = 128, 256, 2
    c = torch.randn((G, M, N), dtype=torch.float32, device="cuda")
    d = torch.full((G, M, N), float("nan"), dtype=torch.float32, device="cuda")
    a = torch.zeros((M, 0), dtype=torch.uint8, device="cuda")
    b = torch.zeros((N, 0), dtype=torch.uint8, device="cuda")
    sfa = torch.zeros((0, M), dtype=torch.int32, device="cuda")
    sfb = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    ks = torch.zeros((G,), dtype=torch.int32, device="cuda")
    lib.dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(a, sfa, b, sfb, c, d, ks)
    torch.cuda.synchronize()
    assert torch.equal(d, c)


@pytest.mark.parametrize("bad_ks", [[256, 200], [128, 128], [512, -128]])
def test_k_grouped_bad_slices_reported(lib, bad_ks):
    # the operands are built for slices [256, 256]; other sizes violate the layout
    p = W.make_k_grouped(G=2, M=128, N=256, tokens=0, seed=8, with_c=False, ks=np.array([256, 256]))
    p.ks = np.array(bad_ks, np.int32)
    run_k_grouped(lib, p)
    assert lib.dg_get_device_status() == 6
    assert lib.dg_get_device_status() == 0


# --------------------------------------------------------------------------------------
# CTA-pair kernel (with 8 SMs in use, small problems have enough tiles to take it)
# --------------------------------------------------------------------------------------

@pytest.fixture
def few_sms(lib):
    lib.dg_set_num_sms(8)
    yield
    lib.dg_set_num_sms(0)


@pytest.mark.parametrize("bn", ["256", "192"])
@pytest.mark.parametrize("ks,M,N,with_c", [
    ([256, 0, 384], 256, 384, True),
    ([128, 512, 0, 640], 300, 272, False),    # ragged M (an odd number of 128-row blocks) and N, an empty expert
    ([1152], 384, 256, True),                 # one expert, K-groups not a multiple of 4
    ([384, 128, 256], 512, 512, True),
])
def test_k_grouped_pair(lib, few_sms, monkeypatch, bn, ks, M, N, with_c):
    monkeypatch.setenv("DG_PAIR_BN", bn)
    p = W.make_k_grouped(G=len(ks), M=M, N=N, tokens=0, seed=700 + M + N, with_c=with_c, ks=np.array(ks))
    d = run_k_grouped(lib, p).cpu().numpy().astype(np.float64)
    ref = _ref(p)
    for g in range(p.G):
        rep = assert_parity(d[g], ref[g], f"pair expert {g} ks={ks}")
        assert rep["max_err"] <= 1e-5 * max(rep["rms"], 1e-30), rep
    assert lib.dg_get_device_status() == 0


def test_k_grouped_pair_in_place_with_empty_expert(lib, few_sms):
    p = W.make_k_grouped(G=3, M=384, N=512, tokens=0, seed=17, with_c=True, ks=np.array([256, 0, 640]))
    c0 = p.c.astype(np.float64)
    d = dev(p.c)
    args = (dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb))
    ks = dev(np.asarray(p.ks, np.int32))
    for _ in range(2):
        lib.dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(*args, d, d, ks)
    torch.cuda.synchronize()
    prod = O.k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(p.a, p.sfa, p.b, p.sfb, None, p.ks, p.M, p.N)
    got = d.cpu().numpy().astype(np.float64)
    assert np.array_equal(got[1], c0[1])          # the empty expert keeps its addend exactly
    for g in (0, 2):
        assert_parity(got[g], c0[g] + 2.0 * prod[g], f"pair in place, expert {g}")
    assert lib.dg_get_device_status() == 0


def test_k_grouped_pair_bad_slices_reported(lib, few_sms):
    p = W.make_k_grouped(G=2, M=256, N=512, tokens=0, seed=18, with_c=False, ks=np.array([256, 256]))
    p.ks = np.array([256, 200], np.int32)
    run_k_grouped(lib, p)
    assert lib.dg_get_device_status() == 6
    assert lib.dg_get_device_status() == 0
