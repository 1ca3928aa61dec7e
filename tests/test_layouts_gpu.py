"""The NN / TN / TT layouts (M-major A given as [K, M], N-major B given as [K, N]) against
the oracle, in tile mode (both tile widths) and stream-K; and bit-identical to the NT form
on the same logical problem when the same kernel configuration runs (the operand layout
changes only how tiles reach shared memory, not the MMAs)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import assert_parity, bf16_bits, bf16_f64, dev, sentinel_like

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


def _stored(p, layout):
    a = p.a if layout[0] == "n" else np.ascontiguousarray(p.a.T)
    b = np.ascontiguousarray(p.b.T) if layout[1] == "n" else p.b
    return a, b


def _run(lib, layout, p):
    a, b = _stored(p, layout)
    c = dev(p.c.view(np.int16), torch.bfloat16) if p.c is not None else None
    d = sentinel_like((p.M, p.N))
    getattr(lib, f"dg_fp8_gemm_{layout}")(dev(a), dev(p.sfa), dev(b), dev(p.sfb), c, d)
    torch.cuda.synchronize()
    return d


def _oracle(layout, p):
    a, b = _stored(p, layout)
    return getattr(O, f"fp8_gemm_{layout}")(a, p.sfa, b, p.sfb, p.c, p.M, p.N, p.K)


@pytest.mark.parametrize("layout", ["nn", "tn", "tt"])
@pytest.mark.parametrize("M,N,K,with_c,bn", [
    (128, 256, 512, False, None),       # stream-K
    (208, 400, 1152, True, None),       # stream-K, ragged M and N, K-groups not a multiple of 4
    (2048, 1536, 512, True, "256"),     # tile mode
    (2048, 1536, 640, False, "128"),
    (1040, 2304, 256, True, "256"),     # tile mode, ragged M
])
def test_layout_parity(lib, monkeypatch, layout, M, N, K, with_c, bn):
    if bn is not None:
        monkeypatch.setenv("DG_FORCE_BN", bn)
    p = W.make_dense(M, N, K, seed=1300 + M + N + K, with_c=with_c)
    d = _run(lib, layout, p)
    assert_parity(bf16_f64(d), _oracle(layout, p), f"{layout} {M}x{N}x{K}")


@pytest.mark.parametrize("bn", ["256", "128"])
def test_layouts_bit_identical_to_nt(lib, monkeypatch, bn):
    # one kernel configuration for all four: the single-CTA tile mode at the same width
    monkeypatch.setenv("DG_FORCE_BN", bn)
    monkeypatch.setenv("DG_PAIR", "0")
    p = W.make_dense(2048, 1536, 768, seed=1400, with_c=True)
    ref = bf16_bits(_run(lib, "nt", p))
    for layout in ("nn", "tn", "tt"):
        assert np.array_equal(bf16_bits(_run(lib, layout, p)), ref), layout


def test_tn_identity_exact(lib):
    # A' = [I | 0] (stored transposed), unit scales: D[i, n] = B''[i, n] exactly
    M, N, K = 128, 256, 256
    rng = np.random.default_rng(9)
    a = np.zeros((M, K), np.uint8)
    a[np.arange(M), np.arange(M)] = 0x38
    b = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    b[(b & 0x7F) == 0x7F] = 0x30
    p = W.Dense(a, W.pack_sf(np.full((M, 2), 127, np.uint8)), b, W.pack_sf(np.full((2, 2), 127, np.uint8)),
                None, M, N, K)
    got = bf16_f64(_run(lib, "tn", p))
    assert np.array_equal(got, O.decode_e4m3(b[:, :M]).T)


def test_t_layout_rejects_m_not_multiple_of_16(lib):
    import ctypes
    raw = lib.load_library()
    x = ctypes.c_void_p(0x10000)
    assert raw.dg_fp8_gemm_tn(x, x, x, x, None, x, 100, 128, 128, None) == 1
    assert raw.dg_fp8_gemm_tt(x, x, x, x, None, x, 100, 128, 128, None) == 1


@pytest.mark.parametrize("bn", [None, "128"])
@pytest.mark.parametrize("counts,N,K", [
    ([130, 0, 170, 1], 144, 256),
    ([128, 256, 5, 300], 400, 640),
])
def test_nn_contiguous_parity(lib, monkeypatch, bn, counts, N, K):
    from gpu_util import SENTINEL
    if bn is not None:
        monkeypatch.setenv("DG_FORCE_BN", bn)
    p = W.make_contiguous(G=len(counts), tokens=sum(counts), N=N, K=K, seed=1500 + N, counts=counts)
    b_kn = np.ascontiguousarray(p.b.transpose(0, 2, 1))
    d = sentinel_like((p.M_total, p.N))
    lib.dg_m_grouped_fp8_gemm_nn_contiguous(dev(p.a), dev(p.sfa), dev(b_kn), dev(p.sfb), d, dev(p.m_indices))
    torch.cuda.synchronize()
    ref, valid = O.m_grouped_fp8_gemm_nn_contiguous(p.a, p.sfa, b_kn, p.sfb, p.m_indices, p.M_total, p.N, p.K, p.G)
    bits = bf16_bits(d)
    assert (bits[~valid] == SENTINEL).all()
    assert_parity(bf16_f64(d)[valid], ref[valid], f"nn contiguous {counts}")
    # the NT form at the same width computes the same bits
    monkeypatch.setenv("DG_FORCE_BN", bn or ("256" if -(-N // 256) * 256 <= -(-N // 128) * 128 else "128"))
    d_nt = sentinel_like((p.M_total, p.N))
    lib.dg_m_grouped_fp8_gemm_nt_contiguous(dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb), d_nt, dev(p.m_indices))
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(d_nt), bits)


@pytest.mark.parametrize("ks,M,N,with_c", [
    ([256, 0, 384], 256, 384, True),
    ([128, 512, 640], 208, 272, False),      # ragged M (multiple of 16) and N
])
def test_tn_k_grouped_parity(lib, monkeypatch, ks, M, N, with_c):
    p = W.make_k_grouped(G=len(ks), M=M, N=N, tokens=0, seed=1600 + M + N, with_c=with_c, ks=np.array(ks))
    a_t, b_t = np.ascontiguousarray(p.a.T), np.ascontiguousarray(p.b.T)
    c = dev(p.c) if p.c is not None else None
    d = torch.full((p.G, M, N), float("nan"), dtype=torch.float32, device="cuda")
    lib.dg_k_grouped_fp8_gemm_tn_contiguous(dev(a_t), dev(p.sfa), dev(b_t), dev(p.sfb), c, d,
                                            dev(np.asarray(p.ks, np.int32)))
    torch.cuda.synchronize()
    got = d.cpu().numpy().astype(np.float64)
    ref = O.k_grouped_fp8_gemm_tn_contiguous(a_t, p.sfa, b_t, p.sfb, p.c, p.ks, M, N)
    for g in range(p.G):
        rep = assert_parity(got[g], ref[g], f"tn k-grouped expert {g}")
        assert rep["max_err"] <= 1e-5 * max(rep["rms"], 1e-30), rep
    # the NT K-grouped form at the same width computes the same bits
    monkeypatch.setenv("DG_FORCE_BN", "256" if -(-N // 256) * 256 <= -(-N // 128) * 128 else "128")
    d_nt = torch.full((p.G, M, N), float("nan"), dtype=torch.float32, device="cuda")
    lib.dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb), c, d_nt,
                                                dev(np.asarray(p.ks, np.int32)))
    torch.cuda.synchronize()
    monkeypatch.delenv("DG_FORCE_BN")
    assert torch.equal(d_nt, d)


# --------------------------------------------------------------------------------------
# CTA-pair kernel (256-wide tiles) with MN-major operands; 8 SMs in use so that small
# problems have enough tiles to take it
# --------------------------------------------------------------------------------------

@pytest.fixture
def few_sms(lib):
    lib.dg_set_num_sms(8)
    yield
    lib.dg_set_num_sms(0)


@pytest.mark.parametrize("layout", ["nn", "tn", "tt"])
@pytest.mark.parametrize("M,N,K,with_c", [
    (512, 512, 640, True),
    (304, 400, 1152, True),     # ragged M (an odd number of 128-row blocks) and N, K-groups not a multiple of 4
    (1024, 768, 2048, False),   # several pair tiles per CTA pair
])
def test_layout_pair_parity(lib, few_sms, layout, M, N, K, with_c):
    p = W.make_dense(M, N, K, seed=1500 + M + N + K, with_c=with_c)
    d = _run(lib, layout, p)
    assert_parity(bf16_f64(d), _oracle(layout, p), f"pair {layout} {M}x{N}x{K}")


def test_layout_pair_bit_identical_to_nt(lib, few_sms, monkeypatch):
    # the four layouts on the 256-wide pair kernel: the same MMAs, only the tiles' shared-
    # memory layout differs
    monkeypatch.setenv("DG_PAIR_BN", "256")
    p = W.make_dense(1024, 1024, 768, seed=1600, with_c=True)
    ref = bf16_bits(_run(lib, "nt", p))
    for layout in ("nn", "tn", "tt"):
        assert np.array_equal(bf16_bits(_run(lib, layout, p)), ref), layout
