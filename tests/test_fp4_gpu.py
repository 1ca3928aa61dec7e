"""GPU parity of the FP8 x FP4 GEMMs (B in E2M1 with one UE8M0 scale per row per 32 K) against
the FP64 oracle, through the C ABI.

Bar as for the FP8 forms: per element |d - ref| <= 1e-2*|ref| + 1e-2*rms(ref) and the
cosine-style difference below 1e-3; bit-exact where the result is exact in BF16 (one-hot
B) and for everything integer indexing decides (padding and masked rows keep the sentinel).
The shapes are chosen to reach every launch form the dispatcher has for FP4 B: the CTA-pair
kernel at each width (256, 240, 192), single-CTA tile mode with 128- and 256-wide tiles,
stream-K with two K-groups per stage (an odd K-group count leaves the last stage half past
K), and split-K over CTA pairs.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import (SENTINEL, assert_parity, bf16_bits, bf16_f64, dev, run_contiguous, run_dense, run_masked,
                      sentinel_like)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_gemm_nt_gb300 as L
    L.load_library()
    return L


@pytest.fixture(autouse=True)
def _clean_status(lib):
    lib.dg_get_device_status()
    yield
    assert lib.dg_get_device_status() == 0, "device status set by a test that expected none"


DENSE_SHAPES = [
    (128, 256, 512, False),      # tile mode, 128-wide tiles
    (1, 16, 128, False),         # one row, one K-group
    (77, 48, 384, True),         # ragged M and N, with C
    (300, 400, 640, True),       # split-K over CTA pairs, ragged tails
    (256, 384, 1152, False),     # stream-K, two K-groups per stage, KG = 9
    (130, 1040, 2048, True),     # split-K, wider
    (513, 272, 256, False),      # tile mode, KG = 2
    (1024, 2560, 256, False),    # >= one tile per SM: the CTA-pair kernel
    (1280, 2432, 384, True),     # the CTA-pair kernel, with C
]


@pytest.mark.parametrize("M,N,K,with_c", DENSE_SHAPES)
def test_fp4_dense_parity(lib, M, N, K, with_c):
    p = W.make_dense_fp4(M, N, K, seed=2000 + M + N + K, with_c=with_c)
    d = run_dense(lib, p)
    ref = O.fp8_fp4_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
    assert_parity(bf16_f64(d), ref, f"fp4 dense {M}x{N}x{K}")


def test_fp4_c_aliases_d(lib):
    p = W.make_dense_fp4(200, 320, 512, seed=5, with_c=True)
    d = run_dense(lib, p, c_alias=True)
    ref = O.fp8_fp4_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, p.M, p.N, p.K)
    assert_parity(bf16_f64(d), ref, "fp4 c aliases d")


@pytest.mark.parametrize("M,N,K", [(40, 64, 512), (300, 400, 640), (256, 384, 1152)])
def test_fp4_one_hot_exact(lib, M, N, K):
    # B row n holds 1.0 (code 2) at one column k0[n] (even and odd positions, every 32-wide
    # block), so D[m, n] = sA * sB * A[m, k0[n]] is exact in BF16: compare bit for bit.
    rng = np.random.default_rng(M + N)
    p = W.make_dense_fp4(M, N, K, seed=7 + M)
    k0 = rng.integers(0, K, size=N)
    b = np.zeros((N, K // 2), np.uint8)
    for n, k in enumerate(k0):
        b[n, k // 2] = 2 << (4 * (k % 2))
    eb = rng.integers(120, 135, size=(N, K // 32)).astype(np.uint8)
    p.b, p.sfb = b, W.pack_sf(eb)
    d = bf16_f64(run_dense(lib, p))
    ref = O.fp8_fp4_gemm_nt(p.a, p.sfa, p.b, p.sfb, None, M, N, K)
    assert np.array_equal(d, ref)


def test_fp4_every_code_and_scale_byte(lib):
    # each B row repeats one E2M1 code over all of K, with different scale bytes per 32-wide
    # block: a wrong nibble order, code table or scale byte shows up in whole columns
    M, N, K = 64, 256, 512
    rng = np.random.default_rng(3)
    p = W.make_dense_fp4(M, N, K, seed=11)
    codes = np.arange(N) % 16
    p.b = np.repeat(((codes | (codes << 4)).astype(np.uint8))[:, None], K // 2, axis=1)
    eb = rng.integers(118, 137, size=(N, K // 32)).astype(np.uint8)
    p.sfb = W.pack_sf(eb)
    d = run_dense(lib, p)
    ref = O.fp8_fp4_gemm_nt(p.a, p.sfa, p.b, p.sfb, None, M, N, K)
    assert_parity(bf16_f64(d), ref, "every code")


@pytest.mark.parametrize("counts,N,K", [([300, 0, 129], 256, 512), ([1, 255, 200, 77], 384, 896)])
def test_fp4_contiguous_parity_and_padding(lib, counts, N, K):
    p = W.make_contiguous(G=len(counts), tokens=sum(counts), N=N, K=K, seed=61 + N, counts=counts,
                          b_format="e2m1")
    d = run_contiguous(lib, p)
    ref, valid = O.m_grouped_fp8_fp4_gemm_nt_contiguous(p.a, p.sfa, p.b, p.sfb, p.m_indices, p.M_total, p.N, p.K,
                                                        p.G)
    bits = bf16_bits(d)
    assert (bits[~valid] == SENTINEL).all(), "padding rows were written"
    assert_parity(bf16_f64(d)[valid], ref[valid], f"fp4 contiguous {counts}")


def test_fp4_contiguous_equals_dense_per_expert(lib):
    p = W.make_contiguous(G=3, tokens=600, N=256, K=512, seed=9, counts=[250, 100, 250], b_format="e2m1")
    d = bf16_bits(run_contiguous(lib, p))
    ea = O.unpack_sf(p.sfa, p.M_total, p.K // 128)
    for g in range(p.G):
        r = np.nonzero(p.m_indices == g)[0]
        q = W.Dense(p.a[r], W.pack_sf(ea[r]), p.b[g], p.sfb[g], None, len(r), p.N, p.K, b_format="e2m1")
        assert np.array_equal(d[r], bf16_bits(run_dense(lib, q))), f"expert {g}"


@pytest.mark.parametrize("masked_m,max_m,N,K", [([0, 1, 129, 256], 256, 448, 512), ([64, 3], 64, 128, 384),
                                                ([200, 7, 0], 200, 192, 1024)])
def test_fp4_masked_parity_and_mask(lib, masked_m, max_m, N, K):
    p = W.make_masked(G=len(masked_m), max_m=max_m, N=N, K=K, seed=71 + N, masked_m=masked_m, b_format="e2m1")
    d = run_masked(lib, p)
    ref, valid = O.m_grouped_fp8_fp4_gemm_nt_masked(p.a, p.sfa, p.b, p.sfb, p.masked_m, p.G, p.max_m, p.N, p.K)
    bits = bf16_bits(d)
    assert (bits[~valid] == SENTINEL).all(), "masked rows were written"
    assert_parity(bf16_f64(d)[valid], ref[valid], f"fp4 masked {masked_m}")


def test_fp4_masked_graph_replay_sees_new_counts(lib):
    # the counts are read on the device: a captured graph replayed after they change computes
    # the new rows without re-capture
    p = W.make_masked(G=4, max_m=128, N=256, K=512, seed=13, masked_m=[5, 0, 128, 60], b_format="e2m1")
    a, sfa, b, sfb = dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb)
    mm = dev(p.masked_m)
    d = sentinel_like((p.G, p.max_m, p.N))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        lib.dg_m_grouped_fp8_fp4_gemm_nt_masked(a, sfa, b, sfb, d, mm)   # warm (maps, attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        lib.dg_m_grouped_fp8_fp4_gemm_nt_masked(a, sfa, b, sfb, d, mm)
    for counts in ([5, 0, 128, 60], [128, 77, 1, 0]):
        d.copy_(sentinel_like(d.shape))
        mm.copy_(torch.tensor(counts, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        ref, valid = O.m_grouped_fp8_fp4_gemm_nt_masked(p.a, p.sfa, p.b, p.sfb, np.array(counts), p.G, p.max_m,
                                                        p.N, p.K)
        bits = bf16_bits(d)
        assert (bits[~valid] == SENTINEL).all()
        assert_parity(bf16_f64(d)[valid], ref[valid], f"replay {counts}")


def test_fp4_misaligned_b_rejected(lib):
    # b must be 32-byte aligned (16U4 tensor maps); a 16-byte offset is refused before launch
    p = W.make_dense_fp4(64, 64, 256, seed=1)
    raw = torch.zeros(p.b.size + 64, dtype=torch.uint8, device="cuda")
    base = raw.data_ptr()
    off = (32 - base % 32) % 32 + 16
    b = raw[off:off + p.b.size].view(p.N, p.K // 2)
    d = sentinel_like((p.M, p.N))
    with pytest.raises(lib.DGError) as e:
        lib.dg_fp8_fp4_gemm_nt(dev(p.a), dev(p.sfa), b, dev(p.sfb), None, d)
    assert e.value.status == 3
    assert (bf16_bits(d) == SENTINEL).all()


# --------------------------------------------------------------------------------------
# FP4 B on the CTA-pair kernel (with 8 SMs in use, small problems have enough tiles)
# --------------------------------------------------------------------------------------

@pytest.fixture
def few_sms(lib):
    lib.dg_set_num_sms(8)
    yield
    lib.dg_set_num_sms(0)


@pytest.fixture(params=[256, 240, 192])
def pair_bn(request, monkeypatch):
    monkeypatch.setenv("DG_PAIR_BN", str(request.param))
    return request.param


@pytest.mark.parametrize("M,N,K,with_c", [
    (256, 256, 128, False),
    (384, 512, 640, True),       # odd number of 128-row blocks
    (300, 400, 1152, True),      # ragged M and N, K-groups not a multiple of 4
    (1024, 768, 2048, False),    # several pair tiles per CTA pair
    (512, 496, 640, True),       # N = 2 x 240 + 16: the last tile's narrow chunk lies past N
])
def test_fp4_pair_dense(lib, few_sms, pair_bn, M, N, K, with_c):
    p = W.make_dense_fp4(M, N, K, seed=3000 + M + N + K, with_c=with_c)
    d = run_dense(lib, p)
    ref = O.fp8_fp4_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
    assert_parity(bf16_f64(d), ref, f"fp4 pair dense {M}x{N}x{K}")


def test_fp4_pair_one_hot_exact(lib, few_sms, pair_bn):
    M, N, K = 512, 512, 640
    rng = np.random.default_rng(pair_bn)
    p = W.make_dense_fp4(M, N, K, seed=17)
    k0 = rng.integers(0, K, size=N)
    b = np.zeros((N, K // 2), np.uint8)
    for n, k in enumerate(k0):
        b[n, k // 2] = 2 << (4 * (k % 2))
    p.b, p.sfb = b, W.pack_sf(rng.integers(120, 135, size=(N, K // 32)).astype(np.uint8))
    d = bf16_f64(run_dense(lib, p))
    assert np.array_equal(d, O.fp8_fp4_gemm_nt(p.a, p.sfa, p.b, p.sfb, None, M, N, K))


@pytest.mark.parametrize("counts,N,K", [([300, 0, 129], 256, 512), ([1, 255, 200, 77], 384, 896)])
def test_fp4_contiguous_single_cta(lib, counts, N, K, monkeypatch):
    monkeypatch.setenv("DG_PAIR", "0")
    p = W.make_contiguous(G=len(counts), tokens=sum(counts), N=N, K=K, seed=81 + N, counts=counts,
                          b_format="e2m1")
    d = run_contiguous(lib, p)
    ref, valid = O.m_grouped_fp8_fp4_gemm_nt_contiguous(p.a, p.sfa, p.b, p.sfb, p.m_indices, p.M_total, p.N, p.K,
                                                        p.G)
    assert (bf16_bits(d)[~valid] == SENTINEL).all()
    assert_parity(bf16_f64(d)[valid], ref[valid], f"fp4 contiguous single-CTA {counts}")


@pytest.mark.parametrize("M,N,K,with_c", [(1024, 2560, 256, False), (1280, 2432, 384, True)])
def test_fp4_dense_single_cta_tile_mode(lib, M, N, K, with_c, monkeypatch):
    # 256- and 128-wide single-CTA tiles (the pair kernel takes these shapes by default)
    monkeypatch.setenv("DG_PAIR", "0")
    p = W.make_dense_fp4(M, N, K, seed=4000 + M + N + K, with_c=with_c)
    d = run_dense(lib, p)
    ref = O.fp8_fp4_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
    assert_parity(bf16_f64(d), ref, f"fp4 single-CTA tile mode {M}x{N}x{K}")
