"""The CTA-pair kernel (two SMs share one 256 x BN tcgen05 MMA) against the oracle, for
each tile width: BN = 256 (one accumulator), BN = 240 (two accumulators, dense form only;
tiles start inside 128-column scale blocks and end with a 48-column chunk) and BN = 192
(two accumulators; every other tile starts in the middle of a scale block).

Dense problems reach it in tile mode (at least as many 128 x 128 tiles as SMs used);
the SM cap is lowered so that small problems qualify. Contiguous problems use it when
DG_PAIR=1 (their default is the single-CTA kernel). DG_PAIR_BN selects the width."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import SENTINEL, assert_parity, bf16_bits, bf16_f64, dev, run_contiguous, run_dense, sentinel_like

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_gemm_nt_gb300 as L
    L.load_library()
    return L


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
    (384, 512, 640, True),       # odd number of 128-row blocks: the last pair's second half is empty
    (300, 400, 1152, True),      # ragged M and N, K-groups not a multiple of 4
    (1024, 768, 2048, False),    # several pair tiles per CTA pair
    (512, 496, 640, True),       # N = 2 x 240 + 16: the last tile's narrow chunk lies past N
])
def test_pair_dense(lib, few_sms, pair_bn, M, N, K, with_c):
    p = W.make_dense(M, N, K, seed=900 + M + N + K, with_c=with_c)
    d = run_dense(lib, p)
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
    assert_parity(bf16_f64(d), ref, f"pair dense {M}x{N}x{K}")
    assert lib.dg_get_device_status() == 0


def test_pair_distinct_block_scales_exact(lib, few_sms, pair_bn):
    # B blocks carry different power-of-two scales, A rows of the two CTA halves too: a
    # scale placed in the wrong TMEM columns or lanes (or, for 192-wide tiles, taken from
    # the wrong block where a tile starts inside one) changes results by a power of two,
    # so the shifted run must equal the base run times the shift exactly.
    p = W.make_dense(256, 512, 512, seed=4)
    base = bf16_f64(run_dense(lib, p))
    ea = O.unpack_sf(p.sfa, 256, 4).copy()
    eb = O.unpack_sf(p.sfb, 4, 4).copy()
    ea[130:140] += 1
    eb[1] -= 2
    eb[2] += 1
    eb[3, 2] -= 1                                 # one K-group of the last block only
    q = W.Dense(p.a, W.pack_sf(ea), p.b, W.pack_sf(eb), None, 256, 512, 512)
    got = bf16_f64(run_dense(lib, q))
    expect = base.copy()
    expect[130:140] *= 2.0
    expect[:, 128:256] *= 0.25
    expect[:, 256:384] *= 2.0
    ref = O.fp8_gemm_nt(q.a, q.sfa, q.b, q.sfb, None, 256, 512, 512)
    assert np.array_equal(got[:, :384], expect[:, :384])
    assert_parity(got, ref, "shifted scales")


@pytest.mark.parametrize("counts,N,K", [
    ([300, 100, 300], 512, 512),        # 3, 1 and 3 blocks per expert
    ([128, 0, 129, 255], 256, 384),
    ([1, 1, 1, 1, 1], 272, 256),
])
def test_pair_contiguous(lib, pair_bn, counts, N, K, monkeypatch):
    if pair_bn == 240:
        pytest.skip("240-wide pair tiles are used by the dense form only")
    monkeypatch.setenv("DG_PAIR", "1")
    p = W.make_contiguous(G=len(counts), tokens=sum(counts), N=N, K=K, seed=950 + N + K, counts=counts)
    d = run_contiguous(lib, p)
    ref, valid = O.m_grouped_fp8_gemm_nt_contiguous(p.a, p.sfa, p.b, p.sfb, p.m_indices, p.M_total, p.N, p.K, p.G)
    assert (bf16_bits(d)[~valid] == SENTINEL).all()
    assert_parity(bf16_f64(d)[valid], ref[valid], f"pair contiguous {counts}")
    assert lib.dg_get_device_status() == 0


def test_pair_timeout_path(lib, few_sms, pair_bn):
    p = W.make_dense(512, 512, 512, seed=5)
    lib.dg_get_device_status()
    lib.dg_set_debug(1, 20_000_000)
    try:
        run_dense(lib, p)
        assert lib.dg_get_device_status() == 5
    finally:
        lib.dg_set_debug(0, 0)
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, None, p.M, p.N, p.K)
    assert_parity(bf16_f64(run_dense(lib, p)), ref, "after pair timeout")
    assert lib.dg_get_device_status() == 0


def test_pair_contiguous_bad_index_reported(lib, monkeypatch):
    monkeypatch.setenv("DG_PAIR", "1")
    p = W.make_contiguous(G=2, tokens=200, N=256, K=256, seed=2, counts=[100, 100])
    p.m_indices[128:128 + 100] = 5          # out-of-range expert for the second segment
    d = run_contiguous(lib, p)
    assert lib.dg_get_device_status() == 6
    assert (bf16_bits(d)[128:] == SENTINEL).all(), "rows of an invalid expert were written"


def test_pair_contiguous_repeated_launches(lib, monkeypatch):
    # the pair rows are listed by the scale-preparation launch before every GEMM; many
    # back-to-back launches (programmatic dependent launch chains prep -> GEMM -> prep ...)
    # must all complete without a timeout and leave the same result
    monkeypatch.setenv("DG_PAIR", "1")
    p = W.make_contiguous(G=8, tokens=3000, N=512, K=1024, seed=77)
    a, sfa, b, sfb, idx = dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb), dev(p.m_indices)
    d = sentinel_like((p.M_total, p.N))
    lib.dg_get_device_status()
    for _ in range(300):
        lib.dg_m_grouped_fp8_gemm_nt_contiguous(a, sfa, b, sfb, d, idx)
    torch.cuda.synchronize()
    assert lib.dg_get_device_status() == 0
    ref, valid = O.m_grouped_fp8_gemm_nt_contiguous(p.a, p.sfa, p.b, p.sfb, p.m_indices, p.M_total, p.N, p.K, p.G)
    assert_parity(bf16_f64(d)[valid], ref[valid], "after 300 launches")
