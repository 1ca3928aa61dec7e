"""Split-K over CTA pairs (dense problems with too few tiles to fill the GPU): each pair of
a cluster computes one 128 x BN tile, each CTA half of the K-groups, and the two FP32
partials are summed in rank order through distributed shared memory.

Checked against the oracle for the widths 64 / 96 / 128, ragged M and N, K-group counts
that split unevenly, with and without C; bit-exact determinism; agreement with the
stream-K path; and the bounded-wait failure path (both CTAs of every pair must still meet
at the cluster barriers, so the kernel ends and the context stays usable)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import SENTINEL, assert_parity, bf16_bits, bf16_f64, run_dense

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
    lib.dg_set_num_sms(0)


SPLIT_SHAPES = [
    # M, N, K, with_c, forced width (None: the library's choice)
    (128, 7168, 4096, True, None),     # the decode geometry: 75 tiles of 96 columns
    (64, 7168, 2048, False, None),
    (100, 6000, 1152, True, None),     # ragged M and N; 9 K-groups split 4 + 5
    (128, 4864, 1024, True, 64),       # 76 tiles of 64 columns
    (77, 9728, 768, False, 128),       # 76 tiles of 128 columns, ragged M
    (128, 7168, 512, True, 96),        # 4 K-groups: two per CTA
]


@pytest.mark.parametrize("M,N,K,with_c,bn", SPLIT_SHAPES)
def test_split_parity(lib, monkeypatch, M, N, K, with_c, bn):
    if bn is not None:
        monkeypatch.setenv("DG_SPLIT_BN", str(bn))
    p = W.make_dense(M, N, K, seed=700 + M + N + K, with_c=with_c)
    d = run_dense(lib, p)
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
    assert_parity(bf16_f64(d), ref, f"split {M}x{N}x{K} bn={bn}")
    assert lib.dg_get_device_status() == 0


def test_split_no_write_outside_d(lib):
    # D is written only inside [M, N]: a larger sentinel-filled buffer keeps its margin
    M, N, K = 100, 6000, 1152
    p = W.make_dense(M, N, K, seed=5, with_c=True)
    big = torch.full((M + 3, N), SENTINEL, dtype=torch.int16).view(torch.bfloat16).cuda()
    d = big[:M]
    lib.dg_fp8_gemm_nt(*(torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (p.a, p.sfa, p.b, p.sfb)),
                       torch.from_numpy(p.c.view(np.int16)).view(torch.bfloat16).cuda(), d)
    torch.cuda.synchronize()
    assert (bf16_bits(big[M:]) == SENTINEL).all()
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
    assert_parity(bf16_f64(d), ref, "split with margin")


def test_split_is_deterministic(lib):
    p = W.make_dense(128, 7168, 2048, seed=11, with_c=True)
    first = bf16_bits(run_dense(lib, p))
    for _ in range(3):
        assert np.array_equal(bf16_bits(run_dense(lib, p)), first)


def test_split_agrees_with_stream_k(lib, monkeypatch):
    p = W.make_dense(128, 7168, 2048, seed=12, with_c=True)
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, p.M, p.N, p.K)
    split = bf16_f64(run_dense(lib, p))
    monkeypatch.setenv("DG_SPLIT", "0")
    stream_k = bf16_f64(run_dense(lib, p))
    assert_parity(split, ref, "split")
    assert_parity(stream_k, ref, "stream-K")
    # two correct summation orders: equal up to a last-bit difference in a few places
    assert np.mean(split != stream_k) < 0.05


def test_split_pow2_shift_bit_exact(lib):
    # scaling one A row's scales by 4 and one B block's by 1/2 scales exactly those outputs
    p = W.make_dense(128, 7168, 1024, seed=13)
    base = bf16_f64(run_dense(lib, p))
    KG = p.K // 128
    ea = O.unpack_sf(p.sfa, p.M, KG).copy()
    eb = O.unpack_sf(p.sfb, p.N // 128, KG).copy()
    ea[5] += 2
    eb[7] -= 1                                   # columns 896..1023
    q = W.Dense(p.a, W.pack_sf(ea), p.b, W.pack_sf(eb), None, p.M, p.N, p.K)
    got = bf16_f64(run_dense(lib, q))
    expect = base.copy()
    expect[5] *= 4.0
    expect[:, 896:1024] *= 0.5
    assert np.array_equal(got, expect)


def test_split_timeout_is_reported_and_context_survives(lib):
    p = W.make_dense(128, 7168, 1024, seed=3)
    lib.dg_set_debug(1, 20_000_000)          # producer issues nothing; waits give up after 20 ms
    try:
        run_dense(lib, p)
        assert lib.dg_get_device_status() == 5   # DG_ERR_TIMEOUT
    finally:
        lib.dg_set_debug(0, 0)
    d = run_dense(lib, p)
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, None, p.M, p.N, p.K)
    assert_parity(bf16_f64(d), ref, "after split timeout")
    assert lib.dg_get_device_status() == 0
