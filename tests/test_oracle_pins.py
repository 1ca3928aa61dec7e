"""Pins for the FP64 oracle: checks against things other than the oracle itself.

Each pin is a function of the oracle module so that the same pins can be run against
deliberately broken copies (planted on the CPU, below): every planted mistake must
fail at least one pin. Sources of truth used here:
  * the OCP E4M3FN and UE8M0 code tables (fixed values) and torch's own decoders;
  * exact rational arithmetic (fractions.Fraction) over the definition, on tiny inputs;
  * closed forms: identity and one-hot operands, the C-only case;
  * exact invariances: power-of-two scale shifts act on exactly one row / one block;
  * the grouped forms equal the dense form run per expert (README "Grouped GEMMs").
"""
from __future__ import annotations

import contextlib
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W


# --------------------------------------------------------------------------------------
# helpers that do not use the oracle's arithmetic
# --------------------------------------------------------------------------------------

def torch_e4m3(codes) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def words_from_codes(codes: np.ndarray) -> np.ndarray:
    """Codes [MN, KG] -> packed words, written with explicit integer arithmetic per word."""
    MN, KG = codes.shape
    KP = -(-KG // 4)
    out = np.zeros((KP, 4 * (-(-MN // 4))), np.int64)
    for q in range(KP):
        for i in range(MN):
            w = 0
            for j in range(4):
                g = 4 * q + j
                if g < KG:
                    w += int(codes[i, g]) * (256 ** j)
            out[q, i] = w
    return out.astype(np.uint32).view(np.int32)


def random_codes(rng, shape, nan_free=True):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    if nan_free:
        c[(c & 0x7F) == 0x7F] = 0x3F
    return c


def brute_force(a, ea, b, eb_blocks, c_bits=None):
    """Exact rational D = C + sum_k sA*sB*A*B, with torch decoding the bytes."""
    M, K = a.shape
    N = b.shape[0]
    A = [[Fraction(float(v)) for v in row] for row in torch_e4m3(a)]
    B = [[Fraction(float(v)) for v in row] for row in torch_e4m3(b)]
    two = Fraction(2)
    D = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                g = k // 128
                acc += A[m][k] * B[n][k] * two ** (int(ea[m, g]) - 127) * two ** (int(eb_blocks[n // 128, g]) - 127)
            if c_bits is not None:
                cv = torch.tensor([int(c_bits[m, n])], dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
                acc += Fraction(float(cv.to(torch.float64).item()))
            D[m, n] = float(acc)
    return D


def dense(O_, a, ea, b, eb, c=None):
    M, K = a.shape
    N = b.shape[0]
    return O_.fp8_gemm_nt(a, words_from_codes(ea), b, words_from_codes(eb), c, M, N, K)


# --------------------------------------------------------------------------------------
# pins (each takes the oracle module under test)
# --------------------------------------------------------------------------------------

def pin_e4m3_table(O_):
    known = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x3C: 1.5, 0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0, 0x80: -0.0, 0xB8: -1.0, 0x81: -(2.0 ** -9)}
    for code, v in known.items():
        assert O_.decode_e4m3(np.array([code], np.uint8))[0] == v, hex(code)
    assert np.isnan(O_.decode_e4m3(np.array([0x7F, 0xFF], np.uint8))).all()
    codes = np.arange(256, dtype=np.uint8)
    ours, ref = O_.decode_e4m3(codes), torch_e4m3(codes)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))


def pin_ue8m0_table(O_):
    codes = np.array([0, 1, 126, 127, 128, 200, 254], np.uint8)
    expect = [2.0 ** -127, 2.0 ** -126, 0.5, 1.0, 2.0, 2.0 ** 73, 2.0 ** 127]
    assert list(O_.decode_ue8m0(codes)) == expect
    assert np.isnan(O_.decode_ue8m0(np.array([255], np.uint8))[0])
    if hasattr(torch, "float8_e8m0fnu"):
        all_codes = np.arange(255, dtype=np.uint8)
        ref = torch.from_numpy(all_codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        assert np.array_equal(O_.decode_ue8m0(all_codes), ref)


def pin_bf16(O_):
    x = np.array([0.0, 1.0, -2.5, 3.140625, 1e-3, -7e4, 2.0 ** -130], np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O_.decode_bf16(bits), ref)


def pin_unpack(O_):
    # word for row i of K-quad q holds groups 4q..4q+3 in bytes 0..3 (LSB first)
    words = np.array([[0x04030201, 0x08070605, 0, 0], [0x0C0B0A09, 0x100F0E0D, 0, 0]], np.uint32).view(np.int32)
    codes = O_.unpack_sf(words, 2, 7)
    assert codes.tolist() == [[1, 2, 3, 4, 9, 10, 11], [5, 6, 7, 8, 13, 14, 15]]


def pin_brute_force(O_):
    rng = np.random.default_rng(7)
    for (M, N, K, with_c) in [(1, 1, 128, False), (2, 3, 256, True), (3, 130, 256, True), (4, 2, 384, False)]:
        a = random_codes(rng, (M, K))
        b = random_codes(rng, (N, K))
        ea = rng.integers(120, 135, size=(M, K // 128)).astype(np.uint8)
        eb = rng.integers(120, 135, size=(-(-N // 128), K // 128)).astype(np.uint8)
        c = rng.integers(0, 2 ** 16, size=(M, N)).astype(np.uint16) if with_c else None
        if c is not None:
            c[(c & 0x7F80) == 0x7F80] = 0x3F80     # keep C finite
        got = dense(O_, a, ea, b, eb, c)
        ref = brute_force(a, ea, b, eb, c)
        np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-300)


def pin_identity(O_):
    # A = [I | 0] with unit scales gives D[i, n] = B[n, i] * sB(block of n, group 0)
    rng = np.random.default_rng(11)
    M, N, K = 4, 256, 256
    a = np.zeros((M, K), np.uint8)
    a[np.arange(M), np.arange(M)] = 0x38            # 1.0
    b = random_codes(rng, (N, K))
    ea = np.full((M, 2), 127, np.uint8)
    eb = np.array([[127, 127], [129, 120]], np.uint8)  # block 1 scaled by 4 in group 0
    got = dense(O_, a, ea, b, eb)
    Bv = torch_e4m3(b)
    expect = Bv[:, :M].T * np.where(np.arange(N) >= 128, 4.0, 1.0)[None, :]
    assert np.array_equal(got, expect)


def pin_one_hot(O_):
    rng = np.random.default_rng(12)
    M, N, K = 3, 200, 384
    b = random_codes(rng, (N, K))
    for (m, k) in [(0, 5), (1, 200), (2, 383)]:
        a = np.zeros((M, K), np.uint8)
        a[m, k] = 0x40                              # 2.0
        ea = np.full((M, 3), 127, np.uint8)
        ea[m, k // 128] = 125                       # x 1/4
        eb = np.full((2, 3), 127, np.uint8)
        eb[1, k // 128] = 130                       # block 1 x 8
        got = dense(O_, a, ea, b, eb)
        expect = np.zeros((M, N))
        expect[m] = 2.0 * 0.25 * torch_e4m3(b[:, k]) * np.where(np.arange(N) >= 128, 8.0, 1.0)
        assert np.array_equal(got, expect)


def pin_pow2_invariance(O_):
    rng = np.random.default_rng(13)
    M, N, K = 5, 300, 512
    a, b = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    ea = rng.integers(124, 131, size=(M, 4)).astype(np.uint8)
    eb = rng.integers(124, 131, size=(3, 4)).astype(np.uint8)
    base = dense(O_, a, ea, b, eb)
    # shift every group of row 2 by +3: row 2 x 8, all other rows unchanged, bit-exactly
    ea2 = ea.copy(); ea2[2] += 3
    got = dense(O_, a, ea2, b, eb)
    expect = base.copy(); expect[2] *= 8.0
    assert np.array_equal(got, expect)
    # shift every group of B block 1 by -2: columns 128..255 x 1/4, others unchanged
    eb2 = eb.copy(); eb2[1] -= 2
    got = dense(O_, a, ea, b, eb2)
    expect = base.copy(); expect[:, 128:256] *= 0.25
    assert np.array_equal(got, expect)
    # a single group's scale only touches that group's contribution
    z = a.copy(); z[:, 128:] = 0
    only_g0 = dense(O_, z, ea, b, eb)
    ea3 = ea.copy(); ea3[:, 1:] = 127 - 20
    assert np.array_equal(dense(O_, z, ea3, b, eb), only_g0)


def pin_c_only(O_):
    rng = np.random.default_rng(14)
    M, N, K = 3, 130, 256
    c = rng.integers(0, 2 ** 16, size=(M, N)).astype(np.uint16)
    c[(c & 0x7F80) == 0x7F80] = 0x4000
    got = dense(O_, np.zeros((M, K), np.uint8), np.full((M, 2), 127, np.uint8),
                random_codes(rng, (N, K)), np.full((2, 2), 127, np.uint8), c)
    ref = torch.from_numpy(c.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(got, ref)


def pin_dequantised_route(O_):
    # Same value by another route: dequantise whole operands, one FP64 matmul over all K.
    p = W.make_dense(17, 260, 640, seed=5, with_c=True)
    got = O_.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, p.M, p.N, p.K)
    KG = p.K // 128
    ea = np.stack([(p.sfa.view(np.uint32)[g // 4, :p.M] >> (8 * (g % 4))) & 0xFF for g in range(KG)], 1)
    NB = -(-p.N // 128)
    eb = np.stack([(p.sfb.view(np.uint32)[g // 4, :NB] >> (8 * (g % 4))) & 0xFF for g in range(KG)], 1)
    Af = torch_e4m3(p.a) * np.exp2(np.repeat(ea.astype(np.float64) - 127, 128, axis=1))
    Bf = torch_e4m3(p.b) * np.exp2(np.repeat(np.repeat(eb.astype(np.float64) - 127, 128, axis=0)[:p.N], 128, axis=1))
    Cf = torch.from_numpy(p.c.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_allclose(got, Cf + Af @ Bf.T, rtol=1e-12, atol=1e-12)


def pin_contiguous_equals_dense(O_):
    p = W.make_contiguous(G=3, tokens=300, N=144, K=256, seed=3, counts=[130, 0, 170])
    D, valid = O_.m_grouped_fp8_gemm_nt_contiguous(p.a, p.sfa, p.b, p.sfb, p.m_indices, p.M_total, p.N, p.K, p.G)
    assert p.M_total == 256 + 256
    assert np.array_equal(valid, p.m_indices >= 0)
    assert np.isnan(D[~valid]).all() and not np.isnan(D[valid]).any()
    KG = p.K // 128
    ea = np.stack([(p.sfa.view(np.uint32)[g // 4, :p.M_total] >> (8 * (g % 4))) & 0xFF for g in range(KG)], 1)
    for g in range(p.G):
        r = np.nonzero(p.m_indices == g)[0]
        if len(r) == 0:
            continue
        NB = -(-p.N // 128)
        eb = np.stack([(p.sfb[g].view(np.uint32)[q // 4, :NB] >> (8 * (q % 4))) & 0xFF for q in range(KG)], 1)
        ref = dense(O_, p.a[r], ea[r].astype(np.uint8), p.b[g], eb.astype(np.uint8))
        assert np.array_equal(D[r], ref)
        # and against exact rationals on a few rows
        bf = brute_force(p.a[r[:2]], ea[r[:2]], p.b[g], eb)
        np.testing.assert_allclose(D[r[:2]], bf, rtol=1e-14)


def pin_masked_equals_dense(O_):
    p = W.make_masked(G=4, max_m=40, N=136, K=256, seed=4, masked_m=[0, 40, 17, 1])
    D, valid = O_.m_grouped_fp8_gemm_nt_masked(p.a, p.sfa, p.b, p.sfb, p.masked_m, p.G, p.max_m, p.N, p.K)
    assert valid.sum(1).tolist() == [0, 40, 17, 1]
    assert np.isnan(D[~valid]).all() and not np.isnan(D[valid]).any()
    KG = p.K // 128
    NB = -(-p.N // 128)
    for g in range(p.G):
        m = int(p.masked_m[g])
        if m == 0:
            continue
        ea = np.stack([(p.sfa[g].view(np.uint32)[q // 4, :m] >> (8 * (q % 4))) & 0xFF for q in range(KG)], 1)
        eb = np.stack([(p.sfb[g].view(np.uint32)[q // 4, :NB] >> (8 * (q % 4))) & 0xFF for q in range(KG)], 1)
        bf = brute_force(p.a[g, :min(m, 2)], ea[:2], p.b[g], eb)
        np.testing.assert_allclose(D[g, :min(m, 2)], bf, rtol=1e-14)
        ref = dense(O_, p.a[g, :m], ea.astype(np.uint8), p.b[g], eb.astype(np.uint8))
        assert np.array_equal(D[g, :m], ref)


def pin_wgrad_brute_force(O_):
    # FP32 addend values that BF16 cannot hold: an addend rounded to BF16, dropped or
    # subtracted fails this exact rational check
    rng = np.random.default_rng(21)
    M, N, K = 3, 130, 256
    a, b = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    ea = rng.integers(122, 133, size=(M, 2)).astype(np.uint8)
    eb = rng.integers(122, 133, size=(2, 2)).astype(np.uint8)
    c = (rng.standard_normal((M, N)) * 3).astype(np.float32)
    c[0, 0] = np.float32(1.0) + np.float32(2.0 ** -20)
    got = O_.wgrad_gemm_fp8_fp8_fp32_nt(a, words_from_codes(ea), b, words_from_codes(eb), c, M, N, K)
    exact = brute_force(a, ea, b, eb)
    for m in range(M):
        for n in range(N):
            want = float(Fraction(float(exact[m, n])) + Fraction(float(c[m, n])))
            assert got[m, n] == pytest.approx(want, rel=1e-15, abs=1e-300), (m, n)
    # no addend: the dense result exactly
    assert np.array_equal(O_.wgrad_gemm_fp8_fp8_fp32_nt(a, words_from_codes(ea), b, words_from_codes(eb),
                                                        None, M, N, K), dense(O_, a, ea, b, eb))


def pin_wgrad_c_only(O_):
    rng = np.random.default_rng(22)
    M, N, K = 4, 96, 128
    c = rng.standard_normal((M, N)).astype(np.float32)
    got = O_.wgrad_gemm_fp8_fp8_fp32_nt(np.zeros((M, K), np.uint8), words_from_codes(np.full((M, 1), 127, np.uint8)),
                                        random_codes(rng, (N, K)), words_from_codes(np.full((1, 1), 127, np.uint8)),
                                        c, M, N, K)
    assert np.array_equal(got, c.astype(np.float64))


def pin_k_grouped_equals_per_expert(O_):
    # each expert's output is the dense FP32-output GEMM of its own K-slice, with its own
    # scales packed separately; an expert with no tokens returns its C; and against exact
    # rationals on a few entries
    rng = np.random.default_rng(23)
    M, N, ks = 5, 200, [256, 0, 384, 128]
    K_total = sum(ks)
    a, b = random_codes(rng, (M, K_total)), random_codes(rng, (N, K_total))
    ea = rng.integers(123, 132, size=(M, K_total // 128)).astype(np.uint8)
    eb = rng.integers(123, 132, size=(2, K_total // 128)).astype(np.uint8)
    c = rng.standard_normal((len(ks), M, N)).astype(np.float32)
    sfa, sfb = W.pack_sf_k_grouped(ea, ks), W.pack_sf_k_grouped(eb, ks)
    assert sfa.shape[0] == 1 + 0 + 1 + 1
    D = O_.k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(a, sfa, b, sfb, c, ks, M, N)
    off = 0
    for g, k in enumerate(ks):
        kg = k // 128
        if k == 0:
            assert np.array_equal(D[g], c[g].astype(np.float64))
            continue
        sl = slice(off, off + k)
        gs = slice(off // 128, off // 128 + kg)
        ref = O_.wgrad_gemm_fp8_fp8_fp32_nt(a[:, sl], words_from_codes(ea[:, gs]), b[:, sl],
                                            words_from_codes(eb[:, gs]), c[g], M, N, k)
        assert np.array_equal(D[g], ref)
        exact = brute_force(a[:2, sl], ea[:2, gs], b[:, sl], eb[:, gs])
        np.testing.assert_allclose(D[g, :2], exact + c[g, :2].astype(np.float64), rtol=1e-14)
        off += k


def pin_layouts(O_):
    # each storage layout against exact rationals over the logical M x K and N x K matrices
    rng = np.random.default_rng(24)
    M, N, K = 3, 140, 256
    a, b = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    ea = rng.integers(123, 132, size=(M, 2)).astype(np.uint8)
    eb = rng.integers(123, 132, size=(2, 2)).astype(np.uint8)
    exact = brute_force(a, ea, b, eb)
    sfa, sfb = words_from_codes(ea), words_from_codes(eb)
    got = {
        "nn": O_.fp8_gemm_nn(a, sfa, np.ascontiguousarray(b.T), sfb, None, M, N, K),
        "tn": O_.fp8_gemm_tn(np.ascontiguousarray(a.T), sfa, np.ascontiguousarray(b.T), sfb, None, M, N, K),
        "tt": O_.fp8_gemm_tt(np.ascontiguousarray(a.T), sfa, b, sfb, None, M, N, K),
    }
    for name, d in got.items():
        np.testing.assert_allclose(d, exact, rtol=1e-14, err_msg=name)


def pin_grouped_layouts(O_):
    # the N-major contiguous form and the TN K-grouped form against exact rationals over the
    # logical matrices
    rng = np.random.default_rng(25)
    K, N = 256, 136
    m_idx = np.array([0] * 2 + [-1] * 126 + [1] * 3 + [-1] * 125, np.int32)
    M_total = len(m_idx)
    a = random_codes(rng, (M_total, K))
    b = random_codes(rng, (2, N, K))
    ea = rng.integers(123, 132, size=(M_total, 2)).astype(np.uint8)
    eb = rng.integers(123, 132, size=(2, 2, 2)).astype(np.uint8)
    sfb = np.stack([words_from_codes(eb[g]) for g in range(2)])
    D, valid = O_.m_grouped_fp8_gemm_nn_contiguous(a, words_from_codes(ea), np.ascontiguousarray(b.transpose(0, 2, 1)),
                                                   sfb, m_idx, M_total, N, K, 2)
    assert np.array_equal(valid, m_idx >= 0)
    for r in np.nonzero(m_idx >= 0)[0][:4]:
        g = m_idx[r]
        np.testing.assert_allclose(D[r], brute_force(a[r:r + 1], ea[r:r + 1], b[g], eb[g])[0], rtol=1e-14)
    M, Nk, ks = 4, 160, [128, 256]
    a2, b2 = random_codes(rng, (M, sum(ks))), random_codes(rng, (Nk, sum(ks)))
    ea2 = rng.integers(123, 132, size=(M, 3)).astype(np.uint8)
    eb2 = rng.integers(123, 132, size=(2, 3)).astype(np.uint8)
    D2 = O_.k_grouped_fp8_gemm_tn_contiguous(np.ascontiguousarray(a2.T), W.pack_sf_k_grouped(ea2, ks),
                                             np.ascontiguousarray(b2.T), W.pack_sf_k_grouped(eb2, ks), None, ks, M, Nk)
    np.testing.assert_allclose(D2[1], brute_force(a2[:, 128:], ea2[:, 1:], b2[:, 128:], eb2[:, 1:]), rtol=1e-14)


# --------------------------------------------------------------------------------------
# FP8 x FP4 pins
# --------------------------------------------------------------------------------------

# E2M1 magnitudes of codes 0..7 as tabulated in the OCP Microscaling Formats (MX) v1.0
# specification (FP4 E2M1: 0, 0.5 subnormal, then 1, 1.5, 2, 3, 4, 6); codes 8..15 negate.
E2M1_OCP = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4),
            Fraction(6)]


def e2m1_value(code: int) -> Fraction:
    return -E2M1_OCP[code & 7] if code & 8 else E2M1_OCP[code & 7]


def fp4_code(packed: np.ndarray, n: int, k: int) -> int:
    """Element k of row n of a packed FP4 matrix: the low nibble holds the even element."""
    return (int(packed[n, k // 2]) >> (4 * (k % 2))) & 0xF


def brute_force_fp4(a, ea, b_packed, eb, c_bits=None):
    """Exact rational D = C + sum_k sA[m, k//128] * sB[n, k//32] * A[m, k] * B[n, k]."""
    M, K = a.shape
    N = b_packed.shape[0]
    A = [[Fraction(float(v)) for v in row] for row in torch_e4m3(a)]
    two = Fraction(2)
    D = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += (A[m][k] * e2m1_value(fp4_code(b_packed, n, k)) * two ** (int(ea[m, k // 128]) - 127)
                        * two ** (int(eb[n, k // 32]) - 127))
            if c_bits is not None:
                cv = torch.tensor([int(c_bits[m, n])], dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
                acc += Fraction(float(cv.to(torch.float64).item()))
            D[m, n] = float(acc)
    return D


def pin_e2m1_table(O_):
    got = O_.decode_e2m1(np.arange(16))
    expect = np.array([float(e2m1_value(c)) for c in range(16)])
    assert np.array_equal(got, expect)
    assert np.signbit(got[8]) and not np.signbit(got[0])


def pin_fp4_brute_force(O_):
    rng = np.random.default_rng(31)
    M, N, K = 3, 5, 256
    a = random_codes(rng, (M, K))
    b = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    ea = rng.integers(120, 135, size=(M, K // 128)).astype(np.uint8)
    eb = rng.integers(120, 135, size=(N, K // 32)).astype(np.uint8)
    c = W.to_bf16_bits(rng.standard_normal((M, N)).astype(np.float32))
    got = O_.fp8_fp4_gemm_nt(a, words_from_codes(ea), b, words_from_codes(eb), c, M, N, K)
    np.testing.assert_allclose(got, brute_force_fp4(a, ea, b, eb, c), rtol=1e-14, atol=0)


def pin_fp4_one_hot(O_):
    # B row n holds a single 1.0 (code 2) at column k0[n]: D[m, n] = sA * sB * A[m, k0[n]]
    rng = np.random.default_rng(32)
    M, N, K = 4, 8, 512
    k0 = np.array([0, 1, 33, 94, 127, 128, 301, 511])
    b = np.zeros((N, K // 2), np.uint8)
    for n, k in enumerate(k0):
        b[n, k // 2] = 2 << (4 * (k % 2))
    a = random_codes(rng, (M, K))
    ea = rng.integers(120, 135, size=(M, K // 128)).astype(np.uint8)
    eb = rng.integers(120, 135, size=(N, K // 32)).astype(np.uint8)
    got = O_.fp8_fp4_gemm_nt(a, words_from_codes(ea), b, words_from_codes(eb), None, M, N, K)
    A = torch_e4m3(a)
    for m in range(M):
        for n, k in enumerate(k0):
            want = A[m, k] * 2.0 ** (int(ea[m, k // 128]) - 127) * 2.0 ** (int(eb[n, k // 32]) - 127)
            assert got[m, n] == want, (m, n, got[m, n], want)


def pin_fp4_matches_fp8_route(O_):
    # Every E2M1 value is an E4M3 value: with B's scales constant over each 128 x 128 block the
    # FP8 x FP4 GEMM is the FP8 GEMM of the same numbers (B re-encoded by value lookup in
    # torch's E4M3 decoding).
    rng = np.random.default_rng(33)
    M, N, K = 6, 136, 384
    a = random_codes(rng, (M, K))
    b = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    e4m3_of = {}
    for code in range(256):
        v = torch_e4m3(np.array([code], np.uint8))[0]
        if not np.isnan(v):
            e4m3_of.setdefault(float(v), code)
    e4m3_of[0.0] = 0
    b8 = np.array([[e4m3_of[float(e2m1_value(fp4_code(b, n, k)))] for k in range(K)] for n in range(N)], np.uint8)
    ea = rng.integers(122, 133, size=(M, K // 128)).astype(np.uint8)
    eb_blocks = rng.integers(122, 133, size=(2, K // 128)).astype(np.uint8)
    eb_rows = np.repeat(np.repeat(eb_blocks, 128, axis=0)[:N], 4, axis=1)     # [N, K/32]
    c = W.to_bf16_bits(rng.standard_normal((M, N)).astype(np.float32))
    got = O_.fp8_fp4_gemm_nt(a, words_from_codes(ea), b, words_from_codes(eb_rows), c, M, N, K)
    want = O_.fp8_gemm_nt(a, words_from_codes(ea), b8, words_from_codes(eb_blocks), c, M, N, K)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def pin_fp4_grouped_equals_dense(O_):
    rng = np.random.default_rng(34)
    G, N, K = 3, 40, 256
    b = rng.integers(0, 256, size=(G, N, K // 2), dtype=np.uint8)
    eb = rng.integers(122, 133, size=(G, N, K // 32)).astype(np.uint8)
    sfb = np.stack([words_from_codes(eb[g]) for g in range(G)])
    m_idx = np.array([2] * 3 + [-1] * 125 + [0] * 2 + [-1] * 126, np.int32)
    R = len(m_idx)
    a = random_codes(rng, (R, K))
    ea = rng.integers(122, 133, size=(R, K // 128)).astype(np.uint8)
    D, valid = O_.m_grouped_fp8_fp4_gemm_nt_contiguous(a, words_from_codes(ea), b, sfb, m_idx, R, N, K, G)
    assert np.array_equal(valid, m_idx >= 0)
    assert np.isnan(D[~valid]).all()
    for r in np.nonzero(m_idx >= 0)[0]:
        g = m_idx[r]
        want = brute_force_fp4(a[r:r + 1], ea[r:r + 1], b[g], eb[g])
        np.testing.assert_allclose(D[r:r + 1], want, rtol=1e-14)
    max_m = 5
    am = random_codes(rng, (G, max_m, K))
    eam = rng.integers(122, 133, size=(G, max_m, K // 128)).astype(np.uint8)
    sfam = np.stack([words_from_codes(eam[g]) for g in range(G)])
    masked = np.array([2, 0, 7], np.int32)          # the last is clamped to max_m
    Dm, vm = O_.m_grouped_fp8_fp4_gemm_nt_masked(am, sfam, b, sfb, masked, G, max_m, N, K)
    assert vm.sum() == 2 + 0 + max_m
    np.testing.assert_allclose(Dm[0, :2], brute_force_fp4(am[0, :2], eam[0, :2], b[0], eb[0]), rtol=1e-14)
    np.testing.assert_allclose(Dm[2], brute_force_fp4(am[2], eam[2], b[2], eb[2]), rtol=1e-14)
    assert np.isnan(Dm[1]).all() and np.isnan(Dm[0, 2:]).all()


def pin_golden(O_):
    # the hand-worked examples under tests/golden/ (each shows its arithmetic in the file)
    from golden_util import all_fixtures, check_oracle, load
    for name in all_fixtures():
        g = load(name)
        if g.form == "pack_sf":
            mn, kg = g.sf.shape
            codes = O_.unpack_sf(g.words.view(np.int32), mn, kg)
            assert np.array_equal(W.pack_sf(codes).view(np.uint32), g.words), name
        else:
            check_oracle(O_, g)


def pin_parity_report(O_):
    """The comparator every GPU parity check goes through, on hand-worked cases: each
    expected outcome follows from the bound |d - ref| <= rel*|ref| + abs_rms*rms(ref) (rms
    over ref) and the strict cosine-style bar, computed here by hand."""
    pr = O_.parity_report
    # ref = [1, 7]: rms = sqrt((1 + 49) / 2) = 5, so element 0's bound is 0.01 + 0.05 = 0.06
    r = pr(np.array([1.0595, 7.0]), np.array([1.0, 7.0]))
    assert r["ok"] and r["n_bad"] == 0 and r["n"] == 2 and r["rms"] == 5.0, r
    r = pr(np.array([1.0605, 7.0]), np.array([1.0, 7.0]))
    assert not r["ok"] and r["n_bad"] == 1, r
    # the relative part uses |ref|: for ref = -1 the bound is still 0.06
    r = pr(np.array([-1.0595, 7.0]), np.array([-1.0, 7.0]))
    assert r["ok"] and r["n_bad"] == 0, r
    # rms is over ref, not d. ref = [100, 0]: rms = 70.7107, element 1's bound 0.707107.
    # d = [101.7, 0.71] fails there (rms(d) would be 71.91, a bound of 0.719, and pass);
    # d = [98.3, 0.7] passes both elements (1.7 <= 1.70711, 0.7 <= 0.70711; rms(d) = 69.51
    # would fail element 1); both cosine-style differences are ~1.7e-4
    r = pr(np.array([101.7, 0.71]), np.array([100.0, 0.0]))
    assert not r["ok"] and r["n_bad"] == 1, r
    r = pr(np.array([98.3, 0.7]), np.array([100.0, 0.0]))
    assert r["ok"] and r["n_bad"] == 0, r
    # rel multiplies |ref|, abs_rms multiplies rms: with rel = 0.02, abs_rms = 0.005 and
    # ref = [1, 7] the bounds are 0.045 and 0.165 (swapped roles would give 0.105, 0.135)
    r = pr(np.array([1.08, 7.0]), np.array([1.0, 7.0]), rel=0.02, abs_rms=0.005)
    assert not r["ok"] and r["n_bad"] == 1, r
    r = pr(np.array([1.0, 7.15]), np.array([1.0, 7.0]), rel=0.02, abs_rms=0.005)
    assert r["ok"] and r["n_bad"] == 0, r
    # an element exactly at its bound passes: rel = abs_rms = 2^-7 gives the exact bounds
    # 6 * 2^-7 and 12 * 2^-7 for ref = [1, 7]
    r = pr(np.array([1.0 + 6 / 128, 7.0 - 12 / 128]), np.array([1.0, 7.0]), rel=2.0 ** -7, abs_rms=2.0 ** -7)
    assert r["n_bad"] == 0 and r["ok"], r
    # cosine-style difference: d = 1 + (e, -e, e, -e) against ref = 1 gives exactly
    # e^2 / (2 + e^2); rel = 0, abs_rms = 1 keeps every element inside its bound (1)
    ones = np.ones(4)
    for e, ok in ((0.0447, True), (0.0448, False)):
        r = pr(ones + e * np.array([1.0, -1.0, 1.0, -1.0]), ones, rel=0.0, abs_rms=1.0)
        assert abs(r["diff"] - e * e / (2 + e * e)) < 1e-15 and r["ok"] == ok and r["n_bad"] == 0, (e, r)
    # the bar is strict: d = (1, 1, 1, 1), ref = (1, 1, 1, -1) give 2*2/8 = 0.5, difference 0.5
    r = pr(np.ones(4), np.array([1.0, 1.0, 1.0, -1.0]), rel=0.0, abs_rms=10.0, cos_max=0.5)
    assert r["diff"] == 0.5 and r["n_bad"] == 0 and not r["ok"], r
    r = pr(np.ones(4), np.array([1.0, 1.0, 1.0, -1.0]), rel=0.0, abs_rms=10.0, cos_max=0.5 + 2.0 ** -20)
    assert r["ok"], r
    # a NaN in d fails its element (and the difference)
    r = pr(np.array([np.nan, 7.0]), np.array([1.0, 7.0]))
    assert not r["ok"] and r["n_bad"] == 1, r
    # nothing to compare: reported ok with n = 0
    r = pr(np.zeros(0), np.zeros(0))
    assert r["ok"] and r["n"] == 0 and r["n_bad"] == 0, r


PINS = [pin_e4m3_table, pin_ue8m0_table, pin_bf16, pin_unpack, pin_brute_force, pin_identity,
        pin_one_hot, pin_pow2_invariance, pin_c_only, pin_dequantised_route,
        pin_contiguous_equals_dense, pin_masked_equals_dense, pin_wgrad_brute_force, pin_wgrad_c_only,
        pin_k_grouped_equals_per_expert, pin_layouts, pin_grouped_layouts, pin_e2m1_table, pin_fp4_brute_force,
        pin_fp4_one_hot, pin_fp4_matches_fp8_route, pin_fp4_grouped_equals_dense, pin_golden,
        pin_parity_report]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(O)


# --------------------------------------------------------------------------------------
# planted mistakes: each must be caught by at least one pin
# --------------------------------------------------------------------------------------

def _mut_table(table_fn):
    @contextlib.contextmanager
    def ctx():
        old = O._E4M3.copy()
        O._E4M3[:] = table_fn(old)
        try:
            yield
        finally:
            O._E4M3[:] = old
    return ctx


def _mut_attr(name, new):
    @contextlib.contextmanager
    def ctx():
        old = getattr(O, name)
        setattr(O, name, new(old))
        try:
            yield
        finally:
            setattr(O, name, old)
    return ctx


def _subnormal_with_implicit_one(t):
    t = t.copy()
    for code in range(256):
        if (code >> 3) & 0xF == 0:
            s = -1.0 if code & 0x80 else 1.0
            t[code] = s * (1 + (code & 7) / 8) * 2.0 ** -6
    return t


def _bias_off_by_one(old):
    return lambda codes: np.ldexp(1.0, np.asarray(codes, np.int64) - 126)


def _byte_order_reversed(old):
    def f(words, mn, kgroups):
        w = np.asarray(words).view(np.uint32)
        out = np.empty((mn, kgroups), np.uint8)
        for g in range(kgroups):
            out[:, g] = (w[g // 4, :mn] >> np.uint32(8 * (3 - g % 4))) & np.uint32(0xFF)
        return out
    return f


def _make_scaled(mode):
    def factory(old):
        def f(a_codes, sa_codes, b_codes, sb_codes, K):
            KG = K // 128
            N = b_codes.shape[0]
            A = O.decode_e4m3(a_codes)
            B = O.decode_e4m3(b_codes)
            if mode == "transposed_b":   # B read as if stored [K, N]
                B = B.reshape(-1)[: N * K].reshape(K, N).T if N != K else B.T
            sA = O.decode_ue8m0(sa_codes)
            blk = (np.arange(N) % 128) if mode == "block_mod" else (np.arange(N) // 128)
            blk = np.minimum(blk, sb_codes.shape[0] - 1)
            sB = O.decode_ue8m0(sb_codes)[blk]
            D = np.zeros((A.shape[0], N))
            groups = range(KG - 1) if mode == "drop_last_group" else range(KG)
            for g in groups:
                ks = slice(g * 128, (g + 1) * 128)
                ga = 0 if mode == "first_scale_only" else g
                D += sA[:, ga:ga + 1] * (A[:, ks] @ B[:, ks].T) * sB[None, :, g]
            return D
        return f
    return factory


def _c_sign(old):
    def f(a, sfa, b, sfb, c, M, N, K, rows=None):
        d = old(a, sfa, b, sfb, None, M, N, K, rows)
        if c is not None:
            r = np.arange(M) if rows is None else np.asarray(rows)
            d = d - O.decode_bf16(np.asarray(c)[r])
        return d
    return f


def _contig_negative_index(old):
    def f(a, sfa, b, sfb, m_indices, M_total, N, K, G, rows=None):
        rows = np.arange(M_total) if rows is None else np.asarray(rows)
        idx = np.asarray(m_indices)[rows]
        D = np.full((len(rows), N), np.nan)
        sa = O.unpack_sf(sfa, M_total, K // 128)
        for r_i, r in enumerate(rows):
            g = idx[r_i]          # -1 silently selects the last expert
            D[r_i] = O._scaled_gemm(a[r:r + 1], sa[r:r + 1], b[g], O.unpack_sf(sfb[g], -(-N // 128), K // 128), K)[0]
        return D, idx >= 0
    return f


def _masked_off_by_one(old):
    def f(a, sfa, b, sfb, masked_m, G, max_m, N, K, groups=None):
        mm = np.minimum(np.asarray(masked_m) + 1, max_m)
        return old(a, sfa, b, sfb, mm, G, max_m, N, K, groups)
    return f


def _wgrad_c_as_bf16(old):
    def f(a, sfa, b, sfb, c, M, N, K, rows=None):
        if c is not None:
            c = torch.from_numpy(np.asarray(c, np.float32)).to(torch.bfloat16).to(torch.float32).numpy()
        return old(a, sfa, b, sfb, c, M, N, K, rows)
    return f


def _wgrad_c_dropped(old):
    def f(a, sfa, b, sfb, c, M, N, K, rows=None):
        return old(a, sfa, b, sfb, None, M, N, K, rows)
    return f


def _k_grouped_global_packing(old):
    # reads the scale words as if packed over the whole K axis (not per expert)
    def f(a, sfa, b, sfb, c, ks, M, N, groups=None, rows=None):
        ks = [int(k) for k in ks]
        K_total = sum(ks)
        KG = K_total // 128
        NB = -(-N // 128)
        ea = O.unpack_sf(np.asarray(sfa), M, min(KG, 4 * np.asarray(sfa).shape[0]))
        eb = O.unpack_sf(np.asarray(sfb), NB, min(KG, 4 * np.asarray(sfb).shape[0]))
        pad = KG - ea.shape[1]
        if pad > 0:
            ea = np.concatenate([ea, np.full((M, pad), 127, ea.dtype)], 1)
            eb = np.concatenate([eb, np.full((NB, pad), 127, eb.dtype)], 1)
        out, off = [], 0
        for g, k in enumerate(ks):
            kg = k // 128
            sl = slice(off * 128, (off + kg) * 128)
            d = O._scaled_gemm(a[:, sl], ea[:, off:off + kg], b[:, sl], eb[:, off:off + kg], k) if kg else np.zeros((M, N))
            out.append((np.asarray(c, np.float32)[g].astype(np.float64) if c is not None else 0) + d)
            off += kg
        return np.stack(out)
    return f


def _tn_forgets_to_transpose_a(old):
    def f(a, sfa, b, sfb, c, M, N, K):
        return O.fp8_gemm_nt(np.asarray(a).reshape(M, K), sfa, np.ascontiguousarray(np.asarray(b).T), sfb, c, M, N, K)
    return f


def _tt_forgets_to_transpose_a(old):
    def f(a, sfa, b, sfb, c, M, N, K):
        return O.fp8_gemm_nt(np.asarray(a).reshape(M, K), sfa, b, sfb, c, M, N, K)
    return f


def _nn_contiguous_reads_b_as_n_major(old):
    def f(a, sfa, b, sfb, m_indices, M_total, N, K, G, rows=None):
        return O.m_grouped_fp8_gemm_nt_contiguous(a, sfa, np.asarray(b).reshape(G, N, K), sfb, m_indices,
                                                  M_total, N, K, G, rows=rows)
    return f


def _tn_k_grouped_reads_b_as_k_major(old):
    def f(a, sfa, b, sfb, c, ks, M, N, groups=None, rows=None):
        K_total = int(np.sum(ks))
        return O.k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(np.ascontiguousarray(np.asarray(a).T), sfa,
                                                      np.asarray(b).reshape(N, K_total), sfb, c, ks, M, N,
                                                      groups=groups, rows=rows)
    return f


def _mut_e2m1(table_fn):
    @contextlib.contextmanager
    def ctx():
        old = O._E2M1.copy()
        O._E2M1[:] = table_fn(old)
        try:
            yield
        finally:
            O._E2M1[:] = old
    return ctx


def _e2m1_subnormal_as_normal(t):
    t = t.copy()
    t[1], t[9] = 1.0, -1.0      # code 1 read with an implicit leading one
    return t


def _fp4_high_nibble_first(old):
    def f(packed, K):
        p = np.asarray(packed, dtype=np.uint8)
        out = np.empty(p.shape[:-1] + (K,), np.uint8)
        out[..., 0::2] = p >> 4
        out[..., 1::2] = p & 0xF
        return out
    return f


def _make_scaled_fp4(mode):
    def factory(old):
        def f(a_codes, sa_codes, b_codes, sb_codes, K):
            A = O.decode_e4m3(a_codes)
            B = O.decode_e2m1(b_codes)
            sA = O.decode_ue8m0(sa_codes)
            sB = O.decode_ue8m0(sb_codes)
            D = np.zeros((A.shape[0], B.shape[0]))
            for j in range(K // 32):
                ks = slice(32 * j, 32 * j + 32)
                jb = 4 * (j // 4) if mode == "b_scale_per_128" else j
                ja = min(j, sA.shape[1] - 1) if mode == "a_scale_per_32" else j // 4
                D += sA[:, ja, None] * (A[:, ks] @ B[:, ks].T) * sB[None, :, jb]
            return D
        return f
    return factory


def _make_parity(mode):
    """Copies of the comparator with one planted mistake each."""
    def factory(old):
        def f(d, ref, rel=1e-2, abs_rms=1e-2, cos_max=1e-3):
            d = np.asarray(d, np.float64)
            ref = np.asarray(ref, np.float64)
            over = d if mode == "rms_over_d" else ref
            rms = float(np.sqrt(np.mean(over * over))) if ref.size else 0.0
            err = np.abs(d - ref)
            if mode == "rel_abs_swapped":
                bound = abs_rms * np.abs(ref) + rel * rms
            elif mode == "signed_ref":
                bound = rel * ref + abs_rms * rms
            else:
                bound = rel * np.abs(ref) + abs_rms * rms
            if mode == "nan_passes":
                bad = err > bound
            elif mode == "strict_bound":
                bad = ~(err < bound)
            else:
                bad = ~(err <= bound)
            denom = float((d * d).sum() + (ref * ref).sum())
            diff = 0.0 if denom == 0.0 else 1.0 - 2.0 * float((d * ref).sum()) / denom
            if mode == "diff_sign_flipped":
                diff = -diff
            ok_cos = diff <= cos_max if mode == "cos_not_strict" else diff < cos_max
            return dict(n=int(ref.size), n_bad=int(bad.sum()), max_err=float(err.max()) if ref.size else 0.0,
                        rms=rms, diff=diff, ok=bool(not bad.any() and ok_cos))
        return f
    return factory


MUTANTS = {
    "subnormal_implicit_one": _mut_table(_subnormal_with_implicit_one),
    "sign_ignored": _mut_table(lambda t: np.abs(t)),
    "ue8m0_bias_126": _mut_attr("decode_ue8m0", _bias_off_by_one),
    "sf_byte_order_reversed": _mut_attr("unpack_sf", _byte_order_reversed),
    "b_transposed": _mut_attr("_scaled_gemm", _make_scaled("transposed_b")),
    "b_block_index_mod": _mut_attr("_scaled_gemm", _make_scaled("block_mod")),
    "dropped_last_group": _mut_attr("_scaled_gemm", _make_scaled("drop_last_group")),
    "a_scale_first_group_only": _mut_attr("_scaled_gemm", _make_scaled("first_scale_only")),
    "c_subtracted": _mut_attr("fp8_gemm_nt", _c_sign),
    "contiguous_pad_uses_last_expert": _mut_attr("m_grouped_fp8_gemm_nt_contiguous", _contig_negative_index),
    "masked_off_by_one": _mut_attr("m_grouped_fp8_gemm_nt_masked", _masked_off_by_one),
    "wgrad_c_rounded_to_bf16": _mut_attr("wgrad_gemm_fp8_fp8_fp32_nt", _wgrad_c_as_bf16),
    "wgrad_c_dropped": _mut_attr("wgrad_gemm_fp8_fp8_fp32_nt", _wgrad_c_dropped),
    "k_grouped_scales_packed_globally": _mut_attr("k_grouped_wgrad_gemm_fp8_fp8_fp32_nt", _k_grouped_global_packing),
    "tn_reads_a_as_k_major": _mut_attr("fp8_gemm_tn", _tn_forgets_to_transpose_a),
    "tt_reads_a_as_k_major": _mut_attr("fp8_gemm_tt", _tt_forgets_to_transpose_a),
    "nn_contiguous_reads_b_as_n_major": _mut_attr("m_grouped_fp8_gemm_nn_contiguous",
                                                  _nn_contiguous_reads_b_as_n_major),
    "tn_k_grouped_reads_b_as_k_major": _mut_attr("k_grouped_fp8_gemm_tn_contiguous",
                                                 _tn_k_grouped_reads_b_as_k_major),
    "fp4_subnormal_as_normal": _mut_e2m1(_e2m1_subnormal_as_normal),
    "fp4_sign_ignored": _mut_e2m1(lambda t: np.abs(t)),
    "fp4_high_nibble_first": _mut_attr("unpack_e2m1", _fp4_high_nibble_first),
    "fp4_b_scale_per_128": _mut_attr("_scaled_gemm_fp4", _make_scaled_fp4("b_scale_per_128")),
    "fp4_a_scale_per_32": _mut_attr("_scaled_gemm_fp4", _make_scaled_fp4("a_scale_per_32")),
    "parity_rms_over_d": _mut_attr("parity_report", _make_parity("rms_over_d")),
    "parity_rel_abs_swapped": _mut_attr("parity_report", _make_parity("rel_abs_swapped")),
    "parity_signed_ref": _mut_attr("parity_report", _make_parity("signed_ref")),
    "parity_nan_passes": _mut_attr("parity_report", _make_parity("nan_passes")),
    "parity_strict_bound": _mut_attr("parity_report", _make_parity("strict_bound")),
    "parity_diff_sign_flipped": _mut_attr("parity_report", _make_parity("diff_sign_flipped")),
    "parity_cos_not_strict": _mut_attr("parity_report", _make_parity("cos_not_strict")),
}


# pins that build exact rationals over grouped problems take ~1-2 s each: tried last
_SLOW_PINS = {"pin_k_grouped_equals_per_expert", "pin_grouped_layouts", "pin_masked_equals_dense",
              "pin_contiguous_equals_dense", "pin_brute_force", "pin_fp4_grouped_equals_dense",
              "pin_wgrad_brute_force", "pin_layouts"}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_is_caught(name):
    caught = None
    with MUTANTS[name]():
        for pin in sorted(PINS, key=lambda f: f.__name__ in _SLOW_PINS):
            try:
                pin(O)
            except (AssertionError, ValueError, IndexError):
                caught = pin.__name__
                break
    assert caught, f"planted mistake {name} passed every pin"


# --------------------------------------------------------------------------------------
# the input generator (not the method): its quantiser keeps values representable
# --------------------------------------------------------------------------------------

def test_quantiser_roundtrip_and_minimal_exponent():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((64, 512)).astype(np.float32) * 3
    x[0, :128] = 0.0
    q, e = W.quantize_rows(x)
    deq = torch_e4m3(q) * np.exp2(np.repeat(e.astype(np.float64) - 127, 128, axis=1))
    np.testing.assert_allclose(deq, x, rtol=2 ** -4, atol=2.0 ** -9 * 4)
    assert e[0, 0] == 127
    amax = np.abs(x.reshape(64, 4, 128)).max(2)
    ok = amax > 0
    assert (amax[ok] / np.exp2(e[ok].astype(np.float64) - 127) <= 448).all()
    assert (amax[ok] / np.exp2(e[ok].astype(np.float64) - 128) > 448).all()


def test_pack_sf_layout():
    e = np.arange(1, 1 + 6 * 5, dtype=np.uint8).reshape(6, 5)
    w = W.pack_sf(e)
    assert w.shape == (2, 8)
    assert np.array_equal(w, words_from_codes(e))
    assert np.array_equal(O.unpack_sf(w, 6, 5), e)


def test_fp4_quantiser_roundtrip_ties_and_packing():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((16, 256)) * 3).astype(np.float32)
    x[0, :32] = 0.0
    packed, e = W.quantize_fp4_rows(x)
    assert packed.shape == (16, 128) and e.shape == (16, 8)
    codes = np.stack([(packed >> 0) & 0xF, (packed >> 4) & 0xF], axis=-1).reshape(16, 256)   # even element low
    vals = np.array([float(e2m1_value(int(c))) for c in codes.reshape(-1)]).reshape(16, 256)
    scale = np.exp2(np.repeat(e.astype(np.float64) - 127, 32, axis=1))
    deq = vals * scale
    # E2M1 has one mantissa bit: within a quarter of the value's binade step, or half the
    # smallest step (0.5 * scale) near zero
    assert (np.abs(deq - x) <= np.maximum(0.25 * np.abs(x), 0.25 * scale) + 1e-12).all()
    assert e[0, 0] == 127 and (codes[0, :32] == 0).all()
    amax = np.abs(x.reshape(16, 8, 32)).max(2)
    ok = amax > 0
    assert (amax[ok] / np.exp2(e[ok].astype(np.float64) - 127) <= 6).all()      # fits E2M1
    assert (amax[ok] / np.exp2(e[ok].astype(np.float64) - 128) > 6).all()       # the least such exponent
    # ties go to the even code: 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0, 1.75 -> 2.0, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    t = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -5.0], np.float32)
    got = [float(e2m1_value(int(c))) for c in W._to_e2m1_codes(t)]
    assert got == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, -4.0]
    assert W.pack_fp4(np.array([[1, 2, 3, 4]], np.uint8)).tolist() == [[0x21, 0x43]]
