"""FP64 CPU oracle for the fine-grained-scaled FP8 GEMM D = C + A @ B.T.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or links this
package: only the tests, the smoke check and the benchmark's CPU-baseline leg do.
It shares no code with the CUDA library (``fp8_gemm_nt_gb300``) and imports nothing
from it; both sides consume the same seeded bytes from ``workloads``.

Sources. Citations name the DeepGEMM README as reproduced on the page "Weight
gradient kernels for dense and MoE models #95" (gitblind.noratr.app, DeepGEMM pull
95), by README section, plus the Hindi summary page "DeepGEMM: ... FP8 GEMM kernel"
(hi.news.hada.io topic 19459) where it restates the same section:

* "Interfaces / Notices": GEMMs are named after D = C + A @ B, the NT layout
  (fp8_gemm_nt computes D = C + A @ B.T), and the SM100 scale format (UE8M0 codes,
  four of them packed into one 32-bit integer; the LHS scales transposed and padded
  for TMA).
* "Grouped GEMMs (contiguous layout)": only M is grouped; N and K are fixed; each
  expert's token rows are concatenated and every segment is aligned to the M block.
* "Grouped GEMMs (masked layout)": a mask tensor gives each group's valid rows and
  only those are computed.

The pages print no formula beyond D = C + A @ B.T, and no scale granularity. This
oracle therefore writes out the plain definition with the granularity the workload
names (A: one scale per row per 128-wide K-group; B: one scale per 128x128 block):

    D[m, n] = C[m, n] + sum_g sA[m, g] * sB[n // 128, g] * sum_{k in group g} A[m, k] * B[n, k]

Readings where the pages are silent (each one is listed in the design notes):
E4M3 is the OCP "E4M3FN" encoding (bias 7, no infinities, S.1111.111 is NaN, max
448); UE8M0 code e means 2**(e - 127) and 255 is NaN; in a packed word, K-group
4q + j sits in byte j (least significant first) of word q; scales are stored
MN-major with the MN extent padded to a multiple of four words; the B scales use
the same MN-major packing over the N-block index.

Exactness. Every E4M3 value is an integer multiple of 2**-9 below 2**9, so each
product A*B is a multiple of 2**-18 below 2**18 and a 128-term group sum stays below
2**25 on the same 2**-18 grid: it is exact in FP64 in any summation order. Scaling
by powers of two is exact (away from the FP64 range ends), so the only rounding in
the result is the FP64 sum over K-groups. The group products use numpy's matmul as
a library step; its blocking cannot change an exact result.

Pins: tests/test_oracle_pins.py checks this module against the OCP code tables,
torch's own FP8/BF16 decoders, brute-force rational arithmetic on tiny inputs,
identity/one-hot operands, exact power-of-two scale invariance, the C-only case and
the grouped-equals-per-expert-dense identity; planted mistakes must fail a pin.
The FP8 x FP4 forms (end of the module) are pinned the same way: the OCP E2M1 table,
exact rationals with an independent nibble unpacking, one-hot closed forms, and the
identity with the FP8 form when every FP4 value and scale is also an FP8 one.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

GROUP_K = 128
BLOCK_N = 128


# --------------------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------------------

def _e4m3_table() -> np.ndarray:
    """All 256 E4M3FN codes decoded from the format's definition."""
    t = np.empty(256, np.float64)
    for code in range(256):
        s = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            t[code] = np.nan                      # the only NaN pattern; no infinities
        elif e == 0:
            t[code] = s * (m / 8.0) * 2.0 ** -6   # subnormal
        else:
            t[code] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return t


_E4M3 = _e4m3_table()


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """E4M3 bytes -> float64 ("FP8 E4M3" operands, README "Interfaces / Notices")."""
    return _E4M3[np.asarray(codes, dtype=np.uint8)]


def decode_ue8m0(codes: np.ndarray) -> np.ndarray:
    """UE8M0 scale codes -> float64: 2**(e-127); code 255 is NaN (README "Interfaces / Notices")."""
    e = np.asarray(codes, dtype=np.int64)
    out = np.ldexp(1.0, e - 127)
    return np.where(e == 255, np.nan, out)


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (a bf16 is the upper half of an IEEE fp32)."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u32.view(np.float32).astype(np.float64)


def unpack_sf(words: np.ndarray, mn: int, kgroups: int) -> np.ndarray:
    """Packed UE8M0 words [ceil(kgroups/4), >=mn] (MN-major) -> codes [mn, kgroups].

    On SM100 the scales are UE8M0 codes packed four to a 32-bit integer, and the LHS
    scales are stored transposed (README "Interfaces / Notices"). Reading: K-group g is
    byte g % 4 of word g // 4 of its row.
    """
    w = np.asarray(words).view(np.uint32)
    out = np.empty((mn, kgroups), np.uint8)
    for g in range(kgroups):
        out[:, g] = (w[g // 4, :mn] >> np.uint32(8 * (g % 4))) & np.uint32(0xFF)
    return out


# --------------------------------------------------------------------------------------
# the GEMM forms
# --------------------------------------------------------------------------------------

def _scaled_gemm(a_codes, sa_codes, b_codes, sb_codes, K: int) -> np.ndarray:
    """sum_g sA[:, g] * sB[n // 128, g] * (A_g @ B_g.T) in FP64.

    a_codes: E4M3 [R, K]; sa_codes: UE8M0 [R, KG]; b_codes: E4M3 [N, K];
    sb_codes: UE8M0 [ceil(N/128), KG] (one per 128x128 block of B).
    """
    KG = K // GROUP_K
    N = b_codes.shape[0]
    A = decode_e4m3(a_codes)                                                # [R, K]
    B = decode_e4m3(b_codes)                                                # [N, K]
    sA = decode_ue8m0(sa_codes)                                             # [R, KG]
    sB = decode_ue8m0(sb_codes)[np.arange(N) // BLOCK_N]                    # [N, KG]
    D = np.zeros((A.shape[0], N), np.float64)
    for g in range(KG):
        ks = slice(g * GROUP_K, (g + 1) * GROUP_K)
        partial = A[:, ks] @ B[:, ks].T                                     # exact
        D += sA[:, g:g + 1] * partial * sB[None, :, g]
    return D


def fp8_gemm_nt(a, sfa, b, sfb, c: Optional[np.ndarray], M: int, N: int, K: int,
                rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """D = C + A @ B.T with fine-grained scales, in FP64 (README "Interfaces / Notices",
    "Normal dense GEMMs (non-grouped)").

    a: uint8 [M, K]; sfa: int32 [ceil(KG/4), ceil4(M)]; b: uint8 [N, K];
    sfb: int32 [ceil(KG/4), ceil4(ceil(N/128))]; c: bf16 bits [M, N] or None.
    rows: optional subset of output rows to compute (default all). Returns [len(rows), N].
    """
    assert K % GROUP_K == 0
    KG = K // GROUP_K
    rows = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    sa = unpack_sf(sfa, M, KG)[rows]
    sb = unpack_sf(sfb, -(-N // BLOCK_N), KG)
    D = _scaled_gemm(np.asarray(a)[rows], sa, np.asarray(b), sb, K)
    if c is not None:
        D = decode_bf16(np.asarray(c)[rows]) + D
    return D


def fp8_gemm_nn(a, sfa, b, sfb, c, M: int, N: int, K: int) -> np.ndarray:
    """D = C + A @ B with A stored [M, K] and B stored [K, N] (README "Interfaces / Notices":
    the SM100 library supports the NT, TN, NN and TT layouts; "Normal dense GEMMs":
    fp8_gemm_{nt, nn, tn, tt}). The layout is storage only: the scales keep their meaning
    (A per row per 128-wide K-group, B per 128 x 128 block of the N x K view)."""
    return fp8_gemm_nt(a, sfa, np.ascontiguousarray(np.asarray(b).T), sfb, c, M, N, K)


def fp8_gemm_tn(a, sfa, b, sfb, c, M: int, N: int, K: int) -> np.ndarray:
    """D = C + A @ B with A stored transposed [K, M] and B stored [K, N] (see fp8_gemm_nn)."""
    return fp8_gemm_nt(np.ascontiguousarray(np.asarray(a).T), sfa, np.ascontiguousarray(np.asarray(b).T), sfb, c,
                       M, N, K)


def fp8_gemm_tt(a, sfa, b, sfb, c, M: int, N: int, K: int) -> np.ndarray:
    """D = C + A @ B.T with A stored transposed [K, M] and B stored [N, K] (see fp8_gemm_nn)."""
    return fp8_gemm_nt(np.ascontiguousarray(np.asarray(a).T), sfa, b, sfb, c, M, N, K)


def wgrad_gemm_fp8_fp8_fp32_nt(a, sfa, b, sfb, c: Optional[np.ndarray], M: int, N: int, K: int,
                               rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """Weight-gradient GEMM with FP32 output: D = C + A @ B.T, C and D FP32 (page "Weight
    gradient kernels for dense and MoE models #95": wgrad_gemm_fp8_fp8_fp32_nt, FP8 x FP8 ->
    FP32, NT layout). The pages give nothing beyond the name, so the reading is the plainest
    one: the same operands and scale format as fp8_gemm_nt, and an FP32 addend C (the
    gradient being accumulated; it may be the output buffer itself).

    c: float32 [M, N] or None. Returns FP64 [len(rows), N].
    """
    assert K % GROUP_K == 0
    KG = K // GROUP_K
    rows = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    sa = unpack_sf(sfa, M, KG)[rows]
    sb = unpack_sf(sfb, -(-N // BLOCK_N), KG)
    D = _scaled_gemm(np.asarray(a)[rows], sa, np.asarray(b), sb, K)
    if c is not None:
        D = np.asarray(c, dtype=np.float32)[rows].astype(np.float64) + D
    return D


def k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(a, sfa, b, sfb, c: Optional[np.ndarray], ks, M: int, N: int,
                                         groups: Optional[Sequence[int]] = None,
                                         rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """K-grouped weight-gradient GEMM for MoE (page "Weight gradient kernels for dense and MoE
    models #95": k_grouped_wgrad_gemm_fp8_fp8_fp32_nt; README "Grouped GEMMs": grouping along
    K, with M and N the same for every group). Expert g owns the K-slice [off_g, off_g + ks[g]) of A
    [M, K_total] and B [N, K_total] (off_g = ks[0] + ... + ks[g-1]) and gets its own FP32
    output: D[g] = C[g] + A[:, slice_g] @ B[:, slice_g].T.

    Readings (the pages name the function only): every ks[g] is a multiple of 128, so scale
    K-groups never straddle experts; the packed scale words are laid out per expert (the
    README lists a separate "K-grouped" packing utility): expert g's K-groups j = 0, 1, ...
    sit in byte j % 4 of word row R_g + j // 4, R_g = sum over h < g of ceil(ks[h] / 512),
    MN-major as elsewhere. An expert with ks[g] = 0 gets D[g] = C[g] (0 without C).

    a: uint8 [M, K_total]; sfa: int32 [sum_g ceil(ks_g/512), ceil4(M)]; b: uint8 [N, K_total];
    sfb: int32 [sum_g ceil(ks_g/512), ceil4(ceil(N/128))]; c: float32 [G, M, N] or None.
    Returns FP64 [len(groups), len(rows), N].
    """
    ks = [int(k) for k in ks]
    G = len(ks)
    assert all(k >= 0 and k % GROUP_K == 0 for k in ks)
    groups = range(G) if groups is None else groups
    rows = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    NB = -(-N // BLOCK_N)
    offs = np.concatenate([[0], np.cumsum(ks)]).astype(np.int64)
    word_rows = np.concatenate([[0], np.cumsum([-(-k // (4 * GROUP_K)) for k in ks])]).astype(np.int64)
    out = np.zeros((len(groups), len(rows), N), np.float64)
    for i, g in enumerate(groups):
        kg = ks[g] // GROUP_K
        if kg > 0:
            w0, w1 = word_rows[g], word_rows[g + 1]
            sa = unpack_sf(np.asarray(sfa)[w0:w1], M, kg)[rows]
            sb = unpack_sf(np.asarray(sfb)[w0:w1], NB, kg)
            ksl = slice(offs[g], offs[g + 1])
            out[i] = _scaled_gemm(np.asarray(a)[rows][:, ksl], sa, np.asarray(b)[:, ksl], sb, ks[g])
        if c is not None:
            out[i] = np.asarray(c, dtype=np.float32)[g][rows].astype(np.float64) + out[i]
    return out


def k_grouped_fp8_gemm_tn_contiguous(a, sfa, b, sfb, c: Optional[np.ndarray], ks, M: int, N: int,
                                     groups: Optional[Sequence[int]] = None,
                                     rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """The K-grouped GEMM with A stored [K_total, M] and B stored [K_total, N] (README
    "Grouped GEMMs (contiguous layout)": k_grouped_fp8_gemm_tn_contiguous, the API that groups
    K instead of M for the weight gradient of MoE layers). Storage only: the same D[g] = C[g] + A_g @ B_g.T as
    k_grouped_wgrad_gemm_fp8_fp8_fp32_nt over the logical [M, K_total] and [N, K_total]."""
    return k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(np.ascontiguousarray(np.asarray(a).T), sfa,
                                                np.ascontiguousarray(np.asarray(b).T), sfb, c, ks, M, N,
                                                groups=groups, rows=rows)


def m_grouped_fp8_gemm_nn_contiguous(a, sfa, b, sfb, m_indices, M_total: int, N: int, K: int, G: int,
                                     rows: Optional[Sequence[int]] = None):
    """Contiguous M-grouped GEMM with each expert's B stored [K, N] (README "Grouped GEMMs
    (contiguous layout)": m_grouped_fp8_gemm_{nt, nn}_contiguous). Storage only: b[g].T is
    the [N, K] matrix of the NT form."""
    bt = np.ascontiguousarray(np.transpose(np.asarray(b), (0, 2, 1)))
    return m_grouped_fp8_gemm_nt_contiguous(a, sfa, bt, sfb, m_indices, M_total, N, K, G, rows=rows)


def m_grouped_fp8_gemm_nt_contiguous(a, sfa, b, sfb, m_indices, M_total: int, N: int, K: int,
                                     G: int, rows: Optional[Sequence[int]] = None):
    """Contiguous M-grouped GEMM (README "Grouped GEMMs (contiguous layout)").

    Row r of A belongs to expert m_indices[r] and is multiplied by that expert's B
    [N, K] and scales; rows with m_indices == -1 are padding and produce nothing.
    Returns (D [R, N] float64 with NaN on padding rows, valid [R] bool).
    """
    KG = K // GROUP_K
    rows = np.arange(M_total) if rows is None else np.asarray(rows, dtype=np.int64)
    idx = np.asarray(m_indices)[rows]
    D = np.full((len(rows), N), np.nan)
    sa = unpack_sf(sfa, M_total, KG)
    NB = -(-N // BLOCK_N)
    for g in range(G):
        sel = np.nonzero(idx == g)[0]
        if len(sel) == 0:
            continue
        r = rows[sel]
        D[sel] = _scaled_gemm(np.asarray(a)[r], sa[r], np.asarray(b[g]), unpack_sf(sfb[g], NB, KG), K)
    return D, idx >= 0


def m_grouped_fp8_gemm_nt_masked(a, sfa, b, sfb, masked_m, G: int, max_m: int, N: int, K: int,
                                 groups: Optional[Sequence[int]] = None):
    """Masked M-grouped GEMM (README "Grouped GEMMs (masked layout)").

    For group g only rows r < masked_m[g] of A[g] are computed, against B[g].
    Returns (D [len(groups), max_m, N] float64 with NaN on masked rows,
    valid [len(groups), max_m] bool). A count above max_m is clamped to max_m.
    """
    KG = K // GROUP_K
    NB = -(-N // BLOCK_N)
    groups = list(range(G)) if groups is None else list(groups)
    D = np.full((len(groups), max_m, N), np.nan)
    valid = np.zeros((len(groups), max_m), bool)
    for i, g in enumerate(groups):
        m = int(min(max(int(masked_m[g]), 0), max_m))
        valid[i, :m] = True
        if m:
            sa = unpack_sf(sfa[g], max_m, KG)[:m]
            D[i, :m] = _scaled_gemm(np.asarray(a[g])[:m], sa, np.asarray(b[g]),
                                    unpack_sf(sfb[g], NB, KG), K)
    return D, valid


# --------------------------------------------------------------------------------------
# FP8 x FP4: E4M3 activations against E2M1 weights
# --------------------------------------------------------------------------------------
# The pages name the GEMM only (the DeepGEMM news entry of 2026.04.16, "FP8xFP4 GEMM", and
# the Mega MoE section, whose linear layers multiply FP8 activations by FP4 weights that carry
# UE8M0 scales).
# Readings, each the plainest one the pages allow:
# * the FP4 operand is OCP MX FP4 (E2M1: sign, 2 exponent bits with bias 1, 1 mantissa
#   bit; +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}; no infinities or NaN), two codes per byte, element
#   2j in the low nibble of byte j of its row (B stored [N, K/2] bytes, K-major as in NT);
# * its UE8M0 scales follow the MX block: one per row per 32 consecutive K-elements, packed
#   four per int32 along K (block 4q + j in byte j of word q) and stored MN-major
#   [K/128, ceil4(N)] words, the same "packed, transposed" format as A's scales;
# * A, its scales, C and D are exactly as in fp8_gemm_nt.
# Exactness: E4M3 x E2M1 products are multiples of 2**-10 below 2**12, so each 32-term block
# sum is exact in FP64 and the only rounding is the FP64 sum over blocks.

FP4_BLOCK_K = 32


def _e2m1_table() -> np.ndarray:
    """All 16 E2M1 codes decoded from the format's definition."""
    t = np.empty(16, np.float64)
    for code in range(16):
        s = -1.0 if code & 0x8 else 1.0
        e = (code >> 1) & 0x3
        m = code & 0x1
        t[code] = s * (0.5 * m if e == 0 else (1.0 + 0.5 * m) * 2.0 ** (e - 1))
    return t


_E2M1 = _e2m1_table()


def decode_e2m1(codes: np.ndarray) -> np.ndarray:
    """E2M1 codes (0..15) -> float64."""
    return _E2M1[np.asarray(codes, dtype=np.uint8) & 0xF]


def unpack_e2m1(packed: np.ndarray, K: int) -> np.ndarray:
    """Packed FP4 bytes [..., K/2] -> codes [..., K]: element 2j is the low nibble of byte j."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (K,), np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def _scaled_gemm_fp4(a_codes, sa_codes, b_codes, sb_codes, K: int) -> np.ndarray:
    """sum_j sA[:, j // 4] * sB[:, j] * (A_j @ B_j.T) over the 32-wide blocks j, in FP64.

    a_codes: E4M3 [R, K]; sa_codes: UE8M0 [R, K/128]; b_codes: E2M1 [N, K];
    sb_codes: UE8M0 [N, K/32] (one per row per 32-wide block of B).
    """
    A = decode_e4m3(a_codes)
    B = decode_e2m1(b_codes)
    sA = decode_ue8m0(sa_codes)
    sB = decode_ue8m0(sb_codes)
    D = np.zeros((A.shape[0], B.shape[0]), np.float64)
    for j in range(K // FP4_BLOCK_K):
        ks = slice(j * FP4_BLOCK_K, (j + 1) * FP4_BLOCK_K)
        D += sA[:, j * FP4_BLOCK_K // GROUP_K, None] * (A[:, ks] @ B[:, ks].T) * sB[None, :, j]
    return D


def fp8_fp4_gemm_nt(a, sfa, b, sfb, c: Optional[np.ndarray], M: int, N: int, K: int,
                    rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """D = C + A @ B.T with A E4M3 (scales 1 x 128) and B E2M1 (scales 1 x 32), in FP64
    (DeepGEMM news 2026.04.16 "FP8xFP4 GEMM"; README "Interfaces / Notices" for A, C, D and
    the scale packing; the readings above for B).

    a: uint8 [M, K]; sfa: int32 [ceil(K/512), ceil4(M)]; b: uint8 [N, K/2] (packed E2M1);
    sfb: int32 [K/128, ceil4(N)]; c: bf16 bits [M, N] or None. Returns FP64 [len(rows), N].
    """
    assert K % GROUP_K == 0
    rows = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    sa = unpack_sf(sfa, M, K // GROUP_K)[rows]
    sb = unpack_sf(sfb, N, K // FP4_BLOCK_K)
    D = _scaled_gemm_fp4(np.asarray(a)[rows], sa, unpack_e2m1(b, K), sb, K)
    if c is not None:
        D = decode_bf16(np.asarray(c)[rows]) + D
    return D


def m_grouped_fp8_fp4_gemm_nt_contiguous(a, sfa, b, sfb, m_indices, M_total: int, N: int, K: int, G: int,
                                         rows: Optional[Sequence[int]] = None):
    """Contiguous M-grouped FP8 x FP4 GEMM (README "Grouped GEMMs (contiguous layout)" with the
    FP4 weights read as in fp8_fp4_gemm_nt): row r uses expert m_indices[r]'s B [N, K/2] and
    scales [K/128, ceil4(N)]; padding rows (-1) produce nothing.
    Returns (D [R, N] float64 with NaN on padding rows, valid [R] bool)."""
    rows = np.arange(M_total) if rows is None else np.asarray(rows, dtype=np.int64)
    idx = np.asarray(m_indices)[rows]
    D = np.full((len(rows), N), np.nan)
    sa = unpack_sf(sfa, M_total, K // GROUP_K)
    for g in range(G):
        sel = np.nonzero(idx == g)[0]
        if len(sel) == 0:
            continue
        r = rows[sel]
        D[sel] = _scaled_gemm_fp4(np.asarray(a)[r], sa[r], unpack_e2m1(b[g], K),
                                  unpack_sf(sfb[g], N, K // FP4_BLOCK_K), K)
    return D, idx >= 0


def m_grouped_fp8_fp4_gemm_nt_masked(a, sfa, b, sfb, masked_m, G: int, max_m: int, N: int, K: int,
                                     groups: Optional[Sequence[int]] = None):
    """Masked M-grouped FP8 x FP4 GEMM (README "Grouped GEMMs (masked layout)" with the FP4
    weights read as in fp8_fp4_gemm_nt): group g computes rows r < masked_m[g] (clamped to
    [0, max_m]) of A[g] against B[g].
    Returns (D [len(groups), max_m, N] with NaN on masked rows, valid [len(groups), max_m])."""
    groups = list(range(G)) if groups is None else list(groups)
    D = np.full((len(groups), max_m, N), np.nan)
    valid = np.zeros((len(groups), max_m), bool)
    for i, g in enumerate(groups):
        m = int(min(max(int(masked_m[g]), 0), max_m))
        valid[i, :m] = True
        if m:
            sa = unpack_sf(sfa[g], max_m, K // GROUP_K)[:m]
            D[i, :m] = _scaled_gemm_fp4(np.asarray(a[g])[:m], sa, unpack_e2m1(b[g], K),
                                        unpack_sf(sfb[g], N, K // FP4_BLOCK_K), K)
    return D, valid


# --------------------------------------------------------------------------------------
# comparison (the parity bar)
# --------------------------------------------------------------------------------------

def parity_report(d: np.ndarray, ref: np.ndarray, rel: float = 1e-2, abs_rms: float = 1e-2,
                  cos_max: float = 1e-3):
    """The parity bar of the GEMM forms against this oracle (the workload's tolerance; the
    pages give only D = C + A @ B.T, README "Interfaces / Notices").

    Every element must satisfy |d - ref| <= rel*|ref| + abs_rms*rms(ref), where rms is taken
    over ref (the oracle), and the cosine-style difference
    1 - 2*sum(d*ref) / (sum(d^2) + sum(ref^2)) must be strictly below cos_max. A NaN in d (or
    ref) fails its element and makes the difference NaN, which also fails. An empty pair of
    arrays compares nothing and is reported ok with n = 0; callers that must compare
    something check n. d, ref are converted to float64."""
    d = np.asarray(d, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    err = np.abs(d - ref)
    bound = rel * np.abs(ref) + abs_rms * rms
    bad = ~(err <= bound)
    denom = float((d * d).sum() + (ref * ref).sum())
    diff = 0.0 if denom == 0.0 else 1.0 - 2.0 * float((d * ref).sum()) / denom
    return dict(n=int(ref.size), n_bad=int(bad.sum()), max_err=float(err.max()) if ref.size else 0.0,
                rms=rms, diff=diff, ok=bool(not bad.any() and diff < cos_max))
