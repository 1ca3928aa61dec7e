"""Seeded synthetic inputs for the fine-grained-scaled FP8 GEMM (D = C + A @ B.T).

This module only *makes inputs*. It holds none of the GEMM's arithmetic: the
kernels and the oracle both consume the bytes produced here, so a choice made
by the quantiser below (how a scale exponent is picked, how a value is rounded
to E4M3) can never cause a parity failure between them.

Input format (the library's boundary format, restated from the DeepGEMM README
as quoted on the pages, "Interfaces / Notices"): A and B are E4M3 bytes, both
K-major ("NT": A is [M, K] row-major, B is [N, K] row-major). Scale factors are
UE8M0 exponents packed four to one int32 (K-group 4q+j in byte j of word q,
little-endian), stored MN-major with the MN extent padded to a multiple of four
words (the transposed, TMA-padded layout). A has one scale per row per 128-wide
K-group; B has one scale per 128x128 block. The pages leave the packing byte
order and the B-scale layout open; these are the plain readings adopted here.

Every generator is deterministic in its seed (numpy PCG64). On the pages the caller
quantises its own inputs (the library does no FP8 casting for them); the recipe
used here is a per-group power-of-two scale that maps the group's
absolute maximum into the E4M3 range, then round-to-nearest-even to E4M3.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

GROUP_K = 128          # K-group width of one scale (A: 1x128, B: 128x128)
BLOCK_N = 128          # N extent of one B scale block
E4M3_MAX = 448.0
MK_ALIGNMENT = 128     # alignment of each expert segment in the contiguous layout


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def ceil4(x: int) -> int:
    return 4 * ceil_div(x, 4)


# --------------------------------------------------------------------------------------
# quantisation (input preparation, not the method)
# --------------------------------------------------------------------------------------

def _to_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    """Round fp32 values (already inside +-448) to E4M3 with torch's RNE cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def _scale_exponents(amax: np.ndarray, vmax: float = E4M3_MAX) -> np.ndarray:
    """Smallest UE8M0 code e (1..254) with amax / 2**(e-127) <= vmax; amax == 0 -> 127."""
    amax = np.asarray(amax, dtype=np.float64)
    with np.errstate(divide="ignore"):
        s = np.ceil(np.log2(np.where(amax > 0, amax, 1.0) / vmax))
    # fix any off-by-one from log2 rounding so that s is the least valid exponent
    s = np.where(np.ldexp(amax, -s.astype(np.int64)) > vmax, s + 1, s)
    s = np.where(np.ldexp(amax, -(s - 1).astype(np.int64)) <= vmax, s - 1, s)
    e = np.clip(s + 127, 1, 254)
    e = np.where(amax > 0, e, 127)
    return e.astype(np.uint8)


def quantize_rows(x: np.ndarray):
    """Per-row, per-128-K-group quantisation. x: fp32 [R, K] -> (E4M3 bytes [R, K], exps [R, K/128])."""
    R, K = x.shape
    assert K % GROUP_K == 0
    xg = x.reshape(R, K // GROUP_K, GROUP_K)
    e = _scale_exponents(np.abs(xg).max(axis=2))
    scaled = np.ldexp(xg.astype(np.float64), -(e.astype(np.int64) - 127)[:, :, None])
    return _to_e4m3_bytes(scaled.reshape(R, K).astype(np.float32)), e


def quantize_blocks(x: np.ndarray):
    """Per-128x128-block quantisation. x: fp32 [N, K] -> (E4M3 bytes [N, K], exps [ceil(N/128), K/128])."""
    N, K = x.shape
    assert K % GROUP_K == 0
    NB = ceil_div(N, BLOCK_N)
    pad = NB * BLOCK_N - N
    xp = np.concatenate([x, np.zeros((pad, K), x.dtype)]) if pad else x
    xb = xp.reshape(NB, BLOCK_N, K // GROUP_K, GROUP_K)
    e = _scale_exponents(np.abs(xb).max(axis=(1, 3)))                   # [NB, KG]
    rows_e = np.repeat(e, BLOCK_N, axis=0)[:N]                          # [N, KG]
    xg = x.reshape(N, K // GROUP_K, GROUP_K).astype(np.float64)
    scaled = np.ldexp(xg, -(rows_e.astype(np.int64) - 127)[:, :, None])
    return _to_e4m3_bytes(scaled.reshape(N, K).astype(np.float32)), e


E2M1_MAX = 6.0
FP4_BLOCK_K = 32       # K extent of one FP4 scale (the MX block)
_E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _to_e2m1_codes(x: np.ndarray) -> np.ndarray:
    """Round values (already inside +-6) to the nearest E2M1 magnitude, ties to the even
    code; the sign goes to bit 3 (zero magnitudes stay +0)."""
    x = np.asarray(x)
    mag = np.abs(x.astype(np.float64))
    mid = (_E2M1_MAGNITUDES[:-1] + _E2M1_MAGNITUDES[1:]) / 2          # 0.25, 0.75, ..., 5
    idx = np.searchsorted(mid, mag, side="left")                          # a tie lands on the lower code
    tie = (idx < len(mid)) & (mag == mid[np.minimum(idx, len(mid) - 1)]) & (idx % 2 == 1)
    idx = (idx + tie).astype(np.uint8)                                    # odd lower code: take the even one
    return np.where((x < 0) & (idx > 0), idx | 8, idx).astype(np.uint8)


def pack_fp4(codes: np.ndarray) -> np.ndarray:
    """E2M1 codes [..., K] -> bytes [..., K/2], element 2j in the low nibble of byte j."""
    c = np.asarray(codes, np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def quantize_fp4_rows(x: np.ndarray):
    """Per-row, per-32-K-block FP4 quantisation (the MX recipe): x fp32 [N, K] ->
    (packed E2M1 bytes [N, K/2], exps [N, K/32])."""
    N, K = x.shape
    assert K % GROUP_K == 0
    xb = x.reshape(N, K // FP4_BLOCK_K, FP4_BLOCK_K)
    e = _scale_exponents(np.abs(xb).max(axis=2), E2M1_MAX)
    scaled = np.ldexp(xb.astype(np.float64), -(e.astype(np.int64) - 127)[:, :, None])
    return pack_fp4(_to_e2m1_codes(scaled.reshape(N, K))), e


def pack_sf(exps: np.ndarray) -> np.ndarray:
    """UE8M0 exponents [MN, KG] -> packed int32 words [ceil(KG/4), ceil4(MN)] (MN-major)."""
    MN, KG = exps.shape
    KP = ceil_div(KG, 4)
    padded = np.zeros((ceil4(MN), KP * 4), np.uint8)
    padded[:MN, :KG] = exps
    # byte j of word q holds K-group 4q + j (little-endian)
    words = padded.reshape(ceil4(MN), KP, 4).copy().view("<u4").reshape(ceil4(MN), KP)
    return np.ascontiguousarray(words.T).view(np.int32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


# --------------------------------------------------------------------------------------
# problem containers
# --------------------------------------------------------------------------------------

@dataclasses.dataclass
class Dense:
    a: np.ndarray              # uint8 [M, K]
    sfa: np.ndarray            # int32 [KP, ceil4(M)]
    b: np.ndarray              # uint8 [N, K]
    sfb: np.ndarray            # int32 [KP, ceil4(ceil(N/128))]
    c: Optional[np.ndarray]    # uint16 bf16 bits [M, N] or None
    M: int
    N: int
    K: int
    layout: str = "nt"         # how a and b are stored on the device (the arrays here are always NT)
    b_format: str = "e4m3"     # "e2m1": b is packed FP4 [N, K/2], sfb per row per 32 K [K/128, ceil4(N)]

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


@dataclasses.dataclass
class Wgrad:
    """Weight-gradient GEMM operands: like Dense, with an FP32 addend / output."""
    a: np.ndarray              # uint8 [M, K]
    sfa: np.ndarray            # int32 [KP, ceil4(M)]
    b: np.ndarray              # uint8 [N, K]
    sfb: np.ndarray            # int32 [KP, ceil4(ceil(N/128))]
    c: Optional[np.ndarray]    # float32 [M, N] or None
    M: int
    N: int
    K: int

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


@dataclasses.dataclass
class KGrouped:
    """K-grouped weight-gradient operands: expert g owns K-slice [off_g, off_g + ks[g])."""
    a: np.ndarray              # uint8 [M, K_total]
    sfa: np.ndarray            # int32 [sum_g ceil(ks_g/512), ceil4(M)], packed per expert
    b: np.ndarray              # uint8 [N, K_total]
    sfb: np.ndarray            # int32 [sum_g ceil(ks_g/512), ceil4(ceil(N/128))], packed per expert
    c: Optional[np.ndarray]    # float32 [G, M, N] or None
    ks: np.ndarray             # int32 [G], multiples of 128
    M: int
    N: int

    @property
    def G(self) -> int:
        return len(self.ks)

    @property
    def K_total(self) -> int:
        return int(self.ks.sum())

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * float(self.ks.sum())


@dataclasses.dataclass
class Contiguous:
    a: np.ndarray              # uint8 [M_total, K]
    sfa: np.ndarray            # int32 [KP, ceil4(M_total)]
    b: np.ndarray              # uint8 [G, N, K]
    sfb: np.ndarray            # int32 [G, KP, ceil4(ceil(N/128))]
    m_indices: np.ndarray      # int32 [M_total], expert id or -1 for padding
    M_total: int
    N: int
    K: int
    G: int
    b_format: str = "e4m3"     # "e2m1": b is packed FP4 [G, N, K/2], sfb [G, K/128, ceil4(N)]

    @property
    def valid_rows(self) -> int:
        return int((self.m_indices >= 0).sum())

    @property
    def flops(self) -> float:
        return 2.0 * self.valid_rows * self.N * self.K


@dataclasses.dataclass
class Masked:
    a: np.ndarray              # uint8 [G, max_m, K]
    sfa: np.ndarray            # int32 [G, KP, ceil4(max_m)]
    b: np.ndarray              # uint8 [G, N, K]
    sfb: np.ndarray            # int32 [G, KP, ceil4(ceil(N/128))]
    masked_m: np.ndarray       # int32 [G]
    G: int
    max_m: int
    N: int
    K: int
    b_format: str = "e4m3"     # "e2m1": b is packed FP4 [G, N, K/2], sfb [G, K/128, ceil4(N)]

    @property
    def flops(self) -> float:
        return 2.0 * float(np.minimum(self.masked_m, self.max_m).sum()) * self.N * self.K


# --------------------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------------------

def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _normal(rng, shape, row_magnitude: bool = False) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if row_magnitude:  # per-row magnitude ~ logU(0.1, 10)
        r = np.exp(rng.uniform(math.log(0.1), math.log(10.0), size=shape[:-1] + (1,)))
        x *= r.astype(np.float32)
    return x


def make_dense(M: int, N: int, K: int, seed: int, with_c: bool = False,
               row_magnitude: bool = False) -> Dense:
    rng = _rng(seed)
    a, ea = quantize_rows(_normal(rng, (M, K), row_magnitude))
    b, eb = quantize_blocks(_normal(rng, (N, K), row_magnitude))
    c = to_bf16_bits(rng.standard_normal((M, N), dtype=np.float32)) if with_c else None
    return Dense(a, pack_sf(ea), b, pack_sf(eb), c, M, N, K)


def make_dense_fp4(M: int, N: int, K: int, seed: int, with_c: bool = False) -> Dense:
    """A quantised like make_dense; B [N, K] quantised to FP4 with one scale per row per 32 K."""
    rng = _rng(seed)
    a, ea = quantize_rows(_normal(rng, (M, K)))
    b, eb = quantize_fp4_rows(_normal(rng, (N, K)))
    c = to_bf16_bits(rng.standard_normal((M, N), dtype=np.float32)) if with_c else None
    return Dense(a, pack_sf(ea), b, pack_sf(eb), c, M, N, K, b_format="e2m1")


def make_wgrad(M: int, N: int, K: int, seed: int, with_c: bool = True) -> Wgrad:
    """A, B quantised like make_dense; C ~ N(0,1) in FP32 (the gradient accumulated so far)."""
    rng = _rng(seed)
    a, ea = quantize_rows(_normal(rng, (M, K)))
    b, eb = quantize_blocks(_normal(rng, (N, K)))
    c = rng.standard_normal((M, N), dtype=np.float32) if with_c else None
    return Wgrad(a, pack_sf(ea), b, pack_sf(eb), c, M, N, K)


def pack_sf_k_grouped(exps: np.ndarray, ks) -> np.ndarray:
    """Exponents [MN, K_total/128] -> words packed per expert K-slice, concatenated along the
    word-row axis: [sum_g ceil(ks_g/512), ceil4(MN)]."""
    parts, off = [], 0
    for k in ks:
        kg = int(k) // GROUP_K
        if kg > 0:
            parts.append(pack_sf(exps[:, off:off + kg]))
        off += kg
    if not parts:
        return np.zeros((0, ceil4(exps.shape[0])), np.int32)
    return np.ascontiguousarray(np.concatenate(parts, axis=0))


def make_k_grouped(G: int, M: int, N: int, tokens: int, seed: int, with_c: bool = True,
                   ks: Optional[np.ndarray] = None) -> KGrouped:
    """Token counts ~ Multinomial(tokens, 1/G) per expert (or given), each rounded up to a
    multiple of 128 (the alignment the K-grouped layout needs); A [M, K_total] and B [N, K_total]
    quantised like make_dense over the concatenated K; C ~ N(0,1) FP32 per expert."""
    rng = _rng(seed)
    if ks is None:
        counts = rng.multinomial(tokens, [1.0 / G] * G)
        ks = np.array([MK_ALIGNMENT * ceil_div(int(c), MK_ALIGNMENT) for c in counts], np.int32)
    ks = np.asarray(ks, dtype=np.int32)
    K_total = int(ks.sum())
    a, ea = quantize_rows(_normal(rng, (M, max(K_total, GROUP_K))))
    b, eb = quantize_blocks(_normal(rng, (N, max(K_total, GROUP_K))))
    a, ea, b, eb = a[:, :K_total], ea[:, :K_total // GROUP_K], b[:, :K_total], eb[:, :K_total // GROUP_K]
    c = rng.standard_normal((len(ks), M, N), dtype=np.float32) if with_c else None
    return KGrouped(np.ascontiguousarray(a), pack_sf_k_grouped(ea, ks), np.ascontiguousarray(b),
                    pack_sf_k_grouped(eb, ks), c, ks, M, N)


def _make_b_grouped(rng, G, N, K, b_format="e4m3"):
    bs, sfbs = [], []
    for _ in range(G):
        if b_format == "e2m1":
            b, eb = quantize_fp4_rows(_normal(rng, (N, K)))
        else:
            b, eb = quantize_blocks(_normal(rng, (N, K)))
        bs.append(b)
        sfbs.append(pack_sf(eb))
    return np.stack(bs), np.stack(sfbs)


def make_contiguous(G: int, tokens: int, N: int, K: int, seed: int,
                    counts: Optional[np.ndarray] = None, b_format: str = "e4m3") -> Contiguous:
    """Token rows split among G experts by a uniform multinomial (or given counts); each
    expert segment padded to a multiple of 128 rows with m_indices = -1 on the padding."""
    rng = _rng(seed)
    if counts is None:
        counts = rng.multinomial(tokens, [1.0 / G] * G)
    counts = np.asarray(counts, dtype=np.int64)
    seg = [MK_ALIGNMENT * ceil_div(int(c), MK_ALIGNMENT) for c in counts]
    M_total = int(sum(seg))
    m_indices = np.full(M_total, -1, np.int32)
    off = 0
    for g, (cnt, s) in enumerate(zip(counts, seg)):
        m_indices[off:off + int(cnt)] = g
        off += s
    a, ea = quantize_rows(_normal(rng, (max(M_total, 1), K)))
    a, ea = a[:M_total], ea[:M_total]
    b, sfb = _make_b_grouped(rng, G, N, K, b_format)
    return Contiguous(a, pack_sf(ea), b, sfb, m_indices, M_total, N, K, G, b_format)


def make_masked(G: int, max_m: int, N: int, K: int, seed: int,
                masked_m: Optional[np.ndarray] = None, b_format: str = "e4m3") -> Masked:
    """A [G, max_m, K]; masked_m ~ U{0..max_m} per expert (or given); rows past masked_m
    hold ordinary random data that the GEMM must ignore."""
    rng = _rng(seed)
    if masked_m is None:
        masked_m = rng.integers(0, max_m + 1, size=G)
    masked_m = np.asarray(masked_m, dtype=np.int32)
    a_list, sfa_list = [], []
    for _ in range(G):
        a, ea = quantize_rows(_normal(rng, (max_m, K)))
        a_list.append(a)
        sfa_list.append(pack_sf(ea))
    b, sfb = _make_b_grouped(rng, G, N, K, b_format)
    return Masked(np.stack(a_list), np.stack(sfa_list), b, sfb, masked_m, G, max_m, N, K, b_format)


# --------------------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------------------

SEED_BASE = 20260

WORKLOADS = {
    "dense_128x256x512": dict(kind="dense", M=128, N=256, K=512, with_c=False),
    "dense_decode_128x7168x16384_c": dict(kind="dense", M=128, N=7168, K=16384, with_c=True),
    "dense_prefill_4096x24576x1536": dict(kind="dense", M=4096, N=24576, K=1536, with_c=False,
                                          row_magnitude=True),
    "contiguous_g8_t32768_n4096_k7168": dict(kind="contiguous", G=8, tokens=32768, N=4096, K=7168),
    "masked_g32_m256_n7168_k2048": dict(kind="masked", G=32, max_m=256, N=7168, K=2048),
    # weight gradient of a 7168 x 4096 projection over 4096 tokens, accumulated into FP32
    "wgrad_7168x4096x4096_c": dict(kind="wgrad", M=7168, N=4096, K=4096, with_c=True),
    # data gradient of a 7168 -> 2048 projection over 4096 tokens: dX = dY @ W, W stored [K, N]
    "dense_nn_4096x7168x2048": dict(kind="dense_layout", layout="nn", M=4096, N=7168, K=2048, with_c=False),
    # MoE weight gradient: 4 experts, 4096 x 7168 each, 16384 tokens split among them
    "k_grouped_wgrad_g4_m4096_n7168_t16384": dict(kind="k_grouped", G=4, M=4096, N=7168, tokens=16384),
    # FP8 x FP4 (weights in FP4 with per-32 UE8M0 scales): the decode and MoE shapes above
    "fp4_dense_decode_128x7168x16384_c": dict(kind="dense_fp4", M=128, N=7168, K=16384, with_c=True),
    "fp4_masked_g32_m256_n7168_k2048": dict(kind="masked", G=32, max_m=256, N=7168, K=2048, b_format="e2m1"),
    "fp4_contiguous_g8_t32768_n4096_k7168": dict(kind="contiguous", G=8, tokens=32768, N=4096, K=7168,
                                                 b_format="e2m1"),
}
WORKLOAD_ORDER = list(WORKLOADS)


def make_workload(name: str):
    spec = dict(WORKLOADS[name])
    seed = SEED_BASE + WORKLOAD_ORDER.index(name)
    kind = spec.pop("kind")
    if kind == "dense":
        return make_dense(seed=seed, **spec)
    if kind == "dense_fp4":
        return make_dense_fp4(seed=seed, **spec)
    if kind == "contiguous":
        return make_contiguous(seed=seed, **spec)
    if kind == "wgrad":
        return make_wgrad(seed=seed, **spec)
    if kind == "dense_layout":
        layout = spec.pop("layout")
        p = make_dense(seed=seed, **spec)
        p.layout = layout          # storage of A ("n": [M, K], "t": [K, M]) and B ("n": [K, N], "t": [N, K])
        return p
    if kind == "k_grouped":
        return make_k_grouped(seed=seed, **spec)
    return make_masked(seed=seed, **spec)


def sentinel_bits() -> int:
    """bf16 quiet-NaN bit pattern used to prefill D: any write to it is detectable bit-exactly."""
    return 0x7FC1
