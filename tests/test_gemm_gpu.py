"""GPU parity tests: the CUDA library (through its C ABI) against the FP64 oracle.

Bar: per element |d - ref| <= 1e-2*|ref| + 1e-2*rms(ref) and the cosine-style
difference below 1e-3 for floating point; bit-exact for everything the integer
indexing decides (padding rows, masked rows, guard values) and for the exact cases
(identity / one-hot operands, power-of-two scale shifts, C-only).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import (SENTINEL, assert_parity, bf16_bits, bf16_f64, dev, run_contiguous, run_dense,
                      run_masked, sentinel_like)

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


# --------------------------------------------------------------------------------------
# dense
# --------------------------------------------------------------------------------------

DENSE_SHAPES = [
    (128, 256, 512, False),     # the small workload
    (1, 16, 128, False),        # single row, single K-group
    (77, 48, 384, True),        # ragged M and N, with C
    (300, 400, 640, True),      # several tiles with ragged tails in M and N, KG = 5
    (256, 384, 1152, False),    # KG = 9: last packed word only partly used
    (130, 1040, 2048, True),
    (513, 272, 256, False),
]


@pytest.mark.parametrize("M,N,K,with_c", DENSE_SHAPES)
def test_dense_parity(lib, M, N, K, with_c):
    p = W.make_dense(M, N, K, seed=1000 + M + N + K, with_c=with_c)
    d = run_dense(lib, p)
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, M, N, K)
    assert_parity(bf16_f64(d), ref, f"dense {M}x{N}x{K}")


def test_dense_row_magnitudes(lib):
    p = W.make_dense(384, 512, 1536, seed=77, row_magnitude=True)
    d = run_dense(lib, p)
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, None, p.M, p.N, p.K)
    assert_parity(bf16_f64(d), ref, "row magnitudes")


def test_dense_c_aliases_d(lib):
    p = W.make_dense(200, 320, 512, seed=5, with_c=True)
    d = run_dense(lib, p, c_alias=True)
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, p.c, p.M, p.N, p.K)
    assert_parity(bf16_f64(d), ref, "c aliases d")


def test_dense_identity_bit_exact(lib):
    # A = [I | 0], unit scales: D[i, n] = B[n, i] exactly (E4M3 values are exact in BF16)
    M, N, K = 128, 256, 256
    rng = np.random.default_rng(3)
    a = np.zeros((M, K), np.uint8)
    a[np.arange(M), np.arange(M)] = 0x38
    b = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    b[(b & 0x7F) == 0x7F] = 0x30
    sfa = W.pack_sf(np.full((M, 2), 127, np.uint8))
    sfb = W.pack_sf(np.full((2, 2), 127, np.uint8))
    p = W.Dense(a, sfa, b, sfb, None, M, N, K)
    d = run_dense(lib, p)
    expect = O.decode_e4m3(b[:, :M]).T
    got = bf16_f64(d)
    assert np.array_equal(got, expect)


def test_dense_one_hot_scales_bit_exact(lib):
    # one nonzero per row at a different K-group; per-row and per-block scales are
    # distinct powers of two, so a wrong scale row/column/byte shows up exactly
    M, N, K = 128, 384, 1024
    rng = np.random.default_rng(4)
    b = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    b[(b & 0x7F) == 0x7F] = 0x30
    a = np.zeros((M, K), np.uint8)
    ks = rng.integers(0, K, size=M)
    a[np.arange(M), ks] = 0x38
    ea = rng.integers(120, 135, size=(M, K // 128)).astype(np.uint8)
    eb = rng.integers(120, 135, size=(N // 128, K // 128)).astype(np.uint8)
    p = W.Dense(a, W.pack_sf(ea), b, W.pack_sf(eb), None, M, N, K)
    d = run_dense(lib, p)
    ref = O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, None, M, N, K)
    ref_bf16 = torch.from_numpy(ref).to(torch.bfloat16).to(torch.float64).numpy()
    got = bf16_f64(d)
    bad = np.argwhere(got != ref_bf16)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:5].tolist()}"


def test_dense_pow2_row_and_block_shift_bit_exact(lib):
    p = W.make_dense(256, 512, 768, seed=9)
    base = bf16_bits(run_dense(lib, p))
    KG = p.K // 128
    ea = O.unpack_sf(p.sfa, p.M, KG).copy()
    ea[17] += 2                                   # row 17 x 4
    eb = O.unpack_sf(p.sfb, 4, KG).copy()
    eb[3] -= 1                                    # columns 384..511 x 1/2
    q = W.Dense(p.a, W.pack_sf(ea), p.b, W.pack_sf(eb), None, p.M, p.N, p.K)
    got = bf16_f64(run_dense(lib, q))
    expect = torch.from_numpy(base.view(np.int16)).view(torch.bfloat16).double().numpy()
    expect[17] *= 4.0
    expect[:, 384:] *= 0.5
    assert np.array_equal(got, expect)


def test_dense_c_only_bit_exact(lib):
    M, N, K = 96, 160, 256
    p = W.make_dense(M, N, K, seed=2, with_c=True)
    p.a[:] = 0
    d = run_dense(lib, p)
    assert np.array_equal(bf16_bits(d), p.c)


def test_dense_m_zero_is_noop(lib):
    p = W.make_dense(1, 32, 128, seed=1)
    d = sentinel_like((1, 32))
    lib.dg_fp8_gemm_nt(dev(p.a)[:0], torch.zeros((1, 0), dtype=torch.int32, device="cuda"), dev(p.b), dev(p.sfb),
                       None, d[:0])
    torch.cuda.synchronize()
    assert (bf16_bits(d) == SENTINEL).all()


# --------------------------------------------------------------------------------------
# contiguous
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("counts,N,K", [
    ([130, 0, 170, 1], 144, 256),
    ([128, 256, 5, 300], 400, 640),
    ([0, 0, 7], 64, 128),
])
def test_contiguous_parity_and_padding(lib, counts, N, K):
    p = W.make_contiguous(G=len(counts), tokens=sum(counts), N=N, K=K, seed=31 + N, counts=counts)
    d = run_contiguous(lib, p)
    ref, valid = O.m_grouped_fp8_gemm_nt_contiguous(p.a, p.sfa, p.b, p.sfb, p.m_indices, p.M_total, p.N, p.K, p.G)
    bits = bf16_bits(d)
    assert (bits[~valid] == SENTINEL).all(), "padding rows were written"
    assert_parity(bf16_f64(d)[valid], ref[valid], f"contiguous {counts}")


def test_contiguous_equals_dense_per_expert(lib):
    p = W.make_contiguous(G=3, tokens=600, N=256, K=512, seed=8, counts=[250, 100, 250])
    d = bf16_bits(run_contiguous(lib, p))
    KG = p.K // 128
    ea = O.unpack_sf(p.sfa, p.M_total, KG)
    for g in range(p.G):
        r = np.nonzero(p.m_indices == g)[0]
        q = W.Dense(p.a[r], W.pack_sf(ea[r]), p.b[g], p.sfb[g], None, len(r), p.N, p.K)
        dd = bf16_bits(run_dense(lib, q))
        assert np.array_equal(d[r], dd), f"expert {g}"


def test_contiguous_bad_index_reported(lib):
    p = W.make_contiguous(G=2, tokens=200, N=64, K=128, seed=2, counts=[100, 100])
    p.m_indices[128:128 + 100] = 5          # out-of-range expert for the second segment
    d = run_contiguous(lib, p)
    assert lib.dg_get_device_status() == 6
    bits = bf16_bits(d)
    assert (bits[128:] == SENTINEL).all(), "rows of an invalid expert were written"
    assert lib.dg_get_device_status() == 0  # cleared by the read


# --------------------------------------------------------------------------------------
# masked
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("masked_m,max_m,N,K", [
    ([0, 40, 17, 1], 40, 136 - 8, 256),
    ([256, 0, 129, 128, 3], 256, 320, 512),
    ([5, 200], 200, 64, 384),
])
def test_masked_parity_and_mask(lib, masked_m, max_m, N, K):
    p = W.make_masked(G=len(masked_m), max_m=max_m, N=N, K=K, seed=41 + N, masked_m=masked_m)
    d = run_masked(lib, p)
    ref, valid = O.m_grouped_fp8_gemm_nt_masked(p.a, p.sfa, p.b, p.sfb, p.masked_m, p.G, p.max_m, p.N, p.K)
    bits = bf16_bits(d)
    assert (bits[~valid] == SENTINEL).all(), "masked rows were written"
    assert_parity(bf16_f64(d)[valid], ref[valid], f"masked {masked_m}")


def test_masked_many_groups_beyond_count_cache(lib):
    # more groups than the kernel caches in shared memory (1024): the counts past the cache
    # are read from global memory; a few non-empty groups on both sides of the boundary
    G, max_m, N, K = 1100, 16, 32, 128
    masked_m = np.zeros(G, np.int32)
    masked_m[[0, 5, 1023, 1024, 1060, 1099]] = [3, 16, 1, 7, 16, 2]
    p = W.make_masked(G=G, max_m=max_m, N=N, K=K, seed=77, masked_m=masked_m)
    d = run_masked(lib, p)
    groups = [0, 5, 1023, 1024, 1060, 1099, 1, 1050]
    ref, valid = O.m_grouped_fp8_gemm_nt_masked(p.a, p.sfa, p.b, p.sfb, p.masked_m, p.G, p.max_m, p.N, p.K,
                                                groups=groups)
    got = bf16_f64(d)[groups]
    assert (bf16_bits(d)[groups][~valid] == SENTINEL).all()
    assert_parity(got[valid], ref[valid], "masked, 1100 groups")
    untouched = np.ones(G, bool)
    untouched[[0, 5, 1023, 1024, 1060, 1099]] = False
    assert (bf16_bits(d)[untouched] == SENTINEL).all()


def test_masked_count_above_max_is_clamped(lib):
    p = W.make_masked(G=2, max_m=64, N=64, K=128, seed=3, masked_m=[100, 10])
    d = run_masked(lib, p)
    assert lib.dg_get_device_status() == 6
    ref, valid = O.m_grouped_fp8_gemm_nt_masked(p.a, p.sfa, p.b, p.sfb, p.masked_m, p.G, p.max_m, p.N, p.K)
    assert valid[0].all() and valid[1].sum() == 10
    assert (bf16_bits(d)[~valid] == SENTINEL).all()
    assert_parity(bf16_f64(d)[valid], ref[valid], "clamped")


# --------------------------------------------------------------------------------------
# scale packing
# --------------------------------------------------------------------------------------

def test_pack_sf_matches_layout(lib):
    rng = np.random.default_rng(0)
    e = rng.integers(1, 255, size=(70, 9)).astype(np.uint8)
    f = np.ldexp(np.ones_like(e, dtype=np.float32), e.astype(np.int32) - 127).astype(np.float32)
    out = lib.dg_pack_sf_ue8m0(dev(f))
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), W.pack_sf(e))
    out_t = lib.dg_pack_sf_ue8m0(dev(np.ascontiguousarray(f.T)), mn_major=True)   # [kgroups, mn] input
    torch.cuda.synchronize()
    assert np.array_equal(out_t.cpu().numpy(), W.pack_sf(e))
    # non-powers of two round up to the next power of two
    g = f * np.float32(1.5)
    g[e >= 254] = f[e >= 254]
    out2 = lib.dg_pack_sf_ue8m0(dev(np.ascontiguousarray(g)))
    torch.cuda.synchronize()
    e2 = np.where(e >= 254, e, e + 1).astype(np.uint8)
    assert np.array_equal(out2.cpu().numpy(), W.pack_sf(e2))


def test_pack_sf_gives_the_fp4_scale_layout(lib):
    # FP4 B's scales (one per row per 32 K) are packed by the same utility: FP32 scales
    # [N, K/32] -> int32 [K/128, ceil4(N)], and a GEMM with them matches the oracle
    p = W.make_dense_fp4(64, 208, 512, seed=21)
    eb = O.unpack_sf(p.sfb, p.N, p.K // 32)
    f = np.ldexp(np.ones(eb.shape, np.float32), eb.astype(np.int32) - 127).astype(np.float32)
    packed = lib.dg_pack_sf_ue8m0(dev(f))
    torch.cuda.synchronize()
    assert np.array_equal(packed.cpu().numpy(), p.sfb)
    d = sentinel_like((p.M, p.N))
    lib.dg_fp8_fp4_gemm_nt(dev(p.a), dev(p.sfa), dev(p.b), packed, None, d)
    torch.cuda.synchronize()
    assert_parity(bf16_f64(d), O.fp8_fp4_gemm_nt(p.a, p.sfa, p.b, p.sfb, None, p.M, p.N, p.K), "packed FP4 scales")


def test_masked_graph_replay_reads_counts_on_the_device(lib):
    # the masked form is captured once into a CUDA graph; replays pick up new per-expert
    # counts written to device memory (the CPU never learns them), as the pages intend for
    # decoding with CUDA graphs
    p = W.make_masked(G=4, max_m=256, N=384, K=512, seed=61, masked_m=[256, 0, 100, 3])
    a, sfa, b, sfb = dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb)
    mm = dev(p.masked_m.astype(np.int32))
    d = sentinel_like((p.G, p.max_m, p.N))
    lib.dg_m_grouped_fp8_gemm_nt_masked(a, sfa, b, sfb, d, mm)          # outside capture: lazy set-up
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        lib.dg_m_grouped_fp8_gemm_nt_masked(a, sfa, b, sfb, d, mm)
    for counts in ([17, 256, 0, 129], [0, 0, 0, 1], [256, 256, 256, 256]):
        counts = np.array(counts, np.int32)
        mm.copy_(torch.from_numpy(counts))
        d.view(torch.int16).fill_(SENTINEL - 65536 if SENTINEL >= 32768 else SENTINEL)
        graph.replay()
        torch.cuda.synchronize()
        ref, valid = O.m_grouped_fp8_gemm_nt_masked(p.a, p.sfa, p.b, p.sfb, counts, p.G, p.max_m, p.N, p.K)
        bits = bf16_bits(d)
        assert (bits[~valid] == SENTINEL).all(), counts
        assert_parity(bf16_f64(d)[valid], ref[valid], f"graph replay {counts.tolist()}")


# --------------------------------------------------------------------------------------
# inputs written by the kernel right before the GEMM (the dispatch step of a MoE layer)
# --------------------------------------------------------------------------------------

def test_masked_counts_written_by_the_previous_kernel(lib):
    # the counts come from a device kernel launched just before each GEMM on the same stream:
    # every launch must read the new values (the kernels read their inputs at L2 after the
    # dependency wait)
    p = W.make_masked(G=8, max_m=256, N=512, K=512, seed=91, masked_m=[0] * 8)
    a, sfa, b, sfb = dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb)
    mm = torch.zeros(8, dtype=torch.int32, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(5)
    for it in range(6):
        d = sentinel_like((p.G, p.max_m, p.N))
        mm.copy_(torch.randint(0, p.max_m + 1, (p.G,), device="cuda", generator=gen, dtype=torch.int32))
        lib.dg_m_grouped_fp8_gemm_nt_masked(a, sfa, b, sfb, d, mm)
        torch.cuda.synchronize()
        counts = mm.cpu().numpy()
        ref, valid = O.m_grouped_fp8_gemm_nt_masked(p.a, p.sfa, p.b, p.sfb, counts, p.G, p.max_m, p.N, p.K)
        bits = bf16_bits(d)
        assert (bits[~valid] == SENTINEL).all(), f"launch {it}: rows past the counts were written"
        assert not (bits[valid] == SENTINEL).any(), f"launch {it}: counted rows were not written"
        assert_parity(bf16_f64(d)[valid], ref[valid], f"launch {it}")


def test_contiguous_indices_written_by_the_previous_kernel(lib):
    # the row -> expert map is rewritten on the device before each launch (experts permuted)
    q = W.make_contiguous(G=3, tokens=600, N=256, K=512, seed=92, counts=[250, 100, 250])
    a, sfa, b, sfb = dev(q.a), dev(q.sfa), dev(q.b), dev(q.sfb)
    idx = dev(q.m_indices)
    base = torch.from_numpy(q.m_indices).cuda()
    for it, perm in enumerate(([0, 1, 2], [2, 0, 1], [1, 2, 0])):
        table = torch.tensor(perm + [-1], dtype=torch.int32, device="cuda")
        idx.copy_(table[base.long()])          # -1 maps to table[-1] = -1
        d = sentinel_like((q.M_total, q.N))
        lib.dg_m_grouped_fp8_gemm_nt_contiguous(a, sfa, b, sfb, d, idx)
        torch.cuda.synchronize()
        m_idx = idx.cpu().numpy()
        ref, valid = O.m_grouped_fp8_gemm_nt_contiguous(q.a, q.sfa, q.b, q.sfb, m_idx, q.M_total, q.N, q.K, q.G)
        assert (bf16_bits(d)[~valid] == SENTINEL).all()
        assert_parity(bf16_f64(d)[valid], ref[valid], f"permutation {perm}")


def test_workspaces_for_many_streams(lib):
    # more streams than the library keeps workspaces for (16): the cache is released and
    # rebuilt; the stream-K shape below uses the workspace on every call, and every stream
    # computes the same bits (stream-K sums its partials in a fixed order)
    p = W.make_dense(256, 384, 1152, seed=55)
    a, sfa, b, sfb = dev(p.a), dev(p.sfa), dev(p.b), dev(p.sfb)
    outs = []
    for s in [torch.cuda.Stream() for _ in range(24)]:
        d = sentinel_like((p.M, p.N))
        with torch.cuda.stream(s):
            lib.dg_fp8_gemm_nt(a, sfa, b, sfb, None, d)
        outs.append(d)
    torch.cuda.synchronize()
    first = bf16_bits(outs[0])
    for i, d in enumerate(outs[1:]):
        assert np.array_equal(bf16_bits(d), first), f"stream {i + 1}"
    assert_parity(bf16_f64(outs[0]), O.fp8_gemm_nt(p.a, p.sfa, p.b, p.sfb, None, p.M, p.N, p.K), "many streams")
