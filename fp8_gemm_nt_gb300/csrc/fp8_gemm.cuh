// Persistent, warp-specialised fine-grained-scaled FP8 GEMM for sm_103a.
//
//   D = C + A @ B.T, A: E4M3 [rows, K] (one UE8M0 scale per row per 128-K group),
//   B: E4M3 [N, K] (one UE8M0 scale per 128x128 block), FP32 accumulation in TMEM,
//   BF16 output. Operation and scale format: DeepGEMM README ("Interfaces / Notices",
//   "Normal dense GEMMs", "Grouped GEMMs (contiguous layout)", "Grouped GEMMs (masked
//   layout)") as reproduced on the page "Weight gradient kernels for dense and MoE
//   models #95".
//
// One CTA per SM walks a sequence of *segments*: a segment is one 128 x BN output tile
// and a range of its K-groups. In tile mode every segment is a whole tile (K-groups
// 0..KG-1), tiles dealt round-robin to the CTAs. In stream-K mode (dense form, used
// when there are fewer tiles than SMs) the flattened (tile, K-group) space is cut into
// one equal contiguous range per CTA; a tile covered by several CTAs is finished by
// the last of them to arrive, which sums the FP32 partials of all contributors in a
// fixed order (so the result does not depend on arrival order) from a workspace.
//
// Roles:
//   warp 0       TMA producer: A tile (128 x 128 B), B tile (BN x 128 B) and, at the
//                first K-group of a segment and every fourth K-group, the packed scale
//                words, into a kStages-deep ring.
//   warp 1       MMA warp: rearranges the scale words into the tcgen05.cp source layout,
//                copies them into TMEM, and one elected thread issues
//                tcgen05.mma.kind::mxf8f6f4.block_scale (K = 32 per instruction, four per
//                K-group, all four reading the group's scale byte via the scale-factor id).
//   warps 2..    epilogue: TMEM -> registers (+C) -> BF16 -> swizzled smem -> TMA store,
//                or predicated row stores for tiles that hold padding / masked rows, or
//                (stream-K) FP32 partials to the workspace and the last-arriver reduction.
// The accumulator is double-buffered in TMEM (kNumAccum = 2) so the epilogue of one
// segment overlaps the main loop of the next.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace dg {

// KGrouped: the K-grouped weight-gradient form (expert g owns a K-slice; FP32 output per expert)
enum class Kind : int { Dense = 0, Contiguous = 1, Masked = 2, KGrouped = 3 };

// Device status bits: bit (1 << s) for dg_status s.
enum : uint32_t { kStatusTimeoutBit = 1u << 5, kStatusBadIndexBit = 1u << 6 };

// Fault injection for the failure-detection tests (host-side switch, default off).
enum : int { kFaultNone = 0, kFaultProducerSilent = 1 };

constexpr int BLOCK_M = 128;
constexpr int BLOCK_K = 128;   // one scale group per pipeline stage
constexpr int SF_BLOCK_N = 128;
constexpr int kPrefetchKGroups = 4;   // K-groups of the first segment prefetched into L2 at launch
constexpr int kMaskCountCache = 1024;   // masked form: group counts cached in shared memory (more: read at L2)

__host__ __device__ constexpr int count_cache_for(Kind k) { return k == Kind::Masked ? kMaskCountCache : 0; }

struct Params {
  int M;   // dense: M; contiguous: M_total; masked: max_m (rows per group)
  int N;
  int K;
  int G;
  const int32_t* m_indices;       // contiguous: expert of each row, -1 = padding
  union {
    const int32_t* masked_m;      // masked: valid rows per group (device)
    const int* pair_count;        // CTA-pair kernel, contiguous form: number of listed pair rows
  };
  const __nv_bfloat16* c;         // dense: optional addend [M, N]
  __nv_bfloat16* d;               // output (used by the predicated store path)
  uint32_t* status;               // device status word
  unsigned long long timeout_ns;  // bound on every pipeline wait
  // stream-K (dense only); sk_ctas == 0 selects tile mode
  int sk_ctas;                    // number of CTAs sharing the K-group space (== gridDim.x)
  int sk_slots;                   // partial slots per tile in the workspace
  float* sk_ws;                   // [tiles][sk_slots][128 * BN] FP32 partials
  int* sk_counters;               // [tiles][epilogue warps], zero between launches
  int fault;                      // kFault*
  // CTA-pair kernel: row counts of the tcgen05.cp-layout scale chunk tensors
  int sf_num_mb;                  // 128-row blocks of A per K-quad
  int sf_nb;                      // B chunk rows per (group, K-quad): two per tile
  // K-grouped form: K-slice length of each expert (device, multiples of 128) and the number
  // of packed scale-word rows (the scales of each expert start a new word row). The CTA-pair
  // kernel's contiguous form instead reads its pair rows, listed per call ({first block,
  // expert, own blocks} each), from the same slot (the two forms never meet; keeping the
  // parameter block small keeps every kernel within its register budget).
  union {
    const int32_t* ks;
    const int* pair_list;
  };
  int sf_k_rows;
};

__host__ __device__ constexpr int ceil_div_c(int a, int b) { return (a + b - 1) / b; }

// kKG = K-groups per pipeline stage (1 or 2). Two K-groups per stage double the bytes
// each TMA round trip moves; on GB300 a single producer thread streams markedly more from
// HBM with 64 KB stages than with 32 KB ones (measured 5.2 vs 4.1 TB/s in a TMA-only
// probe with the decode shape's A and B boxes), which is what the HBM-bound shapes need.
//
// kSplit > 0 (dense only): split-K over a cluster of kSplit CTAs. Each cluster computes one
// tile, CTA r of the cluster K-groups [r, r+1) * K / kSplit of it; the FP32 partials meet
// in shared memory and CTA r sums (in rank order) and stores columns [r, r+1) * BN / kSplit.
//
// kBF4: B is FP4 (E2M1, two per byte) with one UE8M0 scale per row per 32 K. A TMA load of
// the 16U4_ALIGN16B type spreads each 8 bytes of B over a 16-byte shared-memory chunk (the
// upper 8 bytes zero), which is the layout tcgen05.mma reads an E2M1 operand in, so the B
// stage has the FP8 shape (BN rows x 128 bytes per K-group) while the transaction count is
// the global bytes read (BN x 64 per K-group; measured on GB300). Every stage then carries
// the scale words: A's packed word per row (as in FP8) and, per K-group, one word per B row
// holding the scales of its four 32-wide blocks.
// kCountCache: per-group row counts (the masked form's device-side counts) held in shared
// memory, read once per CTA, so that the schedule walk of every role reads them there.
template <int BN, int kStages, int kNumAccum, int kEpiWarps, int kEpiBufs, int kKG = 1, int kSplit = 0,
          bool kBF4 = false, int kCountCache = 0>
struct Config {
  static_assert(kKG == 1 || kKG == 2, "one or two K-groups per stage");
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN must be a multiple of 32 in [64, 256]");
  static_assert(kEpiWarps == 4 || kEpiWarps == 8, "epilogue uses 4 or 8 warps");
  static constexpr int kSfWarp = 2 + kEpiWarps;                 // rearranges the scale words
  static constexpr int kThreads = (3 + kEpiWarps) * 32;
  static constexpr int kColsPerEpiWarp = BN / (kEpiWarps / 4);
  static_assert(kSplit > 0 || kColsPerEpiWarp % 64 == 0, "each epilogue warp stores whole 64-column chunks");
  static_assert(kSplit == 0 || (kEpiWarps == 4 && kNumAccum == 1 && (BN / kSplit) % 8 == 0),
                "split-K: 4 epilogue warps, one accumulator, 8-column slices");

  // shared memory (offsets from a 1024-byte-aligned base)
  static constexpr int A_SUB = BLOCK_M * BLOCK_K;               // one K-group of A
  static constexpr int B_SUB = BN * BLOCK_K;                    // one K-group of B
  static constexpr int A_BYTES = kKG * A_SUB;                   // per stage
  static constexpr int B_BYTES = kKG * B_SUB;
  static constexpr int B_TX = kBF4 ? B_BYTES / 2 : B_BYTES;     // global bytes of a stage's B boxes
  static constexpr int SFB_CHUNKS = ceil_div_c(BN, 128);        // 128-row chunks of B scale rows
  static constexpr int SFB_SETS = kBF4 ? kKG : 1;               // B scale sets in TMEM per scale stage
  static constexpr int SF_RAW_B_BYTES = kBF4 ? BN * 4 * kKG : 8 * 4;   // FP4: BN row words per K-group
  static constexpr int SF_RAW_A = 0;                            // 128 words as loaded (row-major)
  static constexpr int SF_RAW_B = 512;                          // B words as loaded
  static constexpr int SF_UT_A = 512 + ceil_div_c(SF_RAW_B_BYTES > 512 ? SF_RAW_B_BYTES : 512, 128) * 128;
  static constexpr int SF_UT_B = SF_UT_A + 512;                 // SFB_SETS x SFB_CHUNKS x (32 rows x 16 B)
  static constexpr int SF_BYTES = SF_UT_B + SFB_SETS * SFB_CHUNKS * 512;
  static constexpr int SF_TX_BYTES = BLOCK_M * 4 + SF_RAW_B_BYTES;   // SFA box {128,1} + SFB box
  static constexpr int EPI_BUF_BYTES = 32 * 128;                // 32 rows x 64 BF16 columns
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + kStages * A_BYTES;
  static constexpr int OFF_SF = OFF_B + kStages * B_BYTES;
  static constexpr int OFF_EPI = ((OFF_SF + kStages * SF_BYTES + 1023) / 1024) * 1024;
  static constexpr int OFF_BAR = OFF_EPI + kEpiWarps * kEpiBufs * EPI_BUF_BYTES;
  static constexpr int NUM_BARS = 3 * kStages + 2 * kNumAccum + 1;   // + scale-ready per stage
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_COUNTS = OFF_MISC + 16;
  static constexpr int SMEM_BYTES = OFF_COUNTS + 4 * kCountCache + 1024;   // + slack for manual alignment
  static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");

  // tensor memory columns
  static constexpr int ACC_COLS = kNumAccum * BN;
  static constexpr int SFA_COL = ACC_COLS;                      // 2 buffers x 4 columns
  static constexpr int SFB_COL = SFA_COL + 8;                   // 2 buffers x SFB_SETS x 4*SFB_CHUNKS columns
  static constexpr int TMEM_USED = SFB_COL + 2 * SFB_SETS * 4 * SFB_CHUNKS;
  static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64 : TMEM_USED <= 128 ? 128
                                 : TMEM_USED <= 256 ? 256 : 512;
  static_assert(TMEM_USED <= 512, "TMEM budget exceeded");

  // stream-K partial layout: per epilogue warp a 32-row x kColsPerEpiWarp block of float4,
  // float4 (c4, lane) at index c4 * 32 + lane (a warp's 32 lanes write 512 contiguous bytes)
  static constexpr int SK_TILE_FLOATS = BLOCK_M * BN;
  static constexpr int SK_WARP_FLOATS = 32 * kColsPerEpiWarp;
  // split-K: this CTA's FP32 partial, float4 (c4, row) at byte (c4 * 128 + row) * 16, in the
  // ring's shared memory (idle once the CTA's only tile is accumulated)
  static_assert(kSplit == 0 || BN * BLOCK_M * 4 <= OFF_EPI - OFF_A, "split-K partial exceeds the ring");
};

// ------------------------------------------------------------------------------------
// Segment scheduler: every role of a CTA walks the same sequence of segments.
// ------------------------------------------------------------------------------------
struct Segment {
  int g;          // expert (grouped forms), 0 for dense
  int m_blk;      // 128-row block (within the group for the masked form)
  int n_blk;
  int valid_m;    // masked: rows of the group that are valid (clamped count)
  int tile;       // linear tile index (stream-K workspace / counters)
  int kb_begin;   // K-groups [kb_begin, kb_end) of the tile
  int kb_end;
  int n_contrib;  // CTAs contributing to this tile (1 = this segment is the whole tile)
  int slot;       // this CTA's position among them
  bool cta_last;  // stream-K: no further segment for this CTA (its ring smem is free afterwards)
  int k_base;     // K-grouped: first K-group of the expert's slice (0 otherwise)
  int sf_row;     // K-grouped: first packed scale-word row of the expert (0 otherwise)
};

template <Kind kKind, int BN, int kKG = 1, int kSplit = 0>
struct Scheduler {
  int num_n, num_m, total, num_kb, num_kc;   // num_kc: stream-K units (kKG K-groups) per tile
  int g_cur, g_start, g_tiles;   // masked: incremental walk over groups
  int kbase_cur, sfrow_cur;      // K-grouped: K-group and scale-row offsets of expert g_cur
  int t;                         // tile mode: next tile index
  long long u, u_end, U;         // stream-K: this CTA's K-group range, total K-groups
  bool stream_k;
  const int* counts;             // masked: the group counts cached in shared memory (or null)

  __device__ __forceinline__ int raw_mask(const Params& p, int g) const {
    return (counts != nullptr && g < kMaskCountCache) ? counts[g] : ld_cg_s32(p.masked_m + g);
  }

  __device__ __forceinline__ int clamped_mask(const Params& p, int g) const {
    const int m = raw_mask(p, g);
    return m < 0 ? 0 : (m > p.M ? p.M : m);
  }

  __device__ __forceinline__ explicit Scheduler(const Params& p, const int* cached_counts = nullptr) {
    counts = cached_counts;
    num_n = ceil_div_c(p.N, BN);
    num_m = ceil_div_c(p.M, BLOCK_M);
    num_kb = p.K / BLOCK_K;
    num_kc = ceil_div_c(num_kb, kKG);
    g_cur = 0;
    g_start = 0;
    g_tiles = 0;
    t = blockIdx.x;
    kbase_cur = 0;
    sfrow_cur = 0;
    stream_k = false;
    u = u_end = U = 0;
    if constexpr (kSplit > 0) {
      // one tile per cluster; this CTA takes its rank's share of the tile's K units
      total = num_m * num_n;
      t = static_cast<int>(blockIdx.x) / kSplit;
      const int r = static_cast<int>(blockIdx.x) % kSplit;
      u = static_cast<long long>(r) * num_kc / kSplit;
      u_end = static_cast<long long>(r + 1) * num_kc / kSplit;
      return;
    }
    if constexpr (kKind == Kind::KGrouped) {
      total = p.G * num_m * num_n;
      if (blockIdx.x == 0 && threadIdx.x == 0) {
        // every slice a non-negative multiple of 128, the slices covering K, the scale rows
        // matching the per-expert packing; otherwise the layout is violated (reported)
        long long kg_sum = 0, rows = 0;
        bool bad = false;
        for (int g = 0; g < p.G; ++g) {
          const int k = ld_cg_s32(p.ks + g);
          if (k < 0 || k % BLOCK_K != 0) bad = true;
          if (k > 0) {
            kg_sum += k / BLOCK_K;
            rows += (k + 4 * BLOCK_K - 1) / (4 * BLOCK_K);
          }
        }
        if (bad || kg_sum != num_kb || rows != p.sf_k_rows) atomicOr(p.status, kStatusBadIndexBit);
      }
      return;
    }
    if constexpr (kKind == Kind::Masked) {
      total = 0;
      for (int g = 0; g < p.G; ++g) total += ceil_div_c(clamped_mask(p, g), BLOCK_M) * num_n;
      g_tiles = p.G > 0 ? ceil_div_c(clamped_mask(p, 0), BLOCK_M) * num_n : 0;
      if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (int g = 0; g < p.G; ++g) {
          const int m = raw_mask(p, g);
          if (m < 0 || m > p.M) atomicOr(p.status, kStatusBadIndexBit);
        }
      }
    } else {
      total = num_m * num_n;
      if constexpr (kKind == Kind::Dense) {
        if (p.sk_ctas > 0) {
          stream_k = true;
          U = static_cast<long long>(total) * num_kc;
          u = static_cast<long long>(blockIdx.x) * U / p.sk_ctas;
          u_end = static_cast<long long>(blockIdx.x + 1) * U / p.sk_ctas;
        }
      }
    }
  }

  // CTA whose unit range contains flattened unit index v (a unit is kKG K-groups).
  __device__ __forceinline__ int sk_owner(const Params& p, long long v) const {
    return static_cast<int>(((v + 1) * p.sk_ctas - 1) / U);
  }

  // Next segment of this CTA; false when there is none left. Contiguous padding blocks
  // are skipped here (every role skips the same ones).
  __device__ __forceinline__ bool next(const Params& p, Segment& s) {
    s.k_base = 0;
    s.sf_row = 0;
    if constexpr (kKind == Kind::KGrouped) {
      if (t >= total) return false;
      const int cur = t;
      t += gridDim.x;
      const int tpg = num_m * num_n;
      const int g = cur / tpg;
      while (g_cur < g) {   // experts are visited in increasing order
        const int k = ld_cg_s32(p.ks + g_cur);
        if (k > 0) {
          kbase_cur += k / BLOCK_K;
          sfrow_cur += (k + 4 * BLOCK_K - 1) / (4 * BLOCK_K);
        }
        ++g_cur;
      }
      const int local = cur - g * tpg;
      const int k = ld_cg_s32(p.ks + g);
      s.tile = cur;
      s.g = g;
      s.m_blk = local / num_n;
      s.n_blk = local % num_n;
      s.valid_m = p.M;
      s.kb_begin = 0;
      s.kb_end = k > 0 ? k / BLOCK_K : 0;   // 0: an expert without tokens (D = C)
      s.k_base = kbase_cur;
      s.sf_row = sfrow_cur;
      s.n_contrib = 1;
      s.slot = 0;
      s.cta_last = false;
      return true;
    }
    if constexpr (kSplit > 0) {
      if (t >= total || u >= u_end) return false;
      s.tile = t;
      s.m_blk = t / num_n;
      s.n_blk = t % num_n;
      s.g = 0;
      s.valid_m = p.M;
      s.kb_begin = static_cast<int>(u) * kKG;
      s.kb_end = static_cast<int>(u_end) * kKG < num_kb ? static_cast<int>(u_end) * kKG : num_kb;
      s.n_contrib = kSplit;
      s.slot = static_cast<int>(blockIdx.x) % kSplit;
      s.cta_last = true;
      t = total;   // a single segment
      return true;
    }
    if (stream_k) {
      if (u >= u_end) return false;
      const int tile = static_cast<int>(u / num_kc);
      s.tile = tile;
      s.m_blk = tile / num_n;
      s.n_blk = tile % num_n;
      s.g = 0;
      s.valid_m = p.M;
      const int kc_begin = static_cast<int>(u - static_cast<long long>(tile) * num_kc);
      const long long left = u_end - u;
      const int kc_end = static_cast<int>(left < num_kc - kc_begin ? kc_begin + left : num_kc);
      s.kb_begin = kc_begin * kKG;
      s.kb_end = kc_end * kKG < num_kb ? kc_end * kKG : num_kb;
      const int first = sk_owner(p, static_cast<long long>(tile) * num_kc);
      const int last = sk_owner(p, static_cast<long long>(tile) * num_kc + num_kc - 1);
      s.n_contrib = last - first + 1;
      s.slot = static_cast<int>(blockIdx.x) - first;
      u += kc_end - kc_begin;
      s.cta_last = u >= u_end;
      return true;
    }
    while (t < total) {
      const int cur = t;
      t += gridDim.x;
      s.tile = cur;
      s.kb_begin = 0;
      s.kb_end = num_kb;
      s.n_contrib = 1;
      s.slot = 0;
      s.cta_last = false;
      if constexpr (kKind == Kind::Masked) {
        while (cur >= g_start + g_tiles && g_cur + 1 < p.G) {
          g_start += g_tiles;
          ++g_cur;
          g_tiles = ceil_div_c(clamped_mask(p, g_cur), BLOCK_M) * num_n;
        }
        const int local = cur - g_start;
        s.g = g_cur;
        s.m_blk = local / num_n;
        s.n_blk = local % num_n;
        s.valid_m = clamped_mask(p, g_cur);
        return true;
      } else {
        s.m_blk = cur / num_n;
        s.n_blk = cur % num_n;
        s.valid_m = p.M;
        s.g = 0;
        if constexpr (kKind == Kind::Contiguous) {
          const int g = ld_cg_s32(p.m_indices + s.m_blk * BLOCK_M);
          if (g < 0 || g >= p.G) {
            // a block led by an out-of-range index is reported once (by its n = 0 tile)
            if ((g < -1 || g >= p.G) && s.n_blk == 0 && threadIdx.x == 64) atomicOr(p.status, kStatusBadIndexBit);
            continue;
          }
          s.g = g;
        }
        return true;
      }
    }
    return false;
  }
};

// Warp-uniform bounded wait: every lane polls, and the warp proceeds only if all lanes
// saw the phase complete and no other role has aborted.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                          volatile uint32_t* abort_flag) {
  const bool ok = (*abort_flag == 0) && mbar_wait(bar, parity, timeout_ns);
  return __all_sync(0xffffffffu, ok);
}

// C of one output chunk (32 rows x 128 bytes: 64 BF16 or 32 FP32 columns) into a warp's
// staging buffer, in the layout the output staging uses (row r's 16-byte piece j at
// r * 128 + (j ^ (r & 7)) * 16). The warp loads it together, four 128-byte rows per
// instruction (a lane per row would touch 32 lines per instruction), at L2. c0 points at
// lane 0's row and the chunk's first column; rows whose bit in ok_mask is clear and pieces
// at or past `cols` elements (or past `pieces`) read as zero.
template <typename T, int kPieces = 8>
__device__ __forceinline__ void warp_stage_c(uint32_t sbuf, const T* c0, long long ld, uint32_t ok_mask, int cols,
                                             uint32_t lane) {
  constexpr int kPer = 16 / static_cast<int>(sizeof(T));   // elements per 16-byte piece
#pragma unroll
  for (int half = 0; half < 2; ++half) {   // two rounds of four loads in flight (register budget)
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = (4 * half + i) * 32 + static_cast<int>(lane);
      const int r = idx >> 3, j = idx & 7;
      v[i] = make_uint4(0u, 0u, 0u, 0u);
      if (j < kPieces && ((ok_mask >> r) & 1u) && kPer * j < cols) v[i] = ld_cg_v4(c0 + r * ld + kPer * j);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = (4 * half + i) * 32 + static_cast<int>(lane);
      const int r = idx >> 3, j = idx & 7;
      if (j < kPieces) st_shared_v4(sbuf + r * 128 + ((j ^ (r & 7)) * 16), v[i].x, v[i].y, v[i].z, v[i].w);
    }
  }
}

__device__ __forceinline__ void st_global_v4f(float* p, float a, float b, float c, float d) {
  asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

__device__ __forceinline__ float4 ld_global_cg_v4f(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// kOutF32: C and D are FP32 (the weight-gradient form, D = C + A @ B.T accumulated in FP32);
// otherwise BF16. kAMN / kBMN: A given as [K, M] / B given as [K, N] (M- / N-major: the
// "t" A and "n" B layouts of fp8_gemm_{nn,tn,tt}); otherwise K-major [M, K] / [N, K].
// An MN-major operand arrives as 128 x 128-byte boxes (128 K-rows of 128 M/N-bytes, 128-byte
// swizzle) stacked along M/N every 16 KB; its smem descriptor takes LBO = 16 KB (stride
// between 128-byte atoms along M/N) and SBO = 1024 (stride between 8-row groups along K),
// and each 32-deep K step of the MMA advances it by 32 rows = 4 KB.
template <Kind kKind, int BN, int kStages, int kNumAccum, int kEpiWarps, int kEpiBufs, bool kHasC, int kKG = 1,
          int kSplit = 0, bool kOutF32 = false, bool kAMN = false, bool kBMN = false, bool kBF4 = false>
__global__ void __launch_bounds__(
    Config<BN, kStages, kNumAccum, kEpiWarps, kEpiBufs, kKG, kSplit, kBF4, count_cache_for(kKind)>::kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_sfa, const __grid_constant__ CUtensorMap tm_sfb,
                    const __grid_constant__ CUtensorMap tm_d, const Params p) {
  using C = Config<BN, kStages, kNumAccum, kEpiWarps, kEpiBufs, kKG, kSplit, kBF4, count_cache_for(kKind)>;
  static_assert(!kBF4 || (!kAMN && !kBMN && !kOutF32 && kKind != Kind::KGrouped),
                "FP4 B: K-major operands, BF16 output, dense / contiguous / masked forms");
  static_assert(kSplit == 0 || kKind == Kind::Dense, "split-K clusters: dense form only");
  static_assert(!kOutF32 || ((kKind == Kind::Dense || kKind == Kind::KGrouped) && kSplit == 0),
                "FP32 output: dense (tile mode / stream-K) and K-grouped forms only");
  static_assert(kKind != Kind::KGrouped || (kOutF32 && kKG == 1), "the K-grouped form writes FP32, one K-group per stage");
  static_assert((!kAMN && !kBMN) ||
                    (kSplit == 0 && ((kKind == Kind::Dense && !kOutF32) || (kKind == Kind::Contiguous && !kAMN && !kOutF32) ||
                                     (kKind == Kind::KGrouped && kOutF32))),
                "MN-major operands: dense (BF16), contiguous N-major B (BF16), K-grouped (FP32)");
  static_assert(!kBMN || BN % 128 == 0, "an N-major B tile is whole 128-column atoms");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + kStages;
  uint64_t* tfull_bar = bars + 2 * kStages;
  uint64_t* tempty_bar = bars + 2 * kStages + kNumAccum;
  uint64_t* drain_bar = bars + 2 * kStages + 2 * kNumAccum;
  // scale words of a stage rearranged by the scale warp (used on scale stages only)
  uint64_t* sf_ready_bar = bars + 2 * kStages + 2 * kNumAccum + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x / 32;
  const uint32_t lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 2);   // the MMA commit and the scale warp
    }
    for (int a = 0; a < kNumAccum; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    for (int s = 0; s < kStages; ++s) mbar_init(&sf_ready_bar[s], 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_sfa);
    tma_prefetch_desc(&tm_sfb);
    tma_prefetch_desc(&tm_d);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // With programmatic dependent launch this kernel may start while the previous one in the
  // stream is finishing: everything above overlapped it; nothing below may read or write
  // global memory before that grid has completed. The one exception: the dense forms ask L2
  // for the first K-groups of their first segment's A and B boxes now. A prefetch into L2
  // returns nothing to this SM and L2 is the point of coherence, so a load issued after
  // the wait still sees any write the previous grid makes to those bytes.
  if constexpr (kKind == Kind::Dense) {
    if (warp == 0 && lane == 0) {
      Scheduler<kKind, BN, kKG, kSplit> first(p);   // the dense schedule reads no global memory
      Segment s0;
      if (first.next(p, s0)) {
        const int kb_end = s0.kb_begin + kPrefetchKGroups < s0.kb_end ? s0.kb_begin + kPrefetchKGroups : s0.kb_end;
        for (int kb = s0.kb_begin; kb < kb_end; ++kb) {
          if constexpr (kAMN) {
            tma_prefetch_l2_2d(&tm_a, s0.m_blk * BLOCK_M, kb * BLOCK_K);
          } else {
            tma_prefetch_l2_2d(&tm_a, kb * BLOCK_K, s0.m_blk * BLOCK_M);
          }
          if constexpr (kBMN) {
#pragma unroll
            for (int h = 0; h < BN / 128; ++h) tma_prefetch_l2_2d(&tm_b, s0.n_blk * BN + 128 * h, kb * BLOCK_K);
          } else {
            tma_prefetch_l2_2d(&tm_b, kb * BLOCK_K, s0.n_blk * BN);
          }
        }
      }
    }
  }
  grid_dependency_wait();

  auto on_timeout = [&]() {
    atomicOr(p.status, kStatusTimeoutBit);
    *abort_flag = 1;
  };

  const int* cached_counts = nullptr;
  if constexpr (kKind == Kind::Masked) {
    // the group counts, read once at L2 (they may come from the previous kernel) into
    // shared memory for every role's schedule walk
    int* cache = reinterpret_cast<int*>(smem + C::OFF_COUNTS);
    const int n = p.G < kMaskCountCache ? p.G : kMaskCountCache;
    for (int i = threadIdx.x; i < n; i += blockDim.x) cache[i] = ld_cg_s32(p.masked_m + i);
    __syncthreads();
    cached_counts = cache;
  }
  Scheduler<kKind, BN, kKG, kSplit> sched(p, cached_counts);
  Segment seg;

  if (warp == 0) {
    // ================================ TMA producer ================================
    if (lane == 0 && p.fault != kFaultProducerSilent) {
      uint32_t stage = 0, phase = 0, issued = 0;
      while (sched.next(p, seg)) {
        const int row0 = seg.m_blk * BLOCK_M;
        const int n0 = seg.n_blk * BN;
        const int sfb_x = (n0 / SF_BLOCK_N) & ~3;   // 16-byte aligned start of the block-scale window
        for (int kb = seg.kb_begin; kb < seg.kb_end; kb += kKG) {
          if (*abort_flag || !mbar_wait(&empty_bar[stage], phase ^ 1, p.timeout_ns)) {
            on_timeout();
            goto producer_done;
          }
          const bool with_sf = kBF4 || kb == seg.kb_begin || (kb % 4) == 0;
          uint64_t* fb = &full_bar[stage];
          mbar_arrive_expect_tx(fb, C::A_BYTES + C::B_TX + (with_sf ? C::SF_TX_BYTES : 0));
          uint8_t* sa = smem + C::OFF_A + stage * C::A_BYTES;
          uint8_t* sb = smem + C::OFF_B + stage * C::B_BYTES;
          uint8_t* ssf = smem + C::OFF_SF + stage * C::SF_BYTES;
          // (with two K-groups per stage, a second K-group past K reads zeros)
#pragma unroll
          for (int j = 0; j < kKG; ++j) {
            if constexpr (kKind == Kind::Masked) {
              tma_load_3d(sa + j * C::A_SUB, &tm_a, fb, (kb + j) * BLOCK_K, row0, seg.g);
            } else if constexpr (kAMN) {
              tma_load_2d(sa + j * C::A_SUB, &tm_a, fb, row0, (seg.k_base + kb + j) * BLOCK_K);
            } else {
              tma_load_2d(sa + j * C::A_SUB, &tm_a, fb, (seg.k_base + kb + j) * BLOCK_K, row0);
            }
            if constexpr (kBMN) {
#pragma unroll
              for (int h = 0; h < BN / 128; ++h) {
                if constexpr (kKind == Kind::Contiguous) {
                  tma_load_3d(sb + j * C::B_SUB + h * (128 * BLOCK_K), &tm_b, fb, n0 + 128 * h, (kb + j) * BLOCK_K,
                              seg.g);
                } else {
                  tma_load_2d(sb + j * C::B_SUB + h * (128 * BLOCK_K), &tm_b, fb, n0 + 128 * h,
                              (seg.k_base + kb + j) * BLOCK_K);
                }
              }
            } else if constexpr (kKind == Kind::Dense || kKind == Kind::KGrouped) {
              tma_load_2d(sb + j * C::B_SUB, &tm_b, fb, (seg.k_base + kb + j) * BLOCK_K, n0);
            } else {
              tma_load_3d(sb + j * C::B_SUB, &tm_b, fb, (kb + j) * BLOCK_K, n0, seg.g);
            }
          }
          if (with_sf) {
            if constexpr (kKind == Kind::Masked) {
              tma_load_3d(ssf + C::SF_RAW_A, &tm_sfa, fb, row0, kb / 4, seg.g);
            } else {
              tma_load_2d(ssf + C::SF_RAW_A, &tm_sfa, fb, row0, seg.sf_row + kb / 4);
            }
            if constexpr (kBF4) {
              // kKG rows (K-groups) of BN per-row words
              if constexpr (kKind == Kind::Dense) {
                tma_load_2d(ssf + C::SF_RAW_B, &tm_sfb, fb, n0, kb);
              } else {
                tma_load_3d(ssf + C::SF_RAW_B, &tm_sfb, fb, n0, kb, seg.g);
              }
            } else if constexpr (kKind == Kind::Dense || kKind == Kind::KGrouped) {
              tma_load_2d(ssf + C::SF_RAW_B, &tm_sfb, fb, sfb_x, seg.sf_row + kb / 4);
            } else {
              tma_load_3d(ssf + C::SF_RAW_B, &tm_sfb, fb, sfb_x, kb / 4, seg.g);
            }
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    producer_done:
      grid_launch_dependents();   // every load of this CTA is issued: the next grid may be scheduled
      // No TMA write may still be landing in this CTA's shared memory at exit: wait for
      // the last use of every stage (already consumed on the normal path).
      for (uint32_t s = 0; s < kStages && s < issued; ++s) {
        const uint32_t last_use = (issued - 1 - s) / kStages;
        mbar_wait(&full_bar[s], last_use & 1, 50000000ull);
      }
    }
  } else if (warp == 1) {
    // ================================ MMA issuer ==================================
    // A single thread runs the whole loop: waits, scale copies into TMEM, four MMAs per
    // K-group and the commits, with no warp-wide synchronisation per K-group (measured on
    // GB300: each tcgen05.mma issue costs ~75 cycles and a warp-wide wait path ~400, so the
    // loop, not the tensor pipe, set the pace).
    if (lane == 0) {
      // B format field [10,13): 0 = E4M3, 5 = E2M1
      constexpr uint32_t kIdesc = make_idesc_mxf8_e4m3(BLOCK_M, BN) | (kAMN ? 1u << 15 : 0u) |
                                  (kBMN ? 1u << 16 : 0u) | (kBF4 ? 5u << 10 : 0u);
      const uint64_t a_desc0 =
          make_smem_desc(smem_addr(smem + C::OFF_A), kAMN ? 128 * BLOCK_K : 16, 1024, kLayoutSwizzle128B);
      const uint64_t b_desc0 =
          make_smem_desc(smem_addr(smem + C::OFF_B), kBMN ? 128 * BLOCK_K : 16, 1024, kLayoutSwizzle128B);
      // descriptor steps (address >> 4) per 32-deep K step: 32 bytes along a K-major row, or
      // 32 rows of 128 bytes down an MN-major box
      constexpr uint64_t kAStep = kAMN ? (32 * 128) >> 4 : 2;
      constexpr uint64_t kBStep = kBMN ? (32 * 128) >> 4 : 2;
      const uint64_t sf_desc0 = make_smem_desc(smem_addr(smem + C::OFF_SF), 0, 128, kLayoutNone);
      uint32_t stage = 0, phase = 0, seg_iter = 0, sf_iter = 0, sf_parity = 0;
      while (sched.next(p, seg)) {
        const uint32_t acc = seg_iter % kNumAccum;
        const uint32_t acc_phase = (seg_iter / kNumAccum) & 1;
        if (*abort_flag || !mbar_wait(&tempty_bar[acc], acc_phase ^ 1, p.timeout_ns)) {
          on_timeout();
          goto mma_done;
        }
        tc_fence_after();
        {
          const uint32_t d_tmem = tmem_base + acc * BN;
          uint32_t sfa_tmem = 0, sfb_tmem = 0;
          for (int kb = seg.kb_begin; kb < seg.kb_end; kb += kKG) {
            if (!mbar_wait(&full_bar[stage], phase, p.timeout_ns)) {
              on_timeout();
              goto mma_done;
            }
            if (kBF4 || kb == seg.kb_begin || kb % 4 == 0) {
              // the scale warp has rearranged this stage's scale words for tcgen05.cp
              if (!mbar_wait(&sf_ready_bar[stage], (sf_parity >> stage) & 1u, p.timeout_ns)) {
                on_timeout();
                goto mma_done;
              }
              sf_parity ^= 1u << stage;
              tc_fence_after();
              const uint32_t buf = sf_iter & 1;
              ++sf_iter;
              sfa_tmem = tmem_base + C::SFA_COL + 4 * buf;
              sfb_tmem = tmem_base + C::SFB_COL + 4 * C::SFB_SETS * C::SFB_CHUNKS * buf;
              const uint64_t sf_desc = sf_desc0 + ((stage * C::SF_BYTES) >> 4);
              tmem_copy_32x128b_warpx4(sfa_tmem, sf_desc + (C::SF_UT_A >> 4));
#pragma unroll
              for (int ch = 0; ch < C::SFB_SETS * C::SFB_CHUNKS; ++ch)
                tmem_copy_32x128b_warpx4(sfb_tmem + 4 * ch, sf_desc + ((C::SF_UT_B + 512 * ch) >> 4));
            } else {
              tc_fence_after();
            }
            // descriptor address field is (address >> 4): stage and 32-byte K steps add to it
#pragma unroll
            for (int j = 0; j < kKG; ++j) {
              if (kb + j < seg.kb_end) {
                const uint64_t adesc = a_desc0 + ((stage * C::A_BYTES + j * C::A_SUB) >> 4);
                const uint64_t bdesc = b_desc0 + ((stage * C::B_BYTES + j * C::B_SUB) >> 4);
#pragma unroll
                for (int k = 0; k < BLOCK_K / 32; ++k) {
                  // A: byte (kb + j) % 4 of its packed word; B (FP8): the same byte of the block
                  // word, (FP4): byte k of K-group j's row word (the k-th 32-wide block)
                  const uint32_t idesc = idesc_with_sf_id(kIdesc, (kb + j) % 4, kBF4 ? k : (kb + j) % 4);
                  mma_mxf8_block_scale(d_tmem, adesc + kAStep * k, bdesc + kBStep * k, idesc, sfa_tmem,
                                       sfb_tmem + (kBF4 ? 4 * C::SFB_CHUNKS * j : 0),
                                       (kb + j != seg.kb_begin || k != 0) ? 1u : 0u);
                }
              }
            }
            tc_commit(&empty_bar[stage]);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
        tc_commit(&tfull_bar[acc]);
        ++seg_iter;
      }
    mma_done:
      // Every MMA / copy issued above must have finished before TMEM is released.
      tc_commit(drain_bar);
      mbar_wait(drain_bar, 0, 50000000ull);
    }
    __syncwarp();
  } else if (warp == C::kSfWarp) {
    // ================================ scale warp ==================================
    // Walks every stage in order. On a stage that carries scale words it rearranges them
    // into the tcgen05.cp source layout (row r holds, in word c, the word of tile row
    // 32c + r; B's per-block words replicated per row) and signals the MMA thread. It is the
    // second arrival on every stage's empty barrier, so the producer cannot refill a stage
    // this warp has not seen: its parity waits can never alias a later phase.
    uint32_t stage = 0, phase = 0;
    while (sched.next(p, seg)) {
      const int n0 = seg.n_blk * BN;
      const int sfb_x = (n0 / SF_BLOCK_N) & ~3;
      for (int kb = seg.kb_begin; kb < seg.kb_end; kb += kKG) {
        if (!warp_wait(&full_bar[stage], phase, p.timeout_ns, abort_flag)) {
          if (lane == 0) on_timeout();
          goto sf_done;
        }
        if (kBF4 || kb == seg.kb_begin || kb % 4 == 0) {
          const uint32_t sf_base = smem_addr(smem + C::OFF_SF + stage * C::SF_BYTES);
          const uint32_t a0 = ld_shared_u32(sf_base + C::SF_RAW_A + 4 * lane);
          const uint32_t a1 = ld_shared_u32(sf_base + C::SF_RAW_A + 4 * (lane + 32));
          const uint32_t a2 = ld_shared_u32(sf_base + C::SF_RAW_A + 4 * (lane + 64));
          const uint32_t a3 = ld_shared_u32(sf_base + C::SF_RAW_A + 4 * (lane + 96));
          st_shared_v4(sf_base + C::SF_UT_A + 16 * lane, a0, a1, a2, a3);
          if constexpr (kBF4) {
            // K-group s of the stage: tile row r's word at raw word s * BN + r (rows past BN
            // read as 0: their columns are never stored)
#pragma unroll
            for (int s = 0; s < C::SFB_SETS; ++s) {
#pragma unroll
              for (int ch = 0; ch < C::SFB_CHUNKS; ++ch) {
                uint32_t w[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const int r = 128 * ch + static_cast<int>(lane) + 32 * j;
                  w[j] = r < BN ? ld_shared_u32(sf_base + C::SF_RAW_B + 4 * (s * BN + r)) : 0u;
                }
                st_shared_v4(sf_base + C::SF_UT_B + 512 * (s * C::SFB_CHUNKS + ch) + 16 * lane, w[0], w[1], w[2],
                             w[3]);
              }
            }
          } else {
#pragma unroll
            for (int ch = 0; ch < C::SFB_CHUNKS; ++ch) {
              uint32_t w[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int n = n0 + 128 * ch + static_cast<int>(lane) + 32 * j;
                w[j] = ld_shared_u32(sf_base + C::SF_RAW_B + 4 * (n / SF_BLOCK_N - sfb_x));
              }
              st_shared_v4(sf_base + C::SF_UT_B + 512 * ch + 16 * lane, w[0], w[1], w[2], w[3]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sf_ready_bar[stage]);
        }
        if (lane == 0) mbar_arrive(&empty_bar[stage]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  sf_done:
    __syncwarp();
  } else if (kSplit > 0 && warp >= 2 && warp < 2 + kEpiWarps) {
    // ============================ split-K epilogue (cluster) ========================
    // 1. this CTA's FP32 partial: TMEM -> its shared memory; 2. cluster barrier; 3. CTA r
    // sums the partials of its column slice over the cluster's CTAs in rank order (reading
    // the others' shared memory), adds C, rounds to BF16 and stores; the kernel's closing
    // cluster barrier keeps every CTA's shared memory alive until all reads are done.
    // Every thread of the cluster passes both barriers on every path (timeouts included).
    if constexpr (kSplit > 0) {
      const int quad = warp % 4;
      const int row_in_tile = quad * 32 + static_cast<int>(lane);
      const uint32_t part = smem_addr(smem + C::OFF_A);
      constexpr int kSliceCols = BN / kSplit;          // output columns this CTA reduces and stores
      constexpr int kUnits = kSliceCols / 8;           // 8-column (16-byte BF16) units of a row
      bool ok = sched.next(p, seg);
      const int rank = seg.slot;
      const int row = seg.m_blk * BLOCK_M + row_in_tile;
      const bool row_ok = ok && row < p.M;
      // C of this CTA's output slice, staged (coalesced) in the warp's epilogue buffer, which
      // this path does not otherwise use, while the MMAs run
      const uint32_t cstage = smem_addr(smem + C::OFF_EPI + (warp - 2) * C::EPI_BUF_BYTES);
      if constexpr (kHasC) {
        const int gcol0 = seg.n_blk * BN + rank * kSliceCols;
        const uint32_t ok_rows = __ballot_sync(0xffffffffu, row_ok);
        const int row0 = seg.m_blk * BLOCK_M + quad * 32;
        warp_stage_c<__nv_bfloat16, kUnits>(cstage, p.c + static_cast<long long>(row0) * p.N + gcol0, p.N, ok_rows,
                                            p.N - gcol0, lane);
      }
      if (ok) {
        ok = warp_wait(&tfull_bar[0], 0, p.timeout_ns, abort_flag);
        if (!ok && lane == 0) on_timeout();
      }
      if (ok) {
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
#pragma unroll 1
        for (int ch = 0; ch < BN / 32; ++ch) {
          uint32_t v[32];
          tmem_load_32x32b_x32(taddr + 32 * ch, v);
          tmem_load_wait();
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_shared_v4(part + ((8 * ch + q) * BLOCK_M + row_in_tile) * 16, v[4 * q], v[4 * q + 1], v[4 * q + 2],
                         v[4 * q + 3]);
        }
        tc_fence_before();
      }
      __syncwarp();
      cluster_sync();   // partials of every CTA of the cluster are in shared memory
      if (ok && *abort_flag == 0) {
        uint32_t src[kSplit];
#pragma unroll
        for (int r = 0; r < kSplit; ++r) src[r] = r == rank ? part : map_to_rank(smem + C::OFF_A, r);
        // all partial loads first (one round trip), then sums in rank order
        uint4 pv[kSplit][kUnits][2];
#pragma unroll
        for (int r = 0; r < kSplit; ++r) {
#pragma unroll
          for (int u = 0; u < kUnits; ++u) {
            const uint32_t off0 = (((rank * kSliceCols + 8 * u) / 4) * BLOCK_M + row_in_tile) * 16;
            const uint32_t off1 = off0 + BLOCK_M * 16;   // the next float4 column group
            pv[r][u][0] = r == rank ? ld_shared_v4(src[r] + off0) : ld_shared_cluster_v4(src[r] + off0);
            pv[r][u][1] = r == rank ? ld_shared_v4(src[r] + off1) : ld_shared_cluster_v4(src[r] + off1);
          }
        }
#pragma unroll
        for (int u = 0; u < kUnits; ++u) {
          const int gcol = seg.n_blk * BN + rank * kSliceCols + 8 * u;
          float f[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) f[i] = 0.0f;
#pragma unroll
          for (int r = 0; r < kSplit; ++r) {
            f[0] += __uint_as_float(pv[r][u][0].x);
            f[1] += __uint_as_float(pv[r][u][0].y);
            f[2] += __uint_as_float(pv[r][u][0].z);
            f[3] += __uint_as_float(pv[r][u][0].w);
            f[4] += __uint_as_float(pv[r][u][1].x);
            f[5] += __uint_as_float(pv[r][u][1].y);
            f[6] += __uint_as_float(pv[r][u][1].z);
            f[7] += __uint_as_float(pv[r][u][1].w);
          }
          if (row_ok && gcol < p.N) {
            if constexpr (kHasC) {
              const uint4 cvu = ld_shared_v4(cstage + lane * 128 + ((u ^ (lane & 7)) * 16));
              const uint32_t cw[4] = {cvu.x, cvu.y, cvu.z, cvu.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 cf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&cw[e]));
                f[2 * e] = cf.x + f[2 * e];
                f[2 * e + 1] = cf.y + f[2 * e + 1];
              }
            }
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
              w[e] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            st_global_v4(p.d + static_cast<long long>(row) * p.N + gcol, w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  } else if (warp >= 2 && warp < 2 + kEpiWarps) {
    // ================================ epilogue ====================================
    const int ew = warp - 2;
    const int quad = warp % 4;                      // TMEM sub-partition this warp may access
    const int col_part = ew / 4;
    uint8_t* stage_base = smem + C::OFF_EPI + ew * kEpiBufs * C::EPI_BUF_BYTES;
    uint32_t seg_iter = 0, buf_iter = 0;
    constexpr int kChunks = C::kColsPerEpiWarp / 64;

    while (sched.next(p, seg)) {
      const uint32_t acc = seg_iter % kNumAccum;
      const uint32_t acc_phase = (seg_iter / kNumAccum) & 1;
      ++seg_iter;
      if (!warp_wait(&tfull_bar[acc], acc_phase, p.timeout_ns, abort_flag)) {
        if (lane == 0) on_timeout();
        break;
      }
      tc_fence_after();

      const int row_in_tile = quad * 32 + static_cast<int>(lane);
      const int row = seg.m_blk * BLOCK_M + row_in_tile;   // row index within A / D (or within group)
      bool row_ok;
      long long d_row;                                     // linear row of D
      if constexpr (kKind == Kind::Dense) {
        row_ok = row < p.M;
        d_row = row;
      } else if constexpr (kKind == Kind::Contiguous) {
        const int gi = row < p.M ? ld_cg_s32(p.m_indices + row) : -1;
        row_ok = gi == seg.g;
        if (gi != seg.g && gi != -1 && seg.n_blk == 0 && col_part == 0) atomicOr(p.status, kStatusBadIndexBit);
        d_row = row;
      } else {
        row_ok = row < seg.valid_m;
        d_row = static_cast<long long>(seg.g) * p.M + row;
      }
      const uint32_t ok_mask = __ballot_sync(0xffffffffu, row_ok);
      const int n0 = seg.n_blk * BN;
      const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;

      // (+C) -> BF16 -> swizzled smem -> TMA store / predicated rows, for one 64-column chunk
      // (FP32 output: two 32-column halves, each one 128-byte-wide TMA box)
      auto store_chunk = [&](float (&f)[64], int col, bool c_added = false) {
        if constexpr (kOutF32) {
          const float* cbase = reinterpret_cast<const float*>(p.c);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int hcol = col + 32 * h;
            uint8_t* sbuf = stage_base + (buf_iter % kEpiBufs) * C::EPI_BUF_BYTES;
            ++buf_iter;
            if (lane == 0) bulk_wait_group_read<kEpiBufs - 1>();
            __syncwarp();
            const uint32_t srow = smem_addr(sbuf) + lane * 128;
            if constexpr (kHasC) {
              if (!c_added) {
                const long long row0 = __shfl_sync(0xffffffffu, d_row, 0);
                warp_stage_c(smem_addr(sbuf), cbase + row0 * p.N + n0 + hcol, p.N, ok_mask, p.N - (n0 + hcol), lane);
                __syncwarp();
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  const uint4 cv = ld_shared_v4(srow + ((q ^ (lane & 7)) * 16));
                  f[32 * h + 4 * q + 0] = __uint_as_float(cv.x) + f[32 * h + 4 * q + 0];
                  f[32 * h + 4 * q + 1] = __uint_as_float(cv.y) + f[32 * h + 4 * q + 1];
                  f[32 * h + 4 * q + 2] = __uint_as_float(cv.z) + f[32 * h + 4 * q + 2];
                  f[32 * h + 4 * q + 3] = __uint_as_float(cv.w) + f[32 * h + 4 * q + 3];
                }
              }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
              st_shared_v4(srow + ((u ^ (lane & 7)) * 16), __float_as_uint(f[32 * h + 4 * u]),
                           __float_as_uint(f[32 * h + 4 * u + 1]), __float_as_uint(f[32 * h + 4 * u + 2]),
                           __float_as_uint(f[32 * h + 4 * u + 3]));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if constexpr (kKind == Kind::KGrouped) {
                tma_store_3d(&tm_d, sbuf, n0 + hcol, seg.m_blk * BLOCK_M + quad * 32, seg.g);
              } else {
                tma_store_2d(&tm_d, sbuf, n0 + hcol, seg.m_blk * BLOCK_M + quad * 32);
              }
              bulk_commit_group();
            }
          }
          return;
        }
        uint8_t* sbuf = stage_base + (buf_iter % kEpiBufs) * C::EPI_BUF_BYTES;
        ++buf_iter;
        if (lane == 0) bulk_wait_group_read<kEpiBufs - 1>();
        __syncwarp();
        const uint32_t srow = smem_addr(sbuf) + lane * 128;
        if constexpr (kHasC) {
          if (!c_added) {
            const long long row0 = __shfl_sync(0xffffffffu, d_row, 0);
            warp_stage_c(smem_addr(sbuf), p.c + row0 * p.N + n0 + col, p.N, ok_mask, p.N - (n0 + col), lane);
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint4 cv = ld_shared_v4(srow + ((q ^ (lane & 7)) * 16));
              const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 c2 = *reinterpret_cast<const __nv_bfloat162*>(&cw[e]);
                const float2 cf = __bfloat1622float2(c2);
                f[8 * q + 2 * e] = cf.x + f[8 * q + 2 * e];
                f[8 * q + 2 * e + 1] = cf.y + f[8 * q + 2 * e + 1];
              }
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(f[8 * u + 2 * e], f[8 * u + 2 * e + 1]);
            w[e] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          st_shared_v4(srow + ((u ^ (lane & 7)) * 16), w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (kKind == Kind::Dense || ok_mask == 0xffffffffu) {
          if (lane == 0) {
            if constexpr (kKind == Kind::Masked) {
              tma_store_3d(&tm_d, sbuf, n0 + col, seg.m_blk * BLOCK_M + quad * 32, seg.g);
            } else {
              tma_store_2d(&tm_d, sbuf, n0 + col, seg.m_blk * BLOCK_M + quad * 32);
            }
            bulk_commit_group();
          }
        } else if (ok_mask != 0) {
          // Rows of this warp are partly padding / masked: copy only the valid rows, one
          // 128-byte row per warp instruction (lane = two columns).
          const int gcol = n0 + col + 2 * static_cast<int>(lane);
#pragma unroll 1
          for (int r = 0; r < 32; ++r) {
            const long long drow = __shfl_sync(0xffffffffu, d_row, r);
            if (((ok_mask >> r) & 1u) && gcol < p.N) {
              const uint32_t unit = (lane / 4) ^ (r & 7);
              const uint32_t val = ld_shared_u32(smem_addr(sbuf) + r * 128 + unit * 16 + (lane % 4) * 4);
              *reinterpret_cast<uint32_t*>(p.d + drow * p.N + gcol) = val;
            }
          }
        }
      };

      if (seg.n_contrib == 1) {
        // a K-grouped expert without tokens has no MMAs: its accumulator is zero, not TMEM
        const bool empty = kKind == Kind::KGrouped && seg.kb_end <= seg.kb_begin;
#pragma unroll 1
        for (int ch = 0; ch < kChunks; ++ch) {
          const int col = col_part * C::kColsPerEpiWarp + ch * 64;   // column within the tile
          uint32_t v0[32], v1[32];
          const uint32_t taddr = tmem_base + t_lane + acc * BN + col;
          if (!empty) {
            tmem_load_32x32b_x32(taddr, v0);
            tmem_load_32x32b_x32(taddr + 32, v1);
            tmem_load_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v0[i] = v1[i] = 0u;
          }
          if (ch == kChunks - 1) {
            // this warp has read its whole share of the accumulator: hand it back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty_bar[acc]);
          }
          float f[64];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            f[i] = __uint_as_float(v0[i]);
            f[32 + i] = __uint_as_float(v1[i]);
          }
          store_chunk(f, col);
        }
      } else {
        // stream-K: publish this CTA's FP32 partial of the warp's block, then let the last
        // contributor to arrive sum all partials (in slot order) and store the tile.
        float* my_ws = p.sk_ws + (static_cast<long long>(seg.tile) * p.sk_slots + seg.slot) * C::SK_TILE_FLOATS +
                       ew * C::SK_WARP_FLOATS;
#pragma unroll 1
        for (int ch = 0; ch < kChunks; ++ch) {
          const int col = col_part * C::kColsPerEpiWarp + ch * 64;
          uint32_t v0[32], v1[32];
          const uint32_t taddr = tmem_base + t_lane + acc * BN + col;
          tmem_load_32x32b_x32(taddr, v0);
          tmem_load_32x32b_x32(taddr + 32, v1);
          tmem_load_wait();
          if (ch == kChunks - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty_bar[acc]);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t* src = q < 4 ? &v0[8 * q] : &v1[8 * (q - 4)];
            const int c4 = ch * 16 + 2 * q;   // float4 column group within the warp's columns
            st_global_v4f(my_ws + (c4 * 32 + lane) * 4, __uint_as_float(src[0]), __uint_as_float(src[1]),
                          __uint_as_float(src[2]), __uint_as_float(src[3]));
            st_global_v4f(my_ws + ((c4 + 1) * 32 + lane) * 4, __uint_as_float(src[4]), __uint_as_float(src[5]),
                          __uint_as_float(src[6]), __uint_as_float(src[7]));
          }
        }
        __threadfence();
        __syncwarp();
        int arrived = 0;
        int* counter = p.sk_counters + seg.tile * kEpiWarps + ew;
        if (lane == 0) arrived = atomicAdd(counter, 1);
        arrived = __shfl_sync(0xffffffffu, arrived, 0);
        if (arrived == seg.n_contrib - 1) {
          __threadfence();
          const float* tile_ws = p.sk_ws + static_cast<long long>(seg.tile) * p.sk_slots * C::SK_TILE_FLOATS +
                                 ew * C::SK_WARP_FLOATS;
          // This CTA's last segment: the ring's shared memory is idle (every load consumed,
          // every MMA complete), so each warp gathers all contributors' partials of a chunk
          // (and its C rows) with asynchronous copies in one round trip, then sums them in
          // slot order from shared memory.
          constexpr int kRingBytes = C::OFF_EPI - C::OFF_A;
          constexpr int kWarpRing = (kRingBytes / kEpiWarps) & ~1023;
          constexpr int kChunkSlotBytes = 16 * 32 * 16;         // 16 float4 per lane per chunk
          constexpr bool kPrefetchC = kHasC && !kOutF32;        // an FP32 C is added by store_chunk
          constexpr int kCBytes = kPrefetchC ? 32 * 128 : 0;    // 32 rows x 64 BF16 columns
          if (seg.cta_last && seg.n_contrib * kChunkSlotBytes + kCBytes <= kWarpRing) {
            const uint32_t region = smem_addr(smem + C::OFF_A) + ew * kWarpRing;
#pragma unroll 1
            for (int ch = 0; ch < kChunks; ++ch) {
              const int col = col_part * C::kColsPerEpiWarp + ch * 64;
#pragma unroll 1
              for (int s = 0; s < seg.n_contrib; ++s) {
                const float* src = tile_ws + static_cast<long long>(s) * C::SK_TILE_FLOATS;
#pragma unroll
                for (int q = 0; q < 16; ++q)
                  cp_async_16(region + s * kChunkSlotBytes + (q * 32 + lane) * 16,
                              src + ((ch * 16 + q) * 32 + lane) * 4);
              }
              if constexpr (kPrefetchC) {
                if (row_ok) {
                  const __nv_bfloat16* crow = p.c + d_row * p.N + n0 + col;
#pragma unroll
                  for (int q = 0; q < 8; ++q)
                    if (n0 + col + 8 * q < p.N)
                      cp_async_16(region + seg.n_contrib * kChunkSlotBytes + lane * 128 + q * 16, crow + 8 * q);
                }
              }
              cp_async_wait_all();
              __syncwarp();
              float f[64];
#pragma unroll
              for (int i = 0; i < 64; ++i) f[i] = 0.0f;
#pragma unroll 1
              for (int s = 0; s < seg.n_contrib; ++s) {
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                  const uint4 v = ld_shared_v4(region + s * kChunkSlotBytes + (q * 32 + lane) * 16);
                  f[4 * q + 0] += __uint_as_float(v.x);
                  f[4 * q + 1] += __uint_as_float(v.y);
                  f[4 * q + 2] += __uint_as_float(v.z);
                  f[4 * q + 3] += __uint_as_float(v.w);
                }
              }
              if constexpr (kPrefetchC) {
                if (row_ok) {
#pragma unroll
                  for (int q = 0; q < 8; ++q) {
                    if (n0 + col + 8 * q < p.N) {
                      const uint4 cv = ld_shared_v4(region + seg.n_contrib * kChunkSlotBytes + lane * 128 + q * 16);
                      const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                      for (int e = 0; e < 4; ++e) {
                        const float2 cf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&cw[e]));
                        f[8 * q + 2 * e] = cf.x + f[8 * q + 2 * e];
                        f[8 * q + 2 * e + 1] = cf.y + f[8 * q + 2 * e + 1];
                      }
                    }
                  }
                }
              }
              __syncwarp();   // all lanes have read the region before the next chunk's copies land
              store_chunk(f, col, kPrefetchC);
            }
            if (lane == 0) *counter = 0;   // ready for the next launch
            continue;
          }
#pragma unroll 1
          for (int ch = 0; ch < kChunks; ++ch) {
            const int col = col_part * C::kColsPerEpiWarp + ch * 64;
            float f[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) f[i] = 0.0f;
#pragma unroll 1
            for (int s = 0; s < seg.n_contrib; ++s) {
              const float* src = tile_ws + static_cast<long long>(s) * C::SK_TILE_FLOATS;
#pragma unroll
              for (int q = 0; q < 16; ++q) {
                const float4 v = ld_global_cg_v4f(src + ((ch * 16 + q) * 32 + lane) * 4);
                f[4 * q + 0] += v.x;
                f[4 * q + 1] += v.y;
                f[4 * q + 2] += v.z;
                f[4 * q + 3] += v.w;
              }
            }
            store_chunk(f, col);
          }
          if (lane == 0) *counter = 0;   // ready for the next launch
        }
      }
    }
    if (lane == 0) bulk_wait_group_all();
    __syncwarp();
  }

  if constexpr (kSplit > 0) {
    // the epilogue warps passed the first cluster barrier above; everyone passes the last
    __syncwarp();
    if (!(warp >= 2 && warp < 2 + kEpiWarps)) cluster_sync();
    cluster_sync();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace dg
