// CTA-pair variant of the fine-grained-scaled FP8 GEMM for sm_103a: two CTAs of a
// cluster share one tcgen05.mma.cta_group::2 of shape 256 x BN (x 32): BN = 256 with one
// accumulator, or BN = 240 / 192 with two (two 256-column accumulators would leave no TMEM
// columns for the scale factors; 240 columns leave 16 beside each accumulator).
//
// Each CTA of the pair holds 128 rows of A and BN/2 of the BN rows of the B tile in its
// own shared memory; the pair's MMA reads both and each CTA's TMEM receives its 128 x BN
// block of the accumulator. Per SM this halves the B bytes loaded and stored in shared
// memory per FLOP compared with a 128 x BN tile on one SM, which is what bounds the
// single-CTA kernel on GB300 (L2->SM traffic and bytes in flight). With two accumulators
// the MMAs of the next tile run while the epilogue drains the previous one.
//
// Roles (both CTAs run the same code):
//   warp 0      TMA producer: its own A rows, its own half of B and the scale chunks,
//               counted on the full barrier of the leader CTA (rank 0).
//   warp 1      allocates TMEM for the pair; in the leader one thread issues the MMAs
//               (one ready-barrier wait and four MMAs per K-group) and commits to the
//               empty / accumulator-full barriers of both CTAs.
//   warps 2..   epilogue, BN/64 x 4 warps' worth of 64-column chunks: each warp reads its
//               32 TMEM lanes of its chunks into registers, hands the accumulator back to
//               the leader, then adds C, rounds to BF16 and TMA-stores (or stores valid
//               rows only).
//   last warp   (leader) hands each stage to the MMA thread: waits for its operands and,
//               on a stage that carries scale chunks, copies them into TMEM
//               (tcgen05.cp.cta_group::2) and signals through tcgen05.commit. Keeping the
//               copies and the TMA-barrier waits off the issuing thread keeps its MMA stream
//               dense (an issuing thread's own shared-memory accesses stall it).
// The scale words are consumed in the tcgen05.cp source layout, produced beforehand in a
// workspace by sf_to_utccp_kernel: one 512-byte chunk per 128 rows of A per 4 K-groups,
// and two per BN-wide tile of B per 4 K-groups (tile columns 0..127 and 128..255), or per
// K-group for FP4 B (one word per row: the scales of its four 32-wide blocks).
// Operation: D = C + A @ B.T (DeepGEMM README "Interfaces / Notices", "Normal dense GEMMs",
// "Grouped GEMMs (contiguous layout)", as reproduced on the page "Weight gradient kernels
// for dense and MoE models #95").
#pragma once

#include "fp8_gemm.cuh"

namespace dg {

// kBF4: B is FP4 (E2M1 with one UE8M0 per row per 32 K), loaded through 16U4_ALIGN16B maps into
// the same shared-memory shape as E4M3 (the barrier counts half the bytes); every stage then
// carries scale chunks (A's K-quad chunk and this K-group's B chunks).
// kSmallEpi (BF16 output without C): each epilogue warp stages 32-column pieces in 2 KB
// (64-byte rows) instead of 64-column chunks in 4 KB, which leaves room for a sixth stage.
// Measured on GB300, the CTA-pair kernel is bound by the depth of its ring (a stage is
// refilled only after the MMAs that read it complete and its TMA loads land again): 3 / 4 / 5
// stages gave 2500 / 2915 / 3200 TFLOPS on the contiguous G=8 workload.
template <int kStages, int kBN, int kNumAccum, bool kBF4 = false, bool kSmallEpi_ = false>
struct PairConfig {
  static constexpr bool kSmallEpi = kSmallEpi_;
  static constexpr int BN = kBN;                 // tile width of the pair; each CTA loads BN/2 B rows
  static_assert(BN % 16 == 0 && BN >= 128 && BN <= 256, "tile width: a multiple of 16 in [128, 256]");
  static constexpr int kChunks = ceil_div_c(BN, 64);   // epilogue chunks of 64 columns (last may be narrower)
  static constexpr int kTail = BN % 64;                // width of a narrower last chunk (0: none)
  static constexpr int kWarpsPerQuad = kChunks % 2 == 0 ? 2 : kChunks;
  static constexpr int kChunksPerWarp = kChunks / kWarpsPerQuad;
  static constexpr int kEpiWarps = 4 * kWarpsPerQuad;
  static constexpr int kReadyWarp = 2 + kEpiWarps;
  static constexpr int kThreads = (3 + kEpiWarps) * 32;
  static constexpr int A_BYTES = BLOCK_M * BLOCK_K;
  static constexpr int B_BYTES = (BN / 2) * BLOCK_K;
  static constexpr int SFA_BYTES = 512;          // one tcgen05.cp chunk: this CTA's 128 rows
  static constexpr int SFB_BYTES = 1024;         // two chunks: the 256 columns of the pair tile
  static constexpr int SF_STRIDE = SFA_BYTES + SFB_BYTES;   // a multiple of 128 (TMA destinations)
  static constexpr int EPI_BUF_BYTES = kSmallEpi ? 32 * 64 : 32 * 128;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + kStages * A_BYTES;
  static constexpr int OFF_SF = OFF_B + kStages * B_BYTES;
  static constexpr int OFF_EPI = ((OFF_SF + kStages * SF_STRIDE + 1023) / 1024) * 1024;
  static constexpr int OFF_BAR = OFF_EPI + kEpiWarps * EPI_BUF_BYTES;
  // TMEM scale buffers (4 SFA + 8 SFB columns each): two, or with FP4 B (a copy every stage)
  // four where the columns allow, so that copies can run further ahead of the MMAs
  static constexpr int kSfBufs = (kBF4 && kNumAccum * BN + 12 * 4 <= 512) ? 4 : 2;
  // full / empty / ready per stage, tfull / tempty per accumulator, MMA drain, copy drain,
  // one "scale buffer free" barrier per TMEM scale buffer, one "C landed" per epilogue warp
  static constexpr int NUM_BARS = 3 * kStages + 2 * kNumAccum + 2 + kSfBufs + kEpiWarps;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
  static constexpr int TX_AB = 2 * (A_BYTES + (kBF4 ? B_BYTES / 2 : B_BYTES));   // both CTAs, every stage
  static constexpr int TX_SF = 2 * (SFA_BYTES + SFB_BYTES);       // both CTAs, every scale stage
  // TMEM: kNumAccum BN-column accumulators and 2 x 4 SFA / 2 x 8 SFB columns, packed when
  // they fit; otherwise (two 240-column accumulators) the accumulators start at columns 0
  // and 256 and the scale columns sit in the 16 columns after each
  static constexpr bool kPacked = kNumAccum * BN + 12 * kSfBufs <= 512;
  static constexpr int ACC_STRIDE = kPacked ? BN : 256;
  static constexpr int SFA_COL = kPacked ? kNumAccum * BN : BN;
  static constexpr int SFB_COL = kPacked ? SFA_COL + 4 * kSfBufs : 256 + BN;
  static constexpr int TMEM_COLS = 512;
  static_assert(kPacked || (kNumAccum == 2 && BN + 8 <= 256 && 256 + BN + 16 <= TMEM_COLS), "TMEM layout");
  static_assert(!kPacked || SFB_COL + 8 * kSfBufs <= TMEM_COLS, "TMEM columns exceeded");
  static_assert(kPacked || kSfBufs == 2, "unpacked TMEM layout: two scale buffers");
};

// Walks the pair tiles of the sequence t = cluster, += clusters. A pair row is two
// consecutive 128-row blocks; in the contiguous form both blocks belong to one expert (an
// expert with an odd number of blocks ends with a pair whose second block is not its own:
// that CTA's rows are computed and discarded). The contiguous pair rows are listed once per
// call by sf_to_utccp_kernel (first block, expert and own-block count per pair row, and
// their number), so a tile costs one small load.
// K-grouped form: tiles are (expert, pair row, n); every role visits the experts in increasing
// order and carries the running K-group and scale-row offsets of the current one.
template <Kind kKind, int kBN>
struct PairScheduler {
  int num_n, total;
  int t, step;
  int pairs_per_g, g_cur, kbase_cur, sfrow_cur;   // K-grouped walk

  __device__ __forceinline__ PairScheduler(const Params& p, int cluster, int clusters) {
    num_n = ceil_div_c(p.N, kBN);
    t = cluster;
    step = clusters;
    pairs_per_g = ceil_div_c(ceil_div_c(p.M, BLOCK_M), 2);
    g_cur = kbase_cur = sfrow_cur = 0;
    if constexpr (kKind == Kind::Contiguous) {
      total = ld_cg_s32(p.pair_count) * num_n;
    } else if constexpr (kKind == Kind::KGrouped) {
      total = p.G * pairs_per_g * num_n;
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
        if (bad || kg_sum != p.K / BLOCK_K || rows != p.sf_k_rows) atomicOr(p.status, kStatusBadIndexBit);
      }
    } else {
      total = pairs_per_g * num_n;
    }
  }

  // seg.m_blk is the pair's first block; the CTA of rank r works on block m_blk + r.
  __device__ __forceinline__ bool next(const Params& p, Segment& s) {
    if (t >= total) return false;
    s.k_base = 0;
    s.sf_row = 0;
    s.kb_begin = 0;
    s.kb_end = p.K / BLOCK_K;
    s.n_contrib = 1;
    s.slot = 0;
    s.valid_m = p.M;
    if constexpr (kKind == Kind::KGrouped) {
      const int cur = t;
      t += step;
      const int tpg = pairs_per_g * num_n;
      const int g = cur / tpg;
      while (g_cur < g) {
        const int k = ld_cg_s32(p.ks + g_cur);
        if (k > 0) {
          kbase_cur += k / BLOCK_K;
          sfrow_cur += (k + 4 * BLOCK_K - 1) / (4 * BLOCK_K);
        }
        ++g_cur;
      }
      const int local = cur - g * tpg;
      const int k = ld_cg_s32(p.ks + g);
      s.g = g;
      s.m_blk = 2 * (local / num_n);
      s.n_blk = local % num_n;
      s.tile = cur;
      s.kb_end = k > 0 ? k / BLOCK_K : 0;   // 0: an expert without tokens (D = C)
      s.k_base = kbase_cur;
      s.sf_row = sfrow_cur;
      return true;
    }
    const int pair = t / num_n;
    s.n_blk = t % num_n;
    t += step;
    s.tile = pair;
    if constexpr (kKind == Kind::Contiguous) {
      s.m_blk = ld_cg_s32(p.pair_list + 3 * pair);
      s.g = ld_cg_s32(p.pair_list + 3 * pair + 1);
      s.n_contrib = ld_cg_s32(p.pair_list + 3 * pair + 2);   // blocks of the pair that are the expert's
    } else {
      s.g = 0;
      s.m_blk = 2 * pair;
    }
    return true;
  }
};

// kOutF32: FP32 C / D (the dense weight-gradient form), else BF16. kBF4: B in FP4.
// kAMN / kBMN (dense form, 256-wide tiles): A given as [K, M] / B given as [K, N]. Each CTA's
// 128 rows of A and 128 columns of B are then one MN-major atom: a TMA box of 128 K-rows x 128
// M/N-bytes (128-byte swizzle), described with LBO = 16 KB, SBO = 1024 and advanced 4 KB per
// 32-deep K step, with the instruction descriptor's transpose bits set.
template <Kind kKind, int kStages, int kBN, int kNumAccum, bool kHasC, bool kOutF32 = false, bool kBF4 = false,
          bool kAMN = false, bool kBMN = false>
__global__ void __launch_bounds__(PairConfig<kStages, kBN, kNumAccum, kBF4, !kHasC && !kOutF32>::kThreads, 1)
    fp8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                         const __grid_constant__ CUtensorMap tm_sfa, const __grid_constant__ CUtensorMap tm_sfb,
                         const __grid_constant__ CUtensorMap tm_d, const __grid_constant__ CUtensorMap tm_d_tail,
                         const __grid_constant__ CUtensorMap tm_c, const Params p) {
  static_assert(kKind != Kind::Masked, "the masked form uses the single-CTA kernel");
  static_assert(kKind == Kind::Dense || kBN % 64 == 0, "narrow last chunks: dense form only");
  static_assert(!kOutF32 || kKind == Kind::Dense || kKind == Kind::KGrouped, "FP32 output: dense and K-grouped");
  static_assert(kKind != Kind::KGrouped || (kOutF32 && !kBF4), "the K-grouped form: FP8 operands, FP32 output");
  static_assert(!kBF4 || !kOutF32, "FP4 B: BF16 output");
  static_assert((!kAMN && !kBMN) || (kKind == Kind::Dense && kBN == 256 && !kBF4),
                "MN-major operands: the dense form with 256-wide tiles");
  using C = PairConfig<kStages, kBN, kNumAccum, kBF4, !kHasC && !kOutF32>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full_bar = bars;                    // used in the leader only
  uint64_t* empty_bar = bars + kStages;         // both CTAs (leader's commit, multicast)
  uint64_t* tfull_bar = bars + 2 * kStages;     // [kNumAccum] both CTAs (leader's commit, multicast)
  uint64_t* tempty_bar = tfull_bar + kNumAccum;  // [kNumAccum] leader: epilogue warps of both CTAs
  uint64_t* drain_bar = tempty_bar + kNumAccum;
  uint64_t* ready_bar = drain_bar + 1;          // [kStages] leader: stage handed to the MMA thread
  uint64_t* sf_drain_bar = ready_bar + kStages;
  uint64_t* sf_free_bar = sf_drain_bar + 1;     // [kSfBufs] leader: MMAs reading TMEM scale buffer b completed
  uint64_t* c_bar = sf_free_bar + C::kSfBufs;   // [kEpiWarps] this CTA: a C box landed in warp w's staging
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x / 32;
  const uint32_t lane = threadIdx.x % 32;
  const uint32_t rank = cluster_cta_rank() & 1u;
  const bool leader = rank == 0;
  const int num_kb = p.K / BLOCK_K;
  const int KP = (num_kb + 3) / 4;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int i = 0; i < kNumAccum; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], 2 * C::kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    for (int s = 0; s < kStages; ++s) mbar_init(&ready_bar[s], 1);
    mbar_init(sf_drain_bar, 1);
    for (int b = 0; b < C::kSfBufs; ++b) mbar_init(&sf_free_bar[b], 1);
    for (int w = 0; w < C::kEpiWarps; ++w) mbar_init(&c_bar[w], 1);
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
    if constexpr (kHasC) tma_prefetch_desc(&tm_c);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_dependency_wait();   // programmatic dependent launch: no global access before this

  auto on_timeout = [&]() {
    atomicOr(p.status, kStatusTimeoutBit);
    *abort_flag = 1;
  };

  PairScheduler<kKind, kBN> sched(p, static_cast<int>(blockIdx.x / 2), static_cast<int>(gridDim.x / 2));
  Segment seg;

  if (warp == 0) {
    // ================================ TMA producer (both CTAs) ====================
    if (lane == 0 && p.fault != kFaultProducerSilent) {
      uint32_t stage = 0, phase = 0, issued = 0;
      while (sched.next(p, seg)) {
        const int m_blk = seg.m_blk + static_cast<int>(rank);
        const int n0 = seg.n_blk * C::BN;
        for (int kb = 0; kb < seg.kb_end; ++kb) {
          if (*abort_flag || !mbar_wait(&empty_bar[stage], phase ^ 1, p.timeout_ns)) {
            on_timeout();
            goto producer_done;
          }
          const bool with_sf = kBF4 || (kb % 4) == 0;
          const uint32_t fb = map_to_rank(&full_bar[stage], 0);
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], C::TX_AB + (with_sf ? C::TX_SF : 0));
          uint8_t* sa = smem + C::OFF_A + stage * C::A_BYTES;
          uint8_t* sb = smem + C::OFF_B + stage * C::B_BYTES;
          uint8_t* ssf = smem + C::OFF_SF + stage * C::SF_STRIDE;
          if constexpr (kAMN) {
            tma_load_2d_pair(sa, &tm_a, fb, m_blk * BLOCK_M, kb * BLOCK_K);
          } else {
            tma_load_2d_pair(sa, &tm_a, fb, (seg.k_base + kb) * BLOCK_K, m_blk * BLOCK_M);
          }
          if constexpr (kBMN) {
            tma_load_2d_pair(sb, &tm_b, fb, n0 + static_cast<int>(rank) * (C::BN / 2), kb * BLOCK_K);
          } else if constexpr (kKind == Kind::Dense || kKind == Kind::KGrouped) {
            tma_load_2d_pair(sb, &tm_b, fb, (seg.k_base + kb) * BLOCK_K, n0 + static_cast<int>(rank) * (C::BN / 2));
          } else {
            tma_load_3d_pair(sb, &tm_b, fb, kb * BLOCK_K, n0 + static_cast<int>(rank) * (C::BN / 2), seg.g);
          }
          if (with_sf) {
            const int q = seg.sf_row + kb / 4;
            // SFA chunk row: (q, m_blk); SFB chunk rows: (g, q, n-block) and the next one, or
            // with FP4 B (g, kb, n-block): one pair of chunks per K-group; the K-grouped form's
            // word rows q run over all experts (B is not grouped)
            tma_load_2d_pair(ssf, &tm_sfa, fb, 0, q * p.sf_num_mb + m_blk);
            const int b_row = kBF4 ? seg.g * num_kb + kb : (kKind == Kind::KGrouped ? q : seg.g * KP + q);
            tma_load_2d_pair(ssf + C::SFA_BYTES, &tm_sfb, fb, 0, b_row * p.sf_nb + 2 * seg.n_blk);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    producer_done:
      grid_launch_dependents();
      if (leader) {
        for (uint32_t s = 0; s < kStages && s < issued; ++s) {
          const uint32_t last_use = (issued - 1 - s) / kStages;
          mbar_wait(&full_bar[s], last_use & 1, 50000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ================================ MMA issuer (leader) ===========================
    // One thread of the leader runs the whole loop (no warp-wide synchronisation per K-group).
    if (leader && lane == 0) {
      // B format field [10,13): 0 = E4M3, 5 = E2M1
      constexpr uint32_t kIdesc = make_idesc_mxf8_e4m3(2 * BLOCK_M, C::BN) | (kBF4 ? 5u << 10 : 0u) |
                                  (kAMN ? 1u << 15 : 0u) | (kBMN ? 1u << 16 : 0u);
      const uint64_t a_desc0 =
          make_smem_desc(smem_addr(smem + C::OFF_A), kAMN ? 128 * BLOCK_K : 16, 1024, kLayoutSwizzle128B);
      const uint64_t b_desc0 =
          make_smem_desc(smem_addr(smem + C::OFF_B), kBMN ? 128 * BLOCK_K : 16, 1024, kLayoutSwizzle128B);
      // descriptor steps (address >> 4) per 32-deep K step: 32 bytes along a K-major row, or
      // 32 rows of 128 bytes down an MN-major box
      constexpr uint64_t kAStep = kAMN ? (32 * 128) >> 4 : 2;
      constexpr uint64_t kBStep = kBMN ? (32 * 128) >> 4 : 2;
      uint32_t stage = 0, phase = 0, tile_iter = 0, sf_iter = 0;
      while (sched.next(p, seg)) {
        const uint32_t acc = tile_iter % kNumAccum;
        if (*abort_flag || !mbar_wait(&tempty_bar[acc], ((tile_iter / kNumAccum) & 1) ^ 1, p.timeout_ns)) {
          on_timeout();
          goto mma_done;
        }
        tc_fence_after();
        {
          const uint32_t d_tmem = tmem_base + acc * C::ACC_STRIDE;
          uint32_t sfa_tmem = 0, sfb_tmem = 0;
          for (int kb = 0; kb < seg.kb_end; ++kb) {
            if (!mbar_wait(&ready_bar[stage], phase, p.timeout_ns)) {
              on_timeout();
              goto mma_done;
            }
            tc_fence_after();
            if (kBF4 || kb % 4 == 0) {
              // the scales of this K-quad (K-group, FP4 B) are in TMEM buffer sf_iter % kSfBufs; the
              // previous buffer's readers are all issued: it may be refilled once they complete
              if (sf_iter > 0) tc_commit_pair(&sf_free_bar[(sf_iter - 1) % C::kSfBufs]);
              const uint32_t buf = sf_iter % C::kSfBufs;
              ++sf_iter;
              sfa_tmem = tmem_base + C::SFA_COL + 4 * buf;
              sfb_tmem = tmem_base + C::SFB_COL + 8 * buf;
            }
            const uint64_t adesc = a_desc0 + ((stage * C::A_BYTES) >> 4);
            const uint64_t bdesc = b_desc0 + ((stage * C::B_BYTES) >> 4);
#pragma unroll
            for (int k = 0; k < BLOCK_K / 32; ++k) {
              // B's scale byte: the K-group's (FP8) or the k-th 32-wide block's (FP4)
              const uint32_t idesc = idesc_with_sf_id(kIdesc, kb % 4, kBF4 ? k : kb % 4);
              mma_mxf8_block_scale_pair(d_tmem, adesc + kAStep * k, bdesc + kBStep * k, idesc, sfa_tmem, sfb_tmem,
                                        (kb | k) != 0);
            }
            tc_commit_pair(&empty_bar[stage]);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
        tc_commit_pair(&tfull_bar[acc]);
        ++tile_iter;
      }
    mma_done:
      tc_commit_pair(drain_bar);
      mbar_wait(drain_bar, 0, 50000000ull);
    }
    __syncwarp();
  } else if (warp == C::kReadyWarp) {
    // ================================ stage hand-off (leader) =======================
    // Walks the stages in the MMA thread's order. A TMEM scale buffer is refilled only
    // after the MMAs reading its previous contents completed (its use k waits for phase
    // k - 1 of its free barrier; phase k needs this very copy, so the parity cannot alias).
    if (leader && lane == 0) {
      const uint64_t sf_desc0 = make_smem_desc(smem_addr(smem + C::OFF_SF), 0, 128, kLayoutNone);
      uint32_t stage = 0, phase = 0, sf_iter = 0;
      while (sched.next(p, seg)) {
        for (int kb = 0; kb < seg.kb_end; ++kb) {
          if (*abort_flag || !mbar_wait(&full_bar[stage], phase, p.timeout_ns)) {
            on_timeout();
            goto ready_done;
          }
          if (kBF4 || kb % 4 == 0) {
            if (sf_iter >= C::kSfBufs &&
                !mbar_wait(&sf_free_bar[sf_iter % C::kSfBufs], ((sf_iter / C::kSfBufs) - 1) & 1, p.timeout_ns)) {
              on_timeout();
              goto ready_done;
            }
            tc_fence_after();
            const uint32_t buf = sf_iter % C::kSfBufs;
            ++sf_iter;
            const uint32_t sfa_tmem = tmem_base + C::SFA_COL + 4 * buf;
            const uint32_t sfb_tmem = tmem_base + C::SFB_COL + 8 * buf;
            const uint64_t sf_desc = sf_desc0 + ((stage * C::SF_STRIDE) >> 4);
            tmem_copy_32x128b_warpx4_pair(sfa_tmem, sf_desc);
            tmem_copy_32x128b_warpx4_pair(sfb_tmem, sf_desc + (C::SFA_BYTES >> 4));
            tmem_copy_32x128b_warpx4_pair(sfb_tmem + 4, sf_desc + ((C::SFA_BYTES + 512) >> 4));
            tc_commit_pair(&ready_bar[stage]);
          } else {
            mbar_arrive(&ready_bar[stage]);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    ready_done:
      // no copy of this thread may still be running when TMEM is released
      tc_commit_pair(sf_drain_bar);
      mbar_wait(sf_drain_bar, 0, 50000000ull);
    }
    __syncwarp();
  } else {
    // ================================ epilogue (both CTAs) ==========================
    const int ew = warp - 2;
    const int quad = warp % 4;
    const int wq = ew / 4;                         // chunks [wq * kChunksPerWarp, (wq + 1) * kChunksPerWarp)
    constexpr int kCols = 64 * C::kChunksPerWarp;   // this warp's columns (the last warp may use fewer)
    const int col0 = kCols * wq;                     // first tile column of this warp
    uint8_t* sbuf = smem + C::OFF_EPI + ew * C::EPI_BUF_BYTES;
    uint32_t tile_iter = 0;
    uint32_t c_loads = 0;   // C boxes loaded into sbuf (parity of c_bar[ew])
    // C of one staging box (32 rows x 128 bytes at column x of the tile's rows, the layout of
    // the output box) by TMA into sbuf, for the warp to add from shared memory. A tile's first
    // box is issued before the accumulator is ready (it lands while the MMAs run).
    auto issue_c_box = [&](int x) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&c_bar[ew], 32 * 128);
        const int y = (seg.m_blk + static_cast<int>(rank)) * BLOCK_M + quad * 32;
        if constexpr (kKind == Kind::KGrouped) {
          tma_load_3d(sbuf, &tm_c, &c_bar[ew], x, y, seg.g);
        } else {
          tma_load_2d(sbuf, &tm_c, &c_bar[ew], x, y);
        }
      }
    };
    auto wait_c_box = [&]() {
      const bool ok = warp_wait(&c_bar[ew], c_loads & 1, p.timeout_ns, abort_flag);
      ++c_loads;
      if (!ok && lane == 0) on_timeout();
    };
    while (sched.next(p, seg)) {
      const uint32_t acc = tile_iter % kNumAccum;
      if constexpr (kHasC) {
        if (lane == 0) bulk_wait_group_read<0>();   // the previous tile's last store has read sbuf
        __syncwarp();
        issue_c_box(seg.n_blk * C::BN + col0);
      }
      if (!warp_wait(&tfull_bar[acc], (tile_iter / kNumAccum) & 1, p.timeout_ns, abort_flag)) {
        if (lane == 0) on_timeout();
        if constexpr (kHasC) wait_c_box();   // no copy may still be landing at exit
        break;
      }
      if constexpr (kHasC) wait_c_box();
      ++tile_iter;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * C::ACC_STRIDE + col0;
      // One accumulator: the warp's whole share into registers, then TMEM handed back at
      // once (the next tile's MMAs wait for it). Two accumulators: a chunk at a time, TMEM
      // handed back after the last chunk is loaded.
      constexpr int kHeld = kNumAccum == 1 ? kCols : 64;
      uint32_t v[kHeld];
      // an expert of the K-grouped form without tokens had no MMAs: its accumulator is zero
      const bool empty = kKind == Kind::KGrouped && seg.kb_end == 0;
      auto load_chunk = [&](int ch, uint32_t* dst) {
        const int col = col0 + 64 * ch;
        if (empty) {
#pragma unroll
          for (int i = 0; i < 64; ++i) dst[i] = 0u;
        } else if (C::kTail == 0 || col + 64 <= C::BN) {
          tmem_load_32x32b_x32(taddr + 64 * ch, *reinterpret_cast<uint32_t(*)[32]>(dst));
          tmem_load_32x32b_x32(taddr + 64 * ch + 32, *reinterpret_cast<uint32_t(*)[32]>(dst + 32));
        } else {
#pragma unroll
          for (int j = 0; j < C::kTail / 16; ++j) tmem_load_32x32b_x16(taddr + 64 * ch + 16 * j, dst + 16 * j);
        }
      };
      auto release = [&]() {
        tmem_load_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(map_to_rank(&tempty_bar[acc], 0));
      };
      if constexpr (kNumAccum == 1) {
#pragma unroll
        for (int ch = 0; ch < C::kChunksPerWarp; ++ch) load_chunk(ch, &v[64 * ch]);
        release();
      }

      const int m_blk = seg.m_blk + static_cast<int>(rank);
      const int row = m_blk * BLOCK_M + quad * 32 + static_cast<int>(lane);
      bool row_ok;
      if constexpr (kKind == Kind::Dense || kKind == Kind::KGrouped) {
        row_ok = row < p.M;
      } else {
        const int gi = row < p.M ? ld_cg_s32(p.m_indices + row) : -1;
        row_ok = gi == seg.g;
        // a row of the expert's own blocks that names another expert violates the layout
        if (gi != seg.g && gi != -1 && static_cast<int>(rank) < seg.n_contrib && seg.n_blk == 0 && wq == 0)
          atomicOr(p.status, kStatusBadIndexBit);
      }
      const uint32_t ok_mask = __ballot_sync(0xffffffffu, row_ok);
      const long long d_row = row;
      const int n0 = seg.n_blk * C::BN;
#pragma unroll
      for (int ch = 0; ch < C::kChunksPerWarp; ++ch) {
        const int col = col0 + 64 * ch;
        // 64 columns, or the narrower last chunk of a tile whose width is not a multiple of 64
        const bool tail = C::kTail != 0 && col + 64 > C::BN;
        const int units = tail ? C::kTail / 8 : 8;    // 8-column (16-byte) units of the chunk
        const uint32_t* vc = &v[0];
        if constexpr (kNumAccum == 1) {
          vc = &v[64 * ch];
        } else {
          load_chunk(ch, v);
          if (ch == C::kChunksPerWarp - 1) {
            release();
          } else {
            tmem_load_wait();
          }
        }
        float f[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) f[i] = __uint_as_float(vc[i]);
        if constexpr (kOutF32) {
          // FP32: 32-column halves, one 128-byte swizzled TMA box each (tm_d); a 16-column
          // half (the end of a 240-wide tile) as plain 64-byte rows (tm_d_tail)
          const int width = tail ? C::kTail : 64;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int hw = width - 32 * h < 32 ? width - 32 * h : 32;
            if (hw <= 0) break;
            const int hcol = col + 32 * h;
            if (lane == 0) bulk_wait_group_read<0>();
            __syncwarp();
            if constexpr (kHasC) {
              // C arrives by TMA in the swizzled layout, each lane adds its row; the output
              // may use another layout: sync in between
              if (ch != 0 || h != 0) {
                issue_c_box(n0 + hcol);
                wait_c_box();
              }
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                if (n0 + hcol + 4 * q < p.N) {   // (past N nothing is stored)
                  const uint4 cv = ld_shared_v4(smem_addr(sbuf) + lane * 128 + ((q ^ (lane & 7)) * 16));
                  f[32 * h + 4 * q + 0] = __uint_as_float(cv.x) + f[32 * h + 4 * q + 0];
                  f[32 * h + 4 * q + 1] = __uint_as_float(cv.y) + f[32 * h + 4 * q + 1];
                  f[32 * h + 4 * q + 2] = __uint_as_float(cv.z) + f[32 * h + 4 * q + 2];
                  f[32 * h + 4 * q + 3] = __uint_as_float(cv.w) + f[32 * h + 4 * q + 3];
                }
              }
              __syncwarp();
            }
            const bool narrow = hw < 32;
            const uint32_t srow = smem_addr(sbuf) + lane * (narrow ? 64 : 128);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              if (4 * u < hw)
                st_shared_v4(srow + (narrow ? u * 16 : (u ^ (lane & 7)) * 16), __float_as_uint(f[32 * h + 4 * u]),
                             __float_as_uint(f[32 * h + 4 * u + 1]), __float_as_uint(f[32 * h + 4 * u + 2]),
                             __float_as_uint(f[32 * h + 4 * u + 3]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if constexpr (kKind == Kind::KGrouped) {
                tma_store_3d(&tm_d, sbuf, n0 + hcol, m_blk * BLOCK_M + quad * 32, seg.g);
              } else {
                tma_store_2d(narrow ? &tm_d_tail : &tm_d, sbuf, n0 + hcol, m_blk * BLOCK_M + quad * 32);
              }
              bulk_commit_group();
            }
          }
          continue;
        }
        if constexpr (C::kSmallEpi) {
          // 32-column pieces through the 2 KB staging buffer: 64-byte rows in the 64-byte
          // swizzle of tm_d (16-byte unit u of row r at r * 64 + (u ^ ((r >> 1) & 3)) * 16);
          // the 16-column end of a 240-wide tile as plain 32-byte rows (tm_d_tail)
          const int width = tail ? C::kTail : 64;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int pw = width - 32 * h < 32 ? width - 32 * h : 32;   // columns of this piece
            if (pw <= 0) break;
            const int pcol = col + 32 * h;
            if (lane == 0) bulk_wait_group_read<0>();   // the previous piece's store has read sbuf
            __syncwarp();
            const bool narrow = pw < 32;
            const uint32_t srow = smem_addr(sbuf) + lane * (narrow ? 32 : 64);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (8 * u < pw) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const __nv_bfloat162 b2 =
                      __floats2bfloat162_rn(f[32 * h + 8 * u + 2 * e], f[32 * h + 8 * u + 2 * e + 1]);
                  w[e] = *reinterpret_cast<const uint32_t*>(&b2);
                }
                st_shared_v4(srow + (narrow ? u * 16 : (u ^ ((lane >> 1) & 3u)) * 16), w[0], w[1], w[2], w[3]);
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (kKind == Kind::Dense || ok_mask == 0xffffffffu) {
              if (lane == 0) {
                tma_store_2d(narrow ? &tm_d_tail : &tm_d, sbuf, n0 + pcol, m_blk * BLOCK_M + quad * 32);
                bulk_commit_group();
              }
            } else if (ok_mask != 0) {
              // only the expert's rows: two rows per pass, 16 lanes x 4 bytes per row
              const int l = static_cast<int>(lane & 15u);
              const int gcol = n0 + pcol + 2 * l;
#pragma unroll 1
              for (int r0 = 0; r0 < 32; r0 += 2) {
                const int r = r0 + static_cast<int>(lane >> 4);
                const long long drow = __shfl_sync(0xffffffffu, d_row, r);
                if (((ok_mask >> r) & 1u) && 2 * l < pw && gcol < p.N) {
                  const uint32_t off = narrow ? r * 32 + l * 4
                                              : r * 64 + ((static_cast<uint32_t>(l) / 4) ^ ((r >> 1) & 3u)) * 16 +
                                                    (l % 4) * 4;
                  const uint32_t val = ld_shared_u32(smem_addr(sbuf) + off);
                  *reinterpret_cast<uint32_t*>(p.d + drow * p.N + gcol) = val;
                }
              }
              __syncwarp();
            }
          }
          continue;
        }
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
        if constexpr (kHasC) {
          // C arrives by TMA (a full 64-column box, also for the narrow last chunk), each lane
          // adds its row; the narrow chunk's output layout differs: sync before it is written
          if (ch != 0) {
            issue_c_box(n0 + col);
            wait_c_box();
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (q < units && n0 + col + 8 * q < p.N) {   // (past the tile or N nothing is stored)
              const uint4 cv = ld_shared_v4(smem_addr(sbuf) + lane * 128 + ((q ^ (lane & 7)) * 16));
              const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 cf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&cw[e]));
                f[8 * q + 2 * e] = cf.x + f[8 * q + 2 * e];
                f[8 * q + 2 * e + 1] = cf.y + f[8 * q + 2 * e + 1];
              }
            }
          }
          __syncwarp();
        }
        // staging: 64-column chunks in the 128-byte-swizzled layout of tm_d; the narrower
        // last chunk as plain rows of kTail * 2 bytes (tm_d_tail, no swizzle)
        const uint32_t srow = smem_addr(sbuf) + lane * (tail ? C::kTail * 2 : 128);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (u < units) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(f[8 * u + 2 * e], f[8 * u + 2 * e + 1]);
              w[e] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            st_shared_v4(srow + (tail ? u * 16 : (u ^ (lane & 7)) * 16), w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (kKind == Kind::Dense || ok_mask == 0xffffffffu) {
          if (lane == 0) {
            tma_store_2d(tail ? &tm_d_tail : &tm_d, sbuf, n0 + col, m_blk * BLOCK_M + quad * 32);
            bulk_commit_group();
          }
        } else if (ok_mask != 0) {
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
      }
    }
    if (lane == 0) bulk_wait_group_all();
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();
  if (*abort_flag) {
    // an aborted pair may still have a peer's copy in flight towards this CTA: let it land
    for (int i = 0; i < 1000; ++i) nanosleep_ns(1000);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

// Scale words -> tcgen05.cp source chunks, for A and B in one launch. For each (group,
// K-quad, 128-row block of A) a 512-byte chunk whose row j (16 bytes) holds the words of rows
// j, j+32, j+64, j+96 of the block. B holds one word per 128-row block; its chunks follow
// BN-wide tiles instead: chunk 2t + c covers tile rows 128c..128c+127 of tile t (rows
// t*BN + 128c + ...), each row carrying the word of the block it falls in, so that a tile
// may start inside a scale block. Launched as a programmatic dependent of the previous
// kernel in the stream (waits for it before reading or writing global memory).
struct SfPrepArgs {
  // contiguous form: the pair rows (built by the last block of the launch), else null
  const int32_t* m_indices;
  int num_mb, groups_g;
  int* pair_list;       // [num_mb][3]: first block, expert, own blocks (1 or 2)
  int* pair_count;
  uint32_t* status;
  const int32_t* sfa;   // [KP][lda] words
  int32_t* sfa_out;     // [KP][a_blocks][128]
  int a_rows, lda, a_blocks;
  const int32_t* sfb;   // [G][b_kp][ldb] words
  int32_t* sfb_out;     // [G][b_kp][b_chunks][128]
  int groups, b_rows, ldb, b_chunks, tile_bn;
  int kp;               // A's word rows (K-quads)
  int b_kp;             // B's word rows: K-quads (one word per 128-row block), or K-groups with
  int b_per_row;        // b_per_row set (FP4 B: one word per row, its four 32-wide blocks)
};

// Pair rows of the contiguous layout, by one block: block b (of 128 rows) belongs to the
// expert in m_indices[128 b] (outside [0, G): not computed, and reported unless it is -1);
// runs of consecutive blocks of one expert are cut into pairs from the run's first block. A
// block starts a pair iff it is valid and an even distance from its run's first block; pair
// rows are numbered by an exclusive prefix sum of those starts (two block-wide scans per
// chunk of blockDim.x blocks, carried across chunks).
__device__ void build_pair_list(const SfPrepArgs& a) {
  __shared__ int s_g[256 + 1];
  __shared__ int s_scan[256];
  const int tid = threadIdx.x;
  const int nt = blockDim.x;   // 256
  int run_start_carry = -1;    // first block of the run the previous chunk ended in
  int prev_g = -2;             // expert of the block before this chunk
  int count_carry = 0;
  auto expert = [&](int b) {
    const int g = ld_cg_s32(a.m_indices + static_cast<long long>(b) * 128);
    return (g >= 0 && g < a.groups_g) ? g : -1;
  };
  for (int base = 0; base < a.num_mb; base += nt) {
    const int b = base + tid;
    const bool in = b < a.num_mb;
    int raw = -1;
    if (in) {
      raw = ld_cg_s32(a.m_indices + static_cast<long long>(b) * 128);
      if (raw < -1 || raw >= a.groups_g) atomicOr(a.status, kStatusBadIndexBit);
    }
    const int g = in && raw >= 0 && raw < a.groups_g ? raw : -1;
    s_g[tid + 1] = g;
    if (tid == 0) s_g[0] = prev_g;
    __syncthreads();
    // run starts: a valid block whose predecessor has another expert
    int rs = (g >= 0 && s_g[tid] != g) ? b : -1;
    s_scan[tid] = rs;
    __syncthreads();
    for (int off = 1; off < nt; off <<= 1) {           // inclusive prefix max
      const int v = tid >= off ? s_scan[tid - off] : -1;
      __syncthreads();
      s_scan[tid] = max(s_scan[tid], v);
      __syncthreads();
    }
    const int run_start = max(s_scan[tid], run_start_carry);
    const bool start = g >= 0 && ((b - run_start) % 2 == 0);
    const int last_rs = s_scan[nt - 1];
    __syncthreads();
    s_scan[tid] = start ? 1 : 0;
    __syncthreads();
    for (int off = 1; off < nt; off <<= 1) {           // inclusive prefix sum
      const int v = tid >= off ? s_scan[tid - off] : 0;
      __syncthreads();
      s_scan[tid] += v;
      __syncthreads();
    }
    if (start) {
      const int idx = count_carry + s_scan[tid] - 1;
      const int own = (b + 1 < a.num_mb && expert(b + 1) == g) ? 2 : 1;
      a.pair_list[3 * idx + 0] = b;
      a.pair_list[3 * idx + 1] = g;
      a.pair_list[3 * idx + 2] = own;
    }
    const int chunk_count = s_scan[nt - 1];
    run_start_carry = max(run_start_carry, last_rs);
    prev_g = s_g[nt];
    __syncthreads();
    count_carry += chunk_count;
    // a run that ended inside this chunk must not leak into the next one: the next chunk's
    // first valid block restarts its run whenever its expert differs from prev_g, which the
    // run-start flags above take care of; run_start_carry only matters for a continuing run
  }
  if (tid == 0) *a.pair_count = count_carry;
}

__global__ void sf_to_utccp_kernel(const SfPrepArgs a) {
  grid_dependency_wait();
  grid_launch_dependents();
  const bool list_block = a.m_indices != nullptr && blockIdx.x == gridDim.x - 1;
  if (list_block) {
    build_pair_list(a);
    return;
  }
  const int sf_blocks = gridDim.x - (a.m_indices != nullptr ? 1 : 0);
  const long long na = static_cast<long long>(a.kp) * a.a_blocks * 128;
  const long long total = na + static_cast<long long>(a.groups) * a.b_kp * a.b_chunks * 128;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(sf_blocks) * blockDim.x) {
    int32_t val = 0;
    if (idx < na) {
      const int w = static_cast<int>(idx % 128);
      const long long chunk = idx / 128;              // q * a_blocks + b
      const int b = static_cast<int>(chunk % a.a_blocks);
      const long long q = chunk / a.a_blocks;
      const int row = b * 128 + 32 * (w % 4) + w / 4;
      if (row < a.a_rows) val = ld_cg_s32(a.sfa + q * a.lda + row);
      a.sfa_out[idx] = val;
    } else {
      const long long j = idx - na;
      const int w = static_cast<int>(j % 128);
      const long long chunk = j / 128;                // (g * b_kp + q) * b_chunks + c
      const int c = static_cast<int>(chunk % a.b_chunks);
      const long long gq = chunk / a.b_chunks;
      const int row = (c / 2) * a.tile_bn + (c % 2) * 128 + 32 * (w % 4) + w / 4;
      if (row < a.b_rows) val = ld_cg_s32(a.sfb + gq * a.ldb + (a.b_per_row ? row : row / 128));
      a.sfb_out[j] = val;
    }
  }
}

}  // namespace dg
