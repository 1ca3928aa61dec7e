// CTA-pair variant of the fine-grained-scaled FP8 GEMM for sm_103a: two CTAs of a
// cluster share one tcgen05.mma.cta_group::2 of shape 256 x 256 (x 32).
//
// Each CTA of the pair holds 128 rows of A and 128 of the 256 rows of the B tile in its
// own shared memory; the pair's MMA reads both and each CTA's TMEM receives its 128 x 256
// block of the accumulator. Per SM this halves the B bytes loaded and stored in shared
// memory per FLOP compared with a 128 x 256 tile on one SM, which is what bounds the
// single-CTA kernel on GB300 (L2->SM traffic and bytes in flight).
//
// Roles (both CTAs run the same code):
//   warp 0      TMA producer: its own A rows, its own half of B and the scale chunks,
//               counted on the full barrier of the leader CTA (rank 0).
//   warp 1      allocates TMEM for the pair; in the leader one thread copies the scale
//               chunks into TMEM (tcgen05.cp.cta_group::2) and issues the MMAs, then
//               commits to the empty / accumulator-full barriers of both CTAs.
//   warps 2..9  epilogue: each reads its 32 TMEM lanes x 128 columns into registers,
//               hands the accumulator back to the leader, then adds C, rounds to BF16 and
//               TMA-stores (or stores valid rows only).
// The scale words are consumed in the tcgen05.cp source layout, produced beforehand in a
// workspace by sf_to_utccp_kernel (one 512-byte chunk per 128 rows per 4 K-groups).
// Operation: D = C + A @ B.T (DeepGEMM README "Interfaces / Notices", "Normal dense GEMMs",
// "Grouped GEMMs (contiguous layout)", as reproduced on the page "Weight gradient kernels
// for dense and MoE models #95").
#pragma once

#include "fp8_gemm.cuh"

namespace dg {

template <int kStages>
struct PairConfig {
  static constexpr int BN = 256;                 // tile width of the pair; each CTA loads BN/2 B rows
  static constexpr int kEpiWarps = 8;            // two per TMEM sub-partition, 128 columns each
  static constexpr int kThreads = (2 + kEpiWarps) * 32;
  static constexpr int A_BYTES = BLOCK_M * BLOCK_K;
  static constexpr int B_BYTES = (BN / 2) * BLOCK_K;
  static constexpr int SFA_BYTES = 512;          // one tcgen05.cp chunk: this CTA's 128 rows
  static constexpr int SFB_BYTES = 1024;         // two chunks: the 256 columns of the pair tile
  static constexpr int SF_STRIDE = 2048;
  static constexpr int EPI_BUF_BYTES = 32 * 128;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + kStages * A_BYTES;
  static constexpr int OFF_SF = OFF_B + kStages * B_BYTES;
  static constexpr int OFF_EPI = ((OFF_SF + kStages * SF_STRIDE + 1023) / 1024) * 1024;
  static constexpr int OFF_BAR = OFF_EPI + kEpiWarps * EPI_BUF_BYTES;
  static constexpr int NUM_BARS = 2 * kStages + 3;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
  static constexpr int TX_AB = 2 * (A_BYTES + B_BYTES);           // both CTAs, every stage
  static constexpr int TX_SF = 2 * (SFA_BYTES + SFB_BYTES);       // both CTAs, every 4th stage
  // TMEM: one 256-column accumulator, then 2 x 4 SFA columns and 2 x 8 SFB columns
  static constexpr int SFA_COL = BN;
  static constexpr int SFB_COL = BN + 8;
  static constexpr int TMEM_COLS = 512;
};

// Walks the pair tiles of the sequence t = cluster, += clusters. A pair row is two
// consecutive 128-row blocks; in the contiguous form both blocks belong to one expert
// (an expert with an odd number of blocks ends with a pair whose second block is not its
// own: that CTA's rows are computed and discarded).
template <Kind kKind>
struct PairScheduler {
  int num_n, num_mb, total;
  int t, step;
  // contiguous cursor
  int cur_pair, cur_block;

  __device__ __forceinline__ int expert_of(const Params& p, int b) const {
    if (b >= num_mb) return -1;
    const int g = __ldg(p.m_indices + b * BLOCK_M);
    return (g >= 0 && g < p.G) ? g : -1;
  }
  __device__ __forceinline__ int pair_len(const Params& p, int b, int g) const {
    return (b + 1 < num_mb && expert_of(p, b + 1) == g) ? 2 : 1;
  }

  __device__ __forceinline__ PairScheduler(const Params& p, int cluster, int clusters) {
    num_n = ceil_div_c(p.N, PairConfig<1>::BN);
    num_mb = ceil_div_c(p.M, BLOCK_M);
    t = cluster;
    step = clusters;
    cur_pair = 0;
    cur_block = 0;
    if constexpr (kKind == Kind::Contiguous) {
      int pairs = 0;
      for (int b = 0; b < num_mb;) {
        const int g = expert_of(p, b);
        if (g < 0) {
          // a block led by an index outside [-1, G) is skipped and reported (once, by CTA 0)
          if (blockIdx.x == 0 && threadIdx.x == 0) {
            const int raw = __ldg(p.m_indices + b * BLOCK_M);
            if (raw < -1 || raw >= p.G) atomicOr(p.status, kStatusBadIndexBit);
          }
          ++b;
          continue;
        }
        b += pair_len(p, b, g);
        ++pairs;
      }
      total = pairs * num_n;
    } else {
      total = ceil_div_c(num_mb, 2) * num_n;
    }
  }

  // seg.m_blk is the pair's first block; the CTA of rank r works on block m_blk + r.
  __device__ __forceinline__ bool next(const Params& p, Segment& s) {
    if (t >= total) return false;
    const int pair = t / num_n;
    s.n_blk = t % num_n;
    t += step;
    s.kb_begin = 0;
    s.kb_end = p.K / BLOCK_K;
    s.n_contrib = 1;
    s.slot = 0;
    s.tile = pair;
    s.valid_m = p.M;
    if constexpr (kKind == Kind::Contiguous) {
      // advance the cursor to the pair with index `pair` (indices only grow)
      while (true) {
        int g = expert_of(p, cur_block);
        while (g < 0) {
          if (++cur_block >= num_mb) return false;
          g = expert_of(p, cur_block);
        }
        if (cur_pair == pair) {
          s.g = g;
          s.m_blk = cur_block;
          s.n_contrib = pair_len(p, cur_block, g);   // blocks of this pair that belong to the expert
          return true;
        }
        cur_block += pair_len(p, cur_block, g);
        ++cur_pair;
      }
    } else {
      s.g = 0;
      s.m_blk = 2 * pair;
      return true;
    }
  }
};

template <Kind kKind, int kStages, bool kHasC>
__global__ void __launch_bounds__(PairConfig<kStages>::kThreads, 1)
    fp8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                         const __grid_constant__ CUtensorMap tm_sfa, const __grid_constant__ CUtensorMap tm_sfb,
                         const __grid_constant__ CUtensorMap tm_d, const Params p) {
  static_assert(kKind != Kind::Masked, "the masked form uses the single-CTA kernel");
  using C = PairConfig<kStages>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full_bar = bars;                    // used in the leader only
  uint64_t* empty_bar = bars + kStages;         // both CTAs (leader's commit, multicast)
  uint64_t* tfull_bar = bars + 2 * kStages;     // both CTAs (leader's commit, multicast)
  uint64_t* tempty_bar = bars + 2 * kStages + 1;  // leader: 8 epilogue warps x 2 CTAs
  uint64_t* drain_bar = bars + 2 * kStages + 2;
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
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, 2 * C::kEpiWarps);
    mbar_init(drain_bar, 1);
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

  PairScheduler<kKind> sched(p, static_cast<int>(blockIdx.x / 2), static_cast<int>(gridDim.x / 2));
  Segment seg;

  if (warp == 0) {
    // ================================ TMA producer (both CTAs) ====================
    if (lane == 0 && p.fault != kFaultProducerSilent) {
      uint32_t stage = 0, phase = 0, issued = 0;
      while (sched.next(p, seg)) {
        const int m_blk = seg.m_blk + static_cast<int>(rank);
        const int n0 = seg.n_blk * C::BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (*abort_flag || !mbar_wait(&empty_bar[stage], phase ^ 1, p.timeout_ns)) {
            on_timeout();
            goto producer_done;
          }
          const bool with_sf = (kb % 4) == 0;
          const uint32_t fb = map_to_rank(&full_bar[stage], 0);
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], C::TX_AB + (with_sf ? C::TX_SF : 0));
          uint8_t* sa = smem + C::OFF_A + stage * C::A_BYTES;
          uint8_t* sb = smem + C::OFF_B + stage * C::B_BYTES;
          uint8_t* ssf = smem + C::OFF_SF + stage * C::SF_STRIDE;
          tma_load_2d_pair(sa, &tm_a, fb, kb * BLOCK_K, m_blk * BLOCK_M);
          if constexpr (kKind == Kind::Dense) {
            tma_load_2d_pair(sb, &tm_b, fb, kb * BLOCK_K, n0 + static_cast<int>(rank) * (C::BN / 2));
          } else {
            tma_load_3d_pair(sb, &tm_b, fb, kb * BLOCK_K, n0 + static_cast<int>(rank) * (C::BN / 2), seg.g);
          }
          if (with_sf) {
            const int q = kb / 4;
            // SFA chunk row: (q, m_blk); SFB chunk rows: (g, q, n-block) and the next one
            tma_load_2d_pair(ssf, &tm_sfa, fb, 0, q * p.sf_num_mb + m_blk);
            tma_load_2d_pair(ssf + C::SFA_BYTES, &tm_sfb, fb, 0,
                             (seg.g * KP + q) * p.sf_nb + n0 / SF_BLOCK_N);
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
      constexpr uint32_t kIdesc = make_idesc_mxf8_e4m3(2 * BLOCK_M, C::BN);
      const uint64_t a_desc0 = make_smem_desc(smem_addr(smem + C::OFF_A), 16, 1024, kLayoutSwizzle128B);
      const uint64_t b_desc0 = make_smem_desc(smem_addr(smem + C::OFF_B), 16, 1024, kLayoutSwizzle128B);
      const uint64_t sf_desc0 = make_smem_desc(smem_addr(smem + C::OFF_SF), 0, 128, kLayoutNone);
      uint32_t stage = 0, phase = 0, tile_iter = 0, sf_iter = 0;
      while (sched.next(p, seg)) {
        if (*abort_flag || !mbar_wait(tempty_bar, (tile_iter & 1) ^ 1, p.timeout_ns)) {
          on_timeout();
          goto mma_done;
        }
        tc_fence_after();
        {
          uint32_t sfa_tmem = 0, sfb_tmem = 0;
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!mbar_wait(&full_bar[stage], phase, p.timeout_ns)) {
              on_timeout();
              goto mma_done;
            }
            tc_fence_after();
            if (kb % 4 == 0) {
              const uint32_t buf = sf_iter & 1;
              ++sf_iter;
              sfa_tmem = tmem_base + C::SFA_COL + 4 * buf;
              sfb_tmem = tmem_base + C::SFB_COL + 8 * buf;
              const uint64_t sf_desc = sf_desc0 + ((stage * C::SF_STRIDE) >> 4);
              tmem_copy_32x128b_warpx4_pair(sfa_tmem, sf_desc);
              tmem_copy_32x128b_warpx4_pair(sfb_tmem, sf_desc + (C::SFA_BYTES >> 4));
              tmem_copy_32x128b_warpx4_pair(sfb_tmem + 4, sf_desc + ((C::SFA_BYTES + 512) >> 4));
            }
            const uint64_t adesc = a_desc0 + ((stage * C::A_BYTES) >> 4);
            const uint64_t bdesc = b_desc0 + ((stage * C::B_BYTES) >> 4);
            const uint32_t idesc = idesc_with_sf_id(kIdesc, kb % 4, kb % 4);
#pragma unroll
            for (int k = 0; k < BLOCK_K / 32; ++k)
              mma_mxf8_block_scale_pair(tmem_base, adesc + 2 * k, bdesc + 2 * k, idesc, sfa_tmem, sfb_tmem,
                                        (kb | k) != 0);
            tc_commit_pair(&empty_bar[stage]);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
        tc_commit_pair(tfull_bar);
        ++tile_iter;
      }
    mma_done:
      tc_commit_pair(drain_bar);
      mbar_wait(drain_bar, 0, 50000000ull);
    }
    __syncwarp();
  } else {
    // ================================ epilogue (both CTAs) ==========================
    const int ew = warp - 2;
    const int quad = warp % 4;
    const int half = ew / 4;                       // columns [128 * half, 128 * half + 128)
    uint8_t* sbuf = smem + C::OFF_EPI + ew * C::EPI_BUF_BYTES;
    const uint32_t tempty_leader = map_to_rank(tempty_bar, 0);
    uint32_t tile_iter = 0;
    while (sched.next(p, seg)) {
      if (!warp_wait(tfull_bar, tile_iter & 1, p.timeout_ns, abort_flag)) {
        if (lane == 0) on_timeout();
        break;
      }
      ++tile_iter;
      tc_fence_after();
      // the whole share of the accumulator into registers, then hand TMEM back at once
      uint32_t v[128];
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + 128 * half;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t (&vj)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32 * j]);
        tmem_load_32x32b_x32(taddr + 32 * j, vj);
      }
      tmem_load_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader);

      const int m_blk = seg.m_blk + static_cast<int>(rank);
      const int row = m_blk * BLOCK_M + quad * 32 + static_cast<int>(lane);
      bool row_ok;
      if constexpr (kKind == Kind::Dense) {
        row_ok = row < p.M;
      } else {
        const int gi = row < p.M ? __ldg(p.m_indices + row) : -1;
        row_ok = gi == seg.g;
        // a row of the expert's own blocks that names another expert violates the layout
        if (gi != seg.g && gi != -1 && static_cast<int>(rank) < seg.n_contrib && seg.n_blk == 0 && half == 0)
          atomicOr(p.status, kStatusBadIndexBit);
      }
      const uint32_t ok_mask = __ballot_sync(0xffffffffu, row_ok);
      const long long d_row = row;
      const int n0 = seg.n_blk * C::BN;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int col = 128 * half + 64 * ch;
        float f[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) f[i] = __uint_as_float(v[64 * ch + i]);
        if constexpr (kHasC) {
          if (row_ok) {
            const __nv_bfloat16* crow = p.c + d_row * p.N + n0 + col;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              if (n0 + col + 8 * q < p.N) {
                const uint4 cv = ld_global_nc_v4(crow + 8 * q);
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
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
        const uint32_t srow = smem_addr(sbuf) + lane * 128;
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
            tma_store_2d(&tm_d, sbuf, n0 + col, m_blk * BLOCK_M + quad * 32);
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

// Scale words -> tcgen05.cp source chunks. For each (group, K-quad, 128-row block) a
// 512-byte chunk whose row j (16 bytes) holds the words of rows j, j+32, j+64, j+96 of
// the block. With `per_block` set the input holds one word per 128-row block (B scales)
// and every row of the chunk repeats it.
__global__ void sf_to_utccp_kernel(const int32_t* __restrict__ sf, int32_t* __restrict__ out, int groups, int kp,
                                   int mn, int ld, int blocks, int per_block) {
  const long long total = static_cast<long long>(groups) * kp * blocks * 128;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int w = static_cast<int>(idx % 128);
    const long long chunk = idx / 128;              // (g * kp + q) * blocks + b
    const int b = static_cast<int>(chunk % blocks);
    const long long gq = chunk / blocks;            // g * kp + q
    int32_t val = 0;
    if (per_block) {
      if (b < mn) val = __ldg(sf + gq * ld + b);
    } else {
      const int row = b * 128 + 32 * (w % 4) + w / 4;
      if (row < mn) val = __ldg(sf + gq * ld + row);
    }
    out[idx] = val;
  }
}

}  // namespace dg
