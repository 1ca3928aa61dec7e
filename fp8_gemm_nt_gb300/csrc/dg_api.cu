// Host side of libdg: argument validation, TMA descriptor construction, kernel
// selection and launch, the scale-packing kernel and the device status word.
// The C ABI is declared (and documented) in include/dg.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "debug_state.h"
#include "dg.h"
#include "fp8_gemm.cuh"
#include "fp8_gemm_pair.cuh"
#include "workspace_cache.h"

namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<int> g_num_sms_cap{0};
std::atomic<int> g_mk_alignment{128};   // what callers are told to pad expert segments to
std::atomic<int> g_fault{0};
std::atomic<unsigned long long> g_timeout_ns{0};

constexpr int kMaxDevices = 64;
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;   // 2 s per pipeline wait
constexpr int kMinKGroupsPerCta = 4;                            // stream-K: smallest share per CTA
constexpr size_t kSkCounterInts = 4096;                         // stream-K arrival counters per workspace
constexpr size_t kMaxWorkspaces = 16;                           // freeable cached workspaces, per device

// The CUDA runtime calls the workspace cache policy (workspace_cache.h) is written against.
struct CudaApi {
  using Stream = cudaStream_t;
  using Event = cudaEvent_t;
  static int is_capturing(Stream s, bool* capturing) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(s, &st);
    *capturing = st != cudaStreamCaptureStatusNone;
    return static_cast<int>(e);
  }
  static int malloc(void** p, size_t n) { return static_cast<int>(cudaMalloc(p, n)); }
  static int malloc_async(void** p, size_t n, Stream s) { return static_cast<int>(cudaMallocAsync(p, n, s)); }
  static int free_async(void* p, Stream s) { return static_cast<int>(cudaFreeAsync(p, s)); }
  static int memset_async(void* p, size_t n, Stream s) { return static_cast<int>(cudaMemsetAsync(p, 0, n, s)); }
  static int event_create(Event* e) { return static_cast<int>(cudaEventCreateWithFlags(e, cudaEventDisableTiming)); }
  static int event_destroy(Event e) { return static_cast<int>(cudaEventDestroy(e)); }
  static int event_record(Event e, Stream s) { return static_cast<int>(cudaEventRecord(e, s)); }
  static int stream_wait_event(Stream s, Event e) { return static_cast<int>(cudaStreamWaitEvent(s, e, 0)); }
};

struct DeviceState {
  bool ready = false;
  bool supported = false;
  int num_sms = 0;
  uint32_t* status = nullptr;
  dg::WorkspaceCache<cudaStream_t, cudaEvent_t> workspaces;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mutex;

dg_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return DG_ERR_CUDA;
}

// Per-device set-up (once): capability check, SM count, the status word.
dg_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return DG_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return cuda_fail(e);
    s.supported = (major == 10 && minor == 3);
    if (s.supported) {
      if ((e = cudaMalloc(&s.status, sizeof(uint32_t))) != cudaSuccess) return cuda_fail(e);
      if ((e = cudaMemset(s.status, 0, sizeof(uint32_t))) != cudaSuccess) return cuda_fail(e);
    }
    s.ready = true;
  }
  if (!s.supported) return DG_ERR_UNSUPPORTED;
  *out = &s;
  return DG_OK;
}

int sms_to_use(const DeviceState& s) {
  const int cap = g_num_sms_cap.load();
  return (cap > 0 && cap < s.num_sms) ? cap : s.num_sms;
}

unsigned long long wait_timeout_ns() {
  const unsigned long long t = g_timeout_ns.load();
  return t ? t : kWaitTimeoutNs;
}

// The parameter block every launch shares: the problem shape, C and D (BF16, or FP32 for the
// weight-gradient forms, which the kernels reinterpret), the device status word, the wait
// limit and the failure-injection switch.
dg::Params base_params(const DeviceState& ds, int M, int N, int K, int G, const void* c, void* d) {
  dg::Params p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.G = G;
  p.c = static_cast<const __nv_bfloat16*>(c);
  p.d = static_cast<__nv_bfloat16*>(d);
  p.status = ds.status;
  p.timeout_ns = wait_timeout_ns();
  p.fault = g_fault.load();
  return p;
}

// A workspace pointer and the lock that keeps it valid. Workspaces are freed only under
// g_mutex, in stream order after their last use (an event recorded once the kernels that use
// them are enqueued). A caller therefore holds the lease until its kernels are launched and
// done() has recorded that point: another host thread cannot evict the memory in between.
struct WorkspaceLease {
  void* ptr = nullptr;
  DeviceState* ds = nullptr;
  size_t index = 0;
  cudaStream_t stream = nullptr;
  std::unique_lock<std::mutex> lock;

  // After the launches that use the workspace are enqueued (also on a failed launch).
  void done() {
    if (ds && lock.owns_lock()) {
      dg::release<CudaApi>(ds->workspaces, index, stream);
      lock.unlock();
    }
  }
  ~WorkspaceLease() { done(); }
};

// Workspace of at least `bytes` for `stream` (policy in workspace_cache.h): allocated in
// stream order on the first call that needs it (or by dg_reserve_workspace), never with a
// device or stream synchronisation. The stream-K arrival counters at its start are zero when
// allocated and left at zero by every completed launch.
dg_status stream_workspace(DeviceState& ds, cudaStream_t stream, size_t bytes, WorkspaceLease* out) {
  std::unique_lock<std::mutex> lock(g_mutex);
  void* ptr = nullptr;
  size_t index = 0;
  if (const int e = dg::acquire<CudaApi, kMaxWorkspaces>(ds.workspaces, stream, bytes, &ptr, &index))
    return cuda_fail(static_cast<cudaError_t>(e));
  out->ptr = ptr;
  out->ds = &ds;
  out->index = index;
  out->stream = stream;
  out->lock = std::move(lock);
  return DG_OK;
}

// ------------------------------------------------------------------------------------
// TMA descriptors
// ------------------------------------------------------------------------------------
// Programmatic dependent launch: a GEMM may start its prologue while the previous kernel in
// the stream finishes; the kernels wait for that grid before touching global memory. On by
// default (the environment variable DG_PDL=0 makes the default off); dg_set_pdl changes it.
// -1: not yet initialised from the environment.
std::atomic<int> g_pdl{-1};

bool pdl_enabled() {
  int v = g_pdl.load();
  if (v < 0) {
    const char* f = std::getenv("DG_PDL");
    int expected = -1;
    g_pdl.compare_exchange_strong(expected, (f && f[0] == '0') ? 0 : 1);
    v = g_pdl.load();
  }
  return v != 0;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A small per-thread cache of encoded descriptors: repeated calls on the same buffers
// (the common case: weights, activations and outputs reused every step) skip the encode.
struct MapKey {
  const void* base;
  uint64_t dims[3];
  uint64_t strides[2];
  uint32_t box[3];
  int dt, rank, swz;
};

struct MapCacheEntry {
  MapKey key;
  CUtensorMap map;
  bool used;
};

constexpr int kMapCacheSize = 32;
thread_local MapCacheEntry g_map_cache[kMapCacheSize];
thread_local int g_map_cache_next = 0;

bool same_key(const MapKey& a, const MapKey& b) { return std::memcmp(&a, &b, sizeof(MapKey)) == 0; }

// dims/box innermost first; strides in bytes for dims 1..rank-1.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swz) {
  MapKey key;
  std::memset(&key, 0, sizeof(key));
  key.base = base;
  key.dt = static_cast<int>(dt);
  key.rank = rank;
  key.swz = static_cast<int>(swz);
  for (int i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) key.strides[i] = strides[i];
  for (int i = 0; i < kMapCacheSize; ++i) {
    if (g_map_cache[i].used && same_key(g_map_cache[i].key, key)) {
      *m = g_map_cache[i].map;
      return true;
    }
  }
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  cuuint64_t d[5], st[4];
  cuuint32_t b[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
  CUresult r = fn(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, st, b, elem_strides,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  MapCacheEntry& e = g_map_cache[g_map_cache_next];
  g_map_cache_next = (g_map_cache_next + 1) % kMapCacheSize;
  e.key = key;
  e.map = *m;
  e.used = true;
  return true;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline int ceil4(int x) { return 4 * ceil_div(x, 4); }

// ------------------------------------------------------------------------------------
// Kernel configurations
// ------------------------------------------------------------------------------------
template <dg::Kind kKind, int BN, int kStages, int kNumAccum, int kEpiWarps_, int kEpiBufs, bool kHasC,
          int kKG = 1, int kSplit = 0, bool kOutF32 = false, bool kAMN = false, bool kBMN = false, bool kBF4 = false>
struct Launcher {
  static constexpr int kEpiWarps = kEpiWarps_;
  using Cfg = dg::Config<BN, kStages, kNumAccum, kEpiWarps, kEpiBufs, kKG, kSplit, kBF4, dg::count_cache_for(kKind)>;
  static constexpr int kBN = BN;
  static constexpr auto kernel() {
    return dg::fp8_gemm_kernel<kKind, BN, kStages, kNumAccum, kEpiWarps, kEpiBufs, kHasC, kKG, kSplit, kOutF32,
                               kAMN, kBMN, kBF4>;
  }

  // Largest number of co-resident clusters of kSplit CTAs (0 if the kernel cannot run).
  static int max_clusters() {
    static thread_local int dev_cached = -1, value = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev == dev_cached) return value;
    auto kern = kernel();
    value = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = kSplit > 0 ? kSplit : 1;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(kSplit > 0 ? kSplit : 1, 1, 1);
      cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
      cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess) value = n;
    }
    cudaGetLastError();
    dev_cached = dev;
    return value;
  }

  static dg_status launch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                          const CUtensorMap& tsb, const CUtensorMap& td, const dg::Params& p, int grid,
                          cudaStream_t stream) {
    auto kern = kernel();
    static thread_local int attr_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_dev != dev) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
      if (e != cudaSuccess) return cuda_fail(e);
      attr_dev = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    int n_attr = 0;
    if (kSplit > 0) {
      attr[n_attr].id = cudaLaunchAttributeClusterDimension;
      attr[n_attr].val.clusterDim.x = kSplit;
      attr[n_attr].val.clusterDim.y = 1;
      attr[n_attr].val.clusterDim.z = 1;
      ++n_attr;
    }
    if (pdl_enabled()) {
      attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
      ++n_attr;
    }
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tsa, tsb, td, p);
    if (e != cudaSuccess) return cuda_fail(e);
    if (std::getenv("DG_PRINT_CONFIGS"))
      std::fprintf(stderr, "[dg] kind=%d M=%d N=%d K=%d G=%d BN=%d stages=%d accum=%d epi_warps=%d grid=%d smem=%d stream_k=%d split=%d kg=%d fp4=%d\n",
                   static_cast<int>(kKind), p.M, p.N, p.K, p.G, BN, kStages, kNumAccum, kEpiWarps, grid,
                   Cfg::SMEM_BYTES, p.sk_ctas, kSplit, kKG, kBF4 ? 1 : 0);
    return DG_OK;
  }
};

// Split-K over CTA pairs (clusters of two) for problems with too few tiles to fill the GPU:
// one 128 x BN tile per pair, each CTA half of K, two K-groups per 3-stage ring slot; the
// partials are summed through distributed shared memory (no workspace, no atomics).
constexpr int kSplitWays = 2;
template <bool kHasC, int BN, bool kBF4 = false>
using SplitLauncher = Launcher<dg::Kind::Dense, BN, 3, 1, 4, 1, kHasC, 2, kSplitWays, false, false, false, kBF4>;

template <bool kHasC, bool kBF4 = false>
int split_max_clusters(int bn) {
  switch (bn) {
    case 64: return SplitLauncher<kHasC, 64, kBF4>::max_clusters();
    case 96: return SplitLauncher<kHasC, 96, kBF4>::max_clusters();
    case 128: return SplitLauncher<kHasC, 128, kBF4>::max_clusters();
  }
  return 0;
}

template <bool kHasC, bool kBF4 = false>
dg_status launch_split(int bn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                       const CUtensorMap& tsb, const CUtensorMap& td, const dg::Params& p, int grid,
                       cudaStream_t stream) {
  switch (bn) {
    case 64: return SplitLauncher<kHasC, 64, kBF4>::launch(ta, tb, tsa, tsb, td, p, grid, stream);
    case 96: return SplitLauncher<kHasC, 96, kBF4>::launch(ta, tb, tsa, tsb, td, p, grid, stream);
    case 128: return SplitLauncher<kHasC, 128, kBF4>::launch(ta, tb, tsa, tsb, td, p, grid, stream);
  }
  return DG_ERR_INVALID_ARG;
}

// Split-K tile width for a problem with fewer 128 x 128 tiles than SMs: the narrowest of
// 64 / 96 / 128 whose tiles fit one per co-resident CTA pair, if that keeps at least 3/4
// of the SMs busy and gives each CTA two or more K-groups; 0 = use stream-K instead.
// DG_SPLIT=0 disables the split form, DG_SPLIT_BN forces a width (if it fits).
int pick_split_bn(int M, int N, int K, int sms, bool with_c, bool fp4 = false) {
  if (const char* f = std::getenv("DG_SPLIT")) {
    if (f[0] == '0') return 0;
  }
  int forced = 0;
  if (const char* f = std::getenv("DG_SPLIT_BN")) forced = std::atoi(f);
  if (K / 128 < 2 * kSplitWays) return 0;
  const long long m_blocks = ceil_div(M, 128);
  for (int bn : {64, 96, 128}) {
    if (forced && bn != forced) continue;
    const int max_cl = std::min(fp4 ? (with_c ? split_max_clusters<true, true>(bn) : split_max_clusters<false, true>(bn))
                                    : (with_c ? split_max_clusters<true>(bn) : split_max_clusters<false>(bn)),
                                sms / kSplitWays);
    const long long tiles = m_blocks * ceil_div(N, bn);
    if (max_cl > 0 && tiles <= max_cl && tiles * kSplitWays * 4 >= 3LL * sms) return bn;
  }
  return 0;
}

// Tile configurations (BN = tile width). All use 128-row tiles and 4 epilogue warps.
//   128: 5-stage ring, double-buffered accumulators (TMEM 2 x 128 columns)
//   192: 4-stage ring, double-buffered accumulators (TMEM 2 x 192 columns)
//   256: 4-stage ring, single accumulator (TMEM 256 columns; 2 x 256 + scales exceeds 512)
//   128 x 2: two K-groups per stage (64 KB stages, 3 of them), for HBM-bound stream-K shapes
//   FP4 B (kBF4): dense 128, 128 x 2 and 256; contiguous 128 and 256; masked 128 and 192
template <dg::Kind kKind, bool kHasC, bool kOutF32 = false, bool kAMN = false, bool kBMN = false, bool kBF4 = false>
dg_status launch_bn(int bn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                    const CUtensorMap& tsb, const CUtensorMap& td, const dg::Params& p, int grid,
                    cudaStream_t stream, int kgroups_per_stage = 1) {
  if constexpr (kBF4) {
    static_assert(!kOutF32 && !kAMN && !kBMN, "FP4 B: K-major operands, BF16 output");
    if constexpr (kKind == dg::Kind::Dense) {
      if (kgroups_per_stage == 2 && bn == 128)
        return Launcher<kKind, 128, 3, 2, 4, 1, kHasC, 2, 0, false, false, false, true>::launch(ta, tb, tsa, tsb, td,
                                                                                                  p, grid, stream);
    }
    if constexpr (kKind == dg::Kind::Masked) {
      if (bn == 192)
        return Launcher<kKind, 192, 4, 2, 4, 2, kHasC, 1, 0, false, false, false, true>::launch(ta, tb, tsa, tsb, td,
                                                                                                  p, grid, stream);
    }
    if (bn == 128)
      return Launcher<kKind, 128, 5, 2, 4, 2, kHasC, 1, 0, false, false, false, true>::launch(ta, tb, tsa, tsb, td, p,
                                                                                                grid, stream);
    if constexpr (kKind != dg::Kind::Masked) {
      if (bn == 256)
        return Launcher<kKind, 256, 4, 1, 4, 1, kHasC, 1, 0, false, false, false, true>::launch(ta, tb, tsa, tsb, td,
                                                                                                  p, grid, stream);
    }
    return DG_ERR_INVALID_ARG;
  }
  if constexpr (kKind == dg::Kind::Dense) {
    if (kgroups_per_stage == 2 && bn == 128)
      return Launcher<kKind, 128, 3, 2, 4, 1, kHasC, 2, 0, kOutF32, kAMN, kBMN>::launch(ta, tb, tsa, tsb, td, p, grid,
                                                                                        stream);
  }
  if constexpr (kAMN || kBMN) {
    // the MN-major layouts use 128- and 256-wide tiles (an N-major B tile is whole
    // 128-column atoms)
    switch (bn) {
      case 128:
        return Launcher<kKind, 128, 5, 2, 4, 2, kHasC, 1, 0, kOutF32, kAMN, kBMN>::launch(ta, tb, tsa, tsb, td, p,
                                                                                           grid, stream);
      case 256:
        return Launcher<kKind, 256, 4, 1, 4, 1, kHasC, 1, 0, kOutF32, kAMN, kBMN>::launch(ta, tb, tsa, tsb, td, p,
                                                                                           grid, stream);
    }
    return DG_ERR_INVALID_ARG;
  }
  switch (bn) {
    case 128: return Launcher<kKind, 128, 5, 2, 4, 2, kHasC, 1, 0, kOutF32>::launch(ta, tb, tsa, tsb, td, p, grid, stream);
    case 192: return Launcher<kKind, 192, 4, 2, 4, 2, kHasC, 1, 0, kOutF32>::launch(ta, tb, tsa, tsb, td, p, grid, stream);
    case 256: return Launcher<kKind, 256, 4, 1, 4, 1, kHasC, 1, 0, kOutF32>::launch(ta, tb, tsa, tsb, td, p, grid, stream);
  }
  return DG_ERR_INVALID_ARG;
}
constexpr int kEpilogueWarps = 4;

// CTA-pair configurations: 256 x BN tiles over two SMs; BN = 256 with one accumulator, BN = 240
// or 192 with two. Ring: 6 stages per CTA for BF16 output without C (32-column epilogue pieces
// leave the shared memory for it), 5 otherwise.
template <bool kHasC, bool kOutF32>
constexpr int pair_stages() { return (!kHasC && !kOutF32) ? 6 : 5; }

template <dg::Kind kKind, bool kHasC, int kBN, bool kOutF32 = false, bool kBF4 = false, bool kAMN = false,
          bool kBMN = false>
struct PairLauncher {
  static constexpr int kNumAccum = kBN == 256 ? 1 : 2;
  static constexpr int kStages = pair_stages<kHasC, kOutF32>();
  using Cfg = dg::PairConfig<kStages, kBN, kNumAccum, kBF4, !kHasC && !kOutF32>;
  static constexpr auto kernel() {
    return dg::fp8_gemm_pair_kernel<kKind, kStages, kBN, kNumAccum, kHasC, kOutF32, kBF4, kAMN, kBMN>;
  }

  // Largest number of co-resident CTA pairs (0 if the device cannot run the kernel).
  static int max_clusters() {
    static thread_local int dev_cached = -1, value = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev == dev_cached) return value;
    auto kern = kernel();
    value = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) == cudaSuccess &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2, 1, 1);
      cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
      cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess) value = n;
    }
    cudaGetLastError();
    dev_cached = dev;
    return value;
  }

  static dg_status launch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                          const CUtensorMap& tsb, const CUtensorMap& td, const CUtensorMap& td_tail,
                          const CUtensorMap& tc, const dg::Params& p, int clusters, cudaStream_t stream) {
    auto kern = kernel();
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tsa, tsb, td, td_tail, tc, p);
    if (e != cudaSuccess) return cuda_fail(e);
    if (std::getenv("DG_PRINT_CONFIGS"))
      std::fprintf(stderr, "[dg] kind=%d M=%d N=%d K=%d G=%d pair 256x%d accum=%d stages=%d clusters=%d smem=%d fp4=%d\n",
                   static_cast<int>(kKind), p.M, p.N, p.K, p.G, kBN, kNumAccum, kStages, clusters,
                   Cfg::SMEM_BYTES, kBF4 ? 1 : 0);
    return DG_OK;
  }
};

bool pair_enabled() {
  const char* f = std::getenv("DG_PAIR");
  return !(f && f[0] == '0');
}



// Tile width for a problem: DG_FORCE_BN (128, 192 or 256) overrides the heuristic.
// Measured on GB300 (tile mode): wider tiles cut the L2->SM bytes per FLOP, which is what
// limits the 128-wide configuration, so the widest tile that wastes no more columns than
// the narrower ones wins; the masked form (short K, HBM-bound) prefers 192 with its
// double-buffered accumulators.
int pick_bn(dg::Kind kind, int N) {
  if (const char* f = std::getenv("DG_FORCE_BN")) {
    const int v = std::atoi(f);
    if (v == 128 || v == 192 || v == 256) return v;
  }
  if (kind == dg::Kind::Masked) return N > 128 ? 192 : 128;
  const int cands[3] = {256, 192, 128};
  int best = 256;
  long long best_cols = -1;
  for (int bn : cands) {
    const long long cols = static_cast<long long>(ceil_div(N, bn)) * bn;
    if (best_cols < 0 || cols < best_cols) {
      best = bn;
      best_cols = cols;
    }
  }
  return best;
}

// A / B operand maps: E4M3 with 128-byte K boxes and 128-byte swizzle.
bool map_operand_2d(CUtensorMap* m, const void* base, int rows, int K, int box_rows) {
  const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(rows)};
  const uint64_t strides[1] = {static_cast<uint64_t>(K)};
  const uint32_t box[2] = {128, static_cast<uint32_t>(box_rows)};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool map_operand_3d(CUtensorMap* m, const void* base, int G, int rows, int K, int box_rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(rows), static_cast<uint64_t>(G)};
  const uint64_t strides[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(K) * rows};
  const uint32_t box[3] = {128, static_cast<uint32_t>(box_rows), 1};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Packed scale words [(G,) KP, ceil4(mn)] int32, loaded box_x words at a time.
bool map_sf(CUtensorMap* m, const int32_t* base, int G, int mn, int KP, int box_x) {
  const uint64_t w = static_cast<uint64_t>(ceil4(mn));
  if (G <= 0) {
    const uint64_t dims[2] = {w, static_cast<uint64_t>(KP)};
    const uint64_t strides[1] = {w * 4};
    const uint32_t box[2] = {static_cast<uint32_t>(box_x), 1};
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  const uint64_t dims[3] = {w, static_cast<uint64_t>(KP), static_cast<uint64_t>(G)};
  const uint64_t strides[2] = {w * 4, w * 4 * KP};
  const uint32_t box[3] = {static_cast<uint32_t>(box_x), 1, 1};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Output D (BF16), stored 32 rows x 64 columns per TMA store with 128-byte swizzle.
bool map_out(CUtensorMap* m, void* base, int G, int rows, int N) {
  if (G <= 0) {
    const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(rows)};
    const uint64_t strides[1] = {static_cast<uint64_t>(N) * 2};
    const uint32_t box[2] = {64, 32};
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  const uint64_t dims[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(rows), static_cast<uint64_t>(G)};
  const uint64_t strides[2] = {static_cast<uint64_t>(N) * 2, static_cast<uint64_t>(N) * 2 * rows};
  const uint32_t box[3] = {64, 32, 1};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Output D (BF16) in 32-row x 32-column pieces (64-byte rows, 64-byte swizzle): the CTA-pair
// kernel's epilogue for BF16 output without C.
bool map_out_pieces(CUtensorMap* m, void* base, int rows, int N) {
  const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(rows)};
  const uint64_t strides[1] = {static_cast<uint64_t>(N) * 2};
  const uint32_t box[2] = {32, 32};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
}

// MN-major operand ("t" A given as [K, M], "n" B given as [K, N]): boxes of 128 K-rows x 128
// M/N-bytes with 128-byte swizzle; mn must be a multiple of 16 (its row stride in bytes).
bool map_operand_mn(CUtensorMap* m, const void* base, int mn, int K) {
  const uint64_t dims[2] = {static_cast<uint64_t>(mn), static_cast<uint64_t>(K)};
  const uint64_t strides[1] = {static_cast<uint64_t>(mn)};
  const uint32_t box[2] = {128, 128};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// FP32 output D (and C) of the weight-gradient form: 32 rows x 32 columns (128 bytes) per TMA
// store, 128-byte swizzle.
bool map_out_f32(CUtensorMap* m, void* base, int rows, int N) {
  const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(rows)};
  const uint64_t strides[1] = {static_cast<uint64_t>(N) * 4};
  const uint32_t box[2] = {32, 32};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// FP32 output D (and C) of the K-grouped form, [G][rows][N]: 32 x 32 boxes, 128-byte swizzle.
bool map_out_f32_3d(CUtensorMap* m, void* base, int G, int rows, int N) {
  const uint64_t dims[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(rows), static_cast<uint64_t>(G)};
  const uint64_t strides[2] = {static_cast<uint64_t>(N) * 4, static_cast<uint64_t>(N) * rows * 4};
  const uint32_t box[3] = {32, 32, 1};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// FP4 operand ([(G,) rows, K/2] bytes of packed E2M1): 128-element x box_rows boxes of the
// 16U4_ALIGN16B type (each 8 bytes land in a 16-byte shared-memory chunk), 128-byte swizzle.
// The base must be 32-byte aligned and K/2 a multiple of 32 bytes.
bool map_operand_fp4(CUtensorMap* m, const void* base, int G, int rows, int K, int box_rows) {
  const uint64_t row_bytes = static_cast<uint64_t>(K) / 2;
  if (G <= 0) {
    const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(rows)};
    const uint64_t strides[1] = {row_bytes};
    const uint32_t box[2] = {128, static_cast<uint32_t>(box_rows)};
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  const uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(rows), static_cast<uint64_t>(G)};
  const uint64_t strides[2] = {row_bytes, row_bytes * rows};
  const uint32_t box[3] = {128, static_cast<uint32_t>(box_rows), 1};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// FP4 B scale words [(G,) K/128, ceil4(N)] int32 (word (q, n): the four 32-wide blocks of
// K-group q of row n), loaded as box_n words x kg K-groups.
bool map_sf_fp4(CUtensorMap* m, const int32_t* base, int G, int N, int KG, int box_n, int kg) {
  const uint64_t w = static_cast<uint64_t>(ceil4(N));
  if (G <= 0) {
    const uint64_t dims[2] = {w, static_cast<uint64_t>(KG)};
    const uint64_t strides[1] = {w * 4};
    const uint32_t box[2] = {static_cast<uint32_t>(box_n), static_cast<uint32_t>(kg)};
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  const uint64_t dims[3] = {w, static_cast<uint64_t>(KG), static_cast<uint64_t>(G)};
  const uint64_t strides[2] = {w * 4, w * 4 * KG};
  const uint32_t box[3] = {static_cast<uint32_t>(box_n), static_cast<uint32_t>(kg), 1};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Dense / contiguous GEMM on CTA pairs: converts the scale words into tcgen05.cp chunks in
// the stream workspace (two small kernels), then launches the pair kernel.
template <dg::Kind kKind, bool kHasC, int kBN, bool kOutF32 = false, bool kBF4 = false, bool kAMN = false,
          bool kBMN = false>
dg_status run_pair(DeviceState& ds, const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, void* d,
                   dg::Params p, int clusters, cudaStream_t stream) {
  constexpr bool kKG = kKind == dg::Kind::KGrouped;
  // scale word rows: K-quads, or (K-grouped) the per-expert packed rows of all experts
  const int KP = kKG ? p.sf_k_rows : ceil_div(p.K / 128, 4);
  const int num_mb = ceil_div(p.M, 128);
  const int NB = ceil_div(p.N, 128);
  const int sfb_rows = 2 * ceil_div(p.N, kBN);     // two chunks per tile
  const int G = (kKind == dg::Kind::Dense || kKG) ? 1 : p.G;   // groups of B (and its scales)
  const int b_kp = kBF4 ? p.K / 128 : KP;           // B chunk rows per K-group (FP4) or per K-quad
  const size_t sfa_words = static_cast<size_t>(KP) * num_mb * 128;
  const size_t sfb_words = static_cast<size_t>(G) * b_kp * sfb_rows * 128;
  if (static_cast<size_t>(KP) * num_mb > (1u << 30) || static_cast<size_t>(G) * b_kp * sfb_rows > (1u << 30))
    return DG_ERR_UNSUPPORTED;
  // contiguous form: the pair-row list (3 ints per pair row, at most one per block) and its length
  const size_t list_words = kKind == dg::Kind::Contiguous ? 4 + 4 * static_cast<size_t>(ceil_div(3 * num_mb, 4)) : 0;
  WorkspaceLease ws;   // held until both kernels below are launched
  if (dg_status s = stream_workspace(ds, stream, kSkCounterInts * 4 + (sfa_words + sfb_words + list_words) * 4, &ws);
      s != DG_OK)
    return s;
  int32_t* sfa_t = static_cast<int32_t*>(ws.ptr) + kSkCounterInts;
  int32_t* sfb_t = sfa_t + sfa_words;
  int32_t* list = sfb_t + sfb_words;
  {
    dg::SfPrepArgs pa{};
    pa.sfa = sfa;
    pa.sfa_out = sfa_t;
    pa.a_rows = p.M;
    pa.lda = ceil4(p.M);
    pa.a_blocks = num_mb;
    pa.sfb = sfb;
    pa.sfb_out = sfb_t;
    pa.groups = G;
    pa.b_rows = p.N;
    pa.ldb = kBF4 ? ceil4(p.N) : ceil4(NB);
    pa.b_chunks = sfb_rows;
    pa.tile_bn = kBN;
    pa.kp = KP;
    pa.b_kp = b_kp;
    pa.b_per_row = kBF4 ? 1 : 0;
    if constexpr (kKind == dg::Kind::Contiguous) {
      pa.m_indices = p.m_indices;
      pa.num_mb = num_mb;
      pa.groups_g = p.G;
      pa.pair_count = list;
      pa.pair_list = list + 4;   // 16-byte aligned after the count
      pa.status = ds.status;
      p.pair_count = pa.pair_count;
      p.pair_list = pa.pair_list;
    }
    const size_t words = sfa_words + sfb_words;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // (+ one block that lists the contiguous form's pair rows)
    cfg.gridDim = dim3(static_cast<unsigned>(std::min<size_t>((words + 255) / 256, 2048) +
                                             (kKind == dg::Kind::Contiguous ? 1 : 0)),
                       1, 1);
    cfg.blockDim = dim3(256, 1, 1);   // the pair-row scan assumes 256 threads
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, dg::sf_to_utccp_kernel, pa);
    if (e != cudaSuccess) return cuda_fail(e);
  }

  CUtensorMap ta, tb, tsa, tsb, td, td_tail, tc;
  // BF16 output without C: 32-column pieces (see PairConfig::kSmallEpi)
  constexpr bool kSmallEpi = !kHasC && !kOutF32;
  bool ok = (kAMN ? map_operand_mn(&ta, a, p.M, p.K) : map_operand_2d(&ta, a, p.M, p.K, 128)) &&
            (kKG ? map_out_f32_3d(&td, d, p.G, p.M, p.N)
                 : kOutF32 ? map_out_f32(&td, d, p.M, p.N)
                           : kSmallEpi ? map_out_pieces(&td, d, p.M, p.N) : map_out(&td, d, 0, p.M, p.N));
  // C is read by TMA in boxes of the output's geometry (the map of D over C's memory)
  void* c_mem = const_cast<void*>(static_cast<const void*>(p.c));
  if (kHasC)
    ok = ok && (kKG ? map_out_f32_3d(&tc, c_mem, p.G, p.M, p.N)
                    : kOutF32 ? map_out_f32(&tc, c_mem, p.M, p.N) : map_out(&tc, c_mem, 0, p.M, p.N));
  else
    tc = td;
  if constexpr (kSmallEpi ? kBN % 32 != 0 : kBN % 64 != 0) {
    // the narrower end of each tile, 32 rows high, no swizzle: BF16 its last kBN % 64
    // columns (kBN % 32 with 32-column pieces); FP32 its last (kBN % 64) % 32 columns (the
    // rest goes out as 32-column boxes)
    const uint64_t dims[2] = {static_cast<uint64_t>(p.N), static_cast<uint64_t>(p.M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(p.N) * (kOutF32 ? 4 : 2)};
    const uint32_t box[2] = {static_cast<uint32_t>(kOutF32 ? (kBN % 64) % 32 : kSmallEpi ? kBN % 32 : kBN % 64), 32};
    static_assert(!kOutF32 || (kBN % 64) % 32 != 0, "an FP32 narrow box needs a remainder");
    ok = ok && make_map(&td_tail, kOutF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d,
                        dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    td_tail = td;
  }
  // each CTA of the pair loads BN/2 rows of the B tile
  if (kBMN)
    ok = ok && map_operand_mn(&tb, b, p.N, p.K);   // 128-column boxes: one per CTA at width 256
  else if (kBF4)
    ok = ok && map_operand_fp4(&tb, b, kKind == dg::Kind::Dense ? 0 : G, p.N, p.K, kBN / 2);
  else if (kKind == dg::Kind::Dense || kKG)
    ok = ok && map_operand_2d(&tb, b, p.N, p.K, kBN / 2);
  else
    ok = ok && map_operand_3d(&tb, b, G, p.N, p.K, kBN / 2);
  {
    const uint64_t dims_a[2] = {128, static_cast<uint64_t>(KP) * num_mb};
    const uint64_t dims_b[2] = {128, static_cast<uint64_t>(G) * b_kp * sfb_rows};
    const uint64_t strides[1] = {512};
    const uint32_t box_a[2] = {128, 1}, box_b[2] = {128, 2};
    ok = ok && make_map(&tsa, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, sfa_t, dims_a, strides, box_a, CU_TENSOR_MAP_SWIZZLE_NONE);
    ok = ok && make_map(&tsb, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, sfb_t, dims_b, strides, box_b, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (!ok) return DG_ERR_CUDA;
  p.sf_num_mb = num_mb;
  p.sf_nb = sfb_rows;
  return PairLauncher<kKind, kHasC, kBN, kOutF32, kBF4, kAMN, kBMN>::launch(ta, tb, tsa, tsb, td, td_tail, tc, p,
                                                                               clusters, stream);
}

// Pair tile width: DG_PAIR_BN (192, 240 or 256) overrides; 240 is offered for the dense
// form only. Otherwise the width with the smallest estimated makespan: waves of pair tiles
// x cycles per tile. Cycles per K-group and the single accumulator's per-tile cost (the
// MMAs wait for the epilogue to drain it) are fitted to GB300 measurements of
// 4096x24576x1536 (BF16 out: 240 -> 2733, 256 -> 2340, 192 -> 2312 TFLOPS) and
// 7168x4096x4096 (FP32 out: 256 -> 2485, 240 -> 2204): ~512 cycles per K-group at 256
// columns (tensor-bound) + ~2000 per tile, ~556 at 240 and ~535 at 192 (issue-bound).
int pick_pair_bn(long long pair_rows, int N, int K, int clusters, bool dense) {
  if (const char* f = std::getenv("DG_PAIR_BN")) {
    const int v = std::atoi(f);
    if (v == 192 || v == 256 || (v == 240 && dense)) return v;
  }
  const long long kb = K / 128;
  auto makespan = [&](int bn) {
    const long long tiles = pair_rows * ceil_div(N, bn);
    const long long waves = ceil_div(tiles, static_cast<long long>(std::max(clusters, 1)));
    const long long per_tile = bn == 256 ? kb * 512 + 2000 : kb * (bn == 240 ? 556 : 535);
    return waves * per_tile;
  };
  int best = 256;
  for (int bn : {240, 192}) {
    if (bn == 240 && !dense) continue;
    if (makespan(bn) < makespan(best)) best = bn;
  }
  return best;
}

// Launches the pair kernel for kKind if the device can run it; *launched tells whether it did.
template <dg::Kind kKind, bool kOutF32 = false, bool kBF4 = false>
dg_status try_pair(DeviceState& ds, const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                   const void* c, void* d, dg::Params pp, long long pair_rows, int sms, cudaStream_t stream,
                   bool* launched) {
  *launched = false;
  // C: the dense and K-grouped forms
  constexpr bool kTakesC = kKind == dg::Kind::Dense || kKind == dg::Kind::KGrouped;
  if constexpr (!kTakesC) {
    if (c) return DG_ERR_INVALID_ARG;
  }
  constexpr bool kDense = kKind == dg::Kind::Dense;
  constexpr int kWideBN = kDense ? 240 : 192;     // the 240-wide configuration is dense-only
  const bool with_c = kTakesC && c != nullptr;
  const int max_cl = std::min({with_c ? PairLauncher<kKind, kTakesC, 256, kOutF32, kBF4>::max_clusters()
                                      : PairLauncher<kKind, false, 256, kOutF32, kBF4>::max_clusters(),
                               with_c ? PairLauncher<kKind, kTakesC, 192, kOutF32, kBF4>::max_clusters()
                                      : PairLauncher<kKind, false, 192, kOutF32, kBF4>::max_clusters(),
                               with_c ? PairLauncher<kKind, kTakesC, kWideBN, kOutF32, kBF4>::max_clusters()
                                      : PairLauncher<kKind, false, kWideBN, kOutF32, kBF4>::max_clusters()});
  if (max_cl <= 0) return DG_OK;
  const int cl_cap = std::min(max_cl, sms / 2);
  // K-grouped: a tile spans one expert's K slice (their mean stands for the makespan estimate)
  const int k_tile = kKind == dg::Kind::KGrouped ? 128 * std::max(1, pp.K / 128 / std::max(pp.G, 1)) : pp.K;
  const int bn = pick_pair_bn(pair_rows, pp.N, k_tile, cl_cap, kDense);
  const long long pair_tiles = pair_rows * ceil_div(pp.N, bn);
  const int clusters = static_cast<int>(std::min<long long>(cl_cap, pair_tiles));
  *launched = true;
  if (bn == 240) {
    if (with_c) return run_pair<kKind, kTakesC, kWideBN, kOutF32, kBF4>(ds, a, sfa, b, sfb, d, pp, clusters, stream);
    return run_pair<kKind, false, kWideBN, kOutF32, kBF4>(ds, a, sfa, b, sfb, d, pp, clusters, stream);
  }
  if (bn == 256) {
    if (with_c) return run_pair<kKind, kTakesC, 256, kOutF32, kBF4>(ds, a, sfa, b, sfb, d, pp, clusters, stream);
    return run_pair<kKind, false, 256, kOutF32, kBF4>(ds, a, sfa, b, sfb, d, pp, clusters, stream);
  }
  if (with_c) return run_pair<kKind, kTakesC, 192, kOutF32, kBF4>(ds, a, sfa, b, sfb, d, pp, clusters, stream);
  return run_pair<kKind, false, 192, kOutF32, kBF4>(ds, a, sfa, b, sfb, d, pp, clusters, stream);
}

dg_status check_common(int N, int K) {
  if (K <= 0 || K % 128 != 0) return DG_ERR_INVALID_ARG;
  if (N <= 0 || N % 16 != 0) return DG_ERR_INVALID_ARG;
  if (static_cast<long long>(K) / 128 > (1 << 24)) return DG_ERR_INVALID_ARG;
  return DG_OK;
}

// ------------------------------------------------------------------------------------
// scale packing kernel
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ue8m0_ceil(float f, uint32_t* status) {
  const uint32_t bits = __float_as_uint(f);
  if (!(f > 0.0f) || !isfinite(f)) {
    atomicOr(status, dg::kStatusBadIndexBit);
    return 127u;
  }
  const uint32_t e = (bits >> 23) & 0xFFu;
  const uint32_t mant = bits & 0x7FFFFFu;
  uint32_t code;
  if (e == 0) {
    code = mant <= 0x400000u ? 0u : 1u;   // subnormal: (0, 2^-127] -> 2^-127, else 2^-126
  } else {
    code = e + (mant != 0 ? 1u : 0u);
  }
  return code > 254u ? 254u : code;
}

// sf is [mn, kgroups] (K-group contiguous), or [kgroups, mn] with mn_major_in.
__global__ void pack_sf_kernel(const float* __restrict__ sf, int32_t* __restrict__ out, int mn, int kgroups,
                               int mn_major_in, int mn_pad, int kp, uint32_t* status) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(mn_pad) * kp) return;
  const int q = static_cast<int>(idx / mn_pad);
  const int i = static_cast<int>(idx % mn_pad);
  uint32_t w = 0;
  if (i < mn) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int g = 4 * q + j;
      if (g < kgroups) {
        const long long at = mn_major_in ? static_cast<long long>(g) * mn + i : static_cast<long long>(i) * kgroups + g;
        w |= ue8m0_ceil(sf[at], status) << (8 * j);
      }
    }
  }
  out[idx] = static_cast<int32_t>(w);
}

// Dense GEMM on the single-CTA kernel: whole tiles (tile mode) or, with fewer tiles than
// SMs, stream-K. kOutF32: FP32 C / D (weight-gradient form), else BF16.
template <bool kOutF32, bool kAMN = false, bool kBMN = false, bool kBF4 = false>
dg_status run_dense_single(DeviceState& dsr, const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                           const void* c, void* d, int M, int N, int K, int BN, int sms, cudaStream_t stream) {
  DeviceState* ds = &dsr;
  const int KP = ceil_div(K / 128, 4);
  CUtensorMap ta, tb, tsa, tsb, td;
  if (!(kAMN ? map_operand_mn(&ta, a, M, K) : map_operand_2d(&ta, a, M, K, 128)) ||
      !(kBF4 ? map_operand_fp4(&tb, b, 0, N, K, BN) : kBMN ? map_operand_mn(&tb, b, N, K) : map_operand_2d(&tb, b, N, K, BN)) ||
      !map_sf(&tsa, sfa, 0, M, KP, 128) || (!kBF4 && !map_sf(&tsb, sfb, 0, ceil_div(N, 128), KP, 8)) ||
      !(kOutF32 ? map_out_f32(&td, d, M, N) : map_out(&td, d, 0, M, N)))
    return DG_ERR_CUDA;
  dg::Params p = base_params(*ds, M, N, K, 1, c, d);
  const long long tiles = static_cast<long long>(ceil_div(M, 128)) * ceil_div(N, BN);
  int grid = static_cast<int>(tiles < sms ? tiles : sms);
  // Fewer tiles than SMs: share the K-groups of all tiles among all SMs (stream-K) so that
  // every SM streams operands; each CTA gets at least kMinKGroupsPerCta K-groups. The
  // stream-K unit is one pipeline stage: two K-groups for 128-wide tiles (DG_KG=1 selects
  // one K-group per stage), one otherwise.
  int kg = 1;
  if (BN == 128) {
    const char* f = std::getenv("DG_KG");
    kg = (f && f[0] == '1') ? 1 : 2;
  }
  const int num_kc = ceil_div(K / 128, kg);                 // stream-K units per tile
  const long long units = tiles * num_kc;
  const long long sk = std::min<long long>(sms, units * kg / kMinKGroupsPerCta);
  WorkspaceLease ws;   // stream-K only; held until the launch at the end
  if (tiles < sms && sk > tiles) {
    int slots = 1;
    for (long long t = 0; t < tiles; ++t) {
      auto owner = [&](long long v) { return ((v + 1) * sk - 1) / units; };
      const int n = static_cast<int>(owner(t * num_kc + num_kc - 1) - owner(t * num_kc) + 1);
      slots = std::max(slots, n);
    }
    // Layout: a fixed-size counter region first (its position must not depend on the
    // problem shape: completed launches leave it all-zero for the next one), then partials.
    const size_t ws_floats = static_cast<size_t>(tiles) * slots * 128 * BN;
    if (static_cast<size_t>(tiles) * kEpilogueWarps > kSkCounterInts) return DG_ERR_UNSUPPORTED;
    if (dg_status s = stream_workspace(*ds, stream, kSkCounterInts * 4 + ws_floats * 4, &ws); s != DG_OK) return s;
    p.sk_ctas = static_cast<int>(sk);
    p.sk_slots = slots;
    p.sk_counters = static_cast<int*>(ws.ptr);
    p.sk_ws = reinterpret_cast<float*>(static_cast<int*>(ws.ptr) + kSkCounterInts);
    grid = static_cast<int>(sk);
  } else {
    kg = 1;   // tile mode: whole tiles, one K-group per stage
  }
  if constexpr (kBF4) {
    if (!map_sf_fp4(&tsb, sfb, 0, N, K / 128, BN, kg)) return DG_ERR_CUDA;
  }
  if (c)
    return launch_bn<dg::Kind::Dense, true, kOutF32, kAMN, kBMN, kBF4>(BN, ta, tb, tsa, tsb, td, p, grid, stream, kg);
  return launch_bn<dg::Kind::Dense, false, kOutF32, kAMN, kBMN, kBF4>(BN, ta, tb, tsa, tsb, td, p, grid, stream, kg);
}

}  // namespace

namespace dg {
int debug_fault_mode() { return g_fault.load(); }
unsigned long long pipeline_wait_timeout_ns() { return wait_timeout_ns(); }
}  // namespace dg

// ======================================================================================
// C ABI
// ======================================================================================
extern "C" {

dg_status dg_fp8_gemm_nt(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, const void* c,
                         void* d, int M, int N, int K, cudaStream_t stream) {
  if (M < 0) return DG_ERR_INVALID_ARG;
  if (dg_status s = check_common(N, K); s != DG_OK) return s;
  if (M == 0) return DG_OK;   // nothing to read or write: the pointers may be null
  if (!a || !sfa || !b || !sfb || !d) return DG_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(sfa) || !aligned16(b) || !aligned16(sfb) || !aligned16(d) || (c && !aligned16(c)))
    return DG_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if (dg_status s = device_state(&ds); s != DG_OK) return s;

  const int KP = ceil_div(K / 128, 4);
  CUtensorMap ta, tb, tsa, tsb, td;
  const int sms = sms_to_use(*ds);
  const long long tiles128 = static_cast<long long>(ceil_div(M, 128)) * ceil_div(N, 128);
  // fewer tiles than SMs: 128-wide tiles shared over K (stream-K); otherwise the heuristic
  // Fewer 128 x 128 tiles than SMs: stream-K (see below) with DG_SK_BN-wide tiles (default
  // 128); otherwise the tile-mode heuristic.
  int sk_bn = 128;
  if (const char* f = std::getenv("DG_SK_BN")) {
    const int v = std::atoi(f);
    if (v == 128 || v == 192 || v == 256) sk_bn = v;
  }
  const int BN = tiles128 < sms ? sk_bn : pick_bn(dg::Kind::Dense, N);
  if (tiles128 >= sms && M > 128 && pair_enabled() && !std::getenv("DG_FORCE_BN")) {
    {
      dg::Params pp = base_params(*ds, M, N, K, 1, c, d);
      bool launched = false;
      const dg_status s = try_pair<dg::Kind::Dense>(*ds, a, sfa, b, sfb, c, d, pp, ceil_div(M, 256), sms, stream,
                                                    &launched);
      if (launched) return s;
    }
  }
  if (tiles128 < sms) {
    if (const int sbn = pick_split_bn(M, N, K, sms, c != nullptr); sbn > 0) {
      if (!map_operand_2d(&ta, a, M, K, 128) || !map_operand_2d(&tb, b, N, K, sbn) ||
          !map_sf(&tsa, sfa, 0, M, KP, 128) || !map_sf(&tsb, sfb, 0, ceil_div(N, 128), KP, 8) ||
          !map_out(&td, d, 0, M, N))
        return DG_ERR_CUDA;
      dg::Params p = base_params(*ds, M, N, K, 1, c, d);
      const int grid = static_cast<int>(static_cast<long long>(ceil_div(M, 128)) * ceil_div(N, sbn)) * kSplitWays;
      if (c) return launch_split<true>(sbn, ta, tb, tsa, tsb, td, p, grid, stream);
      return launch_split<false>(sbn, ta, tb, tsa, tsb, td, p, grid, stream);
    }
  }
  return run_dense_single<false>(*ds, a, sfa, b, sfb, c, d, M, N, K, BN, sms, stream);
}

}  // extern "C"

namespace {
// fp8_gemm_{nn,tn,tt}: the dense GEMM with A given as [K, M] (kAMN) and/or B as [K, N] (kBMN),
// on the single-CTA kernel (tile mode or stream-K), 128- or 256-wide tiles.
template <bool kAMN, bool kBMN>
dg_status dense_layout_entry(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, const void* c,
                             void* d, int M, int N, int K, cudaStream_t stream) {
  if (M < 0) return DG_ERR_INVALID_ARG;
  if (dg_status s = check_common(N, K); s != DG_OK) return s;
  if (kAMN && M % 16 != 0) return DG_ERR_INVALID_ARG;   // [K, M] rows must be 16-byte multiples
  if (M == 0) return DG_OK;
  if (!a || !sfa || !b || !sfb || !d) return DG_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(sfa) || !aligned16(b) || !aligned16(sfb) || !aligned16(d) || (c && !aligned16(c)))
    return DG_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if (dg_status s = device_state(&ds); s != DG_OK) return s;
  const int sms = sms_to_use(*ds);
  const long long tiles128 = static_cast<long long>(ceil_div(M, 128)) * ceil_div(N, 128);
  if (tiles128 >= sms && M > 128 && pair_enabled() && !std::getenv("DG_FORCE_BN")) {
    // CTA pairs, 256-wide tiles (each CTA's half of an N-major B tile is one 128-column atom)
    const int max_cl = c ? PairLauncher<dg::Kind::Dense, true, 256, false, false, kAMN, kBMN>::max_clusters()
                         : PairLauncher<dg::Kind::Dense, false, 256, false, false, kAMN, kBMN>::max_clusters();
    if (max_cl > 0) {
      dg::Params pp = base_params(*ds, M, N, K, 1, c, d);
      const long long pair_tiles = static_cast<long long>(ceil_div(M, 256)) * ceil_div(N, 256);
      const int clusters = static_cast<int>(std::min<long long>(std::min(max_cl, sms / 2), pair_tiles));
      if (c)
        return run_pair<dg::Kind::Dense, true, 256, false, false, kAMN, kBMN>(*ds, a, sfa, b, sfb, d, pp, clusters,
                                                                                stream);
      return run_pair<dg::Kind::Dense, false, 256, false, false, kAMN, kBMN>(*ds, a, sfa, b, sfb, d, pp, clusters,
                                                                               stream);
    }
  }
  int BN = 128;
  if (tiles128 >= sms) {
    BN = ceil_div(N, 256) * 256 <= ceil_div(N, 128) * 128 ? 256 : 128;   // the wider unless it wastes columns
    if (const char* f = std::getenv("DG_FORCE_BN")) {
      const int v = std::atoi(f);
      if (v == 128 || v == 256) BN = v;
    }
  }
  return run_dense_single<false, kAMN, kBMN>(*ds, a, sfa, b, sfb, c, d, M, N, K, BN, sms, stream);
}
}  // namespace

extern "C" {

dg_status dg_fp8_gemm_nn(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, const void* c,
                         void* d, int M, int N, int K, cudaStream_t stream) {
  return dense_layout_entry<false, true>(a, sfa, b, sfb, c, d, M, N, K, stream);
}

dg_status dg_fp8_gemm_tn(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, const void* c,
                         void* d, int M, int N, int K, cudaStream_t stream) {
  return dense_layout_entry<true, true>(a, sfa, b, sfb, c, d, M, N, K, stream);
}

dg_status dg_fp8_gemm_tt(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, const void* c,
                         void* d, int M, int N, int K, cudaStream_t stream) {
  return dense_layout_entry<true, false>(a, sfa, b, sfb, c, d, M, N, K, stream);
}

dg_status dg_wgrad_gemm_fp8_fp8_fp32_nt(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                        const float* c, float* d, int M, int N, int K, cudaStream_t stream) {
  if (M < 0) return DG_ERR_INVALID_ARG;
  if (dg_status s = check_common(N, K); s != DG_OK) return s;
  if (M == 0) return DG_OK;
  if (!a || !sfa || !b || !sfb || !d) return DG_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(sfa) || !aligned16(b) || !aligned16(sfb) || !aligned16(d) || (c && !aligned16(c)))
    return DG_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if (dg_status s = device_state(&ds); s != DG_OK) return s;
  const int sms = sms_to_use(*ds);
  const long long tiles128 = static_cast<long long>(ceil_div(M, 128)) * ceil_div(N, 128);
  if (tiles128 >= sms && M > 128 && pair_enabled() && !std::getenv("DG_FORCE_BN")) {
    dg::Params pp = base_params(*ds, M, N, K, 1, c, d);
    bool launched = false;
    const dg_status s = try_pair<dg::Kind::Dense, true>(*ds, a, sfa, b, sfb, c, d, pp, ceil_div(M, 256), sms, stream,
                                                        &launched);
    if (launched) return s;
  }
  // Tile mode: 192-wide tiles with two accumulators, so that the FP32 epilogue (twice the
  // bytes of the BF16 one, plus the C read) overlaps the next tile's MMAs (measured on GB300,
  // 7168x4096x4096 accumulated in place: 1916 TFLOPS at 192 vs 1736 at 256 and 1650 at 128).
  const int BN = tiles128 < sms ? 128 : (std::getenv("DG_FORCE_BN") || N <= 128 ? pick_bn(dg::Kind::Dense, N) : 192);
  return run_dense_single<true>(*ds, a, sfa, b, sfb, c, d, M, N, K, BN, sms, stream);
}

}  // extern "C"

namespace {
template <bool kMN>
dg_status k_grouped_entry(const void* a, const int32_t* sfa, const void* b,
                                                const int32_t* sfb, const float* c, float* d, const int32_t* ks,
                                                int G, int M, int N, int K_total, int sf_k_rows,
                                                cudaStream_t stream) {
  if (G <= 0 || M < 0 || K_total < 0 || sf_k_rows < 0) return DG_ERR_INVALID_ARG;
  if (N <= 0 || N % 16 != 0 || K_total % 128 != 0) return DG_ERR_INVALID_ARG;
  if (kMN && M % 16 != 0) return DG_ERR_INVALID_ARG;   // [K, M] rows must be 16-byte multiples
  if (M == 0) return DG_OK;
  if (!d || !ks || (K_total > 0 && (!a || !sfa || !b || !sfb || sf_k_rows == 0))) return DG_ERR_INVALID_ARG;
  if ((K_total > 0 && (!aligned16(a) || !aligned16(sfa) || !aligned16(b) || !aligned16(sfb))) || !aligned16(d) ||
      (c && !aligned16(c)) || (reinterpret_cast<uintptr_t>(ks) & 3u))
    return DG_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if (dg_status s = device_state(&ds); s != DG_OK) return s;
  const size_t out_bytes = static_cast<size_t>(G) * M * N * sizeof(float);
  if (K_total == 0) {
    // no tokens at all: every expert's output is its addend (or zero)
    cudaError_t e = c ? (c == d ? cudaSuccess : cudaMemcpyAsync(d, c, out_bytes, cudaMemcpyDeviceToDevice, stream))
                      : cudaMemsetAsync(d, 0, out_bytes, stream);
    return e == cudaSuccess ? DG_OK : cuda_fail(e);
  }
  const int sms = sms_to_use(*ds);
  if constexpr (!kMN) {
    // CTA pairs when the tiles fill the GPU (K-major operands only)
    const long long tiles128 = static_cast<long long>(G) * ceil_div(M, 128) * ceil_div(N, 128);
    if (tiles128 >= sms && M > 128 && pair_enabled() && !std::getenv("DG_FORCE_BN")) {
      dg::Params pp = base_params(*ds, M, N, K_total, G, c, d);
      pp.ks = ks;
      pp.sf_k_rows = sf_k_rows;
      bool launched = false;
      const dg_status s = try_pair<dg::Kind::KGrouped, true>(*ds, a, sfa, b, sfb, c, d, pp,
                                                             static_cast<long long>(G) * ceil_div(M, 256), sms,
                                                             stream, &launched);
      if (launched) return s;
    }
  }
  int BN = std::getenv("DG_FORCE_BN") || N <= 128 ? pick_bn(dg::Kind::Dense, N) : 192;
  if (kMN && BN == 192) BN = 256;   // an N-major B tile is whole 128-column atoms
  CUtensorMap ta, tb, tsa, tsb, td;
  bool ok = (kMN ? map_operand_mn(&ta, a, M, K_total) : map_operand_2d(&ta, a, M, K_total, 128)) &&
            (kMN ? map_operand_mn(&tb, b, N, K_total) : map_operand_2d(&tb, b, N, K_total, BN)) &&
            map_sf(&tsa, sfa, 0, M, sf_k_rows, 128) && map_sf(&tsb, sfb, 0, ceil_div(N, 128), sf_k_rows, 8);
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M), static_cast<uint64_t>(G)};
    const uint64_t strides[2] = {static_cast<uint64_t>(N) * 4, static_cast<uint64_t>(N) * M * 4};
    const uint32_t box[3] = {32, 32, 1};
    ok = ok && make_map(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, d, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (!ok) return DG_ERR_CUDA;
  dg::Params p = base_params(*ds, M, N, K_total, G, c, d);
  p.ks = ks;
  p.sf_k_rows = sf_k_rows;
  const long long tiles = static_cast<long long>(G) * ceil_div(M, 128) * ceil_div(N, BN);
  if (tiles > (1LL << 30)) return DG_ERR_UNSUPPORTED;
  const int grid = static_cast<int>(std::min<long long>(tiles, sms));
  if (c) return launch_bn<dg::Kind::KGrouped, true, true, kMN, kMN>(BN, ta, tb, tsa, tsb, td, p, grid, stream);
  return launch_bn<dg::Kind::KGrouped, false, true, kMN, kMN>(BN, ta, tb, tsa, tsb, td, p, grid, stream);
}
}  // namespace

extern "C" {

dg_status dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(const void* a, const int32_t* sfa, const void* b,
                                                const int32_t* sfb, const float* c, float* d, const int32_t* ks,
                                                int G, int M, int N, int K_total, int sf_k_rows,
                                                cudaStream_t stream) {
  return k_grouped_entry<false>(a, sfa, b, sfb, c, d, ks, G, M, N, K_total, sf_k_rows, stream);
}

dg_status dg_k_grouped_fp8_gemm_tn_contiguous(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                              const float* c, float* d, const int32_t* ks, int G, int M, int N,
                                              int K_total, int sf_k_rows, cudaStream_t stream) {
  return k_grouped_entry<true>(a, sfa, b, sfb, c, d, ks, G, M, N, K_total, sf_k_rows, stream);
}

dg_status dg_m_grouped_fp8_gemm_nt_contiguous(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                              void* d, const int32_t* m_indices, int M_total, int N, int K, int G,
                                              cudaStream_t stream) {
  if (M_total < 0 || G <= 0) return DG_ERR_INVALID_ARG;
  if (dg_status s = check_common(N, K); s != DG_OK) return s;
  if (M_total == 0) return DG_OK;
  if (!a || !sfa || !b || !sfb || !d || !m_indices) return DG_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(sfa) || !aligned16(b) || !aligned16(sfb) || !aligned16(d) ||
      (reinterpret_cast<uintptr_t>(m_indices) & 3u))
    return DG_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if (dg_status s = device_state(&ds); s != DG_OK) return s;

  // The contiguous form runs on CTA pairs (measured on GB300 for the G=8 workload over 100
  // back-to-back launches: 2860-2950 TFLOPS against 2600-2725 with single-CTA 128 x 256
  // tiles); DG_PAIR=0 or DG_FORCE_BN selects the single-CTA kernel.
  if (pair_enabled() && !std::getenv("DG_FORCE_BN")) {
    {
      dg::Params pp = base_params(*ds, M_total, N, K, G, nullptr, d);
      pp.m_indices = m_indices;
      // the number of pair rows depends on m_indices (device): bound it by the block count
      bool launched = false;
      const dg_status s = try_pair<dg::Kind::Contiguous>(*ds, a, sfa, b, sfb, nullptr, d, pp, ceil_div(M_total, 128),
                                                         sms_to_use(*ds), stream, &launched);
      if (launched) return s;
    }
  }
  const int KP = ceil_div(K / 128, 4);
  CUtensorMap ta, tb, tsa, tsb, td;
  const int BN = pick_bn(dg::Kind::Contiguous, N);
  if (!map_operand_2d(&ta, a, M_total, K, 128) || !map_operand_3d(&tb, b, G, N, K, BN) ||
      !map_sf(&tsa, sfa, 0, M_total, KP, 128) || !map_sf(&tsb, sfb, G, ceil_div(N, 128), KP, 8) ||
      !map_out(&td, d, 0, M_total, N))
    return DG_ERR_CUDA;
  dg::Params p = base_params(*ds, M_total, N, K, G, nullptr, d);
  p.m_indices = m_indices;
  const long long tiles = static_cast<long long>(ceil_div(M_total, 128)) * ceil_div(N, BN);
  const int grid = static_cast<int>(tiles < sms_to_use(*ds) ? tiles : sms_to_use(*ds));
  return launch_bn<dg::Kind::Contiguous, false>(BN, ta, tb, tsa, tsb, td, p, grid, stream);
}

dg_status dg_m_grouped_fp8_gemm_nn_contiguous(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                              void* d, const int32_t* m_indices, int M_total, int N, int K, int G,
                                              cudaStream_t stream) {
  if (M_total < 0 || G <= 0) return DG_ERR_INVALID_ARG;
  if (dg_status s = check_common(N, K); s != DG_OK) return s;
  if (M_total == 0) return DG_OK;
  if (!a || !sfa || !b || !sfb || !d || !m_indices) return DG_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(sfa) || !aligned16(b) || !aligned16(sfb) || !aligned16(d) ||
      (reinterpret_cast<uintptr_t>(m_indices) & 3u))
    return DG_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if (dg_status s = device_state(&ds); s != DG_OK) return s;

  const int KP = ceil_div(K / 128, 4);
  CUtensorMap ta, tb, tsa, tsb, td;
  // 128- or 256-wide tiles (an N-major B tile is whole 128-column atoms), the wider unless
  // it wastes columns
  int BN = ceil_div(N, 256) * 256 <= ceil_div(N, 128) * 128 ? 256 : 128;
  if (const char* f = std::getenv("DG_FORCE_BN")) {
    const int v = std::atoi(f);
    if (v == 128 || v == 256) BN = v;
  }
  CUtensorMap tb_mn;
  {
    // B stored [G][K][N]: boxes of 128 K-rows x 128 N-bytes, 128-byte swizzle
    const uint64_t dims[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K), static_cast<uint64_t>(G)};
    const uint64_t strides[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(N) * K};
    const uint32_t box[3] = {128, 128, 1};
    if (!make_map(&tb_mn, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, b, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return DG_ERR_CUDA;
  }
  tb = tb_mn;
  if (!map_operand_2d(&ta, a, M_total, K, 128) ||
      !map_sf(&tsa, sfa, 0, M_total, KP, 128) || !map_sf(&tsb, sfb, G, ceil_div(N, 128), KP, 8) ||
      !map_out(&td, d, 0, M_total, N))
    return DG_ERR_CUDA;
  dg::Params p = base_params(*ds, M_total, N, K, G, nullptr, d);
  p.m_indices = m_indices;
  const long long tiles = static_cast<long long>(ceil_div(M_total, 128)) * ceil_div(N, BN);
  const int grid = static_cast<int>(tiles < sms_to_use(*ds) ? tiles : sms_to_use(*ds));
  return launch_bn<dg::Kind::Contiguous, false, false, false, true>(BN, ta, tb, tsa, tsb, td, p, grid, stream);
}

dg_status dg_m_grouped_fp8_gemm_nt_masked(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                          void* d, const int32_t* masked_m, int G, int max_m, int N, int K,
                                          cudaStream_t stream) {
  if (G <= 0 || max_m < 0) return DG_ERR_INVALID_ARG;
  if (dg_status s = check_common(N, K); s != DG_OK) return s;
  if (max_m == 0) return DG_OK;
  if (!a || !sfa || !b || !sfb || !d || !masked_m) return DG_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(sfa) || !aligned16(b) || !aligned16(sfb) || !aligned16(d) ||
      (reinterpret_cast<uintptr_t>(masked_m) & 3u))
    return DG_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if (dg_status s = device_state(&ds); s != DG_OK) return s;

  const int KP = ceil_div(K / 128, 4);
  CUtensorMap ta, tb, tsa, tsb, td;
  const int BN = pick_bn(dg::Kind::Masked, N);
  if (!map_operand_3d(&ta, a, G, max_m, K, 128) || !map_operand_3d(&tb, b, G, N, K, BN) ||
      !map_sf(&tsa, sfa, G, max_m, KP, 128) || !map_sf(&tsb, sfb, G, ceil_div(N, 128), KP, 8) ||
      !map_out(&td, d, G, max_m, N))
    return DG_ERR_CUDA;
  dg::Params p = base_params(*ds, max_m, N, K, G, nullptr, d);
  p.masked_m = masked_m;
  const long long tiles = static_cast<long long>(G) * ceil_div(max_m, 128) * ceil_div(N, BN);
  const int grid = static_cast<int>(tiles < sms_to_use(*ds) ? tiles : sms_to_use(*ds));
  return launch_bn<dg::Kind::Masked, false>(BN, ta, tb, tsa, tsb, td, p, grid, stream);
}

dg_status dg_pack_sf_ue8m0(const float* sf_fp32, int32_t* out, int mn, int kgroups, int mn_major_in,
                           cudaStream_t stream) {
  if (!sf_fp32 || !out || mn < 0 || kgroups <= 0 || (mn_major_in != 0 && mn_major_in != 1)) return DG_ERR_INVALID_ARG;
  if (!aligned16(out) || (reinterpret_cast<uintptr_t>(sf_fp32) & 3u)) return DG_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if (dg_status s = device_state(&ds); s != DG_OK) return s;
  const int mn_pad = ceil4(mn);
  const int kp = ceil_div(kgroups, 4);
  const long long n = static_cast<long long>(mn_pad) * kp;
  if (n == 0) return DG_OK;
  const int threads = 256;
  const long long blocks = (n + threads - 1) / threads;
  if (blocks > 0x7FFFFFFFll) return DG_ERR_INVALID_ARG;
  pack_sf_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(sf_fp32, out, mn, kgroups, mn_major_in,
                                                                        mn_pad, kp, ds->status);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DG_OK : cuda_fail(e);
}

int dg_get_mk_alignment_for_contiguous_layout(void) { return g_mk_alignment.load(); }

dg_status dg_set_mk_alignment_for_contiguous_layout(int alignment) {
  if (alignment <= 0 || alignment % dg::BLOCK_M != 0 || alignment > (1 << 20)) return DG_ERR_INVALID_ARG;
  g_mk_alignment.store(alignment);
  return DG_OK;
}

int dg_get_theoretical_mk_alignment_for_contiguous_layout(void) { return dg::BLOCK_M; }

int dg_get_tma_aligned_size(int mn, int elem_bytes) {
  if (mn < 0 || (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)) return -1;
  const int per16 = 16 / elem_bytes;
  return ceil_div(mn, per16) * per16;
}

dg_status dg_set_num_sms(int n) {
  if (n <= 0) {
    g_num_sms_cap.store(0);
    return DG_OK;
  }
  DeviceState* ds = nullptr;
  if (dg_status s = device_state(&ds); s != DG_OK) return s;
  if (n > ds->num_sms) return DG_ERR_INVALID_ARG;
  g_num_sms_cap.store(n);
  return DG_OK;
}

int dg_get_num_sms(void) {
  DeviceState* ds = nullptr;
  if (device_state(&ds) != DG_OK) return g_num_sms_cap.load();
  return sms_to_use(*ds);
}

dg_status dg_get_device_status(cudaStream_t stream) {
  DeviceState* ds = nullptr;
  if (dg_status s = device_state(&ds); s != DG_OK) return s;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  uint32_t v = 0;
  if ((e = cudaMemcpy(&v, ds->status, sizeof(v), cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e);
  if (v == 0) return DG_OK;
  if ((e = cudaMemset(ds->status, 0, sizeof(uint32_t))) != cudaSuccess) return cuda_fail(e);
  if (v & dg::kStatusTimeoutBit) {
    // an aborted stream-K launch may leave its arrival counters non-zero: clear them
    std::lock_guard<std::mutex> lock(g_mutex);
    for (const auto* list : {&ds->workspaces.live, &ds->workspaces.retained})
      for (const auto& w : *list)
        if (w.ptr && (e = cudaMemset(w.ptr, 0, w.bytes)) != cudaSuccess) return cuda_fail(e);
    return DG_ERR_TIMEOUT;
  }
  return DG_ERR_BAD_INDEX;
}

const char* dg_status_string(dg_status s) {
  switch (s) {
    case DG_OK: return "DG_OK";
    case DG_ERR_INVALID_ARG: return "DG_ERR_INVALID_ARG";
    case DG_ERR_UNSUPPORTED: return "DG_ERR_UNSUPPORTED";
    case DG_ERR_MISALIGNED: return "DG_ERR_MISALIGNED";
    case DG_ERR_CUDA: return "DG_ERR_CUDA";
    case DG_ERR_TIMEOUT: return "DG_ERR_TIMEOUT";
    case DG_ERR_BAD_INDEX: return "DG_ERR_BAD_INDEX";
  }
  return "DG_ERR_UNKNOWN";
}

int dg_last_cuda_error(void) { return g_last_cuda_error; }

dg_status dg_reserve_workspace(cudaStream_t stream, size_t bytes) {
  DeviceState* ds = nullptr;
  if (dg_status s = device_state(&ds); s != DG_OK) return s;
  std::lock_guard<std::mutex> lock(g_mutex);
  const int e = dg::reserve<CudaApi, kMaxWorkspaces>(ds->workspaces, stream, bytes);
  if (e < 0) return DG_ERR_INVALID_ARG;   // the stream is being captured
  return e ? cuda_fail(static_cast<cudaError_t>(e)) : DG_OK;
}

dg_status dg_release_workspace(cudaStream_t stream) {
  DeviceState* ds = nullptr;
  if (dg_status s = device_state(&ds); s != DG_OK) return s;
  std::lock_guard<std::mutex> lock(g_mutex);
  const int e = dg::reserve_release<CudaApi>(ds->workspaces, stream);
  if (e < 0) return DG_ERR_INVALID_ARG;
  return e ? cuda_fail(static_cast<cudaError_t>(e)) : DG_OK;
}

size_t dg_get_workspace_size(cudaStream_t stream) {
  DeviceState* ds = nullptr;
  if (device_state(&ds) != DG_OK) return 0;
  std::lock_guard<std::mutex> lock(g_mutex);
  return dg::workspace_bytes(ds->workspaces, stream);
}

dg_status dg_set_pdl(int enable) {
  if (enable != 0 && enable != 1) return DG_ERR_INVALID_ARG;
  g_pdl.store(enable);
  return DG_OK;
}

int dg_get_pdl(void) { return pdl_enabled() ? 1 : 0; }

dg_status dg_set_debug(int fault_mode, unsigned long long wait_timeout_ns) {
  if (fault_mode < 0 || fault_mode > dg::kFaultProducerSilent) return DG_ERR_INVALID_ARG;
  g_fault.store(fault_mode);
  g_timeout_ns.store(wait_timeout_ns);
  return DG_OK;
}

}  // extern "C"

// ======================================================================================
// FP8 x FP4: A E4M3 (scales 1 x 128), B packed E2M1 (one UE8M0 scale per row per 32 K)
// ======================================================================================
namespace {

inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// Tile width for FP4 B: the masked form (short K, HBM-bound) takes 192 when N > 128, the
// others the wider of 256 / 128 unless it wastes columns. DG_FORCE_BN overrides (128 or
// 256; 192 for the masked form).
int pick_bn_fp4(dg::Kind kind, int N) {
  if (const char* f = std::getenv("DG_FORCE_BN")) {
    const int v = std::atoi(f);
    if (v == 128 || (v == 256 && kind != dg::Kind::Masked) || (v == 192 && kind == dg::Kind::Masked)) return v;
  }
  if (kind == dg::Kind::Masked) return N > 128 ? 192 : 128;
  return ceil_div(N, 256) * 256 <= ceil_div(N, 128) * 128 ? 256 : 128;
}

dg_status check_fp4_pointers(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, const void* c,
                             const void* d) {
  if (!a || !sfa || !b || !sfb || !d) return DG_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(sfa) || !aligned32(b) || !aligned16(sfb) || !aligned16(d) || (c && !aligned16(c)))
    return DG_ERR_MISALIGNED;
  return DG_OK;
}

}  // namespace

extern "C" {

dg_status dg_fp8_fp4_gemm_nt(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, const void* c,
                             void* d, int M, int N, int K, cudaStream_t stream) {
  if (M < 0) return DG_ERR_INVALID_ARG;
  if (dg_status s = check_common(N, K); s != DG_OK) return s;
  if (M == 0) return DG_OK;
  if (dg_status s = check_fp4_pointers(a, sfa, b, sfb, c, d); s != DG_OK) return s;
  DeviceState* ds = nullptr;
  if (dg_status s = device_state(&ds); s != DG_OK) return s;
  const int sms = sms_to_use(*ds);
  const long long tiles128 = static_cast<long long>(ceil_div(M, 128)) * ceil_div(N, 128);
  if (tiles128 >= sms && M > 128 && pair_enabled() && !std::getenv("DG_FORCE_BN")) {
    dg::Params pp = base_params(*ds, M, N, K, 1, c, d);
    bool launched = false;
    const dg_status s = try_pair<dg::Kind::Dense, false, true>(*ds, a, sfa, b, sfb, c, d, pp, ceil_div(M, 256), sms,
                                                               stream, &launched);
    if (launched) return s;
  }
  if (tiles128 < sms) {
    // few tiles: split-K over CTA pairs when the tiles fill the GPU that way, else stream-K
    if (const int sbn = pick_split_bn(M, N, K, sms, c != nullptr, true); sbn > 0) {
      CUtensorMap ta, tb, tsa, tsb, td;
      if (!map_operand_2d(&ta, a, M, K, 128) || !map_operand_fp4(&tb, b, 0, N, K, sbn) ||
          !map_sf(&tsa, sfa, 0, M, ceil_div(K / 128, 4), 128) || !map_sf_fp4(&tsb, sfb, 0, N, K / 128, sbn, 2) ||
          !map_out(&td, d, 0, M, N))
        return DG_ERR_CUDA;
      dg::Params p = base_params(*ds, M, N, K, 1, c, d);
      const int grid = static_cast<int>(static_cast<long long>(ceil_div(M, 128)) * ceil_div(N, sbn)) * kSplitWays;
      if (c) return launch_split<true, true>(sbn, ta, tb, tsa, tsb, td, p, grid, stream);
      return launch_split<false, true>(sbn, ta, tb, tsa, tsb, td, p, grid, stream);
    }
    return run_dense_single<false, false, false, true>(*ds, a, sfa, b, sfb, c, d, M, N, K, 128, sms, stream);
  }
  return run_dense_single<false, false, false, true>(*ds, a, sfa, b, sfb, c, d, M, N, K,
                                                     pick_bn_fp4(dg::Kind::Dense, N), sms, stream);
}

dg_status dg_m_grouped_fp8_fp4_gemm_nt_contiguous(const void* a, const int32_t* sfa, const void* b,
                                                  const int32_t* sfb, void* d, const int32_t* m_indices, int M_total,
                                                  int N, int K, int G, cudaStream_t stream) {
  if (M_total < 0 || G <= 0) return DG_ERR_INVALID_ARG;
  if (dg_status s = check_common(N, K); s != DG_OK) return s;
  if (M_total == 0) return DG_OK;
  if (!m_indices) return DG_ERR_INVALID_ARG;
  if (dg_status s = check_fp4_pointers(a, sfa, b, sfb, nullptr, d); s != DG_OK) return s;
  if (reinterpret_cast<uintptr_t>(m_indices) & 3u) return DG_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if (dg_status s = device_state(&ds); s != DG_OK) return s;
  if (pair_enabled() && !std::getenv("DG_FORCE_BN")) {
    dg::Params pp = base_params(*ds, M_total, N, K, G, nullptr, d);
    pp.m_indices = m_indices;
    bool launched = false;
    const dg_status s = try_pair<dg::Kind::Contiguous, false, true>(*ds, a, sfa, b, sfb, nullptr, d, pp,
                                                                    ceil_div(M_total, 128), sms_to_use(*ds), stream,
                                                                    &launched);
    if (launched) return s;
  }
  const int BN = pick_bn_fp4(dg::Kind::Contiguous, N);
  CUtensorMap ta, tb, tsa, tsb, td;
  if (!map_operand_2d(&ta, a, M_total, K, 128) || !map_operand_fp4(&tb, b, G, N, K, BN) ||
      !map_sf(&tsa, sfa, 0, M_total, ceil_div(K / 128, 4), 128) || !map_sf_fp4(&tsb, sfb, G, N, K / 128, BN, 1) ||
      !map_out(&td, d, 0, M_total, N))
    return DG_ERR_CUDA;
  dg::Params p = base_params(*ds, M_total, N, K, G, nullptr, d);
  p.m_indices = m_indices;
  const long long tiles = static_cast<long long>(ceil_div(M_total, 128)) * ceil_div(N, BN);
  const int grid = static_cast<int>(tiles < sms_to_use(*ds) ? tiles : sms_to_use(*ds));
  return launch_bn<dg::Kind::Contiguous, false, false, false, false, true>(BN, ta, tb, tsa, tsb, td, p, grid, stream);
}

dg_status dg_m_grouped_fp8_fp4_gemm_nt_masked(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                              void* d, const int32_t* masked_m, int G, int max_m, int N, int K,
                                              cudaStream_t stream) {
  if (G <= 0 || max_m < 0) return DG_ERR_INVALID_ARG;
  if (dg_status s = check_common(N, K); s != DG_OK) return s;
  if (max_m == 0) return DG_OK;
  if (!masked_m) return DG_ERR_INVALID_ARG;
  if (dg_status s = check_fp4_pointers(a, sfa, b, sfb, nullptr, d); s != DG_OK) return s;
  if (reinterpret_cast<uintptr_t>(masked_m) & 3u) return DG_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if (dg_status s = device_state(&ds); s != DG_OK) return s;
  const int BN = pick_bn_fp4(dg::Kind::Masked, N);
  CUtensorMap ta, tb, tsa, tsb, td;
  if (!map_operand_3d(&ta, a, G, max_m, K, 128) || !map_operand_fp4(&tb, b, G, N, K, BN) ||
      !map_sf(&tsa, sfa, G, max_m, ceil_div(K / 128, 4), 128) || !map_sf_fp4(&tsb, sfb, G, N, K / 128, BN, 1) ||
      !map_out(&td, d, G, max_m, N))
    return DG_ERR_CUDA;
  dg::Params p = base_params(*ds, max_m, N, K, G, nullptr, d);
  p.masked_m = masked_m;
  const long long tiles = static_cast<long long>(G) * ceil_div(max_m, 128) * ceil_div(N, BN);
  const int grid = static_cast<int>(tiles < sms_to_use(*ds) ? tiles : sms_to_use(*ds));
  return launch_bn<dg::Kind::Masked, false, false, false, false, true>(BN, ta, tb, tsa, tsb, td, p, grid, stream);
}

}  // extern "C"
