// dg_fp8_gemm_nt_no_alloc: the dense GEMM for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc at the moment they need a GEMM: an inference server
// that fixes its device-memory footprint at start-up and forbids later allocations, a
// custom allocator that owns all of the device's memory, code running under a memory budget
// where a lazy allocation could fail in the middle of a step, or a latency-critical loop
// that cannot afford the implicit device synchronisation a cudaMalloc / cudaFree may bring.
// The regular entry point dg_fp8_gemm_nt allocates on first use (its status word and, for
// some shapes, a per-stream workspace). This entry point allocates nothing: the stream-K
// scratch (arrival counters and FP32 partial tiles) lives in the file-scope device array
// below, and device-side errors go to a status word the caller passes.
//
// It runs the single-CTA kernel of this library in stream-K mode with one K-group per
// pipeline stage and 128 x 128 tiles, on every SM of the device (dg_set_num_sms does not
// apply): the K-groups of all tiles are split evenly among the CTAs, and a tile split
// between CTAs is summed in a fixed order by its last contributor. Its results therefore
// match dg_fp8_gemm_nt within the parity tolerance (the summation order may differ).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "debug_state.h"
#include "dg.h"
#include "fp8_gemm.cuh"

namespace {

// Scratch for the stream-K arrival counters and partial tiles: 16 MiB, held by every
// GPU that loads this library until the process exits.
constexpr size_t kScratchBytes = size_t(16) << 20;
constexpr size_t kCounterInts = 4096;                 // first 16 KiB: arrival counters
constexpr int kBN = 128;                              // tile width of the stream-K kernel
constexpr int kEpiWarps = 4;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_no_alloc_scratch[kScratchBytes];

// The kernel this entry point launches (stream-K, 128-wide tiles, 5 stages, two accumulators).
using Cfg = dg::Config<kBN, 5, 2, kEpiWarps, 2>;
template <bool kHasC>
constexpr auto kernel() {
  return dg::fp8_gemm_kernel<dg::Kind::Dense, kBN, 5, 2, kEpiWarps, 2, kHasC>;
}

struct DeviceSetup {
  bool done = false;
  bool supported = false;
  int num_sms = 0;
  unsigned char* scratch = nullptr;   // device address of g_no_alloc_scratch on this device
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;

// Once per device, with that device current: capability, SM count, and the device address
// of the scratch array (its host-side name is only a stand-in for the symbol).
dg_status setup_device(DeviceSetup** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DG_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DG_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceSetup& s = g_setup[dev];
  if (!s.done) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DG_ERR_CUDA;
    s.supported = (major == 10 && minor == 3);
    if (s.supported) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_no_alloc_scratch) != cudaSuccess || ptr == nullptr) return DG_ERR_CUDA;
      s.scratch = static_cast<unsigned char*>(ptr);
      // the kernels' dynamic shared-memory limit, once per device (not on every call)
      if (cudaFuncSetAttribute(kernel<true>(), cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) !=
              cudaSuccess ||
          cudaFuncSetAttribute(kernel<false>(), cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) !=
              cudaSuccess)
        return DG_ERR_CUDA;
    }
    s.done = true;
  }
  if (!s.supported) return DG_ERR_UNSUPPORTED;
  *out = &s;
  return DG_OK;
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

bool encode(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
            uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// (the shared-memory attribute was set by setup_device for this device)
template <bool kHasC>
cudaError_t launch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa, const CUtensorMap& tsb,
                   const CUtensorMap& td, const dg::Params& p, int grid, cudaStream_t stream) {
  kernel<kHasC>()<<<grid, Cfg::kThreads, Cfg::SMEM_BYTES, stream>>>(ta, tb, tsa, tsb, td, p);
  return cudaGetLastError();
}

}  // namespace

extern "C" dg_status dg_fp8_gemm_nt_no_alloc(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                             const void* c, void* d, uint32_t* status, int M, int N, int K,
                                             cudaStream_t stream) {
  if (M < 0 || K <= 0 || K % 128 != 0 || N <= 0 || N % 16 != 0) return DG_ERR_INVALID_ARG;
  if (M == 0) return DG_OK;
  if (!a || !sfa || !b || !sfb || !d || !status) return DG_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(sfa) || !aligned16(b) || !aligned16(sfb) || !aligned16(d) || (c && !aligned16(c)) ||
      (reinterpret_cast<uintptr_t>(status) & 3u))
    return DG_ERR_MISALIGNED;
  DeviceSetup* ds = nullptr;
  if (dg_status s = setup_device(&ds); s != DG_OK) return s;

  // Partition of the K-groups of all 128 x 128 tiles among the SMs (stream-K), and the
  // scratch it needs: counters for every tile, and room for one FP32 partial tile per
  // contributor slot of every tile (the largest contributor count of any tile, for all
  // tiles: a conservative bound, as a tile that one CTA computes whole writes no partial).
  const int num_kb = K / 128;
  const long long tiles = static_cast<long long>(ceil_div(M, 128)) * ceil_div(N, kBN);
  const long long kgroups = tiles * num_kb;
  const long long ctas = std::max<long long>(1, std::min<long long>(ds->num_sms, kgroups / 4));
  auto owner = [&](long long v) { return ((v + 1) * ctas - 1) / kgroups; };
  int slots = 1;
  for (long long t = 0; t < tiles; ++t)
    slots = std::max(slots, static_cast<int>(owner(t * num_kb + num_kb - 1) - owner(t * num_kb) + 1));
  const size_t partial_bytes = static_cast<size_t>(tiles) * slots * 128 * kBN * sizeof(float);
  if (static_cast<size_t>(tiles) * kEpiWarps > kCounterInts || kCounterInts * 4 + partial_bytes > kScratchBytes)
    return DG_ERR_INVALID_ARG;   // the problem needs more scratch than the fixed array holds

  const int KP = ceil_div(num_kb, 4);
  const int NB = ceil_div(N, 128);
  CUtensorMap ta, tb, tsa, tsb, td;
  if (!encode(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, K, M, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, K, N, K, 128, kBN, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode(&tsa, CU_TENSOR_MAP_DATA_TYPE_INT32, sfa, 4 * ceil_div(M, 4), KP, 16 * ceil_div(M, 4), 128, 1,
              CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode(&tsb, CU_TENSOR_MAP_DATA_TYPE_INT32, sfb, 4 * ceil_div(NB, 4), KP, 16 * ceil_div(NB, 4), 8, 1,
              CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d, N, M, static_cast<uint64_t>(N) * 2, 64, 32,
              CU_TENSOR_MAP_SWIZZLE_128B))
    return DG_ERR_CUDA;

  // The scratch keeps whatever the previous call left: the arrival counters must start at zero.
  int* counters = reinterpret_cast<int*>(ds->scratch);
  if (cudaMemsetAsync(counters, 0, static_cast<size_t>(tiles) * kEpiWarps * sizeof(int), stream) != cudaSuccess)
    return DG_ERR_CUDA;

  dg::Params p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.G = 1;
  p.c = static_cast<const __nv_bfloat16*>(c);
  p.d = static_cast<__nv_bfloat16*>(d);
  p.status = status;
  p.timeout_ns = dg::pipeline_wait_timeout_ns();
  p.fault = dg::debug_fault_mode();
  p.sk_ctas = static_cast<int>(ctas);
  p.sk_slots = slots;
  p.sk_counters = counters;
  p.sk_ws = reinterpret_cast<float*>(ds->scratch + kCounterInts * 4);
  const cudaError_t e = c ? launch<true>(ta, tb, tsa, tsb, td, p, static_cast<int>(ctas), stream)
                          : launch<false>(ta, tb, tsa, tsb, td, p, static_cast<int>(ctas), stream);
  return e == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}
