/*
 * dg.h -- C ABI of the GB300 (sm_103a) fine-grained-scaled FP8 GEMM library (libdg.so).
 *
 * Operation (DeepGEMM README, as reproduced on the page "Weight gradient kernels for
 * dense and MoE models #95", section "Interfaces / Notices"): every GEMM is named after
 * D = C + A @ B and the suffix gives the storage of A and B; NT keeps A as is and reads B
 * transposed, so fp8_gemm_nt computes
 *
 *     D[m, n] = C[m, n] + sum_g sA[m, g] * sB[n / 128, g] * sum_{k = 128 g}^{128 g + 127} A[m, k] * B[n, k]
 *
 * with A and B in FP8 E4M3 (OCP "E4M3FN"), FP32 accumulation and a BF16 result.
 * Scale granularity: A has one scale per row per 128-wide K-group ("1x128"), B one
 * scale per 128x128 block. Scales are UE8M0 (code e means 2^(e-127)); on SM100 the same
 * section has them packed four to a 32-bit integer: K-group 4q+j is byte j (least
 * significant first) of word q. The section also asks for the LHS scales transposed and
 * padded for TMA: MN-major, with the MN extent padded to a multiple of 4 words (16 bytes).
 *
 * Notation used below: KG = K / 128, KP = ceil(KG / 4), NB = ceil(N / 128),
 * ceil4(x) = 4 * ceil(x / 4).
 *
 * Conventions shared by every entry point:
 *   - Every pointer argument of the GEMM calls is caller-owned DEVICE memory on the
 *     current device; the library never frees or retains it. Row-major means the
 *     last index is contiguous. All base pointers must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream). The returned
 *     status covers host-side validation and the launch only; errors detected on the
 *     device (bad expert index, masked count above max_m, a pipeline wait that timed
 *     out) are recorded in a library-owned device status word and reported by
 *     dg_get_device_status().
 *   - On a non-OK synchronous status nothing is launched and no memory is written.
 *   - Shape limits: K > 0 and K % 128 == 0; N > 0 and N % 16 == 0; M >= 0. An empty
 *     problem (M, M_total or max_m == 0) launches nothing, and its pointers may be NULL.
 *     Rows past M are never read or written.
 *   - Not thread-safe against concurrent dg_set_num_sms(); GEMM calls themselves may
 *     be issued from several host threads.
 *   - Library-owned device memory: a 4-byte status word per device, and a workspace per
 *     (device, stream) for the paths that need one (stream-K partials, the CTA-pair kernel's
 *     scale chunks), allocated in stream order on demand or reserved up front with
 *     dg_reserve_workspace (see there). No GEMM call synchronises the device or a stream.
 *   - CUDA graphs: a captured call uses the workspace its stream already has, so make one
 *     uncaptured call of at least the same size on the capturing stream first (allocating
 *     inside a capture works only in cudaStreamCaptureModeRelaxed). Nothing is freed during a
 *     capture, and a workspace used in one is kept until the process exits, so replays stay
 *     valid however many streams come later.
 */
#ifndef DG_H_
#define DG_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DG_OK = 0,
  DG_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, K % 128 != 0, N % 16 != 0, G <= 0 */
  DG_ERR_UNSUPPORTED = 2,   /* device is not sm_103, or a size past the library's limits */
  DG_ERR_MISALIGNED = 3,    /* a base pointer is not 16-byte aligned */
  DG_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed (see dg_last_cuda_error) */
  DG_ERR_TIMEOUT = 5,       /* device: a pipeline wait exceeded its time limit; the kernel exited */
  DG_ERR_BAD_INDEX = 6      /* device: m_indices[r] >= G or < -1, or masked_m[g] outside [0, max_m] */
} dg_status;

/*
 * Dense GEMM: D = C + A @ B.T ("Normal dense GEMMs (non-grouped)": fp8_gemm_nt).
 *   a   : E4M3 [M, K] row-major (K-major).
 *   sfa : int32 [KP, ceil4(M)]; word (q, m) packs the UE8M0 scales of row m for
 *         K-groups 4q..4q+3.
 *   b   : E4M3 [N, K] row-major (K-major), i.e. B.T is column-major.
 *   sfb : int32 [KP, ceil4(NB)]; word (q, j) packs the scales of the 128x128 block
 *         (rows 128j..128j+127 of b) for K-groups 4q..4q+3.
 *   c   : BF16 [M, N] row-major addend, or NULL for C = 0. May alias d exactly.
 *   d   : BF16 [M, N] row-major output; fully overwritten for rows < M.
 */
dg_status dg_fp8_gemm_nt(const void* a, const int32_t* sfa,
                         const void* b, const int32_t* sfb,
                         const void* c, void* d,
                         int M, int N, int K, cudaStream_t stream);

/*
 * The other memory layouts (README "Interfaces / Notices": the SM100 implementation supports
 * NT, TN, NN and TT; "Normal dense GEMMs": fp8_gemm_{nt, nn, tn, tt}). The same product
 * D = C + A' @ B'' of an M x K matrix A' and a K x N matrix B'', with A and B stored as:
 *   dg_fp8_gemm_nn : a = A' [M, K] row-major (K-major),  b = B'' [K, N] row-major (N-major)
 *   dg_fp8_gemm_tn : a = A'^T [K, M] row-major (M-major), b = B'' [K, N] row-major
 *   dg_fp8_gemm_tt : a = A'^T [K, M] row-major,          b = B''^T [N, K] row-major (as nt)
 * Scales do not depend on the storage: sfa holds one UE8M0 per row of A' (M) per 128-wide
 * K-group, sfb one per 128 (N) x 128 (K) block, packed as for dg_fp8_gemm_nt. An M-major A
 * needs M to be a multiple of 16 (its rows are M bytes); otherwise as dg_fp8_gemm_nt.
 */
dg_status dg_fp8_gemm_nn(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, const void* c,
                         void* d, int M, int N, int K, cudaStream_t stream);
dg_status dg_fp8_gemm_tn(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, const void* c,
                         void* d, int M, int N, int K, cudaStream_t stream);
dg_status dg_fp8_gemm_tt(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb, const void* c,
                         void* d, int M, int N, int K, cudaStream_t stream);

/*
 * Weight-gradient GEMM with FP32 output: D = C + A @ B.T (page "Weight gradient kernels
 * for dense and MoE models #95", wgrad_gemm_fp8_fp8_fp32_nt: FP8 x FP8 -> FP32, NT). The
 * pages give nothing beyond the name; the reading taken is the dense GEMM above with an
 * FP32 addend and output: the gradient accumulated so far is passed as C and may be D
 * itself (c == d), which then accumulates in place.
 *   a, sfa, b, sfb, M, N, K : as dg_fp8_gemm_nt (same scale format and constraints).
 *   c : float32 [M, N] row-major, or NULL (no addend); may alias d.
 *   d : float32 [M, N] row-major.
 * Errors as dg_fp8_gemm_nt. Asynchronous on `stream`.
 */
dg_status dg_wgrad_gemm_fp8_fp8_fp32_nt(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                        const float* c, float* d, int M, int N, int K, cudaStream_t stream);

/*
 * K-grouped weight-gradient GEMM for MoE experts, FP32 output (page "Weight gradient kernels
 * for dense and MoE models #95": k_grouped_wgrad_gemm_fp8_fp8_fp32_nt; README "Grouped GEMMs":
 * grouping along K, with M and N the same for every group). Expert g owns the K-slice
 * [off_g, off_g + ks[g]) of A and B, off_g = ks[0] + ... + ks[g-1], and D[g] = C[g] + A[:, slice_g] @ B[:, slice_g].T.
 *   a   : e4m3 [M, K_total] row-major (the experts' token columns concatenated along K).
 *   sfa : int32 [sf_k_rows][ceil4(M)] UE8M0 words packed per expert: expert g's K-groups
 *         j = 0, 1, ... in byte j % 4 of word row R_g + j / 4, R_g = sum over h < g of
 *         ceil(ks[h] / 512) (each expert starts a new word row).
 *   b   : e4m3 [N, K_total] row-major; sfb : int32 [sf_k_rows][ceil4(ceil(N/128))], the same
 *         per-expert packing over 128 x 128 blocks.
 *   c   : float32 [G, M, N] or NULL; may alias d.   d : float32 [G, M, N].
 *   ks  : DEVICE int32 [G], each a non-negative multiple of 128, summing to K_total; an
 *         expert with ks[g] = 0 gets D[g] = C[g] (zero without C).
 *   sf_k_rows : word rows of sfa / sfb (= sum over g of ceil(ks[g] / 512)).
 * Synchronous errors: G <= 0, M < 0, N not a positive multiple of 16, K_total not a
 * multiple of 128, null or misaligned pointers -> DG_ERR_INVALID_ARG / DG_ERR_MISALIGNED.
 * Device-detected: ks values that are negative, not multiples of 128, do not sum to K_total
 * or do not match sf_k_rows set DG_ERR_BAD_INDEX (reads stay within the declared extents).
 */
dg_status dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt(const void* a, const int32_t* sfa, const void* b,
                                                const int32_t* sfb, const float* c, float* d, const int32_t* ks,
                                                int G, int M, int N, int K_total, int sf_k_rows,
                                                cudaStream_t stream);

/*
 * K-grouped GEMM in the TN layout (README "Grouped GEMMs (contiguous layout)": the API that
 * groups K instead of M, meant for the weight gradient of MoE layers,
 * k_grouped_fp8_gemm_tn_contiguous). The same operation
 * and arguments as dg_k_grouped_wgrad_gemm_fp8_fp8_fp32_nt, with A and B stored token-major:
 *   a : E4M3 [K_total, M] row-major (M contiguous; M a multiple of 16),
 *   b : E4M3 [K_total, N] row-major (N contiguous),
 * so that D[g] = C[g] + A_g @ B_g.T with A_g = a[slice_g, :].T and B_g = b[slice_g, :].T.
 * Output FP32 (a weight gradient; the pages give no output type: the reading taken is the
 * K-grouped weight-gradient form's).
 */
dg_status dg_k_grouped_fp8_gemm_tn_contiguous(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                              const float* c, float* d, const int32_t* ks, int G, int M, int N,
                                              int K_total, int sf_k_rows, cudaStream_t stream);

/*
 * M-grouped GEMM, contiguous layout ("Grouped GEMMs (contiguous layout)":
 * m_grouped_fp8_gemm_nt_contiguous). Only M is grouped; N and K are shared by the G
 * experts. Each expert's token rows are concatenated along M, and each expert segment
 * starts on a multiple of dg_get_mk_alignment_for_contiguous_layout() rows; padding
 * rows are marked -1 in m_indices and form a suffix of their segment.
 *   a         : E4M3 [M_total, K] row-major.
 *   sfa       : int32 [KP, ceil4(M_total)] (as for dense A).
 *   b         : E4M3 [G, N, K] row-major (expert g's weights at b + g*N*K).
 *   sfb       : int32 [G, KP, ceil4(NB)] (expert g's block scales).
 *   d         : BF16 [M_total, N] row-major. Rows with m_indices == -1 are NOT written.
 *   m_indices : int32 [M_total] device array: expert of each row, -1 for padding.
 *               The expert of a 128-row block is read from its first row; a block whose
 *               first row is -1 is skipped entirely.
 */
dg_status dg_m_grouped_fp8_gemm_nt_contiguous(const void* a, const int32_t* sfa,
                                              const void* b, const int32_t* sfb,
                                              void* d, const int32_t* m_indices,
                                              int M_total, int N, int K, int G,
                                              cudaStream_t stream);

/*
 * Contiguous M-grouped GEMM with the weights stored N-major (README "Grouped GEMMs
 * (contiguous layout)": m_grouped_fp8_gemm_{nt, nn}_contiguous): as
 * dg_m_grouped_fp8_gemm_nt_contiguous except b = E4M3 [G, K, N] row-major (expert g's
 * weights at b + g*K*N, N contiguous), i.e. D = A @ B_g for rows of expert g. Scales as for
 * the NT form (sfb per 128 (N) x 128 (K) block of expert g).
 */
dg_status dg_m_grouped_fp8_gemm_nn_contiguous(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                                              void* d, const int32_t* m_indices, int M_total, int N, int K, int G,
                                              cudaStream_t stream);

/*
 * M-grouped GEMM, masked layout ("Grouped GEMMs (masked layout)":
 * m_grouped_fp8_gemm_nt_masked). For expert g only rows r < masked_m[g] are
 * computed; the counts are read on the device, so the call can be captured in a CUDA
 * graph while the host does not know them.
 *   a        : E4M3 [G, max_m, K] row-major.
 *   sfa      : int32 [G, KP, ceil4(max_m)].
 *   b        : E4M3 [G, N, K] row-major.
 *   sfb      : int32 [G, KP, ceil4(NB)].
 *   d        : BF16 [G, max_m, N] row-major. Rows r >= masked_m[g] are NOT written.
 *   masked_m : int32 [G] device array. A count above max_m is clamped to max_m and a
 *              negative one is treated as 0; both set DG_ERR_BAD_INDEX on the device.
 */
dg_status dg_m_grouped_fp8_gemm_nt_masked(const void* a, const int32_t* sfa,
                                          const void* b, const int32_t* sfb,
                                          void* d, const int32_t* masked_m,
                                          int G, int max_m, int N, int K,
                                          cudaStream_t stream);

/*
 * FP8 x FP4 GEMMs: D = C + A @ B.T with A in E4M3 and B in FP4 (DeepGEMM news entry of
 * 2026.04.16, "FP8xFP4 GEMM"; the Mega MoE section of the same README runs its linear layers
 * as FP8 x FP4 products, on FP4 weights that carry UE8M0 scales). The pages say no more; the
 * readings taken here:
 *   - B is OCP MX FP4 (E2M1: +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}), two codes per byte, element 2j
 *     of a row in the low nibble of byte j: b is uint8 [N, K/2] row-major.
 *   - B has one UE8M0 scale per row per 32 consecutive K-elements (the MX block), packed four
 *     per int32 along K and stored MN-major: sfb is int32 [KG, ceil4(N)], word (q, n) holding
 *     the scales of K-elements 128q + 32j .. 128q + 32j + 31 of row n in byte j.
 *   - A, sfa, c and d are exactly as in dg_fp8_gemm_nt (A scales 1 x 128, BF16 C and D).
 *     D[m, n] = C[m, n] + sum_k sA[m, k / 128] * sB[n, k / 32] * A[m, k] * B[n, k].
 * b must be 32-byte aligned (the 16U4 tensor-map type's rule), every other pointer 16-byte
 * aligned (DG_ERR_MISALIGNED otherwise). Shape limits and errors as dg_fp8_gemm_nt.
 */
dg_status dg_fp8_fp4_gemm_nt(const void* a, const int32_t* sfa, const void* b, const int32_t* sfb,
                             const void* c, void* d, int M, int N, int K, cudaStream_t stream);

/*
 * Contiguous M-grouped FP8 x FP4 GEMM: dg_m_grouped_fp8_gemm_nt_contiguous with each expert's
 * B in FP4 as above.
 *   b   : uint8 [G, N, K/2] (packed E2M1), 32-byte aligned.
 *   sfb : int32 [G, KG, ceil4(N)] (per-row, per-32 scales packed as for dg_fp8_fp4_gemm_nt).
 *   a, sfa, d, m_indices, M_total, N, K, G : as dg_m_grouped_fp8_gemm_nt_contiguous.
 */
dg_status dg_m_grouped_fp8_fp4_gemm_nt_contiguous(const void* a, const int32_t* sfa, const void* b,
                                                  const int32_t* sfb, void* d, const int32_t* m_indices,
                                                  int M_total, int N, int K, int G, cudaStream_t stream);

/*
 * Masked M-grouped FP8 x FP4 GEMM: dg_m_grouped_fp8_gemm_nt_masked with each expert's B in FP4.
 *   b   : uint8 [G, N, K/2] (packed E2M1), 32-byte aligned.
 *   sfb : int32 [G, KG, ceil4(N)].
 *   a, sfa, d, masked_m, G, max_m, N, K : as dg_m_grouped_fp8_gemm_nt_masked.
 */
dg_status dg_m_grouped_fp8_fp4_gemm_nt_masked(const void* a, const int32_t* sfa, const void* b,
                                              const int32_t* sfb, void* d, const int32_t* masked_m,
                                              int G, int max_m, int N, int K, cudaStream_t stream);

/*
 * Scale-factor packing ("Utilities": get_mn_major_tma_aligned_packed_ue8m0_tensor /
 * transform_sf_into_required_layout). Converts FP32 scales into the packed, MN-major,
 * TMA-aligned UE8M0 words the GEMMs consume.
 *   sf_fp32 : FP32 device array of one scale per row/block and K-group: [mn, kgroups]
 *             row-major (K-groups contiguous) when mn_major_in is 0, [kgroups, mn]
 *             row-major (rows contiguous) when it is 1; any other value of mn_major_in is
 *             DG_ERR_INVALID_ARG. Each value must be a positive finite number; it is rounded UP to
 *             the next power of two (exact powers of two are kept), then clamped to the
 *             UE8M0 range [2^-127, 2^127]. Non-positive or non-finite values encode 127
 *             (scale 1.0) and set DG_ERR_BAD_INDEX on the device.
 *   out     : int32 [ceil(kgroups/4), ceil4(mn)] device array, fully written (padding
 *             bytes and padding rows are 0).
 */
dg_status dg_pack_sf_ue8m0(const float* sf_fp32, int32_t* out, int mn, int kgroups, int mn_major_in,
                           cudaStream_t stream);

/*
 * Dense GEMM that allocates no device memory (the pages have no counterpart: this is an
 * extra entry point of this library).
 *
 * For callers that cannot allocate when they run the GEMM: servers that fix their
 * device-memory footprint at start-up and forbid later allocations, custom allocators that
 * own all of the device's memory, code under a memory budget where a lazy allocation could
 * fail in the middle of a step, or latency-critical loops that cannot afford the implicit
 * device synchronisation of cudaMalloc / cudaFree. dg_fp8_gemm_nt allocates on first use (a
 * status word, and for some shapes a per-stream workspace); this entry point uses instead a
 * fixed 16 MiB scratch array that the library holds in device memory from the first call on
 * each GPU until the process exits.
 *
 * Computes the same D = C + A @ B.T as dg_fp8_gemm_nt, with the same argument meanings and
 * layouts, on the library's single-CTA kernel in stream-K mode (128 x 128 tiles, one K-group
 * per pipeline stage, the K-groups of all tiles split among every SM of the device;
 * dg_set_num_sms does not apply), so results match dg_fp8_gemm_nt within the parity
 * tolerance. dg_set_debug's fault mode and wait limit apply to it as to every GEMM.
 *   status : caller-owned DEVICE uint32 word (4-byte aligned); device-side errors are OR-ed
 *            into it as bit (1 << DG_ERR_TIMEOUT). It is not cleared by the call.
 * Limits: the problem must fit the scratch: 16 KiB of counters (at most 1024 tiles of
 * 128x128) plus tiles x (largest contributor count of any tile) x 64 KiB of FP32 partials,
 * a conservative bound (the 128x7168x16384 decode shape needs 14.0 MiB of partials). Larger
 * problems return DG_ERR_INVALID_ARG with nothing launched; use dg_fp8_gemm_nt for them.
 * The first call on a device does its set-up: it looks up the scratch array's device
 * address and sets the kernels' shared-memory limit (once per device, with that device
 * current); make that first call before any stream capture. Every call shares the one array
 * and it keeps the previous call's contents: each call clears the counters it needs (an
 * asynchronous memset on `stream`) before its kernel. Calls whose work overlaps on the GPU
 * (different streams, or several host threads) race on the array: keep them ordered on one
 * stream. Calls no cudaMalloc / cudaFree and no allocating library routine.
 */
dg_status dg_fp8_gemm_nt_no_alloc(const void* a, const int32_t* sfa,
                                  const void* b, const int32_t* sfb,
                                  const void* c, void* d, uint32_t* status,
                                  int M, int N, int K, cudaStream_t stream);

/* Row (M) alignment of each expert segment in the contiguous layout, and K alignment of each
 * expert slice in the K-grouped form, that callers should pad to (README "Utilities":
 * set/get_mk_alignment_for_contiguous_layout). Default 128. The setter accepts positive
 * multiples of 128 up to 2^20 (the kernels accept any multiple of 128, so a larger value
 * only changes what callers are told to pad to) and returns DG_ERR_INVALID_ARG otherwise;
 * process-wide. The theoretical minimum ("get_theoretical_mk_alignment_for_contiguous_layout")
 * is the kernels' M block, 128. Host-only: no device is touched. */
int dg_get_mk_alignment_for_contiguous_layout(void);
dg_status dg_set_mk_alignment_for_contiguous_layout(int alignment);
int dg_get_theoretical_mk_alignment_for_contiguous_layout(void);

/* Smallest MN extent >= mn whose size in bytes is a multiple of 16 ("get_tma_aligned_size").
 * elem_bytes must be 1, 2, 4 or 8; returns -1 on a bad argument. */
int dg_get_tma_aligned_size(int mn, int elem_bytes);

/* Cap on the number of SMs the persistent kernels use ("set_num_sms / get_num_sms").
 * n <= 0 restores the default (all SMs of the device). Returns DG_ERR_INVALID_ARG if n
 * exceeds the device's SM count. */
dg_status dg_set_num_sms(int n);
int dg_get_num_sms(void);

/* Per-stream workspaces (no counterpart on the pages: memory management of this library).
 * Some paths need device scratch beyond the caller's buffers: stream-K (partial tiles and
 * arrival counters) and the CTA-pair kernel (scale chunks in the tensor-core copy layout, the
 * contiguous form's pair-row list). The library keeps one workspace per (device, stream),
 * allocated and freed in stream order (cudaMallocAsync / cudaFreeAsync): no GEMM call ever
 * synchronises the device or a stream.
 *   dg_reserve_workspace : makes the current device's workspace for `stream` at least `bytes`
 *     now (allocating in stream order) and keeps it until dg_release_workspace. Afterwards a
 *     GEMM call on that stream whose needs fit allocates, frees and synchronises nothing; a
 *     call that needs more grows it (in stream order). bytes = 0 keeps what the stream has, so
 *     one warm-up call followed by dg_reserve_workspace(stream, 0) pins that call's footprint.
 *     Returns DG_ERR_INVALID_ARG while `stream` is being captured into a graph.
 *   dg_release_workspace : frees it in `stream`'s order (call it before destroying a stream
 *     that had one reserved). A workspace a captured graph refers to is kept until exit.
 *   dg_get_workspace_size : its current size in bytes (0 if the stream has none).
 * Workspaces that are not reserved are created by the first call that needs one; at most 16
 * of them are kept per device, and a call on a further stream evicts the least recently used
 * one after its last use (an event, not a synchronisation). A workspace used inside a graph
 * capture is kept until the process exits. */
dg_status dg_reserve_workspace(cudaStream_t stream, size_t bytes);
dg_status dg_release_workspace(cudaStream_t stream);
size_t dg_get_workspace_size(cudaStream_t stream);

/* Programmatic dependent launch ("Utilities": set_pdl / get_pdl). When on, every GEMM
 * launch of the library (and the CTA-pair path's scale-preparation kernel) may begin its
 * prologue (barrier set-up, TMEM allocation, descriptor prefetch, an L2 prefetch of its first
 * operand boxes) while the preceding kernel in the stream is still running; each kernel
 * waits for that kernel's completion (griddepcontrol.wait) before it reads or writes any
 * global memory the preceding kernel may touch, so results do not depend on the setting.
 * On by default; the environment variable DG_PDL=0 makes the default off. dg_set_pdl takes
 * 1 (on) or 0 (off) and returns DG_ERR_INVALID_ARG for anything else; process-wide, for
 * launches made after the call. dg_get_pdl returns the current setting (1 or 0).
 * dg_fp8_gemm_nt_no_alloc launches without it. Host-only: no device is touched. */
dg_status dg_set_pdl(int enable);
int dg_get_pdl(void);

/* Synchronises `stream`, then returns (and clears) the first error recorded on the
 * current device by any earlier call: DG_ERR_TIMEOUT, DG_ERR_BAD_INDEX, or DG_OK. */
dg_status dg_get_device_status(cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char* dg_status_string(dg_status s);

/* The last CUDA error code seen by the library on this host thread (0 if none). */
int dg_last_cuda_error(void);

/*
 * Test hook for the failure-detection path (no counterpart on the pages).
 *   fault_mode      : 0 = none (default); 1 = the TMA producer of every later GEMM launch
 *                     issues no loads, so the MMA and epilogue waits run out and the
 *                     kernel exits with DG_ERR_TIMEOUT recorded in the status word.
 *   wait_timeout_ns : limit of every pipeline wait in later launches; 0 = default (2 s).
 * Process-wide; affects launches made after the call. Returns DG_ERR_INVALID_ARG for an
 * unknown fault_mode.
 */
dg_status dg_set_debug(int fault_mode, unsigned long long wait_timeout_ns);

/*
 * Diagnostic (no counterpart on the pages): the measured FP8 tensor-core ceiling of the
 * current device. Every SM runs one CTA that issues `iters_per_sm` x 4 block-scaled
 * 128 x 256 x 32 MMAs (kind::mxf8f6f4, E4M3, UE8M0 scales, FP32 accumulation in TMEM)
 * back to back from shared memory, with no other work; the grid is timed with CUDA events
 * on the legacy default stream. Writes the rate in TFLOP/s to *tflops and the kernel time
 * to *ms (ms may be NULL). Synchronous; allocates and frees a 4-byte status word.
 * Returns DG_ERR_INVALID_ARG for iters_per_sm outside [1, 2^20] or a null tflops,
 * DG_ERR_TIMEOUT if the kernel's bounded completion wait ran out, DG_ERR_CUDA otherwise
 * on failure.
 */
dg_status dg_measure_fp8_mma_tflops(int iters_per_sm, double* tflops, double* ms);

#ifdef __cplusplus
}
#endif

#endif /* DG_H_ */
