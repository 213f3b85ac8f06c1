/*
 * libnvfp4moe -- the NVFP4 block-scaled Mixture-of-Experts expert layer on
 * NVIDIA GB300 (sm_103a).
 *
 * The layer (route -> quantise -> permute -> grouped GEMM gate/up with fused
 * SwiGLU and NVFP4 requantisation -> grouped GEMM down -> weighted finalize)
 * is the hot path of the GLM-5-NVFP4 MoE deployment described on the source
 * pages:
 *   "SM120 FP4 Kernel Research Campaign"                      (page A)
 *   "Discovering SM120-Specific CUTLASS MoE Kernels"          (page B)
 *   "Uncovering SM120 CUTLASS Collective Implementations"     (page C)
 * Each call below cites the passage that defines its operation.
 *
 * NVFP4 (page A, section 1: the block-scaled MMA takes e2m1 data and ue4m3
 * scales, four scales per 64 K elements): values are FP4 E2M1 codes, two per
 * byte, element 2i in the LOW nibble of byte i; one unsigned E4M3 scale byte
 * per 16 consecutive elements along K; one FP32 per-tensor scale.  The value
 * of an element is e2m1(code) * ue4m3(scale) * s.
 *
 * Scale layouts.  "Row-major" scales are uint8 [rows, cols/16].  "Blocked"
 * scales are the tensor-core layout: rows are grouped in blocks of 128 and K
 * in blocks of 64 elements (4 scales); block (rb, kb) is 512 contiguous
 * bytes at offset (rb * (cols/64) + kb) * 512, and inside it the 4 scales of
 * row r (r = 0..127 within the block) sit at (r % 32) * 16 + (r / 32) * 4.
 * A blocked buffer holds ceil(rows/128)*128 rows (nvfp4moe_blocked_scales_bytes).
 *
 * Conventions for every call:
 *   - C ABI, returns a status code (NVFP4MOE_OK = 0 on success).  A non-zero
 *     status means nothing was launched; nvfp4moe_last_error_detail() gives
 *     a per-thread message.
 *   - Pointers marked "device" are device memory owned by the caller; the
 *     library never allocates, frees or keeps them.  Host pointers are
 *     marked "host".  Buffers must be 16-byte aligned.
 *   - Work is enqueued on `stream` and never synchronises.  Data-dependent
 *     scalars (global scales, counts) stay on the device.
 *   - Device-side checks (an expert id out of range, a pipeline wait that
 *     exceeded its time limit) do not fault: they skip the offending work and
 *     raise a sticky device flag that nvfp4moe_sync_status() reports.
 *   - Only compute capability 10.3 (GB300) is supported.
 *   - Kernels other than the grouped GEMM (and the cooperative moe_prepare
 *     kernel) are launched with programmatic dependent launch: such a kernel
 *     may be scheduled while the kernel before it in the stream drains, and
 *     waits for that kernel's completion before it reads or writes any
 *     buffer.  Stream order is therefore kept for every caller.
 *     NVFP4MOE_PDL=0 in the environment turns the overlap off.
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define NVFP4MOE_OK                 0
#define NVFP4MOE_ERR_INVALID_ARG    1  /* null/misaligned pointer, bad enum, negative size */
#define NVFP4MOE_ERR_UNSUPPORTED    2  /* shape outside the supported set, or device is not cc 10.3 */
#define NVFP4MOE_ERR_SMEM           3  /* tile pipeline does not fit the device's opt-in shared memory */
#define NVFP4MOE_ERR_WORKSPACE      4  /* workspace smaller than the matching *_workspace_size() */
#define NVFP4MOE_ERR_CUDA           5  /* CUDA runtime error (launch failure, driver entry point missing) */
#define NVFP4MOE_ERR_TIMEOUT        6  /* a device pipeline wait ran out of time (sticky, see sync_status) */
#define NVFP4MOE_ERR_DEVICE_DATA    7  /* device data out of range, e.g. an expert id >= E (sticky) */

/* ---- enums ------------------------------------------------------------- */
#define NVFP4MOE_SCORE_SOFTMAX      0
#define NVFP4MOE_SCORE_SIGMOID      1

#define NVFP4MOE_QUANT_COMPUTE_GLOBAL  1  /* compute s = amax/2688 into *global_scale */
#define NVFP4MOE_QUANT_SCALES_BLOCKED  2  /* write scales in the blocked layout */

#define NVFP4MOE_EPI_BF16           0  /* C = bf16(acc * s_a * s_w[e]) */
#define NVFP4MOE_EPI_SWIGLU_NVFP4   1  /* h = silu(gate) * up, requantised to NVFP4 */
#define NVFP4MOE_EPI_SWIGLU_F32     2  /* h = silu(gate) * up as float32 (unfused check) */
#define NVFP4MOE_EPI_SWIGLU_MXFP4   3  /* h = silu(gate) * up, requantised to MXFP4 (MXFP4 GEMM only) */
#define NVFP4MOE_EPI_FINALIZE_F32   4  /* out_f32[t] += w * bf16(acc) (moe_grouped_gemm_nvfp4_finalize only) */

/* Grouped GEMM tile_n values for token-major tiles (see moe_grouped_gemm_nvfp4). */
#define NVFP4MOE_TILE_TOKEN_MAJOR   (-1)
#define NVFP4MOE_TILE_TOKEN_MAJOR_PAIR (-2)

/* ---- library and device ------------------------------------------------- */

/* Version as major*10000 + minor*100 + patch. */
int nvfp4moe_version(void);

/* Static description of a status code (never NULL). */
const char* nvfp4moe_status_string(int status);

/* Message of the last failed call on the calling host thread ("" if none). */
const char* nvfp4moe_last_error_detail(void);

/* Checks that `device` is a compute capability 10.3 GPU and caches its SM
 * count and opt-in shared memory.  Returns OK, UNSUPPORTED or CUDA. */
int nvfp4moe_device_check(int device);

/* Synchronises `stream`, then reads and clears the sticky device flags
 * raised by earlier calls on the current device.  Returns OK, TIMEOUT,
 * DEVICE_DATA or CUDA. */
int nvfp4moe_sync_status(cudaStream_t stream);

/* Time limit of every bounded device wait of the pipelines -- the mbarrier
 * waits of the grouped GEMM's producer, MMA, scale-factor and epilogue
 * roles, and the grid barriers of moe_prepare -- in microseconds, for the
 * calls launched after it is set (process-wide, all devices).  A wait that
 * exceeds it abandons its kernel without faulting, the kernel raises the
 * sticky TIMEOUT flag and nvfp4moe_sync_status() returns
 * NVFP4MOE_ERR_TIMEOUT (the opaque "Error Internal" failures that page C,
 * "The Thinking Process", runs into are what this status replaces).  A
 * serving loop can lower it to notice a stuck pipeline sooner; a limit
 * shorter than a wait that legitimately occurs (a stage's operands, a
 * tile's accumulator, a grid barrier: microseconds) aborts healthy calls.
 * 0 restores the default, 2000000 (2 s); at most 60000000.  Returns OK or
 * INVALID_ARG.  After a TIMEOUT, zero moe_prepare's workspace again. */
int nvfp4moe_set_wait_limit_us(uint32_t us);
uint32_t nvfp4moe_wait_limit_us(void);

/* Self-test of the bounded waits: one CTA waits, through the grouped GEMM's
 * bounded mbarrier wait and under the current wait limit, for the phase of
 * a shared-memory mbarrier that expects `expected_arrivals` (1..64)
 * arrivals and receives `arrivals` (0..32, one per thread).  With arrivals
 * < expected_arrivals the phase can never complete: the wait gives up after
 * the limit and the next nvfp4moe_sync_status() returns
 * NVFP4MOE_ERR_TIMEOUT; otherwise OK.  Enqueued on `stream`; no memory is
 * touched besides the flag.  No counterpart on the source pages. */
int nvfp4moe_wait_selftest(uint32_t expected_arrivals, uint32_t arrivals, cudaStream_t stream);

/* Bytes of a blocked scale buffer for a [rows, cols] NVFP4 matrix
 * (cols % 64 == 0): ceil(rows/128) * 128 * cols / 16.  0 on bad input. */
size_t nvfp4moe_blocked_scales_bytes(int64_t rows, int64_t cols);
/* Bytes of an MXFP4 blocked scale buffer (see the MXFP4 section): 0 unless cols % 128 == 0. */
size_t nvfp4moe_mxfp4_blocked_scales_bytes(int64_t rows, int64_t cols);

/* Tiled weight layout (NVFP4MOE_W_TILED), an offline re-layout of packed
 * E2M1 weights (NVFP4 or MXFP4 codes alike) for the grouped GEMM: the
 * grouped GEMM reads a weight tile 128 rows x 128 bytes at a time, which in
 * the row-major layout are 128 strips K/2 bytes apart; tiled, each such box
 * is 16384 contiguous bytes (measured on GB300: 6.9 TB/s for the strided
 * boxes of a 3 KB-row matrix, 7.2 TB/s contiguous).  For packed [rows, K/2]
 * (rows % 128 == 0, K % 64 == 0), KC = ceil(K / 256): block (rb, kc), rb <
 * rows / 128, kc < KC, starts at byte (rb * KC + kc) * 16384 and holds
 * bytes [kc * 128, kc * 128 + 128) of rows rb * 128 .. rb * 128 + 127, row by
 * row; bytes past K/2 are zero.  Scales keep their layout. */
#define NVFP4MOE_W_ROWMAJOR 0
#define NVFP4MOE_W_TILED    1
/* Bytes of the tiled copy of a [rows, K/2] packed matrix; 0 on bad input. */
size_t nvfp4moe_tiled_weights_bytes(int64_t rows, int K);
/* Writes the tiled copy of w_packed (device uint8 [rows, K/2], 16-byte
 * aligned) to w_tiled (device, nvfp4moe_tiled_weights_bytes bytes, 16-byte
 * aligned), asynchronously on `stream`.  Returns OK, INVALID_ARG,
 * UNSUPPORTED (rows % 128 or K % 64) or CUDA. */
int nvfp4moe_tile_weights(const uint8_t* w_packed, int64_t rows, int K, uint8_t* w_tiled, cudaStream_t stream);

/* ---- a1: routing ---------------------------------------------------------
 * Top-k expert selection with sigmoid scoring (page A, key finding 8 and its
 * closing paragraph, which name sigmoid as the GLM-5 router's score
 * function) or softmax.  Selection compares float32 v = logits + bias, descending, the
 * lower expert index first on ties; slot j of a token holds its j-th
 * largest v.  Weights (computed in float64, stored float32):
 *   softmax: exp(v_j - max v) / sum over the k selected (renormalize = 1)
 *            or over all E (renormalize = 0);
 *   sigmoid: sigma(v_j), divided by the sum over the k selected when
 *            renormalize = 1.
 * logits  device float32 [T, E] row-major; bias device float32 [E] or NULL;
 * topk_idx device int32 [T, k]; topk_w device float32 [T, k].
 * Limits: 1 <= E <= 1024, 1 <= k <= min(E, 32), T >= 0 (T = 0 is a no-op).
 * NaN logits give an unspecified (but in-range) selection. */
int moe_route_topk(const float* logits, const float* bias, int T, int E, int k,
                   int score_fn, int renormalize,
                   int32_t* topk_idx, float* topk_w, cudaStream_t stream);

/* Batch-aware ("opportunistic") expert routing (page A, Introduction, key
 * finding 6 and section 6: during decode a token trades the experts it
 * weights least for experts other tokens of the batch use already, so
 * fewer experts' weights are streamed; the pages give no algorithm).  This library's reading:
 *   1. each token's primary experts are its top-k_primary by logit + bias
 *      (order and ties as moe_route_topk);
 *   2. the batch's active set S is the union of all tokens' primary experts;
 *   3. each token takes k experts ranked by (member of S first, then value
 *      descending, then lower index): its best k within S, followed -- only
 *      when S holds fewer than k experts -- by its best experts outside S;
 *      slots keep that order;
 *   4. weights as moe_route_topk over the chosen experts.
 * k_primary == k is moe_route_topk.  Same arguments as moe_route_topk plus
 * k_primary in [1, k] and ws: device scratch of at least
 * moe_route_batch_aware_workspace_size(E) bytes, 4-byte aligned (the set S,
 * cleared by the call).  Two kernels and one memset. */
size_t moe_route_batch_aware_workspace_size(int E);
int moe_route_batch_aware(const float* logits, const float* bias, int T, int E, int k, int k_primary,
                          int score_fn, int renormalize, int32_t* topk_idx, float* topk_w,
                          void* ws, size_t ws_bytes, cudaStream_t stream);

/* ---- a2: quantisation ----------------------------------------------------
 * bf16 -> NVFP4 (page A, section 1 operand types; four ue4m3 scales per k64
 * MMA step means one scale per 16 elements).  Per 16-element block along a
 * row: a = max|x|, t = (a / 6) / s in float32, scale byte b = t rounded to
 * the nearest ue4m3 (ties to even, saturating at 448), d = ue4m3(b) * s,
 * code = x / d rounded to the nearest E2M1 (ties to even, saturating at 6)
 * with the sign bit of x; b == 0 gives code 0 for the block.
 * x device bf16 [rows, cols] row-major, cols % 16 == 0
 *   (cols % 64 == 0 with NVFP4MOE_QUANT_SCALES_BLOCKED).
 * global_scale device float32 [1]: read as s, or, with
 *   NVFP4MOE_QUANT_COMPUTE_GLOBAL, written with s = amax(|x|)/2688 (1 if
 *   the tensor is zero) and then used.
 * packed device uint8 [rows, cols/2]; scales device uint8, row-major
 *   [rows, cols/16] or blocked (nvfp4moe_blocked_scales_bytes(rows, cols);
 *   padding rows of the last block are written as 0).
 * ws device workspace of moe_quantize_nvfp4_workspace_size() bytes (may be
 *   NULL when that is 0).  rows = 0 is a no-op (global_scale untouched).
 * NaN or infinite inputs are not supported. */
size_t moe_quantize_nvfp4_workspace_size(int64_t rows, int64_t cols, int flags);
int moe_quantize_nvfp4(const void* x_bf16, int64_t rows, int64_t cols,
                       float* global_scale, int flags,
                       uint8_t* packed, uint8_t* scales,
                       void* ws, size_t ws_bytes, cudaStream_t stream);

/* Row-major scales [rows, cols/16] -> blocked layout (cols % 64 == 0), for
 * NVFP4 data quantised elsewhere.  Padding rows are written as 0. */
int moe_scales_to_blocked(const uint8_t* scales_row_major, int64_t rows, int64_t cols,
                          uint8_t* scales_blocked, cudaStream_t stream);

/* ---- a3: permutation -----------------------------------------------------
 * Expert-first layout with token reordering (page A, section 6: two of its
 * listed techniques, the expert-first layout and reordering tokens so that
 * a fused reduction can gather them back).  Flat id
 * f = t*k + j.  Expert e's rows are the flat ids routed to e in ascending
 * f.  Each expert's rows start at a multiple of 128 in the permuted
 * buffers ("row_offsets"), so that a tensor-core tile never mixes experts.
 * Inputs: topk_idx device int32 [T, k]; xq device uint8 [T, H/2] and
 *   xs device uint8 [T, H/16] (row-major scales) from moe_quantize_nvfp4.
 * Outputs (device):
 *   expert_counts int32 [E]; expert_offsets int32 [E+1] (exclusive scan of
 *   the counts: the unpadded expert-first order); row_offsets int32 [E+1]
 *   (exclusive scan of counts rounded up to 128);
 *   perm_to_flat int32 [rows_capacity]: flat id held by each padded row,
 *   -1 for padding rows; flat_to_perm int32 [T*k]: padded row of each flat id;
 *   a_packed uint8 [rows_capacity, H/2]: row row_offsets[e] + r is the
 *   quantised token of expert e's r-th flat id (padding rows untouched);
 *   a_scales uint8, blocked layout over rows_capacity rows.
 * rows_capacity = moe_permute_rows_capacity(T, E, k).
 * Limits: H % 64 == 0, 1 <= E <= 1024, 1 <= k <= E.  An expert id outside
 * [0, E) is skipped and raises NVFP4MOE_ERR_DEVICE_DATA (sticky). */
int64_t moe_permute_rows_capacity(int T, int E, int k);
size_t moe_permute_workspace_size(int T, int E, int k);
int moe_permute(const int32_t* topk_idx, int T, int E, int k,
                const uint8_t* xq, const uint8_t* xs, int H,
                int32_t* expert_counts, int32_t* expert_offsets, int32_t* row_offsets,
                int32_t* perm_to_flat, int32_t* flat_to_perm,
                uint8_t* a_packed, uint8_t* a_scales,
                void* ws, size_t ws_bytes, cudaStream_t stream);

/* moe_permute without a workspace argument.  No counterpart on the source
 * pages: it exists for callers that cannot allocate device memory when they
 * call -- code running inside a fixed device-memory arena it may not grow,
 * plugins or foreign-function callers that are handed tensors but no
 * allocator, and hot loops where any cudaMalloc/cudaFree (which can
 * synchronise the device) is not acceptable.
 * Same arguments, outputs and limits as moe_permute, minus ws/ws_bytes.  The
 * scratch is a 1 MiB array inside the library (a file-scope device array,
 * resident on every GPU that loads the library until the process exits):
 * at most 131072 routed rows (T*k) and 65536 segment-expert counters
 * (ceil(T*k/1024) * E); larger calls return NVFP4MOE_ERR_UNSUPPORTED
 * without launching.  Nothing is allocated or freed.
 * Each call made outside stream capture looks up the array's device address
 * (cudaGetSymbolAddress) with the calling thread's device current.  A call
 * made while its stream is being captured cannot do that lookup and reuses
 * the address found by the last uncaptured call on the same CUDA context;
 * if there was none (first call on this device, or the device was reset
 * since, which gives it a new context and may move the array), it returns
 * NVFP4MOE_ERR_UNSUPPORTED without launching: make one uncaptured call on
 * each device, and again after a device reset, before capturing.
 * Every call shares the one array and overwrites the part it uses, so no
 * state carries over between calls, but calls whose work overlaps on the
 * GPU (other streams, other host threads) race on it: serialise them. */
int moe_permute_no_alloc(const int32_t* topk_idx, int T, int E, int k,
                         const uint8_t* xq, const uint8_t* xs, int H,
                         int32_t* expert_counts, int32_t* expert_offsets, int32_t* row_offsets,
                         int32_t* perm_to_flat, int32_t* flat_to_perm,
                         uint8_t* a_packed, uint8_t* a_scales, cudaStream_t stream);

/* ---- a1 + a2 + a3 in one launch -------------------------------------------
 * moe_route_topk, moe_quantize_nvfp4 (NVFP4MOE_QUANT_COMPUTE_GLOBAL,
 * row-major scales) and moe_permute fused into one cooperative kernel, for
 * decode-sized batches where each separate launch costs more than its work
 * (page A, Research Report sections 2-4 and Key Findings item 8: a MoE path
 * that is fast at large batch loses at interactive batch sizes to its
 * preprocessing; page B, Discovery: the fused-MoE module's enable_pdl
 * option).  The kernel keeps every CTA resident and separates the steps by
 * grid-wide barriers: route and the partial amax of x, then the global scale,
 * quantisation and segment ranks, then the expert scan, then placement and
 * the gather.  Every output is bit-identical to the three separate calls:
 *   topk_idx, topk_w [T, k] as moe_route_topk (logits device float32 [T, E],
 *     bias device float32 [E] or NULL, score_fn, renormalize) when
 *     k_primary == k, as moe_route_batch_aware when 1 <= k_primary < k (one
 *     more grid barrier);
 *   x_gscale device float32 [1], xq uint8 [T, H/2], xs uint8 [T, H/16] as
 *     moe_quantize_nvfp4 of x (device bf16 [T, H]);
 *   expert_counts .. a_scales as moe_permute (rows_capacity =
 *     moe_permute_rows_capacity(T, E, k)).
 * Limits: T >= 0, 1 <= E <= 1024, 1 <= k <= min(E, 32), H % 64 == 0,
 * T*k <= 2^30.  ws: device, at least moe_prepare_workspace_size(T, E, k)
 * bytes, 256-byte aligned, ZERO-FILLED before its first use (its first 256
 * bytes hold the grid-barrier words; every call that completes leaves them
 * ready for the next call, so zero it once).  After a call that raised
 * NVFP4MOE_ERR_TIMEOUT, zero it again.  Calls sharing one workspace must not
 * overlap on the GPU.  A barrier wait that exceeds its time limit abandons
 * the kernel and raises NVFP4MOE_ERR_TIMEOUT (sticky). */
size_t moe_prepare_workspace_size(int T, int E, int k);
int moe_prepare(const float* logits, const float* bias, const void* x_bf16,
                int T, int E, int k, int k_primary, int H, int score_fn, int renormalize,
                int32_t* topk_idx, float* topk_w, float* x_gscale, uint8_t* xq, uint8_t* xs,
                int32_t* expert_counts, int32_t* expert_offsets, int32_t* row_offsets,
                int32_t* perm_to_flat, int32_t* flat_to_perm,
                uint8_t* a_packed, uint8_t* a_scales,
                void* ws, size_t ws_bytes, cudaStream_t stream);

/* ---- a4/a5: grouped GEMM ---------------------------------------------------
 * The grouped ("array") block-scaled GEMM over experts (page C, Context and
 * the sm120_mma_array_tma_blockwise_scaling collective it finds; page A,
 * section 7: warp-specialised schedules).  For every expert e and every
 * valid row r of e (row = row_offsets[e] + r, r < expert_counts[e]):
 *   acc[row, n] = sum_K A[row, :] * W[e, n, :]   (dequantised, fp32 accumulate)
 * scaled by a_gscale[0] * w_gscale[e].  Epilogues:
 *   NVFP4MOE_EPI_BF16:        c_out bf16 [rows_capacity, N] = bf16(acc).
 *   NVFP4MOE_EPI_SWIGLU_NVFP4: N = 2*I, W rows [0, I) are the gate and
 *       [I, 2I) the up projection; h = silu(gate) * up (float32) is
 *       quantised with per-tensor scale c_gscale[0] exactly as
 *       moe_quantize_nvfp4 does: c_out uint8 [rows_capacity, I/2] packed,
 *       c_scales blocked over rows_capacity rows with I columns.
 *   NVFP4MOE_EPI_SWIGLU_F32:  h as float32, c_out [rows_capacity, I].
 * Padding rows of the outputs are left untouched.
 * a_packed device uint8 [rows_capacity, K/2]; a_scales device blocked;
 * a_gscale device float32 [1]; expert_counts / row_offsets device int32 as
 * written by moe_permute; w_packed device uint8 [E, N, K/2]; w_scales
 * device, blocked per expert ([E] x nvfp4moe_blocked_scales_bytes(N, K));
 * w_gscale device float32 [E].  w_layout: NVFP4MOE_W_ROWMAJOR (w_packed as
 * above) or NVFP4MOE_W_TILED (w_packed is nvfp4moe_tile_weights of that
 * [E*N, K/2] matrix; the same results).
 * m_total = number of routed rows (T*k); it only guides the choice of tiles.
 * tile_n selects the tile orientation.  128, or 256 with NVFP4MOE_EPI_BF16:
 * the widest token tile with weight rows as the MMA's 128-row M side; token
 * tiles start on 128-row boundaries of an expert's rows and each tile's MMA
 * width is the smallest of 32, 64, 128, 256 covering the rows left (capped
 * at tile_n), so a decode expert with 4 rows runs 128 x 32 MMAs.
 * NVFP4MOE_TILE_TOKEN_MAJOR (N % 256 == 0): 128 tokens as M and two 128-row
 * weight tiles (gate and up, or two consecutive output blocks) as one
 * N = 256 operand, which reads each token tile once per K step (for experts
 * with many rows; a partial tile still computes 128 token rows).
 * NVFP4MOE_TILE_TOKEN_MAJOR_PAIR (N % 256 == 0): the same tiles on a pair
 * of neighbouring SMs (a two-CTA cluster issuing cta_group::2 MMAs): 256
 * tokens as M, 128 in each SM, and the 256 weight rows split between the
 * two SMs' shared memory, so each SM stages half the weight bytes per K
 * step; a partial tile still computes 256 token rows.  Runs the static
 * schedule (the workspace is not used).
 * 0: when N % 256 == 0, token-major on CTA pairs from m_total >= 512 * E,
 * token-major from m_total >= 64 * E; otherwise 128.
 * The results do not depend on tile_n beyond float32 summation order.
 * Limits: K % 64 == 0; N % 128 == 0 (BF16) or N % 256 == 0 (SwiGLU);
 * 1 <= E <= 1024; rows_capacity % 128 == 0.  A pipeline that does not fit the
 * device's opt-in shared memory is refused with NVFP4MOE_ERR_SMEM (the
 * message gives the bytes required and the limit, cf. the OutOfResources
 * failure quoted on page A, section "The Research Task").
 * ws: NULL, or a device workspace of moe_grouped_gemm_nvfp4_workspace_size()
 * bytes (256), 256-byte aligned and ZERO-FILLED before its first use.  With a
 * workspace the persistent CTAs claim tiles from a launch-wide counter
 * (dynamic schedule: faster SMs take more tiles); the last CTA to finish
 * leaves the workspace zeroed for the next call, also after a timeout.
 * Without one, CTA c takes tiles c, c + #SMs, ...  Results are identical
 * either way.  Calls sharing a workspace must not overlap on the GPU. */
size_t moe_grouped_gemm_nvfp4_workspace_size(int E, int N, int K, int epilogue);
/* The tile orientation a grouped GEMM call with these arguments runs: tile_n
 * itself when it is not 0 (or N % 256 != 0), else the automatic choice
 * above (NVFP4MOE_TILE_TOKEN_MAJOR_PAIR, NVFP4MOE_TILE_TOKEN_MAJOR or 0 =
 * 128-token tiles with weight rows as M).  Host only; no device access. */
int nvfp4moe_gemm_tile_choice(int E, int N, int64_t m_total, int tile_n);
int moe_grouped_gemm_nvfp4(const uint8_t* a_packed, const uint8_t* a_scales, const float* a_gscale,
                           const int32_t* expert_counts, const int32_t* row_offsets,
                           int E, int64_t rows_capacity, int64_t m_total,
                           const uint8_t* w_packed, const uint8_t* w_scales, const float* w_gscale,
                           int N, int K, int epilogue, const float* c_gscale,
                           void* c_out, uint8_t* c_scales, int tile_n, int w_layout,
                           void* ws, size_t ws_bytes, cudaStream_t stream);

/* moe_grouped_gemm_nvfp4 restricted to the experts whose row count
 * (expert_counts[e], read on the device) lies in [min_rows, max_rows); the
 * other experts' output rows are left untouched.  Two calls over
 * complementary ranges, each with its own tile_n, give the same outputs as
 * one call over all experts (up to float32 summation order): a layer with
 * a few experts holding hundreds of rows and many holding a handful can
 * run the first on token-major tiles and the rest with weight rows as M.
 * m_total should then be the routed rows the call is expected to cover; it
 * only guides tile_n = 0.  1 <= min_rows <= max_rows; otherwise as
 * moe_grouped_gemm_nvfp4 (which is this call with [1, INT32_MAX)).  No
 * counterpart on the source pages beyond their per-regime tile choices. */
int moe_grouped_gemm_nvfp4_range(const uint8_t* a_packed, const uint8_t* a_scales, const float* a_gscale,
                                 const int32_t* expert_counts, const int32_t* row_offsets,
                                 int E, int64_t rows_capacity, int64_t m_total,
                                 const uint8_t* w_packed, const uint8_t* w_scales, const float* w_gscale,
                                 int N, int K, int epilogue, const float* c_gscale,
                                 void* c_out, uint8_t* c_scales, int tile_n, int w_layout,
                                 int32_t min_rows, int32_t max_rows,
                                 void* ws, size_t ws_bytes, cudaStream_t stream);

/* a5 with a6 fused into its epilogue (page C, Context: the grouped GEMM's
 * finalize epilogue; page A, section 6: token reordering with a fused
 * reduction).  The down projection of every valid row r of the experts in
 * [min_rows, max_rows) is rounded to bf16 as in NVFP4MOE_EPI_BF16 (Y), then
 * topk_w[f] * Y[r] is added into out_f32[f / k] with f = perm_to_flat[r]
 * by float32 atomic adds; nothing is written to a [rows, N] buffer.  The
 * order of the k additions into a token's row is not fixed, so unlike
 * moe_finalize the float32 sum is not bit-reproducible from call to call
 * (the difference is float32 rounding).  out_f32: device float32 [T, N],
 * zero before the call (moe_finalize_f32 converts it to bf16 and zeroes it
 * again).  perm_to_flat [rows_capacity] and topk_w [T, k] as written by
 * moe_permute / moe_route_topk.  Other arguments as moe_grouped_gemm_nvfp4_range
 * with epilogue NVFP4MOE_EPI_FINALIZE_F32. */
int moe_grouped_gemm_nvfp4_finalize(const uint8_t* a_packed, const uint8_t* a_scales, const float* a_gscale,
                                    const int32_t* expert_counts, const int32_t* row_offsets,
                                    int E, int64_t rows_capacity, int64_t m_total,
                                    const uint8_t* w_packed, const uint8_t* w_scales, const float* w_gscale,
                                    int N, int K, const int32_t* perm_to_flat, const float* topk_w, int T, int k,
                                    float* out_f32, int tile_n, int w_layout, int32_t min_rows, int32_t max_rows,
                                    void* ws, size_t ws_bytes, cudaStream_t stream);
/* out_bf16 [T, H] = bf16(acc_f32 [T, H]) (round to nearest even), and
 * acc_f32 = 0 afterwards, ready for the next moe_grouped_gemm_nvfp4_finalize.
 * H % 8 == 0; both device pointers 16-byte aligned. */
int moe_finalize_f32(float* acc_f32, int T, int H, void* out_bf16, cudaStream_t stream);

/* ---- MXFP4 variant of a2, a3, a4/a5 -----------------------------------------
 * MXFP4 (page A, sections 2-4: the MXFP4 grouped GEMM that works with
 * specific tile parameters; the pages give the format's name only, so the
 * library takes the OCP microscaling definition): E2M1 values, two per byte
 * as for NVFP4, one E8M0 scale byte per 32 consecutive elements along K
 * (value 2^(b - 127)), no per-tensor scale.  Quantisation of a 32-element
 * block: X = floor(log2(amax)) - 2, clamped to [-127, 127] (-127 for an
 * all-zero block), scale byte X + 127, codes = nearest E2M1 of x / 2^X,
 * ties to the even code, saturating at 6, sign of x.
 * Scale layouts: row-major uint8 [rows, cols/32], or blocked: blocks of 128
 * rows x 128 K elements (4 scales per row), 512 contiguous bytes at
 * (rb * (cols/128) + kb) * 512, row r's 4 scales at (r % 32) * 16 +
 * (r / 32) * 4 (nvfp4moe_mxfp4_blocked_scales_bytes).
 *
 * moe_quantize_mxfp4: x device bf16 [rows, cols] -> packed [rows, cols/2],
 *   scales row-major or blocked (flags NVFP4MOE_QUANT_SCALES_BLOCKED, which
 *   needs cols % 128 == 0; padding rows of a blocked buffer get scale 0).
 *   cols % 32 == 0.  No workspace.
 * moe_permute_mxfp4: moe_permute for MXFP4 rows (xs row-major [T, H/32],
 *   a_scales blocked MXFP4 over rows_capacity rows); H % 128 == 0; the
 *   workspace is moe_permute_workspace_size(T, E, k).
 * moe_grouped_gemm_mxfp4: moe_grouped_gemm_nvfp4 for MXFP4 operands
 *   (kind::mxf4nvf4 with ue8m0 scales, scale_vec::2X): no a_gscale,
 *   w_gscale or c_gscale; w_scales blocked per expert ([E] x
 *   nvfp4moe_mxfp4_blocked_scales_bytes(N, K)); K % 128 == 0; epilogues
 *   NVFP4MOE_EPI_BF16, NVFP4MOE_EPI_SWIGLU_MXFP4 (c_out packed [rows_capacity,
 *   I/2], c_scales blocked MXFP4 over rows_capacity rows with I columns,
 *   quantised as moe_quantize_mxfp4) or NVFP4MOE_EPI_SWIGLU_F32; ws as for
 *   moe_grouped_gemm_nvfp4. */
int moe_quantize_mxfp4(const void* x_bf16, int64_t rows, int64_t cols, int flags,
                       uint8_t* packed, uint8_t* scales, cudaStream_t stream);
int moe_permute_mxfp4(const int32_t* topk_idx, int T, int E, int k,
                      const uint8_t* xq, const uint8_t* xs, int H,
                      int32_t* expert_counts, int32_t* expert_offsets, int32_t* row_offsets,
                      int32_t* perm_to_flat, int32_t* flat_to_perm,
                      uint8_t* a_packed, uint8_t* a_scales,
                      void* ws, size_t ws_bytes, cudaStream_t stream);
/* moe_prepare for the MXFP4 layer: route (as moe_prepare, k_primary
 * included), quantise x by moe_quantize_mxfp4 (xq [T, H/2], row-major xs
 * [T, H/32]; no global scale) and permute as moe_permute_mxfp4, in one
 * cooperative launch.  H % 128 == 0; the workspace is
 * moe_prepare_workspace_size(T, E, k), zero-filled once, as for moe_prepare. */
int moe_prepare_mxfp4(const float* logits, const float* bias, const void* x_bf16,
                      int T, int E, int k, int k_primary, int H, int score_fn, int renormalize,
                      int32_t* topk_idx, float* topk_w, uint8_t* xq, uint8_t* xs,
                      int32_t* expert_counts, int32_t* expert_offsets, int32_t* row_offsets,
                      int32_t* perm_to_flat, int32_t* flat_to_perm,
                      uint8_t* a_packed, uint8_t* a_scales,
                      void* ws, size_t ws_bytes, cudaStream_t stream);
int moe_grouped_gemm_mxfp4(const uint8_t* a_packed, const uint8_t* a_scales,
                           const int32_t* expert_counts, const int32_t* row_offsets,
                           int E, int64_t rows_capacity, int64_t m_total,
                           const uint8_t* w_packed, const uint8_t* w_scales,
                           int N, int K, int epilogue, void* c_out, uint8_t* c_scales, int tile_n,
                           int w_layout, void* ws, size_t ws_bytes, cudaStream_t stream);
/* moe_grouped_gemm_mxfp4 restricted to experts with min_rows <= rows <
 * max_rows (see moe_grouped_gemm_nvfp4_range). */
int moe_grouped_gemm_mxfp4_range(const uint8_t* a_packed, const uint8_t* a_scales,
                                 const int32_t* expert_counts, const int32_t* row_offsets,
                                 int E, int64_t rows_capacity, int64_t m_total,
                                 const uint8_t* w_packed, const uint8_t* w_scales,
                                 int N, int K, int epilogue, void* c_out, uint8_t* c_scales, int tile_n,
                                 int w_layout, int32_t min_rows, int32_t max_rows,
                                 void* ws, size_t ws_bytes, cudaStream_t stream);

/* ---- a6: finalize ----------------------------------------------------------
 * Router-weighted reduce back to token order (page A, section 6: the
 * technique that reorders tokens by expert and fuses the weighted sum back;
 * page C, Context: the finalize epilogue): out[t, :] = sum_{j<k} topk_w[t, j] * y[flat_to_perm[t*k + j], :]
 * accumulated in float32 in slot order, stored as bf16.
 * y device bf16 [rows_capacity, H]; flat_to_perm device int32 [T*k];
 * topk_w device float32 [T, k]; out device bf16 [T, H].  H % 8 == 0.
 * A row index outside [0, rows_capacity) contributes nothing and raises
 * NVFP4MOE_ERR_DEVICE_DATA (sticky). */
int moe_finalize(const void* y_bf16, const int32_t* flat_to_perm, const float* topk_w,
                 int T, int k, int H, int64_t rows_capacity,
                 void* out_bf16, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4MOE_H */
