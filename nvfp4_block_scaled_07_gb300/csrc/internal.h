// Host-side launchers shared between the translation units of libnvfp4moe.
// Arguments are validated by the C entry points (api.cu) before any launcher
// is called; launchers only configure grids and enqueue kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace nvfp4moe {

// Device flag bits (sticky until nvfp4moe_sync_status reads them).
constexpr unsigned kFlagTimeout = 1u;
constexpr unsigned kFlagBadData = 2u;

// Limit of every bounded device wait of the pipelines (mbarrier waits of
// the grouped GEMM, grid barriers of the prepare kernel), in microseconds:
// the value of nvfp4moe_set_wait_limit_us, read at each launch.
constexpr uint32_t kDefaultWaitUs = 2000000;
constexpr uint32_t kMaxWaitUs = 60000000;
uint32_t wait_limit_us();

// Runs the grouped GEMM's bounded mbarrier wait on a barrier that expects
// `expected` arrivals and gets `arrivals` (<= 32).
cudaError_t launch_wait_selftest(uint32_t expected, uint32_t arrivals, cudaStream_t st);

// Segment of flat ids ranked by one warp in the permutation.
constexpr int kPermuteSegment = 1024;

cudaError_t launch_route_topk(const float* logits, const float* bias, int T, int E, int k, int score_fn,
                              int renormalize, int32_t* idx, float* w, cudaStream_t st);

// Batch-aware routing: active_set is a device scratch of ceil(E/32) words
// (zeroed by the launcher).
cudaError_t launch_route_batch_aware(const float* logits, const float* bias, int T, int E, int k, int k_primary,
                                     int score_fn, int renormalize, int32_t* idx, float* w, uint32_t* active_set,
                                     cudaStream_t st);

cudaError_t launch_quantize(const void* x, int64_t rows, int64_t cols, float* global_scale, bool compute_global,
                            bool blocked, uint8_t* packed, uint8_t* scales, unsigned* amax_ws, int num_sms,
                            cudaStream_t st);

cudaError_t launch_scales_to_blocked(const uint8_t* src, int64_t rows, int64_t cols, uint8_t* dst,
                                     int num_sms, cudaStream_t st);

// sf_groups: 4-byte scale groups per row (H/64 for NVFP4, H/128 for MXFP4).
cudaError_t launch_permute(const int32_t* topk_idx, int T, int E, int k, const uint8_t* xq, const uint8_t* xs,
                           int H, int sf_groups, int32_t* counts, int32_t* offsets, int32_t* row_offsets,
                           int32_t* perm_to_flat, int32_t* flat_to_perm, uint8_t* a_packed, uint8_t* a_scales,
                           int64_t rows_capacity, int32_t* ws_rank, int32_t* ws_seg_count, int32_t* ws_seg_base,
                           int num_sms, cudaStream_t st);

cudaError_t launch_quantize_mx(const void* x, int64_t rows, int64_t cols, bool blocked, uint8_t* packed,
                               uint8_t* scales, int num_sms, cudaStream_t st);

// Limits of the permutation that runs on library-owned scratch: routed rows
// (T*k) and per-segment expert counters (ceil(T*k/1024) * E).
constexpr int64_t kNoAllocMaxRoutedRows = 131072;
constexpr int64_t kNoAllocMaxSegmentExperts = 65536;

// Device address of the static scratch for the current device and CUDA
// context (looked up outside stream capture; during capture, the address the
// last uncaptured call on the same context found).  Returns an NVFP4MOE
// status, with the message set on failure.
int permute_scratch_address(cudaStream_t st, int32_t** base);
cudaError_t launch_permute_static_scratch(int32_t* base, const int32_t* topk_idx, int T, int E, int k,
                                          const uint8_t* xq, const uint8_t* xs, int H, int32_t* counts,
                                          int32_t* offsets, int32_t* row_offsets, int32_t* perm_to_flat,
                                          int32_t* flat_to_perm, uint8_t* a_packed, uint8_t* a_scales,
                                          int64_t rows_capacity, int num_sms, cudaStream_t st);

// Route + quantise + permute in one cooperative launch.  Workspace layout
// (bytes from the start, 256-byte aligned pieces): grid-barrier words and
// the batch-aware routing set (512 bytes), per-CTA partial amax, segment ranks [T*k], per-segment expert counts and
// bases [nseg*E] each.  Segments are 256 flat ids up to
// kPrepareShortMaxRows routed rows, 1024 above.
constexpr int64_t kPrepareShortMaxRows = 16384;
constexpr int kPrepareMaxGrid = 1024;

struct PrepareLayout {
  int64_t seg_len, nseg;
  int64_t bar_off, amax_off, rank_off, seg_count_off, seg_base_off, bytes;
};
PrepareLayout prepare_layout(int T, int E, int k);

cudaError_t launch_prepare(const float* logits, const float* bias, const void* x, int T, int E, int k, int k_primary,
                           int H, int score_fn, int renormalize, int32_t* idx, float* w, float* gscale, uint8_t* xq,
                           uint8_t* xs, int32_t* counts, int32_t* offsets, int32_t* row_offsets, int32_t* perm_to_flat,
                           int32_t* flat_to_perm, uint8_t* a_packed, uint8_t* a_scales, int64_t rows_capacity,
                           void* ws, bool mx, int num_sms, cudaStream_t st);

cudaError_t launch_finalize(const void* y, const int32_t* flat_to_perm, const float* w, int T, int k, int H,
                            int64_t rows_capacity, void* out, cudaStream_t st);
cudaError_t launch_finalize_f32(float* acc, int64_t n, void* out, int num_sms, cudaStream_t st);

// Reads and clears the sticky device flags of the kernels in kernels_prep.cu.
cudaError_t prep_read_and_clear_flags(unsigned* flags);

struct GemmArgs {
  const uint8_t* a_packed;
  const uint8_t* a_scales;
  const float* a_gscale;
  const int32_t* counts;
  const int32_t* row_offsets;
  int E;
  int64_t rows_capacity;
  int64_t m_total;
  const uint8_t* w_packed;
  const uint8_t* w_scales;
  const float* w_gscale;
  int N, K, epilogue;
  const float* c_gscale;
  void* c_out;
  uint8_t* c_scales;
  int tile_n;
  bool mx;  // MXFP4 operands (ue8m0 scale per 32 elements, no per-tensor scales)
  bool w_tiled;  // w_packed in the tiled layout (NVFP4MOE_W_TILED)
  void* sched;  // zero-filled 256-byte tile-scheduler workspace, or null for the static schedule
  int32_t min_rows, max_rows;  // experts outside [min_rows, max_rows) get no tiles
  // NVFP4MOE_EPI_FINALIZE_F32: c_out is float32 [T, N]; row r adds
  // topk_w[f] * bf16(acc) into row f / k, f = perm_to_flat[r]
  const int32_t* perm_to_flat;
  const float* topk_w;
  int k;
};

constexpr size_t kGemmWorkspaceBytes = 256;
// tile_n = 0 picks token-major tiles from this many routed rows per expert
// on average (m_total >= kTokenMajorMinRows * E).  Measured on GB300:
// token-major is 10 % faster on the skewed 2048-token batch (64 rows per
// expert on average, a few experts with hundreds) and 1 % slower at a
// uniform 32 rows per expert, where its 128-token tiles are mostly padding.
constexpr int64_t kTokenMajorMinRows = 64;
// ... and token-major tiles on CTA pairs from this many (m_total >=
// kPairMinRows * E): each pair tile is 256 token rows, so smaller experts
// would compute mostly padding.  Measured on GB300 at 2048 rows per expert:
// gate/up 2.66 vs 2.76 ms, down 1.46 vs 1.57 ms against single-SM tiles.
constexpr int64_t kPairMinRows = 512;

// Returns 0 on success or an NVFP4MOE_ERR_* code (message via set_error_detail).
int launch_grouped_gemm(const GemmArgs& a, int num_sms, int smem_optin, cudaStream_t st);

// One 128-row x 128-byte weight box of the tiled layout.
constexpr int64_t kWeightBoxBytes = 128 * 128;
cudaError_t launch_tile_weights(const uint8_t* w_packed, int64_t rows, int K, uint8_t* w_tiled, int num_sms,
                                cudaStream_t st);
cudaError_t gemm_read_and_clear_flags(unsigned* flags);

// Per-thread error message used by nvfp4moe_last_error_detail().
void set_error_detail(const char* fmt, ...);

}  // namespace nvfp4moe
