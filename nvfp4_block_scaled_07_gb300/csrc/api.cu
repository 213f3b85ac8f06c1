// C entry points of libnvfp4moe: argument validation, the per-device
// attribute cache and status plumbing.  The compute lives in
// kernels_prep.cu and grouped_gemm.cu; nothing here allocates device memory.
#include <atomic>
#include <cstdint>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/nvfp4moe.h"
#include "internal.h"

namespace nvfp4moe {

namespace {

thread_local char t_detail[512] = "";

struct DeviceInfo {
  bool checked = false;
  int status = NVFP4MOE_OK;
  int num_sms = 0;
  int smem_optin = 0;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_dev_mutex;

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_detail, sizeof(t_detail), fmt, ap);
  va_end(ap);
  return status;
}

int check_device(int dev, DeviceInfo* out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(NVFP4MOE_ERR_INVALID_ARG, "device %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_devices[dev];
  if (!d.checked) {
    cudaDeviceProp prop;
    cudaError_t err = cudaGetDeviceProperties(&prop, dev);
    if (err != cudaSuccess) return fail(NVFP4MOE_ERR_CUDA, "cudaGetDeviceProperties: %s", cudaGetErrorString(err));
    int optin = 0;
    err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (err != cudaSuccess) return fail(NVFP4MOE_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(err));
    d.num_sms = prop.multiProcessorCount;
    d.smem_optin = optin;
    d.status = (prop.major == 10 && prop.minor == 3) ? NVFP4MOE_OK : NVFP4MOE_ERR_UNSUPPORTED;
    d.checked = true;
    if (d.status != NVFP4MOE_OK)
      snprintf(t_detail, sizeof(t_detail), "device %d is compute capability %d.%d; libnvfp4moe is built for 10.3",
               dev, prop.major, prop.minor);
  }
  if (d.status != NVFP4MOE_OK) return fail(d.status, "device %d is not compute capability 10.3", dev);
  *out = d;
  return NVFP4MOE_OK;
}

int current_device(DeviceInfo* out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return fail(NVFP4MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
  return check_device(dev, out);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_status(cudaError_t err, const char* what) {
  if (err == cudaSuccess) return NVFP4MOE_OK;
  return fail(NVFP4MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(err));
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

void set_error_detail(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_detail, sizeof(t_detail), fmt, ap);
  va_end(ap);
}

}  // namespace nvfp4moe

namespace nvfp4moe {
namespace {
std::atomic<uint32_t> g_wait_limit_us{kDefaultWaitUs};
}  // namespace
uint32_t wait_limit_us() { return g_wait_limit_us.load(std::memory_order_relaxed); }
}  // namespace nvfp4moe

using namespace nvfp4moe;

#define NVFP4MOE_REQUIRE(cond, status, ...) \
  do {                                      \
    if (!(cond)) return fail(status, __VA_ARGS__); \
  } while (0)

extern "C" {

int nvfp4moe_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char* nvfp4moe_status_string(int status) {
  switch (status) {
    case NVFP4MOE_OK: return "ok";
    case NVFP4MOE_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4MOE_ERR_UNSUPPORTED: return "unsupported shape or device";
    case NVFP4MOE_ERR_SMEM: return "tile pipeline exceeds the opt-in shared memory";
    case NVFP4MOE_ERR_WORKSPACE: return "workspace too small";
    case NVFP4MOE_ERR_CUDA: return "CUDA runtime error";
    case NVFP4MOE_ERR_TIMEOUT: return "device pipeline wait timed out";
    case NVFP4MOE_ERR_DEVICE_DATA: return "device data out of range";
    default: return "unknown status";
  }
}

const char* nvfp4moe_last_error_detail(void) { return t_detail; }

int nvfp4moe_device_check(int device) {
  DeviceInfo d;
  t_detail[0] = 0;
  return check_device(device, &d);
}

int nvfp4moe_set_wait_limit_us(uint32_t us) {
  t_detail[0] = 0;
  NVFP4MOE_REQUIRE(us <= kMaxWaitUs, NVFP4MOE_ERR_INVALID_ARG, "wait limit %u us above the maximum %u us", us,
                   kMaxWaitUs);
  g_wait_limit_us.store(us == 0 ? kDefaultWaitUs : us, std::memory_order_relaxed);
  return NVFP4MOE_OK;
}

uint32_t nvfp4moe_wait_limit_us(void) { return wait_limit_us(); }

int nvfp4moe_wait_selftest(uint32_t expected_arrivals, uint32_t arrivals, cudaStream_t stream) {
  t_detail[0] = 0;
  NVFP4MOE_REQUIRE(expected_arrivals >= 1 && expected_arrivals <= 64 && arrivals <= 32, NVFP4MOE_ERR_INVALID_ARG,
                   "expected_arrivals %u (1..64), arrivals %u (0..32)", expected_arrivals, arrivals);
  DeviceInfo d;
  if (int st = current_device(&d)) return st;
  return cuda_status(launch_wait_selftest(expected_arrivals, arrivals, stream), "wait self-test launch");
}

int nvfp4moe_sync_status(cudaStream_t stream) {
  int st = cuda_status(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
  if (st) return st;
  unsigned f1 = 0, f2 = 0;
  st = cuda_status(prep_read_and_clear_flags(&f1), "reading device flags");
  if (st) return st;
  st = cuda_status(gemm_read_and_clear_flags(&f2), "reading device flags");
  if (st) return st;
  const unsigned f = f1 | f2;
  if (f & kFlagTimeout) return fail(NVFP4MOE_ERR_TIMEOUT, "a device wait (grouped GEMM pipeline or prepare grid barrier) exceeded its time limit");
  if (f & kFlagBadData) return fail(NVFP4MOE_ERR_DEVICE_DATA, "an expert id or row index was out of range");
  return NVFP4MOE_OK;
}

size_t nvfp4moe_blocked_scales_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols <= 0 || cols % 64) return 0;
  return size_t(ceil_div(rows, 128) * 128 * (cols / 16));
}

size_t nvfp4moe_mxfp4_blocked_scales_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols <= 0 || cols % 128) return 0;
  return size_t(ceil_div(rows, 128) * 128 * (cols / 32));
}

size_t nvfp4moe_tiled_weights_bytes(int64_t rows, int K) {
  if (rows <= 0 || rows % 128 || K <= 0 || K % 64) return 0;
  return size_t((rows / 128) * ceil_div(int64_t(K), 256) * kWeightBoxBytes);
}

int nvfp4moe_tile_weights(const uint8_t* w_packed, int64_t rows, int K, uint8_t* w_tiled, cudaStream_t stream) {
  t_detail[0] = 0;
  NVFP4MOE_REQUIRE(rows > 0 && rows % 128 == 0 && K > 0 && K % 64 == 0, NVFP4MOE_ERR_UNSUPPORTED,
                   "rows = %lld must be a positive multiple of 128 and K = %d of 64", (long long)rows, K);
  NVFP4MOE_REQUIRE(w_packed && w_tiled && aligned16(w_packed) && aligned16(w_tiled), NVFP4MOE_ERR_INVALID_ARG,
                   "null or misaligned pointer");
  DeviceInfo d;
  if (int st = current_device(&d)) return st;
  return cuda_status(launch_tile_weights(w_packed, rows, K, w_tiled, d.num_sms, stream), "tile weights launch");
}

// ---- a1 ---------------------------------------------------------------------
int moe_route_topk(const float* logits, const float* bias, int T, int E, int k, int score_fn, int renormalize,
                   int32_t* topk_idx, float* topk_w, cudaStream_t stream) {
  t_detail[0] = 0;
  NVFP4MOE_REQUIRE(T >= 0, NVFP4MOE_ERR_INVALID_ARG, "T = %d must be >= 0", T);
  NVFP4MOE_REQUIRE(E >= 1 && E <= 1024, NVFP4MOE_ERR_UNSUPPORTED, "E = %d outside [1, 1024]", E);
  NVFP4MOE_REQUIRE(k >= 1 && k <= E && k <= 32, NVFP4MOE_ERR_UNSUPPORTED, "k = %d outside [1, min(E, 32)]", k);
  NVFP4MOE_REQUIRE(score_fn == NVFP4MOE_SCORE_SOFTMAX || score_fn == NVFP4MOE_SCORE_SIGMOID,
                   NVFP4MOE_ERR_INVALID_ARG, "score_fn %d", score_fn);
  if (T == 0) return NVFP4MOE_OK;
  NVFP4MOE_REQUIRE(logits && topk_idx && topk_w, NVFP4MOE_ERR_INVALID_ARG, "null pointer");
  DeviceInfo d;
  if (int st = current_device(&d)) return st;
  return cuda_status(launch_route_topk(logits, bias, T, E, k, score_fn, renormalize ? 1 : 0, topk_idx, topk_w, stream),
                     "route launch");
}

size_t moe_route_batch_aware_workspace_size(int E) {
  if (E < 1) return 0;
  return size_t(ceil_div(E, 32)) * sizeof(uint32_t);
}

int moe_route_batch_aware(const float* logits, const float* bias, int T, int E, int k, int k_primary, int score_fn,
                          int renormalize, int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes,
                          cudaStream_t stream) {
  t_detail[0] = 0;
  NVFP4MOE_REQUIRE(T >= 0, NVFP4MOE_ERR_INVALID_ARG, "T = %d must be >= 0", T);
  NVFP4MOE_REQUIRE(E >= 1 && E <= 1024, NVFP4MOE_ERR_UNSUPPORTED, "E = %d outside [1, 1024]", E);
  NVFP4MOE_REQUIRE(k >= 1 && k <= E && k <= 32, NVFP4MOE_ERR_UNSUPPORTED, "k = %d outside [1, min(E, 32)]", k);
  NVFP4MOE_REQUIRE(k_primary >= 1 && k_primary <= k, NVFP4MOE_ERR_INVALID_ARG, "k_primary = %d outside [1, k = %d]",
                   k_primary, k);
  NVFP4MOE_REQUIRE(score_fn == NVFP4MOE_SCORE_SOFTMAX || score_fn == NVFP4MOE_SCORE_SIGMOID,
                   NVFP4MOE_ERR_INVALID_ARG, "score_fn %d", score_fn);
  if (T == 0) return NVFP4MOE_OK;
  NVFP4MOE_REQUIRE(logits && topk_idx && topk_w, NVFP4MOE_ERR_INVALID_ARG, "null pointer");
  const size_t need = moe_route_batch_aware_workspace_size(E);
  NVFP4MOE_REQUIRE(ws && ws_bytes >= need && (reinterpret_cast<uintptr_t>(ws) & 3) == 0, NVFP4MOE_ERR_WORKSPACE,
                   "workspace %zu < %zu or misaligned", ws_bytes, need);
  DeviceInfo d;
  if (int st = current_device(&d)) return st;
  return cuda_status(launch_route_batch_aware(logits, bias, T, E, k, k_primary, score_fn, renormalize ? 1 : 0,
                                              topk_idx, topk_w, static_cast<uint32_t*>(ws), stream),
                     "batch-aware route launch");
}

// ---- a2 ---------------------------------------------------------------------
size_t moe_quantize_nvfp4_workspace_size(int64_t rows, int64_t cols, int flags) {
  (void)rows;
  (void)cols;
  return (flags & NVFP4MOE_QUANT_COMPUTE_GLOBAL) ? 16 : 0;
}

int moe_quantize_nvfp4(const void* x_bf16, int64_t rows, int64_t cols, float* global_scale, int flags,
                       uint8_t* packed, uint8_t* scales, void* ws, size_t ws_bytes, cudaStream_t stream) {
  t_detail[0] = 0;
  NVFP4MOE_REQUIRE(rows >= 0 && cols > 0, NVFP4MOE_ERR_INVALID_ARG, "rows %lld cols %lld", (long long)rows,
                   (long long)cols);
  NVFP4MOE_REQUIRE((flags & ~3) == 0, NVFP4MOE_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  const bool blocked = flags & NVFP4MOE_QUANT_SCALES_BLOCKED;
  const bool compute = flags & NVFP4MOE_QUANT_COMPUTE_GLOBAL;
  NVFP4MOE_REQUIRE(cols % 16 == 0, NVFP4MOE_ERR_UNSUPPORTED, "cols %lld is not a multiple of 16", (long long)cols);
  NVFP4MOE_REQUIRE(!blocked || cols % 64 == 0, NVFP4MOE_ERR_UNSUPPORTED,
                   "blocked scales need cols %% 64 == 0 (cols %lld)", (long long)cols);
  if (rows == 0) return NVFP4MOE_OK;
  NVFP4MOE_REQUIRE(x_bf16 && global_scale && packed && scales, NVFP4MOE_ERR_INVALID_ARG, "null pointer");
  NVFP4MOE_REQUIRE(aligned16(x_bf16) && aligned16(packed), NVFP4MOE_ERR_INVALID_ARG,
                   "x and packed must be 16-byte aligned");
  const size_t need = moe_quantize_nvfp4_workspace_size(rows, cols, flags);
  NVFP4MOE_REQUIRE(ws_bytes >= need && (need == 0 || ws), NVFP4MOE_ERR_WORKSPACE, "workspace %zu < %zu", ws_bytes,
                   need);
  DeviceInfo d;
  if (int st = current_device(&d)) return st;
  return cuda_status(launch_quantize(x_bf16, rows, cols, global_scale, compute, blocked, packed, scales,
                                     static_cast<unsigned*>(ws), d.num_sms, stream),
                     "quantize launch");
}

int moe_quantize_mxfp4(const void* x_bf16, int64_t rows, int64_t cols, int flags, uint8_t* packed, uint8_t* scales,
                       cudaStream_t stream) {
  t_detail[0] = 0;
  NVFP4MOE_REQUIRE(rows >= 0 && cols > 0, NVFP4MOE_ERR_INVALID_ARG, "rows %lld cols %lld", (long long)rows,
                   (long long)cols);
  NVFP4MOE_REQUIRE((flags & ~NVFP4MOE_QUANT_SCALES_BLOCKED) == 0, NVFP4MOE_ERR_INVALID_ARG, "unknown flags 0x%x",
                   flags);
  const bool blocked = flags & NVFP4MOE_QUANT_SCALES_BLOCKED;
  NVFP4MOE_REQUIRE(cols % 32 == 0, NVFP4MOE_ERR_UNSUPPORTED, "cols %lld is not a multiple of 32", (long long)cols);
  NVFP4MOE_REQUIRE(!blocked || cols % 128 == 0, NVFP4MOE_ERR_UNSUPPORTED,
                   "blocked scales need cols %% 128 == 0 (cols %lld)", (long long)cols);
  if (rows == 0) return NVFP4MOE_OK;
  NVFP4MOE_REQUIRE(x_bf16 && packed && scales, NVFP4MOE_ERR_INVALID_ARG, "null pointer");
  NVFP4MOE_REQUIRE(aligned16(x_bf16) && aligned16(packed), NVFP4MOE_ERR_INVALID_ARG,
                   "x and packed must be 16-byte aligned");
  DeviceInfo d;
  if (int st = current_device(&d)) return st;
  return cuda_status(launch_quantize_mx(x_bf16, rows, cols, blocked, packed, scales, d.num_sms, stream),
                     "MXFP4 quantize launch");
}

int moe_scales_to_blocked(const uint8_t* scales_row_major, int64_t rows, int64_t cols, uint8_t* scales_blocked,
                          cudaStream_t stream) {
  t_detail[0] = 0;
  NVFP4MOE_REQUIRE(rows >= 0 && cols > 0, NVFP4MOE_ERR_INVALID_ARG, "bad shape");
  NVFP4MOE_REQUIRE(cols % 64 == 0, NVFP4MOE_ERR_UNSUPPORTED, "cols must be a multiple of 64");
  if (rows == 0) return NVFP4MOE_OK;
  NVFP4MOE_REQUIRE(scales_row_major && scales_blocked, NVFP4MOE_ERR_INVALID_ARG, "null pointer");
  NVFP4MOE_REQUIRE((reinterpret_cast<uintptr_t>(scales_row_major) & 3) == 0 && aligned16(scales_blocked),
                   NVFP4MOE_ERR_INVALID_ARG, "misaligned pointer");
  DeviceInfo d;
  if (int st = current_device(&d)) return st;
  return cuda_status(launch_scales_to_blocked(scales_row_major, rows, cols, scales_blocked, d.num_sms, stream),
                     "scale re-layout launch");
}

// ---- a3 ---------------------------------------------------------------------
int64_t moe_permute_rows_capacity(int T, int E, int k) {
  if (T < 0 || E < 1 || k < 1) return 0;
  return ceil_div(int64_t(T) * k + int64_t(E) * 127, 128) * 128;
}

size_t moe_permute_workspace_size(int T, int E, int k) {
  if (T < 0 || E < 1 || k < 1) return 0;
  const int64_t R = int64_t(T) * k;
  const int64_t nseg = ceil_div(R, kPermuteSegment);
  const size_t rank = size_t(ceil_div(R, 64) * 64) * 4;
  const size_t seg = size_t(ceil_div(nseg * E, 64) * 64) * 4;
  return rank + 2 * seg + 256;
}

static int permute_common(const int32_t* topk_idx, int T, int E, int k, const uint8_t* xq, const uint8_t* xs, int H, int scale_block,
                int32_t* expert_counts, int32_t* expert_offsets, int32_t* row_offsets, int32_t* perm_to_flat,
                int32_t* flat_to_perm, uint8_t* a_packed, uint8_t* a_scales, void* ws, size_t ws_bytes,
                cudaStream_t stream) {
  t_detail[0] = 0;
  NVFP4MOE_REQUIRE(T >= 0, NVFP4MOE_ERR_INVALID_ARG, "T = %d", T);
  NVFP4MOE_REQUIRE(E >= 1 && E <= 1024, NVFP4MOE_ERR_UNSUPPORTED, "E = %d outside [1, 1024]", E);
  NVFP4MOE_REQUIRE(k >= 1 && k <= E, NVFP4MOE_ERR_UNSUPPORTED, "k = %d outside [1, E]", k);
  NVFP4MOE_REQUIRE(H > 0 && H % (4 * scale_block) == 0, NVFP4MOE_ERR_UNSUPPORTED,
                   "H = %d must be a positive multiple of %d", H, 4 * scale_block);
  NVFP4MOE_REQUIRE(int64_t(T) * k <= (int64_t(1) << 30), NVFP4MOE_ERR_UNSUPPORTED, "T*k too large");
  NVFP4MOE_REQUIRE(expert_counts && expert_offsets && row_offsets && perm_to_flat, NVFP4MOE_ERR_INVALID_ARG,
                   "null pointer");
  NVFP4MOE_REQUIRE(T == 0 || (topk_idx && xq && xs && flat_to_perm && a_packed && a_scales),
                   NVFP4MOE_ERR_INVALID_ARG, "null pointer");
  NVFP4MOE_REQUIRE(T == 0 || (aligned16(xq) && aligned16(a_packed) && aligned16(a_scales) &&
                              (reinterpret_cast<uintptr_t>(xs) & 3) == 0),
                   NVFP4MOE_ERR_INVALID_ARG, "misaligned pointer");
  const size_t need = moe_permute_workspace_size(T, E, k);
  NVFP4MOE_REQUIRE(ws && ws_bytes >= need, NVFP4MOE_ERR_WORKSPACE, "workspace %zu < %zu", ws_bytes, need);
  DeviceInfo d;
  if (int st = current_device(&d)) return st;
  const int64_t R = int64_t(T) * k;
  const int64_t nseg = ceil_div(R, kPermuteSegment);
  int32_t* rank = static_cast<int32_t*>(ws);
  int32_t* seg_count = rank + ceil_div(R, 64) * 64;
  int32_t* seg_base = seg_count + ceil_div(nseg * E, 64) * 64;
  return cuda_status(launch_permute(topk_idx, T, E, k, xq, xs, H, H / (4 * scale_block), expert_counts, expert_offsets, row_offsets,
                                    perm_to_flat, flat_to_perm, a_packed, a_scales,
                                    moe_permute_rows_capacity(T, E, k), rank, seg_count, seg_base, d.num_sms,
                                    stream),
                     "permute launch");
}

int moe_permute(const int32_t* topk_idx, int T, int E, int k, const uint8_t* xq, const uint8_t* xs, int H,
                int32_t* expert_counts, int32_t* expert_offsets, int32_t* row_offsets, int32_t* perm_to_flat,
                int32_t* flat_to_perm, uint8_t* a_packed, uint8_t* a_scales, void* ws, size_t ws_bytes,
                cudaStream_t stream) {
  return permute_common(topk_idx, T, E, k, xq, xs, H, 16, expert_counts, expert_offsets, row_offsets, perm_to_flat,
                        flat_to_perm, a_packed, a_scales, ws, ws_bytes, stream);
}

int moe_permute_mxfp4(const int32_t* topk_idx, int T, int E, int k, const uint8_t* xq, const uint8_t* xs, int H,
                      int32_t* expert_counts, int32_t* expert_offsets, int32_t* row_offsets, int32_t* perm_to_flat,
                      int32_t* flat_to_perm, uint8_t* a_packed, uint8_t* a_scales, void* ws, size_t ws_bytes,
                      cudaStream_t stream) {
  return permute_common(topk_idx, T, E, k, xq, xs, H, 32, expert_counts, expert_offsets, row_offsets, perm_to_flat,
                        flat_to_perm, a_packed, a_scales, ws, ws_bytes, stream);
}

int moe_permute_no_alloc(const int32_t* topk_idx, int T, int E, int k, const uint8_t* xq, const uint8_t* xs, int H,
                         int32_t* expert_counts, int32_t* expert_offsets, int32_t* row_offsets,
                         int32_t* perm_to_flat, int32_t* flat_to_perm, uint8_t* a_packed, uint8_t* a_scales,
                         cudaStream_t stream) {
  t_detail[0] = 0;
  NVFP4MOE_REQUIRE(T >= 0, NVFP4MOE_ERR_INVALID_ARG, "T = %d", T);
  NVFP4MOE_REQUIRE(E >= 1 && E <= 1024, NVFP4MOE_ERR_UNSUPPORTED, "E = %d outside [1, 1024]", E);
  NVFP4MOE_REQUIRE(k >= 1 && k <= E, NVFP4MOE_ERR_UNSUPPORTED, "k = %d outside [1, E]", k);
  NVFP4MOE_REQUIRE(H > 0 && H % 64 == 0, NVFP4MOE_ERR_UNSUPPORTED, "H = %d must be a positive multiple of 64", H);
  const int64_t R = int64_t(T) * k;
  const int64_t seg_experts = ceil_div(R, kPermuteSegment) * E;
  NVFP4MOE_REQUIRE(R <= kNoAllocMaxRoutedRows && seg_experts <= kNoAllocMaxSegmentExperts, NVFP4MOE_ERR_UNSUPPORTED,
                   "T*k = %lld routed rows and %lld segment-expert counters exceed the library's static scratch "
                   "(at most %lld routed rows and %lld counters); use moe_permute with a workspace",
                   (long long)R, (long long)seg_experts, (long long)kNoAllocMaxRoutedRows,
                   (long long)kNoAllocMaxSegmentExperts);
  NVFP4MOE_REQUIRE(expert_counts && expert_offsets && row_offsets && perm_to_flat, NVFP4MOE_ERR_INVALID_ARG,
                   "null pointer");
  NVFP4MOE_REQUIRE(T == 0 || (topk_idx && xq && xs && flat_to_perm && a_packed && a_scales),
                   NVFP4MOE_ERR_INVALID_ARG, "null pointer");
  NVFP4MOE_REQUIRE(T == 0 || (aligned16(xq) && aligned16(a_packed) && aligned16(a_scales) &&
                              (reinterpret_cast<uintptr_t>(xs) & 3) == 0),
                   NVFP4MOE_ERR_INVALID_ARG, "misaligned pointer");
  DeviceInfo d;
  if (int st = current_device(&d)) return st;
  int32_t* scratch = nullptr;
  if (int st = permute_scratch_address(stream, &scratch)) return st;
  return cuda_status(launch_permute_static_scratch(scratch, topk_idx, T, E, k, xq, xs, H, expert_counts,
                                                   expert_offsets, row_offsets, perm_to_flat, flat_to_perm, a_packed,
                                                   a_scales, moe_permute_rows_capacity(T, E, k), d.num_sms, stream),
                     "permute (static scratch) launch");
}

// ---- a1 + a2 + a3 -----------------------------------------------------------
size_t moe_prepare_workspace_size(int T, int E, int k) {
  if (T < 0 || E < 1 || k < 1) return 0;
  return size_t(prepare_layout(T, E, k).bytes);
}

static int prepare_common(bool mx, const float* logits, const float* bias, const void* x_bf16, int T, int E, int k,
                          int k_primary, int H, int score_fn, int renormalize, int32_t* topk_idx, float* topk_w,
                          float* x_gscale, uint8_t* xq, uint8_t* xs, int32_t* expert_counts, int32_t* expert_offsets,
                          int32_t* row_offsets, int32_t* perm_to_flat, int32_t* flat_to_perm, uint8_t* a_packed,
                          uint8_t* a_scales, void* ws, size_t ws_bytes, cudaStream_t stream) {
  t_detail[0] = 0;
  NVFP4MOE_REQUIRE(T >= 0, NVFP4MOE_ERR_INVALID_ARG, "T = %d must be >= 0", T);
  NVFP4MOE_REQUIRE(E >= 1 && E <= 1024, NVFP4MOE_ERR_UNSUPPORTED, "E = %d outside [1, 1024]", E);
  NVFP4MOE_REQUIRE(k >= 1 && k <= E && k <= 32, NVFP4MOE_ERR_UNSUPPORTED, "k = %d outside [1, min(E, 32)]", k);
  NVFP4MOE_REQUIRE(k_primary >= 1 && k_primary <= k, NVFP4MOE_ERR_INVALID_ARG, "k_primary = %d outside [1, k = %d]",
                   k_primary, k);
  const int hq = mx ? 128 : 64;
  NVFP4MOE_REQUIRE(H > 0 && H % hq == 0, NVFP4MOE_ERR_UNSUPPORTED, "H = %d must be a positive multiple of %d", H, hq);
  NVFP4MOE_REQUIRE(int64_t(T) * k <= (int64_t(1) << 30), NVFP4MOE_ERR_UNSUPPORTED, "T*k too large");
  NVFP4MOE_REQUIRE(score_fn == NVFP4MOE_SCORE_SOFTMAX || score_fn == NVFP4MOE_SCORE_SIGMOID,
                   NVFP4MOE_ERR_INVALID_ARG, "score_fn %d", score_fn);
  NVFP4MOE_REQUIRE((mx || x_gscale) && expert_counts && expert_offsets && row_offsets && perm_to_flat,
                   NVFP4MOE_ERR_INVALID_ARG, "null pointer");
  NVFP4MOE_REQUIRE(T == 0 || (logits && x_bf16 && topk_idx && topk_w && xq && xs && flat_to_perm && a_packed &&
                              a_scales),
                   NVFP4MOE_ERR_INVALID_ARG, "null pointer");
  NVFP4MOE_REQUIRE(T == 0 || (aligned16(x_bf16) && aligned16(xq) && aligned16(a_packed) && aligned16(a_scales) &&
                              (reinterpret_cast<uintptr_t>(xs) & 3) == 0),
                   NVFP4MOE_ERR_INVALID_ARG, "misaligned pointer");
  const size_t need = moe_prepare_workspace_size(T, E, k);
  NVFP4MOE_REQUIRE(ws && ws_bytes >= need, NVFP4MOE_ERR_WORKSPACE, "workspace %zu < %zu", ws_bytes, need);
  NVFP4MOE_REQUIRE((reinterpret_cast<uintptr_t>(ws) & 255) == 0, NVFP4MOE_ERR_INVALID_ARG,
                   "workspace must be 256-byte aligned");
  DeviceInfo d;
  if (int st = current_device(&d)) return st;
  return cuda_status(launch_prepare(logits, bias, x_bf16, T, E, k, k_primary, H, score_fn, renormalize ? 1 : 0,
                                    topk_idx, topk_w, x_gscale, xq, xs, expert_counts, expert_offsets, row_offsets,
                                    perm_to_flat, flat_to_perm, a_packed, a_scales,
                                    moe_permute_rows_capacity(T, E, k), ws, mx, d.num_sms, stream),
                     "prepare launch");
}

int moe_prepare(const float* logits, const float* bias, const void* x_bf16, int T, int E, int k, int k_primary,
                int H, int score_fn, int renormalize, int32_t* topk_idx, float* topk_w, float* x_gscale, uint8_t* xq,
                uint8_t* xs, int32_t* expert_counts, int32_t* expert_offsets, int32_t* row_offsets,
                int32_t* perm_to_flat, int32_t* flat_to_perm, uint8_t* a_packed, uint8_t* a_scales, void* ws,
                size_t ws_bytes, cudaStream_t stream) {
  return prepare_common(false, logits, bias, x_bf16, T, E, k, k_primary, H, score_fn, renormalize, topk_idx, topk_w,
                        x_gscale, xq, xs, expert_counts, expert_offsets, row_offsets, perm_to_flat, flat_to_perm,
                        a_packed, a_scales, ws, ws_bytes, stream);
}

int moe_prepare_mxfp4(const float* logits, const float* bias, const void* x_bf16, int T, int E, int k,
                      int k_primary, int H, int score_fn, int renormalize, int32_t* topk_idx, float* topk_w,
                      uint8_t* xq, uint8_t* xs, int32_t* expert_counts, int32_t* expert_offsets,
                      int32_t* row_offsets, int32_t* perm_to_flat, int32_t* flat_to_perm, uint8_t* a_packed,
                      uint8_t* a_scales, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return prepare_common(true, logits, bias, x_bf16, T, E, k, k_primary, H, score_fn, renormalize, topk_idx, topk_w,
                        nullptr, xq, xs, expert_counts, expert_offsets, row_offsets, perm_to_flat, flat_to_perm,
                        a_packed, a_scales, ws, ws_bytes, stream);
}

// ---- a4/a5 ------------------------------------------------------------------
size_t moe_grouped_gemm_nvfp4_workspace_size(int E, int N, int K, int epilogue) {
  (void)E;
  (void)N;
  (void)K;
  (void)epilogue;
  return kGemmWorkspaceBytes;
}

int nvfp4moe_gemm_tile_choice(int E, int N, int64_t m_total, int tile_n) {
  // tile_n = 0: token-major tiles once experts average kTokenMajorMinRows
  // rows, on CTA pairs from kPairMinRows
  if (tile_n != 0 || N % 256 != 0 || E < 1) return tile_n;
  if (m_total >= kPairMinRows * E) return NVFP4MOE_TILE_TOKEN_MAJOR_PAIR;
  if (m_total >= kTokenMajorMinRows * E) return NVFP4MOE_TILE_TOKEN_MAJOR;
  return 0;
}

static int grouped_gemm_common(bool mx, const uint8_t* a_packed, const uint8_t* a_scales, const float* a_gscale,
                               const int32_t* expert_counts, const int32_t* row_offsets, int E, int64_t rows_capacity,
                               int64_t m_total, const uint8_t* w_packed, const uint8_t* w_scales,
                               const float* w_gscale, int N, int K, int epilogue, const float* c_gscale, void* c_out,
                               uint8_t* c_scales, int tile_n, int w_layout, int32_t min_rows,
                               int32_t max_rows, void* ws, size_t ws_bytes, cudaStream_t stream,
                               const int32_t* perm_to_flat = nullptr, const float* topk_w = nullptr, int T = 0,
                               int k = 0) {
  t_detail[0] = 0;
  NVFP4MOE_REQUIRE(min_rows >= 1 && min_rows <= max_rows, NVFP4MOE_ERR_INVALID_ARG,
                   "expert row range [%d, %d) must have 1 <= min_rows <= max_rows", min_rows, max_rows);
  NVFP4MOE_REQUIRE(w_layout == NVFP4MOE_W_ROWMAJOR || w_layout == NVFP4MOE_W_TILED, NVFP4MOE_ERR_INVALID_ARG,
                   "w_layout %d", w_layout);
  NVFP4MOE_REQUIRE(!ws || (ws_bytes >= kGemmWorkspaceBytes && (reinterpret_cast<uintptr_t>(ws) & 255) == 0),
                   NVFP4MOE_ERR_WORKSPACE, "workspace must be NULL or %zu bytes, 256-byte aligned (got %zu)",
                   kGemmWorkspaceBytes, ws_bytes);
  const int requant = mx ? NVFP4MOE_EPI_SWIGLU_MXFP4 : NVFP4MOE_EPI_SWIGLU_NVFP4;
  const bool fin = epilogue == NVFP4MOE_EPI_FINALIZE_F32;
  NVFP4MOE_REQUIRE(epilogue == NVFP4MOE_EPI_BF16 || epilogue == requant || epilogue == NVFP4MOE_EPI_SWIGLU_F32 ||
                       (fin && !mx && perm_to_flat),
                   NVFP4MOE_ERR_INVALID_ARG, "epilogue %d", epilogue);
  NVFP4MOE_REQUIRE(!fin || (topk_w && T >= 0 && k >= 1 && int64_t(T) * k <= rows_capacity), NVFP4MOE_ERR_INVALID_ARG,
                   "fused finalize needs perm_to_flat, topk_w, T >= 0 and 1 <= k with T*k <= rows_capacity");
  NVFP4MOE_REQUIRE(E >= 1 && E <= 1024, NVFP4MOE_ERR_UNSUPPORTED, "E = %d outside [1, 1024]", E);
  const int kq = mx ? 128 : 64;
  NVFP4MOE_REQUIRE(K >= kq && K % kq == 0, NVFP4MOE_ERR_UNSUPPORTED, "K = %d must be a positive multiple of %d", K,
                   kq);
  const bool swiglu = epilogue != NVFP4MOE_EPI_BF16 && !fin;
  NVFP4MOE_REQUIRE(N > 0 && N % (swiglu ? 256 : 128) == 0, NVFP4MOE_ERR_UNSUPPORTED,
                   "N = %d must be a multiple of %d for this epilogue", N, swiglu ? 256 : 128);
  NVFP4MOE_REQUIRE(int64_t(E) * N < (int64_t(1) << 31), NVFP4MOE_ERR_UNSUPPORTED, "E*N too large");
  NVFP4MOE_REQUIRE(rows_capacity >= 128 && rows_capacity % 128 == 0 && rows_capacity < (int64_t(1) << 31),
                   NVFP4MOE_ERR_INVALID_ARG, "rows_capacity %lld must be a positive multiple of 128",
                   (long long)rows_capacity);
  NVFP4MOE_REQUIRE(m_total >= 0, NVFP4MOE_ERR_INVALID_ARG, "m_total < 0");
  NVFP4MOE_REQUIRE(tile_n == 0 || tile_n == 128 || (!swiglu && tile_n == 256) ||
                       ((tile_n == NVFP4MOE_TILE_TOKEN_MAJOR || tile_n == NVFP4MOE_TILE_TOKEN_MAJOR_PAIR) &&
                        N % 256 == 0),
                   NVFP4MOE_ERR_UNSUPPORTED,
                   "tile_n %d (expected 0, 128, 256 for the bf16 epilogue, or NVFP4MOE_TILE_TOKEN_MAJOR[_PAIR] with "
                   "N %% 256 == 0)",
                   tile_n);
  NVFP4MOE_REQUIRE(a_packed && a_scales && expert_counts && row_offsets && w_packed && w_scales && c_out,
                   NVFP4MOE_ERR_INVALID_ARG, "null pointer");
  NVFP4MOE_REQUIRE(mx || (a_gscale && w_gscale), NVFP4MOE_ERR_INVALID_ARG, "null per-tensor scale pointer");
  NVFP4MOE_REQUIRE(epilogue != NVFP4MOE_EPI_SWIGLU_NVFP4 || (c_gscale && c_scales), NVFP4MOE_ERR_INVALID_ARG,
                   "SWIGLU_NVFP4 needs c_gscale and c_scales");
  NVFP4MOE_REQUIRE(epilogue != NVFP4MOE_EPI_SWIGLU_MXFP4 || c_scales, NVFP4MOE_ERR_INVALID_ARG,
                   "SWIGLU_MXFP4 needs c_scales");
  NVFP4MOE_REQUIRE(aligned16(a_packed) && aligned16(a_scales) && aligned16(w_packed) && aligned16(w_scales) &&
                       aligned16(c_out),
                   NVFP4MOE_ERR_INVALID_ARG, "operands must be 16-byte aligned");
  DeviceInfo d;
  if (int st = current_device(&d)) return st;
  GemmArgs a;
  a.a_packed = a_packed;
  a.a_scales = a_scales;
  a.a_gscale = a_gscale;
  a.counts = expert_counts;
  a.row_offsets = row_offsets;
  a.E = E;
  a.rows_capacity = rows_capacity;
  a.m_total = m_total;
  a.w_packed = w_packed;
  a.w_scales = w_scales;
  a.w_gscale = w_gscale;
  a.N = N;
  a.K = K;
  a.epilogue = epilogue;
  a.c_gscale = c_gscale;
  a.c_out = c_out;
  a.c_scales = c_scales;
  a.tile_n = nvfp4moe_gemm_tile_choice(E, N, m_total, tile_n);
  a.mx = mx;
  a.w_tiled = w_layout == NVFP4MOE_W_TILED;
  a.sched = ws;
  a.min_rows = min_rows;
  a.max_rows = max_rows;
  a.perm_to_flat = perm_to_flat;
  a.topk_w = topk_w;
  a.k = k;
  return launch_grouped_gemm(a, d.num_sms, d.smem_optin, stream);  // detail already set on failure
}

int moe_grouped_gemm_nvfp4(const uint8_t* a_packed, const uint8_t* a_scales, const float* a_gscale,
                           const int32_t* expert_counts, const int32_t* row_offsets, int E, int64_t rows_capacity,
                           int64_t m_total, const uint8_t* w_packed, const uint8_t* w_scales,
                           const float* w_gscale, int N, int K, int epilogue, const float* c_gscale, void* c_out,
                           uint8_t* c_scales, int tile_n, int w_layout, void* ws, size_t ws_bytes,
                           cudaStream_t stream) {
  return grouped_gemm_common(false, a_packed, a_scales, a_gscale, expert_counts, row_offsets, E, rows_capacity,
                             m_total, w_packed, w_scales, w_gscale, N, K, epilogue, c_gscale, c_out, c_scales, tile_n,
                             w_layout, 1, INT32_MAX, ws, ws_bytes, stream);
}

int moe_grouped_gemm_nvfp4_range(const uint8_t* a_packed, const uint8_t* a_scales, const float* a_gscale,
                                 const int32_t* expert_counts, const int32_t* row_offsets, int E,
                                 int64_t rows_capacity, int64_t m_total, const uint8_t* w_packed,
                                 const uint8_t* w_scales, const float* w_gscale, int N, int K, int epilogue,
                                 const float* c_gscale, void* c_out, uint8_t* c_scales, int tile_n, int w_layout,
                                 int32_t min_rows, int32_t max_rows, void* ws, size_t ws_bytes,
                                 cudaStream_t stream) {
  return grouped_gemm_common(false, a_packed, a_scales, a_gscale, expert_counts, row_offsets, E, rows_capacity,
                             m_total, w_packed, w_scales, w_gscale, N, K, epilogue, c_gscale, c_out, c_scales, tile_n,
                             w_layout, min_rows, max_rows, ws, ws_bytes, stream);
}

int moe_grouped_gemm_mxfp4(const uint8_t* a_packed, const uint8_t* a_scales, const int32_t* expert_counts,
                           const int32_t* row_offsets, int E, int64_t rows_capacity, int64_t m_total,
                           const uint8_t* w_packed, const uint8_t* w_scales, int N, int K, int epilogue, void* c_out,
                           uint8_t* c_scales, int tile_n, int w_layout, void* ws, size_t ws_bytes,
                           cudaStream_t stream) {
  return grouped_gemm_common(true, a_packed, a_scales, nullptr, expert_counts, row_offsets, E, rows_capacity, m_total,
                             w_packed, w_scales, nullptr, N, K, epilogue, nullptr, c_out, c_scales, tile_n, w_layout,
                             1, INT32_MAX, ws, ws_bytes, stream);
}

int moe_grouped_gemm_nvfp4_finalize(const uint8_t* a_packed, const uint8_t* a_scales, const float* a_gscale,
                                    const int32_t* expert_counts, const int32_t* row_offsets, int E,
                                    int64_t rows_capacity, int64_t m_total, const uint8_t* w_packed,
                                    const uint8_t* w_scales, const float* w_gscale, int N, int K,
                                    const int32_t* perm_to_flat, const float* topk_w, int T, int k, float* out_f32,
                                    int tile_n, int w_layout, int32_t min_rows, int32_t max_rows, void* ws,
                                    size_t ws_bytes, cudaStream_t stream) {
  return grouped_gemm_common(false, a_packed, a_scales, a_gscale, expert_counts, row_offsets, E, rows_capacity,
                             m_total, w_packed, w_scales, w_gscale, N, K, NVFP4MOE_EPI_FINALIZE_F32, nullptr, out_f32,
                             nullptr, tile_n, w_layout, min_rows, max_rows, ws, ws_bytes, stream, perm_to_flat, topk_w,
                             T, k);
}

int moe_finalize_f32(float* acc_f32, int T, int H, void* out_bf16, cudaStream_t stream) {
  t_detail[0] = 0;
  NVFP4MOE_REQUIRE(T >= 0 && H > 0 && H % 8 == 0, NVFP4MOE_ERR_INVALID_ARG, "T %d H %d (H %% 8 == 0)", T, H);
  NVFP4MOE_REQUIRE(T == 0 || (acc_f32 && out_bf16 && aligned16(acc_f32) && aligned16(out_bf16)),
                   NVFP4MOE_ERR_INVALID_ARG, "null or misaligned pointer");
  DeviceInfo d;
  if (int st = current_device(&d)) return st;
  return cuda_status(launch_finalize_f32(acc_f32, int64_t(T) * H, out_bf16, d.num_sms, stream),
                     "finalize_f32 launch");
}

int moe_grouped_gemm_mxfp4_range(const uint8_t* a_packed, const uint8_t* a_scales, const int32_t* expert_counts,
                                 const int32_t* row_offsets, int E, int64_t rows_capacity, int64_t m_total,
                                 const uint8_t* w_packed, const uint8_t* w_scales, int N, int K, int epilogue,
                                 void* c_out, uint8_t* c_scales, int tile_n, int w_layout, int32_t min_rows,
                                 int32_t max_rows, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return grouped_gemm_common(true, a_packed, a_scales, nullptr, expert_counts, row_offsets, E, rows_capacity, m_total,
                             w_packed, w_scales, nullptr, N, K, epilogue, nullptr, c_out, c_scales, tile_n, w_layout,
                             min_rows, max_rows, ws, ws_bytes, stream);
}

// ---- a6 ---------------------------------------------------------------------
int moe_finalize(const void* y_bf16, const int32_t* flat_to_perm, const float* topk_w, int T, int k, int H,
                 int64_t rows_capacity, void* out_bf16, cudaStream_t stream) {
  t_detail[0] = 0;
  NVFP4MOE_REQUIRE(T >= 0 && k >= 1 && k <= 1024, NVFP4MOE_ERR_INVALID_ARG, "T %d k %d", T, k);
  NVFP4MOE_REQUIRE(H > 0 && H % 8 == 0, NVFP4MOE_ERR_UNSUPPORTED, "H = %d must be a multiple of 8", H);
  NVFP4MOE_REQUIRE(rows_capacity >= 0, NVFP4MOE_ERR_INVALID_ARG, "rows_capacity < 0");
  if (T == 0) return NVFP4MOE_OK;
  NVFP4MOE_REQUIRE(y_bf16 && flat_to_perm && topk_w && out_bf16, NVFP4MOE_ERR_INVALID_ARG, "null pointer");
  NVFP4MOE_REQUIRE(aligned16(y_bf16) && aligned16(out_bf16), NVFP4MOE_ERR_INVALID_ARG, "misaligned pointer");
  DeviceInfo d;
  if (int st = current_device(&d)) return st;
  return cuda_status(launch_finalize(y_bf16, flat_to_perm, topk_w, T, k, H, rows_capacity, out_bf16, stream),
                     "finalize launch");
}

}  // extern "C"
