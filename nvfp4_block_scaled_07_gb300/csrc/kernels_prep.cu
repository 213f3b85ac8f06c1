// Memory-bound kernels of the NVFP4 MoE layer: top-k routing, bf16 -> NVFP4
// quantisation, scale re-layout, expert-first permutation and the weighted
// finalize.  All are HBM/latency bound (no contraction), so they use
// 128-bit loads, one warp per token or row, and grid-stride loops sized to
// a multiple of the SM count.
#include <cfloat>
#include <climits>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace nvfp4moe {

namespace {

__device__ unsigned g_prep_flags = 0;

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
  return v;
}

// ---------------------------------------------------------------------------
// a1: top-k routing ("SM120 FP4 Kernel Research Campaign", key finding 8:
// sigmoid expert scoring; softmax for the tiny layer).  One warp per token;
// lane l holds experts l, l+32, ...; k rounds of a warp arg-max with the
// lower expert index winning ties.
// ---------------------------------------------------------------------------
template <int VPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits,
                                                         const float* __restrict__ bias, int T, int E, int k,
                                                         int score_fn, int renorm, int32_t* __restrict__ idx_out,
                                                         float* __restrict__ w_out) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;  // uniform per warp
  const float* row = logits + int64_t(t) * E;
  float v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    float x = -INFINITY;
    if (e < E) {
      x = bias ? row[e] + bias[e] : row[e];
      if (x != x) x = -INFINITY;  // NaN never wins
    }
    v[i] = x;
  }
  uint32_t used = 0;
  int my_e = 0;
  float my_v = -INFINITY;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = INT_MAX;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((used >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, off);
      const int oe = __shfl_xor_sync(kFull, be, off);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) used |= 1u << (be >> 5);
    if (lane == j) {
      my_e = be;
      my_v = bv;
    }
  }
  const bool mine = lane < k;
  double wj;
  if (score_fn == 0) {  // softmax; slot 0 holds the largest value of all E
    const double vmax = double(__shfl_sync(kFull, my_v, 0));
    const double ex = mine ? exp(double(my_v) - vmax) : 0.0;
    double den;
    if (renorm) {
      den = warp_sum(ex);
    } else {
      double part = 0.0;
#pragma unroll
      for (int i = 0; i < VPL; ++i)
        if (lane + 32 * i < E) part += exp(double(v[i]) - vmax);
      den = warp_sum(part);
    }
    wj = ex / den;
  } else {  // sigmoid of the (biased) logit
    const double sg = mine ? 1.0 / (1.0 + exp(-double(my_v))) : 0.0;
    wj = renorm ? sg / warp_sum(sg) : sg;
  }
  if (mine) {
    idx_out[int64_t(t) * k + lane] = my_e;
    w_out[int64_t(t) * k + lane] = float(wj);
  }
}

// ---------------------------------------------------------------------------
// a2: bf16 -> NVFP4 ("SM120 FP4 Kernel Research Campaign", section 1 operand
// types).  One thread per 16-element block: two 128-bit loads, block amax,
// ue4m3 scale, 16 E2M1 codes packed into 8 bytes.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) amax_kernel(const uint4* __restrict__ x, int64_t nvec,
                                                   unsigned* __restrict__ amax_bits) {
  float m = 0.f;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += int64_t(gridDim.x) * blockDim.x) {
    const uint4 q = x[i];
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < int(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
    atomicMax(amax_bits, __float_as_uint(m));  // non-negative floats order like their bit patterns
  }
}

__global__ void __launch_bounds__(256) quantize_kernel(const uint4* __restrict__ x, int64_t rows, int64_t cols,
                                                       const float* __restrict__ gscale_in,
                                                       const unsigned* __restrict__ amax_bits,
                                                       float* __restrict__ gscale_out, uint8_t* __restrict__ packed,
                                                       uint8_t* __restrict__ scales, int blocked) {
  float s;
  if (amax_bits) {
    const float a = __uint_as_float(*amax_bits);
    s = a > 0.f ? a / kGlobalScaleDivisor : 1.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0) *gscale_out = s;
  } else {
    s = *gscale_in;
  }
  const int64_t bpr = cols / 16;  // blocks per row
  const int64_t nblk = rows * bpr;
  const int64_t nblk_pad = blocked ? ((rows + 127) / 128) * 128 * bpr : nblk;
  const int64_t kblocks = cols / 64;
  for (int64_t b = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; b < nblk_pad;
       b += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = b / bpr, c16 = b - row * bpr;
    uint32_t sb = 0;
    if (b < nblk) {
      const uint4 lo = x[2 * b], hi = x[2 * b + 1];
      const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
      float f[16];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        f[2 * j] = bf16_lo(w[j]);
        f[2 * j + 1] = bf16_hi(w[j]);
      }
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) a = fmaxf(a, fabsf(f[j]));
      const float t = (a / kE2M1Max) / s;
      sb = f32_to_ue4m3(t);
      const float d = ue4m3_to_f32(sb) * s;
      uint32_t p0 = 0, p1 = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        p0 |= e2m1_code(f[j], d) << (4 * j);
        p1 |= e2m1_code(f[8 + j], d) << (4 * j);
      }
      *reinterpret_cast<uint2*>(packed + 8 * b) = make_uint2(p0, p1);
    }
    if (blocked)
      scales[blocked_sf_offset(row, c16 >> 2, kblocks) + (c16 & 3)] = uint8_t(sb);
    else
      scales[b] = uint8_t(sb);
  }
}

// Row-major [rows, cols/16] scales -> blocked layout, one 4-byte group per thread.
__global__ void __launch_bounds__(256) scales_to_blocked_kernel(const uint8_t* __restrict__ src, int64_t rows,
                                                                int64_t cols, uint8_t* __restrict__ dst) {
  const int64_t kblocks = cols / 64;
  const int64_t total = ((rows + 127) / 128) * 128 * kblocks;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = i / kblocks, kb = i - row * kblocks;
    uint32_t v = 0;
    if (row < rows) v = reinterpret_cast<const uint32_t*>(src + row * (cols / 16))[kb];
    *reinterpret_cast<uint32_t*>(dst + blocked_sf_offset(row, kb, kblocks)) = v;
  }
}

// ---------------------------------------------------------------------------
// a3: expert-first permutation ("SM120 FP4 Kernel Research Campaign",
// section 6: expert-first layout and token reordering).  Stable counting
// sort of the flat ids by expert in three steps:
//   rank  - each warp ranks a segment of 1024 flat ids: __match_any groups
//           equal experts inside 32 ids, a per-warp shared counter carries
//           the running count across the segment;
//   scan  - one block turns per-segment counts into per-segment bases,
//           expert counts, offsets and 128-aligned row offsets (warp scans);
//   place - one warp per flat id writes the maps and gathers the packed row
//           and its scales into the expert-padded buffers.
// ---------------------------------------------------------------------------
constexpr int kRankWarps = 8;

__global__ void __launch_bounds__(kRankWarps * 32) permute_rank_kernel(const int32_t* __restrict__ idx, int64_t R,
                                                                       int E, int nseg,
                                                                       int32_t* __restrict__ rank,
                                                                       int32_t* __restrict__ seg_count) {
  extern __shared__ int32_t cnt_all[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = blockIdx.x * kRankWarps + warp;
  if (seg >= nseg) return;  // uniform per warp; no block-wide barrier below
  int32_t* cnt = cnt_all + warp * E;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
  const int64_t base = int64_t(seg) * kPermuteSegment;
  // All ids of the segment first, so their loads are in flight together.
  int ids[kPermuteSegment / 32];
#pragma unroll
  for (int it = 0; it < kPermuteSegment / 32; ++it) {
    const int64_t f = base + it * 32 + lane;
    ids[it] = f < R ? idx[f] : -1;
  }
#pragma unroll
  for (int it = 0; it < kPermuteSegment / 32; ++it) {
    const int64_t f = base + it * 32 + lane;
    int e = ids[it];
    if (f < R && (e < 0 || e >= E)) {
      atomicOr(&g_prep_flags, kFlagBadData);
      e = -1;
    }
    const unsigned grp = __match_any_sync(kFull, e);
    int r = -1;
    if (e >= 0) r = cnt[e] + __popc(grp & lt);
    __syncwarp();
    if (e >= 0 && lane == __ffs(grp) - 1) cnt[e] += __popc(grp);
    __syncwarp();
    if (f < R) rank[f] = r;
  }
  for (int e = lane; e < E; e += 32) seg_count[int64_t(seg) * E + e] = cnt[e];
}

__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot) {
  // blockDim.x == 1024
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(kFull, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kFull, wi, off);
      if (lane >= off) wi += o;
    }
    warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
  }
  __syncthreads();
  const int res = warp_tot[warp] + incl - v;
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(1024) permute_scan_kernel(const int32_t* __restrict__ seg_count, int nseg, int E,
                                                            int32_t* __restrict__ seg_base,
                                                            int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ row_offsets,
                                                            int32_t* __restrict__ perm_to_flat,
                                                            int64_t rows_capacity) {
  __shared__ int warp_tot[32];
  __shared__ int tail_start;
  __shared__ int s_cnt[1024], s_roff[1024];
  const int e = threadIdx.x;
  int run = 0;
  if (e < E) {
    for (int s = 0; s < nseg; ++s) {
      const int c = seg_count[int64_t(s) * E + e];
      seg_base[int64_t(s) * E + e] = run;
      run += c;
    }
  }
  const int cnt = e < E ? run : 0;
  const int padded = (cnt + 127) & ~127;
  const int off = block_exclusive_scan(cnt, warp_tot);
  const int roff = block_exclusive_scan(padded, warp_tot);
  if (e < E) {
    counts[e] = cnt;
    offsets[e] = off;
    row_offsets[e] = roff;
    s_cnt[e] = cnt;
    s_roff[e] = roff;
  }
  if (e == E - 1) {
    offsets[E] = off + cnt;
    row_offsets[E] = roff + padded;
    tail_start = roff + padded;
  }
  __syncthreads();
  // Padding rows of each expert (one warp per expert, coalesced), then the tail.
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int x = warp; x < E; x += 32) {
    const int c = s_cnt[x], pad = (c + 127) & ~127;
    for (int r = c + lane; r < pad; r += 32) perm_to_flat[s_roff[x] + r] = -1;
  }
  for (int64_t p = int64_t(tail_start) + threadIdx.x; p < rows_capacity; p += blockDim.x) perm_to_flat[p] = -1;
}

__global__ void __launch_bounds__(256) permute_place_kernel(const int32_t* __restrict__ idx, int64_t R, int k, int E,
                                                            const int32_t* __restrict__ rank,
                                                            const int32_t* __restrict__ seg_base,
                                                            const int32_t* __restrict__ row_offsets,
                                                            const uint8_t* __restrict__ xq,
                                                            const uint8_t* __restrict__ xs, int H,
                                                            int32_t* __restrict__ perm_to_flat,
                                                            int32_t* __restrict__ flat_to_perm,
                                                            uint8_t* __restrict__ a_packed,
                                                            uint8_t* __restrict__ a_scales) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
  const int64_t kblocks = H / 64;
  for (int64_t f = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); f < R; f += nwarps) {
    const int e = idx[f];
    if (e < 0 || e >= E) continue;  // flagged by the rank step
    const int64_t seg = f / kPermuteSegment;
    const int64_t row = int64_t(row_offsets[e]) + seg_base[seg * E + e] + rank[f];
    if (lane == 0) {
      perm_to_flat[row] = int32_t(f);
      flat_to_perm[f] = int32_t(row);
    }
    const int64_t t = f / k;
    const uint4* src = reinterpret_cast<const uint4*>(xq + t * (H / 2));
    uint4* dst = reinterpret_cast<uint4*>(a_packed + row * (H / 2));
    for (int c = lane; c < H / 32; c += 32) dst[c] = src[c];
    const uint32_t* ssrc = reinterpret_cast<const uint32_t*>(xs + t * (H / 16));
    for (int kb = lane; kb < kblocks; kb += 32)
      *reinterpret_cast<uint32_t*>(a_scales + blocked_sf_offset(row, kb, kblocks)) = ssrc[kb];
  }
}

// ---------------------------------------------------------------------------
// a6: finalize ("SM120 FP4 Kernel Research Campaign", section 6: token
// reordering with fused reduction; "Uncovering SM120 CUTLASS Collective
// Implementations", Context: the finalize epilogue).  Each thread owns 8
// consecutive columns of one token and sums its k expert rows in slot order.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) finalize_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ f2p,
                                                       const float* __restrict__ w, int T, int k, int H,
                                                       int64_t rows_capacity, uint4* __restrict__ out) {
  const int t = blockIdx.x;
  const int c8 = blockIdx.y * blockDim.x + threadIdx.x;  // column group of 8
  if (c8 * 8 >= H) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < k; ++j) {
    const int64_t row = f2p[int64_t(t) * k + j];
    const float wj = w[int64_t(t) * k + j];
    if (row < 0 || row >= rows_capacity) {
      if (c8 == 0) atomicOr(&g_prep_flags, kFlagBadData);
      continue;
    }
    const uint4 q = y[(row * H) / 8 + c8];
    const uint32_t v[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = fmaf(wj, bf16_lo(v[i]), acc[2 * i]);
      acc[2 * i + 1] = fmaf(wj, bf16_hi(v[i]), acc[2 * i + 1]);
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);  // .x = low half
    o[i] = *reinterpret_cast<const uint32_t*>(&p);
  }
  out[(int64_t(t) * H) / 8 + c8] = make_uint4(o[0], o[1], o[2], o[3]);
}

int grid_for(int64_t work_items, int threads, int num_sms, int per_sm) {
  const int64_t need = (work_items + threads - 1) / threads;
  const int64_t cap = int64_t(num_sms) * per_sm;
  return int(need < 1 ? 1 : (need < cap ? need : cap));
}

}  // namespace

cudaError_t launch_route_topk(const float* logits, const float* bias, int T, int E, int k, int score_fn,
                              int renormalize, int32_t* idx, float* w, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int warps = 8;
  const dim3 grid((T + warps - 1) / warps), block(warps * 32);
  const int vpl = (E + 31) / 32;
#define NVFP4MOE_ROUTE(V)                                                                          \
  route_topk_kernel<V><<<grid, block, 0, st>>>(logits, bias, T, E, k, score_fn, renormalize, idx, w); \
  break;
  switch (vpl <= 1 ? 1 : vpl <= 2 ? 2 : vpl <= 4 ? 4 : vpl <= 8 ? 8 : vpl <= 16 ? 16 : 32) {
    case 1: NVFP4MOE_ROUTE(1)
    case 2: NVFP4MOE_ROUTE(2)
    case 4: NVFP4MOE_ROUTE(4)
    case 8: NVFP4MOE_ROUTE(8)
    case 16: NVFP4MOE_ROUTE(16)
    default: NVFP4MOE_ROUTE(32)
  }
#undef NVFP4MOE_ROUTE
  return cudaGetLastError();
}

cudaError_t launch_quantize(const void* x, int64_t rows, int64_t cols, float* global_scale, bool compute_global,
                            bool blocked, uint8_t* packed, uint8_t* scales, unsigned* amax_ws, int num_sms,
                            cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int64_t nblk = rows * (cols / 16);
  if (compute_global) {
    cudaError_t err = cudaMemsetAsync(amax_ws, 0, sizeof(unsigned), st);
    if (err != cudaSuccess) return err;
    amax_kernel<<<grid_for(nblk * 2, 256, num_sms, 8), 256, 0, st>>>(static_cast<const uint4*>(x), nblk * 2,
                                                                       amax_ws);
  }
  const int64_t work = blocked ? ((rows + 127) / 128) * 128 * (cols / 16) : nblk;
  quantize_kernel<<<grid_for(work, 256, num_sms, 8), 256, 0, st>>>(
      static_cast<const uint4*>(x), rows, cols, global_scale, compute_global ? amax_ws : nullptr, global_scale,
      packed, scales, blocked ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_scales_to_blocked(const uint8_t* src, int64_t rows, int64_t cols, uint8_t* dst, int num_sms,
                                     cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int64_t total = ((rows + 127) / 128) * 128 * (cols / 64);
  scales_to_blocked_kernel<<<grid_for(total, 256, num_sms, 8), 256, 0, st>>>(src, rows, cols, dst);
  return cudaGetLastError();
}

cudaError_t launch_permute(const int32_t* topk_idx, int T, int E, int k, const uint8_t* xq, const uint8_t* xs,
                           int H, int32_t* counts, int32_t* offsets, int32_t* row_offsets, int32_t* perm_to_flat,
                           int32_t* flat_to_perm, uint8_t* a_packed, uint8_t* a_scales, int64_t rows_capacity,
                           int32_t* ws_rank, int32_t* ws_seg_count, int32_t* ws_seg_base, int num_sms,
                           cudaStream_t st) {
  const int64_t R = int64_t(T) * k;
  const int nseg = int((R + kPermuteSegment - 1) / kPermuteSegment);
  if (nseg > 0) {
    const size_t smem = size_t(kRankWarps) * E * sizeof(int32_t);
    if (smem > 48 * 1024) {
      cudaError_t err =
          cudaFuncSetAttribute(permute_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (err != cudaSuccess) return err;
    }
    permute_rank_kernel<<<(nseg + kRankWarps - 1) / kRankWarps, kRankWarps * 32, smem, st>>>(topk_idx, R, E, nseg,
                                                                                           ws_rank, ws_seg_count);
  }
  permute_scan_kernel<<<1, 1024, 0, st>>>(ws_seg_count, nseg, E, ws_seg_base, counts, offsets, row_offsets,
                                          perm_to_flat, rows_capacity);
  if (R > 0)
    permute_place_kernel<<<grid_for(R * 32, 256, num_sms, 8), 256, 0, st>>>(
        topk_idx, R, k, E, ws_rank, ws_seg_base, row_offsets, xq, xs, H, perm_to_flat, flat_to_perm, a_packed,
        a_scales);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const void* y, const int32_t* flat_to_perm, const float* w, int T, int k, int H,
                            int64_t rows_capacity, void* out, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const dim3 block(128), grid(T, (H / 8 + 127) / 128);
  finalize_kernel<<<grid, block, 0, st>>>(static_cast<const uint4*>(y), flat_to_perm, w, T, k, H, rows_capacity,
                                          static_cast<uint4*>(out));
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Permutation with library-owned scratch, for callers that cannot allocate
// device memory at call time.  The scratch is one file-scope device array,
// present on every GPU that loads the library until the process exits.
// Host code may not use the array's name as a device address, so its
// address is looked up once per device with cudaGetSymbolAddress.
// ---------------------------------------------------------------------------
static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocMaxRoutedRows + 2 * kNoAllocMaxSegmentExperts];

namespace {
constexpr int kScratchDevices = 64;
std::mutex g_scratch_mutex;
int32_t* g_scratch_addr[kScratchDevices] = {};
}  // namespace

cudaError_t launch_permute_static_scratch(const int32_t* topk_idx, int T, int E, int k, const uint8_t* xq,
                                          const uint8_t* xs, int H, int32_t* counts, int32_t* offsets,
                                          int32_t* row_offsets, int32_t* perm_to_flat, int32_t* flat_to_perm,
                                          uint8_t* a_packed, uint8_t* a_scales, int64_t rows_capacity, int num_sms,
                                          cudaStream_t st) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kScratchDevices) return cudaErrorInvalidDevice;
  int32_t* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      err = cudaGetSymbolAddress(&p, g_permute_scratch);  // device `dev` is current here
      if (err != cudaSuccess) return err;
      g_scratch_addr[dev] = static_cast<int32_t*>(p);
    }
    base = g_scratch_addr[dev];
  }
  int32_t* rank = base;
  int32_t* seg_count = rank + kNoAllocMaxRoutedRows;
  int32_t* seg_base = seg_count + kNoAllocMaxSegmentExperts;
  return launch_permute(topk_idx, T, E, k, xq, xs, H, counts, offsets, row_offsets, perm_to_flat, flat_to_perm,
                        a_packed, a_scales, rows_capacity, rank, seg_count, seg_base, num_sms, st);
}

cudaError_t prep_read_and_clear_flags(unsigned* flags) {
  unsigned zero = 0;
  cudaError_t err = cudaMemcpyFromSymbol(flags, g_prep_flags, sizeof(unsigned));
  if (err != cudaSuccess) return err;
  return cudaMemcpyToSymbol(g_prep_flags, &zero, sizeof(unsigned));
}

}  // namespace nvfp4moe
