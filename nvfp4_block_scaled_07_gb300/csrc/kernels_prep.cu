// Memory-bound kernels of the NVFP4 MoE layer: top-k routing, bf16 -> NVFP4
// quantisation, scale re-layout, expert-first permutation and the weighted
// finalize.  All are HBM/latency bound (no contraction), so they use
// 128-bit loads, one warp per token or row, and grid-stride loops sized to
// a multiple of the SM count.
#include <cuda.h>

#include <cfloat>
#include <climits>
#include <cstdint>
#include <mutex>

#include "../../include/nvfp4moe.h"
#include "common.cuh"
#include "internal.h"
#include "launch.cuh"
#include "sm103_ptx.cuh"

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
//
// Batch-aware routing (same page, key finding 6 and section 6: during
// decode a token gives up the experts it weights least in favour of experts
// other tokens of the batch already use).  Pass 1 marks every token's top-k_primary experts in
// a bit set S; pass 2 ranks each token's experts with members of S first
// (then value, then index) and takes k of them.  Plain top-k is pass 2 with
// every expert a member.
// ---------------------------------------------------------------------------
template <int VPL>
__device__ __forceinline__ void router_values(const float* __restrict__ logits, const float* __restrict__ bias, int t,
                                              int E, int lane, float (&v)[VPL]) {
  const float* row = logits + int64_t(t) * E;
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
}

// k rounds of a warp arg-max.  member_bits bit i: expert lane + 32 i is in
// the preferred set; the first `nmem` rounds (the set's size across the
// warp) choose among members, the rest among non-members.  Lane j < k ends
// with the j-th choice in (my_e, my_v).
template <int VPL>
__device__ __forceinline__ void select_ranked(const float (&v)[VPL], uint32_t member_bits, int nmem, int E, int k,
                                              int lane, int& my_e, float& my_v) {
  uint32_t used = 0;
  my_e = 0;
  my_v = -INFINITY;
  for (int j = 0; j < k; ++j) {
    const uint32_t want = j < nmem ? member_bits : ~member_bits;
    float bv = -INFINITY;
    int be = INT_MAX;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((used >> i) & 1u) && ((want >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
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
}

// Weights of the k chosen experts (lane j < k holds choice j) and the stores.
template <int VPL>
__device__ __forceinline__ void route_weights_store(const float (&v)[VPL], int my_e, float my_v, int t, int E, int k,
                                                   int score_fn, int renorm, int32_t* __restrict__ idx_out,
                                                   float* __restrict__ w_out, int lane) {
  const bool mine = lane < k;
  double wj;
  if (score_fn == 0) {  // softmax; slot 0 holds the token's largest value of all E
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
  } else {
    // Sigmoid of the (biased) logit in float32 (expf is within 2 ulp), the
    // sum over the k selected in float64: the weight is within ~7 ulp of the
    // exact value, far below the 1e-6 relative bar, at a fraction of the
    // float64 cost.
    const float sg = mine ? 1.0f / (1.0f + expf(-my_v)) : 0.0f;
    wj = renorm ? double(sg / float(warp_sum(double(sg)))) : double(sg);
  }
  if (mine) {
    idx_out[int64_t(t) * k + lane] = my_e;
    w_out[int64_t(t) * k + lane] = float(wj);
  }
}

// Lane's member bits of the set S (E/32 words, expert e = bit e % 32 of word e / 32).
template <int VPL>
__device__ __forceinline__ uint32_t member_bits_of(const uint32_t* set, int E, int lane) {
  uint32_t bits = 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (lane + 32 * i < E) bits |= ((__ldcg(set + i) >> lane) & 1u) << i;
  return bits;
}

template <int VPL>
__device__ __forceinline__ int valid_bits_count(uint32_t bits, int E, int lane) {
  uint32_t valid = 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (lane + 32 * i < E) valid |= 1u << i;
  return int(__reduce_add_sync(kFull, unsigned(__popc(bits & valid))));
}

// Plain top-k (active_set == nullptr) or pass 2 of batch-aware routing.
template <int VPL>
__device__ __forceinline__ void route_token(const float* __restrict__ logits, const float* __restrict__ bias, int t,
                                            int E, int k, int score_fn, int renorm, const uint32_t* active_set,
                                            int32_t* __restrict__ idx_out, float* __restrict__ w_out, int lane) {
  float v[VPL];
  router_values<VPL>(logits, bias, t, E, lane, v);
  uint32_t bits = ~0u;
  int nmem = E;
  if (active_set) {
    bits = member_bits_of<VPL>(active_set, E, lane);
    nmem = valid_bits_count<VPL>(bits, E, lane);
  }
  int my_e;
  float my_v;
  select_ranked<VPL>(v, bits, nmem, E, k, lane, my_e, my_v);
  route_weights_store<VPL>(v, my_e, my_v, t, E, k, score_fn, renorm, idx_out, w_out, lane);
}

// Pass 1 of batch-aware routing: the token's top-k_primary join the set S.
template <int VPL>
__device__ __forceinline__ void mark_primary(const float* __restrict__ logits, const float* __restrict__ bias, int t,
                                             int E, int k_primary, uint32_t* active_set, int lane) {
  float v[VPL];
  router_values<VPL>(logits, bias, t, E, lane, v);
  int my_e;
  float my_v;
  select_ranked<VPL>(v, ~0u, E, E, k_primary, lane, my_e, my_v);
  if (lane < k_primary) atomicOr(active_set + (my_e >> 5), 1u << (my_e & 31));
}

template <int VPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits,
                                                         const float* __restrict__ bias, int T, int E, int k,
                                                         int score_fn, int renorm, const uint32_t* active_set,
                                                         int32_t* __restrict__ idx_out, float* __restrict__ w_out) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;  // uniform per warp
  route_token<VPL>(logits, bias, t, E, k, score_fn, renorm, active_set, idx_out, w_out, threadIdx.x & 31);
}

template <int VPL>
__global__ void __launch_bounds__(256) route_mark_kernel(const float* __restrict__ logits,
                                                         const float* __restrict__ bias, int T, int E, int k_primary,
                                                         uint32_t* active_set) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;  // uniform per warp
  mark_primary<VPL>(logits, bias, t, E, k_primary, active_set, threadIdx.x & 31);
}

// ---------------------------------------------------------------------------
// a2: bf16 -> NVFP4 ("SM120 FP4 Kernel Research Campaign", section 1 operand
// types).  One thread per 16-element block: two 128-bit loads, block amax,
// ue4m3 scale, 16 E2M1 codes packed into 8 bytes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float amax8(uint4 q, float m) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
  return m;
}

// The 16 bf16 values in (lo, hi) with per-tensor scale s -> ue4m3 block
// scale (returned) and the packed codes, element 2i in the low nibble.
__device__ __forceinline__ uint32_t nvfp4_block16(uint4 lo, uint4 hi, float s, uint2* packed) {
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
  const uint32_t sb = f32_to_ue4m3(t);
  const float d = ue4m3_to_f32(sb) * s;
  uint32_t p0 = 0, p1 = 0;
  if (d != 0.0f) {  // a zero step gives code 0 for the whole block
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // q = x / d exactly as a float32 division, then the nearest code
      p0 |= e2m1x2(f[2 * j] / d, f[2 * j + 1] / d) << (8 * j);
      p1 |= e2m1x2(f[8 + 2 * j] / d, f[8 + 2 * j + 1] / d) << (8 * j);
    }
  }
  *packed = make_uint2(p0, p1);
  return sb;
}

__device__ __forceinline__ float global_scale_of(float amax) { return amax > 0.f ? amax / kGlobalScaleDivisor : 1.0f; }

__global__ void __launch_bounds__(256) amax_kernel(const uint4* __restrict__ x, int64_t nvec,
                                                   unsigned* __restrict__ amax_bits) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  float m = 0.f;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += int64_t(gridDim.x) * blockDim.x)
    m = amax8(x[i], m);
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
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  float s;
  if (amax_bits) {
    s = global_scale_of(__uint_as_float(*amax_bits));
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
      uint2 pk;
      sb = nvfp4_block16(x[2 * b], x[2 * b + 1], s, &pk);
      *reinterpret_cast<uint2*>(packed + 8 * b) = pk;
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
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int64_t kblocks = cols / 64;
  const int64_t total = ((rows + 127) / 128) * 128 * kblocks;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = i / kblocks, kb = i - row * kblocks;
    uint32_t v = 0;
    if (row < rows) v = reinterpret_cast<const uint32_t*>(src + row * (cols / 16))[kb];
    *reinterpret_cast<uint32_t*>(dst + blocked_sf_offset(row, kb, kblocks)) = v;
  }
}

// MXFP4 (E2M1 with one E8M0 scale per 32 elements, no per-tensor scale).
// One thread per 32-element block: four 128-bit loads, block amax, shared
// exponent, 32 codes packed into 16 bytes.  Scales row-major [rows, cols/32]
// or blocked (128-row x 128-K blocks of 512 bytes, row r's four scales at
// (r % 32) * 16 + (r / 32) * 4).
__global__ void __launch_bounds__(256) quantize_mx_kernel(const uint4* __restrict__ x, int64_t rows, int64_t cols,
                                                          uint8_t* __restrict__ packed, uint8_t* __restrict__ scales,
                                                          int blocked) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int64_t bpr = cols / 32;  // blocks per row
  const int64_t nblk = rows * bpr;
  const int64_t nblk_pad = blocked ? ((rows + 127) / 128) * 128 * bpr : nblk;
  const int64_t groups = cols / 128;
  for (int64_t b = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; b < nblk_pad;
       b += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = b / bpr, c32 = b - row * bpr;
    uint32_t sb = 0;
    if (b < nblk) {
      uint4 q[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) q[j] = x[4 * b + j];
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) a = amax8(q[j], a);
      const int X = mx_exponent(a);
      sb = uint32_t(X + 127);
      const float inv = mx_inv_step(X);
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t v[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) word |= mx_code2(bf16_lo(v[i]), bf16_hi(v[i]), inv) << (8 * i);
        w[j] = word;
      }
      reinterpret_cast<uint4*>(packed)[b] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (blocked)
      scales[blocked_sf_offset(row, c32 >> 2, groups) + (c32 & 3)] = uint8_t(sb);
    else
      scales[b] = uint8_t(sb);
  }
}

// ---------------------------------------------------------------------------
// a3: expert-first permutation ("SM120 FP4 Kernel Research Campaign",
// section 6: expert-first layout and token reordering).  Stable counting
// sort of the flat ids by expert in three steps:
//   rank  - each warp ranks a segment of 32*ITERS flat ids: __match_any
//           groups equal experts inside 32 ids, a per-warp shared counter
//           carries the running count across the segment;
//   scan  - one block turns per-segment counts into per-segment bases,
//           expert counts, offsets and 128-aligned row offsets (warp scans);
//   place - one warp per flat id writes the maps and gathers the packed row
//           and its scales into the expert-padded buffers.
// Data written earlier in the same grid (the fused prepare kernel) is read
// with ld.global.cg, which does not allocate in the non-coherent L1.
// ---------------------------------------------------------------------------
template <int ITERS>
__device__ __forceinline__ void rank_segment(const int32_t* idx, int64_t R, int E, int64_t seg, int32_t* cnt,
                                             int32_t* __restrict__ rank, int32_t* __restrict__ seg_count,
                                             int lane) {
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
  const int64_t base = seg * (ITERS * 32);
  // All ids of the segment first, so their loads are in flight together.
  int ids[ITERS];
#pragma unroll
  for (int it = 0; it < ITERS; ++it) {
    const int64_t f = base + it * 32 + lane;
    ids[it] = f < R ? __ldcg(idx + f) : -1;
  }
#pragma unroll
  for (int it = 0; it < ITERS; ++it) {
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
  for (int e = lane; e < E; e += 32) seg_count[seg * E + e] = cnt[e];
  __syncwarp();
}

constexpr int kRankWarps = 8;

__global__ void __launch_bounds__(kRankWarps * 32) permute_rank_kernel(const int32_t* __restrict__ idx, int64_t R,
                                                                       int E, int nseg,
                                                                       int32_t* __restrict__ rank,
                                                                       int32_t* __restrict__ seg_count) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  extern __shared__ int32_t cnt_all[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = blockIdx.x * kRankWarps + warp;
  if (seg >= nseg) return;  // uniform per warp; no block-wide barrier below
  rank_segment<kPermuteSegment / 32>(idx, R, E, seg, cnt_all + warp * E, rank, seg_count, lane);
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

// One block of 1024 threads (E <= 1024): per-segment bases, counts,
// offsets [E+1] and 128-aligned row offsets [E+1].  G threads per expert (a
// power of two, at most 32, so a group sits in one warp) each sum a run of
// segments, scan the runs with shuffles and write their segments' bases; the
// per-expert totals then go through block scans, thread e = expert e.
// (One thread per expert walking all segments took ~10 us at 128 segments.)
// s_tot: 1024 ints of shared memory.  Returns thread e's expert count and
// row offset.
__device__ __forceinline__ void scan_experts(const int32_t* seg_count, int nseg, int E, int32_t* __restrict__ seg_base,
                                             int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                             int32_t* __restrict__ row_offsets, int* warp_tot, int* s_tot, int* cnt_out,
                                             int* roff_out) {
  int ep = 1;
  while (ep < E) ep <<= 1;
  const int G = min(32, 1024 / ep);
  const int ge = threadIdx.x / G, sub = threadIdx.x % G;
  const int chunk = (nseg + G - 1) / G;
  const int sa = min(nseg, sub * chunk), sb = min(nseg, sa + chunk);
  int local = 0;
  if (ge < E) {
    int s = sa;
    for (; s + 8 <= sb; s += 8) {
      int c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) c[j] = __ldcg(seg_count + int64_t(s + j) * E + ge);
#pragma unroll
      for (int j = 0; j < 8; ++j) local += c[j];
    }
    for (; s < sb; ++s) local += __ldcg(seg_count + int64_t(s) * E + ge);
  }
  int incl = local;
  for (int off = 1; off < G; off <<= 1) {
    const int o = __shfl_up_sync(kFull, incl, off, G);
    if (sub >= off) incl += o;
  }
  if (ge < E) {
    // second pass in batches of 8 loads issued together (a load after each
    // store would wait out a full L2 round trip per segment)
    int run = incl - local;
    int s = sa;
    for (; s + 8 <= sb; s += 8) {
      int c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) c[j] = __ldcg(seg_count + int64_t(s + j) * E + ge);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        seg_base[int64_t(s + j) * E + ge] = run;
        run += c[j];
      }
    }
    for (; s < sb; ++s) {
      const int c = __ldcg(seg_count + int64_t(s) * E + ge);
      seg_base[int64_t(s) * E + ge] = run;
      run += c;
    }
    if (sub == G - 1) s_tot[ge] = incl;
  }
  __syncthreads();
  const int e = threadIdx.x;
  const int cnt = e < E ? s_tot[e] : 0;
  const int padded = (cnt + 127) & ~127;
  const int off = block_exclusive_scan(cnt, warp_tot);
  const int roff = block_exclusive_scan(padded, warp_tot);
  if (e < E) {
    counts[e] = cnt;
    offsets[e] = off;
    row_offsets[e] = roff;
  }
  if (e == E - 1) {
    offsets[E] = off + cnt;
    row_offsets[E] = roff + padded;
  }
  *cnt_out = cnt;
  *roff_out = roff;
}

__global__ void __launch_bounds__(1024) permute_scan_kernel(const int32_t* __restrict__ seg_count, int nseg, int E,
                                                            int32_t* __restrict__ seg_base,
                                                            int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ row_offsets,
                                                            int32_t* __restrict__ perm_to_flat,
                                                            int64_t rows_capacity) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  __shared__ int warp_tot[32];
  __shared__ int tail_start;
  __shared__ int s_cnt[1024], s_roff[1024], s_tot[1024];
  int cnt, roff;
  scan_experts(seg_count, nseg, E, seg_base, counts, offsets, row_offsets, warp_tot, s_tot, &cnt, &roff);
  const int e = threadIdx.x;
  if (e < E) {
    s_cnt[e] = cnt;
    s_roff[e] = roff;
  }
  if (e == E - 1) tail_start = roff + ((cnt + 127) & ~127);
  __syncthreads();
  // Padding rows of each expert (one warp per expert, coalesced), then the tail.
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int x = warp; x < E; x += 32) {
    const int c = s_cnt[x], pad = (c + 127) & ~127;
    for (int r = c + lane; r < pad; r += 32) perm_to_flat[s_roff[x] + r] = -1;
  }
  for (int64_t p = int64_t(tail_start) + threadIdx.x; p < rows_capacity; p += blockDim.x) perm_to_flat[p] = -1;
}

// Placement of up to 32 flat ids by one warp: lane l takes f = f0 + l * step
// (token f / k, slot f % k), finds its row in the expert-padded layout and
// writes both maps; then the warp copies each of those tokens' packed row
// and scales, all of a row's 16-byte chunks in flight at once.  The
// metadata loads of the 32 ids overlap, so a row costs one round trip.
// sf_groups = 4-byte scale groups per row: H/64 for NVFP4, H/128 for MXFP4.
__device__ __forceinline__ void place_rows(int64_t f0, int64_t step, int64_t R, const int32_t* idx, int k, int E,
                                           int seg_len, const int32_t* rank, const int32_t* seg_base,
                                           const int32_t* row_offsets, const uint8_t* xq, const uint8_t* xs, int H,
                                           int sf_groups, int32_t* __restrict__ perm_to_flat,
                                           int32_t* __restrict__ flat_to_perm, uint8_t* __restrict__ a_packed,
                                           uint8_t* __restrict__ a_scales, int lane, bool write_scales = true) {
  const int64_t f = f0 + int64_t(lane) * step;
  int64_t row = -1;
  if (f < R) {
    const int e = __ldcg(idx + f);
    if (e >= 0 && e < E) {  // an id out of range is flagged by the rank step
      const int r = __ldcg(rank + f);
      row = int64_t(__ldcg(row_offsets + e)) + __ldcg(seg_base + (f / seg_len) * E + e) + r;
      perm_to_flat[row] = int32_t(f);
      flat_to_perm[f] = int32_t(row);
    }
  }
  const int nv = H / 32;  // 16-byte chunks of one packed row
  for (int j = 0; j < 32; ++j) {
    const int64_t rj = __shfl_sync(kFull, row, j);
    if (rj < 0) continue;  // uniform across the warp
    const int64_t t = (f0 + int64_t(j) * step) / k;
    const uint4* src = reinterpret_cast<const uint4*>(xq + t * (H / 2));
    uint4* dst = reinterpret_cast<uint4*>(a_packed + rj * (H / 2));
    for (int c0 = 0; c0 < nv; c0 += 256) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + 32 * u + lane;
        if (c < nv) v[u] = __ldcg(src + c);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + 32 * u + lane;
        if (c < nv) dst[c] = v[u];
      }
    }
    if (!write_scales) continue;  // uniform across the warp
    const unsigned* ssrc = reinterpret_cast<const unsigned*>(xs + t * (4 * int64_t(sf_groups)));
    for (int kb = lane; kb < sf_groups; kb += 32)
      *reinterpret_cast<uint32_t*>(a_scales + blocked_sf_offset(rj, kb, sf_groups)) = __ldcg(ssrc + kb);
  }
}

__global__ void __launch_bounds__(256) permute_place_kernel(const int32_t* __restrict__ idx, int64_t R, int k, int E,
                                                            const int32_t* __restrict__ rank,
                                                            const int32_t* __restrict__ seg_base,
                                                            const int32_t* __restrict__ row_offsets,
                                                            const uint8_t* __restrict__ xq,
                                                            const uint8_t* __restrict__ xs, int H, int sf_groups,
                                                            int32_t* __restrict__ perm_to_flat,
                                                            int32_t* __restrict__ flat_to_perm,
                                                            uint8_t* __restrict__ a_packed,
                                                            uint8_t* __restrict__ a_scales) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
  const int64_t w0 = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  for (int64_t f0 = w0; f0 < R; f0 += 32 * nwarps)
    place_rows(f0, nwarps, R, idx, k, E, kPermuteSegment, rank, seg_base, row_offsets, xq, xs, H, sf_groups,
               perm_to_flat, flat_to_perm, a_packed, a_scales, lane);
}

// ---------------------------------------------------------------------------
// a1 + a2 + a3 in one cooperative launch.  Four phases separated by grid
// barriers (every CTA resident, bounded waits):
//   A  route (one warp per token) and per-CTA partial amax of x (NVFP4);
//   B  global scale from the partials, quantisation of x (NVFP4, or MXFP4
//      with no global scale), segment ranks;
//   C  CTA 0 scans the segment counts;
//   D  padding rows, placement and the gather of packed rows and scales.
// Each step is the same device code as in the separate kernels above, so the
// results are identical bit for bit.
// ---------------------------------------------------------------------------
struct PrepareParams {
  const float* logits;
  const float* bias;
  const uint4* x;
  int T, E, k, k_primary, H, score_fn, renorm, nseg;
  int mx;  // MXFP4 (E8M0 scale per 32 elements, no global scale) instead of NVFP4
  int32_t* idx;
  float* w;
  float* gscale;
  uint8_t* xq;
  uint8_t* xs;
  int32_t* counts;
  int32_t* offsets;
  int32_t* row_offsets;
  int32_t* perm_to_flat;
  int32_t* flat_to_perm;
  uint8_t* a_packed;
  uint8_t* a_scales;
  int64_t rows_cap;
  uint32_t* bar;  // [0] arrivals, [32] generation: separate 128-byte lines
  uint32_t wait_us;  // limit of each grid-barrier wait (nvfp4moe_set_wait_limit_us)
  uint32_t* active_set;  // batch-aware routing: E bits, zero between calls
  float* amax_part;
  int32_t* rank;
  int32_t* seg_count;
  int32_t* seg_base;
};

constexpr int kPrepThreads = 1024;
constexpr int kRouteWarps = 16;  // most routing warps per CTA in phase A (NVFP4)
// All CTAs of the grid meet here.  Thread 0 of each CTA arrives on a
// device-scope counter; the last arrival resets it and bumps the generation
// word the others poll (bounded by the launch's wait limit).  Returns false, the same
// in every thread of the CTA, if the wait gave up or the counter held a
// value no launch leaves behind; the caller then abandons the kernel.
__device__ __forceinline__ bool grid_barrier(uint32_t* bar, int* s_ok, uint32_t wait_us) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    uint32_t* count = bar;
    uint32_t* gen = bar + 32;
    const uint32_t g = ptx::ld_acquire_gpu(gen);
    __threadfence();
    const uint32_t arrived = atomicAdd(count, 1u) + 1u;
    if (arrived == gridDim.x) {
      atomicExch(count, 0u);
      __threadfence();
      ptx::red_release_gpu_add(gen, 1u);
    } else if (arrived > gridDim.x) {
      atomicOr(&g_prep_flags, kFlagBadData);
      ok = 0;
    } else {
      const uint64_t t0 = ptx::globaltimer_ns();
      while (ptx::ld_acquire_gpu(gen) == g) {
        if (ptx::globaltimer_ns() - t0 > uint64_t(wait_us) * 1000u) {
          atomicOr(&g_prep_flags, kFlagTimeout);
          ok = 0;
          break;
        }
      }
    }
    __threadfence();
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

template <int VPL, int ITERS>
__global__ void __launch_bounds__(kPrepThreads, 1) prepare_kernel(const PrepareParams p) {
  extern __shared__ int32_t s_rank_cnt[];  // kRankWarps x E
  __shared__ float s_red[32];
  __shared__ int s_ok;
  __shared__ int warp_tot[32];
  __shared__ int s_tot[1024];
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarp = kPrepThreads / 32;
  const int64_t tid = int64_t(blockIdx.x) * kPrepThreads + threadIdx.x;
  const int64_t nthreads = int64_t(gridDim.x) * kPrepThreads;
  const int64_t gw0 = int64_t(warp) * gridDim.x + blockIdx.x;  // warps interleaved across CTAs
  const int64_t gw_stride = int64_t(gridDim.x) * nwarp;
  const int64_t R = int64_t(p.T) * p.k;

  // ---- A: routing (batch-aware: its first pass) and partial amax ----------
  // The first nroute warps of every CTA route (compute and latency bound;
  // as many as give each at most one token, up to kRouteWarps) while the
  // others stream x for its amax (HBM bound), so the two overlap; with no
  // amax (MXFP4) every warp routes.
  const bool batch_aware = p.k_primary < p.k;
  const int nroute = p.mx ? nwarp : min(kRouteWarps, max(1, int((p.T + gridDim.x - 1) / gridDim.x)));
  if (warp < nroute) {
    for (int64_t t = int64_t(warp) * gridDim.x + blockIdx.x; t < p.T; t += int64_t(gridDim.x) * nroute) {
      if (batch_aware)
        mark_primary<VPL>(p.logits, p.bias, int(t), p.E, p.k_primary, p.active_set, lane);
      else
        route_token<VPL>(p.logits, p.bias, int(t), p.E, p.k, p.score_fn, p.renorm, nullptr, p.idx, p.w, lane);
    }
  }
  if (!p.mx) {
    float m = 0.f;
    if (warp >= nroute) {
      // 8 independent 16-byte loads in flight per thread
      const int64_t na = int64_t(gridDim.x) * (kPrepThreads - 32 * nroute);
      const int64_t nvec = int64_t(p.T) * p.H / 8;
      int64_t i = int64_t(blockIdx.x) * (kPrepThreads - 32 * nroute) + (threadIdx.x - 32 * nroute);
      for (; i + 7 * na < nvec; i += 8 * na) {
        uint4 q[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) q[u] = __ldg(p.x + i + u * na);
#pragma unroll
        for (int u = 0; u < 8; ++u) m = amax8(q[u], m);
      }
      for (; i < nvec; i += na) m = amax8(__ldg(p.x + i), m);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    if (warp == 0) {
      m = s_red[lane];
#pragma unroll
      for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
      if (lane == 0) p.amax_part[blockIdx.x] = m;
    }
  }
  if (!grid_barrier(p.bar, &s_ok, p.wait_us)) return;

  // ---- A2 (batch-aware routing only): rank within the batch's active set ------
  if (batch_aware) {
    for (int64_t t = gw0; t < p.T; t += gw_stride)
      route_token<VPL>(p.logits, p.bias, int(t), p.E, p.k, p.score_fn, p.renorm, p.active_set, p.idx, p.w, lane);
    if (!grid_barrier(p.bar, &s_ok, p.wait_us)) return;
  }

  // ---- B: segment ranks, global scale, quantisation --------------------------
  // Warp 0 of every CTA ranks segments while the other warps quantise, so a
  // CTA with a segment does not start its share of the quantisation late
  // (the rank of a 1024-id segment is a long dependent chain).  Warp 1
  // reduces the amax partials (NVFP4); the quantising warps wait for it on a
  // named barrier that warp 0 is not part of.
  if (warp == 0) {
    for (int64_t seg = blockIdx.x; seg < p.nseg; seg += gridDim.x)
      rank_segment<ITERS>(p.idx, R, p.E, seg, s_rank_cnt, p.rank, p.seg_count, lane);
  } else {
  if (warp == 1 && !p.mx) {
    float m = 0.f;
    for (int i = lane; i < int(gridDim.x); i += 32) m = fmaxf(m, __ldcg(p.amax_part + i));
#pragma unroll
    for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
    if (lane == 0) s_red[0] = global_scale_of(m);
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kPrepThreads - 32) : "memory");
  const int64_t qtid = int64_t(blockIdx.x) * (kPrepThreads - 32) + (threadIdx.x - 32);
  const int64_t nq = int64_t(gridDim.x) * (kPrepThreads - 32);
  if (p.mx) {
    // MXFP4: one thread per 32-element block, no global scale
    const int64_t nblk = int64_t(p.T) * (p.H / 32);
    for (int64_t b = qtid; b < nblk; b += nq) {
      uint4 q[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) q[j] = __ldg(p.x + 4 * b + j);
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) a = amax8(q[j], a);
      const int X = mx_exponent(a);
      const float inv = mx_inv_step(X);
      uint32_t wd[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t v[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) word |= mx_code2(bf16_lo(v[i]), bf16_hi(v[i]), inv) << (8 * i);
        wd[j] = word;
      }
      reinterpret_cast<uint4*>(p.xq)[b] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      p.xs[b] = uint8_t(X + 127);
    }
  } else {
    const float s = s_red[0];
    if (blockIdx.x == 0 && threadIdx.x == 32) *p.gscale = s;
    // two independent blocks per iteration: their four loads are in flight together
    const int64_t nblk = int64_t(p.T) * (p.H / 16);
    int64_t b = qtid;
    for (; b + nq < nblk; b += 2 * nq) {
      const int64_t b1 = b + nq;
      const uint4 l0 = __ldg(p.x + 2 * b), h0 = __ldg(p.x + 2 * b + 1);
      const uint4 l1 = __ldg(p.x + 2 * b1), h1 = __ldg(p.x + 2 * b1 + 1);
      uint2 k0, k1;
      const uint32_t s0 = nvfp4_block16(l0, h0, s, &k0);
      const uint32_t s1 = nvfp4_block16(l1, h1, s, &k1);
      *reinterpret_cast<uint2*>(p.xq + 8 * b) = k0;
      *reinterpret_cast<uint2*>(p.xq + 8 * b1) = k1;
      p.xs[b] = uint8_t(s0);
      p.xs[b1] = uint8_t(s1);
    }
    if (b < nblk) {
      uint2 pk;
      const uint32_t sb = nvfp4_block16(__ldg(p.x + 2 * b), __ldg(p.x + 2 * b + 1), s, &pk);
      *reinterpret_cast<uint2*>(p.xq + 8 * b) = pk;
      p.xs[b] = uint8_t(sb);
    }
  }
  }
  if (!grid_barrier(p.bar, &s_ok, p.wait_us)) return;

  // ---- C: expert counts, offsets, row offsets --------------------------------
  if (blockIdx.x == 0) {
    int cnt, roff;
    scan_experts(p.seg_count, p.nseg, p.E, p.seg_base, p.counts, p.offsets, p.row_offsets, warp_tot, s_tot, &cnt,
                 &roff);
  }
  if (!grid_barrier(p.bar, &s_ok, p.wait_us)) return;

  // ---- D: padding rows, placement and gather ---------------------------------
  if (batch_aware && blockIdx.x == 0 && threadIdx.x < (p.E + 31) / 32) p.active_set[threadIdx.x] = 0u;  // read in A2 only
  for (int64_t e = gw0; e < p.E; e += gw_stride) {
    const int c = __ldcg(p.counts + e), ro = __ldcg(p.row_offsets + e);
    const int pad = (c + 127) & ~127;
    for (int r = c + lane; r < pad; r += 32) p.perm_to_flat[ro + r] = -1;
  }
  for (int64_t q = int64_t(__ldcg(p.row_offsets + p.E)) + tid; q < p.rows_cap; q += nthreads) p.perm_to_flat[q] = -1;
  // Large batches (long segments) write the rows' scales in phase E instead:
  // scattered one 4-byte word per 512-byte block, they cost ~90 us of the
  // prefill_t16384 prepare.
  constexpr bool kScalesByBlock = ITERS * 32 > 256;
  const int sfg = p.mx ? p.H / 128 : p.H / 64;  // 4-byte scale words per row
  for (int64_t f0 = gw0; f0 < R; f0 += 32 * gw_stride)
    place_rows(f0, gw_stride, R, p.idx, p.k, p.E, ITERS * 32, p.rank, p.seg_base, p.row_offsets, p.xq, p.xs, p.H, sfg,
               p.perm_to_flat, p.flat_to_perm, p.a_packed, p.a_scales, lane, !kScalesByBlock);

  // ---- E (large batches): row scales by destination block --------------------
  // One warp per (128-row block, 16 scale words): lane i gathers the words of
  // rows i, i + 32, i + 64, i + 96 of the block from the quantised token rows
  // (perm_to_flat is complete after the barrier) and writes each 512-byte
  // block's 16-byte row i, so a warp's stores are 512 contiguous bytes.
  // Padding rows keep their bytes.
  if constexpr (kScalesByBlock) {
    if (!grid_barrier(p.bar, &s_ok, p.wait_us)) return;
    const int64_t nrb = int64_t(__ldcg(p.row_offsets + p.E)) / 128;
    const int kchunks = (sfg + 15) / 16;
    // 16-byte loads of 4 words when every row start is 16-byte aligned (xs
    // itself need only be 4-byte aligned)
    const bool vec = (sfg & 3) == 0 && (reinterpret_cast<uintptr_t>(p.xs) & 15) == 0;
    const uint32_t* xs32 = reinterpret_cast<const uint32_t*>(p.xs);
    for (int64_t item = gw0; item < nrb * kchunks; item += gw_stride) {
      const int64_t rb = item / kchunks;
      const int kb0 = int(item - rb * kchunks) * 16, kb1 = min(kb0 + 16, sfg);
      int64_t src[4];
      bool all = true;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int32_t f = __ldcg(p.perm_to_flat + rb * 128 + lane + 32 * j);
        src[j] = f >= 0 ? int64_t(f / p.k) * sfg : -1;
        all = all && f >= 0;
      }
      uint8_t* dst = p.a_scales + (rb * sfg) * 512 + lane * 16;
      for (int kb = kb0; kb < kb1; kb += 4) {
        uint32_t wv[4][4];  // [row j][word kb + u]
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (src[j] < 0) continue;
          if (vec) {
            const uint4 v = __ldcg(reinterpret_cast<const uint4*>(xs32 + src[j] + kb));
            wv[j][0] = v.x, wv[j][1] = v.y, wv[j][2] = v.z, wv[j][3] = v.w;
          } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) wv[j][u] = kb + u < kb1 ? __ldcg(xs32 + src[j] + kb + u) : 0u;
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (kb + u >= kb1) break;
          uint8_t* d = dst + int64_t(kb + u) * 512;
          if (all) {
            *reinterpret_cast<uint4*>(d) = make_uint4(wv[0][u], wv[1][u], wv[2][u], wv[3][u]);
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (src[j] >= 0) *reinterpret_cast<uint32_t*>(d + 4 * j) = wv[j][u];
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// a6: finalize ("SM120 FP4 Kernel Research Campaign", section 6: token
// reordering with fused reduction; "Uncovering SM120 CUTLASS Collective
// Implementations", Context: the finalize epilogue).  Each thread owns 8
// consecutive columns of one token and sums its k expert rows in slot order.
// ---------------------------------------------------------------------------
constexpr int kFinThreads = 128;

// A CTA covers 256 consecutive 8-column groups of one token; a thread sums
// two of them (c and c + 128), so its k row indices and weights are read once
// for both and up to 16 row loads are in flight together.  The sum still
// runs in slot order for every element.
__global__ void __launch_bounds__(kFinThreads) finalize_kernel(const uint4* __restrict__ y,
                                                               const int32_t* __restrict__ f2p,
                                                               const float* __restrict__ w, int T, int k, int H,
                                                               int64_t rows_capacity, uint4* __restrict__ out) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int t = blockIdx.x;
  const int ncg = H / 8;  // 8-column groups of a row
  const int ca = blockIdx.y * (2 * kFinThreads) + threadIdx.x;
  if (ca >= ncg) return;
  const int cb = ca + kFinThreads;
  const bool has_b = cb < ncg;
  float acc[2][8] = {};
  for (int j0 = 0; j0 < k; j0 += 8) {
    const int n = min(8, k - j0);
    int64_t row[8];
    float wj[8];
    uint4 q[2][8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < n) {
        row[j] = __ldg(f2p + int64_t(t) * k + j0 + j);
        wj[j] = __ldg(w + int64_t(t) * k + j0 + j);
      }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < n && row[j] >= 0 && row[j] < rows_capacity) {
        q[0][j] = y[row[j] * ncg + ca];
        if (has_b) q[1][j] = y[row[j] * ncg + cb];
      }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j >= n) break;
      if (row[j] < 0 || row[j] >= rows_capacity) {
        if (ca == 0) atomicOr(&g_prep_flags, kFlagBadData);
        continue;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (h == 1 && !has_b) break;
        const uint32_t v[4] = {q[h][j].x, q[h][j].y, q[h][j].z, q[h][j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[h][2 * i] = fmaf(wj[j], bf16_lo(v[i]), acc[h][2 * i]);
          acc[h][2 * i + 1] = fmaf(wj[j], bf16_hi(v[i]), acc[h][2 * i + 1]);
        }
      }
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (h == 1 && !has_b) break;
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 p = __floats2bfloat162_rn(acc[h][2 * i], acc[h][2 * i + 1]);  // .x = low half
      o[i] = *reinterpret_cast<const uint32_t*>(&p);
    }
    out[int64_t(t) * ncg + (h ? cb : ca)] = make_uint4(o[0], o[1], o[2], o[3]);
  }
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
#define NVFP4MOE_ROUTE(V)                                                                                      \
  return launch_kernel(route_topk_kernel<V>, grid, block, 0, st, false, logits, bias, T, E, k, score_fn,      \
                       renormalize, static_cast<const uint32_t*>(nullptr), idx, w);
  switch (vpl <= 1 ? 1 : vpl <= 2 ? 2 : vpl <= 4 ? 4 : vpl <= 8 ? 8 : vpl <= 16 ? 16 : 32) {
    case 1: NVFP4MOE_ROUTE(1)
    case 2: NVFP4MOE_ROUTE(2)
    case 4: NVFP4MOE_ROUTE(4)
    case 8: NVFP4MOE_ROUTE(8)
    case 16: NVFP4MOE_ROUTE(16)
    default: NVFP4MOE_ROUTE(32)
  }
#undef NVFP4MOE_ROUTE
}

cudaError_t launch_route_batch_aware(const float* logits, const float* bias, int T, int E, int k, int k_primary,
                                     int score_fn, int renormalize, int32_t* idx, float* w, uint32_t* active_set,
                                     cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  cudaError_t err = cudaMemsetAsync(active_set, 0, size_t((E + 31) / 32) * sizeof(uint32_t), st);
  if (err != cudaSuccess) return err;
  const int warps = 8;
  const dim3 grid((T + warps - 1) / warps), block(warps * 32);
  const int vpl = (E + 31) / 32;
#define NVFP4MOE_ROUTE_BA(V)                                                                                   \
  err = launch_kernel(route_mark_kernel<V>, grid, block, 0, st, false, logits, bias, T, E, k_primary,         \
                      active_set);                                                                             \
  if (err != cudaSuccess) return err;                                                                          \
  return launch_kernel(route_topk_kernel<V>, grid, block, 0, st, false, logits, bias, T, E, k, score_fn,      \
                       renormalize, static_cast<const uint32_t*>(active_set), idx, w);
  switch (vpl <= 1 ? 1 : vpl <= 2 ? 2 : vpl <= 4 ? 4 : vpl <= 8 ? 8 : vpl <= 16 ? 16 : 32) {
    case 1: NVFP4MOE_ROUTE_BA(1)
    case 2: NVFP4MOE_ROUTE_BA(2)
    case 4: NVFP4MOE_ROUTE_BA(4)
    case 8: NVFP4MOE_ROUTE_BA(8)
    case 16: NVFP4MOE_ROUTE_BA(16)
    default: NVFP4MOE_ROUTE_BA(32)
  }
#undef NVFP4MOE_ROUTE_BA
}

cudaError_t launch_quantize(const void* x, int64_t rows, int64_t cols, float* global_scale, bool compute_global,
                            bool blocked, uint8_t* packed, uint8_t* scales, unsigned* amax_ws, int num_sms,
                            cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int64_t nblk = rows * (cols / 16);
  const uint4* xv = static_cast<const uint4*>(x);
  if (compute_global) {
    cudaError_t err = cudaMemsetAsync(amax_ws, 0, sizeof(unsigned), st);
    if (err != cudaSuccess) return err;
    err = launch_kernel(amax_kernel, dim3(grid_for(nblk * 2, 256, num_sms, 8)), dim3(256), 0, st, false, xv,
                        nblk * 2, amax_ws);
    if (err != cudaSuccess) return err;
  }
  const int64_t work = blocked ? ((rows + 127) / 128) * 128 * (cols / 16) : nblk;
  return launch_kernel(quantize_kernel, dim3(grid_for(work, 256, num_sms, 8)), dim3(256), 0, st, false, xv, rows,
                       cols, static_cast<const float*>(global_scale),
                       static_cast<const unsigned*>(compute_global ? amax_ws : nullptr), global_scale, packed, scales,
                       blocked ? 1 : 0);
}

cudaError_t launch_quantize_mx(const void* x, int64_t rows, int64_t cols, bool blocked, uint8_t* packed,
                               uint8_t* scales, int num_sms, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int64_t work = (blocked ? ((rows + 127) / 128) * 128 : rows) * (cols / 32);
  return launch_kernel(quantize_mx_kernel, dim3(grid_for(work, 256, num_sms, 8)), dim3(256), 0, st, false,
                       static_cast<const uint4*>(x), rows, cols, packed, scales, blocked ? 1 : 0);
}

cudaError_t launch_scales_to_blocked(const uint8_t* src, int64_t rows, int64_t cols, uint8_t* dst, int num_sms,
                                     cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const int64_t total = ((rows + 127) / 128) * 128 * (cols / 64);
  return launch_kernel(scales_to_blocked_kernel, dim3(grid_for(total, 256, num_sms, 8)), dim3(256), 0, st, false,
                       src, rows, cols, dst);
}

cudaError_t launch_permute(const int32_t* topk_idx, int T, int E, int k, const uint8_t* xq, const uint8_t* xs,
                           int H, int sf_groups, int32_t* counts, int32_t* offsets, int32_t* row_offsets,
                           int32_t* perm_to_flat, int32_t* flat_to_perm, uint8_t* a_packed, uint8_t* a_scales,
                           int64_t rows_capacity, int32_t* ws_rank, int32_t* ws_seg_count, int32_t* ws_seg_base,
                           int num_sms, cudaStream_t st) {
  const int64_t R = int64_t(T) * k;
  const int nseg = int((R + kPermuteSegment - 1) / kPermuteSegment);
  cudaError_t err;
  if (nseg > 0) {
    const size_t smem = size_t(kRankWarps) * E * sizeof(int32_t);
    if (smem > 48 * 1024) {
      err = cudaFuncSetAttribute(permute_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (err != cudaSuccess) return err;
    }
    err = launch_kernel(permute_rank_kernel, dim3((nseg + kRankWarps - 1) / kRankWarps), dim3(kRankWarps * 32), smem,
                        st, false, topk_idx, R, E, nseg, ws_rank, ws_seg_count);
    if (err != cudaSuccess) return err;
  }
  err = launch_kernel(permute_scan_kernel, dim3(1), dim3(1024), 0, st, false,
                      static_cast<const int32_t*>(ws_seg_count), nseg, E, ws_seg_base, counts, offsets, row_offsets,
                      perm_to_flat, rows_capacity);
  if (err != cudaSuccess || R == 0) return err;
  return launch_kernel(permute_place_kernel, dim3(grid_for(R * 32, 256, num_sms, 8)), dim3(256), 0, st, false,
                       topk_idx, R, k, E, static_cast<const int32_t*>(ws_rank),
                       static_cast<const int32_t*>(ws_seg_base), static_cast<const int32_t*>(row_offsets), xq, xs, H,
                       sf_groups, perm_to_flat, flat_to_perm, a_packed, a_scales);
}

PrepareLayout prepare_layout(int T, int E, int k) {
  PrepareLayout L;
  const int64_t R = int64_t(T) * k;
  L.seg_len = R <= kPrepareShortMaxRows ? 256 : 1024;
  L.nseg = (R + L.seg_len - 1) / L.seg_len;
  auto up = [](int64_t b) { return (b + 255) / 256 * 256; };
  L.bar_off = 0;        // barrier words at bytes 0 and 128, the active-expert set at 192 (<= 128 bytes)
  L.amax_off = 512;
  L.rank_off = L.amax_off + up(int64_t(kPrepareMaxGrid) * 4);
  L.seg_count_off = L.rank_off + up(R * 4);
  L.seg_base_off = L.seg_count_off + up(L.nseg * E * 4);
  L.bytes = L.seg_base_off + up(L.nseg * E * 4);
  return L;
}

namespace {

template <int VPL, int ITERS>
cudaError_t launch_prepare_impl(const PrepareParams& p, int num_sms, cudaStream_t st) {
  const size_t smem = size_t(kRankWarps) * p.E * sizeof(int32_t);
  // The grid barriers need every CTA resident: one CTA per SM must fit.
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prepare_kernel<VPL, ITERS>, kPrepThreads,
                                                                  smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  const int grid = num_sms < kPrepareMaxGrid ? num_sms : kPrepareMaxGrid;
  return launch_kernel(prepare_kernel<VPL, ITERS>, dim3(grid), dim3(kPrepThreads), smem, st, true, p);
}

}  // namespace

cudaError_t launch_prepare(const float* logits, const float* bias, const void* x, int T, int E, int k, int k_primary,
                           int H, int score_fn, int renormalize, int32_t* idx, float* w, float* gscale, uint8_t* xq,
                           uint8_t* xs, int32_t* counts, int32_t* offsets, int32_t* row_offsets, int32_t* perm_to_flat,
                           int32_t* flat_to_perm, uint8_t* a_packed, uint8_t* a_scales, int64_t rows_capacity,
                           void* ws, bool mx, int num_sms, cudaStream_t st) {
  const PrepareLayout L = prepare_layout(T, E, k);
  uint8_t* base = static_cast<uint8_t*>(ws);
  PrepareParams p;
  p.logits = logits;
  p.bias = bias;
  p.x = static_cast<const uint4*>(x);
  p.T = T;
  p.E = E;
  p.k = k;
  p.k_primary = k_primary;
  p.mx = mx ? 1 : 0;
  p.H = H;
  p.score_fn = score_fn;
  p.renorm = renormalize;
  p.nseg = int(L.nseg);
  p.idx = idx;
  p.w = w;
  p.gscale = gscale;
  p.xq = xq;
  p.xs = xs;
  p.counts = counts;
  p.offsets = offsets;
  p.row_offsets = row_offsets;
  p.perm_to_flat = perm_to_flat;
  p.flat_to_perm = flat_to_perm;
  p.a_packed = a_packed;
  p.a_scales = a_scales;
  p.rows_cap = rows_capacity;
  p.bar = reinterpret_cast<uint32_t*>(base + L.bar_off);
  p.wait_us = wait_limit_us();
  p.active_set = reinterpret_cast<uint32_t*>(base + L.bar_off + 192);
  p.amax_part = reinterpret_cast<float*>(base + L.amax_off);
  p.rank = reinterpret_cast<int32_t*>(base + L.rank_off);
  p.seg_count = reinterpret_cast<int32_t*>(base + L.seg_count_off);
  p.seg_base = reinterpret_cast<int32_t*>(base + L.seg_base_off);
  const int vpl = (E + 31) / 32;
  const int v = vpl <= 1 ? 1 : vpl <= 2 ? 2 : vpl <= 4 ? 4 : vpl <= 8 ? 8 : vpl <= 16 ? 16 : 32;
  const bool short_seg = L.seg_len == 256;
#define NVFP4MOE_PREP(V)                                                                           \
  return short_seg ? launch_prepare_impl<V, 8>(p, num_sms, st) : launch_prepare_impl<V, 32>(p, num_sms, st);
  switch (v) {
    case 1: NVFP4MOE_PREP(1)
    case 2: NVFP4MOE_PREP(2)
    case 4: NVFP4MOE_PREP(4)
    case 8: NVFP4MOE_PREP(8)
    case 16: NVFP4MOE_PREP(16)
    default: NVFP4MOE_PREP(32)
  }
#undef NVFP4MOE_PREP
}

namespace {
// Float32 accumulator of the fused finalize -> bf16 output, leaving the
// accumulator zeroed; one thread per 8 values.
__global__ void __launch_bounds__(256) finalize_f32_kernel(float4* __restrict__ acc, int64_t n8, uint4* __restrict__ out) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += int64_t(gridDim.x) * blockDim.x) {
    const float4 a = acc[2 * i], b = acc[2 * i + 1];
    const __nv_bfloat162 v0 = __floats2bfloat162_rn(a.x, a.y), v1 = __floats2bfloat162_rn(a.z, a.w);
    const __nv_bfloat162 v2 = __floats2bfloat162_rn(b.x, b.y), v3 = __floats2bfloat162_rn(b.z, b.w);
    out[i] = make_uint4(*reinterpret_cast<const uint32_t*>(&v0), *reinterpret_cast<const uint32_t*>(&v1),
                        *reinterpret_cast<const uint32_t*>(&v2), *reinterpret_cast<const uint32_t*>(&v3));
    acc[2 * i] = make_float4(0.f, 0.f, 0.f, 0.f);
    acc[2 * i + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}
}  // namespace

cudaError_t launch_finalize_f32(float* acc, int64_t n, void* out, int num_sms, cudaStream_t st) {
  const int64_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  const int64_t want = (n8 + 255) / 256, cap = int64_t(num_sms) * 8;
  return launch_kernel(finalize_f32_kernel, dim3(unsigned(want < cap ? want : cap)), dim3(256), 0, st, false,
                       reinterpret_cast<float4*>(acc), n8, static_cast<uint4*>(out));
}

cudaError_t launch_finalize(const void* y, const int32_t* flat_to_perm, const float* w, int T, int k, int H,
                            int64_t rows_capacity, void* out, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const dim3 block(kFinThreads), grid(T, (H / 8 + 2 * kFinThreads - 1) / (2 * kFinThreads));
  return launch_kernel(finalize_kernel, grid, block, 0, st, false, static_cast<const uint4*>(y), flat_to_perm, w, T,
                       k, H, rows_capacity, static_cast<uint4*>(out));
}

// ---------------------------------------------------------------------------
// Permutation with library-owned scratch, for callers that cannot allocate
// device memory at call time.  The scratch is one file-scope device array,
// present on every GPU that loads the library until the process exits.
// Host code may not use the array's name as a device address, so its
// address comes from cudaGetSymbolAddress, with the device current.
// Outside stream capture the address is looked up on every call; a call
// being captured cannot make that lookup (it may load the module) and uses
// the address the last uncaptured call on the same CUDA context found.  The
// cache is keyed on the context's process-unique id, so a device reset (a
// new primary context, possibly with the array at a new address) is never
// served a stale address.
// ---------------------------------------------------------------------------
static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocMaxRoutedRows + 2 * kNoAllocMaxSegmentExperts];

namespace {
constexpr int kScratchDevices = 64;
struct ScratchAddr {
  unsigned long long ctx_id;  // 0: none recorded
  int32_t* ptr;
};
std::mutex g_scratch_mutex;
ScratchAddr g_scratch_addr[kScratchDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Process-unique id of the calling thread's current CUDA context (the
// driver's cuCtxGetId, reached through the runtime's entry-point table).
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS && *id != 0;
}
}  // namespace

int permute_scratch_address(cudaStream_t st, int32_t** base) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) {
    set_error_detail("cudaGetDevice: %s", cudaGetErrorString(err));
    return NVFP4MOE_ERR_CUDA;
  }
  if (dev < 0 || dev >= kScratchDevices) {
    set_error_detail("device %d: the static scratch keeps addresses for devices 0..%d", dev, kScratchDevices - 1);
    return NVFP4MOE_ERR_UNSUPPORTED;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  err = cudaStreamIsCapturing(st, &cs);
  if (err != cudaSuccess) {
    set_error_detail("cudaStreamIsCapturing: %s", cudaGetErrorString(err));
    return NVFP4MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (cs == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_permute_scratch);  // device `dev` is current here
    if (err != cudaSuccess) {
      set_error_detail("cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(err));
      return NVFP4MOE_ERR_CUDA;
    }
    unsigned long long id = 0;
    g_scratch_addr[dev] = current_context_id(&id) ? ScratchAddr{id, static_cast<int32_t*>(p)} : ScratchAddr{0, nullptr};
    *base = static_cast<int32_t*>(p);
    return NVFP4MOE_OK;
  }
  unsigned long long id = 0;
  if (!current_context_id(&id) || g_scratch_addr[dev].ctx_id != id || !g_scratch_addr[dev].ptr) {
    set_error_detail(
        "moe_permute_no_alloc called during stream capture before any uncaptured call on this device's current "
        "CUDA context: make one uncaptured call first (it looks up the static scratch's device address)");
    return NVFP4MOE_ERR_UNSUPPORTED;
  }
  *base = g_scratch_addr[dev].ptr;
  return NVFP4MOE_OK;
}

cudaError_t launch_permute_static_scratch(int32_t* base, const int32_t* topk_idx, int T, int E, int k,
                                          const uint8_t* xq, const uint8_t* xs, int H, int32_t* counts,
                                          int32_t* offsets, int32_t* row_offsets, int32_t* perm_to_flat,
                                          int32_t* flat_to_perm, uint8_t* a_packed, uint8_t* a_scales,
                                          int64_t rows_capacity, int num_sms, cudaStream_t st) {
  int32_t* rank = base;
  int32_t* seg_count = rank + kNoAllocMaxRoutedRows;
  int32_t* seg_base = seg_count + kNoAllocMaxSegmentExperts;
  return launch_permute(topk_idx, T, E, k, xq, xs, H, H / 64, counts, offsets, row_offsets, perm_to_flat,
                        flat_to_perm, a_packed, a_scales, rows_capacity, rank, seg_count, seg_base, num_sms, st);
}

cudaError_t prep_read_and_clear_flags(unsigned* flags) {
  unsigned zero = 0;
  cudaError_t err = cudaMemcpyFromSymbol(flags, g_prep_flags, sizeof(unsigned));
  if (err != cudaSuccess) return err;
  return cudaMemcpyToSymbol(g_prep_flags, &zero, sizeof(unsigned));
}

}  // namespace nvfp4moe
