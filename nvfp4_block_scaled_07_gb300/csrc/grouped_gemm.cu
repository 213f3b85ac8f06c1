// Grouped NVFP4 block-scaled GEMM over experts on the 5th-generation tensor
// core (tcgen05, sm_103a), with the SwiGLU + NVFP4 requantisation epilogue of
// the gate/up projection fused in.
//
// Source of the operation: "Uncovering SM120 CUTLASS Collective
// Implementations" (Context: the grouped "array" block-scaled GEMM with a
// finalize epilogue, tile shapes limited by shared memory) and "SM120 FP4
// Kernel Research Campaign" (section 1: the block-scaled MMA with e2m1 data
// and ue4m3 scales; section 7: warp-specialised producer/consumer schedules;
// the SM100 column of its hardware table: tcgen05.mma, 256 KB of tensor
// memory, 228 KB of shared memory).  The SM120 kernels the pages study use
// mma.sync in 100 KB of shared memory; this kernel is designed for the GB300
// instead: one 128-row tcgen05 MMA per k64 step with the accumulator in
// tensor memory, operands staged by TMA through a deep mbarrier ring that
// uses the whole opt-in shared memory.
//
// Orientation ("swap AB", the default): the weight rows of one expert form
// the 128-row M side, the expert's tokens form the N side.  Decode-sized experts (a
// handful to ~64 tokens) then fill whole MMAs along M and the kernel
// streams every weight tile from HBM exactly once.  Token tiles start on
// 128-row boundaries (so every scale-factor address in tensor memory stays
// 4-column aligned) and each tile's MMA width is the power of two >= 32 that
// covers the expert's remaining rows, up to BN (128 or 256).
// Token-major orientation (TM, for experts with hundreds of rows): 128
// tokens form M and the stage's two 128-row weight tiles (gate and up, or
// two consecutive output blocks) form one N = 256 operand, so each k64 step
// is a single MMA that reads the token tile once instead of once per weight
// tile (48 instead of 64 KB of shared-memory reads per stage), and each
// epilogue thread holds one token's features in consecutive columns.
//
// Warp roles (one CTA per SM, persistent):
//   warp 0     TMA producer: weight tile(s), token tile, their scale blocks
//   warp 1     tensor-memory owner and MMA issuer (one elected lane)
//   next 4/8   epilogue: tcgen05.ld of the accumulator, scaling, SwiGLU,
//              requantisation or bf16 conversion, global stores (8 warps
//              for SwiGLU, two per lane quarter)
//   last 4     scale factors: shared memory -> tensor memory (tcgen05.st)
//              into a ring of slots the MMAs read their block scales from
// Tiles are (expert, M tile, N tile) with N innermost, so the CTAs working at
// the same time share a weight tile through L2; experts with several token
// tiles and experts with one alternate in the tile list (TileMap).
//
// Every mbarrier wait is bounded (2 s); on expiry the kernel raises a sticky
// flag, drains its own copies and MMAs, frees tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "../../include/nvfp4moe.h"
#include "common.cuh"
#include "internal.h"
#include "launch.cuh"
#include "sm103_ptx.cuh"

namespace nvfp4moe {
namespace {

__device__ unsigned g_gemm_flags = 0;

// Epilogue warps: the SwiGLU requantisation is a long dependent chain per
// token, so two warps per tensor-memory lane quarter split the token chunks
// (which also halves the registers each needs to drain its share of the
// accumulator early).  The CTA-pair bf16 epilogue also takes two warps per
// quarter, each draining half of the 256 accumulator columns in one
// tensor-memory round trip before it releases the accumulator; the other
// bf16 epilogues have one warp per quarter.
__host__ __device__ constexpr int epi_warps(bool swiglu, bool pair) { return swiglu || pair ? 8 : 4; }
// warp 0 producer, warp 1 MMA, then the epilogue warps, then 4 scale-factor
// warps.  Token-major kernels put the roles on warpgroup boundaries (warps 2
// and 3 idle) so that setmaxnreg can move registers from the producer / MMA
// and scale-factor warpgroups to the epilogue warpgroups.
__host__ __device__ constexpr int epi_first(bool wg) { return wg ? 4 : 2; }
__host__ __device__ constexpr int num_threads(bool swiglu, bool wg, bool pair = false) {
  return 32 * (epi_first(wg) + epi_warps(swiglu, pair) + 4);
}
// Registers per thread after the split (setmaxnreg) of a token-major kernel,
// by warpgroup: with two epilogue warpgroups (512 threads, 128 registers a
// thread at launch) or one (single-SM bf16: 384 threads, 168); the split
// must not need more than the launch's registers in total.
__host__ __device__ constexpr int regs_launch(bool wide) { return 65536 / (wide ? 512 : 384) / 8 * 8; }
// producer, MMA issuer and scale-ring producer (one lane each) and an idle warp
__host__ __device__ constexpr int regs_control(bool wide) { return wide ? 64 : 120; }
__host__ __device__ constexpr int regs_scale(bool wide) { return wide ? 80 : 120; }
__host__ __device__ constexpr int regs_epilogue(bool wide) { return wide ? 184 : 256; }
static_assert(num_threads(true, true) == 512 && num_threads(false, true, true) == 512 && num_threads(false, true) == 384,
              "token-major warp layouts");
static_assert(regs_control(true) + 2 * regs_epilogue(true) + regs_scale(true) <= 4 * regs_launch(true),
              "register split exceeds the launch's registers");
static_assert(regs_control(false) + regs_epilogue(false) + regs_scale(false) <= 3 * regs_launch(false),
              "register split exceeds the launch's registers");
constexpr int kBM = 128;           // MMA M (weight rows per tile)
constexpr int kBKBytes = 128;      // bytes of K per stage and row = 256 E2M1 elements
constexpr int kATile = kBM * kBKBytes;
constexpr int kTmemCols = 512;
constexpr int kAccSlotCols = 128;  // two accumulator slots at columns 0 and 128
constexpr int kSfTile = 2048;      // 4 k64 blocks x 512-byte scale blocks
constexpr int kSfColBase = 256;    // scale-factor ring: columns 256..511
constexpr int kSfRingCols = 256;
constexpr int kMaxSfSlots = 8;
constexpr int kMaxStages = 16;
// Token-major bf16 epilogue: a 2 KB shared-memory buffer per epilogue warp
// (32 rows x 64 bytes) from which a TMA store writes each chunk.
constexpr int kOutChunkBytes = 2048;
__host__ __device__ constexpr int out_stage_bytes(bool swiglu, bool tm, bool pair) {
  return tm && !swiglu ? epi_warps(swiglu, pair) * kOutChunkBytes : 0;
}
// mbarriers: full/empty per stage, acc full/empty per slot, drain, sf full/empty per ring slot,
// the tile ring, and the scale copies of each stage
// Ring of claimed tile ids (dynamic schedule): the producer claims ids from
// a launch-wide counter and passes them to the other roles.
constexpr int kTileRing = 16;
__host__ __device__ constexpr int tile_consumers(bool swiglu, bool pair) { return 1 + 4 + epi_warps(swiglu, pair); }  // MMA, SF and epilogue warps
constexpr int kNumBars = 3 * kMaxStages + 5 + 2 * kMaxSfSlots + 2 * kTileRing;
constexpr uint64_t kTimeoutNs = 2000000000ull;   // drains after an abort
constexpr uint64_t kPeerDrainNs = 30000000000ull;  // CTA 1 of a pair waiting for the pair's last MMA
constexpr unsigned kFull = 0xFFFFFFFFu;

struct Params {
  const uint8_t* w_scales;
  const uint8_t* a_scales;
  const float* a_gscale;
  const float* w_gscale;
  const int32_t* counts;
  const int32_t* row_offsets;
  const float* c_gscale;
  void* c_out;
  uint8_t* c_scales;
  int E, N, K, epi;
  int smem_bytes;   // dynamic shared memory of the launch (after 1024-byte alignment slack)
  int stage_cap;    // most pipeline stages to use (2..kMaxStages)
  uint32_t* sched;  // [0] tile counter, [32] finished CTAs (zero between launches); null: static stripes
  int w_tiled;      // weights in the tiled layout (5-D weight map coordinates below)
  int w_kc;         // 128-byte K chunks per weight row (tiled layout)
  int64_t rows_cap;
  uint32_t wait_us;  // limit of every pipeline wait (nvfp4moe_set_wait_limit_us)
  int w_policy;      // L2 policy of weight copies: 0 evict_first, 1 evict_normal, 2 evict_last
  int32_t min_rows, max_rows;  // experts outside [min_rows, max_rows) get no tiles in this launch
  const int32_t* perm_to_flat;  // NVFP4MOE_EPI_FINALIZE_F32: row -> flat id t * k + j
  const float* topk_w;          // ... and the routing weights [T, k]
  int k;
};

// Shared state of the bounded waits of one CTA: the abort flag every role
// polls and the launch's wait limit.
struct WaitCtl {
  int abort;
  uint32_t limit_us;
};

template <int BN, int NA_, bool SWIGLU>
struct Cfg {
  static constexpr int NA = NA_;  // 128-row weight tiles per stage: gate and up, or NA consecutive row blocks
  static_assert(!SWIGLU || NA == 2, "the SwiGLU epilogue pairs a gate tile with an up tile");
  static_assert(NA == 1 || NA == 2, "one or two weight tiles per stage");
  static constexpr int NSFB = BN > 128 ? 2 : 1;      // 128-row scale blocks per token tile
  static constexpr int SfCols = NA * 16 + NSFB * 16;  // tensor-memory columns of one stage's scales
  static constexpr int SfSlots = kSfRingCols / SfCols < kMaxSfSlots ? kSfRingCols / SfCols : kMaxSfSlots;
  static_assert(BN == 128 || BN == 256, "token tiles must start on 128-row scale blocks");
  static_assert(NA * BN <= 2 * kAccSlotCols, "accumulator does not fit the two slots");
  static_assert(SfCols <= 64, "scale-factor buffer overflow");
  // Bytes of one pipeline stage when the widest token tile is `wmax` rows:
  // weight tile(s), token tile, their scale blocks; a multiple of 2048, so
  // every stage and every tile in it stays 1024-byte aligned (128B swizzle).
  __host__ __device__ static constexpr int stage_bytes(int wmax) {
    return NA * kATile + wmax * kBKBytes + NA * kSfTile + (wmax > 128 ? 2 : 1) * kSfTile;
  }
};

// Control block at the start of shared memory: mbarriers, the tensor-memory
// address, flags and the per-expert tile scan; stages start after it on a
// 1024-byte boundary.
__host__ __device__ constexpr int ctrl_bytes(int E) {
  return (kNumBars * 8 + 16 + kTileRing * 4 + (4 + 4 * E) * 4 + 1023) / 1024 * 1024;
}

// Bounded wait on an mbarrier phase.  SPIN polls with test_wait, which
// never suspends the thread: the producer and the MMA issuer use it, since a
// suspended try_wait resumed measurably late after the phase completed
// (~0.2 us per stage at prefill); the other roles wait long stretches and
// use try_wait, which leaves the issue slots to the warps that work.  The
// slow path is kept out of line: a loop or call inlined between two groups
// of MMAs measurably delays the issue of the second group.
template <bool SPIN>
__device__ __forceinline__ uint32_t poll_phase(uint32_t bar, uint32_t parity) {
  return SPIN ? ptx::mbar_test_wait(bar, parity) : ptx::mbar_try_wait(bar, parity);
}

// The slow path of a wait.  The spinning form (producer and MMA issuer,
// both in the first warpgroup) stays out of line; the blocking form is
// inlined into each role, since an out-of-line function shared by
// warpgroups with different register budgets (setmaxnreg) cannot be
// register-allocated.
template <bool SPIN>
__device__ __forceinline__ bool wait_phase_loop(uint32_t bar, uint32_t parity, volatile WaitCtl* wctl) {
  const uint64_t t0 = ptx::globaltimer_ns();
  const uint64_t limit = uint64_t(wctl->limit_us) * 1000u;
  for (uint32_t i = 0;; ++i) {
    if (poll_phase<SPIN>(bar, parity)) return true;
    if ((i & 255u) == 255u) {
      if (wctl->abort) return false;
      if (ptx::globaltimer_ns() - t0 > limit) {
        wctl->abort = 1;
        atomicOr(&g_gemm_flags, kFlagTimeout);
        return false;
      }
    }
  }
}
__device__ __noinline__ bool wait_phase_slow_spin(uint32_t bar, uint32_t parity, volatile WaitCtl* wctl) {
  return wait_phase_loop<true>(bar, parity, wctl);
}

template <bool SPIN = false>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile WaitCtl* abort_flag) {
  if (poll_phase<SPIN>(bar, parity)) return true;
  if constexpr (SPIN) return wait_phase_slow_spin(bar, parity, abort_flag);
  else return wait_phase_loop<false>(bar, parity, abort_flag);
}

// Short bounded wait used only while draining after an abort.
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > kTimeoutNs) return;
  }
}

// Tile t -> expert e, M tile mb, N tile nb and the tile's MMA width w: the
// smallest power of two >= 32 covering the rows left, capped at BN.
// The launch's tile list.  Experts with two or more token tiles (their
// weight tiles are re-read from L2 by every token tile: compute-heavy) form
// class A, experts with one (each weight tile streamed from HBM once) class
// B; each class lists its experts in index order and an expert's tiles M
// tile by M tile, N (token) tile innermost.  Tile t alternates between the
// classes (even t from A, odd from B) until the smaller one runs out, so on
// a skewed batch the compute-heavy and the HBM-bound tiles run side by side
// instead of in two phases; a batch of one class keeps plain expert order.
struct TileMap {
  const int* hdr;   // [0] class-A tiles, [1] class-B tiles, [2] class-A experts, [3] class-B experts
  const int* pre;   // per position: first tile of the expert within its class
  const int* expt;  // per position: expert id (class A first, then class B)
  const int* count; // per expert: rows
};

// Tile t -> expert e, M tile mb, N tile nb and the tile's MMA width w: the
// smallest power of two >= 32 covering the rows left, capped at BN.
__device__ __forceinline__ void decode_tile(int t, const TileMap& m, int BN, int& e, int& mb, int& nb, int& w) {
  const int tA = m.hdr[0], tB = m.hdr[1], nA = m.hdr[2], nB = m.hdr[3];
  const int both = min(tA, tB);
  int cls, local;
  if (t < 2 * both) {
    cls = t & 1;
    local = t >> 1;
  } else {
    cls = tA > tB ? 0 : 1;
    local = t - both;
  }
  int lo = cls ? nA : 0, hi = cls ? nA + nB - 1 : nA - 1;  // last position whose first tile <= local
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (m.pre[mid] <= local) lo = mid;
    else hi = mid - 1;
  }
  e = m.expt[lo];
  const int ntn = (m.count[e] + BN - 1) / BN;
  const int in = local - m.pre[lo];
  mb = in / ntn;
  nb = in - mb * ntn;
  const int rem = m.count[e] - nb * BN;
  w = 32;
  while (w < rem && w < BN) w <<= 1;
}

// Accumulator slots of one tile: a tile whose accumulator fits 128 columns
// takes the next slot (alternating), a wider one takes both, starting at 0.
// Producer (MMA) and consumer (epilogue) walk the same sequence.
struct SlotSeq {
  uint32_t use0 = 0u, use1 = 0u;  // completed uses per slot (phase parity source)
  int next = 0;
  __device__ __forceinline__ uint32_t parity(int slot) const { return (slot ? use1 : use0) & 1u; }
  __device__ __forceinline__ void pick(int cols, int& s0, int& s1) {
    if (cols <= kAccSlotCols) {
      s0 = next;
      s1 = -1;
      next ^= 1;
    } else {
      s0 = 0;
      s1 = 1;
      next = 0;
    }
  }
  __device__ __forceinline__ void done(int s0, int s1) {
    if (s0 == 0 || s1 == 0) ++use0;
    if (s0 == 1 || s1 == 1) ++use1;
  }
};

// NVFP4 requantisation of a 32-token x 32-feature chunk of the SwiGLU output
// held one feature per lane (lane = feature f0 + lane, h[t] = token t), with
// the rounding rules of the quantiser kernel.  The two 16-feature blocks of
// the warp (lanes 0-15 and 16-31) need one scale per token each: a
// reduce-scatter butterfly over the 16 lanes of a block leaves the block
// amax of tokens 2l and 2l+1 in lane l, which computes their scales once and
// shares the dequantisation step back with one shuffle per element.
__device__ __forceinline__ void requant_swiglu_chunk(const float (&h)[32], int lane, float s_h, int64_t row0,
                                                     int nvalid, int f, int n_out, uint8_t* out_codes,
                                                     uint8_t* out_scales) {
  float a[16];
  {
    const bool hi = lane & 8;
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const float keep = hi ? fabsf(h[t + 16]) : fabsf(h[t]);
      const float give = hi ? fabsf(h[t]) : fabsf(h[t + 16]);
      a[t] = fmaxf(keep, __shfl_xor_sync(kFull, give, 8));
    }
  }
#pragma unroll
  for (int step = 4; step >= 1; step >>= 1) {   // 16 -> 8 -> 4 -> 2 tokens per lane
    const bool hi = lane & step;
    const int half = 2 * step;                   // tokens kept after this step
#pragma unroll
    for (int t = 0; t < half; ++t) {
      const float keep = hi ? a[t + half] : a[t];
      const float give = hi ? a[t] : a[t + half];
      a[t] = fmaxf(keep, __shfl_xor_sync(kFull, give, step));
    }
  }
  // lane l of a block now holds the amax of tokens 2(l % 16) and 2(l % 16) + 1
  const int t0 = 2 * (lane & 15);
  uint32_t sb[2];
  float inv[2];  // 1 / step, 0 for a zero step (whose codes are all 0)
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    sb[k] = f32_to_ue4m3((a[k] / kE2M1Max) / s_h);
    const float d = ue4m3_to_f32(sb[k]) * s_h;
    inv[k] = d != 0.0f ? 1.0f / d : 0.0f;
  }
  const int fb = (f & ~31) + (lane & 16);        // first feature of this lane's block
#pragma unroll
  for (int k = 0; k < 2; ++k)
    if (t0 + k < nvalid)
      out_scales[blocked_sf_offset(row0 + t0 + k, fb >> 6, n_out / 64) + ((fb >> 4) & 3)] = uint8_t(sb[k]);
  // Codes: q = h * (1 / step) (within an ulp of h / step; the SwiGLU value is
  // an accumulator result, so its codes are compared with the oracle's
  // statistically) and the hardware conversion of the even/odd feature pair
  // held by lanes 2i and 2i+1; four pairs make the 32-bit word of 8 features.
  uint8_t* row_ptr = out_codes + row0 * (n_out / 2) + (f & ~7) / 2;
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    const float it = __shfl_sync(kFull, inv[t & 1], (lane & 16) + (t >> 1));
    const float q = it != 0.0f ? h[t] * it : 0.0f;
    const float qn = __shfl_xor_sync(kFull, q, 1);
    uint32_t word = (lane & 1) ? 0u : e2m1x2(q, qn) << (8 * ((lane & 7) >> 1));
    word |= __shfl_xor_sync(kFull, word, 2);
    word |= __shfl_xor_sync(kFull, word, 4);
    if ((lane & 7) == 0 && t < nvalid) *reinterpret_cast<uint32_t*>(row_ptr + int64_t(t) * (n_out / 2)) = word;
  }
}

// MXFP4 requantisation of a 32-token x 32-feature chunk of the SwiGLU output
// (lane = feature f0 + lane with f0 % 32 == 0, h[t] = token t): the warp's
// 32 features are one MX block per token.  A reduce-scatter butterfly over
// the 32 lanes leaves token l's block amax in lane l, which derives the
// token's shared exponent and scale byte; every element then takes its
// token's 2^-X from lane t.
__device__ __forceinline__ void requant_swiglu_chunk_mx(const float (&h)[32], int lane, int64_t row0, int nvalid,
                                                        int f, int n_out, uint8_t* out_codes, uint8_t* out_scales) {
  float a[32];
#pragma unroll
  for (int t = 0; t < 32; ++t) a[t] = fabsf(h[t]);
#pragma unroll
  for (int step = 16; step >= 1; step >>= 1) {   // 32 -> 16 -> ... -> 1 token per lane
    const bool hi = lane & step;
#pragma unroll
    for (int t = 0; t < step; ++t) {
      const float keep = hi ? a[t + step] : a[t];
      const float give = hi ? a[t] : a[t + step];
      a[t] = fmaxf(keep, __shfl_xor_sync(kFull, give, step));
    }
  }
  const int X = mx_exponent(a[0]);               // token `lane`
  const float inv = mx_inv_step(X);
  const int f0 = f & ~31;
  if (lane < nvalid)
    out_scales[blocked_sf_offset(row0 + lane, f0 >> 7, n_out / 128) + ((f0 >> 5) & 3)] = uint8_t(X + 127);
  uint8_t* row_ptr = out_codes + row0 * (n_out / 2) + (f & ~7) / 2;
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    const float q = h[t] * __shfl_sync(kFull, inv, t);  // exact: 2^-X scaling
    const float qn = __shfl_xor_sync(kFull, q, 1);
    uint32_t word = (lane & 1) ? 0u : e2m1x2(q, qn) << (8 * ((lane & 7) >> 1));
    word |= __shfl_xor_sync(kFull, word, 2);
    word |= __shfl_xor_sync(kFull, word, 4);
    if ((lane & 7) == 0 && t < nvalid) *reinterpret_cast<uint32_t*>(row_ptr + int64_t(t) * (n_out / 2)) = word;
  }
}

// Token-major epilogue: NVFP4 requantisation of 32 consecutive features of
// one token row held by one thread (h[i] = feature f0 + i as float bits,
// f0 % 32 == 0), two 16-feature blocks, with the rounding steps of
// requant_swiglu_chunk.  The 16 code bytes are one 16-byte store.
__device__ __forceinline__ void requant_row32(const uint32_t (&h)[32], float s_h, int64_t row, int f0, int n_out,
                                              uint8_t* out_codes, uint8_t* out_scales) {
  uint32_t wd[4];
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(__uint_as_float(h[16 * b + i])));
    const uint32_t sb = f32_to_ue4m3((a / kE2M1Max) / s_h);
    const float d = ue4m3_to_f32(sb) * s_h;
    const float inv = d != 0.0f ? 1.0f / d : 0.0f;
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      uint32_t word = 0;
#pragma unroll
      for (int pr = 0; pr < 4; ++pr) {
        const int i = 16 * b + 8 * w + 2 * pr;
        const float q0 = inv != 0.0f ? __uint_as_float(h[i]) * inv : 0.0f;
        const float q1 = inv != 0.0f ? __uint_as_float(h[i + 1]) * inv : 0.0f;
        word |= e2m1x2(q0, q1) << (8 * pr);
      }
      wd[2 * b + w] = word;
    }
    const int fb = f0 + 16 * b;
    out_scales[blocked_sf_offset(row, fb >> 6, n_out / 64) + ((fb >> 4) & 3)] = uint8_t(sb);
  }
  *reinterpret_cast<uint4*>(out_codes + row * (n_out / 2) + f0 / 2) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
}

// MXFP4 counterpart: the 32 features are one MX block (requant_swiglu_chunk_mx).
__device__ __forceinline__ void requant_row32_mx(const uint32_t (&h)[32], int64_t row, int f0, int n_out,
                                                 uint8_t* out_codes, uint8_t* out_scales) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(__uint_as_float(h[i])));
  const int X = mx_exponent(a);
  const float inv = mx_inv_step(X);
  uint32_t wd[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
      const int i = 8 * w + 2 * pr;
      word |= e2m1x2(__uint_as_float(h[i]) * inv, __uint_as_float(h[i + 1]) * inv) << (8 * pr);
    }
    wd[w] = word;
  }
  out_scales[blocked_sf_offset(row, f0 >> 7, n_out / 128) + ((f0 >> 5) & 3)] = uint8_t(X + 127);
  *reinterpret_cast<uint4*>(out_codes + row * (n_out / 2) + f0 / 2) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
}

template <int BN, int NA, bool SWIGLU, bool MX, bool TM, bool PAIR = false, bool FIN = false>
__global__ void __launch_bounds__(num_threads(SWIGLU, TM, PAIR), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_c, const __grid_constant__ CUtensorMap tmap_sf,
                        const __grid_constant__ CUtensorMap tmap_asf, const Params p) {
  using C = Cfg<BN, NA, SWIGLU>;
  static_assert(!TM || (BN == 128 && NA == 2), "token-major tiles: 128 tokens x two 128-row weight tiles");
  static_assert(!PAIR || TM, "CTA pairs run token-major tiles");
  // FIN: the bf16 epilogue adds each row, times its routing weight, into its
  // token's float32 row (NVFP4MOE_EPI_FINALIZE_F32); its own instantiation,
  // so the plain bf16 kernels keep their register allocation.
  static_assert(!FIN || (!SWIGLU && !MX), "the fused finalize follows the NVFP4 down projection");
  // CTA pair (cluster of two, cta_group::2 MMAs): a tile is 256 tokens, 128
  // in each CTA, against the stage's two weight tiles, one in each CTA's
  // shared memory; CTA 0 of the pair issues the MMAs for both.
  constexpr int TB = PAIR ? 2 * kBM : BN;      // token rows per tile
  constexpr int NW = PAIR ? 1 : C::NA;         // weight tiles in this CTA's stage
  const uint32_t crank = PAIR ? ptx::cluster_ctarank() : 0u;
  uint32_t* const sched = PAIR ? nullptr : p.sched;  // pairs run static stripes
  // Token-major kernels tie each stage's scale-factor slot in tensor memory
  // to its shared-memory stage, and the scale-factor warps arrive on the
  // stage's full barrier: the MMA thread then waits on one barrier and
  // commits once per stage.  Its MMAs queue only about one deep, so every
  // handshake between stages leaves the tensor core idle.
  constexpr bool kTied = TM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  int* s_wmax = reinterpret_cast<int*>(tmem_slot + 1);
  volatile WaitCtl* abort_flag = reinterpret_cast<volatile WaitCtl*>(tmem_slot + 2);
  volatile int* s_tq = reinterpret_cast<volatile int*>(tmem_slot + 4);   // claimed tile ids
  int* s_map = reinterpret_cast<int*>(tmem_slot + 4 + kTileRing);  // TileMap header
  int* s_pre = s_map + 4;
  int* s_expt = s_pre + p.E;
  int* s_count = s_expt + p.E;
  int* s_rowoff = s_count + p.E;
  const TileMap tiles{s_map, s_pre, s_expt, s_count};
  const int ctrl = ctrl_bytes(p.E);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = ptx::smem_u32(bars);
  // full[s] = bar0 + 8s, empty[s] = bar0 + 8(kMaxStages+s), acc_full[b], acc_empty[b], drain
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (uint32_t(kMaxStages) + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * uint32_t(2 * kMaxStages + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * uint32_t(2 * kMaxStages + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * uint32_t(2 * kMaxStages + 4);
  auto sff_bar = [&](uint32_t r) { return bar0 + 8u * (uint32_t(2 * kMaxStages + 5) + r); };
  auto sfe_bar = [&](uint32_t r) { return bar0 + 8u * (uint32_t(2 * kMaxStages + 5 + kMaxSfSlots) + r); };
  auto tqf_bar = [&](uint32_t q) { return bar0 + 8u * (uint32_t(2 * kMaxStages + 5 + 2 * kMaxSfSlots) + q); };
  auto tqe_bar = [&](uint32_t q) {
    return bar0 + 8u * (uint32_t(2 * kMaxStages + 5 + 2 * kMaxSfSlots + kTileRing) + q);
  };
  // the scale blocks of stage s (token-major: of scale ring slot s), copied ahead of its operands
  auto sfc_bar = [&](uint32_t s) {
    return bar0 + 8u * (uint32_t(2 * kMaxStages + 5 + 2 * kMaxSfSlots + 2 * kTileRing) + s);
  };

  const int MT = SWIGLU ? p.N / 2 / kBM : p.N / (kBM * NA);  // M tiles per expert
  // Single-CTA token-major kernels keep the scale blocks out of the operand
  // stages, in a deeper shared-memory ring of their own that a second
  // producer thread (lane 0 of warp 2) fills ahead of the operands, and the
  // scale-factor warps move a slot into tensor memory as soon as the MMAs of
  // the stage's previous use are done (measured on GB300: skewed_t2048 0.711
  // -> 0.676 ms per layer).  Pair tiles keep them in the stage: with the
  // ring, their copy pipeline alone ran faster (gate/up without MMAs 2.38 ->
  // 1.87 ms at prefill) but the whole kernel slower (2.63 -> 2.76 ms).
  constexpr bool kRing = TM && !PAIR;
  constexpr int nprod = kRing ? 2 : 1;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      // the producer's expect_tx, plus (tied scale slots) one arrival per scale-factor warp of each CTA
      ptx::mbar_init(full_bar(s), kTied ? 1 + (PAIR ? 8 : 4) : 1);
      ptx::mbar_init(empty_bar(s), 1);
      ptx::mbar_init(sfc_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(accf_bar(b), 1);
      ptx::mbar_init(acce_bar(b), (PAIR ? 2 : 1) * epi_warps(SWIGLU, PAIR));  // both CTAs' epilogues drain it
    }
    ptx::mbar_init(drain_bar, 1);
    for (int r = 0; r < kMaxSfSlots; ++r) {
      ptx::mbar_init(sff_bar(r), PAIR ? 8 : 4);  // one arrival per scale-factor warp (of both CTAs)
      // MMA completion; token-major: the scale ring slot read by this CTA's 4 scale-factor warps
      ptx::mbar_init(sfe_bar(r), kRing ? 4 : 1);
    }
    for (int q = 0; q < kTileRing; ++q) {
      ptx::mbar_init(tqf_bar(q), 1);
      ptx::mbar_init(tqe_bar(q), tile_consumers(SWIGLU, PAIR) + nprod - 1);  // (+ the scale-copy producer)
    }
    abort_flag->abort = 0;
    abort_flag->limit_us = p.wait_us;
    ptx::fence_barrier_init();
    ptx::prefetch_tmap(&tmap_w);
    ptx::prefetch_tmap(&tmap_a);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  // Everything above touches only this CTA's own resources; from here on the
  // kernel reads the previous kernel's outputs (counts, operands, scales).
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  if (warp == 2) {
    // The tile list (TileMap): per-expert token tiles, the class of each
    // expert, each class's positions and tile prefixes, and the widest token
    // tile of the launch; experts whose rows would leave the padded buffers
    // are skipped and flagged.
    const int per = (p.E + 31) / 32;
    const int beg = min(lane * per, p.E), end = min(beg + per, p.E);
    int nA = 0, tA = 0, nB = 0, tB = 0, wmax = 32;
    for (int e = beg; e < end; ++e) {
      int c = p.counts[e];
      const int ro = p.row_offsets[e];
      const int64_t padded = (int64_t(c) + 127) / 128 * 128;
      if (c < 0 || ro < 0 || (ro & 127) || int64_t(ro) + padded > p.rows_cap) {
        atomicOr(&g_gemm_flags, kFlagBadData);
        c = 0;
      }
      if (c < p.min_rows || c >= p.max_rows) c = 0;  // another launch covers this expert
      s_count[e] = c;
      s_rowoff[e] = ro;
      const int ntn = (c + TB - 1) / TB;
      if (ntn >= 2) ++nA, tA += MT * ntn;
      else if (ntn == 1) ++nB, tB += MT;
      int w = 32;
      while (w < c && w < BN) w <<= 1;
      if (c > 0) wmax = max(wmax, w);
    }
    int inA = nA, itA = tA, inB = nB, itB = tB;  // inclusive scans over the lanes
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int a = __shfl_up_sync(kFull, inA, off), b = __shfl_up_sync(kFull, itA, off);
      const int c = __shfl_up_sync(kFull, inB, off), d = __shfl_up_sync(kFull, itB, off);
      if (lane >= off) inA += a, itA += b, inB += c, itB += d;
      wmax = max(wmax, __shfl_xor_sync(kFull, wmax, off));
    }
    const int expertsA = __shfl_sync(kFull, inA, 31);
    int posA = inA - nA, preA = itA - tA, posB = expertsA + inB - nB, preB = itB - tB;
    for (int e = beg; e < end; ++e) {
      const int ntn = (s_count[e] + TB - 1) / TB;
      if (ntn >= 2) {
        s_expt[posA] = e, s_pre[posA] = preA;
        ++posA, preA += MT * ntn;
      } else if (ntn == 1) {
        s_expt[posB] = e, s_pre[posB] = preB;
        ++posB, preB += MT;
      }
    }
    if (lane == 31) {
      s_map[0] = itA, s_map[1] = itB, s_map[2] = inA, s_map[3] = inB;
      *s_wmax = wmax;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  // A pair's CTAs signal each other's barriers from here on: both must have
  // initialised theirs.
  if constexpr (PAIR) ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = s_map[0] + s_map[1];
  const int kblocks = p.K / 64;
  const int nkt = (kblocks + 3) / 4;
  const int sf_k = MX ? p.K / 128 : kblocks;     // 512-byte scale blocks along K per 128 rows
  const int sf_per_kt = MX ? 2 : 4;              // of them per 256-element K stage
  // Stage geometry for this launch: as many stages as fit once the token
  // slot is sized for the widest tile actually present.
  const int wmax = TM ? kBM : *s_wmax;  // token-major: every token tile is 128 rows
  // With a scale ring: operand stages hold the weight and token tiles only,
  // and each slot of the ring the weight tiles' and the token tile's scale
  // blocks of one K stage (sf_slot bytes); the stages take what the ring's
  // two slots leave, the ring what the stages leave (at most kMaxSfSlots).
  // Otherwise the scale blocks ride in the stage.
  const int sf_slot = (C::NA + (wmax > 128 ? 2 : 1)) * kSfTile;
  const int stage = NW * kATile + wmax * kBKBytes + (kRing ? 0 : sf_slot);
  const int off_b = NW * kATile;
  const int off_sfa = kRing ? 0 : off_b + wmax * kBKBytes;  // in the stage, or in the ring slot
  const int off_sfb = off_sfa + C::NA * kSfTile;
  const int room = p.smem_bytes - ctrl - out_stage_bytes(SWIGLU, TM, PAIR);
  const int S = min(kTied ? C::SfSlots : kMaxStages, min(p.stage_cap, (room - (kRing ? 2 * sf_slot : 0)) / stage));
  const int R = kRing ? min(kMaxSfSlots, (room - S * stage) / sf_slot) : 0;  // scale ring slots
  const uint32_t smem_base = ptx::smem_u32(smem) + uint32_t(ctrl);
  const uint32_t sf_ring = smem_base + uint32_t(S * stage);
  const uint32_t out_base = sf_ring + uint32_t(R * sf_slot);  // token-major bf16 chunk buffers

  // The i-th tile of this CTA: the static stripe blockIdx.x + i * gridDim.x,
  // or (dynamic schedule) the i-th id the producer claimed, read from the
  // ring; lane 0 of a warp role reads it and releases the slot.  Returns -1
  // if the wait was abandoned.
  auto next_tile = [&](uint32_t i, bool whole_warp) -> int {
    if (PAIR) return int((blockIdx.x >> 1) + i * (gridDim.x >> 1));
    if (!sched) return int(blockIdx.x + i * gridDim.x);
    const uint32_t q = i % uint32_t(kTileRing), ph = (i / uint32_t(kTileRing)) & 1u;
    int t = -1;
    if (!whole_warp || lane == 0) {
      if (whole_warp ? wait_phase(tqf_bar(q), ph, abort_flag) : wait_phase<true>(tqf_bar(q), ph, abort_flag)) {
        t = s_tq[q];
        ptx::mbar_arrive(tqe_bar(q));
      }
    }
    if (whole_warp) t = __shfl_sync(kFull, t, 0);
    return t;
  };

  // ---- warp roles (bodies as lambdas; dispatched below) ----
  auto role_producer = [&](int who) {
    // ---------------- TMA producer ----------------
    // who: 0 (lane 0 of warp 0) copies the operand stages, and their scale
    // blocks unless the kernel has a scale ring; 1 (lane 0 of warp 2) fills
    // the scale ring.
    // weights stream through once at decode; token-major (many rows per
    // expert) re-reads each weight tile for every token tile
    const uint64_t pol_w = p.w_policy == 2   ? ptx::policy_evict_last()
                           : p.w_policy == 1 ? ptx::policy_evict_normal()
                                             : ptx::policy_evict_first();
    const uint64_t pol_a = ptx::policy_evict_last();   // token tiles are re-read by every M tile
    uint32_t it = 0;          // stages issued (for the drain after an abort)
    uint32_t s = 0, ph = 0;   // ring position of stage it and its phase parity (scale ring: who 1)
    const uint32_t ring = who == 0 ? uint32_t(S) : uint32_t(R);
    bool ok = true;
    // Dynamic schedule: producer 0 claims the next id one tile ahead, so the
    // atomic's latency overlaps the current tile's copies; the scale ring's
    // producer reads the ids from the ring like the other roles.
    int next = who != 0 ? 0 : sched ? int(atomicAdd(sched, 1u)) : int(PAIR ? blockIdx.x >> 1 : blockIdx.x);
    for (uint32_t i = 0; ok; ++i) {
      int t;
      if (who == 0) {
        t = next;
        if (sched) {
          const uint32_t q = i % uint32_t(kTileRing), ph = (i / uint32_t(kTileRing)) & 1u;
          if (!wait_phase<true>(tqe_bar(q), ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          s_tq[q] = t;
          ptx::mbar_arrive(tqf_bar(q));
        }
        if (t >= total) break;
        next = sched ? int(atomicAdd(sched, 1u)) : t + int(PAIR ? gridDim.x >> 1 : gridDim.x);
      } else {
        t = next_tile(i, false);
        if (t < 0) ok = false;
        if (t < 0 || t >= total) break;
      }
      int e, mb, nb, w;
      decode_tile(t, tiles, TB, e, mb, nb, w);
      if constexpr (TM) w = kBM;
      const int arow = s_rowoff[e] + nb * TB + int(crank) * kBM;  // this CTA's token rows
      const int sfb_chunks = w > 128 ? 2 : 1;
      // weight tiles: gate/up pair rows f and I + f; otherwise NA consecutive 128-row blocks
      // The stage's NA weight tiles are one box of the 5-D weight map (see
      // encode_weight_map): coordinates (kt * wdx, wc1, wc2 + kt * wdz, wc3, wc4).
      const int wdx = p.w_tiled ? 0 : kBKBytes, wdz = p.w_tiled ? 1 : 0;
      const int wblk = SWIGLU ? mb : e * (p.N / kBM) + mb * NA;  // first 128-row block of the tile
      const int wc1 = (!p.w_tiled && SWIGLU) ? mb * kBM : 0;
      // a pair's CTA loads one of the stage's two weight tiles: the up tile
      // (or the second output block) in CTA 1
      const int wc2 = p.w_tiled ? 0 : (SWIGLU ? 2 * e : wblk) + int(crank);
      const int wc3 = p.w_tiled ? wblk + (SWIGLU ? 0 : int(crank)) : 0;
      const int wc4 = (p.w_tiled && SWIGLU) ? 2 * e + int(crank) : 0;
      // The weight tiles' scale blocks of a stage are one box of the scale map
      // (see encode_weight_scale_map) at (64 sf_per_kt kt, sc1, sc2): a stage
      // advances sf_per_kt 512-byte blocks; the token tile's start at asf.
      const int sc1 = SWIGLU ? mb : e * (p.N / kBM) + mb * NA, sc2 = SWIGLU ? 2 * e : 0;
      const uint8_t* asf = p.a_scales + size_t(arow / kBM) * sf_k * 512;
      const uint32_t op_bytes = uint32_t(NW * kATile + w * kBKBytes);
      for (int kt = 0; kt < nkt; ++kt, ++it) {
        if (who == 1) {
          // Token-major scale ring: slot s is free once this CTA's
          // scale-factor warps have read it into registers.  This thread
          // runs ahead of the operands and waits with try_wait: spinning
          // here takes issue slots from the epilogue warps on its SM
          // sub-partition.
          if (!wait_phase(sfe_bar(s), ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t slot = sf_ring + s * uint32_t(sf_slot);
          ptx::mbar_arrive_expect_tx(sfc_bar(s), uint32_t(sf_slot));
          ptx::tma_load_3d(slot, &tmap_sf, sfc_bar(s), kt * sf_per_kt * 64, sc1, sc2, pol_w);
          ptx::tma_load_3d(slot + C::NA * kSfTile, &tmap_asf, sfc_bar(s), kt * sf_per_kt * 64, arow / kBM, 0, pol_a);
          if (++s == ring) s = 0, ph ^= 1u;
          continue;
        }
        if (!wait_phase<true>(empty_bar(s), ph ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t st = smem_base + s * uint32_t(stage);
        // The scale blocks first, on their own barrier: the scale-factor
        // warps move them into tensor memory while the operands are in flight.
        const int nkb = min(4, kblocks - 4 * kt);
        // 512-byte scale blocks of this stage per 128 rows: one per k64 step
        // (NVFP4) or per k128 step (MXFP4, K % 128 == 0)
        const uint32_t sf_bytes = uint32_t((MX ? nkb / 2 : nkb) * 512);
        const size_t sf_off = size_t(kt) * (sf_per_kt * 512);
        // scale boxes are always full (bytes past the scales read as zero)
        if constexpr (kRing) {
          // (the scale ring's producer copies them)
        } else if constexpr (BN == 128) {  // one 128-row token chunk: its scales are a box of the token scale map
          ptx::mbar_arrive_expect_tx(sfc_bar(s), uint32_t((C::NA + 1) * kSfTile));
          ptx::tma_load_3d(st + off_sfa, &tmap_sf, sfc_bar(s), kt * sf_per_kt * 64, sc1, sc2, pol_w);
          ptx::tma_load_3d(st + off_sfb, &tmap_asf, sfc_bar(s), kt * sf_per_kt * 64, arow / kBM, 0, pol_a);
        } else {
          ptx::mbar_arrive_expect_tx(sfc_bar(s), uint32_t(C::NA * kSfTile) + sfb_chunks * sf_bytes);
          ptx::tma_load_3d(st + off_sfa, &tmap_sf, sfc_bar(s), kt * sf_per_kt * 64, sc1, sc2, pol_w);
          for (int c = 0; c < sfb_chunks; ++c)
            ptx::bulk_load(st + off_sfb + c * kSfTile, asf + size_t(c) * sf_k * 512 + sf_off, sf_bytes, sfc_bar(s),
                           pol_a);
        }
        if constexpr (PAIR) {
          // Both CTAs' operands complete on CTA 0's full barrier, which
          // expects the bytes of both.
          const uint32_t fb = ptx::mapa(full_bar(s), 0);
          if (crank == 0) ptx::mbar_arrive_expect_tx(full_bar(s), 2 * op_bytes);
          ptx::tma_load_5d_pair(st, &tmap_w, fb, kt * wdx, wc1, wc2 + kt * wdz, wc3, wc4, pol_w);
          ptx::tma_load_2d_pair(st + off_b, &tmap_a, fb, kt * kBKBytes, arow, pol_a);
        } else {
          ptx::mbar_arrive_expect_tx(full_bar(s), op_bytes);
          ptx::tma_load_5d(st, &tmap_w, full_bar(s), kt * wdx, wc1, wc2 + kt * wdz, wc3, wc4, pol_w);
          if constexpr (TM) {  // a 128-row token tile: one box (the map's box is 128 rows here)
            ptx::tma_load_2d(st + off_b, &tmap_a, full_bar(s), kt * kBKBytes, arow, pol_a);
          } else {
            for (int r = 0; r < w; r += 32)  // the token tile in 32-row boxes
              ptx::tma_load_2d(st + off_b + r * kBKBytes, &tmap_a, full_bar(s), kt * kBKBytes, arow + r, pol_a);
          }
        }
        if (++s == uint32_t(S)) s = 0, ph ^= 1u;
      }
    }
    if (!ok) {
      // Let every copy this thread issued land before the CTA can exit: the
      // scale ring's and (not token-major) the stages' own barriers complete
      // once the bytes are in.  A token-major stage's full barrier also waits
      // for the scale-factor warps, and a pair's CTA 1 copies complete on CTA
      // 0's barriers, which CTA 1 cannot wait on: there, any copy still in
      // flight gets 1 ms to land.
      const uint32_t first = it > ring ? it - ring : 0u;
      for (uint32_t i = first; i < it; ++i) {
        if (TM && who == 0) break;
        drain_phase(sfc_bar(i % ring), (i / ring) & 1u);
        if (!TM && crank == 0) drain_phase(full_bar(i % ring), (i / ring) & 1u);
      }
      if (TM && who == 0) {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::globaltimer_ns() - t0 < 1000000ull) {
        }
      }
    }
  };
  auto role_peer_wait = [&]() {
    // CTA 1 of a pair issues no MMAs; its tensor memory is freed once CTA 0's
    // last MMA (which writes it) has completed.  CTA 0 signals that at the end
    // of its MMA role, also after an abort, so this wait spans the whole
    // kernel: its limit is kPeerDrainNs instead of the per-stage limit.
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(drain_bar, 0)) {
      if (ptx::globaltimer_ns() - t0 > kPeerDrainNs) {
        atomicOr(&g_gemm_flags, kFlagTimeout);
        break;
      }
    }
  };
  auto role_mma = [&]() {
    // ---------------- MMA issuer ----------------
    // The tensor core queues about one MMA, so whatever this thread does
    // between two groups of MMAs (waits, commits, address arithmetic) leaves
    // it idle.  The loop therefore keeps that work small: ring positions are
    // wrap-around counters, both barriers of a stage are polled once with the
    // bounded slow path out of line, and (default orientation) two K stages
    // of a tile are waited for together and issued back to back (a probe on
    // one SM: 904 -> 709 cycles per 8 MMAs against 518 for MMAs alone).
    uint32_t s = 0, ph = 0;  // pipeline stage and its phase parity
    uint32_t r = 0, rph = 0;  // scale-factor ring slot and its parity
    SlotSeq slots;
    bool ok = true;
    // a pair's MMAs signal the barrier at the same offset in both CTAs
    auto commit = [](uint32_t bar) {
      if constexpr (PAIR) ptx::tc_commit_pair(bar);
      else ptx::tc_commit(bar);
    };
    for (uint32_t i = 0; ok; ++i) {
      const int t = next_tile(i, false);
      if (t < 0 || t >= total) break;
      int e, mb, nb, w;
      decode_tile(t, tiles, TB, e, mb, nb, w);
      if constexpr (TM) w = kBM;
      int s0, s1;
      slots.pick(C::NA * w, s0, s1);
      if (!wait_phase<true>(acce_bar(s0), slots.parity(s0) ^ 1u, abort_flag)) break;
      if (s1 >= 0 && !wait_phase<true>(acce_bar(s1), slots.parity(s1) ^ 1u, abort_flag)) break;
      ptx::tc_fence_after();
      const uint32_t idesc = TM ? ptx::idesc_nvfp4(PAIR ? 2 * kBM : kBM, C::NA * kBM, MX) : ptx::idesc_nvfp4(kBM, w, MX);
      const uint32_t d0 = tmem + uint32_t(s0 * kAccSlotCols);
      // The MMAs of K stage kt from pipeline stage st and scale slot sf: a
      // full stage (4 k64 blocks) is one fully unrolled sequence.
      auto issue_stage = [&](int kt, uint32_t st, uint32_t sf) {
        const int nkb = min(4, kblocks - 4 * kt);
        const uint64_t bdesc = ptx::desc_kmajor_sw128(st + off_b);
        auto mma_block = [&](int kb) {
          {
#pragma unroll
            for (int j = 0; j < C::NA; ++j) {
              if constexpr (MX)
                ptx::tc_mma_mxfp4(d0 + j * w, ptx::desc_kmajor_sw128(st + j * kATile) + 2 * kb, bdesc + 2 * kb, idesc,
                                  sf + j * 16 + kb * 4, sf + C::NA * 16 + kb * 4 * C::NSFB, (kt | kb) != 0 ? 1u : 0u);
              else
                ptx::tc_mma_nvfp4(d0 + j * w, ptx::desc_kmajor_sw128(st + j * kATile) + 2 * kb, bdesc + 2 * kb, idesc,
                                  sf + j * 16 + kb * 4, sf + C::NA * 16 + kb * 4 * C::NSFB, (kt | kb) != 0 ? 1u : 0u);
            }
          }
        };
        if (nkb == 4) {
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) mma_block(kb);
        } else {
          for (int kb = 0; kb < nkb; ++kb) mma_block(kb);
        }
      };
      if constexpr (TM) {
        // Token-major: wait for the next stage, then issue it and every
        // following stage of the tile whose operands and scales are already
        // in, back to back (a test of the barrier, no wait), so the MMA
        // queue is refilled with as little thread work between stages as
        // the data allows.  The MMA thread shares its SM sub-partition with
        // busy epilogue warps, and clock64 in it at prefill showed ~330
        // cycles of loop work between two stages, more than the ~256 cycles
        // of MMAs still queued; this loop measured (CTA pairs, prefill)
        // gate/up 2.63 -> 2.41 ms and down 1.46 -> 1.36 ms against one stage
        // per iteration of the general loop.  Stage s's descriptors are stage 0's plus
        // s * stage / 16 in the start-address field (shared addresses stay
        // below 2^18, so the 14-bit field never carries).
        const uint64_t wdesc0 = ptx::desc_kmajor_sw128(smem_base);
        const uint64_t adesc0 = ptx::desc_kmajor_sw128(smem_base + off_b);
        const uint32_t stage16 = uint32_t(stage) >> 4;
        // The next stage's barrier is tested before the stage's last MMA and
        // (CTA pairs) the stage's commit is issued after the first MMA of the
        // next stage of the group, so neither sits between two stages' MMAs:
        // with about one MMA queued, every cycle of this thread between the
        // last MMA of a stage and the first of the next one idles the tensor
        // core (an extra commit or barrier test per stage each cost ~3.5 % of
        // the prefill gate/up GEMM).  Single-SM kernels, with one stage
        // fewer, commit at once: the later release measured 4 % slower there.
        int kt = 0;
        uint32_t ps = 0;    // last stage whose MMAs are issued and not yet committed
        bool pend = false;  // (within a group of stages issued back to back)
        while (kt < nkt) {
          if (!ptx::mbar_test_wait(full_bar(s), ph) && !wait_phase<true>(full_bar(s), ph, abort_flag)) {
            ok = false;
            break;
          }
          bool more;
          do {
            ptx::tc_fence_after();
            const uint64_t so = uint64_t(s * stage16);
            const uint32_t sf = tmem + uint32_t(kSfColBase) + s * uint32_t(C::SfCols);
            const int nkb = min(4, kblocks - 4 * kt);
            uint32_t sn = s + 1, phn = ph;
            if (sn == uint32_t(S)) sn = 0, phn ^= 1u;
            auto mma = [&](int kb) {
              const uint64_t adesc = adesc0 + so + 2 * kb, wdesc = wdesc0 + so + 2 * kb;
              const uint32_t acc = (kt | kb) != 0 ? 1u : 0u;
              const uint32_t sfa = sf + C::NA * 16 + kb * 4, sfw = sf + kb * 8;
              if constexpr (PAIR && MX) ptx::tc_mma_mxfp4_pair(d0, adesc, wdesc, idesc, sfa, sfw, acc);
              else if constexpr (PAIR) ptx::tc_mma_nvfp4_pair(d0, adesc, wdesc, idesc, sfa, sfw, acc);
              else if constexpr (MX) ptx::tc_mma_mxfp4(d0, adesc, wdesc, idesc, sfa, sfw, acc);
              else ptx::tc_mma_nvfp4(d0, adesc, wdesc, idesc, sfa, sfw, acc);
            };
            mma(0);
            if (PAIR && pend) commit(empty_bar(ps));  // frees stage ps (and its scale slot) once its MMAs have read it
            if (nkb == 4) {
              mma(1);
              mma(2);
              more = kt + 1 < nkt && ptx::mbar_test_wait(full_bar(sn), phn);
              mma(3);
            } else {
              for (int kb = 1; kb < nkb; ++kb) mma(kb);
              more = kt + 1 < nkt && ptx::mbar_test_wait(full_bar(sn), phn);
            }
            if (!PAIR) commit(empty_bar(s));
            ps = s, pend = PAIR;
            ++kt, s = sn, ph = phn;
          } while (more);
          if (pend) commit(empty_bar(ps));  // the group's last stage
          pend = false;
        }
      } else {
      // The default orientation issues its N <= 128 MMAs two stages at a time.
      for (int kt = 0; kt < nkt; kt += 2) {
        const bool two = kt + 1 < nkt;
        uint32_t s2 = s + 1, ph2 = ph, r2 = r + 1, rph2 = rph;
        if (s2 == uint32_t(S)) s2 = 0, ph2 ^= 1u;
        if (r2 == uint32_t(C::SfSlots)) r2 = 0, rph2 ^= 1u;
        // A stage's scales are in tensor memory once the scale-factor warps
        // arrive, which they do only after its copies have landed; the
        // stage's own barrier is complete by then and is checked as well.
        // (Tied slots: the scale-factor warps arrive on the stage's barrier.)
        uint32_t ready = kTied ? ptx::mbar_test_wait(full_bar(s), ph)
                               : ptx::mbar_test_wait(sff_bar(r), rph) & ptx::mbar_test_wait(full_bar(s), ph);
        if (two)
          ready &= kTied ? ptx::mbar_test_wait(full_bar(s2), ph2)
                         : ptx::mbar_test_wait(sff_bar(r2), rph2) & ptx::mbar_test_wait(full_bar(s2), ph2);
        if (!ready) {
          if ((!kTied && !wait_phase<true>(sff_bar(r), rph, abort_flag)) ||
              !wait_phase<true>(full_bar(s), ph, abort_flag) ||
              (two && ((!kTied && !wait_phase<true>(sff_bar(r2), rph2, abort_flag)) ||
                       !wait_phase<true>(full_bar(s2), ph2, abort_flag)))) {
            ok = false;
            break;
          }
        }
        ptx::tc_fence_after();
        issue_stage(kt, smem_base + s * uint32_t(stage), tmem + uint32_t(kSfColBase + (kTied ? s : r) * C::SfCols));
        commit(empty_bar(s));  // frees the stage (and, tied, its scale slot) once these MMAs have read it
        if (!kTied) commit(sfe_bar(r));
        if (two) {
          issue_stage(kt + 1, smem_base + s2 * uint32_t(stage),
                      tmem + uint32_t(kSfColBase + (kTied ? s2 : r2) * C::SfCols));
          commit(empty_bar(s2));
          if (!kTied) commit(sfe_bar(r2));
          s = s2 + 1, ph = ph2, r = r2 + 1, rph = rph2;
        } else {
          s = s2, ph = ph2, r = r2, rph = rph2;
        }
        if (s == uint32_t(S)) s = 0, ph ^= 1u;
        if (r == uint32_t(C::SfSlots)) r = 0, rph ^= 1u;
      }
      }
      if (!ok) break;
      commit(accf_bar(s0));
      if (s1 >= 0) commit(accf_bar(s1));
      slots.done(s0, s1);
    }
    commit(drain_bar);  // every MMA of this CTA (pair) done before tensor memory is freed
    drain_phase(drain_bar, 0);
  };
  auto role_scale = [&]() {
    // ---------------- scale factors: shared memory -> tensor memory ----------------
    // Each of the four warps writes its 32-lane quarter of every scale block
    // (the tensor core reads the 512-byte block of 128 rows as four 32-bit
    // columns per lane, the same in every quarter): lane i loads the block's
    // 16-byte row i and stores it as 4 columns.  Doing this with tcgen05.st
    // from these warps keeps the MMA issue stream free of copies, which would
    // otherwise serialise with the MMAs of the previous stage.  The warps
    // wait only for the stage's scale copies, which the producer issues
    // ahead of its operands, so this work is off the path from the operand
    // copies to the MMAs.
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    // column of weight tile j's scales for k64 step kb within a ring slot:
    // per tile (swap AB, the tile is one MMA's A operand) or interleaved per
    // step (token-major, the two tiles are one N = 256 B operand)
    auto wcol = [](int j, int kb) { return TM ? kb * 8 + j * 4 : j * 16 + kb * 4; };
    uint32_t s = 0, ph = 0, r = 0, rph = 0;
    bool ok = true;
    for (uint32_t i = 0; ok; ++i) {
      const int t = next_tile(i, true);
      if (t < 0 || t >= total) break;
      int e, mb, nb, w;
      decode_tile(t, tiles, TB, e, mb, nb, w);
      if constexpr (TM) w = kBM;
      const int sfb_chunks = w > 128 ? 2 : 1;
      for (int kt = 0; kt < nkt; ++kt) {
        // Tied slots: the stage's scale copies are issued only after the MMAs
        // that last read its slot have completed, so their arrival is enough.
        // With a scale ring (slot r) the copies run ahead; the stage's
        // tensor-memory slot s is free once the MMAs of its previous use have
        // completed (its empty barrier).
        if (kRing) {
          if (!wait_phase(sfc_bar(r), rph, abort_flag)) {
            ok = false;
            break;
          }
        } else if ((!kTied && !wait_phase(sfe_bar(r), rph ^ 1u, abort_flag)) || !wait_phase(sfc_bar(s), ph, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t st = kRing ? sf_ring + r * uint32_t(sf_slot) : smem_base + s * uint32_t(stage);
        const uint32_t sf = tmem + lane_base + uint32_t(kSfColBase + (kTied ? s : r) * C::SfCols);
        const int nkb = min(4, kblocks - 4 * kt);
        if constexpr (TM) {
          // Token-major slots are 48 contiguous columns: the weight tiles'
          // scales (step kb, tile j at 8 kb + 4 j) fill columns 0-31 and the
          // token tile's (4 kb) columns 32-47, so the whole slot goes out in
          // two stores (one 32-column and one 16-column tcgen05.st) instead
          // of twelve 4-column ones.  All four steps are stored; the MMAs of
          // a short last stage read only its first nkb.
          uint32_t wv[32], av[16];
          auto put = [](uint32_t* d, const uint4& v) { d[0] = v.x, d[1] = v.y, d[2] = v.z, d[3] = v.w; };
          if constexpr (MX) {
            // A 512-byte MXFP4 block holds 4 ue8m0 scales per row for 128 K
            // elements: bytes 0-1 go to k64 step 2m, bytes 2-3 to step 2m + 1.
            auto lo = [](const uint4& v) { return make_uint4(v.x & 0xFFFFu, v.y & 0xFFFFu, v.z & 0xFFFFu, v.w & 0xFFFFu); };
            auto hi = [](const uint4& v) { return make_uint4(v.x >> 16, v.y >> 16, v.z >> 16, v.w >> 16); };
#pragma unroll
            for (int m = 0; m < 2; ++m) {
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const uint4 v = ptx::lds128(st + off_sfa + j * kSfTile + m * 512 + lane * 16);
                put(wv + (2 * m) * 8 + j * 4, lo(v));
                put(wv + (2 * m + 1) * 8 + j * 4, hi(v));
              }
              const uint4 v = ptx::lds128(st + off_sfb + m * 512 + lane * 16);
              put(av + (2 * m) * 4, lo(v));
              put(av + (2 * m + 1) * 4, hi(v));
            }
          } else {
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
#pragma unroll
              for (int j = 0; j < 2; ++j) put(wv + kb * 8 + j * 4, ptx::lds128(st + off_sfa + j * kSfTile + kb * 512 + lane * 16));
              put(av + kb * 4, ptx::lds128(st + off_sfb + kb * 512 + lane * 16));
            }
          }
          if constexpr (kRing) {
            // The ring slot is read: hand it back, then wait for the
            // tensor-memory slot.  The proxy fence orders these generic-proxy
            // reads before the TMA (async-proxy) writes the slot's next
            // copies make once the arrival is seen; without it some slots
            // were overwritten before they were read (wrong scales in whole
            // token tiles, found by comparing tile orientations bit for bit).
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(sfe_bar(r));
            if (!wait_phase(empty_bar(s), ph ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
          }
          ptx::tmem_st_32x32b_x32(sf, wv);
          ptx::tmem_st_32x32b_x16(sf + 32, av);
        } else if constexpr (MX) {
          // A 512-byte MXFP4 block holds 4 ue8m0 scales per row for 128 K
          // elements: bytes 0-1 go to the k64 step 2m, bytes 2-3 to 2m + 1,
          // each into bytes 0-1 of that step's cell.
          for (int m = 0; m < nkb / 2; ++m) {
#pragma unroll
            for (int j = 0; j < C::NA; ++j) {
              const uint4 v = ptx::lds128(st + off_sfa + j * kSfTile + m * 512 + lane * 16);
              ptx::tmem_st_32x32b_x4(sf + wcol(j, 2 * m), v.x & 0xFFFFu, v.y & 0xFFFFu, v.z & 0xFFFFu,
                                     v.w & 0xFFFFu);
              ptx::tmem_st_32x32b_x4(sf + wcol(j, 2 * m + 1), v.x >> 16, v.y >> 16, v.z >> 16, v.w >> 16);
            }
            for (int c = 0; c < sfb_chunks; ++c) {
              const uint4 v = ptx::lds128(st + off_sfb + c * kSfTile + m * 512 + lane * 16);
              ptx::tmem_st_32x32b_x4(sf + C::NA * 16 + (2 * m) * 4 * C::NSFB + c * 4, v.x & 0xFFFFu, v.y & 0xFFFFu,
                                     v.z & 0xFFFFu, v.w & 0xFFFFu);
              ptx::tmem_st_32x32b_x4(sf + C::NA * 16 + (2 * m + 1) * 4 * C::NSFB + c * 4, v.x >> 16, v.y >> 16,
                                     v.z >> 16, v.w >> 16);
            }
          }
        } else {
          for (int kb = 0; kb < nkb; ++kb) {
#pragma unroll
            for (int j = 0; j < C::NA; ++j) {
              const uint4 v = ptx::lds128(st + off_sfa + j * kSfTile + kb * 512 + lane * 16);
              ptx::tmem_st_32x32b_x4(sf + wcol(j, kb), v.x, v.y, v.z, v.w);
            }
            for (int c = 0; c < sfb_chunks; ++c) {
              const uint4 v = ptx::lds128(st + off_sfb + c * kSfTile + kb * 512 + lane * 16);
              ptx::tmem_st_32x32b_x4(sf + C::NA * 16 + kb * 4 * C::NSFB + c * 4, v.x, v.y, v.z, v.w);
            }
          }
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          // CTA 0 of a pair issues the MMAs; tied slots arrive on the stage's full barrier
          const uint32_t b = kTied ? full_bar(s) : sff_bar(r);
          if constexpr (PAIR) ptx::mbar_arrive_cluster(ptx::mapa(b, 0));
          else ptx::mbar_arrive(b);
        }
        if (++s == uint32_t(S)) s = 0, ph ^= 1u;
        if (++r == uint32_t(kRing ? R : C::SfSlots)) r = 0, rph ^= 1u;
      }
    }
  };
  auto role_epilogue = [&]() {
    // ---------------- epilogue ----------------
    const int q = warp & 3;            // tensor-memory lane quarter this warp may access
    constexpr int kParts = epi_warps(SWIGLU, PAIR) / 4;  // warps sharing a quarter split the columns or token chunks
    const int part = (warp - epi_first(TM)) / 4;
    const int lrow = q * 32 + lane;    // accumulator row = output feature within the tile
    const float a_gs = MX ? 1.0f : *p.a_gscale;   // MXFP4 has no per-tensor scales
    const bool f32_out = p.epi == NVFP4MOE_EPI_SWIGLU_F32;
    const float s_h = (SWIGLU && !f32_out && !MX) ? *p.c_gscale : 1.0f;
    const int n_out = SWIGLU ? p.N / 2 : p.N;
    SlotSeq slots;
    for (uint32_t i = 0;; ++i) {
      const int t = next_tile(i, true);
      if (t < 0 || t >= total) break;
      int e, mb, nb, w;
      decode_tile(t, tiles, TB, e, mb, nb, w);
      if constexpr (TM) w = kBM;
      int s0, s1;
      slots.pick(C::NA * w, s0, s1);
      if (!wait_phase(accf_bar(s0), slots.parity(s0), abort_flag)) break;
      if (s1 >= 0 && !wait_phase(accf_bar(s1), slots.parity(s1), abort_flag)) break;
      ptx::tc_fence_after();
      // this CTA's token rows of the tile (a pair's CTA 1 holds rows 128..255)
      const int valid = min(w, s_count[e] - nb * TB - int(crank) * kBM);
      const int64_t row0 = int64_t(s_rowoff[e]) + int64_t(nb) * TB + int(crank) * kBM;
      const float scale = MX ? 1.0f : a_gs * p.w_gscale[e];
      const uint32_t tbase = tmem + (uint32_t(q * 32) << 16) + uint32_t(s0 * kAccSlotCols);
      const int f = (SWIGLU ? mb : mb * NA) * kBM + lrow;  // output column (of tile 0)
      // h = silu(gate) * up of a chunk, computed in place over the gate
      // registers (a warp holds one raw chunk and one finished one).
      auto swiglu = [&](uint32_t (&g)[32], const uint32_t (&u)[32]) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float gf = __uint_as_float(g[i]) * scale;
          const float uf = __uint_as_float(u[i]) * scale;
          g[i] = __float_as_uint(gf * ptx::rcp_approx(1.0f + __expf(-gf)) * uf);
        }
      };
      auto release = [&]() {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR) {  // CTA 0 issues the next tile's MMAs into both CTAs' accumulators
            ptx::mbar_arrive_cluster(ptx::mapa(acce_bar(s0), 0));
            if (s1 >= 0) ptx::mbar_arrive_cluster(ptx::mapa(acce_bar(s1), 0));
          } else {
            ptx::mbar_arrive(acce_bar(s0));
            if (s1 >= 0) ptx::mbar_arrive(acce_bar(s1));
          }
        }
      };
      if constexpr (TM) {
        // Token-major: accumulator lane = token row of the tile, column =
        // weight row of the N = 256 operand.
        const int64_t row = row0 + q * 32 + lane;
        const bool row_ok = q * 32 + lane < valid;
        if constexpr (SWIGLU) {
          // Features [64 part, 64 part + 64) of the tile's 128: gate in
          // columns c, up in 128 + c; both 32-feature chunks are loaded at
          // once and the accumulator released before any arithmetic.
          static_assert(kParts == 2, "two epilogue warps per lane quarter");
          const int c0 = 64 * part;
          uint32_t h0[32], u0[32], g[32], u[32];
          ptx::tmem_ld_32x32b_x32(tbase + c0, h0);
          ptx::tmem_ld_32x32b_x32(tbase + kBM + c0, u0);
          ptx::tmem_ld_32x32b_x32(tbase + c0 + 32, g);
          ptx::tmem_ld_32x32b_x32(tbase + kBM + c0 + 32, u);
          ptx::tmem_ld_wait();
          release();
          swiglu(h0, u0);
          swiglu(g, u);
          if (row_ok) {
            const int fo = mb * kBM + c0;  // output feature of h0[0]
            if (f32_out) {
              float4* out = reinterpret_cast<float4*>(static_cast<float*>(p.c_out) + row * n_out + fo);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                out[i] = make_float4(__uint_as_float(h0[4 * i]), __uint_as_float(h0[4 * i + 1]),
                                     __uint_as_float(h0[4 * i + 2]), __uint_as_float(h0[4 * i + 3]));
                out[8 + i] = make_float4(__uint_as_float(g[4 * i]), __uint_as_float(g[4 * i + 1]),
                                         __uint_as_float(g[4 * i + 2]), __uint_as_float(g[4 * i + 3]));
              }
            } else if constexpr (MX) {
              requant_row32_mx(h0, row, fo, n_out, static_cast<uint8_t*>(p.c_out), p.c_scales);
              requant_row32_mx(g, row, fo + 32, n_out, static_cast<uint8_t*>(p.c_out), p.c_scales);
            } else {
              requant_row32(h0, s_h, row, fo, n_out, static_cast<uint8_t*>(p.c_out), p.c_scales);
              requant_row32(g, s_h, row, fo + 32, n_out, static_cast<uint8_t*>(p.c_out), p.c_scales);
            }
          }
        } else {
          if constexpr (kParts == 2) {
          // bf16: columns c = output features mb * 256 + c, 64 bytes per
          // chunk and row.  Two warps per lane quarter: warp part p takes
          // columns 128 p .. 128 p + 127 (four 32-column chunks), loads them
          // in one tensor-memory round trip and releases the accumulator
          // before any arithmetic (with one warp per quarter the second
          // round trip waited for the first one's conversion, ~1.5k cycles
          // of accumulator drain per tile at prefill), then packs them to
          // bf16.  A thread's row is 14 KB away from its neighbour's, so each
          // chunk is staged in this warp's 2 KB buffer and written by a TMA
          // store (full 64-byte row segments) when all 32 rows of the quarter
          // belong to the expert; a partial quarter stores per thread and
          // leaves the padding rows untouched.
          constexpr int kMine = C::NA * kBM / 32 / 2;  // this warp's 32-column chunks
          const int cbase = kMine * part;              // its first chunk
          uint32_t pk[kMine][16];
          {
            uint32_t g[kMine][32];
#pragma unroll
            for (int j = 0; j < kMine; ++j) ptx::tmem_ld_32x32b_x32(tbase + 32 * (cbase + j), g[j]);
            ptx::tmem_ld_wait();
            release();
#pragma unroll
            for (int j = 0; j < kMine; ++j)
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(g[j][2 * i]) * scale,
                                                               __uint_as_float(g[j][2 * i + 1]) * scale);
                pk[j][i] = *reinterpret_cast<const uint32_t*>(&v);
              }
          }
          if constexpr (FIN) {
            // fused finalize: this thread's token row, times its routing
            // weight, added into the token's float32 row
            if (row_ok) {
              const int fl = __ldg(p.perm_to_flat + row);
              const float wt = __ldg(p.topk_w + fl);
              float* dst = static_cast<float*>(p.c_out) + int64_t(fl / p.k) * n_out + mb * (C::NA * kBM);
#pragma unroll
              for (int j = 0; j < kMine; ++j)
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[j][i]));
                  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[j][i + 1]));
                  ptx::red_add_v4(dst + 32 * (cbase + j) + 2 * i, wt * a.x, wt * a.y, wt * b.x, wt * b.y);
                }
            }
            slots.done(s0, s1);
            continue;
          }
          const bool quarter_full = q * 32 + 32 <= valid;
          const uint32_t obuf = out_base + uint32_t((warp - epi_first(TM)) * kOutChunkBytes);
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.c_out) + row * n_out + mb * (C::NA * kBM);
#pragma unroll
          for (int j = 0; j < kMine; ++j) {
            const int c = cbase + j;
            if (quarter_full) {
              if (lane == 0) ptx::bulk_wait_read_all();  // the previous chunk's store has read the buffer
              __syncwarp();
#pragma unroll
              for (int i = 0; i < 4; ++i)
                ptx::sts128(obuf + uint32_t(lane * 64 + i * 16), pk[j][4 * i], pk[j][4 * i + 1], pk[j][4 * i + 2],
                            pk[j][4 * i + 3]);
              ptx::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                ptx::tma_store_2d(&tmap_c, obuf, mb * (C::NA * kBM) + 32 * c, int(row0 + q * 32));
                ptx::bulk_commit();
              }
            } else if (row_ok) {
              uint4* o = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                o[i] = make_uint4(pk[j][4 * i], pk[j][4 * i + 1], pk[j][4 * i + 2], pk[j][4 * i + 3]);
            }
          }
          } else {
          // bf16: columns c = output features mb * 256 + c, 64 bytes per
          // chunk and row.  The whole row (256 columns) is packed to bf16 in
          // registers, two chunks per tensor-memory round trip, and the
          // accumulator released before any store.  A thread's row is 14 KB
          // away from its neighbour's, so each chunk is staged in this warp's
          // 2 KB buffer and written by a TMA store (full 64-byte row
          // segments) when all 32 rows of the quarter belong to the expert;
          // a partial quarter stores per thread and leaves the padding rows
          // untouched.
          // Four 32-column chunks per tensor-memory round trip (two round
          // trips for the row), packed to bf16 in registers.
          constexpr int kChunks = C::NA * kBM / 32;
          constexpr int kPerTrip = 4;
          uint32_t pk[kChunks][16];
#pragma unroll
          for (int c = 0; c < kChunks; c += kPerTrip) {
            uint32_t g[kPerTrip][32];
#pragma unroll
            for (int j = 0; j < kPerTrip; ++j) ptx::tmem_ld_32x32b_x32(tbase + 32 * (c + j), g[j]);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < kPerTrip; ++j)
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(g[j][2 * i]) * scale,
                                                               __uint_as_float(g[j][2 * i + 1]) * scale);
                pk[c + j][i] = *reinterpret_cast<const uint32_t*>(&v);
              }
          }
          release();
          if constexpr (FIN) {
            // fused finalize: this thread's token row, times its routing
            // weight, added into the token's float32 row
            if (row_ok) {
              const int fl = __ldg(p.perm_to_flat + row);
              const float wt = __ldg(p.topk_w + fl);
              float* dst = static_cast<float*>(p.c_out) + int64_t(fl / p.k) * n_out + mb * (C::NA * kBM);
#pragma unroll
              for (int c = 0; c < kChunks; ++c)
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[c][i]));
                  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[c][i + 1]));
                  ptx::red_add_v4(dst + 32 * c + 2 * i, wt * a.x, wt * a.y, wt * b.x, wt * b.y);
                }
            }
            slots.done(s0, s1);
            continue;
          }
          const bool quarter_full = q * 32 + 32 <= valid;
          const uint32_t obuf = out_base + uint32_t(q * kOutChunkBytes);
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.c_out) + row * n_out + mb * (C::NA * kBM);
#pragma unroll
          for (int c = 0; c < kChunks; ++c) {
            if (quarter_full) {
              if (lane == 0) ptx::bulk_wait_read_all();  // the previous chunk's store has read the buffer
              __syncwarp();
#pragma unroll
              for (int i = 0; i < 4; ++i)
                ptx::sts128(obuf + uint32_t(lane * 64 + i * 16), pk[c][4 * i], pk[c][4 * i + 1], pk[c][4 * i + 2],
                            pk[c][4 * i + 3]);
              ptx::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                ptx::tma_store_2d(&tmap_c, obuf, mb * (C::NA * kBM) + 32 * c, int(row0 + q * 32));
                ptx::bulk_commit();
              }
            } else if (row_ok) {
              uint4* o = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                o[i] = make_uint4(pk[c][4 * i], pk[c][4 * i + 1], pk[c][4 * i + 2], pk[c][4 * i + 3]);
            }
          }
          }
        }
      } else if constexpr (SWIGLU) {
        // Drain this warp's chunks (at most two: BN = 128 and two warps per
        // lane quarter) into h = silu(gate) * up, release the accumulator so
        // the next tile's MMAs can start, then requantise from registers.
        static_assert(BN == 128 && kParts == 2, "two 32-token chunks per epilogue warp");
        // The accumulator is released once both chunks are in registers; the
        // second chunk's SwiGLU (bound by the special-function units) runs
        // after that.
        uint32_t h0[32], g[32], u[32];
        const bool have0 = 32 * part < valid, have1 = 32 * part + 64 < valid;
        if (have0) {
          ptx::tmem_ld_32x32b_x32(tbase + 32 * part, h0);
          ptx::tmem_ld_32x32b_x32(tbase + w + 32 * part, u);
          ptx::tmem_ld_wait();
          swiglu(h0, u);
        }
        if (have1) {
          ptx::tmem_ld_32x32b_x32(tbase + 32 * part + 64, g);
          ptx::tmem_ld_32x32b_x32(tbase + w + 32 * part + 64, u);
          ptx::tmem_ld_wait();
        }
        release();
        if (have1) swiglu(g, u);
        float hb[2][32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          hb[0][i] = __uint_as_float(h0[i]);
          hb[1][i] = __uint_as_float(g[i]);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c0 = 32 * part + 64 * j;
          if (c0 < valid) {
            if (f32_out) {
              float* out = static_cast<float*>(p.c_out) + (row0 + c0) * n_out + f;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (c0 + i < valid) out[int64_t(i) * n_out] = hb[j][i];
            } else if constexpr (MX) {
              requant_swiglu_chunk_mx(hb[j], lane, row0 + c0, valid - c0, f, n_out, static_cast<uint8_t*>(p.c_out),
                                      p.c_scales);
            } else {
              requant_swiglu_chunk(hb[j], lane, s_h, row0 + c0, valid - c0, f, n_out,
                                   static_cast<uint8_t*>(p.c_out), p.c_scales);
            }
          }
        }
      } else {
        // NVFP4MOE_EPI_FINALIZE_F32: each row's bf16 values, times the
        // row's routing weight, are added into its token's float32 row.
        constexpr bool scatter = FIN;
        for (int c0 = 32 * part; c0 < valid; c0 += 32 * kParts) {
#pragma unroll
          for (int j = 0; j < NA; ++j) {  // NA consecutive 128-row blocks of the tile
            uint32_t g[32];
            ptx::tmem_ld_32x32b_x32(tbase + j * w + c0, g);
            ptx::tmem_ld_wait();
            const int col = f + j * kBM;
            if constexpr (scatter) {
              float* acc = static_cast<float*>(p.c_out);
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (c0 + i < valid) {
                  const int fl = __ldg(p.perm_to_flat + row0 + c0 + i);
                  const float y = __bfloat162float(__float2bfloat16_rn(__uint_as_float(g[i]) * scale));
                  atomicAdd(acc + int64_t(fl / p.k) * n_out + col, __ldg(p.topk_w + fl) * y);
                }
            } else {
              __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.c_out);
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (c0 + i < valid) out[(row0 + c0 + i) * n_out + col] = __float2bfloat16_rn(__uint_as_float(g[i]) * scale);
            }
          }
        }
        release();
      }
      slots.done(s0, s1);
    }
    if constexpr (TM && !SWIGLU) {
      if (lane == 0) ptx::bulk_wait_all();  // this warp's TMA stores have completed
    }
  };
  // Teardown, reached by every thread: all roles done, tensor memory freed
  // by warp 1 (for a pair: by both CTAs together, once both are done with
  // it), no CTA of a pair leaving while the other may still signal it.
  auto teardown = [&]() {
    ptx::tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) ptx::cluster_sync();
    if (warp == 1) {
      __syncwarp();
      ptx::tc_fence_after();
      if constexpr (PAIR) ptx::tmem_dealloc_pair(tmem, kTmemCols);
      else ptx::tmem_dealloc(tmem, kTmemCols);
    }
    if constexpr (PAIR) ptx::cluster_sync();
    // Dynamic schedule: the last CTA to finish (every producer has stopped
    // claiming by then) leaves both counters at zero for the next launch.
    if (sched && threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(p.sched + 32, 1u) == gridDim.x - 1) {
        atomicExch(p.sched, 0u);
        atomicExch(p.sched + 32, 0u);
      }
    }
  };
  if constexpr (TM) {
    // Token-major kernels branch by warpgroup first: each warpgroup sets its
    // register budget (setmaxnreg) at the top of its branch, so the
    // epilogue warpgroups get the registers the producer / MMA and the
    // scale-factor warpgroups leave unused and can hold their whole share of
    // the accumulator (budgets at regs_control).  Each branch runs its own
    // copy of the teardown, so no code is shared by warps with different
    // budgets.
    const int wg = warp >> 2;
    if (wg == 0) {
      ptx::setmaxnreg_dec<regs_control(epi_warps(SWIGLU, PAIR) == 8)>();
      if (lane == 0 && (warp == 0 || (kRing && warp == 2))) {
        role_producer(warp == 0 ? 0 : 1);
      } else if (warp == 1 && lane == 0) {
        if (PAIR && crank != 0) role_peer_wait();
        else role_mma();
      }
      __syncwarp();
      teardown();
    } else if (wg == (epi_first(TM) + epi_warps(SWIGLU, PAIR)) / 4) {
      ptx::setmaxnreg_dec<regs_scale(epi_warps(SWIGLU, PAIR) == 8)>();
      role_scale();
      teardown();
    } else {
      ptx::setmaxnreg_inc<regs_epilogue(epi_warps(SWIGLU, PAIR) == 8)>();
      role_epilogue();
      teardown();
    }
  } else {
    if (warp == 0 && lane == 0) role_producer(0);
    else if (warp == 1 && lane == 0) role_mma();
    else if (warp >= epi_first(TM) + epi_warps(SWIGLU, PAIR)) role_scale();
    else if (warp >= epi_first(TM)) role_epilogue();
    teardown();
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D byte tensor [rows, row_bytes] -> TMA map with a [box_rows, 128 B] box, 128B swizzle.
bool encode_kmajor_map(CUtensorMap* m, const void* base, int64_t rows, int64_t row_bytes, int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cuuint64_t(row_bytes), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(row_bytes)};
  cuuint32_t box[2] = {cuuint32_t(kBKBytes), cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Weight map: a 5-D byte view of the weights whose box {128 B, 128 rows, ...}
// holds the `tiles` weight tiles of one pipeline stage back to back (one copy
// per stage; a CTA of a pair loads one of the two, tiles = 1).  Coordinates (kt * dx, c1, c2 + kt * dz, c3, c4):
//   row-major, SwiGLU: [K/2 B][I rows][2E halves (gate, up)]   box {128, 128, 2}
//                      at (128 kt, 128 mb, 2e)
//   row-major, other:  [K/2 B][128 rows][E N / 128 blocks]      box {128, 128, NA}
//                      at (128 kt, 0, first block)
//   tiled, SwiGLU:     [128 B][128 rows][kc chunks][I / 128 blocks][2E halves]
//                      box {128, 128, 1, 1, 2} at (0, 0, kt, mb, 2e)
//   tiled, other:      [128 B][128 rows][kc chunks][E N / 128 blocks]
//                      box {128, 128, 1, NA} at (0, 0, kt, first block)
// Unit dimensions fill the view to 5-D.
bool encode_weight_map(CUtensorMap* m, const GemmArgs& a, bool swiglu, int tiles) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const int64_t kh = a.K / 2, kc = (a.K + 255) / 256, nblk = int64_t(a.E) * a.N / kBM, half = a.N / 2;
  cuuint64_t dims[5];
  cuuint64_t strides[4];
  cuuint32_t box[5] = {cuuint32_t(kBKBytes), cuuint32_t(kBM), 1, 1, 1};
  if (!a.w_tiled) {
    if (swiglu) {
      dims[0] = kh, dims[1] = half, dims[2] = 2 * int64_t(a.E);
      strides[0] = kh, strides[1] = half * kh;
    } else {
      dims[0] = kh, dims[1] = kBM, dims[2] = nblk;
      strides[0] = kh, strides[1] = kBM * kh;
    }
    box[2] = cuuint32_t(tiles);
    dims[3] = dims[4] = 1;
    strides[2] = strides[3] = strides[1] * dims[2];
  } else {
    dims[0] = kBKBytes, dims[1] = kBM, dims[2] = kc;
    strides[0] = kBKBytes, strides[1] = kWeightBoxBytes, strides[2] = kc * kWeightBoxBytes;
    if (swiglu) {
      dims[3] = half / kBM, dims[4] = 2 * int64_t(a.E);
      strides[3] = (half / kBM) * kc * kWeightBoxBytes;
      box[4] = cuuint32_t(tiles);
    } else {
      dims[3] = nblk, dims[4] = 1;
      strides[3] = nblk * kc * kWeightBoxBytes;
      box[3] = cuuint32_t(tiles);
    }
  }
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<uint8_t*>(a.w_packed), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Weight scale map: the blocked scales of the weights as 8-byte elements,
// [sf_k * 64 elements per 128-row block][row blocks][halves], whose box
// {256, 1, 2} (SwiGLU: gate and up blocks of the same features) or
// {256, NA, 1} (NA consecutive blocks) is 2 KB per weight tile from the
// stage's first block, at (64 sf_per_kt kt, block, half): an NVFP4 stage's
// four blocks, or an MXFP4 stage's two and the next stage's (unused); past
// the last K block the box reads zeros.
bool encode_weight_scale_map(CUtensorMap* m, const GemmArgs& a, bool swiglu, int na) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const int64_t sf_k = a.mx ? a.K / 128 : a.K / 64;  // 512-byte blocks per 128-row block
  const int64_t row_elems = sf_k * 64, nblk = int64_t(a.E) * a.N / kBM;
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3] = {cuuint32_t(kSfTile / 8), 1, 1};
  dims[0] = row_elems;
  strides[0] = sf_k * 512;
  if (swiglu) {
    dims[1] = a.N / 2 / kBM, dims[2] = 2 * int64_t(a.E);
    box[2] = 2;
  } else {
    dims[1] = nblk, dims[2] = 1;
    box[1] = cuuint32_t(na);
  }
  strides[1] = strides[0] * dims[1];
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint8_t*>(a.w_scales), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Token scale map: the blocked scales of the permuted activations as 8-byte
// elements, [sf_k * 64 elements per 128-row block][row blocks], whose box
// {256, 1, 1} is one stage's 2 KB for a 128-row token tile at
// (64 sf_per_kt kt, row block, 0), zero-filled past the last K block.
bool encode_token_scale_map(CUtensorMap* m, const GemmArgs& a) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const int64_t sf_k = a.mx ? a.K / 128 : a.K / 64;
  cuuint64_t dims[3] = {cuuint64_t(sf_k * 64), cuuint64_t(a.rows_capacity / kBM), 1};
  cuuint64_t strides[2] = {cuuint64_t(sf_k * 512), cuuint64_t(sf_k * 512 * (a.rows_capacity / kBM))};
  cuuint32_t box[3] = {cuuint32_t(kSfTile / 8), 1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint8_t*>(a.a_scales), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 [rows, cols] output written by 32-row x 32-column TMA stores (64-byte
// rows in shared memory, no swizzle).
bool encode_bf16_store_map(CUtensorMap* m, void* base, int64_t rows, int64_t cols) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(cols * 2)};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Stage cap: NVFP4MOE_STAGE_CAP in the environment (2..16) overrides the
// default of as many stages as fit, for pipeline-depth studies.
int stage_cap_from_env() {
  static const int cap = [] {
    const char* v = std::getenv("NVFP4MOE_STAGE_CAP");
    const int c = v ? std::atoi(v) : kMaxStages;
    return c < 2 ? 2 : (c > kMaxStages ? kMaxStages : c);
  }();
  return cap;
}

// CTA pairs of a kernel that can be resident at once (clusters of two), per
// device, looked up once.
template <typename K>
int max_pairs(K kernel, int threads, size_t smem, int num_sms) {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) return 0;
  cached[dev] = std::min(n, num_sms / 2);
  return cached[dev];
}

// L2 policy of the weight copies of token-major kernels: NVFP4MOE_WPOL
// (0 evict_first, 1 evict_normal, 2 evict_last), for cache studies.
int w_policy_from_env(int dflt) {
  static const int v = [] {
    const char* e = std::getenv("NVFP4MOE_WPOL");
    return e ? std::atoi(e) : -1;
  }();
  return v >= 0 && v <= 2 ? v : dflt;
}

template <int BN, int NA, bool SWIGLU, bool MX, bool TM = false, bool PAIR = false, bool FIN = false>
int launch_impl(const GemmArgs& a, int num_sms, int smem_optin, cudaStream_t st) {
  using C = Cfg<BN, NA, SWIGLU>;
  // The whole opt-in shared memory is requested; the kernel sizes its stages
  // for the widest token tile present.  Two stages of the widest possible
  // tile must fit.
  const int64_t usable = int64_t(smem_optin) - 1024 - ctrl_bytes(a.E);
  const int worst = PAIR ? kATile + kBM * kBKBytes + NA * kSfTile + kSfTile : C::stage_bytes(BN);
  if (usable < 2 * int64_t(worst) + out_stage_bytes(SWIGLU, TM, PAIR)) {
    set_error_detail(
        "grouped GEMM tile %dx%d (%s) needs %lld bytes of shared memory for a 2-stage pipeline; Hardware limit: %d",
        kBM * NA, BN, SWIGLU ? "gate/up" : "down",
        (long long)(1024 + ctrl_bytes(a.E) + 2 * int64_t(worst) + out_stage_bytes(SWIGLU, TM, PAIR)), smem_optin);
    return NVFP4MOE_ERR_SMEM;
  }
  const size_t smem = size_t(smem_optin);
  CUtensorMap tw, ta, tc, tsf, tasf;
  const int w_kc = (a.K + 255) / 256;
  if (!encode_weight_map(&tw, a, SWIGLU, PAIR ? 1 : (SWIGLU ? 2 : NA)) || !encode_weight_scale_map(&tsf, a, SWIGLU, NA) ||
      !encode_token_scale_map(&tasf, a) ||
      !encode_kmajor_map(&ta, a.a_packed, a.rows_capacity, a.K / 2, TM ? kBM : 32) ||
      !(out_stage_bytes(SWIGLU, TM, PAIR) && a.epilogue != NVFP4MOE_EPI_FINALIZE_F32
            ? encode_bf16_store_map(&tc, a.c_out, a.rows_capacity, a.N)
            : encode_kmajor_map(&tc, a.a_packed, a.rows_capacity, a.K / 2, 32))) {
    set_error_detail("cuTensorMapEncodeTiled failed or is unavailable");
    return NVFP4MOE_ERR_CUDA;
  }
  auto kernel = grouped_gemm_kernel<BN, NA, SWIGLU, MX, TM, PAIR, FIN>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (err != cudaSuccess) {
    set_error_detail("cudaFuncSetAttribute: %s", cudaGetErrorString(err));
    return NVFP4MOE_ERR_CUDA;
  }
  Params p;
  p.w_scales = a.w_scales;
  p.a_scales = a.a_scales;
  p.a_gscale = a.a_gscale;
  p.w_gscale = a.w_gscale;
  p.counts = a.counts;
  p.row_offsets = a.row_offsets;
  p.c_gscale = a.c_gscale;
  p.c_out = a.c_out;
  p.c_scales = a.c_scales;
  p.E = a.E;
  p.N = a.N;
  p.K = a.K;
  p.epi = a.epilogue;
  p.smem_bytes = int(smem) - 1024;
  p.stage_cap = stage_cap_from_env();
  p.rows_cap = a.rows_capacity;
  p.sched = static_cast<uint32_t*>(a.sched);
  p.w_tiled = a.w_tiled ? 1 : 0;
  p.w_kc = w_kc;
  p.wait_us = wait_limit_us();
  p.min_rows = a.min_rows;
  p.max_rows = a.max_rows;
  p.perm_to_flat = a.perm_to_flat;
  p.topk_w = a.topk_w;
  p.k = a.k;
  // Pair tiles serve experts with many rows: every weight tile is re-read by
  // each of the expert's token tiles, so the weights stay in L2 (evict_last;
  // measured at 2048 rows per expert: gate/up 2.76 -> 2.66 ms, down 1.58 ->
  // 1.46 ms against evict_first).
  p.w_policy = PAIR ? w_policy_from_env(2) : TM ? w_policy_from_env(0) : 0;
  // Launched without programmatic dependent launch: measured on GB300, a
  // grouped GEMM launched with it streamed its weight tiles about 2.5%
  // slower per tile, more than the few microseconds of launch latency it
  // hides.  The kernel still starts with griddepcontrol.wait (a no-op here),
  // so the kernel after it may be launched with the attribute.
  if constexpr (PAIR) {
    // Clusters of two CTAs on neighbouring SMs, as many as can be resident
    // at once (the kernel is persistent: pair c takes tiles c, c + #pairs, ...).
    const int pairs = max_pairs(kernel, num_threads(SWIGLU, TM, PAIR), smem, num_sms);
    if (pairs < 1) {
      set_error_detail("no CTA pair of the grouped GEMM fits on this device");
      return NVFP4MOE_ERR_SMEM;
    }
    p.sched = nullptr;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(num_threads(SWIGLU, TM, PAIR));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, kernel, tw, ta, tc, tsf, tasf, p);
    if (err == cudaSuccess) err = cudaGetLastError();
  } else {
    kernel<<<num_sms, num_threads(SWIGLU, TM, PAIR), smem, st>>>(tw, ta, tc, tsf, tasf, p);
    err = cudaGetLastError();
  }
  if (err != cudaSuccess) {
    set_error_detail("grouped GEMM launch: %s", cudaGetErrorString(err));
    return NVFP4MOE_ERR_CUDA;
  }
  return NVFP4MOE_OK;
}

}  // namespace

template <bool MX>
int launch_format(const GemmArgs& a, int num_sms, int smem_optin, cudaStream_t st) {
  const bool swiglu = a.epilogue != NVFP4MOE_EPI_BF16 && a.epilogue != NVFP4MOE_EPI_FINALIZE_F32;
  const int bn = a.tile_n == 0 ? 128 : a.tile_n;
  // Two 128-row weight tiles per stage whenever N allows: each stage carries
  // twice the weight bytes and two accumulation chains, and every token tile
  // loaded serves 256 output features (measured: the down GEMM at decode
  // 0.48 -> 0.30 ms, at 2048 rows per expert 4.02 -> 2.78 ms).
  const bool pair = a.N % (2 * kBM) == 0;
  if constexpr (!MX) {
    if (a.epilogue == NVFP4MOE_EPI_FINALIZE_F32) {
      if (a.tile_n == NVFP4MOE_TILE_TOKEN_MAJOR_PAIR && pair)
        return launch_impl<128, 2, false, false, true, true, true>(a, num_sms, smem_optin, st);
      if (a.tile_n == NVFP4MOE_TILE_TOKEN_MAJOR && pair)
        return launch_impl<128, 2, false, false, true, false, true>(a, num_sms, smem_optin, st);
      if (bn == 128 && pair) return launch_impl<128, 2, false, false, false, false, true>(a, num_sms, smem_optin, st);
      if (bn == 128) return launch_impl<128, 1, false, false, false, false, true>(a, num_sms, smem_optin, st);
      set_error_detail("tile_n %d is not supported with the fused finalize", a.tile_n);
      return NVFP4MOE_ERR_UNSUPPORTED;
    }
  }
  if (a.tile_n == NVFP4MOE_TILE_TOKEN_MAJOR_PAIR && pair) {
    if (swiglu) return launch_impl<128, 2, true, MX, true, true>(a, num_sms, smem_optin, st);
    return launch_impl<128, 2, false, MX, true, true>(a, num_sms, smem_optin, st);
  }
  if (a.tile_n == NVFP4MOE_TILE_TOKEN_MAJOR && pair) {
    if (swiglu) return launch_impl<128, 2, true, MX, true>(a, num_sms, smem_optin, st);
    return launch_impl<128, 2, false, MX, true>(a, num_sms, smem_optin, st);
  }
  if (swiglu && bn == 128) return launch_impl<128, 2, true, MX>(a, num_sms, smem_optin, st);
  if (!swiglu && bn == 128 && pair) return launch_impl<128, 2, false, MX>(a, num_sms, smem_optin, st);
  if (!swiglu && bn == 128) return launch_impl<128, 1, false, MX>(a, num_sms, smem_optin, st);
  if (!swiglu && bn == 256) return launch_impl<256, 1, false, MX>(a, num_sms, smem_optin, st);
  set_error_detail("tile_n %d is not supported for this epilogue", a.tile_n);
  return NVFP4MOE_ERR_UNSUPPORTED;
}

namespace {

// Tiled weight layout: one thread per 16 bytes of the output.  Output unit u
// is byte 16 * (u % 8) of row (u / 8) % 128 of box u / 1024; box b holds
// row block b / kc, K chunk b % kc.  Bytes past the row's end are zero.
__global__ void __launch_bounds__(256) tile_weights_kernel(const uint4* __restrict__ w, int64_t rows, int row_bytes,
                                                           int kc, uint4* __restrict__ out) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int64_t units = rows / kBM * kc * (kWeightBoxBytes / 16);
  const int row16 = row_bytes / 16;
  for (int64_t u = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; u < units; u += int64_t(gridDim.x) * blockDim.x) {
    const int64_t box = u >> 10;
    const int r = int(u >> 3) & 127, c16 = int(u & 7);
    const int64_t rb = box / kc;
    const int col16 = int(box - rb * kc) * 8 + c16;  // 16-byte column within the row
    out[u] = col16 < row16 ? __ldg(w + (rb * kBM + r) * row16 + col16) : make_uint4(0u, 0u, 0u, 0u);
  }
}

}  // namespace

cudaError_t launch_tile_weights(const uint8_t* w_packed, int64_t rows, int K, uint8_t* w_tiled, int num_sms,
                                cudaStream_t st) {
  const int kc = (K + 255) / 256;
  const int64_t units = rows / kBM * kc * (kWeightBoxBytes / 16);
  const int64_t want = (units + 255) / 256, cap = int64_t(num_sms) * 16;
  return launch_kernel(tile_weights_kernel, dim3(unsigned(want < cap ? want : cap)), dim3(256), 0, st, false,
                       reinterpret_cast<const uint4*>(w_packed), rows, K / 2, kc, reinterpret_cast<uint4*>(w_tiled));
}

int launch_grouped_gemm(const GemmArgs& a, int num_sms, int smem_optin, cudaStream_t st) {
  return a.mx ? launch_format<true>(a, num_sms, smem_optin, st) : launch_format<false>(a, num_sms, smem_optin, st);
}

namespace {

// One CTA waits, through the grouped GEMM's bounded wait, for a phase of an
// mbarrier that expects `expected` arrivals and receives `arrivals` (one per
// thread, arrivals <= 32): with arrivals < expected the phase never
// completes and the wait gives up after the launch's wait limit, raising
// the sticky timeout flag.
__global__ void __launch_bounds__(32, 1) wait_selftest_kernel(uint32_t expected, uint32_t arrivals, uint32_t wait_us) {
  __shared__ uint64_t bar;
  __shared__ WaitCtl ctl;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), expected);
    ctl.abort = 0;
    ctl.limit_us = wait_us;
    ptx::fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x < arrivals) ptx::mbar_arrive(ptx::smem_u32(&bar));
  __syncwarp();
  if (threadIdx.x == 0) wait_phase(ptx::smem_u32(&bar), 0, &ctl);
}

}  // namespace

cudaError_t launch_wait_selftest(uint32_t expected, uint32_t arrivals, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(expected, arrivals, wait_limit_us());
  return cudaGetLastError();
}

cudaError_t gemm_read_and_clear_flags(unsigned* flags) {
  unsigned zero = 0;
  cudaError_t err = cudaMemcpyFromSymbol(flags, g_gemm_flags, sizeof(unsigned));
  if (err != cudaSuccess) return err;
  return cudaMemcpyToSymbol(g_gemm_flags, &zero, sizeof(unsigned));
}

}  // namespace nvfp4moe
