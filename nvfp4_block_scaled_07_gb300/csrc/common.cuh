// Device helpers shared by the libnvfp4moe kernels (sm_103a only).
//
// NVFP4 codec: E2M1 codes with one unsigned E4M3 (ue4m3) scale per 16
// elements and a float32 per-tensor scale -- the operand types of the
// block-scaled MMA ("SM120 FP4 Kernel Research Campaign", section 1).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace nvfp4moe {

constexpr float kE2M1Max = 6.0f;
constexpr float kGlobalScaleDivisor = 2688.0f;   // 6 * 448: largest E2M1 * largest ue4m3

// Offset of the 4-byte scale group (row, kb) in the blocked scale layout:
// blocks of 128 rows x 64 K elements, 512 bytes each, row r of a block at
// (r % 32) * 16 + (r / 32) * 4.  kblocks = cols / 64.
__host__ __device__ __forceinline__ int64_t blocked_sf_offset(int64_t row, int64_t kb, int64_t kblocks) {
  return ((row >> 7) * kblocks + kb) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4;
}

// Round a non-negative float to the nearest ue4m3 byte, ties to even,
// saturating at 448 (0x7E).  Works on the float32 bit pattern.
__device__ __forceinline__ uint32_t f32_to_ue4m3(float t) {
  if (!(t < 448.0f)) return 0x7Eu;                  // also catches +inf
  const uint32_t bits = __float_as_uint(t);
  const int e = int(bits >> 23) - 127;              // unbiased exponent of t
  if (e < -6) {
    // ue4m3 subnormal range: value = m * 2^-9, m in 0..8 (8 is the first normal)
    return uint32_t(__float2int_rn(t * 512.0f));    // exact scaling, RNE to integer
  }
  const uint32_t mant = bits & 0x7FFFFFu;
  uint32_t m3 = mant >> 20;
  const uint32_t rest = mant & 0xFFFFFu;
  if (rest > 0x80000u || (rest == 0x80000u && (m3 & 1u))) ++m3;   // RNE on the dropped 20 bits
  uint32_t code = (uint32_t(e + 7) << 3) + m3;                      // mantissa carry bumps the exponent
  return code > 0x7Eu ? 0x7Eu : code;
}

// Value of a ue4m3 byte (valid bytes 0..0x7E).
__device__ __forceinline__ float ue4m3_to_f32(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  if (e == 0) return float(m) * (1.0f / 512.0f);
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Two E2M1 codes in one byte (lo in the low nibble) by the hardware
// conversion: the nearest of {0, .5, 1, 1.5, 2, 3, 4, 6} in magnitude, ties
// to the even code, saturating at 6, the sign kept (so small negatives give
// -0, code 0x8).
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// ---- MXFP4: E2M1 with one E8M0 scale 2^X per 32 elements ----------------------
// X = floor(log2(amax)) - 2 (2 = exponent of E2M1's largest value, 6 = 1.5 * 2^2),
// clamped to [-127, 127]; an all-zero block takes X = -127.  floor(log2) is
// read off the float32 bits (normal or subnormal), so it is exact.
__device__ __forceinline__ int mx_exponent(float amax) {
  const uint32_t bits = __float_as_uint(amax);
  if (bits == 0u) return -127;
  const int e_field = int(bits >> 23);
  const int fl = e_field ? e_field - 127 : (31 - __clz(int(bits))) - 149;
  const int x = fl - 2;
  return x < -127 ? -127 : (x > 127 ? 127 : x);
}

// 2^-X as a float32 (exact: X <= 125 for any finite bf16/float32 amax, and
// 2^127 is representable for X = -127).
__device__ __forceinline__ float mx_inv_step(int x) { return __uint_as_float(uint32_t(127 - x) << 23); }

// Two MXFP4 codes in one byte (x * 2^-X is exact, so the conversion rounds the true quotient).
__device__ __forceinline__ uint32_t mx_code2(float lo, float hi, float inv_step) {
  return e2m1x2(lo * inv_step, hi * inv_step);
}

}  // namespace nvfp4moe
