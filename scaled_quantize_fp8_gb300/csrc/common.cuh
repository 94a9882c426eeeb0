// Device helpers shared by the quantize and GEMM kernels of the FP8 linear layer.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "fp8lin.h"

namespace fp8lin {

constexpr int kTile = 128;          // quantize tile: 128 x 128 source elements
constexpr int kMxBlock = 32;        // MXFP8 block length
constexpr int kBwBlock = 128;       // blockwise block length

// First error wins: a device-side condition is recorded once, later ones are dropped.
__device__ __forceinline__ void report_status(int32_t* st, int32_t code) {
  if (st != nullptr) atomicCAS(st, 0, code);
}

// bf16 pair in a 32-bit word -> two floats (exact widening).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Magnitude maxima of packed bf16 pairs. The packed bf16 max propagates NaN, so a block or
// tensor holding a NaN reports a NaN magnitude (any bit pattern above +Inf, 0x7F80, once the
// sign is cleared); otherwise the result is the exact largest |x|.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t acc, uint32_t w) {
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&acc);
  __nv_bfloat162 b = __habs2(*reinterpret_cast<__nv_bfloat162*>(&w));
  __nv_bfloat162 m = __hmax2_nan(a, b);
  return *reinterpret_cast<uint32_t*>(&m);
}
// Fold a packed pair of magnitudes into one 15-bit magnitude pattern.
__device__ __forceinline__ uint32_t fold_bf16x2(uint32_t m) {
  return max(m & 0x7FFFu, (m >> 16) & 0x7FFFu);
}
// amax (as a float) from the 15-bit bf16 magnitude pattern.
__device__ __forceinline__ float amax_from_bits(uint32_t m) { return __uint_as_float(m << 16); }

// Two floats -> two E4M3 codes (round to nearest even, saturating to +-448; the hardware
// conversion). Byte 0 of the result is `a`, byte 1 is `b`.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// NaN inputs keep their sign: code 0x7F | sign. Only called when a NaN is present.
__device__ __forceinline__ uint32_t fix_nan_code(uint32_t code, float x) {
  if (x != x) code = 0x7Fu | ((__float_as_uint(x) >> 24) & 0x80u);
  return code;
}

// Eight bf16 (one 16-byte vector) times s -> eight codes packed in a uint2.
__device__ __forceinline__ uint2 encode8(uint4 v, float s, bool has_nan) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = __fmul_rn(bf16_lo(w[i]), s);
    const float b = __fmul_rn(bf16_hi(w[i]), s);
    uint32_t p = cvt_e4m3x2(a, b);
    if (has_nan) {
      p = fix_nan_code(p & 0xFFu, bf16_lo(w[i])) | (fix_nan_code(p >> 8, bf16_hi(w[i])) << 8);
    }
    c[i] = p;
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// 2^k as a float for k in [-149, 127] (exact; subnormal below 2^-126).
__device__ __forceinline__ float exp2i(int k) {
  return k >= -126 ? __uint_as_float(uint32_t(k + 127) << 23)
                   : __uint_as_float(1u << (k + 149));
}

// Per-tensor / per-block scale from an amax: s = fp32(448/amax) * 2^-margin, s = 1 for
// amax 0 / Inf / NaN, an infinite s becomes FLT_MAX. Returns s; *s_inv = fp32(1/s).
__device__ __forceinline__ float scale_from_amax(float amax, int margin, float* s_inv) {
  float s;
  if (!(amax > 0.0f) || !(amax <= 3.402823466e38f)) {
    s = 1.0f;
  } else {
    s = __fdiv_rn(448.0f, amax);
  }
  if (margin != 0) s = __fmul_rn(s, exp2i(-margin));
  if (s > 3.402823466e38f) s = 3.402823466e38f;
  *s_inv = __fdiv_rn(1.0f, s);
  return s;
}

// MXFP8 E8M0 byte from a block amax given as a 15-bit bf16 magnitude pattern: the smallest e
// with amax <= 448 * 2^e (448 = 1.75 * 2^8), -127 below 2^-126, clamped to [-127, 127];
// 0xFF (NaN) when the block holds Inf/NaN. Also returns the multiplier 2^-e (1 for NaN).
__device__ __forceinline__ uint32_t mx_scale_byte(uint32_t amax_bits, float* mult) {
  const uint32_t bexp = (amax_bits >> 7) & 0xFFu;     // biased exponent of the bf16 value
  if (bexp == 0xFFu) {
    *mult = 1.0f;
    return 0xFFu;
  }
  int e;
  if (bexp == 0u) {
    e = -127;
  } else {
    const int E = int(bexp) - 127;
    e = E - 8 + (((amax_bits & 0x7Fu) > 0x60u) ? 1 : 0);   // mantissa > 0.75 <=> m > 1.75
    e = max(-127, min(127, e));
  }
  *mult = exp2i(-e);
  return uint32_t(e + 127);
}

// Offset of the E8M0 byte of row r, 32-block kb in the tiled order used by the tensor
// core's block-scale path (512-byte atoms of 128 rows x 4 blocks).
__host__ __device__ __forceinline__ int64_t mx_scale_offset(int64_t r, int64_t kb, int64_t cols) {
  return ((r >> 7) * (cols >> 7) + (kb >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 +
         (kb & 3);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace fp8lin
