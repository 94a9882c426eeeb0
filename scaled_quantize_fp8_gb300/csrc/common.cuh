// Device helpers shared by the quantize and GEMM kernels of the FP8 linear layer.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "fp8lin.h"

namespace fp8lin {

constexpr int kTile = 128;          // quantize tile: 128 x 128 source elements

// FP8 storage formats: E4M3 for everything, E5M2 for gradients under the hybrid format.
enum Fp8Fmt : int { F8_E4M3 = 0, F8_E5M2 = 1 };
template <int F8>
__host__ __device__ constexpr float fp8_max() { return F8 == F8_E5M2 ? 57344.0f : 448.0f; }
constexpr int kMxBlock = 32;        // MXFP8 block length
constexpr int kBwBlock = 128;       // blockwise block length

// First error wins: a device-side condition is recorded once, later ones are dropped.
// Programmatic dependent launch (no-ops when the kernel was launched without the attribute):
// let the next kernel in the stream begin launching, and wait until the previous kernel has
// completed and its writes are visible (before this kernel's first global memory access).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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
    const float2 ab = __fmul2_rn(make_float2(bf16_lo(w[i]), bf16_hi(w[i])), make_float2(s, s));
    const float a = ab.x, b = ab.y;
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

// The scale alone (the first half of scale_from_amax below, for callers that do not store
// s_inv).
__device__ __forceinline__ float scale_only_from_amax(float amax, int margin,
                                                      float fmax = 448.0f, bool pow2 = false) {
  float s;
  if (!(amax > 0.0f) || !(amax <= 3.402823466e38f)) {
    s = 1.0f;
  } else {
    s = __fdiv_rn(fmax, amax);
  }
  if (margin != 0) s = __fmul_rn(s, exp2i(-margin));
  if (s > 3.402823466e38f) s = 3.402823466e38f;
  if (pow2) {
    const uint32_t b = __float_as_uint(s);
    s = __uint_as_float(b >= 0x00800000u ? (b & 0xFF800000u)
                                         : (b == 0u ? 0u : (0x80000000u >> __clz(b))));
  }
  return s;
}

// Per-tensor / per-block scale from an amax: s = fp32(fmax/amax) * 2^-margin (fmax = 448 for
// E4M3, 57344 for E5M2), rounded down to a power of two when pow2 is set, s = 1 for
// amax 0 / Inf / NaN, an infinite s becomes FLT_MAX. Returns s; *s_inv = fp32(1/s).
__device__ __forceinline__ float scale_from_amax(float amax, int margin, float* s_inv,
                                                 float fmax = 448.0f, bool pow2 = false) {
  float s;
  if (!(amax > 0.0f) || !(amax <= 3.402823466e38f)) {
    s = 1.0f;
  } else {
    s = __fdiv_rn(fmax, amax);
  }
  if (margin != 0) s = __fmul_rn(s, exp2i(-margin));
  if (s > 3.402823466e38f) s = 3.402823466e38f;
  if (pow2) {
    // largest power of two <= s: keep the exponent (normal), or the top set bit (subnormal)
    const uint32_t b = __float_as_uint(s);
    s = __uint_as_float(b >= 0x00800000u ? (b & 0xFF800000u)
                                         : (b == 0u ? 0u : (0x80000000u >> __clz(b))));
  }
  *s_inv = __fdiv_rn(1.0f, s);
  return s;
}

// MXFP8 E8M0 byte from a block amax given as a 15-bit bf16 magnitude pattern: the smallest e
// with amax <= 448 * 2^e (448 = 1.75 * 2^8, so e = E - 8, plus one when the mantissa exceeds
// 1.75), -127 below 2^-126, clamped to [-127, 127] (a finite bf16 amax never exceeds e = 120);
// 0xFF (NaN) when the block holds Inf/NaN. Also returns the multiplier 2^-e (1 for NaN).
__device__ __forceinline__ uint32_t mx_scale_byte(uint32_t amax_bits, float* mult) {
  const int bexp = int((amax_bits >> 7) & 0xFFu);
  int e = bexp - 135 + int((amax_bits & 0x7Fu) > 0x60u);
  e = max(e, -127);
  const bool nan = bexp == 0xFF;
  *mult = nan ? 1.0f : __uint_as_float(uint32_t(127 - e) << 23);
  return nan ? 0xFFu : uint32_t(e + 127);
}

// E8M0 byte of a power-of-two dequantisation factor 2^k, k in [-127, 127]: the float's biased
// exponent field (2^-127, a float subnormal, has field 0, which is also its E8M0 byte).
__device__ __forceinline__ uint32_t e8m0_of_pow2(float s_inv) {
  return (__float_as_uint(s_inv) >> 23) & 0xFFu;
}

// Four floats -> four E4M3 codes in one word (byte i holds the code of x_i).
__device__ __forceinline__ uint32_t cvt_e4m3x4(float x0, float x1, float x2, float x3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  return r;
}

// Four floats -> four E5M2 codes (round to nearest even, saturating to +-57344).
__device__ __forceinline__ uint32_t cvt_e5m2x4(float x0, float x1, float x2, float x3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e5m2x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e5m2x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  return r;
}
template <int F8>
__device__ __forceinline__ uint32_t cvt_fp8x4(float x0, float x1, float x2, float x3) {
  if constexpr (F8 == F8_E5M2) return cvt_e5m2x4(x0, x1, x2, x3);
  else return cvt_e4m3x4(x0, x1, x2, x3);
}

// Two words of packed bf16 (4 values) times s -> one word of 4 codes.
// Two packed fp32 multiplies, each lane rounded like __fmul_rn (the quantize kernels, which
// have registers to spare); encode4_scalar is the same arithmetic in four scalar multiplies,
// for register-bound callers (a packed operand needs an aligned register pair).
template <int F8 = F8_E4M3>
__device__ __forceinline__ uint32_t encode4_scalar(uint32_t w0, uint32_t w1, float s) {
  return cvt_fp8x4<F8>(__fmul_rn(bf16_lo(w0), s), __fmul_rn(bf16_hi(w0), s),
                       __fmul_rn(bf16_lo(w1), s), __fmul_rn(bf16_hi(w1), s));
}
template <int F8 = F8_E4M3>
__device__ __forceinline__ uint32_t encode4(uint32_t w0, uint32_t w1, float s) {
  const float2 s2 = make_float2(s, s);
  const float2 a = __fmul2_rn(make_float2(bf16_lo(w0), bf16_hi(w0)), s2);
  const float2 b = __fmul2_rn(make_float2(bf16_lo(w1), bf16_hi(w1)), s2);
  return cvt_fp8x4<F8>(a.x, a.y, b.x, b.y);
}

// Give the codes of NaN inputs the NaN code with the input's sign (rare path).
__device__ __forceinline__ uint32_t fix_nan4(uint32_t code, uint32_t w0, uint32_t w1) {
  const uint32_t in[4] = {w0 & 0xFFFFu, w0 >> 16, w1 & 0xFFFFu, w1 >> 16};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if ((in[k] & 0x7FFFu) > 0x7F80u) {
      const uint32_t c = 0x7Fu | ((in[k] >> 8) & 0x80u);
      code = (code & ~(0xFFu << (8 * k))) | (c << (8 * k));
    }
  }
  return code;
}

// Offset of the E8M0 byte of row r, 32-block kb in the tiled order used by the tensor
// core's block-scale path (512-byte atoms of 128 rows x 4 blocks).
__host__ __device__ __forceinline__ int64_t mx_scale_offset(int64_t r, int64_t kb, int64_t cols) {
  return ((r >> 7) * (cols >> 7) + (kb >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 +
         (kb & 3);
}

// One 32-byte global store (256-bit vector; the address must be 32-byte aligned).
__device__ __forceinline__ void stg_v8(void* p, uint4 a, uint4 b) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x),
               "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}
// A 32-byte segment whose halves may fall outside the tensor: whole-sector store when
// allowed (aligned and both halves in range), else one 16-byte store per valid half.
__device__ __forceinline__ void store_seg32(void* p, uint4 a, uint4 b, bool lo_ok, bool hi_ok,
                                            bool v8) {
  if (v8 && lo_ok && hi_ok) {
    stg_v8(p, a, b);
  } else {
    if (lo_ok) reinterpret_cast<uint4*>(p)[0] = a;
    if (hi_ok) reinterpret_cast<uint4*>(p)[1] = b;
  }
}

// 16-byte read-only load with an L2 cache policy (see ptx::l2_evict_last_policy). Not
// volatile: the compiler may batch several of them ahead of their uses (read-only data).
__device__ __forceinline__ uint4 ldg_nc_v4_policy(const void* p, uint64_t policy) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p), "l"(policy));
  return v;
}
// The same without a policy, also free to be scheduled ahead of its uses.
__device__ __forceinline__ uint4 ldg_nc_v4_sched(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// Bring the L2 line holding p in from DRAM ahead of its use (no register holds anything).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace fp8lin
