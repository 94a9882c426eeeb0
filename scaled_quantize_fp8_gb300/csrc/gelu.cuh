// GeLU of the transformer MLP block with the activation input kept in FP8 (Megatron Core
// "Low-Precision Training Guide"): a = gelu(h) in the forward pass, dh = da * gelu'(h) in the
// backward pass with h decoded from its MXFP8 row copy. Shared by the standalone MLP quantize
// kernels and the fused GEMM epilogues, so both produce bit-identical values.
//
// gelu(h) = h Phi(h) (exact erf form, no tanh approximation), evaluated in fp32 and rounded
// to bf16. The per-CTA shared-memory tables hold exactly the values the direct fp32
// evaluation returns, so a lookup and a direct evaluation never disagree.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "internal.cuh"

namespace fp8lin {

constexpr int kGeluExpLo = -14, kGeluExps = 18;       // gelu table: |h| in [2^-14, 2^4)
constexpr int kGeluEntries = kGeluExps * 128 * 2;     // bf16 input: 7-bit mantissa, sign
constexpr int kDgeluExpLo = -20, kDgeluExps = 24;     // gelu' table: |h| in [2^-20, 2^4)
constexpr int kDgeluEntries = kDgeluExps * 8 * 2;     // E4M3-derived input: 3-bit mantissa
// table bytes, rounded up to 1 KiB multiples so buffers behind them stay aligned
constexpr uint32_t kGeluTableBytes = 9216;
constexpr uint32_t kDgeluTableBytes = 2048;
static_assert(kGeluEntries * 2 <= int(kGeluTableBytes), "gelu table size");
static_assert(kDgeluEntries * 4 <= int(kDgeluTableBytes), "gelu' table size");

__device__ __forceinline__ uint32_t bf16_rn_bits(float f) {
  return uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(f)));
}
// Two floats rounded to bf16 in one conversion (low half = a), the same rounding as above.
__device__ __forceinline__ uint32_t bf16x2_rn_bits(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// E4M3 code pair -> two floats (exact, through the hardware f16x2 conversion).
__device__ __forceinline__ float2 e4m3x2_to_f2(uint16_t codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
  const __half2 h = *reinterpret_cast<const __half2*>(&h2);
  return __half22float2(h);
}

// Standard normal CDF Phi(h) = 0.5 erfc(-h / sqrt 2) in fp32, and optionally exp(-h^2 / 2).
// erfc(z), z >= 0, uses the Chebyshev-fitted form of Numerical Recipes ("erfcc", Press et al.,
// Numerical Recipes in C, 2nd ed., section 6.2): erfc(z) = t exp(-z^2 + P(t)), t = 1/(1 + z/2),
// with a stated fractional error below 1.2e-7 for all z >= 0. For h >= 0, Phi = 1 - erfc/2.
// The fast exponential is exact enough here (bf16 output); below h = -13 its result would be
// flushed, so that rare tail takes the full-range expf.
__device__ __forceinline__ float phi_cdf(float h, float* gauss) {
  const float z = fabsf(h) * 0.70710678118654752f;
  const float t = __fdividef(1.0f, fmaf(0.5f, z, 1.0f));
  float P = 0.17087277f;
  P = fmaf(P, t, -0.82215223f);
  P = fmaf(P, t, 1.48851587f);
  P = fmaf(P, t, -1.13520398f);
  P = fmaf(P, t, 0.27886807f);
  P = fmaf(P, t, -0.18628806f);
  P = fmaf(P, t, 0.09678418f);
  P = fmaf(P, t, 0.37409196f);
  P = fmaf(P, t, 1.00002368f);
  P = fmaf(P, t, -1.26551223f);
  const float z2 = z * z;
  const float arg = P - z2;
  const float e = z > 9.0f ? expf(arg) : __expf(arg);
  const float half_erfc = 0.5f * t * e;
  if (gauss != nullptr) *gauss = 0.3989422804014327f * (z > 9.0f ? expf(-z2) : __expf(-z2));
  return h >= 0.0f ? 1.0f - half_erfc : half_erfc;
}
// gelu(h) = h Phi(h); gelu'(h) = Phi(h) + h phi(h), phi(h) = exp(-h^2/2) / sqrt(2 pi).
__device__ __forceinline__ float gelu_f32(float h) { return h * phi_cdf(h, nullptr); }
__device__ __forceinline__ float gelu_grad_f32(float h) {
  // A dequantised FP8 value can exceed the fp32 range (a code near 448 times 2^120); its
  // gelu' is then the limit: 1 above, +0 below. (Inf/NaN inputs never get here as such: their
  // MXFP8 block carries the NaN scale.)
  if (fabsf(h) > 3.402823466e38f) return h > 0.0f ? 1.0f : 0.0f;
  float g;
  const float c = phi_cdf(h, &g);
  return fmaf(h, g, c);
}

// Direct evaluations for inputs outside the tables: rare, kept out of line so the unrolled
// tile loop stays small enough for the instruction cache.
static __device__ __noinline__ uint32_t gelu_bf16_direct(uint32_t hb) {
  return bf16_rn_bits(gelu_f32(__uint_as_float(hb << 16)));
}
static __device__ __noinline__ float gelu_grad_direct(float h) { return gelu_grad_f32(h); }

// gelu over bf16 inputs through the CTA's shared-memory table: every bf16 h with |h| in
// [2^-14, 2^4) has an entry holding bf16(gelu_f32(h)), so the lookup returns exactly what the
// direct evaluation would; other inputs (tiny, large, Inf/NaN) are evaluated directly.
__device__ __forceinline__ uint32_t gelu_table_lookup(const void* table, uint32_t hb) {
  const uint32_t e = ((hb >> 7) & 0xFFu) - uint32_t(kGeluExpLo + 127);
  if (e < uint32_t(kGeluExps)) {
    const uint32_t idx = (e << 8) | ((hb & 0x7Fu) << 1) | (hb >> 15);
    return reinterpret_cast<const uint16_t*>(table)[idx];
  }
  return gelu_bf16_direct(hb);
}
// gelu'(h) for h decoded from an E4M3 code times a power of two (at most 3 mantissa bits):
// table entries hold gelu_grad_f32 of each such value with |h| in [2^-20, 2^4); zero gives 1/2;
// anything else is evaluated directly.
__device__ __forceinline__ float dgelu_table_lookup(const void* table, float h) {
  const uint32_t bits = __float_as_uint(h);
  const uint32_t e = ((bits >> 23) & 0xFFu) - uint32_t(kDgeluExpLo + 127);
  if (e < uint32_t(kDgeluExps)) {
    const uint32_t idx = (e << 4) | (((bits >> 20) & 7u) << 1) | (bits >> 31);
    return reinterpret_cast<const float*>(table)[idx];
  }
  if ((bits & 0x7FFFFFFFu) == 0u) return 0.5f;
  return gelu_grad_direct(h);
}

// Fill the tables cooperatively (thread `tid` of `nthreads`); the caller synchronises.
__device__ __forceinline__ void gelu_table_fill(void* table, int tid, int nthreads) {
  uint16_t* tb = reinterpret_cast<uint16_t*>(table);
  for (int idx = tid; idx < kGeluEntries; idx += nthreads) {
    const uint32_t bits = (uint32_t(idx & 1) << 15) |
                          (uint32_t((idx >> 8) + kGeluExpLo + 127) << 7) |
                          uint32_t((idx >> 1) & 0x7F);
    tb[idx] = uint16_t(bf16_rn_bits(gelu_f32(__uint_as_float(bits << 16))));
  }
}
__device__ __forceinline__ void dgelu_table_fill(void* table, int tid, int nthreads) {
  float* tb = reinterpret_cast<float*>(table);
  for (int idx = tid; idx < kDgeluEntries; idx += nthreads) {
    const uint32_t bits = (uint32_t(idx & 1) << 31) |
                          (uint32_t((idx >> 4) + kDgeluExpLo + 127) << 23) |
                          (uint32_t((idx >> 1) & 7) << 20);
    tb[idx] = gelu_grad_f32(__uint_as_float(bits));
  }
}

// Table lookups for a word of two bf16 without branching: each half's index is its bits
// rotated left by one ((magnitude << 1) | sign, the table order) minus the first entry's, so
// inputs outside the table wrap to indices >= kGeluEntries. Those are clamped (a wrong but
// harmless read) and reported through *miss (the running maximum of the indices): a caller
// that sees *miss >= kGeluEntries recomputes the word with gelu_bf16x2.
__device__ __forceinline__ uint32_t gelu_bf16x2_nobranch(const void* table, uint32_t w,
                                                         uint32_t* miss) {
  constexpr uint32_t kBias = 0x10000u - (uint32_t(kGeluExpLo + 127) << 8);
  const uint32_t r = ((w << 1) & 0xFFFEFFFEu) | ((w >> 15) & 0x00010001u);
  const uint32_t ilo = (r + kBias) & 0xFFFFu;
  const uint32_t ihi = (r + (kBias << 16)) >> 16;
  *miss = max(*miss, max(ilo, ihi));
  const uint16_t* tb = reinterpret_cast<const uint16_t*>(table);
  const uint32_t last = uint32_t(kGeluEntries - 1);
  return uint32_t(tb[min(ilo, last)]) | (uint32_t(tb[min(ihi, last)]) << 16);
}

// gelu over a word of two bf16 (low half first).
__device__ __forceinline__ uint32_t gelu_bf16x2(const void* table, uint32_t w) {
  return gelu_table_lookup(table, w & 0xFFFFu) | (gelu_table_lookup(table, w >> 16) << 16);
}

// dh = bf16(da * gelu'(h)) for two elements: da as a bf16 pair, h as an E4M3 code pair times
// the block's power-of-two scale hs (NaN for a NaN block).
__device__ __forceinline__ uint32_t dgelu_bf16x2(const void* table, uint32_t da, uint16_t hcodes,
                                                 float hs) {
  const float2 hv = e4m3x2_to_f2(hcodes);
  const float d0 = __fmul_rn(__uint_as_float(da << 16),
                             dgelu_table_lookup(table, __fmul_rn(hv.x, hs)));
  const float d1 = __fmul_rn(__uint_as_float(da & 0xFFFF0000u),
                             dgelu_table_lookup(table, __fmul_rn(hv.y, hs)));
  return bf16x2_rn_bits(d0, d1);
}

// gelu'(h) as the standalone kernels define it: 1/2 at h = +-0, gelu_grad_f32 elsewhere (the
// values their table lookups return).
__device__ __forceinline__ float gelu_grad_value(float h) {
  return (__float_as_uint(h) & 0x7FFFFFFFu) == 0u ? 0.5f : gelu_grad_f32(h);
}

// gelu' by (E8M0 scale byte, E4M3 code) for the fused dgrad epilogue. Within one MXFP8 block the
// scale byte is fixed, so h = decode(code) * 2^(sb - 127) is a function of the code byte alone:
// row sb - kDgeluSbLo of the table holds gelu_grad_value of each of the 256 codes (zero,
// subnormals and NaN included), and the per-element work is a single indexed load. Blocks whose
// scale byte falls outside the rows (|h| above about 2^5 or below 2^-17 in the whole block) take
// the direct evaluation.
constexpr int kDgeluSbLo = 110, kDgeluSbRows = 16;
constexpr uint32_t kDgeluCodeTableBytes = kDgeluSbRows * 256 * 4;

__device__ __forceinline__ void dgelu_code_table_fill(void* table, int tid, int nthreads) {
  float* tb = reinterpret_cast<float*>(table);
  for (int idx = tid; idx < kDgeluSbRows * 256; idx += nthreads) {
    const int sb = kDgeluSbLo + (idx >> 8);
    const float hv = e4m3x2_to_f2(uint16_t(idx & 0xFF)).x;
    tb[idx] = gelu_grad_value(__fmul_rn(hv, exp2i(sb - 127)));
  }
}

// dh for two elements of a block outside the table rows: direct evaluation (rare, out of line).
static __device__ __noinline__ uint32_t dgelu_bf16x2_direct(uint32_t da, uint32_t hcodes,
                                                           float hs) {
  const float2 hv = e4m3x2_to_f2(uint16_t(hcodes));
  const float d0 = __fmul_rn(__uint_as_float(da << 16), gelu_grad_value(__fmul_rn(hv.x, hs)));
  const float d1 =
      __fmul_rn(__uint_as_float(da & 0xFFFF0000u), gelu_grad_value(__fmul_rn(hv.y, hs)));
  return bf16x2_rn_bits(d0, d1);
}

}  // namespace fp8lin
