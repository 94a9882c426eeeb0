// Quantize-cast of fp32 master weights straight to E4M3 (no bf16 rounding on the way): the
// optimizer keeps fp32 weights and the forward pass needs their FP8 copies each step
// (cast_master_weights_to_fp8 in the training stack the Megatron Core "Low-Precision Training
// Guide" builds on). The recipes and their readings are those of the bf16 quantize kernels
// (tensorwise, delayed, MXFP8 1x32, blockwise 128x128 for weights); only the input differs:
// amaxes are taken over the fp32 values and codes are encode(fp32(x * s)).
//
// One CTA (256 threads) per 128 x 128 source tile: the fp32 tile is staged in shared memory
// (rows padded to 132 floats so a warp reading one row or one column hits distinct banks);
// thread (r, h) writes row r's codes for columns 64h .. 64h+63, thread (c, h) the column copy
// of column c over rows 64h .. 64h+63, 32 codes (one 32-byte sector) at a time. Weights are a
// small share of a step's bytes, so this kernel favours simplicity over the TMA pipeline of
// the bf16 quantizer.
#include <algorithm>

#include "common.cuh"
#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace fp8lin {

enum MMode : int { M_TENSOR = 0, M_MX = 1, M_BW128 = 2 };

struct MasterParams {
  const float* x;             // [R][C] fp32
  int64_t R, C;
  int tiles_c, tiles_r;
  uint8_t* row;               // [R][C] codes or null
  uint8_t* col;               // [C][R] codes or null
  void* row_scale;            // MXFP8 E8M0 (tiled atoms) / 128x128 s_inv grid [R/128][C/128]
  void* col_scale;            // ... of the column copy ([C/128][R/128] for 128x128)
  const float* scale_in;      // delayed: device scale to cast with
  const uint32_t* part_in;    // tensorwise: per-CTA 31-bit magnitude maxima
  int n_part_in;
  float* amax_out;            // tensorwise: written by CTA 0
  float* scale_out;
  float* scale_inv_out;
  uint32_t* part_out;         // delayed: this tile's 31-bit magnitude maximum
  int margin;
  bool v8;                    // row and column copies start on 32-byte boundaries
};

constexpr int kMLd = 132;     // padded row length of the shared tile (floats)
constexpr uint32_t kMasterSmem = 128 * kMLd * 4;

__device__ __forceinline__ uint32_t mag31(float x) { return __float_as_uint(x) & 0x7FFFFFFFu; }

// E8M0 byte from an fp32 block amax given as its 31-bit magnitude pattern: the smallest e with
// amax <= 448 * 2^e (e = E - 8, plus one when the mantissa exceeds 1.75), -127 below 2^-126,
// 0xFF for an Inf/NaN block; *mult = 2^-e (1 for NaN). A finite fp32 amax never exceeds e = 120.
__device__ __forceinline__ uint32_t mx_scale_byte_f32(uint32_t mag, float* mult) {
  const int bexp = int(mag >> 23);
  int e = bexp - 135 + int((mag & 0x7FFFFFu) > 0x600000u);
  e = max(e, -127);
  const bool nan = bexp == 0xFF;
  *mult = nan ? 1.0f : __uint_as_float(uint32_t(127 - e) << 23);
  return nan ? 0xFFu : uint32_t(e + 127);
}

// 32 fp32 values times s -> 32 E4M3 codes (NaN inputs keep their sign), stored as one segment.
__device__ __forceinline__ void encode32_store(const float* v, float s, bool has_nan,
                                               uint8_t* dst, bool lo_ok, bool hi_ok, bool v8) {
  uint32_t c[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float2 a = __fmul2_rn(make_float2(v[4 * q], v[4 * q + 1]), make_float2(s, s));
    const float2 b = __fmul2_rn(make_float2(v[4 * q + 2], v[4 * q + 3]), make_float2(s, s));
    c[q] = cvt_e4m3x4(a.x, a.y, b.x, b.y);
    if (has_nan) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (v[4 * q + k] != v[4 * q + k])
          c[q] = (c[q] & ~(0xFFu << (8 * k))) |
                 ((0x7Fu | ((__float_as_uint(v[4 * q + k]) >> 24) & 0x80u)) << (8 * k));
    }
  }
  store_seg32(dst, make_uint4(c[0], c[1], c[2], c[3]), make_uint4(c[4], c[5], c[6], c[7]), lo_ok,
              hi_ok, v8);
}

__device__ __forceinline__ uint32_t block_max_256(uint32_t v, uint32_t* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  uint32_t m = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) m = max(m, red[i]);
  return m;
}

template <int MODE>
__global__ void __launch_bounds__(256) quantize_master_kernel(const MasterParams p) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float4 msm_raw[];
  float* tile = reinterpret_cast<float*>(msm_raw);
  __shared__ uint32_t red[8];
  const int t = threadIdx.x;
  const int tr = int(blockIdx.x) / p.tiles_c, tc = int(blockIdx.x) % p.tiles_c;
  const int64_t r0 = int64_t(tr) * 128, c0 = int64_t(tc) * 128;

  // ---- stage the fp32 tile (zeros outside the tensor): all 16 of a thread's 16-byte copies
  // in flight at once, global -> shared without passing through registers
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int idx = i * 256 + t, r = idx >> 5, c4 = idx & 31;
    const bool in = r0 + r < p.R && c0 + 4 * c4 < p.C;
    const float* src = in ? p.x + (r0 + r) * p.C + c0 + 4 * c4 : p.x;
    ptx::cp_async_16_zfill(tile + r * kMLd + 4 * c4, src, in ? 16u : 0u);
  }
  ptx::cp_async_commit();
  ptx::cp_async_wait<0>();
  __syncthreads();

  const int r = t >> 1, h = t & 1;          // row pass: row r, columns 64h .. 64h+63
  // ---- tile-wide / tensor-wide scale
  float s = 1.0f, sinv = 1.0f;
  bool nan_all = false;
  if constexpr (MODE != M_MX) {
    uint32_t m = 0;
#pragma unroll 8
    for (int k = 0; k < 64; ++k) m = max(m, mag31(tile[r * kMLd + 64 * h + k]));
    const uint32_t tm = block_max_256(m, red);
    if constexpr (MODE == M_BW128) {
      nan_all = tm > 0x7F800000u;
      s = scale_from_amax(__uint_as_float(tm), p.margin, &sinv);
      if (t == 0) {
        if (p.row_scale) reinterpret_cast<float*>(p.row_scale)[tr * p.tiles_c + tc] = sinv;
        if (p.col_scale) reinterpret_cast<float*>(p.col_scale)[tc * p.tiles_r + tr] = sinv;
      }
    } else if (p.scale_in != nullptr) {
      s = *p.scale_in;                      // delayed: cast with the history's scale
      if (t == 0) p.part_out[blockIdx.x] = tm;
      nan_all = tm > 0x7F800000u;
    } else {
      uint32_t g = 0;                       // tensorwise: reduce the per-CTA partials
      for (int i = t; i < p.n_part_in; i += 256) g = max(g, p.part_in[i]);
      g = block_max_256(g, red);
      nan_all = g > 0x7F800000u;
      s = scale_from_amax(__uint_as_float(g), p.margin, &sinv);
      if (blockIdx.x == 0 && t == 0) {
        *p.amax_out = __uint_as_float(g);
        *p.scale_out = s;
        *p.scale_inv_out = sinv;
      }
    }
  }

  // ---- row-wise copy
  if (p.row != nullptr && r0 + r < p.R) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int64_t cc = c0 + 64 * h + 32 * j;
      if (cc >= p.C) break;
      float v[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 f = *reinterpret_cast<const float4*>(tile + r * kMLd + 64 * h + 32 * j + 4 * q);
        v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
      }
      float sc = s;
      bool nan = nan_all;
      if constexpr (MODE == M_MX) {
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < 32; ++k) m = max(m, mag31(v[k]));
        const uint32_t sb = mx_scale_byte_f32(m, &sc);
        nan = m > 0x7F800000u;
        reinterpret_cast<uint8_t*>(p.row_scale)[mx_scale_offset(r0 + r, cc >> 5, p.C)] =
            uint8_t(sb);
      }
      encode32_store(v, sc, nan, p.row + (r0 + r) * p.C + cc, true, cc + 16 < p.C, p.v8);
    }
  }

  // ---- column-wise copy: column c over rows 64h .. 64h+63
  const int c = t & 127, hc = t >> 7;
  if (p.col != nullptr && c0 + c < p.C) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int64_t rr = r0 + 64 * hc + 32 * j;
      if (rr >= p.R) break;
      float v[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = tile[(64 * hc + 32 * j + k) * kMLd + c];
      float sc = s;
      bool nan = nan_all;
      if constexpr (MODE == M_MX) {
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < 32; ++k) m = max(m, mag31(v[k]));
        const uint32_t sb = mx_scale_byte_f32(m, &sc);
        nan = m > 0x7F800000u;
        reinterpret_cast<uint8_t*>(p.col_scale)[mx_scale_offset(c0 + c, rr >> 5, p.R)] =
            uint8_t(sb);
      }
      encode32_store(v, sc, nan, p.col + (c0 + c) * p.R + rr, true, rr + 16 < p.R, p.v8);
    }
  }
}

// Tensorwise first pass over fp32: per-CTA max of the 31-bit magnitudes (a NaN pattern
// compares above +Inf, so a NaN anywhere makes the amax NaN).
__global__ void __launch_bounds__(512) amax_partial_f32_kernel(const float* __restrict__ x,
                                                               int64_t n_vec,
                                                               uint32_t* __restrict__ part) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ uint32_t red[16];
  uint32_t m = 0;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const float4* x4 = reinterpret_cast<const float4*>(x);
  auto fold = [](uint32_t acc, float4 v) {
    return max(max(acc, max(mag31(v.x), mag31(v.y))), max(mag31(v.z), mag31(v.w)));
  };
  int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n_vec; i += 4 * stride) {       // four loads in flight per thread
    const float4 a = __ldg(x4 + i), b = __ldg(x4 + i + stride);
    const float4 c = __ldg(x4 + i + 2 * stride), d = __ldg(x4 + i + 3 * stride);
    m = fold(fold(fold(fold(m, a), b), c), d);
  }
  for (; i < n_vec; i += stride) m = fold(m, __ldg(x4 + i));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = 0;
    for (int k = 0; k < int(blockDim.x >> 5); ++k) r = max(r, red[k]);
    part[blockIdx.x] = r;
  }
}

// Delayed: reduce the per-tile 31-bit maxima into the tensor's amax.
__global__ void __launch_bounds__(1024) amax_finalize_f32_kernel(const uint32_t* __restrict__ part,
                                                                 int n, float* __restrict__ amax) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ uint32_t red[32];
  uint32_t m = 0;
  // eight independent loads in flight per thread
  for (int base = threadIdx.x; base < n; base += 8 * int(blockDim.x)) {
    uint32_t v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int j = base + k * int(blockDim.x);
      v[k] = j < n ? __ldg(part + j) : 0u;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) m = max(m, v[k]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = 0;
    for (int k = 0; k < int(blockDim.x >> 5); ++k) r = max(r, red[k]);
    *amax = __uint_as_float(r);
  }
}

__global__ void master_empty_kernel(float* amax, float* scale, float* scale_inv, int margin) {
  pdl_launch_dependents();
  pdl_wait();
  if (amax) *amax = 0.0f;
  if (scale) {
    float si;
    *scale = scale_from_amax(0.0f, margin, &si);
    if (scale_inv) *scale_inv = si;
  }
}

template <int MODE>
static cudaError_t launch_master(MasterParams p, cudaStream_t st) {
  auto a32 = [](const void* q) { return q == nullptr || reinterpret_cast<uintptr_t>(q) % 32 == 0; };
  p.v8 = a32(p.row) && a32(p.col) && p.C % 32 == 0 && p.R % 32 == 0;
  static ContextOnce attr_done{};
  const cudaError_t ae = once_per_context(attr_done, [] {
    return cudaFuncSetAttribute(quantize_master_kernel<MODE>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, int(kMasterSmem));
  });
  if (ae != cudaSuccess) return ae;
  return launch_kernel(quantize_master_kernel<MODE>, dim3(unsigned(p.tiles_r * p.tiles_c)),
                       dim3(256), kMasterSmem, st, nullptr, p);
}

cudaError_t quantize_master_launch(int kind, int margin, const float* x, int64_t R, int64_t C,
                                   bool want_row, bool want_col, fp8_tensor* out,
                                   void* workspace, cudaStream_t st) {
  if (R == 0 || C == 0) {
    if (kind == FP8_RECIPE_TENSORWISE || kind == FP8_RECIPE_DELAYED) {
      return launch_kernel(master_empty_kernel, dim3(1), dim3(1), 0, st, nullptr, out->amax,
                           kind == FP8_RECIPE_TENSORWISE ? out->scale : nullptr, out->scale_inv,
                           margin);
    }
    return cudaSuccess;
  }
  MasterParams p{};
  p.x = x;
  p.R = R;
  p.C = C;
  p.tiles_r = int((R + 127) / 128);
  p.tiles_c = int((C + 127) / 128);
  p.row = want_row ? out->row : nullptr;
  p.col = want_col ? out->col : nullptr;
  p.row_scale = want_row ? out->row_scale : nullptr;
  p.col_scale = want_col ? out->col_scale : nullptr;
  p.margin = margin;
  switch (kind) {
    case FP8_RECIPE_TENSORWISE: {
      // as many partials as the bf16 path uses, so fp8_workspace_bytes covers both
      const int ctas = amax_partial_ctas(R * C / 8);
      uint32_t* part = reinterpret_cast<uint32_t*>(workspace);
      const cudaError_t e = launch_kernel(amax_partial_f32_kernel, dim3(ctas), dim3(512), 0, st,
                                          nullptr, x, R * C / 4, part);
      if (e != cudaSuccess) return e;
      p.part_in = part;
      p.n_part_in = ctas;
      p.amax_out = out->amax;
      p.scale_out = out->scale;
      p.scale_inv_out = out->scale_inv;
      return launch_master<M_TENSOR>(p, st);
    }
    case FP8_RECIPE_DELAYED: {
      p.scale_in = out->scale;
      p.part_out = reinterpret_cast<uint32_t*>(workspace);
      cudaError_t e = launch_master<M_TENSOR>(p, st);
      if (e != cudaSuccess) return e;
      return launch_kernel(amax_finalize_f32_kernel, dim3(1), dim3(1024), 0, st, nullptr,
                           static_cast<const uint32_t*>(p.part_out), p.tiles_r * p.tiles_c,
                           out->amax);
    }
    case FP8_RECIPE_MXFP8:
      return launch_master<M_MX>(p, st);
    case FP8_RECIPE_BLOCKWISE:
      return launch_master<M_BW128>(p, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fp8lin
