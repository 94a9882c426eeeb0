// Quantize-cast kernels of the FP8 linear layer: bf16 -> E4M3 codes + scales, row-wise copy
// [R][C] and column-wise (transposed) copy [C][R], for the four recipes of the Megatron Core
// "Low-Precision Training Guide" (Recipe Reference: delayed, tensorwise, mxfp8, blockwise),
// plus the MLP activation variants that keep the GeLU input in FP8.
//
// One CTA (256 threads) owns a 128 x 128 source tile. It reads the tile once from HBM with
// 16-byte non-allocating loads, writes the row-wise codes straight from registers (a
// half-warp covers one 128-byte row segment), parks the bf16 tile in shared memory, and
// writes the column-wise codes from there (each thread emits 32 consecutive bytes of two
// transposed rows, i.e. whole 32-byte sectors). Scales are staged in shared memory and
// written as one coalesced block per tile. HBM traffic per element: 2 bytes read, 1 byte
// per copy written, plus the scales.
#include <algorithm>

#include "common.cuh"
#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace fp8lin {

enum QMode : int { Q_TENSOR = 0, Q_MX = 1, Q_BW1x128 = 2, Q_BW128 = 3 };
enum QEpi : int { EPI_NONE = 0, EPI_GELU = 1, EPI_DGELU = 2 };

struct QuantParams {
  const uint16_t* x;          // [R][C] bf16 (h for GELU, da for DGELU)
  int64_t R, C;
  int tiles_c;
  uint8_t* row;               // [R][C] codes or null
  uint8_t* col;               // [C][R] codes or null
  void* row_scale;
  void* col_scale;
  // per-tensor recipes
  const float* scale_in;      // delayed: device scale to cast with
  const uint32_t* part_in;    // tensorwise: per-CTA amax partials (15-bit bf16 magnitudes)
  int n_part_in;
  float* amax_out;            // tensorwise: CTA 0 writes amax/scale/scale_inv
  float* scale_out;
  float* scale_inv_out;
  uint32_t* part_out;         // delayed: this tile's amax partial
  int margin;
  // MLP epilogues
  int32_t* status;            // device status word (may be null)
  uint16_t* y_bf16;           // GELU: a = gelu(h) in bf16; DGELU: dh in bf16 (optional)
  uint8_t* aux_row;           // GELU: h row codes; DGELU: h row codes (read)
  uint8_t* aux_scale;         // GELU: h row E8M0 (written); DGELU: h row E8M0 (read)
};

__device__ __forceinline__ uint32_t bf16_rn_bits(float f) {
  return uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(f)));
}

// E4M3 code pair -> two floats (exact, through the hardware f16x2 conversion).
__device__ __forceinline__ float2 e4m3x2_to_f2(uint16_t codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
  const __half2 h = *reinterpret_cast<const __half2*>(&h2);
  return __half22float2(h);
}

__device__ __forceinline__ float gelu_f32(float h) { return h * normcdff(h); }
__device__ __forceinline__ float gelu_grad_f32(float h) {
  return normcdff(h) + h * (0.3989422804014327f * expf(-0.5f * h * h));
}

// Max of the 15-bit magnitudes of the eight bf16 in a vector.
__device__ __forceinline__ uint32_t vec_amax_bits(uint4 v) {
  uint32_t m = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(0u, v.x), v.y), v.z), v.w);
  return fold_bf16x2(m);
}

// Block-wide max of a per-thread value (256 threads), result broadcast to all threads.
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* red) {
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

// 32 column values (low or high halves of 32 words) times s -> 32 codes in two uint4.
__device__ __forceinline__ void encode_col32(const uint32_t* w, bool hi, float s, bool nan,
                                             uint4* out) {
  uint32_t c[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t pk = 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float x0 = hi ? bf16_hi(w[4 * j + 2 * k]) : bf16_lo(w[4 * j + 2 * k]);
      const float x1 = hi ? bf16_hi(w[4 * j + 2 * k + 1]) : bf16_lo(w[4 * j + 2 * k + 1]);
      uint32_t p = cvt_e4m3x2(__fmul_rn(x0, s), __fmul_rn(x1, s));
      if (nan) p = fix_nan_code(p & 0xFFu, x0) | (fix_nan_code(p >> 8, x1) << 8);
      pk |= p << (16 * k);
    }
    c[j] = pk;
  }
  out[0] = make_uint4(c[0], c[1], c[2], c[3]);
  out[1] = make_uint4(c[4], c[5], c[6], c[7]);
}

struct QuantSmem {
  uint32_t tile[2][128][64];        // double-buffered bf16 tile, [row][col/2] pairs (64 KiB)
  uint8_t sc_row[512];              // MXFP8 scale atom of the row copy
  uint8_t sc_col[512];              // ... of the column copy
  float scf_row[128];               // blockwise 1x128 s_inv staging
  float scf_col[128];
  uint32_t red[8];
  uint32_t red_col[4][128];
  uint64_t bar[2];                  // TMA completion, one per buffer
  int abort_flag;
};
constexpr uint64_t kQuantWaitBudget = 4000000000ull;   // ~2 s at 2 GHz
constexpr int kQuantCtasPerSm = 3;                     // 3 x ~69 KiB of shared memory

// Quantise one 128 x 128 tile held in shared memory (see the file comment for the scheme).
template <int MODE, int EPI>
__device__ __forceinline__ void quantize_one_tile(const QuantParams& p, QuantSmem& S,
                                                  uint32_t (*tile)[64], int tile_id,
                                                  float s_tensor, bool tensor_nan) {
  const int t = threadIdx.x;
  const int tr = tile_id / p.tiles_c, tc = tile_id % p.tiles_c;
  // 32-bit index arithmetic: the host guarantees R * C < 2^31.
  const uint32_t r0 = uint32_t(tr) * kTile, c0 = uint32_t(tc) * kTile;
  const int vcol = t & 15, rb = t >> 4;
  const uint32_t R = uint32_t(p.R), C = uint32_t(p.C);
  const bool col_ok = (c0 + 8 * vcol) < C;
  const uint32_t rowoff0 = (r0 + rb) * C + c0 + 8 * vcol;   // element offset of v[0]

  // ---- this thread's eight 16-byte vectors (out-of-range parts of the tile read as zero)
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = *reinterpret_cast<const uint4*>(&tile[rb + 16 * i][4 * vcol]);

  // ---- MLP epilogues: turn the input into the tensor to quantise
  if constexpr (EPI == EPI_GELU) {
    // h row copy (MXFP8, blocks of 32 along C) first, then a = bf16(gelu(h)).
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t m = vec_amax_bits(v[i]);
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
      float mult;
      const uint32_t b = mx_scale_byte(m, &mult);
      const uint32_t r = r0 + rb + 16 * i;
      const uint32_t off = rowoff0 + 16 * i * C;
      if (r < R && col_ok) {
        *reinterpret_cast<uint2*>(p.aux_row + off) = encode8(v[i], mult, m > 0x7F80u);
        if ((vcol & 3) == 0) p.aux_scale[mx_scale_offset(r, (c0 + 8 * vcol) >> 5, C)] = uint8_t(b);
      }
      uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w[k] = bf16_rn_bits(gelu_f32(bf16_lo(w[k]))) | (bf16_rn_bits(gelu_f32(bf16_hi(w[k]))) << 16);
      }
      v[i] = make_uint4(w[0], w[1], w[2], w[3]);
      if (p.y_bf16 != nullptr && r < R && col_ok)
        *reinterpret_cast<uint4*>(p.y_bf16 + off) = v[i];
      *reinterpret_cast<uint4*>(&tile[rb + 16 * i][4 * vcol]) = v[i];   // for the column pass
    }
  } else if constexpr (EPI == EPI_DGELU) {
    // dh = bf16(da * gelu'(h)) with h decoded from its MXFP8 row copy.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t r = r0 + rb + 16 * i;
      const uint32_t off = rowoff0 + 16 * i * C;
      if (r < R && col_ok) {
        const uint2 hc = *reinterpret_cast<const uint2*>(p.aux_row + off);
        const uint32_t sb = p.aux_scale[mx_scale_offset(r, (c0 + 8 * vcol) >> 5, C)];
        const float hs = sb == 0xFFu ? __uint_as_float(0x7FC00000u) : exp2i(int(sb) - 127);
        const uint32_t cw[2] = {hc.x, hc.y};
        uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 hv = e4m3x2_to_f2(uint16_t(cw[k >> 1] >> (16 * (k & 1))));
          const float h0 = __fmul_rn(hv.x, hs), h1 = __fmul_rn(hv.y, hs);
          const float d0 = __fmul_rn(bf16_lo(w[k]), gelu_grad_f32(h0));
          const float d1 = __fmul_rn(bf16_hi(w[k]), gelu_grad_f32(h1));
          w[k] = bf16_rn_bits(d0) | (bf16_rn_bits(d1) << 16);
        }
        v[i] = make_uint4(w[0], w[1], w[2], w[3]);
        if (p.y_bf16 != nullptr) *reinterpret_cast<uint4*>(p.y_bf16 + off) = v[i];
      }
      *reinterpret_cast<uint4*>(&tile[rb + 16 * i][4 * vcol]) = v[i];
    }
  }

  // ---- per-thread magnitude max
  uint32_t lmax = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) lmax = max(lmax, vec_amax_bits(v[i]));

  // ---- the tile-wide scale (per-tensor and 128x128 recipes)
  float s_tile = s_tensor, sinv_tile = 1.0f;
  bool tile_nan = tensor_nan;
  if constexpr (MODE == Q_TENSOR) {
    if (p.part_out != nullptr) {                              // delayed: record this tile's amax
      const uint32_t tm = block_max_u32(lmax, S.red);
      tile_nan = tm > 0x7F80u;
      if (t == 0) p.part_out[tile_id] = tm;
    }
  } else if constexpr (MODE == Q_BW128) {
    const uint32_t tm = block_max_u32(lmax, S.red);
    tile_nan = tm > 0x7F80u;
    s_tile = scale_from_amax(amax_from_bits(tm), p.margin, &sinv_tile);
    if (t == 0) {
      const int tiles_r = int((R + 127) >> 7);
      if (p.row_scale) reinterpret_cast<float*>(p.row_scale)[tr * p.tiles_c + tc] = sinv_tile;
      if (p.col_scale) reinterpret_cast<float*>(p.col_scale)[tc * tiles_r + tr] = sinv_tile;
    }
  }

  // ---- row-wise copy from registers
  if (p.row != nullptr) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t r = r0 + rb + 16 * i;
      const int lr = rb + 16 * i;
      uint2 codes;
      if constexpr (MODE == Q_TENSOR || MODE == Q_BW128) {
        codes = encode8(v[i], s_tile, tile_nan);
      } else if constexpr (MODE == Q_MX) {
        uint32_t m = vec_amax_bits(v[i]);
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
        float mult;
        const uint32_t b = mx_scale_byte(m, &mult);
        codes = encode8(v[i], mult, m > 0x7F80u);
        if ((vcol & 3) == 0) S.sc_row[(lr & 31) * 16 + (lr >> 5) * 4 + (vcol >> 2)] = uint8_t(b);
      } else {  // Q_BW1x128: the block is the whole 128-wide tile row (16 lanes)
        uint32_t m = vec_amax_bits(v[i]);
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        float sinv;
        const float s = scale_from_amax(amax_from_bits(m), p.margin, &sinv);
        codes = encode8(v[i], s, m > 0x7F80u);
        if (vcol == 0) S.scf_row[lr] = sinv;
      }
      if (r < R && col_ok) *reinterpret_cast<uint2*>(p.row + rowoff0 + 16 * i * C) = codes;
    }
  }

  if (p.col != nullptr) {
    if constexpr (EPI != EPI_NONE) __syncthreads();          // transformed tile written back

    // ---- column-wise copy: thread owns source columns 2pp, 2pp+1 and rows 32q .. 32q+31
    const int pp = t & 63, q = t >> 6;
    uint32_t w[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) w[j] = tile[32 * q + j][pp];
    uint32_t mw = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) mw = absmax_bf16x2(mw, w[j]);
    const uint32_t ma = mw & 0x7FFFu, mb = (mw >> 16) & 0x7FFFu;   // columns 2pp and 2pp+1

    float sa = s_tile, sb = s_tile;
    bool na = tile_nan, nb = tile_nan;
    if constexpr (MODE == Q_MX) {
      float fa, fb;
      const uint32_t ba = mx_scale_byte(ma, &fa), bb = mx_scale_byte(mb, &fb);
      sa = fa;
      sb = fb;
      na = ma > 0x7F80u;
      nb = mb > 0x7F80u;
      const int ca = 2 * pp, cb = 2 * pp + 1;
      S.sc_col[(ca & 31) * 16 + (ca >> 5) * 4 + q] = uint8_t(ba);
      S.sc_col[(cb & 31) * 16 + (cb >> 5) * 4 + q] = uint8_t(bb);
    } else if constexpr (MODE == Q_BW1x128) {
      S.red_col[q][2 * pp] = ma;
      S.red_col[q][2 * pp + 1] = mb;
      __syncthreads();
      const uint32_t fa = max(max(S.red_col[0][2 * pp], S.red_col[1][2 * pp]),
                              max(S.red_col[2][2 * pp], S.red_col[3][2 * pp]));
      const uint32_t fb = max(max(S.red_col[0][2 * pp + 1], S.red_col[1][2 * pp + 1]),
                              max(S.red_col[2][2 * pp + 1], S.red_col[3][2 * pp + 1]));
      float ia, ib;
      sa = scale_from_amax(amax_from_bits(fa), p.margin, &ia);
      sb = scale_from_amax(amax_from_bits(fb), p.margin, &ib);
      na = fa > 0x7F80u;
      nb = fb > 0x7F80u;
      if (q == 0) {
        S.scf_col[2 * pp] = ia;
        S.scf_col[2 * pp + 1] = ib;
      }
    }

    uint4 out[2];
    const uint32_t rr = r0 + 32 * q;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t c = c0 + 2 * pp + h;
      encode_col32(w, h == 1, h == 0 ? sa : sb, h == 0 ? na : nb, out);
      if (c < C) {
        uint8_t* dst = p.col + c * R + rr;
        if (rr < R) *reinterpret_cast<uint4*>(dst) = out[0];
        if (rr + 16 < R) *reinterpret_cast<uint4*>(dst + 16) = out[1];
      }
    }
  }

  // ---- scales of the copies written from staging
  if constexpr (MODE == Q_MX || MODE == Q_BW1x128) {
    __syncthreads();
    if constexpr (MODE == Q_MX) {
      const int tiles_r = int(R >> 7);
      if (t < 32 && p.row != nullptr)
        reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.row_scale) +
                                 (uint32_t(tr) * p.tiles_c + tc) * 512)[t] =
            reinterpret_cast<const uint4*>(S.sc_row)[t];
      if (t >= 32 && t < 64 && p.col != nullptr)
        reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.col_scale) +
                                 (uint32_t(tc) * tiles_r + tr) * 512)[t - 32] =
            reinterpret_cast<const uint4*>(S.sc_col)[t - 32];
    } else {
      if (t < 128 && p.row != nullptr)
        reinterpret_cast<float*>(p.row_scale)[uint32_t(tc) * R + r0 + t] = S.scf_row[t];
      if (t >= 128 && p.col != nullptr)
        reinterpret_cast<float*>(p.col_scale)[uint32_t(tr) * C + c0 + (t - 128)] =
            S.scf_col[t - 128];
    }
  }
}

// Bounded wait on a TMA completion barrier (all threads); false once the budget is spent.
__device__ __forceinline__ bool quant_wait(QuantSmem& S, int b, uint32_t parity, int32_t* st) {
  if (ptx::mbar_try_wait(&S.bar[b], parity)) return true;
  const uint64_t t0 = ptx::clock64_();
  while (!ptx::mbar_try_wait(&S.bar[b], parity)) {
    if (*reinterpret_cast<volatile int*>(&S.abort_flag)) return false;
    if (ptx::clock64_() - t0 > kQuantWaitBudget) {
      *reinterpret_cast<volatile int*>(&S.abort_flag) = 1;
      report_status(st, FP8_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Persistent quantize kernel: each CTA walks tiles blockIdx.x, +gridDim.x, ...; thread 0
// issues the TMA load of the next tile into the other buffer before the current one is
// processed, so HBM reads overlap the conversion and the stores.
template <int MODE, int EPI>
__global__ void __launch_bounds__(256, kQuantCtasPerSm) quantize_tile_kernel(const __grid_constant__ CUtensorMap tmX,
                                                            const QuantParams p) {
  extern __shared__ uint8_t qsm_raw[];
  QuantSmem& S = *reinterpret_cast<QuantSmem*>(
      (reinterpret_cast<uintptr_t>(qsm_raw) + 127) & ~uintptr_t(127));
  const int t = threadIdx.x;
  const int tiles_r = int((p.R + 127) >> 7);
  const int n_tiles = tiles_r * p.tiles_c;

  if (t == 0) {
    ptx::mbar_init(&S.bar[0], 1);
    ptx::mbar_init(&S.bar[1], 1);
    S.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();

  // per-tensor scale once per CTA: tensorwise from the amax partials, delayed from memory
  float s_tensor = 1.0f;
  bool tensor_nan = false;
  if constexpr (MODE == Q_TENSOR) {
    if (p.scale_in != nullptr) {
      s_tensor = *p.scale_in;
    } else {
      uint32_t m = 0;
      for (int i = t; i < p.n_part_in; i += 256) m = max(m, p.part_in[i]);
      m = block_max_u32(m, S.red);
      tensor_nan = m > 0x7F80u;
      float sinv;
      s_tensor = scale_from_amax(amax_from_bits(m), p.margin, &sinv);
      if (blockIdx.x == 0 && t == 0) {
        *p.amax_out = amax_from_bits(m);
        *p.scale_out = s_tensor;
        *p.scale_inv_out = sinv;
      }
    }
  }

  auto issue = [&](int tile_id, int b) {
    const int tr = tile_id / p.tiles_c, tc = tile_id % p.tiles_c;
    ptx::mbar_arrive_expect_tx(&S.bar[b], 128 * 128 * 2);
    ptx::tma_load_2d(&S.tile[b][0][0], &tmX, tc * kTile, tr * kTile, &S.bar[b]);
  };

  int tile = blockIdx.x;
  if (t == 0 && tile < n_tiles) issue(tile, 0);
  for (int i = 0; tile < n_tiles; ++i, tile += gridDim.x) {
    const int b = i & 1;
    const int next = tile + int(gridDim.x);
    if (t == 0 && next < n_tiles) issue(next, b ^ 1);
    if (!quant_wait(S, b, uint32_t(i >> 1) & 1u, p.status)) break;
    quantize_one_tile<MODE, EPI>(p, S, S.tile[b], tile, s_tensor, tensor_nan);
    __syncthreads();                                 // buffer b is refilled next iteration
  }
  if (*reinterpret_cast<volatile int*>(&S.abort_flag)) {
    const uint64_t t0 = ptx::clock64_();             // let the outstanding copy land
    while (ptx::clock64_() - t0 < 20000000ull) {
    }
  }
}

// Tensorwise first pass: per-CTA max of the 15-bit bf16 magnitudes over a grid-strided
// sweep of 16-byte vectors (four independent loads in flight per thread).
__global__ void __launch_bounds__(512) amax_partial_kernel(const uint16_t* __restrict__ x,
                                                           int64_t n_vec,
                                                           uint32_t* __restrict__ part) {
  __shared__ uint32_t red[16];
  uint32_t m = 0;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n_vec; i += 4 * stride) {
    uint4 a = ldg_nc_v4(x + 8 * i), b = ldg_nc_v4(x + 8 * (i + stride));
    uint4 c = ldg_nc_v4(x + 8 * (i + 2 * stride)), d = ldg_nc_v4(x + 8 * (i + 3 * stride));
    m = max(m, max(max(vec_amax_bits(a), vec_amax_bits(b)), max(vec_amax_bits(c), vec_amax_bits(d))));
  }
  for (; i < n_vec; i += stride) m = max(m, vec_amax_bits(ldg_nc_v4(x + 8 * i)));
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

// Delayed recipe: reduce the per-tile partials written by the cast into the tensor's amax.
__global__ void __launch_bounds__(1024) amax_finalize_kernel(const uint32_t* __restrict__ part,
                                                             int n, float* __restrict__ amax) {
  __shared__ uint32_t red[32];
  uint32_t m = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) m = max(m, part[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = 0;
    for (int k = 0; k < int(blockDim.x >> 5); ++k) r = max(r, red[k]);
    *amax = amax_from_bits(r);
  }
}

// Empty tensor: amax 0; tensorwise also writes scale/scale_inv for amax 0.
__global__ void empty_scalars_kernel(float* amax, float* scale, float* scale_inv, int margin) {
  if (amax) *amax = 0.0f;
  if (scale) {
    float si;
    *scale = scale_from_amax(0.0f, margin, &si);
    if (scale_inv) *scale_inv = si;
  }
}

// Delayed scaling history update (one CTA): push amax_new at head, advance head, and derive
// the next scale from the max over the whole window (the `max` compute algorithm).
__global__ void __launch_bounds__(1024) amax_history_update_kernel(
    float* __restrict__ hist, int32_t* __restrict__ head, int len,
    const float* __restrict__ amax_new, float* __restrict__ scale,
    float* __restrict__ scale_inv, int margin) {
  __shared__ float red[32];
  __shared__ int nan_seen;
  const int h = *head;
  if (threadIdx.x == 0) nan_seen = 0;
  __syncthreads();
  const float a_new = *amax_new;
  float m = 0.0f;
  for (int i = threadIdx.x; i < len; i += blockDim.x) {
    const float a = (i == h) ? a_new : hist[i];
    if (a != a) nan_seen = 1;
    m = fmaxf(m, a);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = red[0];
    for (int k = 1; k < int(blockDim.x >> 5); ++k) r = fmaxf(r, red[k]);
    if (nan_seen) r = __uint_as_float(0x7FC00000u);
    hist[h] = a_new;
    *head = (h + 1) % len;
    float si;
    *scale = scale_from_amax(r, margin, &si);
    *scale_inv = si;
  }
}

// ------------------------------------------------------------------------------------
// Host-side launchers (called from the C ABI after argument checks)
// ------------------------------------------------------------------------------------

int amax_partial_ctas(int64_t n_vec) {
  const int sms = num_sms();
  int64_t want = (n_vec + 2047) / 2048;                    // >= 4 vectors per thread
  return int(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(sms) * 4)));
}

size_t quantize_workspace_bytes(int kind, int64_t R, int64_t C) {
  if (kind != FP8_RECIPE_DELAYED && kind != FP8_RECIPE_TENSORWISE) return 0;
  if (R <= 0 || C <= 0) return 0;
  const int64_t tiles = ((R + 127) / 128) * ((C + 127) / 128);
  const int64_t parts = kind == FP8_RECIPE_DELAYED ? tiles : amax_partial_ctas(R * C / 8);
  return size_t(parts) * sizeof(uint32_t);
}

template <int MODE, int EPI>
static cudaError_t launch_tiles(const QuantParams& p, cudaStream_t st) {
  const int tiles_r = int((p.R + 127) / 128);
  const int n = tiles_r * p.tiles_c;
  CUtensorMap map;
  if (!make_tmap_2d(&map, p.x, 2, p.C, p.R, kTile, kTile, false)) return cudaErrorInvalidValue;
  const int smem = int(sizeof(QuantSmem)) + 128;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(quantize_tile_kernel<MODE, EPI>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int grid = std::max(1, std::min(n, num_sms() * kQuantCtasPerSm));
  quantize_tile_kernel<MODE, EPI><<<grid, 256, smem, st>>>(map, p);
  return cudaGetLastError();
}

cudaError_t quantize_launch(int kind, int role, int margin, const uint16_t* x, int64_t R,
                            int64_t C, bool want_row, bool want_col, fp8_tensor* out,
                            void* workspace, int32_t* status, cudaStream_t st) {
  QuantParams p{};
  p.status = status;
  p.x = x;
  p.R = R;
  p.C = C;
  p.tiles_c = int((C + 127) / 128);
  p.row = want_row ? out->row : nullptr;
  p.col = want_col ? out->col : nullptr;
  p.row_scale = want_row ? out->row_scale : nullptr;
  p.col_scale = want_col ? out->col_scale : nullptr;
  p.margin = margin;
  if (R == 0 || C == 0) {
    if (kind == FP8_RECIPE_TENSORWISE || kind == FP8_RECIPE_DELAYED) {
      empty_scalars_kernel<<<1, 1, 0, st>>>(out->amax,
                                            kind == FP8_RECIPE_TENSORWISE ? out->scale : nullptr,
                                            out->scale_inv, margin);
      return cudaGetLastError();
    }
    return cudaSuccess;
  }
  switch (kind) {
    case FP8_RECIPE_TENSORWISE: {
      const int64_t n_vec = R * C / 8;
      const int ctas = amax_partial_ctas(n_vec);
      uint32_t* part = reinterpret_cast<uint32_t*>(workspace);
      amax_partial_kernel<<<ctas, 512, 0, st>>>(x, n_vec, part);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      p.part_in = part;
      p.n_part_in = ctas;
      p.amax_out = out->amax;
      p.scale_out = out->scale;
      p.scale_inv_out = out->scale_inv;
      return launch_tiles<Q_TENSOR, EPI_NONE>(p, st);
    }
    case FP8_RECIPE_DELAYED: {
      p.scale_in = out->scale;
      p.part_out = reinterpret_cast<uint32_t*>(workspace);
      cudaError_t e = launch_tiles<Q_TENSOR, EPI_NONE>(p, st);
      if (e != cudaSuccess) return e;
      const int n = int((R + 127) / 128) * p.tiles_c;
      amax_finalize_kernel<<<1, 1024, 0, st>>>(p.part_out, n, out->amax);
      return cudaGetLastError();
    }
    case FP8_RECIPE_MXFP8:
      return launch_tiles<Q_MX, EPI_NONE>(p, st);
    case FP8_RECIPE_BLOCKWISE:
      return role == FP8_ROLE_WEIGHT ? launch_tiles<Q_BW128, EPI_NONE>(p, st)
                                     : launch_tiles<Q_BW1x128, EPI_NONE>(p, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t gelu_quantize_launch(const uint16_t* h, int64_t R, int64_t C, uint16_t* a_bf16,
                                 fp8_tensor* a_q, fp8_tensor* h_q, int32_t* status,
                                 cudaStream_t st) {
  if (R == 0 || C == 0) return cudaSuccess;
  QuantParams p{};
  p.status = status;
  p.x = h;
  p.R = R;
  p.C = C;
  p.tiles_c = int(C / 128);
  p.row = a_q->row;
  p.col = a_q->col;
  p.row_scale = a_q->row_scale;
  p.col_scale = a_q->col_scale;
  p.y_bf16 = a_bf16;
  p.aux_row = h_q->row;
  p.aux_scale = reinterpret_cast<uint8_t*>(h_q->row_scale);
  return launch_tiles<Q_MX, EPI_GELU>(p, st);
}

cudaError_t dgelu_quantize_launch(const uint16_t* da, const fp8_tensor* h_q, int64_t R,
                                  int64_t C, uint16_t* dh_bf16, fp8_tensor* dh_q,
                                  int32_t* status, cudaStream_t st) {
  if (R == 0 || C == 0) return cudaSuccess;
  QuantParams p{};
  p.status = status;
  p.x = da;
  p.R = R;
  p.C = C;
  p.tiles_c = int(C / 128);
  p.row = dh_q->row;
  p.col = dh_q->col;
  p.row_scale = dh_q->row_scale;
  p.col_scale = dh_q->col_scale;
  p.y_bf16 = dh_bf16;
  p.aux_row = h_q->row;
  p.aux_scale = reinterpret_cast<uint8_t*>(h_q->row_scale);
  return launch_tiles<Q_MX, EPI_DGELU>(p, st);
}

cudaError_t amax_update_launch(float* hist, int32_t* head, int len, const float* amax_new,
                               float* scale, float* scale_inv, int margin, cudaStream_t st) {
  amax_history_update_kernel<<<1, 1024, 0, st>>>(hist, head, len, amax_new, scale, scale_inv,
                                                 margin);
  return cudaGetLastError();
}

}  // namespace fp8lin
