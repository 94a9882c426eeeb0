// Quantize-cast kernels of the FP8 linear layer: bf16 -> E4M3 codes + scales, row-wise copy
// [R][C] and column-wise (transposed) copy [C][R], for the four recipes of the Megatron Core
// "Low-Precision Training Guide" (Recipe Reference: delayed, tensorwise, mxfp8, blockwise),
// plus the MLP activation variants that keep the GeLU input in FP8.
//
// A persistent kernel: two CTAs of 256 threads per SM, each walking 128 x 128 source tiles
// (blockIdx.x, then + gridDim.x, ...). Thread 0 streams the tiles with TMA (two 64-column
// boxes, 128-byte swizzle) into a ring of three shared-memory buffers, so two tiles are in
// flight while one is converted.
//   Row-wise codes   written straight from registers (a half-warp covers one 128-byte row
//                    segment).
//   Column-wise      written from the shared-memory tile: each thread emits 32 consecutive
//   codes            bytes of two transposed rows, i.e. whole 32-byte sectors, with one
//                    256-bit store.
//   Scales           staged in shared memory and written as one coalesced block per tile.
// HBM traffic per element: 2 bytes read, 1 byte per copy written, plus the scales. Each
// launch uses programmatic dependent launch: the next kernel may start launching at once, and
// this one waits for the previous kernel before its first global memory access.
#include <algorithm>

#include "common.cuh"
#include "gelu.cuh"
#include "internal.cuh"
#include "sm100_ptx.cuh"

namespace fp8lin {

enum QMode : int { Q_TENSOR = 0, Q_MX = 1, Q_BW1x128 = 2, Q_BW128 = 3 };
// MLP epilogue kinds (MlpEpi) and the GeLU tables come from gelu.cuh.
template <int EPI>
__host__ __device__ constexpr uint32_t quant_table_bytes() {
  return EPI == EPI_GELU ? kGeluTableBytes : (EPI == EPI_DGELU ? kDgeluTableBytes : 0u);
}

struct QuantParams {
  const uint16_t* x;          // [R][C] bf16 (h for GELU, da for DGELU)
  int64_t R, C;
  int tiles_c;
  uint8_t* row;               // [R][C] codes or null
  uint8_t* col;               // [C][R] codes (or bf16 when col_bf16), or null
  bool col_bf16;              // column copy = bf16 transpose (wgrad kept in bf16)
  bool col_v8;                // column copy rows start on 32-byte boundaries (256-bit stores)
  bool pow2;                  // blockwise: power-of-two block scales
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
  // Failure-detection test hook (0 otherwise): extra bytes CTA 0's first tile expects, so its
  // barrier never completes and the bounded wait runs out (fp8_test_quantize_stalled).
  uint32_t stall_tx;
  // Tensorwise cast pass: the amax pass has just read the input with an L2 evict_last policy.
  // Walk the tiles in reverse (the most recently read first) and read them with evict_first,
  // so the second read is served from L2 and leaves it.
  bool l2_reread;
};

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


// Shared-memory layout of the quantize kernel (offsets from a 1024-byte aligned base):
//   [0, 5120)           control and staging (QuantCtl)
//   [5120, 103424)      three tile buffers, each two 16 KiB halves (64 columns x 128 rows of
//                       bf16) written by TMA with the 128-byte swizzle: logical 16-byte chunk
//                       c of row r sits at physical chunk c ^ (r % 8). Two tiles are in
//                       flight while the third is converted. For per-tensor and 128x128
//                       scales the row-wise codes are written back over the first half of the
//                       buffer being converted (same swizzle) and read back transposed.
struct QuantCtl {
  uint8_t sc_row[512];              // MXFP8 scale atom of the row copy
  uint8_t sc_col[512];              // ... of the column copy
  float scf_row[128];               // blockwise 1x128 s_inv staging
  float scf_col[128];
  uint32_t red[8];
  uint32_t red_col[4][128];
  uint64_t bar[4];                  // TMA completion, one per buffer
  int abort_flag;
};
constexpr uint32_t kQCtlBytes = 5120;
// Three tile buffers per CTA (two tiles in flight while one is converted), two CTAs per SM.
// (Three CTAs of two buffers each, which the per-tensor casts' register count would allow,
// measured 4-5% slower for tensorwise and delayed at 8192 x 4096.)
template <int MODE, int EPI>
__host__ __device__ constexpr int quant_bufs() { return 3; }
template <int EPI>
__host__ __device__ constexpr uint32_t quant_tiles_off() {
  return kQCtlBytes + quant_table_bytes<EPI>();
}
constexpr uint32_t kQTileBytes = 32768;
static_assert(sizeof(QuantCtl) <= kQCtlBytes, "control block too large");
constexpr uint64_t kQuantWaitBudget = 4000000000ull;   // ~2 s at 2 GHz

template <int MODE>
__host__ __device__ constexpr bool uses_code_tile() { return false; }
template <int MODE, int EPI>
__host__ __device__ constexpr uint32_t quant_smem_bytes() {
  return 1024 + quant_tiles_off<EPI>() + quant_bufs<MODE, EPI>() * kQTileBytes;
}
template <int MODE, int EPI>
__host__ __device__ constexpr int quant_ctas_per_sm() { return 2; }

// Byte offset of logical 16-byte chunk c (0..7) of row r in a 128-byte-swizzled 128-row block.
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t c) {
  return r * 128u + (((c ^ r) & 7u) << 4);
}

// Quantise one 128 x 128 tile held in shared memory.
//   Row pass: warp w, lane = 16 h + 4 rr + cc: row r = 32 i + 4 w + rr (i = 0..3), columns
//   64 h + 16 cc .. +15 (two 16-byte chunks). A 1x32 MXFP8 block is two lanes, a 1x128 block
//   eight. Each lane writes 16 codes (one 16-byte store); a warp covers four 128-byte rows.
//   Column pass: thread (pp = t % 64, q = t / 64) owns source columns 2pp, 2pp+1 over rows
//   32q .. 32q+31 and writes 32 consecutive bytes of each transposed row (re-quantised for
//   MXFP8 and 1x128); per-tensor and 128x128 scales transpose the row codes instead.
template <int MODE, int EPI, int F8>
__device__ __forceinline__ void quantize_one_tile(const QuantParams& p, QuantCtl& S,
                                                  uint8_t* tile, uint8_t* codes,
                                                  const void* table, int tile_id,
                                                  float s_tensor, bool tensor_nan) {
  const int t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  const int h = lane >> 4, rr = (lane >> 2) & 3, cc = lane & 3;
  const int tr = tile_id / p.tiles_c, tc = tile_id % p.tiles_c;
  // 32-bit index arithmetic: the host guarantees R * C < 2^31.
  const uint32_t r0 = uint32_t(tr) * kTile, c0 = uint32_t(tc) * kTile;
  const uint32_t R = uint32_t(p.R), C = uint32_t(p.C);
  const uint32_t ccol = 64u * h + 16u * cc;            // first column of this lane's 16
  const bool col_ok = (c0 + ccol) < C;
  uint8_t* half = tile + h * 16384;

  // ---- this lane's 4 x 16 bf16 (out-of-range parts of the tile read as zero)
  uint32_t w[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t r = 32u * i + 4u * warp + rr;
    const uint4 a = *reinterpret_cast<const uint4*>(half + swz(r, 2 * cc));
    const uint4 b = *reinterpret_cast<const uint4*>(half + swz(r, 2 * cc + 1));
    w[i][0] = a.x; w[i][1] = a.y; w[i][2] = a.z; w[i][3] = a.w;
    w[i][4] = b.x; w[i][5] = b.y; w[i][6] = b.z; w[i][7] = b.w;
  }

  // ---- MLP epilogues: turn the input into the tensor to quantise (and write it back)
  uint4 hcodes[4];
  uint32_t hscale[4];
  if constexpr (EPI == EPI_DGELU) {
    // all of this lane's h codes and scales in flight together
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t r = 32u * i + 4u * warp + rr;
      hcodes[i] = make_uint4(0u, 0u, 0u, 0u);
      hscale[i] = 127u;
      if ((r0 + r < R) && col_ok) {
        hcodes[i] = ldg_nc_v4(p.aux_row + (r0 + r) * C + c0 + ccol);
        hscale[i] = __ldg(p.aux_scale + mx_scale_offset(r0 + r, (c0 + ccol) >> 5, C));
      }
    }
  }
  if constexpr (EPI != EPI_NONE) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t r = 32u * i + 4u * warp + rr;
      const bool ok = (r0 + r < R) && col_ok;
      const uint32_t off = (r0 + r) * C + c0 + ccol;
      if constexpr (EPI == EPI_GELU) {
        // h's own MXFP8 row copy first (the FP8 input store), then a = bf16(gelu(h))
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) m = absmax_bf16x2(m, w[i][k]);
        m = fold_bf16x2(m);
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
        float mult;
        const uint32_t sb = mx_scale_byte(m, &mult);
        uint4 hc = make_uint4(encode4<F8>(w[i][0], w[i][1], mult), encode4<F8>(w[i][2], w[i][3], mult),
                              encode4<F8>(w[i][4], w[i][5], mult), encode4<F8>(w[i][6], w[i][7], mult));
        if (m > 0x7F80u) {
          hc.x = fix_nan4(hc.x, w[i][0], w[i][1]); hc.y = fix_nan4(hc.y, w[i][2], w[i][3]);
          hc.z = fix_nan4(hc.z, w[i][4], w[i][5]); hc.w = fix_nan4(hc.w, w[i][6], w[i][7]);
        }
        if (ok) {
          *reinterpret_cast<uint4*>(p.aux_row + off) = hc;
          if ((cc & 1) == 0) p.aux_scale[mx_scale_offset(r0 + r, (c0 + ccol) >> 5, C)] = uint8_t(sb);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) w[i][k] = gelu_bf16x2(table, w[i][k]);
      } else {
        // dh = bf16(da * gelu'(h)), h decoded from its MXFP8 row copy (loaded up front)
        if (ok) {
          const uint4 hc = hcodes[i];
          const uint32_t sb = hscale[i];
          const float hs = sb == 0xFFu ? __uint_as_float(0x7FC00000u) : exp2i(int(sb) - 127);
          const uint32_t cw[4] = {hc.x, hc.y, hc.z, hc.w};
#pragma unroll
          for (int k = 0; k < 8; ++k)
            w[i][k] = dgelu_bf16x2(table, w[i][k], uint16_t(cw[k >> 1] >> (16 * (k & 1))), hs);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) w[i][k] = 0u;
        }
      }
      if (p.y_bf16 != nullptr && ok) {
        *reinterpret_cast<uint4*>(p.y_bf16 + off) = make_uint4(w[i][0], w[i][1], w[i][2], w[i][3]);
        *reinterpret_cast<uint4*>(p.y_bf16 + off + 8) = make_uint4(w[i][4], w[i][5], w[i][6], w[i][7]);
      }
      if (p.col != nullptr) {
        *reinterpret_cast<uint4*>(half + swz(r, 2 * cc)) = make_uint4(w[i][0], w[i][1], w[i][2], w[i][3]);
        *reinterpret_cast<uint4*>(half + swz(r, 2 * cc + 1)) = make_uint4(w[i][4], w[i][5], w[i][6], w[i][7]);
      }
    }
  }

  // ---- the tile-wide scale (per-tensor and 128x128 recipes)
  float s_tile = s_tensor, sinv_tile = 1.0f;
  bool tile_nan = tensor_nan;
  const bool need_tile_amax =
      MODE == Q_BW128 || (MODE == Q_TENSOR && p.part_out != nullptr);
  if (need_tile_amax) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int k = 0; k < 8; ++k) m = absmax_bf16x2(m, w[i][k]);
    const uint32_t tm = block_max_u32(fold_bf16x2(m), S.red);
    tile_nan = tm > 0x7F80u;
    if constexpr (MODE == Q_TENSOR) {
      if (t == 0) p.part_out[tile_id] = tm;               // delayed: record this tile's amax
    } else {
      s_tile = scale_from_amax(amax_from_bits(tm), p.margin, &sinv_tile, fp8_max<F8>(), p.pow2);
      const int tiles_r = int((R + 127) >> 7);
      if (p.pow2) {
        // power-of-two scales are stored as E8M0 bytes in the MXFP8 layout (one 512-byte atom
        // per 128 x 128 tile and copy, every byte the tile's scale)
        const uint32_t b = e8m0_of_pow2(sinv_tile) * 0x01010101u;
        const uint4 v = make_uint4(b, b, b, b);
        if (t < 32 && p.row_scale)
          reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.row_scale) +
                                   (uint32_t(tr) * p.tiles_c + tc) * 512)[t] = v;
        if (t >= 32 && t < 64 && p.col_scale && !p.col_bf16)
          reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.col_scale) +
                                   (uint32_t(tc) * tiles_r + tr) * 512)[t - 32] = v;
      } else if (t == 0) {
        if (p.row_scale) reinterpret_cast<float*>(p.row_scale)[tr * p.tiles_c + tc] = sinv_tile;
        if (p.col_scale && !p.col_bf16)
          reinterpret_cast<float*>(p.col_scale)[tc * tiles_r + tr] = sinv_tile;
      }
    }
  }

  // ---- row-wise copy (and the code tile for the transposed copy)
  const bool code_tile = uses_code_tile<MODE>() && !p.col_bf16;
  if (code_tile && p.col != nullptr) __syncthreads();   // every lane holds its bf16 in registers
  // 1x128 blocks: a row's block spans the 8 lanes with this lane's rr (both h, all cc). Each of
  // the four rows i of a lane gets its amax from those lanes; lane cc = i then computes that
  // row's scale (one division pair a lane instead of four) and hands it to the other seven.
  float s_bw[4] = {1.0f, 1.0f, 1.0f, 1.0f};
  uint32_t m_bw[4] = {0u, 0u, 0u, 0u};
  if constexpr (MODE == Q_BW1x128) {
    if (p.row != nullptr) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) m = absmax_bf16x2(m, w[i][k]);
        m = fold_bf16x2(m);
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m_bw[i] = max(m, __shfl_xor_sync(0xffffffffu, m, 16));
      }
      const uint32_t mine = cc == 0 ? m_bw[0] : cc == 1 ? m_bw[1] : cc == 2 ? m_bw[2] : m_bw[3];
      float sinv;
      const float s_mine = scale_from_amax(amax_from_bits(mine), p.margin, &sinv, fp8_max<F8>(),
                                           p.pow2);
      if (h == 0) S.scf_row[32u * cc + 4u * warp + rr] = sinv;
#pragma unroll
      for (int i = 0; i < 4; ++i) s_bw[i] = __shfl_sync(0xffffffffu, s_mine, (lane & ~3) | i);
    }
  }
  if (p.row != nullptr || code_tile) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t r = 32u * i + 4u * warp + rr;
      float s = s_tile;
      bool nan = tile_nan;
      if constexpr (MODE == Q_MX) {
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) m = absmax_bf16x2(m, w[i][k]);
        m = fold_bf16x2(m);
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
        const uint32_t sb = mx_scale_byte(m, &s);
        if ((cc & 1) == 0) S.sc_row[(r & 31) * 16 + (r >> 5) * 4 + 2 * h + (cc >> 1)] = uint8_t(sb);
        nan = m > 0x7F80u;
      } else if constexpr (MODE == Q_BW1x128) {
        s = s_bw[i];
        nan = m_bw[i] > 0x7F80u;
      }
      uint4 q4 = make_uint4(encode4<F8>(w[i][0], w[i][1], s), encode4<F8>(w[i][2], w[i][3], s),
                            encode4<F8>(w[i][4], w[i][5], s), encode4<F8>(w[i][6], w[i][7], s));
      if (nan) {
        q4.x = fix_nan4(q4.x, w[i][0], w[i][1]); q4.y = fix_nan4(q4.y, w[i][2], w[i][3]);
        q4.z = fix_nan4(q4.z, w[i][4], w[i][5]); q4.w = fix_nan4(q4.w, w[i][6], w[i][7]);
      }
      if (p.row != nullptr && (r0 + r < R) && col_ok)
        *reinterpret_cast<uint4*>(p.row + (r0 + r) * C + c0 + ccol) = q4;
      if (code_tile && p.col != nullptr) *reinterpret_cast<uint4*>(codes + swz(r, 4 * h + cc)) = q4;
    }
  }

  if (p.col != nullptr) {
    // The MLP epilogues wrote their transformed tile back into the buffer (and a code tile
    // would be read transposed): wait for every lane's writes. Otherwise the column pass reads
    // the tile as TMA delivered it, which every thread has already seen complete.
    if constexpr (EPI != EPI_NONE || uses_code_tile<MODE>()) __syncthreads();
    if (p.col_bf16) {
      // ---- column-wise copy in bf16 (wgrad kept in bf16): the plain transpose. Thread
      // (pp, q) owns source columns 2pp, 2pp+1 over rows 32q .. 32q+31 (64 bytes each).
      const int pp = t & 63, q = t >> 6;
      const uint8_t* hb = tile + (pp >> 5) * 16384;
      const uint32_t chunk = (pp & 31) >> 2, wofs = 4u * (pp & 3);
      uint32_t lo[16], hi[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t x0 = *reinterpret_cast<const uint32_t*>(hb + swz(32u * q + 2 * j, chunk) + wofs);
        const uint32_t x1 = *reinterpret_cast<const uint32_t*>(hb + swz(32u * q + 2 * j + 1, chunk) + wofs);
        lo[j] = __byte_perm(x0, x1, 0x5410);
        hi[j] = __byte_perm(x0, x1, 0x7632);
      }
      const uint32_t rr0 = r0 + 32u * q, cA = c0 + 2u * pp;
      if (cA < C) {
        uint16_t* dst = reinterpret_cast<uint16_t*>(p.col) + cA * R + rr0;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t* src = k == 0 ? lo : hi;
          uint16_t* d = dst + k * R;
          const bool ok0 = rr0 < R, ok1 = rr0 + 16 < R;
          store_seg32(d, make_uint4(src[0], src[1], src[2], src[3]),
                      make_uint4(src[4], src[5], src[6], src[7]), ok0, ok0, p.col_v8);
          store_seg32(d + 16, make_uint4(src[8], src[9], src[10], src[11]),
                      make_uint4(src[12], src[13], src[14], src[15]), ok1, ok1, p.col_v8);
        }
      }
    } else if constexpr (uses_code_tile<MODE>()) {
      // ---- column-wise copy = byte transpose of the row codes. Thread (pp, q): source
      // columns 2pp, 2pp+1 over rows 32q .. 32q+31; each transposed row segment is one
      // 32-byte sector.
      const int pp = t & 63, q = t >> 6;
      const uint32_t chunk = uint32_t(pp) >> 3, bofs = 2u * (pp & 7);
      uint32_t ca[8], cb[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t x[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t r = 32u * q + 4u * j + k;
          x[k] = *reinterpret_cast<const uint16_t*>(codes + swz(r, chunk) + bofs);
        }
        const uint32_t lo = __byte_perm(x[0], x[1], 0x5410), hi = __byte_perm(x[2], x[3], 0x5410);
        ca[j] = __byte_perm(lo, hi, 0x6420);
        cb[j] = __byte_perm(lo, hi, 0x7531);
      }
      const uint32_t rr0 = r0 + 32u * q, cA = c0 + 2u * pp;
      if (cA < C) {
        uint8_t* dst = p.col + cA * R + rr0;
        const bool ok0 = rr0 < R, ok1 = rr0 + 16 < R;
        store_seg32(dst, make_uint4(ca[0], ca[1], ca[2], ca[3]), make_uint4(ca[4], ca[5], ca[6], ca[7]),
                    ok0, ok1, p.col_v8);
        store_seg32(dst + R, make_uint4(cb[0], cb[1], cb[2], cb[3]),
                    make_uint4(cb[4], cb[5], cb[6], cb[7]), ok0, ok1, p.col_v8);
      }
    } else {
      // ---- column-wise copy re-quantised along the rows
      const int pp = t & 63, q = t >> 6;
      const uint8_t* hb = tile + (pp >> 5) * 16384;
      const uint32_t chunk = (pp & 31) >> 2, wofs = 4u * (pp & 3);
      uint32_t x[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint32_t r = 32u * q + j;
        x[j] = *reinterpret_cast<const uint32_t*>(hb + swz(r, chunk) + wofs);
      }
      float sa, sb;
      bool nan_here;
      if constexpr (MODE == Q_TENSOR || MODE == Q_BW128) {
        // one scale for the whole tile: the same codes as the row copy, transposed
        sa = sb = s_tile;
        nan_here = tile_nan;
      } else {
      uint32_t mw = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) mw = absmax_bf16x2(mw, x[j]);
      const uint32_t ma = mw & 0x7FFFu, mb = (mw >> 16) & 0x7FFFu;   // columns 2pp and 2pp+1
      nan_here = ma > 0x7F80u || mb > 0x7F80u;
      if constexpr (MODE == Q_MX) {
        const uint32_t ba = mx_scale_byte(ma, &sa), bb = mx_scale_byte(mb, &sb);
        const int ca = 2 * pp, cb = 2 * pp + 1;
        S.sc_col[(ca & 31) * 16 + (ca >> 5) * 4 + q] = uint8_t(ba);
        S.sc_col[(cb & 31) * 16 + (cb >> 5) * 4 + q] = uint8_t(bb);
      } else {
        S.red_col[q][2 * pp] = ma;
        S.red_col[q][2 * pp + 1] = mb;
        __syncthreads();
        const uint32_t fa = max(max(S.red_col[0][2 * pp], S.red_col[1][2 * pp]),
                                max(S.red_col[2][2 * pp], S.red_col[3][2 * pp]));
        const uint32_t fb = max(max(S.red_col[0][2 * pp + 1], S.red_col[1][2 * pp + 1]),
                                max(S.red_col[2][2 * pp + 1], S.red_col[3][2 * pp + 1]));
        if (q == 0) {                  // the threads that store the dequantisation factors
          float ia, ib;
          sa = scale_from_amax(amax_from_bits(fa), p.margin, &ia, fp8_max<F8>(), p.pow2);
          sb = scale_from_amax(amax_from_bits(fb), p.margin, &ib, fp8_max<F8>(), p.pow2);
          S.scf_col[2 * pp] = ia;
          S.scf_col[2 * pp + 1] = ib;
        } else {
          sa = scale_only_from_amax(amax_from_bits(fa), p.margin, fp8_max<F8>(), p.pow2);
          sb = scale_only_from_amax(amax_from_bits(fb), p.margin, fp8_max<F8>(), p.pow2);
        }
      }
      }
      // codes of column 2pp (low halves) and 2pp+1 (high halves), 32 rows each
      uint32_t ca[8], cb[8];
      const float2 sab = make_float2(sa, sb);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        // one packed multiply a word: (low half x sa, high half x sb)
        float2 y[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          y[k] = __fmul2_rn(make_float2(bf16_lo(x[4 * j + k]), bf16_hi(x[4 * j + k])), sab);
        ca[j] = cvt_fp8x4<F8>(y[0].x, y[1].x, y[2].x, y[3].x);
        cb[j] = cvt_fp8x4<F8>(y[0].y, y[1].y, y[2].y, y[3].y);
      }
      if (nan_here) {                                                   // NaN present
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t lo01 = (x[4 * j] & 0xFFFFu) | (x[4 * j + 1] << 16);
          const uint32_t lo23 = (x[4 * j + 2] & 0xFFFFu) | (x[4 * j + 3] << 16);
          const uint32_t hi01 = (x[4 * j] >> 16) | (x[4 * j + 1] & 0xFFFF0000u);
          const uint32_t hi23 = (x[4 * j + 2] >> 16) | (x[4 * j + 3] & 0xFFFF0000u);
          ca[j] = fix_nan4(ca[j], lo01, lo23);
          cb[j] = fix_nan4(cb[j], hi01, hi23);
        }
      }
      const uint32_t rr0 = r0 + 32u * q;
      const uint32_t cA = c0 + 2u * pp;
      if (cA < C) {
        uint8_t* dst = p.col + cA * R + rr0;
        const bool ok0 = rr0 < R, ok1 = rr0 + 16 < R;
        store_seg32(dst, make_uint4(ca[0], ca[1], ca[2], ca[3]), make_uint4(ca[4], ca[5], ca[6], ca[7]),
                    ok0, ok1, p.col_v8);
        store_seg32(dst + R, make_uint4(cb[0], cb[1], cb[2], cb[3]),
                    make_uint4(cb[4], cb[5], cb[6], cb[7]), ok0, ok1, p.col_v8);
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
      if (t >= 32 && t < 64 && p.col != nullptr && !p.col_bf16)
        reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.col_scale) +
                                 (uint32_t(tc) * tiles_r + tr) * 512)[t - 32] =
            reinterpret_cast<const uint4*>(S.sc_col)[t - 32];
    } else if (p.pow2) {
      // E8M0 bytes in the MXFP8 layout: each 1x128 block's byte for its four 1x32 blocks, the
      // 128 rows (columns) of this tile filling one 512-byte atom of the row (column) copy
      const int u = t & 127;
      const uint32_t off = uint32_t(u & 31) * 16 + uint32_t(u >> 5) * 4;
      if (t < 128 && p.row != nullptr)
        *reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(p.row_scale) +
                                     (uint32_t(tr) * p.tiles_c + tc) * 512 + off) =
            e8m0_of_pow2(S.scf_row[u]) * 0x01010101u;
      if (t >= 128 && p.col != nullptr && !p.col_bf16)
        *reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(p.col_scale) +
                                     (uint32_t(tc) * uint32_t(R >> 7) + tr) * 512 + off) =
            e8m0_of_pow2(S.scf_col[u]) * 0x01010101u;
    } else {
      if (t < 128 && p.row != nullptr)
        reinterpret_cast<float*>(p.row_scale)[uint32_t(tc) * R + r0 + t] = S.scf_row[t];
      if (t >= 128 && p.col != nullptr && !p.col_bf16)
        reinterpret_cast<float*>(p.col_scale)[uint32_t(tr) * C + c0 + (t - 128)] =
            S.scf_col[t - 128];
    }
  }
}

// Bounded wait on a TMA completion barrier (all threads); false once the budget is spent.
__device__ __forceinline__ bool quant_wait(QuantCtl& S, int b, uint32_t parity, int32_t* st) {
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
// issues the TMA loads of the next tile into the other buffer before the current one is
// processed, so HBM reads overlap the conversion and the stores.
template <int MODE, int EPI, int F8>
__global__ void __launch_bounds__(256, quant_ctas_per_sm<MODE, EPI>())
    quantize_tile_kernel(const __grid_constant__ CUtensorMap tmX, const QuantParams p) {
  static_assert(F8 == F8_E4M3 || (MODE != Q_MX && EPI == EPI_NONE), "E5M2: per-tensor / blockwise");
  extern __shared__ uint8_t qsm_raw[];
  uint8_t* base = ptx::align_smem<1024>(qsm_raw);
  QuantCtl& S = *reinterpret_cast<QuantCtl*>(base);
  constexpr int kQBufs = quant_bufs<MODE, EPI>();
  uint8_t* tiles = base + quant_tiles_off<EPI>();
  void* table = base + kQCtlBytes;
  const int t = threadIdx.x;
  const int tiles_r = int((p.R + 127) >> 7);
  const int n_tiles = tiles_r * p.tiles_c;

  pdl_launch_dependents();
  if (t == 0) {
    for (int b = 0; b < kQBufs; ++b) ptx::mbar_init(&S.bar[b], 1);
    S.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();                      // the previous kernel's writes are visible from here on

  // the i-th tile of the walk: in order, or last first for the tensorwise re-read
  auto tile_at = [&](int seq) { return p.l2_reread ? n_tiles - 1 - seq : seq; };
  uint64_t policy = 0;
  if (p.l2_reread && t == 0) policy = ptx::l2_evict_first_policy();
  auto issue = [&](int seq, int b) {
    const int tile_id = tile_at(seq);
    const int tr = tile_id / p.tiles_c, tc = tile_id % p.tiles_c;
    uint8_t* dst = tiles + b * kQTileBytes;
    ptx::mbar_arrive_expect_tx(&S.bar[b], kQTileBytes + (seq == 0 ? p.stall_tx : 0u));
    if (p.l2_reread) {
      ptx::tma_load_2d_hint(dst, &tmX, tc * kTile, tr * kTile, &S.bar[b], policy);
      ptx::tma_load_2d_hint(dst + 16384, &tmX, tc * kTile + 64, tr * kTile, &S.bar[b], policy);
    } else {
      ptx::tma_load_2d(dst, &tmX, tc * kTile, tr * kTile, &S.bar[b]);
      ptx::tma_load_2d(dst + 16384, &tmX, tc * kTile + 64, tr * kTile, &S.bar[b]);
    }
  };

  // prologue: the first kQBufs - 1 tiles in flight
  if (t == 0) {
    for (int j = 0; j < kQBufs - 1; ++j) {
      const int tl = int(blockIdx.x) + j * int(gridDim.x);
      if (tl < n_tiles) issue(tl, j);
    }
  }
  // per-tensor scale once per CTA (the first tiles are already in flight): tensorwise from the
  // amax partials, delayed from memory
  float s_tensor = 1.0f;
  bool tensor_nan = false;
  if constexpr (MODE == Q_TENSOR) {
    if (p.scale_in != nullptr) {
      s_tensor = *p.scale_in;
    } else {
      uint32_t m = 0;
      for (int base = t; base < p.n_part_in; base += 4 * 256) {   // four loads in flight
        uint32_t v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = base + 256 * k;
          v[k] = j < p.n_part_in ? __ldg(p.part_in + j) : 0u;
        }
        m = max(max(m, max(v[0], v[1])), max(v[2], v[3]));
      }
      m = block_max_u32(m, S.red);
      tensor_nan = m > 0x7F80u;
      float sinv;
      s_tensor = scale_from_amax(amax_from_bits(m), p.margin, &sinv, fp8_max<F8>(), p.pow2);
      if (blockIdx.x == 0 && t == 0) {
        *p.amax_out = amax_from_bits(m);
        *p.scale_out = s_tensor;
        *p.scale_inv_out = sinv;
      }
    }
  }

  // MLP kernels: fill the GeLU table while the first tiles are in flight
  if constexpr (EPI == EPI_GELU) gelu_table_fill(table, t, 256);
  else if constexpr (EPI == EPI_DGELU) dgelu_table_fill(table, t, 256);
  if constexpr (EPI != EPI_NONE) __syncthreads();

  int tile = blockIdx.x;
  for (int i = 0; tile < n_tiles; ++i, tile += gridDim.x) {
    const int b = i % kQBufs;
    const int ahead = tile + (kQBufs - 1) * int(gridDim.x);
    if (t == 0 && ahead < n_tiles) issue(ahead, (i + kQBufs - 1) % kQBufs);
    if constexpr (EPI == EPI_DGELU) {
      // the h codes this lane will read for that tile: into L2 while it is in flight
      if (ahead < n_tiles) {
        const int tid = tile_at(ahead);
        const uint32_t ar0 = uint32_t(tid / p.tiles_c) * kTile, ac0 = uint32_t(tid % p.tiles_c) * kTile;
        const int lane = t & 31, h = lane >> 4, rr = (lane >> 2) & 3, cc = lane & 3;
        const uint32_t col = ac0 + 64u * h + 16u * cc;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t r = ar0 + 32u * k + 4u * (t >> 5) + rr;
          if (r < uint32_t(p.R) && col < uint32_t(p.C))
            prefetch_l2(p.aux_row + r * uint32_t(p.C) + col);
        }
      }
    }
    if (!quant_wait(S, b, uint32_t(i / kQBufs) & 1u, p.status)) break;
    uint8_t* buf = tiles + b * kQTileBytes;
    quantize_one_tile<MODE, EPI, F8>(p, S, buf, buf, table, tile_at(tile), s_tensor,
                                     tensor_nan);
    // buffer b is refilled by TMA next iteration: the MLP epilogues wrote their transformed
    // tile into it with ordinary stores, which must be ordered before the async copy
    if constexpr (EPI != EPI_NONE || uses_code_tile<MODE>()) ptx::fence_proxy_async_smem();
    __syncthreads();
  }
  if (*reinterpret_cast<volatile int*>(&S.abort_flag)) {
    const uint64_t t0 = ptx::clock64_();             // let the outstanding copies land
    while (ptx::clock64_() - t0 < 20000000ull) {
    }
  }
}

// Several tensors of one block-scaled recipe in one launch: one persistent grid walks the
// tiles of all of them (tensor 0's first, then tensor 1's, ...), so a set of small tensors runs
// at the rate of one large one instead of paying a launch's ramp and tail each. Every tile is
// quantised exactly as the single-tensor kernel quantises it. FAM 0 is MXFP8; FAM 1 is
// blockwise, where each tensor has its own mode (1x128 or 128x128 blocks by role, E4M3 or, for
// a hybrid-format gradient, E5M2).
constexpr int kQuantGroupMax = 4;
enum GroupMode : int { GM_MX = 0, GM_BW1x128 = 1, GM_BW128 = 2, GM_BW1x128_E5 = 3, GM_BW128_E5 = 4 };
struct QuantGroup {
  CUtensorMap map[kQuantGroupMax];
  QuantParams p[kQuantGroupMax];
  int first[kQuantGroupMax + 1];    // first global tile of each tensor; first[n] = all tiles
  int mode[kQuantGroupMax];         // GroupMode of each tensor
  int n;
  uint32_t stall_tx;                // test hook (0 otherwise): extra bytes tile 0 expects
};

template <int FAM>
__global__ void __launch_bounds__(256, quant_ctas_per_sm<Q_MX, EPI_NONE>())
    quantize_group_kernel(const __grid_constant__ QuantGroup g) {
  extern __shared__ uint8_t qsm_raw[];
  uint8_t* base = ptx::align_smem<1024>(qsm_raw);
  QuantCtl& S = *reinterpret_cast<QuantCtl*>(base);
  constexpr int kQBufs = quant_bufs<Q_MX, EPI_NONE>();
  uint8_t* tiles = base + quant_tiles_off<EPI_NONE>();
  const int t = threadIdx.x;
  const int n_tiles = g.first[g.n];
  int32_t* status = g.p[0].status;

  pdl_launch_dependents();
  if (t == 0) {
    for (int b = 0; b < kQBufs; ++b) ptx::mbar_init(&S.bar[b], 1);
    S.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();

  auto tensor_of = [&](int tile) {
    int k = 0;
    while (k + 1 < g.n && tile >= g.first[k + 1]) ++k;
    return k;
  };
  auto issue = [&](int tile, int b) {
    const int k = tensor_of(tile);
    const int local = tile - g.first[k];
    const int tc_n = g.p[k].tiles_c;
    const int tr = local / tc_n, tc = local % tc_n;
    uint8_t* dst = tiles + b * kQTileBytes;
    ptx::mbar_arrive_expect_tx(&S.bar[b], kQTileBytes + (tile == 0 ? g.stall_tx : 0u));
    ptx::tma_load_2d(dst, &g.map[k], tc * kTile, tr * kTile, &S.bar[b]);
    ptx::tma_load_2d(dst + 16384, &g.map[k], tc * kTile + 64, tr * kTile, &S.bar[b]);
  };

  if (t == 0) {
    for (int j = 0; j < kQBufs - 1; ++j) {
      const int tl = int(blockIdx.x) + j * int(gridDim.x);
      if (tl < n_tiles) issue(tl, j);
    }
  }
  int tile = blockIdx.x;
  for (int i = 0; tile < n_tiles; ++i, tile += gridDim.x) {
    const int b = i % kQBufs;
    const int ahead = tile + (kQBufs - 1) * int(gridDim.x);
    if (t == 0 && ahead < n_tiles) issue(ahead, (i + kQBufs - 1) % kQBufs);
    if (!quant_wait(S, b, uint32_t(i / kQBufs) & 1u, status)) break;
    uint8_t* buf = tiles + b * kQTileBytes;
    const int k = tensor_of(tile);
    const int local = tile - g.first[k];
    if constexpr (FAM == 0) {
      quantize_one_tile<Q_MX, EPI_NONE, F8_E4M3>(g.p[k], S, buf, buf, nullptr, local, 1.0f,
                                                  false);
    } else {
      switch (g.mode[k]) {
        case GM_BW128:
          quantize_one_tile<Q_BW128, EPI_NONE, F8_E4M3>(g.p[k], S, buf, buf, nullptr, local,
                                                         1.0f, false);
          break;
        case GM_BW1x128_E5:
          quantize_one_tile<Q_BW1x128, EPI_NONE, F8_E5M2>(g.p[k], S, buf, buf, nullptr, local,
                                                           1.0f, false);
          break;
        case GM_BW128_E5:
          quantize_one_tile<Q_BW128, EPI_NONE, F8_E5M2>(g.p[k], S, buf, buf, nullptr, local,
                                                         1.0f, false);
          break;
        default:
          quantize_one_tile<Q_BW1x128, EPI_NONE, F8_E4M3>(g.p[k], S, buf, buf, nullptr, local,
                                                           1.0f, false);
          break;
      }
    }
    __syncthreads();
  }
  if (*reinterpret_cast<volatile int*>(&S.abort_flag)) {
    const uint64_t t0 = ptx::clock64_();             // let the outstanding copies land
    while (ptx::clock64_() - t0 < 20000000ull) {
    }
  }
}

// Tensorwise first pass: per-CTA max of the 15-bit bf16 magnitudes over a grid-strided
// sweep of 16-byte vectors. Each thread keeps a batch of sixteen independent loads in flight
// (out-of-range ones read nothing), so a 64 MB tensor takes two round trips to DRAM with
// tens of MB in flight across the GPU. With KEEP the input is read with an L2 evict_last
// policy, so the cast pass that follows finds it in L2.
constexpr int kAmaxThreads = 256;
constexpr int kAmaxBatch = 16;
constexpr int kAmaxCtasPerSm = 4;             // 64 registers a thread (the batch is 64 of them)
template <bool KEEP>
__device__ __forceinline__ uint4 amax_load(const uint16_t* x, int64_t v, uint64_t pol) {
  if constexpr (KEEP) return ldg_nc_v4_policy(x + 8 * v, pol);
  else return ldg_nc_v4_sched(x + 8 * v);
}
template <bool KEEP>
__global__ void __launch_bounds__(kAmaxThreads, kAmaxCtasPerSm)
    amax_partial_kernel(const uint16_t* __restrict__ x, int64_t n_vec,
                        uint32_t* __restrict__ part) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ uint32_t red[kAmaxThreads / 32];
  uint64_t pol = 0;
  if constexpr (KEEP) pol = ptx::l2_evict_last_policy();
  uint32_t m = 0;
  const int64_t stride = int64_t(gridDim.x) * kAmaxThreads;
  for (int64_t i = int64_t(blockIdx.x) * kAmaxThreads + threadIdx.x; i < n_vec;
       i += kAmaxBatch * stride) {
    uint4 v[kAmaxBatch];
#pragma unroll
    for (int k = 0; k < kAmaxBatch; ++k) {
      const int64_t j = i + k * stride;
      v[k] = j < n_vec ? amax_load<KEEP>(x, j, pol) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < kAmaxBatch; ++k) m = max(m, vec_amax_bits(v[k]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = 0;
    for (int k = 0; k < kAmaxThreads / 32; ++k) r = max(r, red[k]);
    part[blockIdx.x] = r;
  }
}

// Delayed recipe: reduce the per-tile partials written by the cast into the tensor's amax.
__global__ void __launch_bounds__(1024) amax_finalize_kernel(const uint32_t* __restrict__ part,
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
    *amax = amax_from_bits(r);
  }
}

// Empty tensor: amax 0; tensorwise also writes scale/scale_inv for amax 0.
__global__ void empty_scalars_kernel(float* amax, float* scale, float* scale_inv, int margin,
                                     float fmax) {
  pdl_launch_dependents();
  pdl_wait();
  if (amax) *amax = 0.0f;
  if (scale) {
    float si;
    *scale = scale_from_amax(0.0f, margin, &si, fmax);
    if (scale_inv) *scale_inv = si;
  }
}

// Delayed scaling history update (one CTA): push amax_new at head, advance head, and derive
// the next scale from the max over the whole window (compute algorithm `max`, algo 0) or from
// amax_new alone (`most_recent`, algo 1).
__global__ void __launch_bounds__(1024) amax_history_update_kernel(
    float* __restrict__ hist, int32_t* __restrict__ head, int len,
    const float* __restrict__ amax_new, float* __restrict__ scale,
    float* __restrict__ scale_inv, int margin, float fmax, int algo) {
  pdl_launch_dependents();
  pdl_wait();
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
    if (algo == 1) r = a_new;
    hist[h] = a_new;
    *head = (h + 1) % len;
    float si;
    *scale = scale_from_amax(r, margin, &si, fmax);
    *scale_inv = si;
  }
}

// ------------------------------------------------------------------------------------
// Host-side launchers (called from the C ABI after argument checks)
// ------------------------------------------------------------------------------------

int amax_partial_ctas(int64_t n_vec) {
  const int sms = num_sms();
  // one batch of sixteen vectors per thread, up to one wave of resident CTAs
  int64_t want = (n_vec + kAmaxThreads * kAmaxBatch - 1) / (kAmaxThreads * kAmaxBatch);
  return int(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(sms) * kAmaxCtasPerSm)));
}

size_t quantize_workspace_bytes(int kind, int64_t R, int64_t C) {
  if (kind != FP8_RECIPE_DELAYED && kind != FP8_RECIPE_TENSORWISE) return 0;
  if (R <= 0 || C <= 0) return 0;
  const int64_t tiles = ((R + 127) / 128) * ((C + 127) / 128);
  const int64_t parts = kind == FP8_RECIPE_DELAYED ? tiles : amax_partial_ctas(R * C / 8);
  return size_t(parts) * sizeof(uint32_t);
}

template <int MODE, int EPI, int F8 = F8_E4M3>
static cudaError_t launch_tiles(QuantParams p, cudaStream_t st) {
  const int64_t col_row_bytes = p.R * (p.col_bf16 ? 2 : 1);
  p.col_v8 = p.col != nullptr && (reinterpret_cast<uintptr_t>(p.col) % 32 == 0) &&
             (col_row_bytes % 32 == 0);
  const int tiles_r = int((p.R + 127) / 128);
  const int n = tiles_r * p.tiles_c;
  CUtensorMap map;
  if (!make_tmap_2d(&map, p.x, 2, p.C, p.R, 64, kTile, true)) return cudaErrorInvalidValue;
  constexpr int smem = int(quant_smem_bytes<MODE, EPI>());
  static ContextOnce attr_done{};
  const cudaError_t ae = once_per_context(attr_done, [&] {
    return cudaFuncSetAttribute(quantize_tile_kernel<MODE, EPI, F8>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (ae != cudaSuccess) return ae;
  const int grid = std::max(1, std::min(n, num_sms() * quant_ctas_per_sm<MODE, EPI>()));
  return launch_kernel(quantize_tile_kernel<MODE, EPI, F8>, dim3(grid), dim3(256), smem, st,
                       nullptr, map, p);
}

cudaError_t quantize_launch(int kind, int role, int fmt, bool pow2, int margin,
                            const uint16_t* x, int64_t R, int64_t C, bool want_row,
                            bool want_col, bool col_bf16, fp8_tensor* out, void* workspace,
                            int32_t* status, cudaStream_t st, uint32_t stall_tx) {
  const bool e5 = fmt == F8_E5M2;
  QuantParams p{};
  p.pow2 = pow2 && kind == FP8_RECIPE_BLOCKWISE;
  p.status = status;
  p.stall_tx = stall_tx;
  p.col_bf16 = col_bf16;
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
      return launch_kernel(empty_scalars_kernel, dim3(1), dim3(1), 0, st, nullptr, out->amax,
                           kind == FP8_RECIPE_TENSORWISE ? out->scale : nullptr, out->scale_inv,
                           margin, e5 ? fp8_max<F8_E5M2>() : fp8_max<F8_E4M3>());
    }
    return cudaSuccess;
  }
  switch (kind) {
    case FP8_RECIPE_TENSORWISE: {
      const int64_t n_vec = R * C / 8;
      const int ctas = amax_partial_ctas(n_vec);
      uint32_t* part = reinterpret_cast<uint32_t*>(workspace);
      // Keep the input in L2 between the two passes when it fits in well under half of L2
      // (the codes written by the cast pass share the cache).
      const bool keep = R * C * 2 <= l2_bytes() / 2;
      const cudaError_t e =
          keep ? launch_kernel(amax_partial_kernel<true>, dim3(ctas), dim3(kAmaxThreads), 0, st,
                               nullptr, x, n_vec, part)
               : launch_kernel(amax_partial_kernel<false>, dim3(ctas), dim3(kAmaxThreads), 0, st,
                               nullptr, x, n_vec, part);
      if (e != cudaSuccess) return e;
      p.l2_reread = keep;
      p.part_in = part;
      p.n_part_in = ctas;
      p.amax_out = out->amax;
      p.scale_out = out->scale;
      p.scale_inv_out = out->scale_inv;
      return e5 ? launch_tiles<Q_TENSOR, EPI_NONE, F8_E5M2>(p, st)
                : launch_tiles<Q_TENSOR, EPI_NONE>(p, st);
    }
    case FP8_RECIPE_DELAYED: {
      p.scale_in = out->scale;
      p.part_out = reinterpret_cast<uint32_t*>(workspace);
      cudaError_t e = e5 ? launch_tiles<Q_TENSOR, EPI_NONE, F8_E5M2>(p, st)
                         : launch_tiles<Q_TENSOR, EPI_NONE>(p, st);
      if (e != cudaSuccess) return e;
      const int n = int((R + 127) / 128) * p.tiles_c;
      return launch_kernel(amax_finalize_kernel, dim3(1), dim3(1024), 0, st, nullptr,
                           static_cast<const uint32_t*>(p.part_out), n, out->amax);
    }
    case FP8_RECIPE_MXFP8:
      if (e5) return cudaErrorInvalidValue;
      return launch_tiles<Q_MX, EPI_NONE>(p, st);
    case FP8_RECIPE_BLOCKWISE:
      if (role == FP8_ROLE_WEIGHT)
        return e5 ? launch_tiles<Q_BW128, EPI_NONE, F8_E5M2>(p, st)
                  : launch_tiles<Q_BW128, EPI_NONE>(p, st);
      return e5 ? launch_tiles<Q_BW1x128, EPI_NONE, F8_E5M2>(p, st)
                : launch_tiles<Q_BW1x128, EPI_NONE>(p, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t quantize_group_launch(int kind, bool pow2, int margin, int n,
                                  const QuantGroupItem* items, int32_t* status, cudaStream_t st,
                                  uint32_t stall_tx) {
  if (n < 1 || n > kQuantGroupMax) return cudaErrorInvalidValue;
  if (kind != FP8_RECIPE_MXFP8 && kind != FP8_RECIPE_BLOCKWISE) return cudaErrorInvalidValue;
  const bool bw = kind == FP8_RECIPE_BLOCKWISE;
  QuantGroup g{};
  g.stall_tx = stall_tx;
  int total = 0, k = 0;
  for (int i = 0; i < n; ++i) {
    const QuantGroupItem& it = items[i];
    if (it.R == 0 || it.C == 0) continue;                 // nothing to write for it
    QuantParams& p = g.p[k];
    p.status = status;
    p.pow2 = bw && pow2;
    p.margin = margin;
    g.mode[k] = !bw ? GM_MX
                    : it.role == FP8_ROLE_WEIGHT ? (it.e5 ? GM_BW128_E5 : GM_BW128)
                                                 : (it.e5 ? GM_BW1x128_E5 : GM_BW1x128);
    p.col_bf16 = it.col_bf16;
    p.x = it.x;
    p.R = it.R;
    p.C = it.C;
    p.tiles_c = int((it.C + 127) / 128);
    p.row = it.want_row ? it.out->row : nullptr;
    p.col = it.want_col ? it.out->col : nullptr;
    p.row_scale = it.want_row ? it.out->row_scale : nullptr;
    p.col_scale = it.want_col ? it.out->col_scale : nullptr;
    const int64_t col_row_bytes = p.R * (p.col_bf16 ? 2 : 1);
    p.col_v8 = p.col != nullptr && (reinterpret_cast<uintptr_t>(p.col) % 32 == 0) &&
               (col_row_bytes % 32 == 0);
    if (!make_tmap_2d(&g.map[k], p.x, 2, p.C, p.R, 64, kTile, true))
      return cudaErrorInvalidValue;
    g.first[k] = total;
    total += int((p.R + 127) / 128) * p.tiles_c;
    ++k;
  }
  g.n = k;
  g.first[k] = total;
  if (total == 0) return cudaSuccess;
  constexpr int smem = int(quant_smem_bytes<Q_MX, EPI_NONE>());
  static_assert(quant_smem_bytes<Q_MX, EPI_NONE>() == quant_smem_bytes<Q_BW128, EPI_NONE>() &&
                    quant_smem_bytes<Q_MX, EPI_NONE>() == quant_smem_bytes<Q_BW1x128, EPI_NONE>(),
                "the group kernels size shared memory like the single-tensor ones");
  static ContextOnce attr_mx{}, attr_bw{};
  auto kern = bw ? quantize_group_kernel<1> : quantize_group_kernel<0>;
  const cudaError_t ae = once_per_context(bw ? attr_bw : attr_mx, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (ae != cudaSuccess) return ae;
  const int grid = std::max(1, std::min(total, num_sms() * quant_ctas_per_sm<Q_MX, EPI_NONE>()));
  return launch_kernel(kern, dim3(grid), dim3(256), smem, st, nullptr, g);
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
                               float* scale, float* scale_inv, int margin, float fmax,
                               int algo, cudaStream_t st) {
  return launch_kernel(amax_history_update_kernel, dim3(1), dim3(1024), 0, st, nullptr, hist,
                       head, len, amax_new, scale, scale_inv, margin, fmax, algo);
}

}  // namespace fp8lin
