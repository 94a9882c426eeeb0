// Scaled FP8 GEMMs of the FP8 linear layer on the sm_103a tensor core (tcgen05 + TMEM + TMA).
//
// Every GEMM of the layer is "TN": D[M][N] = sum_k A[M][K] * B[N][K] with both operands
// K-major, because the column-wise FP8 copies are physically transposed:
//   fprop   X.W^T from the row copies;
//   dgrad   dY.(W^T)^T from dY's row copy and W's column copy;
//   wgrad   (dY^T).(X^T)^T from the two column copies.
// A per-tensor or 128x128 operand whose column copy was not made is read MN-major from its
// row copy instead.
//
// Scaling, per recipe of the Megatron Core "Low-Precision Training Guide" (Recipe Reference):
//   G_TENSOR  delayed / tensorwise: fp32 accumulation of the raw codes, times
//             s_inv(A) * s_inv(B) in the epilogue.
//   G_MX      mxfp8 (and power-of-two blockwise): the tensor core applies the E8M0 scale of
//             every 32-wide K block of A and B during accumulation
//             (tcgen05.mma kind::mxf8f6f4.block_scale).
//   G_BLOCK   blockwise: each 128-wide K chunk is accumulated alone into TMEM. Epilogue
//             warps promote it into fp32 registers times s_inv(A row, chunk) * s_inv(B, chunk)
//             (B: the 128x128 tile scale, or the per-row 1x128 scale for wgrad).
//   G_BF16    bf16 x bf16 (wgrad with --fp8-wgrad off).
//
// Structure: a persistent kernel. One CTA pair (cluster of two, cta_group::2) per two SMs
// runs 256 x 256 tiles; blockwise, and problems with one 128-row half, use one CTA per SM on
// 128 x 256 tiles. Tiles come in a grouped order (16 M tiles per N step).
//   warp 0        streams A/B tiles (and MX scale atoms) with TMA into a 4-6 stage ring.
//   warp 1        allocates TMEM; one thread of the leader CTA issues the MMAs.
//   epilogue      warps 2.. drain TMEM, scale, round to bf16 and store. There are 8 of them,
//                 or 16 for blockwise and the fused MLP epilogues (GeLU / dGeLU with MXFP8
//                 quantisation of their outputs).
//   MXFP8 adds    a warp that copies each stage's scale factors into TMEM.
// Accumulators are double-buffered in TMEM (512 columns), so a tile's epilogue overlaps the
// next tile's main loop. MXFP8 keeps one accumulator buffer, because its scale factors take
// the other columns; its epilogue frees TMEM as soon as it has read it.
//
// Every barrier wait has a clock budget. On expiry the kernel:
//   - records FP8_ERR_TIMEOUT in the caller's status word;
//   - lets in-flight copies land;
//   - frees TMEM and returns.
// Each kernel launches with programmatic dependent launch: it waits for the previous kernel
// only before its first global memory access.
#include <algorithm>
#include <cstdio>

#include "common.cuh"
#include "gelu.cuh"
#include "sm100_ptx.cuh"
#include "internal.cuh"

namespace fp8lin {

constexpr int kBM = 128;                      // accumulator rows per CTA (TMEM lanes)
constexpr int kBN = 256;                      // accumulator columns per tile
constexpr int kBKBytes = 128;                 // one 128-byte swizzle row of K per stage
// Epilogue warps: 8 for plain stores (two per TMEM lane quadrant, 128 columns each); 16 for
// the fused MLP epilogues and the blockwise promotion (four per quadrant, 64 columns each),
// whose per-chunk work needs more warps in flight to hide its latency. Warp 0 is the TMA
// producer, warp 1 the MMA issuer.
template <int MODE, int EPI>
__host__ __device__ constexpr int epi_warps() {
  return (EPI != EPI_NONE || MODE == G_BLOCK) ? 16 : 8;
}
// The blockwise kernel splits the register file between warpgroups: warpgroup 0 (warps 0-3:
// TMA producer, MMA issuer, two idle warps) gives registers to the four promoting epilogue
// warpgroups (warps 4-19) with setmaxnreg. (The fused MLP epilogues measured 3% slower on
// dGeLU with the same split, so they keep 19 warps at 96 registers.)
template <int MODE, int EPI>
__host__ __device__ constexpr bool reg_split() { return MODE == G_BLOCK; }
// First epilogue warp.
template <int MODE, int EPI>
__host__ __device__ constexpr int epi_first_warp() { return reg_split<MODE, EPI>() ? 4 : 2; }
// The split: launched at kSplitLaunchRegs a thread (20 warps), warpgroup 0 drops to
// kSplitWg0Regs and the epilogue warpgroups rise to kSplitEpiRegs.
// 128 x 32 + 512 x 112 = 640 x 96: the pool the CTA was launched with, exactly.
constexpr int kSplitLaunchRegs = 96, kSplitWg0Regs = 32, kSplitEpiRegs = 112;
static_assert(128 * kSplitWg0Regs + 512 * kSplitEpiRegs <= 640 * kSplitLaunchRegs,
              "register split within the launch pool");
// MXFP8 kernels add one warp that copies each stage's scale factors into TMEM, so the MMA
// issuer's instruction stream holds nothing but MMAs (warp 2 with the register split, else
// the warp after the epilogue warps).
template <int MODE, int EPI>
__host__ __device__ constexpr int gemm_threads() {
  return 32 * epi_first_warp<MODE, EPI>() + 32 * epi_warps<MODE, EPI>() +
         ((MODE == G_MX && !reg_split<MODE, EPI>()) ? 32 : 0);
}
constexpr uint32_t kTileABytes = kBM * kBKBytes;      // 16 KiB
constexpr uint32_t kSfStageBytes = 2048;              // SFA 512 B at 0, SFB 2 x 512 B at 512
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCols = 16;                      // MX scale-factor columns per stage
static_assert(256 + kSfCols * 6 <= 512, "MX scale-factor columns behind the accumulator");
constexpr uint64_t kWaitBudgetCycles = 4000000000ull;   // ~2 s at 2 GHz

// Per-configuration geometry. A single CTA (CTA2 = 0) owns a 128 x 256 tile and loads the
// whole 256-row B tile; a CTA pair (CTA2 = 1) owns a 256 x 256 tile, each CTA loading its own
// 128 rows of A and 128 of the 256 rows of B, so a stage is 32 KiB and six of them fit. The
// fused MLP epilogues add a 2 KiB transpose buffer per epilogue warp and a GeLU table behind
// the control block (those kernels give up stages for them: five for the pair, three for a
// single CTA).
constexpr uint32_t kEpiStageBytes = 2048;              // one warp's 32 x 32 bf16 chunk
template <int EPI>
__host__ __device__ constexpr uint32_t epi_smem_bytes() {
  return EPI == EPI_NONE ? 0u
                         : epi_warps<G_MX, EPI>() * kEpiStageBytes +
                               (EPI == EPI_GELU ? kGeluTableBytes : kDgeluCodeTableBytes);
}
template <int CTA2, int EPI = EPI_NONE>
struct Geo {
  static constexpr int kStages = CTA2 ? (EPI == EPI_NONE ? 6 : 5) : (EPI == EPI_NONE ? 4 : 3);
  static constexpr uint32_t kTileBBytes = (CTA2 ? kBN / 2 : kBN) * kBKBytes;
  static constexpr uint32_t kStageBytes = kTileABytes + kTileBBytes + kSfStageBytes;
  static constexpr uint32_t kSmemBytes =
      1024 + kStages * kStageBytes + 512 + epi_smem_bytes<EPI>();
  static constexpr int kTileM = CTA2 ? 2 * kBM : kBM;     // output rows per tile
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct SharedCtl {
  uint64_t full[6];
  uint64_t empty[6];
  uint64_t sfr[6];                  // MX: stage's scale factors are in TMEM
  uint64_t accf[2];
  uint64_t acce[2];
  uint32_t tmem_base;
  int abort_flag;
};

// Tile order: the persistent CTAs (pairs) take consecutive tile indices, so consecutive
// indices walk a group of kTileGroup M tiles before the next N tile. The tiles in flight at
// once then share a few A and B panels (about 16 x 5 of them for 76 pairs) instead of
// sweeping all of A for one or two B panels, which keeps the re-reads in L2. (Measured on the
// MLP step: groups of 16 M tiles beat 4, 8 and 32.) The group's panels are the ones reused
// across rounds of tiles, so the group runs along the smaller operand: with M > N the roles
// of M and N are exchanged (gn). On the MLP step's K = 16384 fprop/dgrad (M 8192, N 4096)
// that cut the DRAM bytes per launch from 571 to 475 MB, on its wgrad with M 16384, N 4096
// from 470 to 339 MB; groups of 8 on the exchanged side read more (519 MB).
constexpr int kTileGroup = 16;
__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, bool gn, int* mt,
                                            int* nt) {
  // gn: the same order with the roles of M and N exchanged
  const int ta = gn ? tiles_n : tiles_m, tb = gn ? tiles_m : tiles_n;
  const int group_tiles = kTileGroup * tb;
  const int first = (tile / group_tiles) * kTileGroup;
  const int ga = min(ta - first, kTileGroup);              // tiles of the grouped side
  const int r = tile % group_tiles;
  const int a = first + r % ga, b = r / ga;
  *mt = gn ? b : a;
  *nt = gn ? a : b;
}

// K order of a tile: a CTA (pair) walks the K blocks of its tiles alternately forwards and
// backwards. All units run about in step, so the tiles of one round end on the K blocks that
// the next round's tiles (which share the group's panels: consecutive rounds move along the
// other side within a group) start on, while those are still in L2. Blockwise keeps the
// forward order (its epilogue promotes the chunks in order).
template <int MODE>
__device__ __forceinline__ int k_block(int tile, int unit, int n_units, int kk, int nk) {
  if constexpr (MODE == G_BLOCK) return kk;
  return (((tile - unit) / n_units) & 1) ? nk - 1 - kk : kk;
}

// After a first test, the polls suspend the waiting thread (up to kSleepHintNs each; it resumes
// as soon as the phase completes) instead of spinning: a warp that waits for a whole main loop
// (the epilogue warps) then takes no issue slots from the MMA and scale-factor warps beside it.
constexpr uint32_t kSleepHintNs = 20000;
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, SharedCtl* ctl,
                                         int32_t* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::clock64_();
  while (true) {
    if (ptx::mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (*reinterpret_cast<volatile int*>(&ctl->abort_flag)) return false;
    if (ptx::clock64_() - t0 > kWaitBudgetCycles) {
      *reinterpret_cast<volatile int*>(&ctl->abort_flag) = 1;
      report_status(status, FP8_ERR_TIMEOUT);
      return false;
    }
  }
}

template <int MODE, int CTA2>
__device__ __forceinline__ uint32_t instr_desc() {
  // [4,6) D format (1 = f32) | [7,10) A fmt | [10,13) B fmt | [15] A major | [16] B major
  // | [17,23) N >> 3 | [24,29) M >> 4. E4M3 = 0, bf16 = 1. The pair's MMA has M = 256.
  const uint32_t M = CTA2 ? 2 * kBM : kBM;
  uint32_t d = (uint32_t(kBN >> 3) << 17) | ((M >> 4) << 24);
  if constexpr (MODE == G_MX) {
    d |= (1u << 23);                          // scale factors are E8M0
  } else if constexpr (MODE == G_BF16) {
    d |= (1u << 4) | (1u << 7) | (1u << 10);
  } else {
    d |= (1u << 4);
  }
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Store one thread's row segment of NC fp32 values (columns n .. n+NC-1 of row m).
template <int NC>
__device__ __forceinline__ void store_row(const GemmParams& p, int m, int n, const float* v) {
  if (m >= p.M) return;
  const bool v8 = p.d_v8 != 0;
  if (p.d_fp32) {
    float* dst = reinterpret_cast<float*>(p.D) + int64_t(m) * p.ldd + n;
#pragma unroll
    for (int j = 0; j < NC; j += 8) {
      // N is a multiple of 16, so a segment starting inside the row ends inside it
      const bool ok = n + j < p.N;
      store_seg32(dst + j,
                  make_uint4(__float_as_uint(v[j]), __float_as_uint(v[j + 1]),
                             __float_as_uint(v[j + 2]), __float_as_uint(v[j + 3])),
                  make_uint4(__float_as_uint(v[j + 4]), __float_as_uint(v[j + 5]),
                             __float_as_uint(v[j + 6]), __float_as_uint(v[j + 7])),
                  ok, ok, v8);
    }
  } else {
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.D) + int64_t(m) * p.ldd + n;
#pragma unroll
    for (int j = 0; j < NC; j += 16) {
      const bool ok = n + j < p.N;
      store_seg32(dst + j,
                  make_uint4(pack_bf16x2(v[j], v[j + 1]), pack_bf16x2(v[j + 2], v[j + 3]),
                             pack_bf16x2(v[j + 4], v[j + 5]), pack_bf16x2(v[j + 6], v[j + 7])),
                  make_uint4(pack_bf16x2(v[j + 8], v[j + 9]), pack_bf16x2(v[j + 10], v[j + 11]),
                             pack_bf16x2(v[j + 12], v[j + 13]), pack_bf16x2(v[j + 14], v[j + 15])),
                  ok, ok, v8);
    }
  }
}

// Read NC consecutive accumulator columns of this thread's TMEM lane.
template <int NC>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, float* out) {
#pragma unroll
  for (int c = 0; c < NC / 32; ++c) {
    uint32_t r[32];
    ptx::tmem_ld_32x32b_x32(taddr + 32 * c, r);
#pragma unroll
    for (int j = 0; j < 32; ++j) out[32 * c + j] = __uint_as_float(r[j]);
  }
}

// Read 64 accumulator columns and round them to bf16 pairs (low half = even column), the
// values a bf16 store of the tile would hold.
__device__ __forceinline__ void tmem_load64_bf16(uint32_t taddr, uint32_t* out) {
  uint32_t r0[32], r1[32];
  ptx::tmem_ld_32x32b_x32(taddr, r0);
  ptx::tmem_ld_32x32b_x32(taddr + 32, r1);
  ptx::tmem_wait_ld();
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    out[j] = pack_bf16x2(__uint_as_float(r0[2 * j]), __uint_as_float(r0[2 * j + 1]));
    out[16 + j] = pack_bf16x2(__uint_as_float(r1[2 * j]), __uint_as_float(r1[2 * j + 1]));
  }
}

// One MXFP8 block of 32 bf16 (16 pairs, in order): E8M0 byte by the ceil rule, codes of
// x * 2^-e stored as 32 bytes at dst. The same arithmetic as the quantize kernels.
__device__ __forceinline__ uint32_t quantize_block32(const uint32_t* w, uint8_t* dst, bool v8) {
  uint32_t mx = 0;
#pragma unroll
  for (int k = 0; k < 16; ++k) mx = absmax_bf16x2(mx, w[k]);
  mx = fold_bf16x2(mx);
  float mult;
  const uint32_t sb = mx_scale_byte(mx, &mult);
  uint32_t c[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) c[q] = encode4_scalar(w[2 * q], w[2 * q + 1], mult);
  if (mx > 0x7F80u) {
#pragma unroll
    for (int q = 0; q < 8; ++q) c[q] = fix_nan4(c[q], w[2 * q], w[2 * q + 1]);
  }
  store_seg32(dst, make_uint4(c[0], c[1], c[2], c[3]), make_uint4(c[4], c[5], c[6], c[7]), true,
              true, v8);
  return sb;
}

// Fused MLP epilogue for one thread: row m, columns n .. n+63 of the output (v: 32 bf16
// pairs), in two 32-column chunks. GELU writes h's MXFP8 row copy, then a = gelu(h);
// DGELU forms dh = da * gelu'(h) from h's codes (hc, 64 bytes) and scales (hsc, 2 bytes).
// The result's row copy is thread-local (a chunk is one 1x32 block); for the column copy
// the warp parks its 32 x 32 chunk in shared memory and lane c reads back column c over the
// warp's 32 rows mrow0 .. mrow0+31, which is one 32-row block of the transposed copy.
template <int EPI>
__device__ __forceinline__ void mlp_epilogue(const GemmParams& p, const uint32_t* v,
                                             const uint4* hc, uint32_t hsc, int m, int n,
                                             int mrow0, uint8_t* stage, const void* table,
                                             int lane) {
  const bool v8 = p.o_v8 != 0;
  uint32_t sc_h = 0, sc_o = 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) w[k] = v[16 * j + k];
    if constexpr (EPI == EPI_GELU) {
      sc_h |= quantize_block32(w, p.h_row + int64_t(m) * p.N + n + 32 * j, v8) << (8 * j);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        uint32_t miss = 0;
        const uint32_t a = gelu_bf16x2_nobranch(table, w[k], &miss);
        // an input outside the table (rare): the exact per-element path
        w[k] = miss >= uint32_t(kGeluEntries) ? gelu_bf16x2(table, w[k]) : a;
      }
    } else {
      const uint32_t sb = (hsc >> (8 * j)) & 0xFFu;
      const uint32_t hw[8] = {hc[2 * j].x,     hc[2 * j].y,     hc[2 * j].z,     hc[2 * j].w,
                              hc[2 * j + 1].x, hc[2 * j + 1].y, hc[2 * j + 1].z, hc[2 * j + 1].w};
      if (sb - uint32_t(kDgeluSbLo) < uint32_t(kDgeluSbRows)) {
        // gelu' straight from the code byte through this block's table row
        const float* row = reinterpret_cast<const float*>(table) + (sb - kDgeluSbLo) * 256;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint32_t c = hw[k >> 1] >> (16 * (k & 1));
          const float d0 = __fmul_rn(bf16_lo(w[k]), row[c & 0xFFu]);
          const float d1 = __fmul_rn(bf16_hi(w[k]), row[(c >> 8) & 0xFFu]);
          w[k] = bf16x2_rn_bits(d0, d1);
        }
      } else {
        const float hs = sb == 0xFFu ? __uint_as_float(0x7FC00000u) : exp2i(int(sb) - 127);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          w[k] = dgelu_bf16x2_direct(w[k], hw[k >> 1] >> (16 * (k & 1)), hs);
      }
    }
    sc_o |= quantize_block32(w, p.o_row + int64_t(m) * p.N + n + 32 * j, v8) << (8 * j);

    // column copy: rows of 64 bytes, 16-byte chunk q of row r at q ^ ((r / 2) % 4)
    __syncwarp();                                   // the previous chunk has been read
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(stage + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4)) =
          make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    __syncwarp();
    uint32_t cw[16];
#pragma unroll
    for (int r = 0; r < 32; r += 2) {
      const uint32_t off = (uint32_t(((lane >> 3) ^ ((r >> 1) & 3))) << 4) + 2u * (lane & 7);
      const uint32_t lo = *reinterpret_cast<const uint16_t*>(stage + r * 64 + off);
      const uint32_t hi = *reinterpret_cast<const uint16_t*>(stage + (r + 1) * 64 + off);
      cw[r >> 1] = lo | (hi << 16);
    }
    const int c = n + 32 * j + lane;
    const uint32_t sbc = quantize_block32(cw, p.o_col + int64_t(c) * p.M + mrow0, v8);
    p.o_col_scale[mx_scale_offset(c, mrow0 >> 5, p.M)] = uint8_t(sbc);
  }
  const int64_t so = mx_scale_offset(m, n >> 5, p.N);     // two consecutive blocks
  if constexpr (EPI == EPI_GELU) *reinterpret_cast<uint16_t*>(p.h_scale + so) = uint16_t(sc_h);
  *reinterpret_cast<uint16_t*>(p.o_row_scale + so) = uint16_t(sc_o);
}

template <int MODE, int B128, int CTA2, int EPI>
__device__ __forceinline__ void gemm_tn_body(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                             const CUtensorMap& tmSFA, const CUtensorMap& tmSFB,
                                             const GemmParams& p) {
  using G = Geo<CTA2, EPI>;
  constexpr int kEpiWarps = epi_warps<MODE, EPI>();
  static_assert(EPI == EPI_NONE || MODE == G_MX, "fused MLP epilogues are MXFP8 only");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = ptx::align_smem<1024>(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + G::kStages * kTileABytes;
  uint8_t* sSF = sB + G::kStages * G::kTileBBytes;
  SharedCtl* ctl = reinterpret_cast<SharedCtl*>(sSF + G::kStages * kSfStageBytes);
  uint8_t* sEpi = reinterpret_cast<uint8_t*>(ctl) + 512;   // fused epilogues only

  constexpr int kNumAcc = (MODE == G_MX) ? 1 : 2;
  constexpr int kElem = (MODE == G_BF16) ? 2 : 1;
  constexpr int kBKElems = kBKBytes / kElem;
  constexpr uint32_t kBRows = CTA2 ? kBN / 2 : kBN;     // B rows this CTA loads per stage

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = CTA2 ? ptx::cluster_rank() : 0u;
  const bool leader = rank == 0;
  const int unit = CTA2 ? int(blockIdx.x >> 1) : int(blockIdx.x);       // CTA or CTA pair
  const int n_units = CTA2 ? int(gridDim.x >> 1) : int(gridDim.x);
  const int tiles_m = (p.M + G::kTileM - 1) / G::kTileM;
  const int tiles_n = (p.N + kBN - 1) / kBN;
  const int n_tiles = tiles_m * tiles_n;
  const int nk = (p.K + kBKElems - 1) / kBKElems;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < G::kStages; ++s) {
      ptx::mbar_init(&ctl->full[s], 1);
      ptx::mbar_init(&ctl->empty[s], 1);
      ptx::mbar_init(&ctl->sfr[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&ctl->accf[b], 1);
      ptx::mbar_init(&ctl->acce[b], CTA2 ? 2 * kEpiWarps : kEpiWarps);
    }
    ctl->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (CTA2) {
      ptx::tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(&ctl->tmem_base, kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  __syncthreads();
  if constexpr (CTA2) ptx::cluster_sync();           // peer barriers initialised
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_wait();                      // the previous kernel's writes are visible from here on
  constexpr int kEpiBase = epi_first_warp<MODE, EPI>();

  // ------------------------------------------------------------ scale-factor copier (MXFP8)
  auto sf_copier = [&]() {
    // (leader) Once a stage's loads have landed, copy its E8M0 atoms from shared memory into
    // that stage's TMEM columns (A's own atom, then the pair's two B atoms) and signal the MMA
    // issuer through sfr. A stage's columns are rewritten only after its smem slot has been
    // released by the MMAs that read them and refilled.
    if (lane == 0 && leader) {
      const uint32_t sf_base = tmem + 256;
      int s = 0;
      uint32_t ph = 0;
      for (int tile = unit; tile < n_tiles; tile += n_units) {
        for (int kk = 0; kk < nk; ++kk) {
          if (!wait_bar(&ctl->full[s], ph, ctl, p.status)) goto sf_done;
          ptx::tc_fence_after();
          const uint32_t sfa_t = sf_base + kSfCols * uint32_t(s), sfb_t = sfa_t + 4;
          const uint32_t sf = ptx::smem_u32(sSF + s * kSfStageBytes);
          const uint64_t d0 = ptx::smem_desc(sf, 0, 128, ptx::kSwizzleNone);
          const uint64_t d1 = ptx::smem_desc(sf + 512, 0, 128, ptx::kSwizzleNone);
          const uint64_t d2 = ptx::smem_desc(sf + 1024, 0, 128, ptx::kSwizzleNone);
          if constexpr (CTA2) {
            ptx::tmem_cp_32x128b_warpx4_pair(sfa_t, d0);
            ptx::tmem_cp_32x128b_warpx4_pair(sfb_t, d1);
            ptx::tmem_cp_32x128b_warpx4_pair(sfb_t + 4, d2);
            ptx::mma_commit_pair(&ctl->sfr[s], 0x1);     // the leader's barrier only
          } else {
            ptx::tmem_cp_32x128b_warpx4(sfa_t, d0);
            ptx::tmem_cp_32x128b_warpx4(sfb_t, d1);
            ptx::tmem_cp_32x128b_warpx4(sfb_t + 4, d2);
            ptx::mma_commit(&ctl->sfr[s]);
          }
          if (++s == G::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    sf_done:;
    }
  };

  if (warp < kEpiBase) {
    // With the register split warpgroup 0 hands registers to the epilogue warps (the
    // blockwise promotion holds a 64-column accumulator and a 32-column partial-sum piece).
    if constexpr (reg_split<MODE, EPI>()) ptx::setmaxnreg_dec<kSplitWg0Regs>();
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        if constexpr (MODE == G_MX && CTA2) {
          ptx::prefetch_tmap(&tmSFA);
          ptx::prefetch_tmap(&tmSFB);
        }
        int s = 0;
        uint32_t ph = 0;
        const int kblocks128 = p.K / 128;       // MX scale atoms per operand row tile
        for (int tile = unit; tile < n_tiles; tile += n_units) {
          int mt, nt;
          tile_coords(tile, tiles_m, tiles_n, p.group_n != 0, &mt, &nt);
          const int m0 = mt * G::kTileM + int(rank) * kBM;
          const int n0 = nt * kBN + int(rank) * int(kBRows);
          for (int kk = 0; kk < nk; ++kk) {
            const int kb = k_block<MODE>(tile, unit, n_units, kk, nk);
            if (!wait_bar(&ctl->empty[s], ph ^ 1u, ctl, p.status)) goto producer_done;
            const uint32_t stall = (unit == 0 && tile == 0 && kk == 0) ? p.stall_tx : 0u;
            uint8_t* a_dst = sA + s * kTileABytes;
            uint8_t* b_dst = sB + s * G::kTileBBytes;
            if constexpr (CTA2) {
              // Both CTAs' loads complete on the leader's barrier, which expects all of them.
              // MXFP8: each CTA also brings its own 512-byte A-scale atom and both B-scale atoms
              // of the pair's 256 B rows (the scale-factor arrays are viewed as rows of 256 B).
              const uint32_t bar = ptx::map_to_rank(&ctl->full[s], 0);
              constexpr uint32_t sf_bytes = MODE == G_MX ? 512u + 1024u : 0u;
              if (leader)
                ptx::mbar_arrive_expect_tx(&ctl->full[s],
                                           2 * (kTileABytes + G::kTileBBytes + sf_bytes) + stall);
              // a K-major tile is 128 bytes of K x rows; an MN-major one 128 of M (N) x 128 K rows
              if (p.a_mn) ptx::tma_load_2d_pair(a_dst, &tmA, m0, kb * kBKElems, bar);
              else ptx::tma_load_2d_pair(a_dst, &tmA, kb * kBKElems, m0, bar);
              if (p.b_mn) ptx::tma_load_2d_pair(b_dst, &tmB, n0, kb * kBKElems, bar);
              else ptx::tma_load_2d_pair(b_dst, &tmB, kb * kBKElems, n0, bar);
              if constexpr (MODE == G_MX) {
                uint8_t* sf = sSF + s * kSfStageBytes;
                const int nb_pair = nt * kBN;                        // first B row of the pair
                ptx::tma_load_2d_pair(sf, &tmSFA, 0, 2 * ((m0 >> 7) * kblocks128 + kb), bar);
                ptx::tma_load_2d_pair(sf + 512, &tmSFB, 0,
                                      2 * ((nb_pair >> 7) * kblocks128 + kb), bar);
                ptx::tma_load_2d_pair(sf + 1024, &tmSFB, 0,
                                      2 * (((nb_pair >> 7) + 1) * kblocks128 + kb), bar);
              }
            } else {
              uint32_t bytes = kTileABytes + G::kTileBBytes + stall;
              const bool sfb_hi = (n0 + 128) < p.N;
              if constexpr (MODE == G_MX) bytes += 512u + (sfb_hi ? 1024u : 512u);
              ptx::mbar_arrive_expect_tx(&ctl->full[s], bytes);
              if (p.a_mn) ptx::tma_load_2d(a_dst, &tmA, m0, kb * kBKElems, &ctl->full[s]);
              else ptx::tma_load_2d(a_dst, &tmA, kb * kBKElems, m0, &ctl->full[s]);
              if (p.b_mn) {
                // the 256-wide B tile as two 128-column boxes, 16 KiB apart
                ptx::tma_load_2d(b_dst, &tmB, n0, kb * kBKElems, &ctl->full[s]);
                ptx::tma_load_2d(b_dst + 16384, &tmB, n0 + 128, kb * kBKElems, &ctl->full[s]);
              } else {
                ptx::tma_load_2d(b_dst, &tmB, kb * kBKElems, n0, &ctl->full[s]);
              }
              if constexpr (MODE == G_MX) {
                uint8_t* sf = sSF + s * kSfStageBytes;
                ptx::bulk_load(sf, p.sfa + (int64_t(m0 >> 7) * kblocks128 + kb) * 512, 512,
                               &ctl->full[s]);
                ptx::bulk_load(sf + 512, p.sfb + (int64_t(n0 >> 7) * kblocks128 + kb) * 512, 512,
                               &ctl->full[s]);
                if (sfb_hi)
                  ptx::bulk_load(sf + 1024,
                                 p.sfb + (int64_t((n0 >> 7) + 1) * kblocks128 + kb) * 512, 512,
                                 &ctl->full[s]);
              }
            }
            if (++s == G::kStages) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
      producer_done:;
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer (leader)
      if (lane == 0 && leader) {
        // operand formats (E4M3 = 0, E5M2 = 1) in descriptor bits 7-9 (A) and 10-12 (B)
        uint32_t idesc = instr_desc<MODE, CTA2>();
        if constexpr (MODE == G_TENSOR || MODE == G_BLOCK)
          idesc |= (uint32_t(p.a_fmt) << 7) | (uint32_t(p.b_fmt) << 10) |
                   (uint32_t(p.a_mn) << 15) | (uint32_t(p.b_mn) << 16);   // operand majorness
        if constexpr (MODE == G_MX)      // E5M2 gradients of power-of-two blockwise under hybrid
          idesc |= (uint32_t(p.a_fmt) << 7) | (uint32_t(p.b_fmt) << 10);
        const uint32_t sf_base = tmem + 256;      // MX scale factors: kSfCols columns a stage
        // Operand descriptors of stage 0's first K = 32 slice. Between stages and slices only the
        // start-address field (bits 0-13, 16-byte units) changes, and an address inside shared
        // memory never carries out of it, so the loop steps the descriptors by plain adds.
        // K-major: rows of 128 bytes of K, the k-th slice 32 bytes in. MN-major: rows of 128 MN
        // elements, one per K, the slice 32 rows = 4 KiB in; 8-row swizzle atoms 1 KiB apart
        // (SBO), 128-column chunks 16 KiB apart (LBO).
        const uint64_t adesc0 =
            ptx::smem_desc(ptx::smem_u32(sA), p.a_mn ? 16384 : 16, 1024, ptx::kSwizzle128B);
        const uint64_t bdesc0 =
            ptx::smem_desc(ptx::smem_u32(sB), p.b_mn ? 16384 : 16, 1024, ptx::kSwizzle128B);
        const uint32_t astep = p.a_mn ? 4096 / 16 : 32 / 16, bstep = p.b_mn ? 4096 / 16 : 32 / 16;
        // MX: the instruction descriptor of K slice k also selects the slice's scale factors
        uint32_t idk[kBKBytes / 32];
  #pragma unroll
        for (int k = 0; k < kBKBytes / 32; ++k)
          idk[k] = MODE == G_MX ? idesc | (uint32_t(k) << 29) | (uint32_t(k) << 4) : idesc;
        int s = 0;
        uint32_t ph = 0;
        uint32_t u = 0;
        // stage s's operand descriptors and scale-factor columns, stepped with s
        uint64_t ad_s = adesc0, bd_s = bdesc0;
        uint32_t sfa_t = sf_base;
        auto commit = [&](uint64_t* bar) {
          if constexpr (CTA2) ptx::mma_commit_pair(bar, 0x3);
          else ptx::mma_commit(bar);
        };
        for (int tile = unit; tile < n_tiles; tile += n_units) {
          uint32_t d_t = tmem;
          if constexpr (MODE != G_BLOCK) {
            const uint32_t b = u % kNumAcc;
            if (!wait_bar(&ctl->acce[b], ((u / kNumAcc) & 1u) ^ 1u, ctl, p.status)) goto mma_done;
            ptx::tc_fence_after();
            d_t = tmem + b * kBN;
          }
          for (int kk = 0; kk < nk; ++kk) {
            uint32_t b = 0;
            if constexpr (MODE == G_BLOCK) {
              b = u & 1u;
              if (!wait_bar(&ctl->acce[b], ((u >> 1) & 1u) ^ 1u, ctl, p.status)) goto mma_done;
              ptx::tc_fence_after();
              d_t = tmem + b * kBN;
            }
            // MX: the scale-factor warp signals once the stage's operands have landed and its
            // scales are in TMEM; other modes wait for the operands themselves
            uint64_t* ready = MODE == G_MX ? &ctl->sfr[s] : &ctl->full[s];
            if (!wait_bar(ready, ph, ctl, p.status)) goto mma_done;
            ptx::tc_fence_after();
            const uint32_t sfb_t = sfa_t + 4;
  #pragma unroll
            for (int k = 0; k < kBKBytes / 32; ++k) {
              const uint64_t ad = ad_s + astep * uint32_t(k);
              const uint64_t bd = bd_s + bstep * uint32_t(k);
              const uint32_t acc_on = MODE == G_BLOCK ? uint32_t(k != 0) : uint32_t((kk | k) != 0);
              if constexpr (CTA2) {
                if constexpr (MODE == G_BF16) {
                  ptx::mma_f16_pair(d_t, ad, bd, idesc, acc_on);
                } else if constexpr (MODE == G_MX) {
                  ptx::mma_mxf8f6f4_pair(d_t, ad, bd, idk[k], sfa_t, sfb_t, acc_on);
                } else {
                  ptx::mma_f8f6f4_pair(d_t, ad, bd, idesc, acc_on);
                }
              } else if constexpr (MODE == G_MX) {
                ptx::mma_mxf8f6f4(d_t, ad, bd, idk[k], sfa_t, sfb_t, acc_on);
              } else if constexpr (MODE == G_BF16) {
                ptx::mma_f16(d_t, ad, bd, idesc, acc_on);
              } else {
                ptx::mma_f8f6f4(d_t, ad, bd, idesc, acc_on);
              }
            }
            commit(&ctl->empty[s]);
            if constexpr (MODE == G_BLOCK) {
              commit(&ctl->accf[b]);
              ++u;
            }
            if (++s == G::kStages) {
              s = 0;
              ph ^= 1u;
              ad_s = adesc0;
              bd_s = bdesc0;
              sfa_t = sf_base;
            } else {
              ad_s += kTileABytes >> 4;
              bd_s += G::kTileBBytes >> 4;
              sfa_t += kSfCols;
            }
          }
          if constexpr (MODE != G_BLOCK) {
            commit(&ctl->accf[u % kNumAcc]);
            ++u;
          }
        }
      mma_done:;
      }
    } else if (warp == 2) {
      if constexpr (MODE == G_MX && reg_split<MODE, EPI>()) sf_copier();
    }
  } else if (warp < kEpiBase + kEpiWarps) {
    // ------------------------------------------------------------ epilogue warps
    if constexpr (reg_split<MODE, EPI>()) ptx::setmaxnreg_inc<kSplitEpiRegs>();
    const int ew = warp - kEpiBase;
    const int quad = warp & 3;            // TMEM lane quadrant this warp may access
    constexpr int kCols = 4 * kBN / kEpiWarps;              // accumulator columns per warp

    const int slice = ew >> 2;            // which kCols columns of the 256-wide tile
    const int row = 32 * quad + lane;
    const uint32_t t_lane = tmem + (uint32_t(32 * quad) << 16) + uint32_t(slice * kCols);
    // accumulator-empty arrivals go to the leader's barrier (a remote arrive from the peer)
    auto release_acc = [&](uint32_t b) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CTA2) ptx::mbar_arrive_cluster(ptx::map_to_rank(&ctl->acce[b], 0));
        else ptx::mbar_arrive(&ctl->acce[b]);
      }
    };
    if constexpr (EPI != EPI_NONE) {
      // ---- fused MLP epilogue (MXFP8, single accumulator)
      uint8_t* stage = sEpi + ew * kEpiStageBytes;
      void* table = sEpi + kEpiWarps * kEpiStageBytes;
      const int et = int(threadIdx.x) - 32 * kEpiBase;       // thread index among them
      if constexpr (EPI == EPI_GELU) gelu_table_fill(table, et, 32 * kEpiWarps);
      else dgelu_code_table_fill(table, et, 32 * kEpiWarps);
      asm volatile("bar.sync 1, %0;" ::"r"(32 * kEpiWarps) : "memory");   // epilogue warps only
      uint32_t u = 0;
      for (int tile = unit; tile < n_tiles; tile += n_units) {
        int mt, nt;
        tile_coords(tile, tiles_m, tiles_n, p.group_n != 0, &mt, &nt);
        const int m0 = mt * G::kTileM + int(rank) * kBM;
        const int n0 = nt * kBN;
        const int m = m0 + row, n = n0 + slice * kCols;
        const int mrow0 = m0 + 32 * quad;
        // M and N are multiples of 128, so a warp's 32 rows x 64 columns are all in or all out
        const bool live = mrow0 < p.M && n < p.N;
        uint4 hc[4];
        uint32_t hsc = 0;
        if constexpr (EPI == EPI_DGELU) {
          // h's codes and scales do not depend on the accumulator: fetch them first, and ask
          // L2 for the next tile's (its loads then wait on L2, not on DRAM)
          if (live) {
            const uint8_t* src = p.h_row + int64_t(m) * p.N + n;
#pragma unroll
            for (int i = 0; i < 4; ++i) hc[i] = ldg_nc_v4(src + 16 * i);
            hsc = __ldg(reinterpret_cast<const uint16_t*>(p.h_scale +
                                                          mx_scale_offset(m, n >> 5, p.N)));
          }
          const int nx = tile + n_units;
          if (nx < n_tiles) {
            int mt2, nt2;
            tile_coords(nx, tiles_m, tiles_n, p.group_n != 0, &mt2, &nt2);
            const int m2 = mt2 * G::kTileM + int(rank) * kBM + row, n2 = nt2 * kBN + slice * kCols;
            if (m2 < p.M && n2 < p.N) {
              prefetch_l2(p.h_row + int64_t(m2) * p.N + n2);          // 64 bytes, one line
              if ((lane & 7) == 0)
                prefetch_l2(p.h_scale + mx_scale_offset(m2, n2 >> 5, p.N));
            }
          }
        }
        if (!wait_bar(&ctl->accf[0], u & 1u, ctl, p.status)) break;
        ptx::tc_fence_after();
        uint32_t v[32];
        tmem_load64_bf16(t_lane, v);
        release_acc(0);
        ++u;
        if (live) mlp_epilogue<EPI>(p, v, hc, hsc, m, n, mrow0, stage, table, lane);
      }
    } else {
    float alpha = 1.0f;
    if constexpr (MODE == G_TENSOR) alpha = __fmul_rn(*p.a_sinv, *p.b_sinv);
    uint32_t u = 0;
    float acc[kCols];
    for (int tile = unit; tile < n_tiles; tile += n_units) {
      int mt, nt;
      tile_coords(tile, tiles_m, tiles_n, p.group_n != 0, &mt, &nt);
      const int m0 = mt * G::kTileM + int(rank) * kBM;
      const int n0 = nt * kBN;
      const int m = m0 + row, n = n0 + slice * kCols;
      if constexpr (MODE != G_BLOCK) {
        const uint32_t b = u % kNumAcc;
        if (!wait_bar(&ctl->accf[b], (u / kNumAcc) & 1u, ctl, p.status)) break;
        ptx::tc_fence_after();
        tmem_load_cols<kCols>(t_lane + b * kBN, acc);
        ptx::tmem_wait_ld();
        release_acc(b);
        ++u;
        if constexpr (MODE == G_TENSOR) {
#pragma unroll
          for (int j = 0; j < kCols; ++j) acc[j] = __fmul_rn(acc[j], alpha);
        }
      } else {
        // Blockwise promotion: chunk kb's partial sum P (fp32 in TMEM) is added into the
        // register accumulator as acc += P * (s_inv(A row, kb) * s_inv(B, kb)), two columns
        // per packed FMA. Chunk kb + 1's scales are fetched while chunk kb is promoted. With
        // per-row B scales (1x128, wgrad) the warp's 64 column scales of a chunk go straight
        // from global to the warp's slice of the (otherwise unused) scale-factor region of
        // shared memory with cp.async, two chunk buffers a warp, and are read back as
        // broadcasts, so no registers hold them in flight.
        static_assert(MODE != G_BLOCK || B128 || kEpiWarps * kCols * 8 <= G::kStages * kSfStageBytes,
                      "per-warp B-scale buffers fit in the scale-factor region");
        const int kblocks = p.K / 128;
        float2 acc2[kCols / 2];
#pragma unroll
        for (int j = 0; j < kCols / 2; ++j) acc2[j] = make_float2(0.0f, 0.0f);
        auto load_sa = [&](int kb) { return m < p.M ? __ldg(p.a_bs + int64_t(kb) * p.M + m) : 0.0f; };
        auto load_sb = [&](int kb) {
          float v = 0.0f;
          if (n < p.N)
            v = p.b_mn ? __ldg(p.b_bs + int64_t(kb) * (p.N >> 7) + (n >> 7))   // grid [K][N]
                       : __ldg(p.b_bs + int64_t(n >> 7) * kblocks + kb);        // grid [N][K]
          return v;
        };
        float2* sbw = reinterpret_cast<float2*>(sSF) + ew * kCols;      // 2 x 32 float2
        auto fetch_sb = [&](int kb) {
          float2* dst = sbw + (kb & 1) * (kCols / 2) + lane;
          if (n < p.N) ptx::cp_async_8(dst, p.b_bs + int64_t(kb) * p.N + n + 2 * lane);
          else *dst = make_float2(0.0f, 0.0f);
          ptx::cp_async_commit();
        };
        float sa_nx = load_sa(0);
        float sb_nx = 0.0f;
        if constexpr (B128 != 0) sb_nx = load_sb(0);
        else {
          __syncwarp();                    // the previous tile's reads of buffer 0 are done
          fetch_sb(0);
        }
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          const float sa = sa_nx;
          const float sb = sb_nx;
          if (kb + 1 < kblocks) {
            sa_nx = load_sa(kb + 1);
            if constexpr (B128 != 0) sb_nx = load_sb(kb + 1);
          }
          if constexpr (B128 == 0) {
            __syncwarp();                  // chunk kb - 1's reads of the other buffer are done
            if (kb + 1 < kblocks) {
              fetch_sb(kb + 1);
              ptx::cp_async_wait<1>();     // chunk kb's group has landed
            } else {
              ptx::cp_async_wait<0>();
            }
            __syncwarp();
          }
          const uint32_t b = u & 1u;
          if (!wait_bar(&ctl->accf[b], (u >> 1) & 1u, ctl, p.status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const float f = __fmul_rn(sa, sb);
          const float2 f2 = make_float2(f, f), sa2 = make_float2(sa, sa);
          // 32 columns a TMEM load (two round trips a chunk): the epilogue warpgroups run with
          // kSplitEpiRegs registers, room for the 64-column accumulator and a 32-column piece
          const float4* sb4 = reinterpret_cast<const float4*>(sbw + (kb & 1) * (kCols / 2));
#pragma unroll
          for (int c = 0; c < kCols / 32; ++c) {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(t_lane + b * kBN + 32 * c, r);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float2 pr = make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
              if constexpr (B128 != 0) {
                acc2[16 * c + j] = __ffma2_rn(pr, f2, acc2[16 * c + j]);
              } else {
                // (P * s_inv(B column)) * s_inv(A row): the partials take the column scale in
                // place, so no product registers are needed
                const float4 q = sb4[8 * c + (j >> 1)];
                pr = __fmul2_rn(pr, (j & 1) ? make_float2(q.z, q.w) : make_float2(q.x, q.y));
                acc2[16 * c + j] = __ffma2_rn(pr, sa2, acc2[16 * c + j]);
              }
            }
          }
          release_acc(b);
          ++u;
        }
        if constexpr (B128 == 0) ptx::cp_async_wait<0>();   // nothing left in flight on exit
#pragma unroll
        for (int j = 0; j < kCols / 2; ++j) {
          acc[2 * j] = acc2[j].x;
          acc[2 * j + 1] = acc2[j].y;
        }
        if (!ok) break;
      }
      store_row<kCols>(p, m, n, acc);
    }
    }
  } else if constexpr (MODE == G_MX && !reg_split<MODE, EPI>()) {
    sf_copier();
  }

  __syncthreads();
  if (*reinterpret_cast<volatile int*>(&ctl->abort_flag)) {
    // Let copies and MMAs already in flight land before the CTA's memory is released.
    const uint64_t t0 = ptx::clock64_();
    while (ptx::clock64_() - t0 < 20000000ull) {
    }
  }
  if constexpr (CTA2) ptx::cluster_sync();           // the pair is done with both TMEMs
  if (warp == 1) {
    ptx::tc_fence_after();
    if constexpr (CTA2) ptx::tmem_dealloc_pair(tmem, kTmemCols);
    else ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Plain GEMMs: 10 warps (11 for MXFP8); some SM sub-partitions hold three of them, so at most
// 168 registers a thread.
template <int MODE, int B128, int CTA2>
__global__ void __maxnreg__(168)
    gemm_tn_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmSFA,
                   const __grid_constant__ CUtensorMap tmSFB, const GemmParams p) {
  gemm_tn_body<MODE, B128, CTA2, EPI_NONE>(tmA, tmB, tmSFA, tmSFB, p);
}

// Fused MLP GEMMs: 19 warps (TMA producer, MMA issuer, 16 epilogue warps, scale-factor
// copier), five on three of the sub-partitions, so at most 96 registers.
template <int CTA2, int EPI>
__global__ void __maxnreg__(96)
    gemm_mlp_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmSFA,
                    const __grid_constant__ CUtensorMap tmSFB, const GemmParams p) {
  gemm_tn_body<G_MX, 1, CTA2, EPI>(tmA, tmB, tmSFA, tmSFB, p);
}

// Blockwise GEMMs: 20 warps (warpgroup 0: TMA producer, MMA issuer and two idle warps; four
// warpgroups of promoting epilogue warps), launched at kSplitLaunchRegs registers a thread;
// setmaxnreg then moves registers from warpgroup 0 (kSplitWg0Regs) to the epilogue warpgroups
// (kSplitEpiRegs).
template <int MODE, int B128, int CTA2>
__global__ void __maxnreg__(kSplitLaunchRegs)
    gemm_wide_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmSFA,
                     const __grid_constant__ CUtensorMap tmSFB, const GemmParams p) {
  gemm_tn_body<MODE, B128, CTA2, EPI_NONE>(tmA, tmB, tmSFA, tmSFB, p);
}

// ------------------------------------------------------------------------------------
// Host side: tensor maps and launch
// ------------------------------------------------------------------------------------

// 2D K-major operand [rows][k] (elements of elem_bytes), box = 128 bytes of K x box_rows.
static bool make_operand_map(CUtensorMap* map, const void* base, int64_t rows, int64_t k,
                             int elem_bytes, int box_rows) {
  return make_tmap_2d(map, base, elem_bytes, k, rows, kBKBytes / elem_bytes, box_rows, true);
}

template <int MODE, int B128, int CTA2, int EPI = EPI_NONE>
static cudaError_t launch_mode(const GemmLaunch& g, cudaStream_t st) {
  using G = Geo<CTA2, EPI>;
  static_assert(EPI == EPI_NONE || (MODE == G_MX && B128 == 1), "fused: MXFP8 only");
  CUtensorMap ma, mb;
  const int eb = MODE == G_BF16 ? 2 : 1;
  // K-major operands [rows][K]: boxes of 128 bytes of K x the tile's rows; MN-major operands
  // [K][rows]: boxes of 128 rows' worth of columns x 128 K rows
  const bool okA = g.p.a_mn ? make_tmap_2d(&ma, g.A, 1, g.p.M, g.p.K, 128, kBKBytes, true)
                            : make_operand_map(&ma, g.A, g.p.M, g.p.K, eb, kBM);
  const bool okB = g.p.b_mn ? make_tmap_2d(&mb, g.B, 1, g.p.N, g.p.K, 128, kBKBytes, true)
                            : make_operand_map(&mb, g.B, g.p.N, g.p.K, eb, CTA2 ? kBN / 2 : kBN);
  if (!okA || !okB) return cudaErrorInvalidValue;
  // MXFP8 scale arrays viewed as rows of 256 bytes (two rows per 512-byte atom) for TMA.
  CUtensorMap msfa = ma, msfb = mb;
  if (MODE == G_MX && CTA2) {
    const int64_t kb = g.p.K / 128;
    if (!make_tmap_2d(&msfa, g.p.sfa, 1, 256, 2 * (int64_t(g.p.M) / 128) * kb, 256, 2, false))
      return cudaErrorInvalidValue;
    if (!make_tmap_2d(&msfb, g.p.sfb, 1, 256, 2 * (int64_t(g.p.N) / 128) * kb, 256, 2, false))
      return cudaErrorInvalidValue;
  }
  auto kern = [] {
    if constexpr (EPI != EPI_NONE) return gemm_mlp_kernel<CTA2, EPI>;
    else if constexpr (MODE == G_BLOCK) return gemm_wide_kernel<MODE, B128, CTA2>;
    else return gemm_tn_kernel<MODE, B128, CTA2>;
  }();
  static ContextOnce attr_done{};
  cudaError_t ae = once_per_context(attr_done, [&] {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(G::kSmemBytes));
    if (e == cudaSuccess && CTA2)
      (void)cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
    if (e == cudaSuccess && reg_split<MODE, EPI>()) {
      // The register split (setmaxnreg) is sized for a launch at exactly kSplitLaunchRegs a
      // thread; with fewer the epilogue warps could never get theirs.
      cudaFuncAttributes fa{};
      e = cudaFuncGetAttributes(&fa, kern);
      if (e == cudaSuccess && fa.numRegs != kSplitLaunchRegs) e = cudaErrorInvalidConfiguration;
    }
    return e;
  });
  if (ae != cudaSuccess) return ae;
  const int sms = num_sms();
  const int tiles = ((g.p.M + G::kTileM - 1) / G::kTileM) * ((g.p.N + kBN - 1) / kBN);
  const int units = std::max(1, std::min(tiles, CTA2 ? sms / 2 : sms));
  cudaLaunchAttribute cluster;
  cluster.id = cudaLaunchAttributeClusterDimension;
  cluster.val.clusterDim.x = CTA2 ? 2 : 1;
  cluster.val.clusterDim.y = 1;
  cluster.val.clusterDim.z = 1;
  return launch_kernel(kern, dim3(unsigned(units * (CTA2 ? 2 : 1))),
                       dim3(gemm_threads<MODE, EPI>()), G::kSmemBytes, st, &cluster, ma, mb,
                       msfa, msfb, g.p);
}

cudaError_t gemm_launch(const GemmLaunch& g, cudaStream_t st) {
  if (g.p.M == 0 || g.p.N == 0) return cudaSuccess;
  GemmLaunch gl = g;
  const int64_t pitch = gl.p.ldd * (gl.p.d_fp32 ? 4 : 2);
  gl.p.d_v8 = (reinterpret_cast<uintptr_t>(gl.p.D) % 32 == 0) && (pitch % 32 == 0);
  if ((gl.p.a_mn && gl.mode != G_TENSOR) ||
      (gl.p.b_mn && gl.mode != G_TENSOR && !(gl.mode == G_BLOCK && gl.p.b_is_128)))
    return cudaErrorInvalidValue;                       // MN-major: per-tensor / 128x128 only
  if (gl.epi != EPI_NONE) {
    if (gl.mode != G_MX) return cudaErrorInvalidValue;
    auto a32 = [](const void* q) { return reinterpret_cast<uintptr_t>(q) % 32 == 0; };
    gl.p.o_v8 = a32(gl.p.o_row) && a32(gl.p.o_col) && (gl.epi != EPI_GELU || a32(gl.p.h_row));
  }
  // Group along the smaller operand: its panels are the ones kept in L2 across the rounds of
  // tiles, while the larger one streams through once per group.
  gl.p.group_n = gl.p.M > gl.p.N;

  // CTA pairs whenever there are at least two 128-row halves to give them.
  // (Blockwise keeps the single CTA: its per-chunk promotion would couple the pair's
  // epilogues to every K step.)
  const bool pair = gl.p.M > kBM;
  switch (gl.mode) {
    case G_TENSOR:
      return pair ? launch_mode<G_TENSOR, 1, 1>(gl, st) : launch_mode<G_TENSOR, 1, 0>(gl, st);
    case G_MX: {
      const bool p2 = pair && gl.p.N > kBM;
      if (gl.epi == EPI_GELU)
        return p2 ? launch_mode<G_MX, 1, 1, EPI_GELU>(gl, st)
                  : launch_mode<G_MX, 1, 0, EPI_GELU>(gl, st);
      if (gl.epi == EPI_DGELU)
        return p2 ? launch_mode<G_MX, 1, 1, EPI_DGELU>(gl, st)
                  : launch_mode<G_MX, 1, 0, EPI_DGELU>(gl, st);
      return p2 ? launch_mode<G_MX, 1, 1>(gl, st) : launch_mode<G_MX, 1, 0>(gl, st);
    }
    case G_BLOCK:
      return gl.p.b_is_128 ? launch_mode<G_BLOCK, 1, 0>(gl, st) : launch_mode<G_BLOCK, 0, 0>(gl, st);
    case G_BF16:
      return pair ? launch_mode<G_BF16, 1, 1>(gl, st) : launch_mode<G_BF16, 1, 0>(gl, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fp8lin
