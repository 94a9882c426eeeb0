// Host-side interfaces between the C ABI (api.cu) and the kernel files.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "fp8lin.h"

struct CUtensorMap_st;

namespace fp8lin {

// ---- tma.cu
// 2-D tensor map over a row-major [rows][inner] array (elements of elem_bytes); box of
// box_inner x box_rows elements; optional 128-byte swizzle; out-of-bounds reads fill zeros.
bool make_tmap_2d(CUtensorMap_st* map, const void* base, int elem_bytes, int64_t inner,
                  int64_t rows, int box_inner, int box_rows, bool swizzle128);
int num_sms();      // of the current device
int64_t l2_bytes(); // L2 cache size of the current device

// Programmatic dependent launch: every kernel of the library lets the next kernel in its
// stream start launching as soon as all of its own CTAs are running, and waits for the kernel
// before it (griddepcontrol.wait) before its first global memory access. The next kernel's
// launch and prologue (barrier setup, TMEM allocation) then overlap this one's tail.
// Environment FP8LIN_PDL=0 turns the launch attribute off (read once per process).
bool pdl_enabled();

// cudaLaunchKernelEx with the programmatic-serialisation attribute (when enabled) plus up to
// one extra attribute (a cluster shape).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, const cudaLaunchAttribute* extra, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (extra != nullptr) attr[n++] = *extra;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Unique id of the calling thread's current CUDA context (cuCtxGetId), or 0 when no context
// is current or the driver cannot say. Ids are never reused within a process, so a setup
// keyed on them is redone in a new context: after cudaDeviceReset, or when the caller makes
// its own context current.
unsigned long long current_context_id();

// Errors of a CUDA call as a status; FP8_ERR_CUDA also records the error's text for
// fp8_last_cuda_error() (per host thread).
fp8_status cuda_status(cudaError_t e);

constexpr int kMaxDevices = 64;

// The contexts in which a per-context setup has run: one slot per device, holding the id of
// the context it last ran in.
struct ContextOnce {
  std::atomic<unsigned long long> ctx[kMaxDevices];
};

// Run set() (an idempotent per-context setup such as cudaFuncSetAttribute) the first time the
// current context reaches this flag; later calls in the same context skip it. A different
// context on the device (after cudaDeviceReset, or another context made current) runs it
// again. Thread-safe: concurrent first calls may both run set(), which is harmless. Devices
// beyond kMaxDevices, or a context whose id is unknown, run it every time.
template <class Set>
cudaError_t once_per_context(ContextOnce& done, Set set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool slot = dev >= 0 && dev < kMaxDevices;
  unsigned long long id = current_context_id();
  if (slot && id != 0 && done.ctx[dev].load(std::memory_order_acquire) == id) return cudaSuccess;
  e = set();
  if (e != cudaSuccess) return e;
  if (id == 0) id = current_context_id();          // set() may have made the context current
  if (slot && id != 0) done.ctx[dev].store(id, std::memory_order_release);
  return cudaSuccess;
}

// ---- quantize.cu
size_t quantize_workspace_bytes(int kind, int64_t R, int64_t C);
int amax_partial_ctas(int64_t n_vec);      // CTAs (= partials) of the tensorwise amax pass
// fmt: 0 = E4M3, 1 = E5M2 (gradients under the hybrid format; not for MXFP8)
// pow2: power-of-two block scales (blockwise only)
cudaError_t quantize_launch(int kind, int role, int fmt, bool pow2, int margin,
                            const uint16_t* x, int64_t R, int64_t C, bool want_row,
                            bool want_col, bool col_bf16, fp8_tensor* out, void* workspace,
                            int32_t* status, cudaStream_t st, uint32_t stall_tx = 0);
// One tensor of a grouped quantize (fp8_quantize_group), checked by the caller.
struct QuantGroupItem {
  const uint16_t* x;
  int64_t R, C;
  int role;
  bool want_row, want_col, col_bf16;
  bool e5;                  // blockwise, hybrid format, role GRAD: E5M2 codes
  fp8_tensor* out;
};
// kind: FP8_RECIPE_MXFP8 or FP8_RECIPE_BLOCKWISE (pow2 and margin apply to blockwise).
cudaError_t quantize_group_launch(int kind, bool pow2, int margin, int n,
                                  const QuantGroupItem* items, int32_t* status, cudaStream_t st,
                                  uint32_t stall_tx = 0);
cudaError_t gelu_quantize_launch(const uint16_t* h, int64_t R, int64_t C, uint16_t* a_bf16,
                                 fp8_tensor* a_q, fp8_tensor* h_q, int32_t* status,
                                 cudaStream_t st);
cudaError_t dgelu_quantize_launch(const uint16_t* da, const fp8_tensor* h_q, int64_t R,
                                  int64_t C, uint16_t* dh_bf16, fp8_tensor* dh_q,
                                  int32_t* status, cudaStream_t st);
cudaError_t amax_update_launch(float* hist, int32_t* head, int len, const float* amax_new,
                               float* scale, float* scale_inv, int margin, float fmax,
                               int algo, cudaStream_t st);

// ---- master.cu (fp32 master weights -> E4M3, role WEIGHT)
cudaError_t quantize_master_launch(int kind, int margin, const float* x, int64_t R, int64_t C,
                                   bool want_row, bool want_col, fp8_tensor* out,
                                   void* workspace, cudaStream_t st);

// ---- gemm.cu
enum GMode : int { G_TENSOR = 0, G_MX = 1, G_BLOCK = 2, G_BF16 = 3 };

// Epilogue kinds of the MLP block's fused steps (GeLU forward / backward).
enum MlpEpi : int { EPI_NONE = 0, EPI_GELU = 1, EPI_DGELU = 2 };

struct GemmParams {
  int M, N, K;              // D[M][N] = sum_k A[M][K] B[N][K]; K in elements
  void* D;
  int64_t ldd;
  int d_fp32;
  int d_v8;                 // D and its row pitch are 32-byte aligned (256-bit stores)
  const float* a_sinv;      // G_TENSOR: per-tensor dequantisation factors
  const float* b_sinv;
  const uint8_t* sfa;       // G_MX: E8M0 scales in the tiled atom order
  const uint8_t* sfb;
  const float* a_bs;        // G_BLOCK: A 1x128 s_inv, [K/128][M]
  const float* b_bs;        // G_BLOCK: B 128x128 grid [N/128][K/128] or 1x128 [K/128][N]
  int b_is_128;
  int32_t* status;          // device status word (may be null)
  int a_fmt, b_fmt;         // G_TENSOR / G_BLOCK operand formats: 0 = E4M3, 1 = E5M2
  // MN-major operands (G_TENSOR: A and/or B; G_BLOCK: B, a 128x128 weight): the operand is
  // stored [K][M] / [K][N] (the other copy of the tensor) and read transposed by the MMA. For
  // G_BLOCK the B scales are then the row grid [K/128][N/128].
  int a_mn, b_mn;
  // Fused MLP epilogues (G_MX only; the tile is quantised instead of stored, D unused):
  //   GELU : h = bf16(acc) -> h_row/h_scale (MXFP8 row copy), a = gelu(h) -> o_*
  //   DGELU: da = bf16(acc), h read from h_row/h_scale, dh = da * gelu'(h) -> o_*
  uint8_t* h_row;           // [M][N] codes
  uint8_t* h_scale;         // E8M0, tiled atoms of the [M][N] tensor
  uint8_t* o_row;           // [M][N] codes of a / dh
  uint8_t* o_row_scale;
  uint8_t* o_col;           // [N][M] codes (column-wise copy)
  uint8_t* o_col_scale;     // E8M0, tiled atoms of the [N][M] tensor
  int o_v8;                 // all of the above code arrays are 32-byte aligned
  // Failure-detection test hook (0 otherwise): extra bytes the first stage of the first CTA
  // (pair) expects, so that stage's barrier never completes and the kernel's bounded waits
  // run out (fp8_test_linear_fwd_stalled).
  uint32_t stall_tx;
  // Tile order: 0 walks a group of M tiles first (A's panels are reused from L2 across the
  // rounds of tiles), 1 a group of N tiles (B's panels are). The host picks the smaller operand.
  int group_n;
};

struct GemmLaunch {
  int mode;                 // GMode
  int epi;                  // MlpEpi (0 = plain bf16/fp32 store)
  const void* A;            // [M][K] codes (bf16 for G_BF16)
  const void* B;            // [N][K]
  GemmParams p;
};

cudaError_t gemm_launch(const GemmLaunch& g, cudaStream_t st);

}  // namespace fp8lin
