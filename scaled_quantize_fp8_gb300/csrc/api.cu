// extern "C" entry points of the FP8 linear-layer library (declared in include/fp8lin.h).
// Arguments are checked on the host before anything is enqueued; every launch goes to the
// caller's stream; no entry point allocates, frees or synchronises.
#include <cstdint>
#include <cstring>

#include "internal.cuh"
#include "fp8lin_test.h"


using namespace fp8lin;

namespace {
thread_local const char* g_last_cuda_error = "";
}  // namespace

fp8_status fp8lin::cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return FP8_OK;
  g_last_cuda_error = cudaGetErrorString(e);
  return FP8_ERR_CUDA;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fp8_status check_ptr(const void* p) {
  if (p == nullptr) return FP8_ERR_NULL;
  if (!aligned16(p)) return FP8_ERR_ALIGN;
  return FP8_OK;
}

#define FP8_TRY(expr)                    \
  do {                                   \
    const fp8_status _s = (expr);        \
    if (_s != FP8_OK) return _s;         \
  } while (0)

fp8_status check_recipe(const fp8_recipe* r) {
  if (r == nullptr) return FP8_ERR_NULL;
  if (r->kind < FP8_RECIPE_DELAYED || r->kind > FP8_RECIPE_BLOCKWISE) return FP8_ERR_UNSUPPORTED;
  if (r->format != FP8_FORMAT_E4M3 && r->format != FP8_FORMAT_HYBRID) return FP8_ERR_UNSUPPORTED;
  if (r->format == FP8_FORMAT_HYBRID && r->kind == FP8_RECIPE_MXFP8)
    return FP8_ERR_UNSUPPORTED;                                  // mxfp8 is E4M3 only
  if (r->margin < -64 || r->margin > 64) return FP8_ERR_UNSUPPORTED;
  if (r->amax_compute_algo != 0 && r->amax_compute_algo != 1)   // max, most_recent
    return FP8_ERR_UNSUPPORTED;
  if (r->kind == FP8_RECIPE_DELAYED && r->amax_history_len < 1) return FP8_ERR_SHAPE;
  if (r->power_2_scales != 0 && r->kind != FP8_RECIPE_BLOCKWISE) return FP8_ERR_UNSUPPORTED;
  return FP8_OK;
}

// Storage format of a tensor with this role: E5M2 (1) for gradients under the hybrid format,
// E4M3 (0) otherwise.
int fmt_of(const fp8_recipe* r, int role) {
  return (r->format == FP8_FORMAT_HYBRID && role == FP8_ROLE_GRAD) ? 1 : 0;
}

// The GEMM path of a recipe: blockwise with power-of-two scales stores its scales as E8M0
// bytes in the MXFP8 layout, so its GEMMs run on the block-scaled (MXFP8) tensor-core path.
int gemm_kind(const fp8_recipe* r) {
  return (r->kind == FP8_RECIPE_BLOCKWISE && r->power_2_scales != 0) ? int(FP8_RECIPE_MXFP8)
                                                                      : r->kind;
}

// Row/column multiple a recipe needs: 128 for the block recipes, 16 for per-tensor scales.
int64_t shape_quantum(int kind) {
  return (kind == FP8_RECIPE_MXFP8 || kind == FP8_RECIPE_BLOCKWISE) ? 128 : 16;
}

// Scale pointers a recipe needs for one copy.
fp8_status check_copy(int kind, const uint8_t* codes, const void* scale) {
  FP8_TRY(check_ptr(codes));
  if (kind == FP8_RECIPE_MXFP8 || kind == FP8_RECIPE_BLOCKWISE) FP8_TRY(check_ptr(scale));
  return FP8_OK;
}

fp8_status check_scalars(int kind, const fp8_tensor* t) {
  if (kind == FP8_RECIPE_TENSORWISE || kind == FP8_RECIPE_DELAYED) {
    if (t->amax == nullptr || t->scale == nullptr || t->scale_inv == nullptr) return FP8_ERR_NULL;
  }
  return FP8_OK;
}

}  // namespace

extern "C" {

const char* fp8_status_str(fp8_status s) {
  switch (s) {
    case FP8_OK: return "ok";
    case FP8_ERR_NULL: return "null pointer";
    case FP8_ERR_ALIGN: return "pointer not 16-byte aligned";
    case FP8_ERR_SHAPE: return "bad shape";
    case FP8_ERR_UNSUPPORTED: return "unsupported recipe option";
    case FP8_ERR_CUDA: return "CUDA launch failed";
    case FP8_ERR_TIMEOUT: return "device wait timed out";
    case FP8_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

const char* fp8_last_cuda_error(void) { return g_last_cuda_error; }

size_t fp8_workspace_bytes(const fp8_recipe* recipe, int64_t rows, int64_t cols) {
  if (recipe == nullptr) return 0;
  return quantize_workspace_bytes(recipe->kind, rows, cols);
}

namespace {
// The checks fp8_quantize makes on one tensor's arguments (the recipe already checked), apart
// from the workspace. Sets *col_bf16: the column copy is the bf16 transpose.
fp8_status check_quantize_args(const fp8_recipe* recipe, const void* x_bf16, int64_t rows,
                               int64_t cols, int32_t role, int32_t want_row, int32_t want_col,
                               const fp8_tensor* out, bool* col_bf16) {
  if (out == nullptr) return FP8_ERR_NULL;
  if (role < FP8_ROLE_ACTIVATION || role > FP8_ROLE_GRAD) return FP8_ERR_UNSUPPORTED;
  if (!want_row && !want_col) return FP8_ERR_SHAPE;
  const int kind = recipe->kind;
  const int64_t q = shape_quantum(kind);
  if (rows < 0 || cols < 0 || rows % q != 0 || cols % q != 0) return FP8_ERR_SHAPE;
  if (rows * cols >= (int64_t(1) << 31)) return FP8_ERR_SHAPE;   // 32-bit element offsets
  FP8_TRY(check_scalars(kind, out));
  *col_bf16 = recipe->fp8_wgrad == 0 && role != FP8_ROLE_WEIGHT;
  if (rows != 0 && cols != 0) {
    FP8_TRY(check_ptr(x_bf16));
    if (want_row) FP8_TRY(check_copy(kind, out->row, out->row_scale));
    if (want_col) {
      if (*col_bf16) FP8_TRY(check_ptr(out->col));
      else FP8_TRY(check_copy(kind, out->col, out->col_scale));
    }
  }
  return FP8_OK;
}

fp8_status quantize_impl(const fp8_recipe* recipe, const void* x_bf16, int64_t rows,
                         int64_t cols, int32_t role, int32_t want_row, int32_t want_col,
                         fp8_tensor* out, void* workspace, size_t ws_bytes, int32_t* dev_status,
                         cudaStream_t stream, uint32_t stall_tx) {
  FP8_TRY(check_recipe(recipe));
  bool col_bf16 = false;
  FP8_TRY(check_quantize_args(recipe, x_bf16, rows, cols, role, want_row, want_col, out,
                              &col_bf16));
  const int kind = recipe->kind;
  const bool empty = rows == 0 || cols == 0;
  if (!empty) {
    const size_t need = quantize_workspace_bytes(kind, rows, cols);
    if (need > 0 && (workspace == nullptr || ws_bytes < need)) return FP8_ERR_WORKSPACE;
    if (need > 0 && !aligned16(workspace)) return FP8_ERR_ALIGN;
  }
  out->rows = rows;
  out->cols = cols;
  out->role = role;
  out->kind = kind;
  out->col_bf16 = col_bf16 ? 1 : 0;
  return cuda_status(quantize_launch(kind, role, fmt_of(recipe, role),
                                     recipe->power_2_scales != 0, recipe->margin,
                                     reinterpret_cast<const uint16_t*>(x_bf16), rows, cols,
                                     want_row != 0, want_col != 0, col_bf16, out, workspace,
                                     dev_status, stream, stall_tx));
}
}  // namespace

fp8_status fp8_quantize(const fp8_recipe* recipe, const void* x_bf16, int64_t rows, int64_t cols,
                        int32_t role, int32_t want_row, int32_t want_col, fp8_tensor* out,
                        void* workspace, size_t ws_bytes, int32_t* dev_status,
                        cudaStream_t stream) {
  return quantize_impl(recipe, x_bf16, rows, cols, role, want_row, want_col, out, workspace,
                       ws_bytes, dev_status, stream, 0u);
}

fp8_status fp8_test_quantize_stalled(const fp8_recipe* recipe, const void* x_bf16, int64_t rows,
                                     int64_t cols, int32_t role, int32_t want_row,
                                     int32_t want_col, fp8_tensor* out, void* workspace,
                                     size_t ws_bytes, int32_t* dev_status, cudaStream_t stream) {
  if (dev_status == nullptr) return FP8_ERR_NULL;     // the outcome is only visible there
  return quantize_impl(recipe, x_bf16, rows, cols, role, want_row, want_col, out, workspace,
                       ws_bytes, dev_status, stream, 16u);
}

namespace {
fp8_status quantize_group_impl(const fp8_recipe* recipe, int32_t n,
                               const fp8_quantize_item* items, int32_t* dev_status,
                               cudaStream_t stream, uint32_t stall_tx) {
  FP8_TRY(check_recipe(recipe));
  if (recipe->kind != FP8_RECIPE_MXFP8 && recipe->kind != FP8_RECIPE_BLOCKWISE)
    return FP8_ERR_UNSUPPORTED;
  if (items == nullptr) return FP8_ERR_NULL;
  if (n < 1 || n > FP8_QUANTIZE_GROUP_MAX) return FP8_ERR_SHAPE;
  fp8lin::QuantGroupItem q[FP8_QUANTIZE_GROUP_MAX];
  for (int i = 0; i < n; ++i) {
    const fp8_quantize_item& it = items[i];
    bool col_bf16 = false;
    FP8_TRY(check_quantize_args(recipe, it.x_bf16, it.rows, it.cols, it.role, it.want_row,
                                it.want_col, it.out, &col_bf16));
    q[i] = {reinterpret_cast<const uint16_t*>(it.x_bf16), it.rows, it.cols, it.role,
            it.want_row != 0, it.want_col != 0, col_bf16, fmt_of(recipe, it.role) == 1, it.out};
  }
  for (int i = 0; i < n; ++i) {
    fp8_tensor* out = items[i].out;
    out->rows = items[i].rows;
    out->cols = items[i].cols;
    out->role = items[i].role;
    out->kind = recipe->kind;
    out->col_bf16 = q[i].col_bf16 ? 1 : 0;
  }
  return cuda_status(fp8lin::quantize_group_launch(recipe->kind, recipe->power_2_scales != 0,
                                                   recipe->margin, n, q, dev_status, stream,
                                                   stall_tx));
}
}  // namespace

fp8_status fp8_quantize_group(const fp8_recipe* recipe, int32_t n,
                              const fp8_quantize_item* items, int32_t* dev_status,
                              cudaStream_t stream) {
  return quantize_group_impl(recipe, n, items, dev_status, stream, 0u);
}

fp8_status fp8_test_quantize_group_stalled(const fp8_recipe* recipe, int32_t n,
                                           const fp8_quantize_item* items, int32_t* dev_status,
                                           cudaStream_t stream) {
  if (dev_status == nullptr) return FP8_ERR_NULL;     // the outcome is only visible there
  return quantize_group_impl(recipe, n, items, dev_status, stream, 16u);
}

fp8_status fp8_quantize_master(const fp8_recipe* recipe, const float* w_f32, int64_t rows,
                               int64_t cols, int32_t want_row, int32_t want_col, fp8_tensor* out,
                               void* workspace, size_t ws_bytes, int32_t* dev_status,
                               cudaStream_t stream) {
  (void)dev_status;                         // no device-side waits in this path
  FP8_TRY(check_recipe(recipe));
  if (out == nullptr) return FP8_ERR_NULL;
  if (recipe->power_2_scales != 0) return FP8_ERR_UNSUPPORTED;
  if (!want_row && !want_col) return FP8_ERR_SHAPE;
  const int kind = recipe->kind;
  const int64_t q = shape_quantum(kind);
  if (rows < 0 || cols < 0 || rows % q != 0 || cols % q != 0) return FP8_ERR_SHAPE;
  if (rows * cols >= (int64_t(1) << 31)) return FP8_ERR_SHAPE;
  FP8_TRY(check_scalars(kind, out));
  const bool empty = rows == 0 || cols == 0;
  if (!empty) {
    FP8_TRY(check_ptr(w_f32));
    if (want_row) FP8_TRY(check_copy(kind, out->row, out->row_scale));
    if (want_col) FP8_TRY(check_copy(kind, out->col, out->col_scale));
    const size_t need = quantize_workspace_bytes(kind, rows, cols);
    if (need > 0 && (workspace == nullptr || ws_bytes < need)) return FP8_ERR_WORKSPACE;
    if (need > 0 && !aligned16(workspace)) return FP8_ERR_ALIGN;
  }
  out->rows = rows;
  out->cols = cols;
  out->role = FP8_ROLE_WEIGHT;
  out->kind = kind;
  out->col_bf16 = 0;
  return cuda_status(quantize_master_launch(kind, recipe->margin, w_f32, rows, cols,
                                            want_row != 0, want_col != 0, out, workspace,
                                            stream));
}

fp8_status fp8_amax_update(const fp8_recipe* recipe, fp8_amax_history* hist, int32_t role,
                           const float* amax_new, float* scale, float* scale_inv,
                           cudaStream_t stream) {
  FP8_TRY(check_recipe(recipe));
  if (recipe->kind != FP8_RECIPE_DELAYED) return FP8_ERR_UNSUPPORTED;
  if (role < FP8_ROLE_ACTIVATION || role > FP8_ROLE_GRAD) return FP8_ERR_UNSUPPORTED;
  if (hist == nullptr || hist->history == nullptr || hist->head == nullptr || amax_new == nullptr ||
      scale == nullptr || scale_inv == nullptr)
    return FP8_ERR_NULL;
  if (hist->len < 1 || hist->len != recipe->amax_history_len) return FP8_ERR_SHAPE;
  const float fmax = fmt_of(recipe, role) == 1 ? 57344.0f : 448.0f;
  return cuda_status(amax_update_launch(hist->history, hist->head, hist->len, amax_new, scale,
                                        scale_inv, recipe->margin, fmax,
                                        recipe->amax_compute_algo, stream));
}

}  // extern "C"

namespace {

// One TN GEMM D[M][N] = A[M][Kr] . B[N][Kr]^T for the recipe, from two quantised copies.
struct Operand {
  const uint8_t* codes;
  const void* scale;        // per recipe (see fp8lin.h)
  const float* scale_inv;   // per-tensor recipes
  int role;
  int fmt;                  // 0 = E4M3, 1 = E5M2
  int mn = 0;               // 1: codes are the other copy, read MN-major (transposed)
};

// The copy a backward GEMM reads for the transposed operand: the column-wise copy (K-major)
// when it exists; otherwise, for per-tensor scales and 128x128 weight tiles (where both copies
// hold the same codes), the row-wise copy read MN-major, so the quantizer may skip the column
// copy for those tensors.
Operand transposed_operand(const fp8_recipe* recipe, const fp8_tensor* t) {
  const bool same_codes = recipe->kind == FP8_RECIPE_TENSORWISE ||
                          recipe->kind == FP8_RECIPE_DELAYED ||
                          (recipe->kind == FP8_RECIPE_BLOCKWISE && t->role == FP8_ROLE_WEIGHT &&
                           recipe->power_2_scales == 0);   // pow2: the MX path is K-major only
  if (t->col == nullptr && t->row != nullptr && same_codes)
    return Operand{t->row, t->row_scale, t->scale_inv, t->role, fmt_of(recipe, t->role), 1};
  return Operand{t->col, t->col_scale, t->scale_inv, t->role, fmt_of(recipe, t->role), 0};
}

fp8_status run_gemm(int kind, const Operand& a, const Operand& b, int64_t M, int64_t N,
                    int64_t Kr, void* D, int fp32_out, int32_t* status, cudaStream_t st,
                    uint32_t stall_tx = 0) {
  FP8_TRY(check_ptr(a.codes));
  FP8_TRY(check_ptr(b.codes));
  FP8_TRY(check_ptr(D));
  const int64_t q = shape_quantum(kind);
  if (M % q || N % q || Kr % q) return FP8_ERR_SHAPE;
  if (M > (int64_t(1) << 30) || N > (int64_t(1) << 30) || Kr > (int64_t(1) << 30))
    return FP8_ERR_SHAPE;
  if (M == 0 || N == 0) return FP8_OK;
  if (Kr == 0) {
    return cuda_status(cudaMemsetAsync(D, 0, size_t(M) * N * (fp32_out ? 4 : 2), st));
  }
  GemmLaunch g{};
  g.A = a.codes;
  g.B = b.codes;
  g.p.M = int(M);
  g.p.N = int(N);
  g.p.K = int(Kr);
  g.p.D = D;
  g.p.ldd = N;
  g.p.d_fp32 = fp32_out;
  g.p.status = status;
  g.p.a_fmt = a.fmt;
  g.p.b_fmt = b.fmt;
  g.p.a_mn = a.mn;
  g.p.b_mn = b.mn;
  g.p.stall_tx = stall_tx;
  switch (kind) {
    case FP8_RECIPE_TENSORWISE:
    case FP8_RECIPE_DELAYED:
      if (a.scale_inv == nullptr || b.scale_inv == nullptr) return FP8_ERR_NULL;
      g.mode = G_TENSOR;
      g.p.a_sinv = a.scale_inv;
      g.p.b_sinv = b.scale_inv;
      break;
    case FP8_RECIPE_MXFP8:
      FP8_TRY(check_ptr(a.scale));
      FP8_TRY(check_ptr(b.scale));
      g.mode = G_MX;
      g.p.sfa = reinterpret_cast<const uint8_t*>(a.scale);
      g.p.sfb = reinterpret_cast<const uint8_t*>(b.scale);
      break;
    case FP8_RECIPE_BLOCKWISE:
      FP8_TRY(check_ptr(a.scale));
      FP8_TRY(check_ptr(b.scale));
      if (a.role == FP8_ROLE_WEIGHT) return FP8_ERR_UNSUPPORTED;   // A is always 1x128
      g.mode = G_BLOCK;
      g.p.a_bs = reinterpret_cast<const float*>(a.scale);
      g.p.b_bs = reinterpret_cast<const float*>(b.scale);
      g.p.b_is_128 = b.role == FP8_ROLE_WEIGHT;
      break;
    default:
      return FP8_ERR_UNSUPPORTED;
  }
  return cuda_status(gemm_launch(g, st));
}

fp8_status run_bf16_gemm(const void* a, const void* b, int64_t M, int64_t N, int64_t Kr, void* D,
                         int fp32_out, int32_t* status, cudaStream_t st) {
  FP8_TRY(check_ptr(a));
  FP8_TRY(check_ptr(b));
  FP8_TRY(check_ptr(D));
  if (M % 16 || N % 16 || Kr % 16) return FP8_ERR_SHAPE;
  if (M > (int64_t(1) << 30) || N > (int64_t(1) << 30) || Kr > (int64_t(1) << 30))
    return FP8_ERR_SHAPE;
  if (M == 0 || N == 0) return FP8_OK;
  if (Kr == 0) return cuda_status(cudaMemsetAsync(D, 0, size_t(M) * N * (fp32_out ? 4 : 2), st));
  GemmLaunch g{};
  g.mode = G_BF16;
  g.A = a;
  g.B = b;
  g.p.M = int(M);
  g.p.N = int(N);
  g.p.K = int(Kr);
  g.p.D = D;
  g.p.ldd = N;
  g.p.d_fp32 = fp32_out;
  g.p.status = status;
  return cuda_status(gemm_launch(g, st));
}

// MXFP8 GEMM whose epilogue quantises the tile (fused MLP steps); D is never written.
fp8_status run_fused_mx(int epi, const Operand& a, const Operand& b, int64_t M, int64_t N,
                        int64_t Kr, uint8_t* h_row, uint8_t* h_scale, fp8_tensor* out,
                        int32_t* status, cudaStream_t st) {
  if (M % 128 || N % 128 || Kr % 128) return FP8_ERR_SHAPE;
  if (M > (int64_t(1) << 30) || N > (int64_t(1) << 30) || Kr > (int64_t(1) << 30) ||
      M * N >= (int64_t(1) << 31))
    return FP8_ERR_SHAPE;
  if (M == 0 || N == 0) return FP8_OK;
  if (Kr == 0) return FP8_ERR_SHAPE;            // no accumulator to quantise
  FP8_TRY(check_ptr(a.codes));
  FP8_TRY(check_ptr(b.codes));
  FP8_TRY(check_ptr(a.scale));
  FP8_TRY(check_ptr(b.scale));
  FP8_TRY(check_copy(FP8_RECIPE_MXFP8, h_row, h_scale));
  FP8_TRY(check_copy(FP8_RECIPE_MXFP8, out->row, out->row_scale));
  FP8_TRY(check_copy(FP8_RECIPE_MXFP8, out->col, out->col_scale));
  GemmLaunch g{};
  g.mode = G_MX;
  g.epi = epi;
  g.A = a.codes;
  g.B = b.codes;
  g.p.M = int(M);
  g.p.N = int(N);
  g.p.K = int(Kr);
  g.p.ldd = N;
  g.p.status = status;
  g.p.sfa = reinterpret_cast<const uint8_t*>(a.scale);
  g.p.sfb = reinterpret_cast<const uint8_t*>(b.scale);
  g.p.h_row = h_row;
  g.p.h_scale = h_scale;
  g.p.o_row = out->row;
  g.p.o_row_scale = reinterpret_cast<uint8_t*>(out->row_scale);
  g.p.o_col = out->col;
  g.p.o_col_scale = reinterpret_cast<uint8_t*>(out->col_scale);
  return cuda_status(gemm_launch(g, st));
}

fp8_status check_tensor(const fp8_recipe* r, const fp8_tensor* t) {
  if (t == nullptr) return FP8_ERR_NULL;
  if (t->kind != r->kind) return FP8_ERR_UNSUPPORTED;
  return FP8_OK;
}

}  // namespace

extern "C" {

fp8_status fp8_linear_fwd(const fp8_recipe* recipe, const fp8_tensor* x, const fp8_tensor* w,
                          void* y, int32_t y_fp32, int32_t* dev_status, cudaStream_t stream) {
  FP8_TRY(check_recipe(recipe));
  FP8_TRY(check_tensor(recipe, x));
  FP8_TRY(check_tensor(recipe, w));
  if (x->cols != w->cols) return FP8_ERR_SHAPE;
  const Operand a{x->row, x->row_scale, x->scale_inv, x->role,
                    fmt_of(recipe, x->role)};
  const Operand b{w->row, w->row_scale, w->scale_inv, w->role,
                    fmt_of(recipe, w->role)};
  return run_gemm(gemm_kind(recipe), a, b, x->rows, w->rows, x->cols, y, y_fp32, dev_status, stream);
}

fp8_status fp8_test_linear_fwd_stalled(const fp8_recipe* recipe, const fp8_tensor* x,
                                       const fp8_tensor* w, void* y, int32_t* dev_status,
                                       cudaStream_t stream) {
  FP8_TRY(check_recipe(recipe));
  FP8_TRY(check_tensor(recipe, x));
  FP8_TRY(check_tensor(recipe, w));
  if (x->cols != w->cols) return FP8_ERR_SHAPE;
  if (dev_status == nullptr) return FP8_ERR_NULL;     // the outcome is only visible there
  const Operand a{x->row, x->row_scale, x->scale_inv, x->role, fmt_of(recipe, x->role)};
  const Operand b{w->row, w->row_scale, w->scale_inv, w->role, fmt_of(recipe, w->role)};
  return run_gemm(gemm_kind(recipe), a, b, x->rows, w->rows, x->cols, y, 0, dev_status, stream,
                  16u);
}

fp8_status fp8_linear_bwd(const fp8_recipe* recipe, const fp8_tensor* dy,
                          const fp8_tensor* x_saved, const fp8_tensor* w, void* dx, void* dw,
                          int32_t out_fp32, int32_t* dev_status, cudaStream_t stream) {
  FP8_TRY(check_recipe(recipe));
  FP8_TRY(check_tensor(recipe, dy));
  const int64_t M = dy->rows, N = dy->cols;
  if (dx != nullptr) {
    FP8_TRY(check_tensor(recipe, w));
    if (w->rows != N) return FP8_ERR_SHAPE;
    const int64_t K = w->cols;
    // dgrad: dX[M][K] = dY[M][N] . (W^T)[K][N]^T
    const Operand a{dy->row, dy->row_scale, dy->scale_inv, dy->role,
                    fmt_of(recipe, dy->role)};
    const Operand b = transposed_operand(recipe, w);
    FP8_TRY(run_gemm(gemm_kind(recipe), a, b, M, K, N, dx, out_fp32, dev_status, stream));
  }
  if (dw != nullptr) {
    FP8_TRY(check_tensor(recipe, x_saved));
    if (x_saved->rows != M) return FP8_ERR_SHAPE;
    const int64_t K = x_saved->cols;
    const bool bf16 = recipe->fp8_wgrad == 0;
    if (dy->col_bf16 != (bf16 ? 1 : 0) || x_saved->col_bf16 != (bf16 ? 1 : 0))
      return FP8_ERR_UNSUPPORTED;              // copies quantised under another --fp8-wgrad
    if (bf16) {
      // wgrad in bf16: dW[N][K] = (dY^T)[N][M] . (X^T)[K][M]^T from the bf16 transposes
      return run_bf16_gemm(dy->col, x_saved->col, N, K, M, dw, out_fp32, dev_status, stream);
    }
    // wgrad: dW[N][K] = (dY^T)[N][M] . (X^T)[K][M]^T
    const Operand a = transposed_operand(recipe, dy);
    const Operand b = transposed_operand(recipe, x_saved);
    FP8_TRY(run_gemm(gemm_kind(recipe), a, b, N, K, M, dw, out_fp32, dev_status, stream));
  }
  return FP8_OK;
}

fp8_status fp8_linear_fwd_gelu(const fp8_recipe* recipe, const fp8_tensor* x,
                               const fp8_tensor* w, fp8_tensor* a_q, fp8_tensor* h_q,
                               int32_t* dev_status, cudaStream_t stream) {
  FP8_TRY(check_recipe(recipe));
  if (recipe->kind != FP8_RECIPE_MXFP8) return FP8_ERR_UNSUPPORTED;
  FP8_TRY(check_tensor(recipe, x));
  FP8_TRY(check_tensor(recipe, w));
  if (a_q == nullptr || h_q == nullptr) return FP8_ERR_NULL;
  if (x->cols != w->cols) return FP8_ERR_SHAPE;
  const int64_t M = x->rows, N = w->rows;
  const Operand a{x->row, x->row_scale, x->scale_inv, x->role,
                    fmt_of(recipe, x->role)};
  const Operand b{w->row, w->row_scale, w->scale_inv, w->role,
                    fmt_of(recipe, w->role)};
  FP8_TRY(run_fused_mx(EPI_GELU, a, b, M, N, x->cols, h_q->row,
                       reinterpret_cast<uint8_t*>(h_q->row_scale), a_q, dev_status, stream));
  for (fp8_tensor* t : {a_q, h_q}) {
    t->rows = M;
    t->cols = N;
    t->kind = FP8_RECIPE_MXFP8;
    t->role = FP8_ROLE_ACTIVATION;
    t->col_bf16 = 0;
  }
  return FP8_OK;
}

fp8_status fp8_linear_dgrad_dgelu(const fp8_recipe* recipe, const fp8_tensor* dy,
                                  const fp8_tensor* w, const fp8_tensor* h_q, fp8_tensor* dh_q,
                                  int32_t* dev_status, cudaStream_t stream) {
  FP8_TRY(check_recipe(recipe));
  if (recipe->kind != FP8_RECIPE_MXFP8) return FP8_ERR_UNSUPPORTED;
  FP8_TRY(check_tensor(recipe, dy));
  FP8_TRY(check_tensor(recipe, w));
  FP8_TRY(check_tensor(recipe, h_q));
  if (dh_q == nullptr) return FP8_ERR_NULL;
  const int64_t M = dy->rows, N = w->cols;
  if (w->rows != dy->cols || h_q->rows != M || h_q->cols != N) return FP8_ERR_SHAPE;
  // dgrad: dA[M][N] = dY[M][H] . (W^T)[N][H]^T
  const Operand a{dy->row, dy->row_scale, dy->scale_inv, dy->role,
                    fmt_of(recipe, dy->role)};
  const Operand b{w->col, w->col_scale, w->scale_inv, w->role,
                    fmt_of(recipe, w->role)};
  FP8_TRY(run_fused_mx(EPI_DGELU, a, b, M, N, dy->cols, h_q->row,
                       reinterpret_cast<uint8_t*>(h_q->row_scale), dh_q, dev_status, stream));
  dh_q->rows = M;
  dh_q->cols = N;
  dh_q->kind = FP8_RECIPE_MXFP8;
  dh_q->role = FP8_ROLE_GRAD;
  dh_q->col_bf16 = 0;
  return FP8_OK;
}

fp8_status fp8_gelu_quantize(const fp8_recipe* recipe, const void* h_bf16, int64_t rows,
                             int64_t cols, void* a_bf16, fp8_tensor* a_q, fp8_tensor* h_q,
                             int32_t* dev_status, cudaStream_t stream) {
  FP8_TRY(check_recipe(recipe));
  if (recipe->kind != FP8_RECIPE_MXFP8) return FP8_ERR_UNSUPPORTED;
  if (a_q == nullptr || h_q == nullptr) return FP8_ERR_NULL;
  if (rows < 0 || cols < 0 || rows % 128 || cols % 128) return FP8_ERR_SHAPE;
  if (rows * cols >= (int64_t(1) << 31)) return FP8_ERR_SHAPE;
  if (rows > 0 && cols > 0) {
    FP8_TRY(check_ptr(h_bf16));
    FP8_TRY(check_copy(FP8_RECIPE_MXFP8, a_q->row, a_q->row_scale));
    FP8_TRY(check_copy(FP8_RECIPE_MXFP8, a_q->col, a_q->col_scale));
    FP8_TRY(check_copy(FP8_RECIPE_MXFP8, h_q->row, h_q->row_scale));
    if (a_bf16 != nullptr && !aligned16(a_bf16)) return FP8_ERR_ALIGN;
  }
  for (fp8_tensor* t : {a_q, h_q}) {
    t->rows = rows;
    t->cols = cols;
    t->kind = FP8_RECIPE_MXFP8;
    t->role = FP8_ROLE_ACTIVATION;
  }
  return cuda_status(gelu_quantize_launch(reinterpret_cast<const uint16_t*>(h_bf16), rows, cols,
                                          reinterpret_cast<uint16_t*>(a_bf16), a_q, h_q, dev_status,
                                          stream));
}

fp8_status fp8_dgelu_quantize(const fp8_recipe* recipe, const void* da_bf16,
                              const fp8_tensor* h_q, void* dh_bf16, fp8_tensor* dh_q,
                              int32_t* dev_status, cudaStream_t stream) {
  FP8_TRY(check_recipe(recipe));
  if (recipe->kind != FP8_RECIPE_MXFP8) return FP8_ERR_UNSUPPORTED;
  if (h_q == nullptr || dh_q == nullptr) return FP8_ERR_NULL;
  if (h_q->kind != FP8_RECIPE_MXFP8) return FP8_ERR_UNSUPPORTED;
  const int64_t rows = h_q->rows, cols = h_q->cols;
  if (rows < 0 || cols < 0 || rows % 128 || cols % 128) return FP8_ERR_SHAPE;
  if (rows * cols >= (int64_t(1) << 31)) return FP8_ERR_SHAPE;
  if (rows > 0 && cols > 0) {
    FP8_TRY(check_ptr(da_bf16));
    FP8_TRY(check_copy(FP8_RECIPE_MXFP8, h_q->row, h_q->row_scale));
    FP8_TRY(check_copy(FP8_RECIPE_MXFP8, dh_q->row, dh_q->row_scale));
    FP8_TRY(check_copy(FP8_RECIPE_MXFP8, dh_q->col, dh_q->col_scale));
    if (dh_bf16 != nullptr && !aligned16(dh_bf16)) return FP8_ERR_ALIGN;
  }
  dh_q->rows = rows;
  dh_q->cols = cols;
  dh_q->kind = FP8_RECIPE_MXFP8;
  dh_q->role = FP8_ROLE_GRAD;
  return cuda_status(dgelu_quantize_launch(reinterpret_cast<const uint16_t*>(da_bf16), h_q, rows,
                                           cols, reinterpret_cast<uint16_t*>(dh_bf16), dh_q,
                                           dev_status, stream));
}

}  // extern "C"
