/*
 * fp8lin.h — C ABI of the GB300 (sm_103a) FP8 linear-layer library.
 *
 * The operations follow the recipes of the Megatron Core developer guide page
 * "Low-Precision Training Guide": section "Hardware and Recipe Compatibility" (the recipe
 * names delayed / tensorwise / mxfp8 / blockwise and the --fp8-format values), section
 * "Recipe Reference" (what each recipe scales by), section "Numerical Stability Knobs"
 * (--fp8-margin, --fp8-amax-history-len, --fp8-amax-compute-algo, --fp8-wgrad), and the
 * TransformerEngine issue "How to reduce cuda memory usage of fp8?" (the backward pass runs
 * from cached FP8 copies of the layer input instead of a bf16 copy). The MegaDLMs summary
 * "Benefits of Using FP8 Precision with MegaDLMs and Required Hardware" (section "Python API
 * Configuration") is the source of the MLP entry points that keep the GeLU input in FP8.
 *
 * Numerics (readings where the pages are silent):
 *   E4M3 is OCP E4M3FN (max 448, min subnormal 2^-9, no Inf). A code is
 *   encode(fp32(x * s)): round to nearest even, +-Inf and finite overflow saturate to
 *   +-448, NaN -> 0x7F with the input's sign bit.
 *   Per-tensor / per-block scale: s = fp32(448 / amax) * 2^-margin (IEEE division), s = 1
 *   when amax is 0, Inf or NaN, an infinite s becomes FLT_MAX; s_inv = fp32(1 / s).
 *   MXFP8 E8M0 exponent of a 1x32 block: the smallest e with amax <= 448 * 2^e, clamped to
 *   [-127, 127], -127 when amax < 2^-126; byte e + 127; codes encode(x * 2^-e). A block
 *   holding Inf or NaN gets byte 0xFF and codes encode(x).
 *   GEMMs accumulate in fp32 and round once to bf16 (round to nearest even).
 *
 * Layouts (all tensors row-major, all pointers device pointers unless stated):
 *   X[M,K] activations, W[N,K] weights (the layer computes Y = X W^T), dY[M,N] gradients.
 *   A quantised tensor of source shape [R,C] has a row-wise copy row[R][C] (blocks along C)
 *   and a column-wise copy col[C][R] = the quantised transpose (blocks along R).
 *   Scale storage per recipe:
 *     DELAYED, TENSORWISE: fp32 scalars amax, scale, scale_inv (one for the tensor).
 *     MXFP8: uint8 E8M0, R*C/32 bytes per copy, in the tiled order that the tensor core's
 *       block-scale path reads: the byte of row r, 32-block kb of a copy with C columns is
 *         ((r/128) * (C/128) + kb/4) * 512 + (r%32) * 16 + ((r%128)/32) * 4 + kb%4.
 *     BLOCKWISE, role ACTIVATION or GRAD (1x128 blocks): fp32 s_inv, R*C/128 floats per
 *       copy, block-major: s_inv of row r, 128-block kb at kb * R + r.
 *     BLOCKWISE, role WEIGHT (128x128 blocks): fp32 s_inv, row copy [R/128][C/128],
 *       column copy [C/128][R/128] (the transposed grid). col = byte transpose of row.
 *
 * Ownership and ordering: the caller owns every buffer. No entry point allocates or frees
 * device memory, synchronises the device or the stream, or keeps state between calls (the
 * one exception is fp8_quantize_static_scratch, whose scratch array in the library image
 * keeps the last call's amax partials: see its "Sharing" note); all work is enqueued on the
 * caller's stream in stream order. Every entry point is safe to call
 * from several host threads on different streams. The kernels are launched with programmatic
 * dependent launch: a kernel may start its setup while the preceding kernel in the stream
 * finishes. It waits for that kernel's completion, and for the visibility of its writes,
 * before its first global memory access, so stream order holds for every buffer. Setting the
 * environment variable FP8LIN_PDL=0 launches without the attribute.
 *
 * Errors: argument errors are found on the host before anything is enqueued and returned as
 * a status (nothing is launched then). Conditions seen on the device (a pipeline wait that
 * ran out of its time budget) are written to *dev_status (int32, caller-zeroed; may be NULL)
 * and the kernel returns early; the caller reads it after its own synchronisation.
 */
#ifndef FP8LIN_H
#define FP8LIN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FP8_OK = 0,
  FP8_ERR_NULL = 1,         /* a required pointer is NULL */
  FP8_ERR_ALIGN = 2,        /* a pointer is not 16-byte aligned */
  FP8_ERR_SHAPE = 3,        /* sizes negative, not multiples of the required block, or
                               inconsistent between operands */
  FP8_ERR_UNSUPPORTED = 4,  /* a recipe option this library does not implement */
  FP8_ERR_CUDA = 5,         /* a CUDA launch or query failed */
  FP8_ERR_TIMEOUT = 6,      /* device-side only: a pipeline wait exceeded its budget */
  FP8_ERR_WORKSPACE = 7     /* workspace missing or smaller than fp8_workspace_bytes() */
} fp8_status;

/* --fp8-recipe values (section "Hardware and Recipe Compatibility"). */
typedef enum {
  FP8_RECIPE_DELAYED = 0,
  FP8_RECIPE_TENSORWISE = 1,
  FP8_RECIPE_MXFP8 = 2,
  FP8_RECIPE_BLOCKWISE = 3
} fp8_recipe_kind;

/* --fp8-format values ("Hardware and Recipe Compatibility": e4m3 for every recipe, hybrid for
 * delayed, tensorwise and blockwise). The pages do not define hybrid; this library reads it as
 * E4M3 for activations and weights and E5M2 for gradients (role FP8_ROLE_GRAD): OCP E5M2, bias
 * 15, 2 mantissa bits, largest finite value 57344, encoded like E4M3 (round to nearest even,
 * finite overflow and infinities saturate to +-57344, NaN -> 0x7F with its sign) with 57344 in
 * place of 448 in the scale rule. MXFP8 takes E4M3 only (hybrid -> FP8_ERR_UNSUPPORTED). */
typedef enum { FP8_FORMAT_E4M3 = 0, FP8_FORMAT_HYBRID = 1 } fp8_format;

/* Which block shape the blockwise recipe uses for a tensor: 1x128 for activations and
 * gradients, 128x128 for weights (recipe entry "blockwise"). Ignored by other recipes. */
typedef enum { FP8_ROLE_ACTIVATION = 0, FP8_ROLE_WEIGHT = 1, FP8_ROLE_GRAD = 2 } fp8_role;

/* The recipe statement, one field per flag. */
typedef struct {
  int32_t kind;               /* fp8_recipe_kind (--fp8-recipe) */
  int32_t format;             /* fp8_format (--fp8-format) */
  int32_t margin;             /* --fp8-margin, in [-64, 64]; s is multiplied by 2^-margin */
  int32_t amax_history_len;   /* --fp8-amax-history-len (DELAYED), >= 1 */
  int32_t amax_compute_algo;  /* --fp8-amax-compute-algo: 0 = max (the page's minimum
                                 config), 1 = most_recent (the newest amax alone) */
  int32_t fp8_wgrad;          /* --fp8-wgrad: 1 = wgrad GEMM in FP8, 0 = in bf16 */
  int32_t power_2_scales;     /* BLOCKWISE only: 1 = each block scale rounded down to a power
                                 of two, stored as E8M0 bytes in the MXFP8 scale layout (each
                                 1x128 or 128x128 block's byte repeated for its 1x32 blocks),
                                 and the GEMMs run on the MXFP8 block-scaled tensor-core path;
                                 0 = plain fp32 s_inv. Other recipes: must be 0 */
} fp8_recipe;

/* A quantised tensor: codes and scales of both copies, all device memory owned by the
 * caller. row / col may be NULL when that copy is not wanted. */
typedef struct {
  uint8_t *row;          /* [rows][cols] FP8 codes (E5M2 for gradients under hybrid) */
  uint8_t *col;          /* [cols][rows] FP8 codes */
  void *row_scale;       /* MXFP8: uint8 E8M0; BLOCKWISE: float s_inv (E8M0 in the MXFP8
                            layout with power_2_scales); else unused */
  void *col_scale;       /* same for the column-wise copy */
  float *amax;           /* DELAYED/TENSORWISE: amax of this tensor (written) */
  float *scale;          /* TENSORWISE: written. DELAYED: read (the scale from history) */
  float *scale_inv;      /* TENSORWISE: written. DELAYED: read */
  int64_t rows, cols;    /* source shape [R, C] */
  int32_t kind;          /* recipe the codes were made with (set by fp8_quantize) */
  int32_t role;          /* fp8_role */
  int32_t col_bf16;      /* 1: `col` holds the bf16 transpose (set by fp8_quantize) */
} fp8_tensor;

/* Delayed-scaling state: a rolling window of the last `len` amax values. */
typedef struct {
  float *history;        /* [len] fp32, start as zeros */
  int32_t *head;         /* next slot to write, starts at 0 */
  int32_t len;           /* --fp8-amax-history-len */
} fp8_amax_history;

/* Bytes of scratch memory fp8_quantize needs for this recipe and shape (0 if none). The
 * tensorwise and delayed recipes reduce the amax through per-tile partial maxima. */
size_t fp8_workspace_bytes(const fp8_recipe *recipe, int64_t rows, int64_t cols);

/*
 * fp8_quantize — bf16 tensor -> FP8 codes plus scales, row-wise and/or column-wise copy
 * (E4M3; E5M2 for role FP8_ROLE_GRAD under the hybrid format).
 *
 * Recipe entries "tensorwise" (scale from this tensor's own amax), "delayed" (scale read from
 * out->scale / out->scale_inv, which fp8_amax_update derived from earlier steps; this call
 * writes this tensor's amax to out->amax for the next update), "mxfp8" (E8M0 per 1x32 block)
 * and "blockwise" (1x128 or 128x128 by role).
 *   x_bf16     [rows][cols] bf16, 16-byte aligned, read only.
 *   rows, cols >= 0. MXFP8 and BLOCKWISE need both to be multiples of 128; TENSORWISE and
 *              DELAYED need multiples of 16. An empty tensor writes amax 0, scale 1.
 *   want_row / want_col: which copies to write (at least one). With recipe->fp8_wgrad == 0
 *              (--fp8-wgrad off) and a role other than WEIGHT, the column-wise copy is the
 *              transposed tensor in bf16 ([cols][rows], 2 bytes per element, no scales): it
 *              is only read by the wgrad GEMM, which then runs in bf16.
 *   out        codes/scales destinations (see the layouts above); out->rows/cols/role/kind
 *              are set by this call.
 *   workspace  device scratch of at least fp8_workspace_bytes() (may be NULL when that is 0).
 * Returns FP8_OK or a host-detected error (nothing launched on error).
 * Source: the Megatron Core "Low-Precision Training Guide", section "Recipe Reference"
 * (entries delayed, tensorwise, mxfp8 and blockwise: what each recipe scales by) and section
 * "Hardware and Recipe Compatibility" (E4M3 / hybrid formats); the two copies are the cached
 * FP8 data and FP8 transpose of the TransformerEngine issue "How to reduce cuda memory usage
 * of fp8?".
 */
fp8_status fp8_quantize(const fp8_recipe *recipe, const void *x_bf16, int64_t rows,
                        int64_t cols, int32_t role, int32_t want_row, int32_t want_col,
                        fp8_tensor *out, void *workspace, size_t ws_bytes,
                        int32_t *dev_status, cudaStream_t stream);

/*
 * fp8_quantize_master — fp32 master weights -> E4M3 codes plus scales (role WEIGHT), with no
 * bf16 rounding in between (the weight cast of an optimizer that keeps fp32 weights). The
 * recipes are those of fp8_quantize for a weight: tensorwise / delayed per-tensor scale,
 * MXFP8 1x32 blocks (row copy along cols, column copy along rows), blockwise 128x128 tiles;
 * amaxes are taken over the fp32 values and a code is encode(fp32(x * s)). The column copy is
 * always FP8. Arguments, layouts, workspace (fp8_workspace_bytes of the same shape) and
 * errors as for fp8_quantize; w_f32 is [rows][cols] fp32, 16-byte aligned.
 * power_2_scales is not supported here (FP8_ERR_UNSUPPORTED).
 * Source: the TransformerEngine issue "How to reduce cuda memory usage of fp8?" (with
 * --fp8-param-gather the distributed optimizer casts the fp32 master weight straight into the
 * FP8 weight) and the Megatron Core "Low-Precision Training Guide", section "Recipe
 * Reference" (the weight's scaling under each recipe).
 */
fp8_status fp8_quantize_master(const fp8_recipe *recipe, const float *w_f32, int64_t rows,
                               int64_t cols, int32_t want_row, int32_t want_col,
                               fp8_tensor *out, void *workspace, size_t ws_bytes,
                               int32_t *dev_status, cudaStream_t stream);

/*
 * fp8_quantize_group — fp8_quantize of up to FP8_QUANTIZE_GROUP_MAX bf16 tensors under one
 * block-scaled recipe in one launch. One persistent grid walks the tiles of all the tensors,
 * so a layer's activation and weights are quantised at the rate of one large tensor instead
 * of each paying a launch's ramp-up and tail. Source: the Megatron Core "Low-Precision
 * Training Guide", section "Recipe Reference", entries mxfp8 (an E8M0 scale per 1x32 block)
 * and blockwise (1x128 activation / gradient blocks, 128x128 weight blocks); the codes and
 * scales are exactly those fp8_quantize writes for each tensor on its own, the hybrid format
 * and power-of-two block scales included.
 *   recipe     kind FP8_RECIPE_MXFP8 or FP8_RECIPE_BLOCKWISE; the per-tensor recipes
 *              (tensorwise, delayed) return FP8_ERR_UNSUPPORTED.
 *   n          number of items, 1 .. FP8_QUANTIZE_GROUP_MAX (else FP8_ERR_SHAPE).
 *   items      n descriptions in host memory, read during the call only. Each field means
 *              what the same-named argument of fp8_quantize means (x_bf16, rows, cols, role,
 *              want_row, want_col, out), with the same shape, alignment and layout rules and
 *              the same --fp8-wgrad handling of the column copy. No output may overlap
 *              another item's output or any input.
 * Every item is checked before anything is launched: on the first failing item its status is
 * returned and nothing runs. out->rows/cols/role/kind/col_bf16 are set as by fp8_quantize.
 * Needs no workspace.
 */
#define FP8_QUANTIZE_GROUP_MAX 4
typedef struct fp8_quantize_item {
  const void *x_bf16;
  int64_t rows;
  int64_t cols;
  int32_t role;
  int32_t want_row;
  int32_t want_col;
  fp8_tensor *out;
} fp8_quantize_item;

fp8_status fp8_quantize_group(const fp8_recipe *recipe, int32_t n,
                              const fp8_quantize_item *items, int32_t *dev_status,
                              cudaStream_t stream);

/*
 * fp8_amax_update — delayed scaling: push *amax_new into the history (the oldest of `len`
 * entries drops out) and write scale = f(max(history)), scale_inv = 1/scale with f the
 * per-tensor rule above (--fp8-amax-history-len, --fp8-margin), or with
 * --fp8-amax-compute-algo most_recent scale = f(*amax_new) (the history is still recorded).
 * role: fp8_role of the tensor this history belongs to (under the hybrid format a gradient's
 * scale uses the E5M2 maximum 57344). One CTA; reads and writes device memory only.
 * Source: the Megatron Core "Low-Precision Training Guide", section "Recipe Reference" entry
 * delayed (the scale comes from a rolling amax history) and section "Numerical Stability
 * Knobs" (--fp8-amax-history-len, --fp8-amax-compute-algo max / most_recent, --fp8-margin).
 */
fp8_status fp8_amax_update(const fp8_recipe *recipe, fp8_amax_history *hist, int32_t role,
                           const float *amax_new, float *scale, float *scale_inv,
                           cudaStream_t stream);

/*
 * fp8_linear_fwd — fprop Y[M,N] = deq(X)[M,K] . deq(W)[N,K]^T (fp32 accumulation).
 * Source: the Megatron Core "Low-Precision Training Guide", section "When to Use Low
 * Precision" (the linear layers' GEMMs run on FP8 tensor cores) and section "Recipe
 * Reference" (what each recipe scales by: one scale per tensor, one E8M0 scale per 1x32
 * block, 1x128 / 128x128 blocks).
 * Uses x->row and w->row. x and w must come from the same recipe. Tensor scales are applied
 * after accumulation, MXFP8 block scales by the tensor core during accumulation, blockwise
 * scales per 128-wide K chunk. y is bf16 [M][N] (y_fp32 = 0) or fp32 [M][N] (y_fp32 = 1,
 * for accumulation checks). M, N multiples of 16 (128 for MXFP8/BLOCKWISE), K multiple of
 * 128 (16 for DELAYED/TENSORWISE).
 */
fp8_status fp8_linear_fwd(const fp8_recipe *recipe, const fp8_tensor *x, const fp8_tensor *w,
                          void *y, int32_t y_fp32, int32_t *dev_status, cudaStream_t stream);

/*
 * fp8_linear_bwd — dgrad dX[M,K] = deq(dY)[M,N] . deq(W^T)[K,N]^T from dy->row and w->col,
 * and wgrad dW[N,K] = deq(dY^T)[N,M] . deq(X^T)[K,M]^T from dy->col and x_saved->col (the
 * copies cached in the forward pass). Where both copies hold the same codes — per-tensor
 * scales (DELAYED, TENSORWISE) and 128x128 weight tiles (BLOCKWISE, role WEIGHT) — a tensor
 * whose col is NULL is read from its row copy instead, as an MN-major (transposed) tensor-core
 * operand, so those tensors can be quantised with want_col = 0. With recipe->fp8_wgrad == 0
 * (--fp8-wgrad off) those two column copies are bf16 transposes (see fp8_quantize) and the
 * wgrad GEMM runs in bf16 with fp32 accumulation. dx or dw may be NULL to skip that GEMM. Outputs are bf16 (out_fp32 = 0)
 * or fp32 (out_fp32 = 1).
 * Source: the MegaDLMs summary "Benefits of Using FP8 Precision with MegaDLMs and Required
 * Hardware", section "Training Speed Improvements" (the backward pass's GEMMs in FP8), the
 * TransformerEngine issue "How to reduce cuda memory usage of fp8?" (the backward pass reads
 * the FP8 copies cached in the forward pass: the transpose on Hopper, the data itself on
 * Blackwell), and the "Low-Precision Training Guide" section "Numerical Stability Knobs"
 * (--fp8-wgrad: wgrad in FP8 or in bf16).
 */
fp8_status fp8_linear_bwd(const fp8_recipe *recipe, const fp8_tensor *dy,
                          const fp8_tensor *x_saved, const fp8_tensor *w, void *dx, void *dw,
                          int32_t out_fp32, int32_t *dev_status, cudaStream_t stream);

/*
 * fp8_gelu_quantize — MLP activation with its input kept in FP8 for the backward pass
 * (activation_func_fp8_input_store): a = bf16(gelu(h)) with gelu(h) = h * Phi(h) in fp32,
 * quantised (row and column copies) into a_q, and h itself quantised (row copy) into h_q.
 * a_bf16 may be NULL (only needed for bf16 wgrad or inspection). MXFP8 recipe only.
 * Source: the MegaDLMs summary "Benefits of Using FP8 Precision with MegaDLMs and Required
 * Hardware", section "Python API Configuration" (activation_func_fp8_input_store: the
 * activation's input is stored in FP8 for the backward pass) and section "Memory and Storage
 * Optimization"; the quantisation is the "Low-Precision Training Guide" Recipe Reference
 * entry mxfp8.
 */
fp8_status fp8_gelu_quantize(const fp8_recipe *recipe, const void *h_bf16, int64_t rows,
                             int64_t cols, void *a_bf16, fp8_tensor *a_q, fp8_tensor *h_q,
                             int32_t *dev_status, cudaStream_t stream);

/*
 * fp8_dgelu_quantize — dh = bf16(da * gelu'(deq(h_q))) in fp32, gelu'(h) = Phi(h) + h phi(h),
 * reading h back from its FP8 row copy, then quantised (row and column copies) into dh_q.
 * dh_bf16 may be NULL. MXFP8 recipe only.
 * Source: as fp8_gelu_quantize (the backward of the activation whose input was stored in
 * FP8).
 */
fp8_status fp8_dgelu_quantize(const fp8_recipe *recipe, const void *da_bf16,
                              const fp8_tensor *h_q, void *dh_bf16, fp8_tensor *dh_q,
                              int32_t *dev_status, cudaStream_t stream);

/*
 * fp8_linear_fwd_gelu — fc1 of the MLP block with the GeLU step fused into the GEMM
 * epilogue (MXFP8 recipe only): h = bf16(deq(X) . deq(W)^T) exactly as fp8_linear_fwd would
 * store it, but instead of writing h the epilogue writes h's MXFP8 row copy into h_q (the FP8
 * input store of the activation) and a = bf16(gelu(h)) as MXFP8 row and column copies into
 * a_q. Byte-identical to fp8_linear_fwd followed by fp8_gelu_quantize, without the bf16 round
 * trip of h through memory. x, w as for fp8_linear_fwd (row copies); a_q needs row, col and
 * both scale arrays, h_q needs row and row_scale, all 16-byte aligned (32-byte aligned code
 * arrays get 256-bit stores). M = x->rows and N = w->rows multiples of 128. On return a_q and
 * h_q describe [M][N] MXFP8 activations.
 * Source: as fp8_linear_fwd and fp8_gelu_quantize (the quantisation fused into the producing
 * GEMM is this library's design, not a step of the pages).
 */
fp8_status fp8_linear_fwd_gelu(const fp8_recipe *recipe, const fp8_tensor *x,
                               const fp8_tensor *w, fp8_tensor *a_q, fp8_tensor *h_q,
                               int32_t *dev_status, cudaStream_t stream);

/*
 * fp8_linear_dgrad_dgelu — dgrad of fc2 with the GeLU backward fused into the GEMM epilogue
 * (MXFP8 only): da = bf16(deq(dY) . deq(W^T)^T) from dy->row and w->col as fp8_linear_bwd
 * would store it, then dh = bf16(da * gelu'(deq(h_q))) with h read back from its FP8 row copy
 * (written by fp8_linear_fwd_gelu or fp8_gelu_quantize), quantised as MXFP8 row and column
 * copies into dh_q. Byte-identical to fp8_linear_bwd (dx only) followed by fp8_dgelu_quantize.
 * h_q must be [dy->rows][w->cols]; dh_q needs row, col and both scale arrays.
 * Source: as fp8_linear_bwd and fp8_dgelu_quantize.
 */
fp8_status fp8_linear_dgrad_dgelu(const fp8_recipe *recipe, const fp8_tensor *dy,
                                  const fp8_tensor *w, const fp8_tensor *h_q, fp8_tensor *dh_q,
                                  int32_t *dev_status, cudaStream_t stream);

/*
 * fp8_quantize_static_scratch — fp8_quantize for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a convenience of this library. Some callers cannot
 * hand the library a workspace (code inside a host framework whose allocator owns the whole
 * device pool, or loops that must not pay for cudaMalloc's implicit synchronisation). This
 * entry point takes the same arguments as fp8_quantize minus the workspace, and reduces the
 * tensorwise / delayed amax partials in a fixed 256 KiB array inside the library's device
 * image (held by every GPU that loads the library until the process exits). It allocates
 * nothing.
 *   Limit: tensors needing more than 65536 partials (delayed: more than 65536 128x128 tiles)
 *   return FP8_ERR_WORKSPACE; MXFP8 and blockwise need no scratch.
 *   Set-up: the first call in each CUDA context looks up the array's device address
 *   (cudaGetSymbolAddress) with that context's device current; make that first call before
 *   any stream capture. A new context on a device (after cudaDeviceReset, or a context the
 *   caller made current) gets its own lookup on its first call.
 *   Sharing: every call on a device uses the same array, which keeps the last call's
 *   contents (nothing in it needs to start at zero); calls whose work overlaps on the GPU
 *   (different streams, or several host threads) race on it and must be serialised by the
 *   caller.
 */
fp8_status fp8_quantize_static_scratch(const fp8_recipe *recipe, const void *x_bf16,
                                       int64_t rows, int64_t cols, int32_t role,
                                       int32_t want_row, int32_t want_col, fp8_tensor *out,
                                       int32_t *dev_status, cudaStream_t stream);

/* Human-readable name of a status. */
const char *fp8_status_str(fp8_status status);

/* Text of the CUDA error behind the calling thread's most recent FP8_ERR_CUDA ("" if none).
 * The string is owned by the library and stays valid until the thread's next failing call. */
const char *fp8_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8LIN_H */
