/*
 * fp8lin_test.h — test hooks of the FP8 linear-layer library (not for production use).
 *
 * Failure detection. Every wait inside the library's kernels (the GEMM pipeline's mbarrier
 * waits between its TMA, MMA, scale-factor and epilogue roles; the quantize kernels' TMA
 * waits) has a clock budget of about two seconds. When a wait runs out, the kernel:
 *   - records FP8_ERR_TIMEOUT in the caller's device status word;
 *   - tells its other roles to stop;
 *   - lets the copies it has in flight land;
 *   - frees its tensor memory and returns.
 * The CUDA context stays usable. The hooks below make such a wait run out on purpose,
 * without faulting, trapping or hanging the GPU, so tests can check that path. There is one
 * hook for the GEMM pipeline, one for the quantize kernels and one for the grouped quantize.
 */
#ifndef FP8LIN_TEST_H
#define FP8LIN_TEST_H

#include "fp8lin.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * fp8_linear_fwd with a stall planted in the GEMM pipeline. The first stage of the first
 * CTA (pair) expects 16 more bytes than its TMA loads deliver, so that stage never becomes
 * ready.
 *
 * Arguments are as for fp8_linear_fwd, with a bf16 y; dev_status is required.
 *
 * On the device, the MMA issuer's wait runs out after its budget. *dev_status then becomes
 * FP8_ERR_TIMEOUT, unless it already held a nonzero status. Outputs of the stalled CTA's
 * tiles are left unwritten; other CTAs finish their tiles.
 *
 * Host-side errors are those of fp8_linear_fwd, plus FP8_ERR_NULL when dev_status is NULL.
 * Takes about two seconds of GPU time.
 */
fp8_status fp8_test_linear_fwd_stalled(const fp8_recipe *recipe, const fp8_tensor *x,
                                       const fp8_tensor *w, void *y, int32_t *dev_status,
                                       cudaStream_t stream);

/*
 * fp8_quantize with a stall planted in the quantize kernel's TMA pipeline. CTA 0's first
 * tile expects 16 more bytes than its TMA loads deliver.
 *
 * Arguments are as for fp8_quantize; dev_status is required.
 *
 * On the device, CTA 0's wait runs out after its budget. *dev_status then becomes
 * FP8_ERR_TIMEOUT, unless it already held a nonzero status. CTA 0's tiles are left
 * unwritten, and under delayed scaling the amax reported for the call is then not
 * meaningful. The other CTAs finish their tiles.
 *
 * Host-side errors are those of fp8_quantize, plus FP8_ERR_NULL when dev_status is NULL.
 * Takes about two seconds of GPU time.
 */
fp8_status fp8_test_quantize_stalled(const fp8_recipe *recipe, const void *x_bf16, int64_t rows,
                                     int64_t cols, int32_t role, int32_t want_row,
                                     int32_t want_col, fp8_tensor *out, void *workspace,
                                     size_t ws_bytes, int32_t *dev_status, cudaStream_t stream);

/*
 * fp8_quantize_group with a stall planted in the grouped kernel's TMA pipeline. The group's
 * first tile (the first item's, loaded by CTA 0) expects 16 more bytes than its TMA loads
 * deliver.
 *
 * Arguments are as for fp8_quantize_group; dev_status is required.
 *
 * On the device, CTA 0's wait runs out after its budget. *dev_status then becomes
 * FP8_ERR_TIMEOUT, unless it already held a nonzero status. CTA 0's tiles are left unwritten;
 * the other CTAs finish theirs.
 *
 * Host-side errors are those of fp8_quantize_group, plus FP8_ERR_NULL when dev_status is
 * NULL. Takes about two seconds of GPU time.
 */
fp8_status fp8_test_quantize_group_stalled(const fp8_recipe *recipe, int32_t n,
                                           const fp8_quantize_item *items, int32_t *dev_status,
                                           cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8LIN_TEST_H */
