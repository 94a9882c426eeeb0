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
 * The CUDA context stays usable. The hook below makes such a wait run out on purpose,
 * without faulting, trapping or hanging the GPU, so tests can check that path.
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

#ifdef __cplusplus
}
#endif

#endif /* FP8LIN_TEST_H */
