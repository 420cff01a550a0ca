/*
 * mc_selftest.h -- diagnostic entry points of libmc (not part of the method).
 *
 * They exercise the building blocks of the tensor-core kernels in isolation so a
 * test can compare each against a plain matrix product on the GPU.
 */
#ifndef MC_SELFTEST_H_
#define MC_SELFTEST_H_

#include "mc.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * mc_selftest_umma -- one 128x128x128 tcgen05 MMA chain on a single CTA.
 *   X, W : bf16 [128][128] row-major, device, 16-byte aligned.
 *   D    : fp32 [128][128] row-major, device, written (form 4 writes columns 0..63).
 *   form : 0  D = X W^T, both operands from shared memory, both K-major
 *          1  D = X W^T, X from tensor memory, W K-major
 *          2  D = X W,   X from tensor memory, W MN-major
 *          3  D = X^T W, both from shared memory, both MN-major
 *          4  D[:, 0:64] = X W[0:64]^T, X from tensor memory, 64-row K-major W
 *          5  D = X W,   X from shared memory K-major, W MN-major
 *   Returns MC_OK, MC_ERR_NULL/MC_ERR_ALIGN/MC_ERR_MODE on bad arguments,
 *   MC_ERR_CUDA if the launch fails.  Synchronises the stream and returns
 *   MC_ERR_DEVICE_TIMEOUT if a bounded device wait gave up.
 */
int mc_selftest_umma(const void *X, const void *W, float *D, int form, mc_stream_t stream);

/*
 * mc_selftest_wait_timeout -- launches one CTA that waits on an mbarrier no
 * thread ever arrives at, with a limit of limit_ms milliseconds (1..5000), then
 * gives up, records the timeout and exits.  Synchronises the stream.  Returns
 * MC_ERR_DEVICE_TIMEOUT when the bounded wait behaved (the expected answer),
 * MC_OK if the wait wrongly completed, MC_ERR_CUDA on a launch failure.
 */
int mc_selftest_wait_timeout(int limit_ms, mc_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MC_SELFTEST_H_ */
