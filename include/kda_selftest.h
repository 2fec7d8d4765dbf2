/*
 * kda_selftest.h -- test-only entry points of libkda.
 *
 * The chunked prefill kernels feed tcgen05.mma from shared-memory tiles in a
 * 128-byte-swizzled layout through hand-built descriptors. The pages describe
 * the intra-chunk products only as dense tensor-core matmuls (Kimi K3 --
 * Architecture Notes, section 1.2, "K3's answer"); this entry point runs ONE
 * such product in isolation so a test can compare it with a host matrix
 * product and pin every descriptor setting the kernels use.
 */
#ifndef KDA_SELFTEST_H
#define KDA_SELFTEST_H

#include <stdint.h>

#include "kda.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * kda_selftest_umma -- D = (negate_a ? -A : A) . B^T on the tensor cores.
 *
 *   A  [M, K] fp32, row-major, device           (M = 64 or 128)
 *   B  [N, K] fp32, row-major, device           (16 <= N <= 256, N % 16 == 0)
 *   fmt operand format the inputs are rounded to before the product:
 *      0 = fp16, 1 = bf16 (kind::f16), 2 = tf32 (kind::tf32, round to nearest)
 *   sw64: K-major 16-bit operands use the 64-byte swizzle (rows of 32 elements)
 *      instead of the 128-byte one
 *   D  [128, N] fp32, device: the raw accumulator, one row per tensor-memory
 *      lane (for M = 128 row m is lane m; for M = 64 the test learns the lanes)
 *   K  16 .. 128, a multiple of 16
 *   a_mn_major / b_mn_major: stage the operand with M (or N) contiguous
 *      (16-bit formats; M or N a multiple of 64) instead of K contiguous
 *   *_lbo, *_sbo: the leading / stride byte offsets put in each descriptor
 *   status: device int, set to 1 if the MMA completion wait gave up
 *
 * One CTA, 128 threads, about 129 KB of shared memory. Enqueued on `stream`.
 */
kda_status kda_selftest_umma(const float *A, const float *B, float *D, int32_t M, int32_t N, int32_t K,
                             int32_t fmt, int32_t sw64, int32_t a_mn_major, int32_t b_mn_major, int32_t negate_a,
                             uint32_t a_lbo,
                             uint32_t a_sbo, uint32_t b_lbo, uint32_t b_sbo, int32_t *status, void *stream);

/*
 * kda_selftest_wait_timeout -- runs the library's bounded mbarrier wait on a
 * phase that nothing completes, so that a test can check the failure path
 * without faulting the GPU: the wait gives up after its limit (about 2 s),
 * records KDA_ERR_TIMEOUT in the device error word (which the next
 * kda_check_device_error reports and clears) and the kernel returns normally,
 * leaving the context usable. No counterpart on the pages: this is the
 * library's own failure detection.
 *
 *   status  device uint32, set to 1 when the wait gave up (0 if it had not)
 *
 * One CTA of 32 threads. Enqueued on `stream`; returns KDA_ERR_INVALID_ARG for
 * a null or misaligned status pointer.
 */
kda_status kda_selftest_wait_timeout(uint32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_SELFTEST_H */
