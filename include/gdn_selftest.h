/*
 * gdn_selftest.h -- self-test entry points of libgdn_gb300.so.
 *
 * Not part of the method: these exist so that a test suite can check, on the
 * device, the building blocks the tensor-core kernels rely on (shared-memory
 * tile layouts, tcgen05 descriptors, TMEM read-back) against a reference
 * product computed elsewhere.
 */
#ifndef GDN_GB300_SELFTEST_H
#define GDN_GB300_SELFTEST_H

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * gdn_selftest_mma -- D = A * B (times 2 when `twice`) on one CTA with
 * tcgen05.mma kind::f16 (M = 128), using the shared-memory layouts of the
 * chunk kernel.
 *   A  bf16 [128, K] row-major (device)    B  bf16 [K, N] row-major (device)
 *   D  fp32 [128, N] row-major (device, written)
 *   K  64 or 128;  N  64 or 128 (b_stacked requires N = 64)
 *   a_mn       0: A K-major in shared memory; 1: A M-major in shared memory;
 *              2: A in TMEM (row m in lane m, bf16 pairs per 32-bit column,
 *              written with tcgen05.st), the form of the chain's S and U
 *              operands
 *   b_mn       store B N-major (else K-major)
 *   b_stacked  K-major B placed in the first 64 rows of a 128-row tile
 *   twice      issue the MMA sequence twice with accumulation
 * Returns GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_TIMEOUT (the completion wait
 * gave up) or GDN_ERR_CUDA. Synchronises `stream`.
 */
int gdn_selftest_mma(const void* A, const void* B, float* D, int K, int N,
                     int a_mn, int b_mn, int b_stacked, int twice,
                     gdn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_SELFTEST_H */
