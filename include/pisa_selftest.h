/*
 * pisa_selftest.h - diagnostic entry point of the PISA library.
 *
 * Not part of the attention path. It checks the tensor-core building blocks
 * the attention kernel relies on (TMA loads with 128-byte swizzle, tcgen05.mma
 * with shared-memory and tensor-memory operands, tcgen05.ld/st) on one
 * 128 x 128 x 128 bf16 product, and the bounded-wait error path.
 */
#ifndef PISA_SELFTEST_H
#define PISA_SELFTEST_H

#include <stdint.h>

#include "pisa.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * pisa_selftest_tc
 *
 * a, b, bt  device bf16 [128][128], row-major, 16-byte aligned.
 * out       device float32 [4][128][128]:
 *             out[0] = a * b^T   (B read K-major from shared memory)
 *             out[1] = a * bt    (B read MN-major from shared memory)
 *             out[2] = a * bt    (A read from tensor memory, B MN-major)
 *             out[3] = a^T * bt  (A and B read MN-major from shared memory)
 * mode      0: compute the four products.
 *           1: wait on an mbarrier that is never signalled; the bounded wait
 *              must expire and store PISA_ERR_TIMEOUT in *dev_status (out is
 *              not written). The kernel returns normally.
 * dev_status optional device int32 (zeroed by the caller).
 * stream    cudaStream_t as void*.
 * Returns PISA_OK, PISA_ERR_INVALID_ARG or PISA_ERR_CUDA.
 */
int pisa_selftest_tc(const void* a, const void* b, const void* bt, float* out, int mode,
                     int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PISA_SELFTEST_H */
