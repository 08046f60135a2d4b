/*
 * Test-only entry points of gb300gemm (not for production callers).
 *
 * The pages describe no failure handling; this hook exists so that the
 * library's bounded waits can be exercised without faulting a GPU: with
 * fault = 1 the producer of each following run withholds its first
 * arrival on the shared-memory ring, the MMA issuer's wait for that stage
 * runs out after the plan's timeout (gemm_plan_set_timeout), the kernel
 * records GEMM_ERR_TIMEOUT, stops its other roles, frees its tensor memory
 * and returns.  fault = 0 restores normal runs.  Returns
 * GEMM_ERR_INVALID_ARG for a NULL plan or another fault value.
 */
#ifndef GB300GEMM_TESTING_H
#define GB300GEMM_TESTING_H

#include "gb300gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

gemm_status gemm_testing_set_fault(gemm_plan_t p, int fault);

/*
 * The fp16/bf16 CTA-pair plans' tile-width rule alone, without a device: the
 * columns (256 or 224) of the pair tile that a plan for M x N x K with a row-major A,
 * column-major B and D of type d (GEMM_F32 or GEMM_BF16) takes when `units`
 * pairs run at once (76 on a GB300).  *tile_n is written on GEMM_OK;
 * GEMM_ERR_INVALID_ARG for NULL tile_n, non-positive sizes or another d.
 */
gemm_status gemm_testing_pair_tile_n(int64_t M, int64_t N, int64_t K, gemm_dtype d, int units, int *tile_n);

#ifdef __cplusplus
}
#endif

#endif /* GB300GEMM_TESTING_H */
