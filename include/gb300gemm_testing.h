/*
 * Test-only entry point of gb300gemm (not for production callers).
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

#ifdef __cplusplus
}
#endif

#endif /* GB300GEMM_TESTING_H */
