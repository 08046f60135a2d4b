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

/*
 * Per-role clock trace of the GEMM kernels, for finding what a kernel waits on.  Only a
 * library compiled with GB300_TRACE=1 (the "trace" build variant, libgb300gemm_trace.so)
 * keeps it; the default build compiles every mark out.  gemm_testing_trace_slots()
 * returns the number of 64-bit counters kept per CTA (0 in a build without the trace).
 * gemm_testing_set_trace points the plan's later gemm_run calls at a caller-owned device
 * buffer of at least grid * slots * 8 bytes (grid from gemm_plan_get_info), to which each
 * CTA adds its counters (the caller clears it; counter i of CTA c at index c * slots + i,
 * in the order of the trace counter list of the Python binding: kernel cycles and ns,
 * producer wait / issue / stages, MMA issuer waits for an accumulator, operands and
 * scales, its issue time, k-blocks, pieces, first and last MMA, the scale copier's wait
 * and issue, the epilogue warps' accumulator wait, TMEM loads, C wait, store work,
 * pieces and end).  NULL stops tracing.  GEMM_ERR_UNSUPPORTED in a build without the
 * trace or for a chain plan, GEMM_ERR_INVALID_ARG for a NULL plan or a buffer too small.
 */
int gemm_testing_trace_slots(void);
gemm_status gemm_testing_set_trace(gemm_plan_t p, void *dev_buffer, int64_t bytes);

#ifdef __cplusplus
}
#endif

#endif /* GB300GEMM_TESTING_H */
