/*
 * Test-only entry points of gb300gemm (not for production callers).
 *
 * The pages describe no failure handling; this hook exists so that the
 * library's bounded waits can be exercised without faulting a GPU: with
 * fault = 1 the producer of each following run withholds its first
 * arrival on the shared-memory ring, the MMA issuer's wait for that stage
 * runs out after the plan's timeout (gemm_plan_set_timeout), the kernel
 * records GEMM_ERR_TIMEOUT, stops its other roles, frees its tensor memory
 * and returns.  With fault = 2 (GEMM plans) the producer computes A's row
 * coordinates one tiled extent too far: the copies read only the fill value
 * (D comes out wrong, nothing faults) and the checks build of the library
 * reports GEMM_ERR_CHECK.  fault = 0 restores normal runs.  Returns
 * GEMM_ERR_INVALID_ARG for a NULL plan, another fault value, or fault = 2 on a
 * chain plan.
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
 * The e4m3 CTA-pair plans' tile-width rule alone, without a device: 256 (one accumulator) or
 * 224 (two accumulators, the narrow form) columns for M x N x K with D of type d (GEMM_F32 or
 * GEMM_BF16) when `units` pairs run at once.  Plans with a row-major (N-contiguous) B keep 256
 * whatever the rule says.  *tile_n is written on GEMM_OK; GEMM_ERR_INVALID_ARG for NULL
 * tile_n, non-positive sizes or another d.
 */
gemm_status gemm_testing_e4m3_pair_tile_n(int64_t M, int64_t N, int64_t K, gemm_dtype d, int units, int *tile_n);

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

/*
 * TMEM data-movement probe: the tcgen05.ld example shapes of "Tensor Memory（TMEM）"
 * (section "Shape 和 Repeat Factor": .16x128b.x1 / .x2 / .x4 / .x8 move 16 lanes x 128
 * bits x num and give each thread 2 / 4 / 8 / 16 registers; section "每个 warp 能访问
 * 哪些 TMEM lanes": warp w of a warpgroup reaches lanes 32w..32w+31), run on the GPU.
 * One CTA of four warps writes (lane << 16) | column into every TMEM cell with
 * tcgen05.st.32x32b (each warp its own window), then each warp reads its window at its
 * first lane with .16x128b.x1 (column 0), .x2 (column 32), .x4 (column 64), .x8 (column
 * 128) and .32x32b.x32 (column 256).  host_out receives, for warp w and thread t, the
 * 62 registers of the five loads in that order (2 + 4 + 8 + 16 + 32 = 62 words) at
 * index (32w + t) * 62; n_words must be at least 128 * 62.  Synchronises the device.
 * GEMM_ERR_INVALID_ARG for NULL or too small a buffer, GEMM_ERR_UNSUPPORTED on another
 * device, GEMM_ERR_CUDA if a CUDA call fails.
 */
gemm_status gemm_testing_tmem_ld_probe(uint32_t *host_out, int64_t n_words);

/*
 * Shared-memory cost of the epilogue's staging patterns, measured alone: one CTA of four
 * warps, each issuing `iters` rounds of 128-bit accesses (load = 1: ld.shared.v4, 0:
 * st.shared.v4) in its own 4 KiB buffer; *clk_per_access = SM clocks per warp-wide access
 * (slowest warp).  pattern 0: bf16 D staging (64-byte rows, 16-byte chunk c of row r at
 * c ^ ((r / 2) % 4), the TMA's 64-byte swizzle); 1: fp32 C / D staging (128-byte rows,
 * chunk c at c ^ (r % 8), the 128-byte swizzle); 2: linear (a warp's 512 bytes
 * contiguous); 3 and 4: the rows of 0 and 1 without the swizzle.  Synchronises the
 * device.  GEMM_ERR_INVALID_ARG for a NULL output, a pattern outside 0..4, load not 0 or 1
 * or iters outside 1..2^20; GEMM_ERR_UNSUPPORTED on another device; GEMM_ERR_CUDA.
 */
gemm_status gemm_testing_staging_probe(int pattern, int load, int64_t iters, double *clk_per_access);

/*
 * The persistent kernels' work schedule, run on the host (no device needed): the pieces
 * that unit `unit` (a CTA, or a CTA pair) of a grid of `units` processes, in order, six
 * ints each in out[6 * i ..]: tile row tm, tile column tn (0 for the chain), k-blocks
 * [kb0, kb1), role (0 a whole tile or split-K slice, 1 the end of a tile that the previous
 * unit's span starts, 2 the start of a tile that the next unit's span ends) and flag slot.
 * chain = 0: the GEMM kernels (tiles_m x tiles_n tiles rasterised in groups of group_m
 * tile rows, splits K slices per tile); chain = 1: the two-product chain (tiles_m tiles;
 * tiles_n, group_m and splits ignored).  sk_units > 0 selects stream-K: the first
 * sk_dp_tiles tiles (a multiple of units) whole, then equal spans of the rest, with
 * sk_units == units and splits == 1.  At most max_pieces are written; *n_pieces gets the
 * count.  GEMM_ERR_INVALID_ARG for NULL pointers or values outside these ranges.
 */
gemm_status gemm_testing_schedule(int chain, int tiles_m, int tiles_n, int group_m, int num_kb, int splits,
                                  int sk_dp_tiles, int sk_units, int unit, int units, int *out, int max_pieces,
                                  int *n_pieces);

#ifdef __cplusplus
}
#endif

#endif /* GB300GEMM_TESTING_H */
