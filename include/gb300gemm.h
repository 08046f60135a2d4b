/*
 * gb300gemm — tensor-core matrix multiply-accumulate D = A·B + C on one
 * NVIDIA GB300 (sm_103a), behind a plain C ABI.
 *
 * The operation is the one the three tensor-core generations share
 * ("Tensor Core 数据布局的演进", overview: D = AB + C, A and B the multiplied
 * matrices, C the addend, D the result), computed with fp32 accumulation:
 *
 *     D[i][j] = C[i][j] + sum_k a[i][k] * b[k][j]          (0 <= i < M, 0 <= j < N)
 *
 * Operands a and b are fp16 or bf16 values, or — block scaled — low-precision
 * values each multiplied by a scale shared by `blk` consecutive K elements
 * ("Tensor Core 数据布局的演进", section "Block-Scaled MMA 的 Scale Factors":
 * SFA[m][sfk] scales row m of A in K block sfk, SFB[n][sfk] scales column n
 * of B; section "scale_vec 的 Word 内复制": one, two or four scales per row
 * and MMA step):
 *
 *     a[i][k] = A[i][k] * sf(SFA[i][k/blk]),   b[k][j] = B[k][j] * sf(SFB[j][k/blk])
 *
 *   block_scaled = GEMM_SCALE_UE8M0_32: blk = 32, sf(c) = 2^(c - 127) (UE8M0),
 *                  A and B OCP e4m3 (scale_vec::1X) or OCP e2m1 (2X);
 *   block_scaled = GEMM_SCALE_UE4M3_16: blk = 16, sf(c) = the unsigned e4m3
 *                  value of c (UE4M3, bit 7 zero), A and B OCP e2m1 (4X).
 *
 * Memory layout (all buffers packed; no leading-dimension arguments):
 *   A    M x K, row-major (element (i,k) at A[i*K + k]) or, with
 *        a_row_major = 0, column-major (at A[k*M + i]).
 *   B    K x N, column-major (element (k,j) at B[j*K + k]) or, with
 *        b_row_major = 1, row-major (at B[k*N + j]).  The tensor core reads
 *        either order: K-major operands and M/N-major ones (described to it
 *        by the shared-memory descriptor's layout and the instruction
 *        descriptor's transpose bits).
 *   C    M x N fp32 row-major, or NULL for C = 0.
 *   D    M x N row-major, fp32 or bf16 (round to nearest even).
 *   SFA  M x ceil(K/blk) scale codes, row-major (block-scaled plans only).
 *   SFB  N x ceil(K/blk) scale codes, row-major (block-scaled plans only).
 *   e2m1 operands are packed two per byte along K, element 2t in bits 0..3
 *   of byte t; they must be K-major (A row-major, B column-major).
 *
 * Every global row stride and every base pointer must be a multiple of
 * 16 bytes: the tensor-memory-accelerator copy engine needs one dimension of
 * stride 1 and 16-byte aligned strides for the others ("(二) CUTLASS —— 掌握
 * Tensor Memory Accelerator（TMA）", section "使用 TMA 处理 remainder tiles
 * 以及 stride 要求": pad the tensor before calling otherwise).  For 16-bit
 * operands the contiguous extent (K, or M / N for column- / row-major A / B)
 * must be a multiple of 8, for e4m3 of 16, for e2m1 (K) of 32; for C and
 * fp32 D N % 4 == 0, for bf16 D N % 8 == 0.  M, N and K need not be multiples of
 * any tile size: the copy engine predicates the remainder tiles.
 *
 * Ownership: the caller owns every device buffer.  A plan owns host state and
 * one small device status word.  Calls on one plan are not thread-safe; calls
 * on different plans are.  No entry point aborts the process: each returns a
 * gemm_status.
 */
#ifndef GB300GEMM_H
#define GB300GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,   /* null plan/pointer, dimension <= 0, bad enum value */
    GEMM_ERR_UNSUPPORTED = 2,   /* dtype / layout combination or device not handled */
    GEMM_ERR_ALIGNMENT = 3,     /* a base pointer or row stride is not a multiple of 16 bytes */
    GEMM_ERR_CUDA = 4,          /* a CUDA runtime or driver call failed */
    GEMM_ERR_TIMEOUT = 5,       /* a bounded wait inside a kernel ran out; the kernel gave up */
    GEMM_ERR_CHECK = 6          /* an on-device check of a copy coordinate failed (the checks
                                   build of the library only; see gb300gemm_testing.h) */
} gemm_status;

typedef enum {
    GEMM_F16 = 0,
    GEMM_BF16 = 1,
    GEMM_E4M3 = 2,
    GEMM_F32 = 3,
    GEMM_E2M1 = 4               /* OCP FP4 E2M1, two elements per byte (block-scaled only) */
} gemm_dtype;

/* gemm_plan_create block_scaled modes */
#define GEMM_SCALE_NONE       0  /* fp16 / bf16 operands, no scales */
#define GEMM_SCALE_UE8M0_32   1  /* UE8M0 scale per 32 K elements: e4m3 or e2m1 operands */
#define GEMM_SCALE_UE4M3_16   2  /* UE4M3 scale per 16 K elements: e2m1 operands */

/* gemm_plan_create flags */
#define GEMM_FLAG_SYNC        0x1u  /* gemm_run synchronises its stream and returns the kernel status */
#define GEMM_FLAG_FORCE_1CTA  0x2u  /* use single-CTA tiles (cta_group::1) even where pairs would be chosen */
#define GEMM_FLAG_FORCE_2CTA  0x4u  /* use CTA-pair tiles (cta_group::2) even where single CTAs would be chosen */
#define GEMM_FLAG_DETERMINISTIC 0x8u /* bitwise-reproducible results run to run: no split-K (see gemm_plan_set_split_k) */

typedef struct gemm_plan *gemm_plan_t;

/* What a plan will launch (for tests, benchmarks and logs). */
typedef struct {
    int cta_group;          /* 1: one CTA per tile, 2: CTA pairs (cta_group::2) share a tile */
    int tile_m, tile_n;     /* output tile of one CTA (group) */
    int tile_k;             /* K elements per pipeline stage */
    int stages;             /* shared-memory ring depth */
    int grid;               /* CTAs launched (persistent) */
    int tiles;              /* output tiles */
    int smem_bytes;         /* dynamic shared memory per CTA */
    int launches_per_run;   /* kernels one gemm_run enqueues */
    int sm_count;           /* SMs of the device the plan was made for */
    int splits;             /* K slices per output tile (1 = no split-K) */
    int stream_k;           /* 1: the last waves' tiles are shared out as equal spans of K (stream-K) */
} gemm_plan_info;

/*
 * Validate a problem and choose its kernel.  M, N, K > 0.  ab and block_scaled
 * go together as GEMM_F16 or GEMM_BF16 with GEMM_SCALE_NONE, GEMM_E4M3 with
 * GEMM_SCALE_UE8M0_32, or GEMM_E2M1 with GEMM_SCALE_UE8M0_32 or
 * GEMM_SCALE_UE4M3_16 (other pairs: GEMM_ERR_UNSUPPORTED; a block_scaled
 * value outside 0..2: GEMM_ERR_INVALID_ARG).  c must be GEMM_F32; d is
 * GEMM_F32 or GEMM_BF16.  a_row_major and b_row_major choose the storage
 * order of A and B (all four combinations for 16- and 8-bit operands; a
 * block-scaled e4m3 plan with row-major B needs CTA pairs, so
 * GEMM_FLAG_FORCE_1CTA then returns GEMM_ERR_UNSUPPORTED; e2m1 operands
 * must be K-major, a_row_major = 1 and b_row_major = 0).  Row-stride alignment (see above) is checked here and
 * returns GEMM_ERR_ALIGNMENT.  The plan is bound to the CUDA device current
 * at creation, which must be compute capability 10.3.  *out is set only on
 * GEMM_OK.
 */
gemm_status gemm_plan_create(gemm_plan_t *out, int64_t M, int64_t N, int64_t K,
                             gemm_dtype ab, gemm_dtype c, gemm_dtype d,
                             int a_row_major, int b_row_major, int block_scaled,
                             unsigned flags);

/*
 * Enqueue D = A·B + C on cuda_stream (a cudaStream_t; NULL = legacy default
 * stream).  A, B, D: device pointers, non-NULL, 16-byte aligned; C: device
 * pointer or NULL (C = 0); SFA, SFB: device pointers for block-scaled plans,
 * ignored otherwise.  D must not overlap A, B, C, SFA or SFB.  Returns after
 * enqueueing (asynchronous) unless the plan has GEMM_FLAG_SYNC, in which case
 * it waits for the stream and returns the kernel's status.
 */
gemm_status gemm_run(gemm_plan_t p, const void *A, const void *B, const void *C, void *D,
                     const uint8_t *SFA, const uint8_t *SFB, void *cuda_stream);

/*
 * The same product with HOST buffers (any host memory; page-locked memory
 * copies fastest): copies A, B, C (and SFA, SFB) to device buffers the plan
 * owns (allocated on first use, freed by gemm_plan_destroy), runs the kernel,
 * copies D back and waits for it.  Returns the kernel's status.  For fp16/bf16
 * plans with row-major A and at least two chunks of 1024 rows, the product runs
 * as a pipeline over up to 8 row chunks on three plan-owned streams (after the
 * work already queued on cuda_stream): B and then each chunk's rows of A and C
 * are copied up, each chunk's product starts as soon as its rows have landed,
 * and its rows of D are copied back while the next chunks are copied up.
 */
gemm_status gemm_run_host(gemm_plan_t p, const void *A, const void *B, const void *C, void *D,
                          const uint8_t *SFA, const uint8_t *SFB, void *cuda_stream);

/*
 * Wait for the stream of the plan's last run, read the plan's device status
 * word (GEMM_OK, GEMM_ERR_TIMEOUT if a kernel gave up on a wait, or, in the
 * checks build only, GEMM_ERR_CHECK if a copy coordinate failed its check; the
 * first error a run records stands) and reset it to GEMM_OK.
 */
gemm_status gemm_plan_last_status(gemm_plan_t p);

/* Fill *info with the plan's launch configuration. */
gemm_status gemm_plan_get_info(gemm_plan_t p, gemm_plan_info *info);

/*
 * Set the limit, in nanoseconds, of every wait inside the plan's kernels
 * (default 1e9).  When a wait runs out the kernel records GEMM_ERR_TIMEOUT in
 * the status word, its other roles stop, it frees its tensor memory and it
 * returns; the CUDA context stays usable.
 */
gemm_status gemm_plan_set_timeout(gemm_plan_t p, uint64_t ns);

/*
 * Split-K ("(二) CUTLASS —— 掌握 Tensor Memory Accelerator（TMA）", section
 * "TMA Store Reduce": a TMA store can add its shared-memory tile into global
 * memory instead of overwriting it).  With splits > 1 each output tile's K
 * range is cut into that many slices that run as separate work units: a
 * small kernel first sets D = C (or 0), then every slice adds its partial
 * product into D with a TMA reduce-add.  This fills the GPU when there are
 * fewer output tiles than SMs.  splits = 0 lets the plan choose (it splits
 * fp32-D problems whose tiles fill at most half the GPU and whose K spans
 * at least 8 k-blocks), 1 turns split-K off; splits is clamped to the number
 * of k-blocks.  Requires fp32 D (GEMM_ERR_UNSUPPORTED otherwise): rounding
 * every partial sum to bf16 would cost accuracy.  The order in which slices
 * are added varies between runs, so results may differ in the last bits; a
 * plan created with GEMM_FLAG_DETERMINISTIC never splits (splits > 1 then
 * returns GEMM_ERR_UNSUPPORTED).
 */
gemm_status gemm_plan_set_split_k(gemm_plan_t p, int splits);

/*
 * Stream-K scheduling of the same product (a property of this library; the pages have
 * no counterpart to it, and it does not change what is computed).  When an fp32-D plan
 * has more output tiles than its persistent grid runs at once but not a whole number of
 * waves, the CTAs (or CTA pairs) first take whole tiles round by round, then share the
 * last one to two waves' worth of tiles out as equal spans of K blocks, so that all of
 * them finish together.  A tile cut between two spans is finished by the span that
 * covers its first K block: the other stores its partial sum into D and publishes it
 * with a flag (plan-owned, a few hundred bytes); the finishing CTA waits for the flag (a
 * bounded wait: GEMM_ERR_TIMEOUT if it runs out) and adds its own part and C into D with
 * a TMA reduce-add.  Results do not depend on timing (each tile is summed in a fixed
 * order), so the schedule is allowed with GEMM_FLAG_DETERMINISTIC; it is never combined
 * with split-K.  enable = 1 (the default) uses it where it was measured to pay — fp32 D,
 * at least 64 K blocks per tile and fewer than 4 waves — and 0 never; other values
 * return GEMM_ERR_INVALID_ARG.  Runs of one stream-K plan must not overlap on the GPU
 * (they share the flags).  Chain plans (gemm_chain_plan_create) take it only on
 * request (enable = 1; it measured slower than whole tiles on the shapes tried): they
 * then share out the first product's K blocks the same way when their tiles make more
 * than one wave but fewer than 4 and not a whole number, with at least 16 K blocks per
 * tile; the finishing CTA adds the other span's partial T (handed over through a
 * plan-owned buffer of 128 x N1 fp32 values per CTA of the grid) before rounding.
 */
gemm_status gemm_plan_set_stream_k(gemm_plan_t p, int enable);

/*
 * SM clock meter of a plan's runs (a measurement aid; the pages have no counterpart and
 * it does not change what is computed).  The SM clock under a dense tensor load sits
 * well below its maximum and moves with the power limit, so a per-clock roofline needs
 * the clock the kernel itself ran at.  enable = 1 allocates a 16-byte device counter on
 * first use and clears it; every later gemm_run and gemm_run_host of the plan then has
 * thread 0 of each CTA add its SM clock cycles (clock64) and globaltimer nanoseconds,
 * from kernel entry to exit, into that counter (two atomic adds per CTA).  enable = 0
 * stops counting; other values return GEMM_ERR_INVALID_ARG; chain plans return
 * GEMM_ERR_UNSUPPORTED.  gemm_plan_read_clock_meter synchronises the device, reads and
 * clears the counter, and returns *sm_mhz = cycles / nanoseconds * 1000 (the mean SM
 * clock over every counted CTA lifetime) and *cta_seconds (those lifetimes summed); both
 * are 0 when nothing was counted.  Runs that overlap on the GPU add into one counter.
 */
gemm_status gemm_plan_set_clock_meter(gemm_plan_t p, int enable);
gemm_status gemm_plan_read_clock_meter(gemm_plan_t p, double *sm_mhz, double *cta_seconds);

/* Release the plan (its status word and any host-run buffers).  NULL is a no-op. */
gemm_status gemm_plan_destroy(gemm_plan_t p);

/*
 * Allocation-free variant of gemm_run for the fp16/bf16 kernel (the pages
 * have no counterpart to this entry point; it is a property of this library).
 *
 * Some callers cannot call cudaMalloc: a host program whose device memory is
 * all owned by its own allocator and that forbids allocations behind its
 * back, a latency-critical loop that cannot afford the device-wide
 * synchronisation cudaMalloc and cudaFree imply, or a plug-in held to a fixed
 * memory budget.  The plan API does allocate (each plan's device status
 * word), so this entry point takes no plan and allocates nothing: the
 * kernel's only memory beyond A, B, C and D — its 4-byte status word — lives
 * in a file-scope __device__ array of 256 bytes that every GPU which loads
 * the library holds until the process exits.  A kernel needing more scratch
 * than the array holds would be rejected with GEMM_ERR_INVALID_ARG.
 *
 * Arguments mean what they mean for gemm_plan_create + gemm_run with
 * a_row_major = 1, b_row_major = 0, c = GEMM_F32 and no flags: ab is GEMM_F16
 * or GEMM_BF16, d is GEMM_F32 or GEMM_BF16, C may be NULL.  The caller owns
 * and passes every input and output.  The kernel takes the CTA mode such a
 * plan would (CTA pairs when M >= 1024 and N >= 1024), but always with
 * 128 x 256 (single CTA) or 256 x 256 (pair) tiles, the 4-warp epilogue and
 * no split-K or stream-K; a plan may choose 256 x 224 pair tiles, the 8-warp
 * epilogue, split-K or stream-K instead, so results can differ from
 * gemm_run's in the order of the fp32 sums (both meet the same accuracy
 * bound) and in speed.
 *
 * With wait = 0 the call returns after enqueueing and the kernel's status is
 * not reported: a GEMM_ERR_TIMEOUT stays in the array until the next call
 * clears it.  With wait != 0 it synchronises cuda_stream and returns the
 * kernel's status (GEMM_ERR_TIMEOUT if a bounded wait ran out); that
 * synchronisation is not allowed on a stream being captured into a graph,
 * so wait != 0 on a capturing stream returns GEMM_ERR_INVALID_ARG before
 * anything is enqueued.
 *
 * The first call on a device does a one-time set-up there (it looks up the
 * array's device address with cudaGetSymbolAddress and sets the kernel's
 * shared-memory limit); make that first call before any stream capture.  All
 * calls on a device share the one array, and each call clears the status word
 * before its kernel runs, so calls whose kernels overlap on the GPU (for
 * example on two streams at once) race on it; serialise them.
 */
gemm_status gemm_run_noalloc(int64_t M, int64_t N, int64_t K, gemm_dtype ab, gemm_dtype d,
                             const void *A, const void *B, const void *C, void *D,
                             void *cuda_stream, int wait);

/*
 * Two chained products with the intermediate kept on chip ("Tensor Core 数据布局的
 * 演进", section "TMEM 中的累加器": some tcgen05.mma forms read their A operand from
 * tensor memory, so a first product's result can feed a second one without a
 * round trip through global memory):
 *
 *     T[i][j] = sum_k a[i][k] * b[k][j]               (fp32 accumulation)
 *     P[i][j] = T[i][j] rounded to the operand type   (round to nearest even)
 *     D[i][n] = C[i][n] + sum_j P[i][j] * e[j][n]      (fp32 accumulation)
 *
 * A is M x K row-major, B is K x N1 column-major (element (k,j) at B[j*K + k]),
 * E is N1 x N2 column-major (element (j,n) at E[n*N1 + j]), C is M x N2 fp32
 * row-major or NULL, D is M x N2 row-major fp32 or bf16.  ab (A, B, E and P) is
 * GEMM_F16 or GEMM_BF16.  1 <= N1, N2 <= 256 (both products' accumulators share
 * one SM's 512 tensor-memory columns; otherwise GEMM_ERR_UNSUPPORTED); K and N1
 * multiples of 8, N2 a multiple of 4 (fp32 D) or 8 (bf16 D), else
 * GEMM_ERR_ALIGNMENT.  The plan runs CTA pairs (256-row tiles, each CTA holding
 * half of B's and E's rows) when M > 128 and N1 and N2, rounded up to multiples of
 * 16, are multiples of 32, else single CTAs; GEMM_FLAG_FORCE_1CTA and
 * GEMM_FLAG_FORCE_2CTA choose the form (GEMM_FLAG_FORCE_2CTA with an N1 or N2 that
 * does not round to a multiple of 32: GEMM_ERR_UNSUPPORTED).  The plan works with
 * gemm_plan_last_status, gemm_plan_get_info, gemm_plan_set_timeout and
 * gemm_plan_destroy; gemm_run / gemm_run_host reject it (GEMM_ERR_INVALID_ARG),
 * and gemm_plan_set_split_k accepts only 0 or 1.  Pointers, streams, errors and
 * GEMM_FLAG_SYNC behave as for gemm_run; gemm_chain_run_host is the host-buffer
 * form (like gemm_run_host).
 */
gemm_status gemm_chain_plan_create(gemm_plan_t *out, int64_t M, int64_t N1, int64_t N2, int64_t K,
                                   gemm_dtype ab, gemm_dtype d, unsigned flags);
gemm_status gemm_chain_run(gemm_plan_t p, const void *A, const void *B, const void *E, const void *C,
                           void *D, void *cuda_stream);
gemm_status gemm_chain_run_host(gemm_plan_t p, const void *A, const void *B, const void *E, const void *C,
                                void *D, void *cuda_stream);

/* Static description of a status code. */
/*
 * Tensor-pipe rate probe (measurement, not part of the GEMM path).  Launches one
 * CTA (cta_group = 1) or CTA pair (cta_group = 2) per SM; in each, one thread
 * issues `iters` groups of four back-to-back tcgen05.mma of the GEMM kernels'
 * instruction shape (M = 128 * cta_group, N = 256, 32 bytes of K per
 * instruction: K = 16 for f16/bf16, 32 for e4m3, 64 for e2m1) from operands
 * already in shared memory into one TMEM accumulator, and times the stream
 * with the SM clock and the globaltimer ("Tensor Core 数据布局的演进", section on
 * Blackwell: tcgen05.mma reads A and B from shared memory and accumulates in TMEM;
 * "Tensor Memory（TMEM）": the accumulator's columns are allocated per CTA).  ab / block_scaled pick
 * the kind as for gemm_plan_create.  1 <= iters <= 2^20.  Synchronises the
 * device first and again before returning; meant for an otherwise idle GPU.
 * Errors: GEMM_ERR_INVALID_ARG (out NULL, cta_group not 1 or 2, iters out of
 * range), GEMM_ERR_UNSUPPORTED (another kind or device), GEMM_ERR_CUDA,
 * GEMM_ERR_TIMEOUT (a CTA's wait ran out).  *out is written only on GEMM_OK.
 */
typedef struct {
    double flop_per_clk_per_sm;  /* dense FLOP per SM clock (median over CTA groups; 2 FLOP per multiply-add) */
    double sm_mhz;               /* SM clock during the run (median of clocks / globaltimer time) */
    double tflops;               /* whole-GPU rate: FLOPs of every CTA group / kernel time (CUDA events) */
    double ms;                   /* kernel time */
    int sms;                     /* CTAs launched (one per SM) */
} gemm_tensor_rate;
gemm_status gemm_measure_tensor_rate(gemm_dtype ab, int block_scaled, int cta_group, int64_t iters,
                                     gemm_tensor_rate *out);

const char *gemm_status_string(gemm_status s);

#ifdef __cplusplus
}
#endif

#endif /* GB300GEMM_H */
