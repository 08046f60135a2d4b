// Host/device shared declarations of the GEMM library (not part of the C ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "gb300gemm.h"

namespace gb300 {

constexpr int TILE_M = 128;   // rows of D per CTA
constexpr int TILE_N = 256;   // columns of D per CTA (and per CTA pair)
constexpr int TILE_K16 = 64;  // 16-bit K elements per stage (one 128-byte swizzle row)

// Kernel parameters common to every GEMM kernel (passed by value).
struct KParams {
    int M, N, K;
    int tiles_m, tiles_n, num_tiles;
    int num_kb;          // K blocks (pipeline stages consumed per tile)
    int group_m;         // tile rasterisation: M tiles per group
    int has_c;
    int a_mn, b_mn;      // operand stored MN-major (M or N contiguous) instead of K-major
    int splits;          // K slices per tile (split-K); > 1: D already holds C, slices reduce-add into it
    uint32_t idesc;      // tcgen05 instruction descriptor
    int *status;         // device status word (sticky error code)
    uint64_t timeout_ns; // limit of every wait
    int fault;           // test hook: 1 = producer withholds its first arrival
    const uint8_t *sfa;  // block-scaled: packed scale factors (device)
    const uint8_t *sfb;
    // stream-K (sk != 0): the first sk_dp_tiles tiles go to the units whole, round by round;
    // the (tile, k-block) iterations of the remaining tiles are cut into sk_units equal
    // spans, one per unit.  A tile cut between two spans is finished by the unit whose
    // span covers its first k-block: the other unit stores its partial sum into D (fp32)
    // and publishes `epoch` in sk_flags[unit * CG + rank]; the finishing unit then adds
    // its own into D.
    int sk;
    int sk_dp_tiles;
    int sk_units;
    int epoch;
    int *sk_flags;
    // clock meter (non-null: thread 0 of every CTA adds its SM cycles and globaltimer
    // nanoseconds, from entry to exit, into clk_meter[0] and clk_meter[1])
    unsigned long long *clk_meter;
    // per-role clock accounting, TRACE_SLOTS counters per CTA (a GB300_TRACE=1 build only)
    unsigned long long *trace;
};

// Counters of the per-role trace (GB300_TRACE=1 builds), per CTA, in SM clock cycles
// unless noted.  Waits are the cycles a role spent in a barrier wait; issue/ld/store the
// cycles between its waits.  Epilogue counters are summed over the epilogue warps.
enum TraceSlot : int {
    TR_KERNEL_CLK = 0,   // entry to exit of thread 0
    TR_KERNEL_NS,        // the same span in globaltimer nanoseconds
    TR_PROD_WAIT,        // producer: waits for a free stage (empty[s])
    TR_PROD_ISSUE,       // producer: arming barriers and issuing the stage's TMA loads
    TR_PROD_STAGES,      // producer: stages filled (count)
    TR_MMA_WAIT_ACC,     // MMA issuer: waits for a free accumulator (tempty)
    TR_MMA_WAIT_AB,      // MMA issuer: waits for a stage's operands (full[s])
    TR_MMA_WAIT_SF,      // MMA issuer: (unused: with copier warps full[s] covers the stage's scales)
    TR_MMA_ISSUE,        // MMA issuer: scale copies (no copier), MMAs and commits
    TR_MMA_KBLOCKS,      // MMA issuer: k-blocks consumed (count)
    TR_MMA_PIECES,       // MMA issuer: work pieces (count)
    TR_MMA_FIRST,        // MMA issuer: entry to its first k-block's operands landing
    TR_MMA_END,          // MMA issuer: entry to the completion of its last MMA
    TR_CP_WAIT,          // copier: waits for a stage's scales in shared memory (sffull[s])
    TR_CP_ISSUE,         // copier: scale copies and commits
    TR_EPI_WAIT_ACC,     // epilogue: waits for a finished accumulator (tfull)
    TR_EPI_TMEM_LD,      // epilogue: tcgen05.ld and wait::ld
    TR_EPI_WAIT_C,       // epilogue: waits for a C box (and the partial sum of a stream-K tile)
    TR_EPI_STORE,        // epilogue: add C, convert, stage, issue the TMA store
    TR_EPI_PIECES,       // epilogue: pieces handled (count, summed over warps)
    TR_EPI_END,          // epilogue: entry to the last store issued (max over warps)
    TRACE_SLOTS = 24
};

// Tensor maps a kernel takes: A, B, C, D, and the packed scale factors (block-scaled only).
constexpr int NUM_MAPS = 6;

// A launch: grid, cluster width and dynamic shared memory.
struct LaunchShape {
    int grid;
    int cluster;
    int smem;
};

// bf16/fp16 kernel family (gemm_f16.cu)
struct F16Config {
    int cta_group;   // 1 or 2
    int out_bf16;    // D is bf16 (else fp32)
    int wide_epi = 0;   // pairs with fp32 D: 8 epilogue warps and one stage fewer (short K)
    int tile_n = TILE_N;   // pairs: TILE_N or F16_NARROW_N columns per tile
};
// the narrower pair tile the fp16/bf16 plans may choose when it fills the waves better
constexpr int F16_NARROW_N = 224;
int f16_stages(const F16Config &cfg);
int f16_smem_bytes(const F16Config &cfg);
cudaError_t f16_prepare(const F16Config &cfg);   // set the kernel's shared-memory limit
cudaError_t f16_max_active_clusters(const F16Config &cfg, int *clusters);
cudaError_t f16_launch(const F16Config &cfg, const LaunchShape &shape, const CUtensorMap *maps,
                       const KParams &p, cudaStream_t stream);

// split-K preparation (gemm_f16.cu): D = C, or D = 0 without C (fp32, n elements, n % 4 == 0)
cudaError_t init_d_launch(float *D, const float *C, size_t n, int sm_count, cudaStream_t stream);

// Operand kinds of the tensor-core kernel (tcgen05.mma kinds):
//   KIND_F16   fp16 / bf16, kind::f16
//   KIND_MXF8  e4m3 with a UE8M0 scale per 32 K, kind::mxf8f6f4 scale_vec::1X
//   KIND_MXF4  e2m1 with a UE8M0 scale per 32 K, kind::mxf4 scale_vec::2X
//   KIND_NVF4  e2m1 with a UE4M3 scale per 16 K, kind::mxf4nvf4 scale_vec::4X
enum GemmKind { KIND_F16 = 0, KIND_MXF8 = 1, KIND_MXF4 = 2, KIND_NVF4 = 3 };

// plan family of the two-product chain (gemm_chain.cu)
constexpr int FAMILY_CHAIN = 4;

// Static shape of a block-scaled kernel instance (per CTA group)
struct ScaledShape {
    int tile_n;      // columns of D per tile
    int stages;      // ring depth
    int smem;        // dynamic shared memory per CTA
    int bk;          // K elements per stage
    int sfa_bytes;   // packed SFA bytes per stage (one 512-byte block per 4 scales of 128 rows)
    int sfb_bytes;   // packed SFB bytes per stage (every column of the tile)
    int epi_box;     // columns of the epilogue's C / D boxes (32 or 16)
};

// A block-scaled kernel family: its instances (CTA group 1 / 2 x D fp32 / bf16, and for e4m3 a
// narrow CTA-pair form: 256 x 224 tiles with two accumulators; `narrow` selects it, and
// families without one (has_narrow false) ignore it)
struct ScaledFamily {
    ScaledShape (*shape)(int cta_group, bool narrow);
    cudaError_t (*prepare)(int cta_group, int out_bf16, bool narrow);      // set the kernel's shared-memory limit
    cudaError_t (*max_active_clusters)(int cta_group, int out_bf16, bool narrow, int *clusters);
    cudaError_t (*launch)(int cta_group, int out_bf16, bool narrow, const LaunchShape &shape, const CUtensorMap *maps,
                          const KParams &p, cudaStream_t stream);
    bool has_narrow;
};
// the narrow e4m3 pair tile's columns
constexpr int MXF8_NARROW_N = 224;
const ScaledFamily &family_mxf8();   // gemm_mxf8.cu
const ScaledFamily &family_mxf4();   // gemm_mxf4.cu
const ScaledFamily &family_nvf4();   // gemm_nvf4.cu

// Pack row-major scale factors SFA (M x sfk) and SFB (N x sfk) into the kernels'
// 512-byte TMEM-order blocks (gemm_sfpack.cu).  n_wg: groups of four scale columns
// per row of the packed layout (stages x scale words per stage); scales outside the
// matrices read as `pad` (the format's 1.0).
cudaError_t sf_pack(const uint8_t *sfa, const uint8_t *sfb, uint8_t *out_a, uint8_t *out_b, int M, int N, int sfk,
                    int row_blocks, int tiles_n, int tile_n, int n_wg, uint8_t pad, cudaStream_t stream);

// Two chained products D = C + round(A·B)·E (gemm_chain.cu): parameters of one launch
struct ChainParams {
    int M, K, N1, N2;
    int n1p, n2p;        // N1 and N2 rounded up to the MMA's N granule (16)
    int num_kb1;         // 64-element K blocks of the first product
    int num_kb2;         // 64-element K blocks of the second product (over n1p)
    int tiles;           // tiles of D (128 rows per CTA, 256 per CTA pair)
    int has_c;
    int f16;             // operands (and the rounded intermediate) fp16, else bf16
    uint32_t idesc1, idesc2;
    int *status;
    uint64_t timeout_ns;
    int fault;
    // stream-K over the first product's k-blocks (sk != 0; as in KParams): a tile cut
    // between two spans is finished by the unit whose span covers its first k-block; the
    // other stores its partial T (fp32, n1p columns rounded up to 32, of each of its CTA's 128 rows) in
    // sk_part[unit * CG + rank] and publishes `epoch` in sk_flags[unit * CG + rank]
    int sk;
    int sk_dp_tiles;
    int sk_units;
    int epoch;
    int *sk_flags;
    float *sk_part;
};
constexpr int CHAIN_MAX_N = 256;   // N1 and N2 limits: both products' accumulators share 512 TMEM columns
int chain_smem_bytes(int cta_group);
int chain_stages(int cta_group);
cudaError_t chain_prepare(int out_bf16, int cta_group);
cudaError_t chain_max_active_clusters(int out_bf16, int cta_group, int *clusters);
// grid: CTAs (a multiple of cta_group); tiles of 128 * cta_group rows
cudaError_t chain_launch(int out_bf16, int cta_group, int grid, const CUtensorMap *maps, const ChainParams &p,
                         cudaStream_t stream);

constexpr int EPI_COLS = 32;  // epilogue chunk width (columns)

}  // namespace gb300
