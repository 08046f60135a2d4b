// C ABI of the GEMM library (include/gb300gemm.h): plan validation, kernel
// choice, tensor-map encoding and launch.
//
// Tensor maps ("(二) CUTLASS —— 掌握 Tensor Memory Accelerator（TMA）", host
// code: a copy descriptor built on the host from the global tensor and the
// shared-memory tile, passed to the kernel as a __grid_constant__ parameter)
// are encoded with the driver's cuTensorMapEncodeTiled, fetched through the
// runtime's entry-point query so that the library does not link libcuda.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include <cudaTypedefs.h>

#include "gemm_internal.h"
#include "ptx.cuh"

using namespace gb300;

// M tiles per rasterisation group (tuning knobs)
#ifndef GB300_GROUP_M_PAIRS
#define GB300_GROUP_M_PAIRS 12
#endif
#ifndef GB300_GROUP_M_SINGLE
#define GB300_GROUP_M_SINGLE 16
#endif

// stream-K needs at least this many k-blocks per tile (32 lost 10 % on block-scaled e4m3 4096^3,
// whose 128-element k-blocks make K = 4096 only 32 of them)
#ifndef GB300_SK_MIN_KB
#define GB300_SK_MIN_KB 64
#endif

// L2 fill granularity of the 32-column C boxes (128-byte rows; 128-byte fills saved 3 % of the
// DRAM reads at 8192^3 and changed no timing, so the default stays 256)
#ifndef GB300_C_PROMO32
#define GB300_C_PROMO32 CU_TENSOR_MAP_L2_PROMOTION_L2_256B
#endif

// gemm_run_host splits a product into at most this many row chunks
#ifndef GB300_HOST_CHUNKS
#define GB300_HOST_CHUNKS 8
#endif
#ifndef GB300_HOST_MIN_ROWS
#define GB300_HOST_MIN_ROWS 1024
#endif
constexpr int HOST_CHUNKS = GB300_HOST_CHUNKS;        // row chunks of the host-buffer pipeline (at most)
constexpr int HOST_MIN_ROWS = GB300_HOST_MIN_ROWS;    // rows of the smallest chunk

struct gemm_plan {
    int64_t M, N, K;
    gemm_dtype ab, c, d;
    int block_scaled;
    int a_mn, b_mn;           // A column-major (M contiguous), B row-major (N contiguous)
    unsigned flags;
    int device;
    int sm_count;
    int cta_group;
    int stages;
    int tiles_m, tiles_n, tiles;
    int grid;
    int smem;
    int group_m;
    uint64_t timeout_ns;
    int fault;
    int *status;              // device word
    int family;               // GemmKind of the kernel: fp16/bf16, or block-scaled e4m3 / e2m1
    int splits;               // K slices per tile (1 = no split-K)
    int capacity;             // work units the persistent grid runs at once (CTAs or CTA pairs)
    int split_request;        // 0 = choose automatically, n >= 1 = asked for
    int sk_request;           // stream-K: 1 = where it balances the waves (default), 0 = never
    int wide_epi;             // fp16/bf16 pairs, fp32 D, short K: the 8-epilogue-warp kernel
    bool narrow;              // block-scaled pairs: the family's narrow pair form (e4m3: 256 x 224 tiles)
    int sk;                   // stream-K chosen
    int sk_dp_tiles;          // stream-K: tiles the units take whole before their spans
    int *sk_flags;            // stream-K: one flag per (slot, CTA of the group)
    float *sk_part;           // chain stream-K: one partial T per (slot, CTA of the group)
    uint32_t epoch;           // stream-K: runs so far (the value a run's flags carry)
    int tile_n;
    int epi_box;              // columns of the epilogue's C / D boxes (32 or 16)
    int tile_k;               // K elements per stage
    int num_kb;
    int sfa_stage_bytes, sfb_stage_bytes;   // block-scaled: packed scales per stage (per CTA)
    int64_t N2;               // chain plans: columns of D (N is the intermediate's N1)
    const void *lastE;
    void *hE;
    uint8_t *ws_a, *ws_b;     // block-scaled: packed scale factors (workspace)
    // device buffers of gemm_run_host (allocated on first use)
    void *hA, *hB, *hC, *hD;
    // gemm_run_host's pipeline: copy-in, compute and copy-out streams and their events
    bool pipe_ready;
    cudaStream_t pipe_in, pipe_comp, pipe_out;
    cudaEvent_t pipe_entry, pipe_in_done[HOST_CHUNKS], pipe_k_done[HOST_CHUNKS];
    uint8_t *hSFA, *hSFB;
    // tensor maps of the last run, reused while the pointers repeat
    const void *lastA, *lastB, *lastC, *lastD;
    CUtensorMap maps[NUM_MAPS];   // A, B, C, D, packed SFA, packed SFB (chain plans: A, B, C, D, E)
    bool maps_valid;
    unsigned long long *clk_meter;   // clock meter: SM cycles, globaltimer ns (device, allocated on first use)
    bool clk_meter_on;
    unsigned long long *trace;       // per-role trace buffer (caller-owned, trace builds only)
};

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

int elem_bits(gemm_dtype t) { return t == GEMM_E2M1 ? 4 : t == GEMM_E4M3 ? 8 : (t == GEMM_F32 ? 32 : 16); }

// bytes of n elements of type t (4-bit elements are packed two per byte)
size_t bytes_of(gemm_dtype t, int64_t n) { return (size_t)((n * elem_bits(t) + 7) / 8); }

// the family's scale-format 1.0: pads the packed scales outside the matrices
uint8_t unit_scale(int family) { return family == KIND_NVF4 ? 0x38 : 127; }

// K elements sharing one scale
int scale_block(int family) { return family == KIND_NVF4 ? 16 : 32; }

const ScaledFamily &scaled_family(int family) {
    return family == KIND_MXF4 ? family_mxf4() : (family == KIND_NVF4 ? family_nvf4() : family_mxf8());
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2-D row-major tensor [outer][inner] with a box of box_outer x box_inner elements; `promo`
// is the L2 fill granularity of the copies (lines fetched around each box row)
bool encode_2d(CUtensorMap *m, CUtensorMapDataType dt, int ebytes, const void *ptr, uint64_t inner, uint64_t outer,
               uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw,
               CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
    if (!encoder()) return false;      // the driver's encoder is looked up on first use
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * (uint64_t)ebytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          sw, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

CUtensorMapDataType tma_dtype(gemm_dtype t) {
    switch (t) {
    case GEMM_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case GEMM_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    case GEMM_F32: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    default: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
    }
}

// Tensor maps of A, B, C and D for the plan's operands with M rows (maps[0..3])
bool encode_operand_maps(const gemm_plan *p, CUtensorMap *maps, const void *A, const void *B, const void *C, void *D,
                         int64_t M) {
    std::memset(maps, 0, 4 * sizeof(CUtensorMap));
    // 4-bit operands are mapped as bytes (two K elements each, K-major only)
    const bool fp4 = p->ab == GEMM_E2M1;
    const int eb = fp4 ? 1 : elem_bits(p->ab) / 8;
    const uint64_t k_units = fp4 ? (uint64_t)p->K / 2 : (uint64_t)p->K;
    const uint32_t bk = 128u / (uint32_t)eb;                       // tensor-map elements in a 128-byte row
    const uint32_t b_rows = (uint32_t)(p->tile_n / p->cta_group);
    // K-major operand: [rows][K], box of bk x rows; MN-major operand: [K][rows], box one
    // 128-byte atom (atom elements) wide along the rows and bk deep along K
    const uint32_t atom = 128u / (uint32_t)eb;
    bool ok = (p->a_mn ? encode_2d(&maps[0], tma_dtype(p->ab), eb, A, M, p->K, atom, bk, CU_TENSOR_MAP_SWIZZLE_128B)
                       : encode_2d(&maps[0], tma_dtype(p->ab), eb, A, k_units, M, bk, TILE_M, CU_TENSOR_MAP_SWIZZLE_128B)) &&
              (p->b_mn ? encode_2d(&maps[1], tma_dtype(p->ab), eb, B, p->N, p->K, atom, bk, CU_TENSOR_MAP_SWIZZLE_128B)
                       : encode_2d(&maps[1], tma_dtype(p->ab), eb, B, k_units, p->N, bk, b_rows, CU_TENSOR_MAP_SWIZZLE_128B));
    // C and D boxes: 32 rows x epi_box columns, swizzled over their row (fp32: 128 or 64
    // bytes, bf16: 64 or 32 bytes), as the epilogue stages them
    const uint32_t box = (uint32_t)p->epi_box;
    const CUtensorMapSwizzle sw32 = box == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const CUtensorMapSwizzle sw16 = box == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
    // C is read once, with an evict-first hint: a 64-byte box row fills only its own 64 bytes
    // of L2 (a 256-byte fill would be evicted before the neighbouring boxes read it)
    if (ok && C)
        ok = encode_2d(&maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, p->N, M, box, 32, sw32,
                       box == 32 ? GB300_C_PROMO32 : CU_TENSOR_MAP_L2_PROMOTION_L2_64B);
    if (ok) {
        if (p->d == GEMM_BF16)
            ok = encode_2d(&maps[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, p->N, M, box, 32, sw16);
        else
            ok = encode_2d(&maps[3], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, p->N, M, box, 32, sw32);
    }
    return ok;
}

gemm_status encode_maps(gemm_plan *p, const void *A, const void *B, const void *C, void *D) {
    if (p->maps_valid && A == p->lastA && B == p->lastB && C == p->lastC && D == p->lastD) return GEMM_OK;
    if (!encoder()) return GEMM_ERR_CUDA;
    // maps 4 and 5 (scale factors) belong to the plan and stay
    if (!encode_operand_maps(p, p->maps, A, B, C, D, p->M)) {
        p->maps_valid = false;
        return GEMM_ERR_CUDA;
    }
    p->lastA = A;
    p->lastB = B;
    p->lastC = C;
    p->lastD = D;
    p->maps_valid = true;
    return GEMM_OK;
}

// The column width of an fp16/bf16 CTA-pair tile: 256 x 224 tiles when they fill the
// persistent rounds of `units` pairs clearly better than 256 x 256 ones.  Estimated
// efficiency (each factor measured on GB300) = used share of the tile columns x busy share of
// the rounds (0.89 where stream-K would balance them) x, for 224, the 3.5 % its extra operand
// bytes per FLOP cost at 8192^3, or, for 256 with fp32 D and short K, the gain of the wide
// epilogue (+14 % at 16 k-blocks, +3.5 % at 33); 224 must win by 2 %.
int pair_tile_n(int64_t M, int64_t N, int64_t K, bool f32, int units) {
    const int64_t tiles_m = (M + 2 * TILE_M - 1) / (2 * TILE_M), kb = (K + TILE_K16 - 1) / TILE_K16;
    auto eff = [&](int bn) {
        const int64_t tn = (N + bn - 1) / bn, tiles = tiles_m * tn;
        const int64_t rounds = (tiles + units - 1) / units;
        const bool sk = f32 && kb >= 64 && tiles >= units && tiles % units != 0 && tiles < 4 * units;
        double e = (double)N / (double)(tn * bn);
        e *= sk ? 0.89 : (double)tiles / (double)(rounds * units);
        if (bn == F16_NARROW_N) e *= 0.965;
        else if (f32 && kb <= 40 && 2 * tiles > units) e *= 1.0 + 0.1 * (double)(40 - kb) / 24.0;
        return e;
    };
    return eff(F16_NARROW_N) > 1.02 * eff(TILE_N) ? F16_NARROW_N : TILE_N;
}

// The column width of an e4m3 CTA-pair tile: 256 (one accumulator, drained to registers
// before the next tile starts) or 224 (two accumulators, the next tile accumulating while the
// epilogue drains).  Estimated efficiency = used share of the tile columns x busy share of the
// rounds (0.89 where stream-K balances them) x, for 256, the tile boundary it waits at (~3.8
// k-blocks' time per tile after the first of a unit) or, for 224, the 7 % more operand bytes
// per FLOP; 224 must win by 5 %.  Measured (one GPU call, 200 runs): 4096^3 224 +16 %,
// 4096 x 4096 x 8192 +6 %; 8192^3 -3 %, 6144^3 -2 %, 3072 x 3072 x 8192 -3 %: the rule
// takes 224 for the first two only.
int e4m3_pair_tile_n(int64_t M, int64_t N, int64_t K, bool f32, int units) {
    const int64_t tiles_m = (M + 2 * TILE_M - 1) / (2 * TILE_M), kb = (K + 127) / 128;
    auto eff = [&](int bn) {
        const int64_t tn = (N + bn - 1) / bn, tiles = tiles_m * tn;
        const int64_t rounds = (tiles + units - 1) / units;
        const bool sk = f32 && kb >= GB300_SK_MIN_KB && tiles >= units && tiles % units != 0 && tiles < 4 * units;
        double e = (double)N / (double)(tn * bn);
        e *= sk ? 0.89 : (double)tiles / (double)(rounds * units);
        if (bn == MXF8_NARROW_N) e *= 0.93;
        else e *= 1.0 - 3.8 / (double)kb * (1.0 - 1.0 / (double)rounds);
        return e;
    };
    return eff(MXF8_NARROW_N) > 1.05 * eff(TILE_N) ? MXF8_NARROW_N : TILE_N;
}

gemm_status configure_f16(gemm_plan *p) {
    int cg = (p->M >= 1024 && p->N >= 1024) ? 2 : 1;
    if (p->flags & GEMM_FLAG_FORCE_1CTA) cg = 1;
    if (p->flags & GEMM_FLAG_FORCE_2CTA) cg = 2;
    F16Config cfg{cg, p->d == GEMM_BF16};
    if (f16_prepare(cfg) != cudaSuccess) return GEMM_ERR_CUDA;
    int units = p->sm_count / cg;
    if (cg == 2) {
        int clusters = 0;
        if (f16_max_active_clusters(cfg, &clusters) == cudaSuccess && clusters > 0) units = clusters;
    }
    p->tiles_m = (int)((p->M + TILE_M * cg - 1) / (TILE_M * cg));
    // pairs: 256 x 224 tiles where they fill the persistent rounds clearly better (pair_tile_n);
    // an N-contiguous B needs whole 64-element atoms per CTA (112 rows are not): it keeps 256
    if (cg == 2 && !p->b_mn) {
        if (pair_tile_n(p->M, p->N, p->K, p->d == GEMM_F32, units) == F16_NARROW_N) {
            cfg.tile_n = F16_NARROW_N;
            if (f16_prepare(cfg) != cudaSuccess) return GEMM_ERR_CUDA;
            int clusters = 0;
            if (f16_max_active_clusters(cfg, &clusters) == cudaSuccess && clusters > 0) units = clusters;
        }
    }
    p->cta_group = cg;
    p->stages = f16_stages(cfg);
    p->smem = f16_smem_bytes(cfg);
    p->tile_n = cfg.tile_n;
    p->epi_box = EPI_COLS;
    p->tile_k = TILE_K16;
    p->num_kb = (int)((p->K + TILE_K16 - 1) / TILE_K16);
    p->tiles_n = (int)((p->N + p->tile_n - 1) / p->tile_n);
    p->tiles = p->tiles_m * p->tiles_n;
    p->capacity = units;
    p->grid = cg * (p->tiles < units ? p->tiles : units);
    p->group_m = cg == 2 ? GB300_GROUP_M_PAIRS : GB300_GROUP_M_SINGLE;
    return GEMM_OK;
}

gemm_status configure_scaled(gemm_plan *p) {
    const ScaledFamily &fam = scaled_family(p->family);
    int cg = (p->M >= 1024 && p->N >= 1024) ? 2 : 1;
    if (p->flags & GEMM_FLAG_FORCE_1CTA) cg = 1;
    if (p->flags & GEMM_FLAG_FORCE_2CTA) cg = 2;
    // single-CTA e4m3 tiles hold 224 rows of B, not a whole number of 128-element atoms:
    // an N-contiguous B needs CTA pairs (128 rows each)
    if (p->b_mn && cg == 1) {
        if (p->flags & GEMM_FLAG_FORCE_1CTA) return GEMM_ERR_UNSUPPORTED;
        cg = 2;
    }
    const int bf = p->d == GEMM_BF16;
    // e4m3 pairs: the narrow form where it fills the rounds clearly better (an N-contiguous B
    // needs whole 128-element atoms per CTA, which its 112 rows are not)
    p->narrow = false;
    if (cg == 2 && fam.has_narrow && !p->b_mn) {
        int units = p->sm_count / 2, clusters = 0;
        if (fam.prepare(cg, bf, false) == cudaSuccess && fam.max_active_clusters(cg, bf, false, &clusters) == cudaSuccess &&
            clusters > 0)
            units = clusters;
        p->narrow = e4m3_pair_tile_n(p->M, p->N, p->K, p->d == GEMM_F32, units) == MXF8_NARROW_N;
    }
    if (fam.prepare(cg, bf, p->narrow) != cudaSuccess) return GEMM_ERR_CUDA;
    const ScaledShape sh = fam.shape(cg, p->narrow);
    p->cta_group = cg;
    p->tile_n = sh.tile_n;
    p->epi_box = sh.epi_box;
    p->stages = sh.stages;
    p->smem = sh.smem;
    p->tile_k = sh.bk;
    p->sfa_stage_bytes = sh.sfa_bytes;
    p->sfb_stage_bytes = sh.sfb_bytes;
    p->num_kb = (int)((p->K + sh.bk - 1) / sh.bk);
    p->tiles_m = (int)((p->M + TILE_M * cg - 1) / (TILE_M * cg));
    p->tiles_n = (int)((p->N + p->tile_n - 1) / p->tile_n);
    p->tiles = p->tiles_m * p->tiles_n;
    int units = p->sm_count / cg;
    if (cg == 2) {
        int clusters = 0;
        if (fam.max_active_clusters(cg, bf, p->narrow, &clusters) == cudaSuccess && clusters > 0) units = clusters;
    }
    p->capacity = units;
    p->grid = cg * (p->tiles < units ? p->tiles : units);
    p->group_m = cg == 2 ? GB300_GROUP_M_PAIRS : GB300_GROUP_M_SINGLE;
    // workspace: the packed SFA of every (128 rows, stage), the packed SFB of every (tile column, stage)
    const int row_blocks = p->tiles_m * cg;
    const size_t a_bytes = (size_t)row_blocks * p->num_kb * sh.sfa_bytes;
    const size_t b_bytes = (size_t)p->tiles_n * p->num_kb * sh.sfb_bytes;
    if (cudaMalloc(&p->ws_a, a_bytes) != cudaSuccess || cudaMalloc(&p->ws_b, b_bytes) != cudaSuccess) {
        cudaFree(p->ws_a);
        cudaFree(p->ws_b);
        p->ws_a = p->ws_b = nullptr;
        return GEMM_ERR_CUDA;
    }
    if (!encoder()) return GEMM_ERR_CUDA;
    if (!encode_2d(&p->maps[4], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p->ws_a, 128, a_bytes / 128, 128,
                   (uint32_t)(sh.sfa_bytes / 128), CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&p->maps[5], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p->ws_b, 128, b_bytes / 128, 128,
                   (uint32_t)(sh.sfb_bytes / 128), CU_TENSOR_MAP_SWIZZLE_NONE))
        return GEMM_ERR_CUDA;
    return GEMM_OK;
}

// Split-K: when the output tiles cannot fill the GPU, cut each tile's K range into
// slices that run as separate work units and add their partial products into D
// (fp32 only: rounding every partial sum to bf16 would cost accuracy).
// Stream-K: when there are more tiles than units but not a whole number of waves, the
// last one to two waves' worth of tiles is shared out as equal spans of k-blocks, so
// that every unit finishes at about the same time (deterministic: every tile is summed
// in a fixed order).
gemm_status choose_splits(gemm_plan *p) {
    const int units = p->capacity;
    int s = 1;
    if (p->split_request >= 1) {
        s = p->split_request;
    } else if (p->d == GEMM_F32 && 2 * p->tiles <= units && p->num_kb >= 8) {
        s = units / p->tiles;
        if (s > p->num_kb / 4) s = p->num_kb / 4;
        if (s > 16) s = 16;
    }
    if (s > p->num_kb) s = p->num_kb;
    if (s < 1 || p->d != GEMM_F32 || (p->flags & GEMM_FLAG_DETERMINISTIC)) s = 1;
    p->splits = s;
    // more work units than tiles: the persistent grid may grow up to the machine
    const int work = p->tiles * s;
    p->grid = p->cta_group * (work < units ? work : units);
    // fp32 D only (the partial sums meet in D itself), and as measured on GB300 only with
    // long tiles (>= 64 k-blocks: the cut pieces' extra epilogue work stays small) and few
    // waves (below 4 the idle part of the last wave is a large share; above, the power the
    // idle SMs leave lets the busy ones clock higher)
    p->sk = s == 1 && p->sk_request && p->d == GEMM_F32 && p->tiles >= units && p->tiles % units != 0 &&
            p->num_kb >= GB300_SK_MIN_KB && p->tiles < 4 * units;
    if (p->sk) {
        p->sk_dp_tiles = (p->tiles / units - 1) * units;
        p->grid = p->cta_group * units;
        if (!p->sk_flags) {
            const size_t fl = (size_t)units * p->cta_group * sizeof(int);
            if (cudaMalloc(&p->sk_flags, fl) != cudaSuccess || cudaMemset(p->sk_flags, 0, fl) != cudaSuccess) {
                cudaFree(p->sk_flags);
                p->sk_flags = nullptr;
                p->sk = 0;
                return GEMM_ERR_CUDA;
            }
        }
    }
    // whole-tile fp16/bf16 pairs with fp32 D and short K: the tile's C-in/D-out epilogue
    // outlasts the next tile's main loop, so twice the epilogue warps (one stage fewer)
    // pay; with bf16 D or longer K they lose (measured on GB300).  Single CTAs that take at
    // most one short tile each: the run is mostly that tile's epilogue, which 8 warps
    // halve (either D type)
    if (p->family == KIND_F16) {
        F16Config cfg{p->cta_group, p->d == GEMM_BF16, 0, p->tile_n};
        cfg.wide_epi = (p->cta_group == 2 && p->tile_n == TILE_N && p->d == GEMM_F32 && s == 1 && !p->sk &&
                        p->num_kb <= 40) ||
                       (p->cta_group == 1 && s == 1 && !p->sk && p->tiles <= units && p->num_kb <= 40);
        if (cfg.wide_epi && f16_prepare(cfg) != cudaSuccess) return GEMM_ERR_CUDA;
        p->wide_epi = cfg.wide_epi;
        p->stages = f16_stages(cfg);
        p->smem = f16_smem_bytes(cfg);
    }
    return GEMM_OK;
}

// Chain plans: stream-K over the first product (on request only: gemm_plan_set_stream_k)
// when the tiles make more than one wave but not a whole number of them (fewer than 4) and
// K is long enough that a handed-over partial T (n1p fp32 columns of 128 rows per CTA) is
// small next to the work it balances.  Measured on 32768 x 4096, N1 = N2 = 256 (pairs, 128
// tiles on 76 units) and 20480 x 1024: 8-10 % slower than whole tiles, so it is off by default.
#ifndef GB300_CHAIN_SK_MIN_KB
#define GB300_CHAIN_SK_MIN_KB 16
#endif
gemm_status choose_chain_schedule(gemm_plan *p) {
    const int units = p->grid / p->cta_group;
    p->sk = p->sk_request && p->tiles > units && p->tiles % units != 0 && p->tiles < 4 * units &&
            p->num_kb >= GB300_CHAIN_SK_MIN_KB;
    if (!p->sk) return GEMM_OK;
    p->sk_dp_tiles = (p->tiles / units - 1) * units;
    if (!p->sk_flags) {
        const size_t row = (size_t)((p->N + 31) / 32 * 32);     // whole 32-column chunks of T
        const size_t fl = (size_t)units * p->cta_group * sizeof(int);
        const size_t pt = (size_t)units * p->cta_group * TILE_M * row * sizeof(float);
        if (cudaMalloc(&p->sk_flags, fl) != cudaSuccess || cudaMemset(p->sk_flags, 0, fl) != cudaSuccess ||
            cudaMalloc(&p->sk_part, pt) != cudaSuccess) {
            cudaFree(p->sk_flags);
            cudaFree(p->sk_part);
            p->sk_flags = nullptr;
            p->sk_part = nullptr;
            p->sk = 0;
            return GEMM_ERR_CUDA;
        }
    }
    return GEMM_OK;
}

}  // namespace

extern "C" {

const char *gemm_status_string(gemm_status s) {
    switch (s) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_UNSUPPORTED: return "unsupported dtype, layout or device";
    case GEMM_ERR_ALIGNMENT: return "pointer or row stride not a multiple of 16 bytes";
    case GEMM_ERR_CUDA: return "CUDA call failed";
    case GEMM_ERR_TIMEOUT: return "a bounded wait inside the kernel ran out";
    case GEMM_ERR_CHECK: return "an on-device check of a copy coordinate failed";
    default: return "unknown status";
    }
}

gemm_status gemm_plan_create(gemm_plan_t *out, int64_t M, int64_t N, int64_t K, gemm_dtype ab, gemm_dtype c,
                             gemm_dtype d, int a_row_major, int b_row_major, int block_scaled, unsigned flags) {
    if (!out || M <= 0 || N <= 0 || K <= 0) return GEMM_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_INVALID_ARG;
    if ((unsigned)ab > GEMM_E2M1 || (unsigned)c > GEMM_E2M1 || (unsigned)d > GEMM_E2M1) return GEMM_ERR_INVALID_ARG;
    if (block_scaled < GEMM_SCALE_NONE || block_scaled > GEMM_SCALE_UE4M3_16) return GEMM_ERR_INVALID_ARG;
    if ((flags & GEMM_FLAG_FORCE_1CTA) && (flags & GEMM_FLAG_FORCE_2CTA)) return GEMM_ERR_INVALID_ARG;
    if (c != GEMM_F32 || (d != GEMM_F32 && d != GEMM_BF16)) return GEMM_ERR_UNSUPPORTED;
    // operand type and scale mode: fp16/bf16 unscaled, e4m3 with UE8M0 / 32, e2m1 with
    // UE8M0 / 32 or UE4M3 / 16
    int family;
    if ((ab == GEMM_F16 || ab == GEMM_BF16) && block_scaled == GEMM_SCALE_NONE)
        family = KIND_F16;
    else if (ab == GEMM_E4M3 && block_scaled == GEMM_SCALE_UE8M0_32)
        family = KIND_MXF8;
    else if (ab == GEMM_E2M1 && block_scaled == GEMM_SCALE_UE8M0_32)
        family = KIND_MXF4;
    else if (ab == GEMM_E2M1 && block_scaled == GEMM_SCALE_UE4M3_16)
        family = KIND_NVF4;
    else
        return GEMM_ERR_UNSUPPORTED;
    // 4-bit operands: K-major only (the tensor core reads packed 4-bit data K-major)
    if (ab == GEMM_E2M1 && (!a_row_major || b_row_major)) return GEMM_ERR_UNSUPPORTED;

    // 16-byte row strides (the copy engine's stride rule): A rows hold K (row-major) or M
    // (column-major) elements, B rows K (column-major) or N (row-major), C and D rows N
    const int64_t a_row = a_row_major ? K : M, b_row = b_row_major ? N : K;
    if ((a_row * elem_bits(ab)) % 128 != 0 || (b_row * elem_bits(ab)) % 128 != 0 || (N * 32) % 128 != 0 ||
        (N * elem_bits(d)) % 128 != 0)
        return GEMM_ERR_ALIGNMENT;

    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return GEMM_ERR_UNSUPPORTED;

    gemm_plan *p = new (std::nothrow) gemm_plan();
    if (!p) return GEMM_ERR_CUDA;
    p->M = M;
    p->N = N;
    p->K = K;
    p->ab = ab;
    p->c = c;
    p->d = d;
    p->block_scaled = block_scaled;
    p->family = family;
    p->a_mn = !a_row_major;
    p->b_mn = b_row_major != 0;
    p->flags = flags;
    p->device = dev;
    p->sm_count = prop.multiProcessorCount;
    p->timeout_ns = 1000000000ull;
    gemm_status st = family == KIND_F16 ? configure_f16(p) : configure_scaled(p);
    if (st != GEMM_OK) {
        cudaFree(p->ws_a);
        cudaFree(p->ws_b);
        delete p;
        return st;
    }
    p->sk_request = 1;
    if (choose_splits(p) != GEMM_OK || cudaMalloc(&p->status, sizeof(int)) != cudaSuccess) {
        cudaFree(p->ws_a);
        cudaFree(p->ws_b);
        cudaFree(p->sk_flags);
        delete p;
        return GEMM_ERR_CUDA;
    }
    if (cudaMemset(p->status, 0, sizeof(int)) != cudaSuccess) {
        cudaFree(p->status);
        delete p;
        return GEMM_ERR_CUDA;
    }
    *out = p;
    return GEMM_OK;
}

gemm_status gemm_run(gemm_plan_t p, const void *A, const void *B, const void *C, void *D, const uint8_t *SFA,
                     const uint8_t *SFB, void *cuda_stream) {
    if (!p || !A || !B || !D || p->family == FAMILY_CHAIN) return GEMM_ERR_INVALID_ARG;
    if (p->family != KIND_F16 && (!SFA || !SFB)) return GEMM_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (C && !aligned16(C))) return GEMM_ERR_ALIGNMENT;
    gemm_status st = encode_maps(p, A, B, C, D);
    if (st != GEMM_OK) return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(cuda_stream);
    KParams kp{};
    kp.M = (int)p->M;
    kp.N = (int)p->N;
    kp.K = (int)p->K;
    kp.tiles_m = p->tiles_m;
    kp.tiles_n = p->tiles_n;
    kp.num_tiles = p->tiles;
    kp.num_kb = p->num_kb;
    kp.group_m = p->group_m;
    kp.has_c = C != nullptr;
    kp.a_mn = p->a_mn;
    kp.b_mn = p->b_mn;
    kp.splits = p->splits;
    if (p->splits > 1) {
        // D starts as C (or 0); every K slice then adds its partial product into it
        if (init_d_launch(static_cast<float *>(D), static_cast<const float *>(C), (size_t)p->M * p->N, p->sm_count,
                          stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
        kp.has_c = 0;
    }
    kp.status = p->status;
    kp.timeout_ns = p->timeout_ns;
    kp.fault = p->fault;
    kp.clk_meter = p->clk_meter_on ? p->clk_meter : nullptr;
    kp.trace = p->trace;
    if (p->sk) {
        kp.sk = 1;
        kp.sk_dp_tiles = p->sk_dp_tiles;
        kp.sk_units = p->grid / p->cta_group;
        kp.epoch = (int)(++p->epoch & 0x7FFFFFFF);
        if (kp.epoch == 0) kp.epoch = p->epoch = 1;
        kp.sk_flags = p->sk_flags;
    }
    LaunchShape shape{p->grid, p->cta_group, p->smem};
    if (p->family != KIND_F16) {
        const uint32_t tm = (uint32_t)(TILE_M * p->cta_group), tn = (uint32_t)p->tile_n;
        kp.idesc = p->family == KIND_MXF8
                       ? idesc_mxf8(tm, tn, 0, 0) | ((uint32_t)p->a_mn << 15) | ((uint32_t)p->b_mn << 16)
                       : idesc_mxf4(tm, tn, p->family == KIND_NVF4);
        kp.sfa = p->ws_a;
        kp.sfb = p->ws_b;
        const int sfk = (int)((p->K + scale_block(p->family) - 1) / scale_block(p->family));
        const int n_wg = p->num_kb * (p->sfa_stage_bytes / 512);
        if (sf_pack(SFA, SFB, p->ws_a, p->ws_b, kp.M, kp.N, sfk, p->tiles_m * p->cta_group, p->tiles_n, p->tile_n,
                    n_wg, unit_scale(p->family), stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (scaled_family(p->family).launch(p->cta_group, p->d == GEMM_BF16, p->narrow, shape, p->maps, kp, stream) !=
            cudaSuccess)
            return GEMM_ERR_CUDA;
    } else {
        kp.idesc = idesc_f16(p->ab == GEMM_BF16 ? 1u : 0u, (uint32_t)(TILE_M * p->cta_group), (uint32_t)p->tile_n) |
                   ((uint32_t)p->a_mn << 15) | ((uint32_t)p->b_mn << 16);
        F16Config cfg{p->cta_group, p->d == GEMM_BF16, p->wide_epi, p->tile_n};
        if (f16_launch(cfg, shape, p->maps, kp, stream) != cudaSuccess) return GEMM_ERR_CUDA;
    }
    if (p->flags & GEMM_FLAG_SYNC) {
        if (cudaStreamSynchronize(stream) != cudaSuccess) return GEMM_ERR_CUDA;
        return gemm_plan_last_status(p);
    }
    return GEMM_OK;
}

namespace {

gemm_status pipe_setup(gemm_plan *p) {
    if (p->pipe_ready) return GEMM_OK;
    bool ok = cudaStreamCreateWithFlags(&p->pipe_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->pipe_comp, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->pipe_out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p->pipe_entry, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < HOST_CHUNKS; ++i)
        ok = cudaEventCreateWithFlags(&p->pipe_in_done[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->pipe_k_done[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return GEMM_ERR_CUDA;
    p->pipe_ready = true;
    return GEMM_OK;
}

void pipe_destroy(gemm_plan *p) {
    if (!p->pipe_ready) return;
    cudaStreamDestroy(p->pipe_in);
    cudaStreamDestroy(p->pipe_comp);
    cudaStreamDestroy(p->pipe_out);
    cudaEventDestroy(p->pipe_entry);
    for (int i = 0; i < HOST_CHUNKS; ++i) {
        cudaEventDestroy(p->pipe_in_done[i]);
        cudaEventDestroy(p->pipe_k_done[i]);
    }
}

// The plan's kernel on rows [0, rows) of device operands A, C, D (and, block-scaled, the
// same rows of SFA with all of SFB): whole tiles, no split-K or stream-K
gemm_status launch_rows(gemm_plan *p, const void *A, const void *B, const void *C, void *D, const uint8_t *SFA,
                        const uint8_t *SFB, int64_t rows, cudaStream_t stream) {
    CUtensorMap maps[NUM_MAPS];
    std::memset(maps, 0, sizeof maps);
    if (!encode_operand_maps(p, maps, A, B, C, D, rows)) return GEMM_ERR_CUDA;
    maps[4] = p->maps[4];                 // packed-scale workspaces (block-scaled plans)
    maps[5] = p->maps[5];
    const int cg = p->cta_group;
    KParams kp{};
    kp.M = (int)rows;
    kp.N = (int)p->N;
    kp.K = (int)p->K;
    kp.tiles_m = (int)((rows + TILE_M * cg - 1) / (TILE_M * cg));
    kp.tiles_n = p->tiles_n;
    kp.num_tiles = kp.tiles_m * kp.tiles_n;
    kp.num_kb = p->num_kb;
    kp.group_m = p->group_m;
    kp.has_c = C != nullptr;
    kp.a_mn = p->a_mn;
    kp.b_mn = p->b_mn;
    kp.splits = 1;
    kp.status = p->status;
    kp.timeout_ns = p->timeout_ns;
    kp.fault = p->fault;
    kp.clk_meter = p->clk_meter_on ? p->clk_meter : nullptr;
    const int units = kp.num_tiles < p->capacity ? kp.num_tiles : p->capacity;
    LaunchShape shape{cg * units, cg, p->smem};
    if (p->family != KIND_F16) {
        const uint32_t tm = (uint32_t)(TILE_M * cg), tn = (uint32_t)p->tile_n;
        kp.idesc = p->family == KIND_MXF8 ? idesc_mxf8(tm, tn, 0, 0) | ((uint32_t)p->b_mn << 16)
                                          : idesc_mxf4(tm, tn, p->family == KIND_NVF4);
        kp.sfa = p->ws_a;
        kp.sfb = p->ws_b;
        const int sfk = (int)((p->K + scale_block(p->family) - 1) / scale_block(p->family));
        const int n_wg = p->num_kb * (p->sfa_stage_bytes / 512);
        if (sf_pack(SFA, SFB, p->ws_a, p->ws_b, kp.M, kp.N, sfk, kp.tiles_m * cg, p->tiles_n, p->tile_n, n_wg,
                    unit_scale(p->family), stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
        return scaled_family(p->family).launch(cg, p->d == GEMM_BF16, p->narrow, shape, maps, kp, stream) == cudaSuccess
                   ? GEMM_OK
                   : GEMM_ERR_CUDA;
    }
    kp.idesc = idesc_f16(p->ab == GEMM_BF16 ? 1u : 0u, (uint32_t)(TILE_M * cg), (uint32_t)p->tile_n) |
               ((uint32_t)p->b_mn << 16);
    F16Config cfg{cg, p->d == GEMM_BF16, p->wide_epi, p->tile_n};
    return f16_launch(cfg, shape, maps, kp, stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

// Host-buffer run as a pipeline over row chunks (row-major A, no split-K): B (and SFB)
// first, then each chunk's rows of A, C (and SFA) go up on one stream, its product runs on
// a second as soon as they have landed (block-scaled: after packing the chunk's scales), and
// its rows of D come back on a third, so that transfers in both directions and the kernels
// overlap.  The chunks' kernels share the scale workspaces in stream order.
gemm_status run_host_pipelined(gemm_plan *p, const void *A, const void *B, const void *C, void *D,
                               const uint8_t *SFA, const uint8_t *SFB, int64_t chunk, cudaStream_t stream) {
    if (pipe_setup(p) != GEMM_OK) return GEMM_ERR_CUDA;
    const size_t a_row = bytes_of(p->ab, p->K), c_row = (size_t)p->N * 4, d_row = bytes_of(p->d, p->N);
    const size_t b_bytes = bytes_of(p->ab, p->K * p->N);
    const char *hA = static_cast<const char *>(A), *hC = static_cast<const char *>(C);
    char *hD = static_cast<char *>(D);
    char *dA = static_cast<char *>(p->hA), *dC = static_cast<char *>(p->hC), *dD = static_cast<char *>(p->hD);
    // the pipeline starts after the work already queued on the caller's stream
    if (cudaEventRecord(p->pipe_entry, stream) != cudaSuccess ||
        cudaStreamWaitEvent(p->pipe_in, p->pipe_entry, 0) != cudaSuccess ||
        cudaStreamWaitEvent(p->pipe_comp, p->pipe_entry, 0) != cudaSuccess ||
        cudaStreamWaitEvent(p->pipe_out, p->pipe_entry, 0) != cudaSuccess ||
        cudaMemcpyAsync(p->hB, B, b_bytes, cudaMemcpyHostToDevice, p->pipe_in) != cudaSuccess)
        return GEMM_ERR_CUDA;
    const bool scaled = p->family != KIND_F16;
    const size_t sfk = scaled ? (size_t)((p->K + scale_block(p->family) - 1) / scale_block(p->family)) : 0;
    uint8_t *dSFA = static_cast<uint8_t *>(p->hSFA);
    if (scaled && cudaMemcpyAsync(p->hSFB, SFB, (size_t)p->N * sfk, cudaMemcpyHostToDevice, p->pipe_in) != cudaSuccess)
        return GEMM_ERR_CUDA;
    int i = 0;
    for (int64_t r0 = 0; r0 < p->M; r0 += chunk, ++i) {
        const int64_t rows = p->M - r0 < chunk ? p->M - r0 : chunk;
        if (cudaMemcpyAsync(dA + r0 * a_row, hA + r0 * a_row, rows * a_row, cudaMemcpyHostToDevice, p->pipe_in) !=
                cudaSuccess ||
            (C && cudaMemcpyAsync(dC + r0 * c_row, hC + r0 * c_row, rows * c_row, cudaMemcpyHostToDevice,
                                  p->pipe_in) != cudaSuccess) ||
            (scaled && cudaMemcpyAsync(dSFA + r0 * sfk, SFA + r0 * sfk, rows * sfk, cudaMemcpyHostToDevice,
                                       p->pipe_in) != cudaSuccess) ||
            cudaEventRecord(p->pipe_in_done[i], p->pipe_in) != cudaSuccess ||
            cudaStreamWaitEvent(p->pipe_comp, p->pipe_in_done[i], 0) != cudaSuccess)
            return GEMM_ERR_CUDA;
        const gemm_status st =
            launch_rows(p, dA + r0 * a_row, p->hB, C ? dC + r0 * c_row : nullptr, dD + r0 * d_row,
                        scaled ? dSFA + r0 * sfk : nullptr, static_cast<const uint8_t *>(p->hSFB), rows, p->pipe_comp);
        if (st != GEMM_OK) return st;
        if (cudaEventRecord(p->pipe_k_done[i], p->pipe_comp) != cudaSuccess ||
            cudaStreamWaitEvent(p->pipe_out, p->pipe_k_done[i], 0) != cudaSuccess ||
            cudaMemcpyAsync(hD + r0 * d_row, dD + r0 * d_row, rows * d_row, cudaMemcpyDeviceToHost, p->pipe_out) !=
                cudaSuccess)
            return GEMM_ERR_CUDA;
    }
    // D's last rows are home once the copy-out stream drains (it waited for every kernel)
    if (cudaStreamSynchronize(p->pipe_out) != cudaSuccess) return GEMM_ERR_CUDA;
    return gemm_plan_last_status(p);
}

}  // namespace

gemm_status gemm_run_host(gemm_plan_t p, const void *A, const void *B, const void *C, void *D, const uint8_t *SFA,
                          const uint8_t *SFB, void *cuda_stream) {
    if (!p || !A || !B || !D || p->family == FAMILY_CHAIN) return GEMM_ERR_INVALID_ARG;
    const size_t a_bytes = bytes_of(p->ab, p->M * p->K);
    const size_t b_bytes = bytes_of(p->ab, p->K * p->N);
    const size_t c_bytes = (size_t)p->M * p->N * 4;
    const size_t d_bytes = bytes_of(p->d, p->M * p->N);
    if (!p->hA) {
        if (cudaMalloc(&p->hA, a_bytes) != cudaSuccess || cudaMalloc(&p->hB, b_bytes) != cudaSuccess ||
            cudaMalloc(&p->hC, c_bytes) != cudaSuccess || cudaMalloc(&p->hD, d_bytes) != cudaSuccess)
            return GEMM_ERR_CUDA;
    }
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(cuda_stream);
    const size_t sfk = p->family != KIND_F16 ? (size_t)((p->K + scale_block(p->family) - 1) / scale_block(p->family)) : 0;
    if (p->family != KIND_F16) {
        if (!SFA || !SFB) return GEMM_ERR_INVALID_ARG;
        if (!p->hSFA && (cudaMalloc(&p->hSFA, (size_t)p->M * sfk) != cudaSuccess ||
                         cudaMalloc(&p->hSFB, (size_t)p->N * sfk) != cudaSuccess))
            return GEMM_ERR_CUDA;
    }
    // row-major A (contiguous row chunks), whole tiles, and room for two or more chunks of at
    // least HOST_MIN_ROWS rows: the pipelined form
    if (!p->a_mn && p->splits == 1) {
        const int64_t tile = (int64_t)TILE_M * p->cta_group;
        int64_t chunk = (p->M + HOST_CHUNKS - 1) / HOST_CHUNKS;
        chunk = (chunk + tile - 1) / tile * tile;
        if (chunk < HOST_MIN_ROWS) chunk = HOST_MIN_ROWS;
        if (p->M >= 2 * chunk) return run_host_pipelined(p, A, B, C, D, SFA, SFB, chunk, stream);
    }
    if (cudaMemcpyAsync(p->hA, A, a_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaMemcpyAsync(p->hB, B, b_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (C && cudaMemcpyAsync(p->hC, C, c_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) return GEMM_ERR_CUDA;
    if (p->family != KIND_F16) {
        if (cudaMemcpyAsync(p->hSFA, SFA, (size_t)p->M * sfk, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
            cudaMemcpyAsync(p->hSFB, SFB, (size_t)p->N * sfk, cudaMemcpyHostToDevice, stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
    }
    const unsigned saved = p->flags;
    p->flags &= ~GEMM_FLAG_SYNC;
    gemm_status st = gemm_run(p, p->hA, p->hB, C ? p->hC : nullptr, p->hD, p->hSFA, p->hSFB, cuda_stream);
    p->flags = saved;
    if (st != GEMM_OK) return st;
    if (cudaMemcpyAsync(D, p->hD, d_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return GEMM_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GEMM_ERR_CUDA;
    return gemm_plan_last_status(p);
}

gemm_status gemm_plan_last_status(gemm_plan_t p) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p->status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_CUDA;
    if (v != 0 && cudaMemset(p->status, 0, sizeof(int)) != cudaSuccess) return GEMM_ERR_CUDA;
    return (gemm_status)v;
}

gemm_status gemm_plan_get_info(gemm_plan_t p, gemm_plan_info *info) {
    if (!p || !info) return GEMM_ERR_INVALID_ARG;
    info->cta_group = p->cta_group;
    info->tile_m = TILE_M * p->cta_group;
    info->tile_n = p->tile_n;
    info->tile_k = p->tile_k;
    info->stages = p->stages;
    info->grid = p->grid;
    info->tiles = p->tiles;
    info->smem_bytes = p->smem;
    // block-scaled plans also launch the scale-packing kernel, split-K plans the D = C kernel
    const bool scaled = p->family != KIND_F16 && p->family != FAMILY_CHAIN;
    info->launches_per_run = (scaled ? 2 : 1) + (p->splits > 1 ? 1 : 0);
    info->splits = p->splits;
    info->stream_k = p->sk;
    info->sm_count = p->sm_count;
    return GEMM_OK;
}

gemm_status gemm_plan_set_timeout(gemm_plan_t p, uint64_t ns) {
    if (!p || ns == 0) return GEMM_ERR_INVALID_ARG;
    p->timeout_ns = ns;
    return GEMM_OK;
}

gemm_status gemm_plan_set_split_k(gemm_plan_t p, int splits) {
    if (!p || splits < 0) return GEMM_ERR_INVALID_ARG;
    if (p->family == FAMILY_CHAIN) return splits > 1 ? GEMM_ERR_UNSUPPORTED : GEMM_OK;
    if (splits > 1 && (p->d != GEMM_F32 || (p->flags & GEMM_FLAG_DETERMINISTIC))) return GEMM_ERR_UNSUPPORTED;
    p->split_request = splits;
    return choose_splits(p);
}

gemm_status gemm_plan_set_stream_k(gemm_plan_t p, int enable) {
    if (!p || enable < 0 || enable > 1) return GEMM_ERR_INVALID_ARG;
    p->sk_request = enable;
    if (p->family == FAMILY_CHAIN) return choose_chain_schedule(p);
    return choose_splits(p);
}

gemm_status gemm_plan_destroy(gemm_plan_t p) {
    if (!p) return GEMM_OK;
    cudaFree(p->status);
    cudaFree(p->hA);
    cudaFree(p->hB);
    cudaFree(p->hC);
    cudaFree(p->hD);
    cudaFree(p->hSFA);
    cudaFree(p->hSFB);
    cudaFree(p->hE);
    pipe_destroy(p);
    cudaFree(p->ws_a);
    cudaFree(p->ws_b);
    cudaFree(p->sk_flags);
    cudaFree(p->sk_part);
    cudaFree(p->clk_meter);
    delete p;
    return GEMM_OK;
}

// ------------------------------------------------------------ two-product chain

gemm_status gemm_chain_plan_create(gemm_plan_t *out, int64_t M, int64_t N1, int64_t N2, int64_t K, gemm_dtype ab,
                                   gemm_dtype d, unsigned flags) {
    if (!out || M <= 0 || N1 <= 0 || N2 <= 0 || K <= 0) return GEMM_ERR_INVALID_ARG;
    if (M > INT32_MAX || K > INT32_MAX) return GEMM_ERR_INVALID_ARG;
    if ((unsigned)ab > GEMM_E2M1 || (unsigned)d > GEMM_E2M1) return GEMM_ERR_INVALID_ARG;
    if ((flags & GEMM_FLAG_FORCE_1CTA) && (flags & GEMM_FLAG_FORCE_2CTA)) return GEMM_ERR_INVALID_ARG;
    if ((ab != GEMM_F16 && ab != GEMM_BF16) || (d != GEMM_F32 && d != GEMM_BF16)) return GEMM_ERR_UNSUPPORTED;
    // both products' accumulators share the 512 tensor-memory columns of one SM
    if (N1 > CHAIN_MAX_N || N2 > CHAIN_MAX_N) return GEMM_ERR_UNSUPPORTED;
    // 16-byte rows: A and B hold K elements, E N1, C N2 fp32, D N2
    if ((K * 2) % 16 != 0 || (N1 * 2) % 16 != 0 || (N2 * 4) % 16 != 0 || (N2 * elem_bits(d) / 8) % 16 != 0)
        return GEMM_ERR_ALIGNMENT;
    // CTA pairs (256-row tiles, each CTA taking in half of B's and E's rows) unless the rows fit
    // one CTA tile or an operand's padded N is not a multiple of 32 (the pair's MMA shapes are
    // kept to N = 32, 64, ..., 256)
    const int64_t n1p = (N1 + 15) / 16 * 16, n2p = (N2 + 15) / 16 * 16;
    const bool pair_ok = n1p % 32 == 0 && n2p % 32 == 0;
    if ((flags & GEMM_FLAG_FORCE_2CTA) && !pair_ok) return GEMM_ERR_UNSUPPORTED;

    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return GEMM_ERR_UNSUPPORTED;
    const int cg = (flags & GEMM_FLAG_FORCE_2CTA) || (!(flags & GEMM_FLAG_FORCE_1CTA) && pair_ok && M > TILE_M) ? 2 : 1;
    if (chain_prepare(d == GEMM_BF16, cg) != cudaSuccess) return GEMM_ERR_CUDA;
    int clusters = 0;
    if (chain_max_active_clusters(d == GEMM_BF16, cg, &clusters) != cudaSuccess || clusters <= 0)
        return GEMM_ERR_CUDA;

    gemm_plan *p = new (std::nothrow) gemm_plan();
    if (!p) return GEMM_ERR_CUDA;
    p->M = M;
    p->N = N1;
    p->N2 = N2;
    p->K = K;
    p->ab = ab;
    p->c = GEMM_F32;
    p->d = d;
    p->a_mn = p->b_mn = 0;
    p->flags = flags;
    p->device = dev;
    p->sm_count = prop.multiProcessorCount;
    p->timeout_ns = 1000000000ull;
    p->family = FAMILY_CHAIN;
    p->cta_group = cg;
    p->stages = chain_stages(cg);
    p->smem = chain_smem_bytes(cg);
    p->tile_n = (int)n2p;
    p->tile_k = TILE_K16;
    p->num_kb = (int)((K + TILE_K16 - 1) / TILE_K16);
    p->tiles_m = (int)((M + TILE_M * cg - 1) / (TILE_M * cg));
    p->tiles_n = 1;
    p->tiles = p->tiles_m;
    p->capacity = clusters;
    p->grid = cg * (p->tiles < clusters ? p->tiles : clusters);
    p->splits = 1;
    p->sk_request = 0;
    if (cudaMalloc(&p->status, sizeof(int)) != cudaSuccess) {
        delete p;
        return GEMM_ERR_CUDA;
    }
    if (cudaMemset(p->status, 0, sizeof(int)) != cudaSuccess || choose_chain_schedule(p) != GEMM_OK) {
        gemm_plan_destroy(p);
        return GEMM_ERR_CUDA;
    }
    *out = p;
    return GEMM_OK;
}

namespace {

gemm_status encode_chain_maps(gemm_plan *p, const void *A, const void *B, const void *E, const void *C, void *D) {
    if (p->maps_valid && A == p->lastA && B == p->lastB && E == p->lastE && C == p->lastC && D == p->lastD)
        return GEMM_OK;
    if (!encoder()) return GEMM_ERR_CUDA;
    std::memset(p->maps, 0, sizeof p->maps);
    const CUtensorMapDataType dt = tma_dtype(p->ab);
    // B and E boxes: the rows one CTA holds (all of them, or half in a CTA pair)
    const uint32_t n1p = (uint32_t)((p->N + 15) / 16 * 16), n2p = (uint32_t)p->tile_n, cg = (uint32_t)p->cta_group;
    bool ok = encode_2d(&p->maps[0], dt, 2, A, p->K, p->M, TILE_K16, TILE_M, CU_TENSOR_MAP_SWIZZLE_128B) &&
              encode_2d(&p->maps[1], dt, 2, B, p->K, p->N, TILE_K16, n1p / cg, CU_TENSOR_MAP_SWIZZLE_128B) &&
              encode_2d(&p->maps[4], dt, 2, E, p->N, p->N2, TILE_K16, n2p / cg, CU_TENSOR_MAP_SWIZZLE_128B);
    if (ok && C)
        ok = encode_2d(&p->maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, p->N2, p->M, EPI_COLS, 32,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (ok)
        ok = p->d == GEMM_BF16 ? encode_2d(&p->maps[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, p->N2, p->M, EPI_COLS,
                                           32, CU_TENSOR_MAP_SWIZZLE_64B)
                               : encode_2d(&p->maps[3], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, p->N2, p->M, EPI_COLS,
                                           32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) {
        p->maps_valid = false;
        return GEMM_ERR_CUDA;
    }
    p->lastA = A;
    p->lastB = B;
    p->lastE = E;
    p->lastC = C;
    p->lastD = D;
    p->maps_valid = true;
    return GEMM_OK;
}

}  // namespace

gemm_status gemm_chain_run(gemm_plan_t p, const void *A, const void *B, const void *E, const void *C, void *D,
                           void *cuda_stream) {
    if (!p || !A || !B || !E || !D || p->family != FAMILY_CHAIN) return GEMM_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(E) || !aligned16(D) || (C && !aligned16(C)))
        return GEMM_ERR_ALIGNMENT;
    gemm_status st = encode_chain_maps(p, A, B, E, C, D);
    if (st != GEMM_OK) return st;
    ChainParams cp{};
    cp.M = (int)p->M;
    cp.K = (int)p->K;
    cp.N1 = (int)p->N;
    cp.N2 = (int)p->N2;
    cp.n1p = (int)((p->N + 15) / 16 * 16);
    cp.n2p = p->tile_n;
    cp.num_kb1 = p->num_kb;
    cp.num_kb2 = (cp.n1p + TILE_K16 - 1) / TILE_K16;
    cp.tiles = p->tiles;
    cp.has_c = C != nullptr;
    cp.f16 = p->ab == GEMM_F16;
    const uint32_t bf = p->ab == GEMM_BF16 ? 1u : 0u;
    cp.idesc1 = idesc_f16(bf, (uint32_t)(TILE_M * p->cta_group), (uint32_t)cp.n1p);
    cp.idesc2 = idesc_f16(bf, (uint32_t)(TILE_M * p->cta_group), (uint32_t)cp.n2p);
    cp.status = p->status;
    cp.timeout_ns = p->timeout_ns;
    cp.fault = p->fault;
    if (p->sk) {
        cp.sk = 1;
        cp.sk_dp_tiles = p->sk_dp_tiles;
        cp.sk_units = p->grid / p->cta_group;
        cp.epoch = (int)(++p->epoch & 0x7FFFFFFF);
        if (cp.epoch == 0) cp.epoch = p->epoch = 1;
        cp.sk_flags = p->sk_flags;
        cp.sk_part = p->sk_part;
    }
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(cuda_stream);
    if (chain_launch(p->d == GEMM_BF16, p->cta_group, p->grid, p->maps, cp, stream) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (p->flags & GEMM_FLAG_SYNC) {
        if (cudaStreamSynchronize(stream) != cudaSuccess) return GEMM_ERR_CUDA;
        return gemm_plan_last_status(p);
    }
    return GEMM_OK;
}

gemm_status gemm_chain_run_host(gemm_plan_t p, const void *A, const void *B, const void *E, const void *C, void *D,
                                void *cuda_stream) {
    if (!p || !A || !B || !E || !D || p->family != FAMILY_CHAIN) return GEMM_ERR_INVALID_ARG;
    const size_t a_bytes = (size_t)p->M * p->K * 2, b_bytes = (size_t)p->K * p->N * 2,
                 e_bytes = (size_t)p->N * p->N2 * 2, c_bytes = (size_t)p->M * p->N2 * 4,
                 d_bytes = bytes_of(p->d, p->M * p->N2);
    if (!p->hA) {
        if (cudaMalloc(&p->hA, a_bytes) != cudaSuccess || cudaMalloc(&p->hB, b_bytes) != cudaSuccess ||
            cudaMalloc(&p->hE, e_bytes) != cudaSuccess || cudaMalloc(&p->hC, c_bytes) != cudaSuccess ||
            cudaMalloc(&p->hD, d_bytes) != cudaSuccess)
            return GEMM_ERR_CUDA;
    }
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(cuda_stream);
    if (cudaMemcpyAsync(p->hA, A, a_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaMemcpyAsync(p->hB, B, b_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaMemcpyAsync(p->hE, E, e_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (C && cudaMemcpyAsync(p->hC, C, c_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) return GEMM_ERR_CUDA;
    const unsigned saved = p->flags;
    p->flags &= ~GEMM_FLAG_SYNC;
    gemm_status st = gemm_chain_run(p, p->hA, p->hB, p->hE, C ? p->hC : nullptr, p->hD, cuda_stream);
    p->flags = saved;
    if (st != GEMM_OK) return st;
    if (cudaMemcpyAsync(D, p->hD, d_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return GEMM_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GEMM_ERR_CUDA;
    return gemm_plan_last_status(p);
}

// Test hook (declared in include/gb300gemm_testing.h): the pair tile-width rule alone.
gemm_status gemm_testing_pair_tile_n(int64_t M, int64_t N, int64_t K, gemm_dtype d, int units, int *tile_n) {
    if (!tile_n || M <= 0 || N <= 0 || K <= 0 || units <= 0 || (d != GEMM_F32 && d != GEMM_BF16))
        return GEMM_ERR_INVALID_ARG;
    *tile_n = pair_tile_n(M, N, K, d == GEMM_F32, units);
    return GEMM_OK;
}

// Test hook (declared in include/gb300gemm_testing.h): the e4m3 CTA-pair tile-width rule alone.
gemm_status gemm_testing_e4m3_pair_tile_n(int64_t M, int64_t N, int64_t K, gemm_dtype d, int units, int *tile_n) {
    if (!tile_n || M <= 0 || N <= 0 || K <= 0 || units <= 0 || (d != GEMM_F32 && d != GEMM_BF16))
        return GEMM_ERR_INVALID_ARG;
    *tile_n = e4m3_pair_tile_n(M, N, K, d == GEMM_F32, units);
    return GEMM_OK;
}

gemm_status gemm_plan_set_clock_meter(gemm_plan_t p, int enable) {
    if (!p || enable < 0 || enable > 1) return GEMM_ERR_INVALID_ARG;
    if (p->family == FAMILY_CHAIN) return GEMM_ERR_UNSUPPORTED;
    if (enable) {
        if (!p->clk_meter && cudaMalloc(&p->clk_meter, 2 * sizeof(unsigned long long)) != cudaSuccess) {
            p->clk_meter = nullptr;
            return GEMM_ERR_CUDA;
        }
        if (cudaMemset(p->clk_meter, 0, 2 * sizeof(unsigned long long)) != cudaSuccess) return GEMM_ERR_CUDA;
    }
    p->clk_meter_on = enable != 0;
    return GEMM_OK;
}

gemm_status gemm_plan_read_clock_meter(gemm_plan_t p, double *sm_mhz, double *cta_seconds) {
    if (!p || !sm_mhz || !cta_seconds) return GEMM_ERR_INVALID_ARG;
    *sm_mhz = 0.0;
    *cta_seconds = 0.0;
    if (!p->clk_meter) return GEMM_OK;
    unsigned long long v[2] = {0, 0};
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(v, p->clk_meter, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(p->clk_meter, 0, sizeof v) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (v[1] > 0) {
        *sm_mhz = (double)v[0] / (double)v[1] * 1e3;
        *cta_seconds = (double)v[1] * 1e-9;
    }
    return GEMM_OK;
}

// Test hook (declared in include/gb300gemm_testing.h): the per-role trace of a
// GB300_TRACE=1 build.
#ifndef GB300_TRACE
#define GB300_TRACE 0
#endif
int gemm_testing_trace_slots(void) { return GB300_TRACE ? (int)TRACE_SLOTS : 0; }

gemm_status gemm_testing_set_trace(gemm_plan_t p, void *dev_buffer, int64_t bytes) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    if (!GB300_TRACE || p->family == FAMILY_CHAIN) return GEMM_ERR_UNSUPPORTED;
    if (dev_buffer && bytes < (int64_t)p->grid * TRACE_SLOTS * (int64_t)sizeof(unsigned long long))
        return GEMM_ERR_INVALID_ARG;
    p->trace = static_cast<unsigned long long *>(dev_buffer);
    return GEMM_OK;
}

// Test hook (declared in include/gb300gemm_testing.h): make the next runs'
// producer withhold one arrival so that a bounded wait runs out (1), or shift its A
// rows past the tiled extent (2).
gemm_status gemm_testing_set_fault(gemm_plan_t p, int fault) {
    if (!p || fault < 0 || fault > 2 || (fault == 2 && p->family == FAMILY_CHAIN)) return GEMM_ERR_INVALID_ARG;
    p->fault = fault;
    return GEMM_OK;
}

}  // extern "C"
