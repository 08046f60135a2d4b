// Persistent, warp-specialised tensor-core GEMM for sm_103a (shared by the
// fp16/bf16 kernels and the block-scaled e4m3 and e2m1 kernels):
//   D = A·B + C, A (M x K) and B (K x N), fp32 accumulation in tensor
//   memory, C fp32, D fp32 or bf16.
//
// One CTA (cta_group::1) or one CTA pair (cta_group::2) owns a 128 x BN or
// 256 x BN output tile at a time and walks the tile list persistently.
// Warp roles (192 threads; 64 + 32 * EPI_WARPS + a copier warp in general):
//   warp 0      TMA producer: fills a STAGES-deep shared-memory ring of
//               A (128 rows) and B (BN/CG rows) boxes of 128-byte K rows,
//               128-byte swizzled, running STAGES k-blocks ahead of the MMA
//               ("(二) CUTLASS —— 掌握 Tensor Memory Accelerator（TMA）":
//               prefetch distance fetch_batch = compute_batch + num_stages;
//               one thread issues each copy, completion is an mbarrier
//               transaction count).  Block-scaled kernels also copy the
//               stage's packed scale factors (with COPIER, first and onto a
//               barrier of their own, sffull[s], so the copier can start early).
//   warp 1      allocates 512 TMEM columns (two BN-column fp32 accumulators,
//               plus scale-factor slots when block-scaled) and, in lane 0 of
//               the pair's leader CTA, issues tcgen05.mma from shared-memory
//               descriptors into TMEM ("Tensor Core 数据布局的演进",
//               Blackwell: A/B in SMEM --tcgen05.mma--> C/D in TMEM); for
//               block scaling it first moves the stage's scales SMEM -> TMEM
//               with tcgen05.cp (same page: SFA, SFB: GMEM --TMA--> SMEM
//               --tcgen05.cp--> TMEM --tcgen05.mma-->).
//   warps 2+EPI.. (block-scaled instances with COPIER, COPIERS warps) wait for the
//               stage's scales (sffull[s]), share the copies SMEM -> TMEM ahead of the
//               MMA issuer and commit their completion to the stage's full[s], which
//               then stands for operands and scales both (one wait per k-block for the
//               MMA issuer), so that copies and MMAs come from different threads and
//               overlap.
//   warps 2..5  epilogue warps (2..9 with EPI_WARPS = 8): warp w reads TMEM lanes 32*(w%4)..+31
//               ("Tensor Memory（TMEM）": each warp of a warpgroup reaches its
//               own 32-lane window) with tcgen05.ld + tcgen05.wait::ld, adds C
//               (TMA-loaded, 128-byte swizzled), converts, stages D in shared
//               memory and writes it with a TMA store (proxy fence before the
//               store, bulk-group wait before the buffer is reused).
// Every wait is bounded: when one runs out the kernel records
// GEMM_ERR_TIMEOUT, its roles stop, and it still frees its tensor memory.
#pragma once

#include <cstdint>
#include <type_traits>


#include "gemm_internal.h"
#include "ptx.cuh"

namespace gb300 {

// Compile-time shape of one kernel instance.
//   CG      1 = single CTA per tile, 2 = CTA pair (cta_group::2)
//   OUT_BF16  D is bf16 (else fp32)
//   KIND    operand kind (GemmKind): fp16/bf16, or block-scaled e4m3 (1X),
//           e2m1 with UE8M0 per 32 (2X) or e2m1 with UE4M3 per 16 (4X)
//   BN      tile columns (MMA N)
//   STAGES  depth of the shared-memory operand ring (k-blocks the producer runs ahead)
//   ACC_BUFS  TMEM accumulators: 2 = the epilogue drains one while the MMA fills
//             the other; 1 = the epilogue copies the accumulator to registers
//             and frees it before converting and storing (leaves TMEM columns
//             for scale slots at N = 256)
//   EPI_WARPS epilogue warps: 4 (one per TMEM lane window) or 8 (two per window,
//             each taking half of the tile's columns)
//   COPIER  block-scaled: a warp of its own issues the scale-factor copies (the
//           MMA thread then issues MMAs only)
//   EPI_BUFS  staging buffers per epilogue warp: 2 = the next box's C loads while this
//             box is stored; 1 = one box at a time (leaves shared memory for a stage)
//   EPI_BOX   columns of a C / D staging box (32 rows each): 32 (4 KiB of fp32, 128-byte
//             rows) or 16 (2 KiB, 64-byte rows: half the staging, room for a stage)
//   COPIERS   with COPIER: warps that share a stage's scale copies (1 or 2; each
//             tcgen05.cp costs its issuing thread ~70 clocks, so 12 copies per k-block
//             outlast the k-block's MMAs on one thread)
template <int CG_, bool OUT_BF16_, int KIND_, int BN_, int STAGES_, int ACC_BUFS_ = 2, int EPI_WARPS_ = 4,
          bool COPIER_ = false, int EPI_BUFS_ = 2, int EPI_BOX_ = 32, int COPIERS_ = 1>
struct TileCfg {
    static constexpr int CG = CG_;
    static constexpr bool OUT_BF16 = OUT_BF16_;
    static constexpr int KIND = KIND_;
    static constexpr bool SCALED = KIND != KIND_F16;
    static constexpr int BN = BN_;
    static constexpr int STAGES = STAGES_;
    static constexpr int ACC_BUFS = ACC_BUFS_;
    static constexpr int EPI_WARPS = EPI_WARPS_;
    static constexpr int EPI_BUFS = EPI_BUFS_;
    static_assert(EPI_BUFS == 1 || EPI_BUFS == 2, "epilogue staging buffers");
    static constexpr int EPI_BOX = EPI_BOX_;
    static_assert(EPI_BOX == 32 || EPI_BOX == 16, "epilogue box width");
    static constexpr int BOXES = EPI_COLS / EPI_BOX;            // boxes per 32-column TMEM chunk
    static constexpr bool COPIER = COPIER_ && KIND_ != KIND_F16;
    static constexpr int COPY_WARP = 2 + EPI_WARPS;             // the first copier warp
    static constexpr int COPIERS = COPIER ? COPIERS_ : 0;
    static_assert(COPIERS_ == 1 || COPIERS_ == 2, "copier warps");
    static constexpr int THREADS = 64 + 32 * EPI_WARPS + 32 * COPIERS;
    static constexpr int WCOLS = BN * 4 / EPI_WARPS;             // columns one epilogue warp handles
    static constexpr int WCHUNKS = WCOLS / EPI_COLS;
    static_assert(ACC_BUFS == 1 || ACC_BUFS == 2, "accumulator buffers");
    static_assert(EPI_WARPS == 4 || EPI_WARPS == 8, "epilogue warps");
    static_assert(WCOLS % EPI_COLS == 0, "epilogue columns per warp");
    static constexpr int ELEM_BITS = KIND == KIND_F16 ? 16 : (KIND == KIND_MXF8 ? 8 : 4);
    static constexpr int BK = 1024 / ELEM_BITS;                 // K elements per stage: one 128-byte row
    static constexpr int MMA_K = 256 / ELEM_BITS;               // K per instruction: 32 bytes
    // K extent of an operand box in tensor-map elements (4-bit operands are mapped as bytes)
    static constexpr int TMA_BK = ELEM_BITS == 4 ? 128 : BK;
    // MN-major operands (8- and 16-bit kinds): boxes one 128-byte swizzle atom wide along
    // M (or N) and BK rows of K
    static constexpr bool MN_OK = ELEM_BITS >= 8;
    static constexpr int ATOM_MN = 1024 / ELEM_BITS;            // M/N elements of one atom
    static constexpr int ATOM_BYTES = BK * 128;                 // one atom column of a stage
    static constexpr int A_BYTES = TILE_M * 128;                // 16 KiB
    static constexpr int B_ROWS = BN / CG;                      // B rows held by one CTA
    static constexpr int B_BYTES = B_ROWS * 128;
    // Block scales: SF_BLOCK K elements share a scale; a row's scales of one stage fill
    // SF_WORDS 32-bit words (four scales each); an MMA step reads SF_PER_MMA of them.
    static constexpr int SF_BLOCK = KIND == KIND_NVF4 ? 16 : 32;
    static constexpr int SF_WORDS = SCALED ? BK / SF_BLOCK / 4 : 0;
    static constexpr int SF_PER_MMA = MMA_K / SF_BLOCK;
    static constexpr int HALVES = (BN + 127) / 128;             // 128-column groups of the tile
    // scales of one stage in one CTA: SFA of its 128 rows, SFB of all BN columns of the
    // tile (each CTA of a pair computes every column of its rows); 512 bytes per word of
    // 128 rows, SFB words ordered (word, 128-column group)
    static constexpr int SFA_BYTES = 512 * SF_WORDS;
    static constexpr int SFB_BYTES = 512 * SF_WORDS * HALVES;
    static constexpr int TX_BYTES = CG * (A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES);
    // with a copier warp the scales land on a barrier of their own (sffull), ahead of A and B
    static constexpr int TX_AB = CG * (A_BYTES + B_BYTES);
    static constexpr int TX_SF = CG * (SFA_BYTES + SFB_BYTES);
    static constexpr int EPI_BUF = 32 * EPI_BOX * 4;            // one 32-row fp32 box
    // Every region a swizzled TMA copy or a swizzled MMA descriptor addresses
    // starts on a 1024-byte boundary: the 128-byte swizzle permutes 16-byte
    // chunks by address bits 7..9, so an offset of 512 would shift the row phase.
    static constexpr int align1k(int x) { return (x + 1023) / 1024 * 1024; }
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SF = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_EPI = align1k(OFF_SF + STAGES * (SFA_BYTES + SFB_BYTES));
    static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_BUFS * EPI_BUF;
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0 && OFF_B % 1024 == 0, "operand stages 1024-aligned");
    static_assert(OFF_EPI % 1024 == 0 && EPI_BUF % 1024 == 0, "epilogue staging 1024-aligned");
    // full[STAGES], empty[STAGES], tmem_full[2], tmem_empty[2], cload[EPI_WARPS][2], drain,
    // epi_sync, then with COPIER: cdrain, sffull[STAGES] (the stage's scales are in shared
    // memory).  With COPIER, full[s] also counts the copier warps' commits: the stage's
    // scales are in TMEM.
    static constexpr int NBAR = 2 * STAGES + 2 + 2 + 2 * EPI_WARPS + 2 + (COPIER ? STAGES + 1 : 0);
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;         // tmem base slot, abort flag
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;     // + alignment slack
    // TMEM columns: accumulators [0, ACC_BUFS*BN), then one scale slot per stage: SFA
    // in 4 columns per word, SFB in 4 columns per (word, 128 columns of the tile).  A
    // slot is reused only when its stage is refilled, i.e. after the MMAs that read it
    // have completed.
    static constexpr int SF_SLOT = 4 * SF_WORDS * (1 + HALVES);
    static constexpr int SF_COL0 = ACC_BUFS * BN;
    static_assert(ACC_BUFS * BN + STAGES * SF_SLOT <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared-memory budget");
    static_assert(BN % EPI_COLS == 0 && BN % 16 == 0 && BN <= 256, "tile N");
    static_assert(!SCALED || (SF_WORDS >= 1 && SF_PER_MMA >= 1 && 4 % SF_PER_MMA == 0), "scale vector");
};

// The work schedule below is plain integer code that also runs on the host, where a test
// hook (gemm_schedule.cu) enumerates it without a device.
#define GB300_HD __host__ __device__ __forceinline__

GB300_HD void tile_coords(int t, int tiles_m, int group_m, int &tm, int &tn, int tiles_n) {
    // groups of group_m M-tiles walk N together so that a wave of CTAs shares
    // A rows and B columns in L2
    const int per_group = group_m * tiles_n;
    const int g = t / per_group;
    const int first_m = g * group_m;
    const int gsize = tiles_m - first_m < group_m ? tiles_m - first_m : group_m;
    const int r = t - g * per_group;
    tm = first_m + r % gsize;
    tn = r / gsize;
}

// Work unit u = (tile, K slice): the splits slices of a tile are consecutive units, so
// they run at about the same time on neighbouring CTAs.  Slice s covers k-blocks
// [s * num_kb / splits, (s + 1) * num_kb / splits), never empty (splits <= num_kb).
GB300_HD void unit_coords(int u, const KParams &p, int &tm, int &tn, int &kb0, int &kb1) {
    const int t = u / p.splits, s = u - t * p.splits;
    tile_coords(t, p.tiles_m, p.group_m, tm, tn, p.tiles_n);
    kb0 = (int)((int64_t)s * p.num_kb / p.splits);
    kb1 = (int)((int64_t)(s + 1) * p.num_kb / p.splits);
}

// K blocks of a unit walk forward in even persistent rounds and backward in odd ones
// (round = how many units this CTA has taken before), so that a round starts on the
// A and B slices the previous round read last, which are the likeliest still in L2.
#ifndef GB300_SERPENTINE_K
#define GB300_SERPENTINE_K 1
#endif
GB300_HD int kb_at(int j, int kb0, int kb1, uint32_t round) {
    return (GB300_SERPENTINE_K && (round & 1u)) ? kb1 - 1 - j : kb0 + j;
}

// A piece of work: K blocks [kb0, kb1) of tile (tm, tn).  ROLE_TILE pieces cover a
// whole tile (or, with split-K, one slice); stream-K pieces that cover only part of a
// tile are ROLE_EARLY (ends the tile, starts a span: stores its partial sum into D and
// publishes flag `slot`) or ROLE_FINAL (starts the tile, ends a span: adds into D once
// flag `slot` is published).
enum : int { ROLE_TILE = 0, ROLE_EARLY = 1, ROLE_FINAL = 2 };
struct Work {
    int tm, tn, kb0, kb1, role, slot;
};

// Stream-K spans: the k-blocks of tiles [dp_tiles, tiles) in (tile, k-block) order, cut into
// `units` equal spans; unit u's span is [g, g_end).
GB300_HD void span_of(int unit, int tiles, int dp_tiles, int num_kb, int units, int64_t &g, int64_t &g_end) {
    const int64_t base = (int64_t)dp_tiles * num_kb;
    const int64_t total = (int64_t)(tiles - dp_tiles) * num_kb;
    g = base + (int64_t)unit * total / units;
    g_end = base + (int64_t)(unit + 1) * total / units;
}

// The next piece of a span (g advances past it): k-blocks [kb0, kb1) of flat tile index t
// (returned).  A span is at least one tile long, so only its first piece can start inside a
// tile (the end of a tile that the previous unit starts: ROLE_EARLY, published in this
// unit's slot) and only its last can end inside one (ROLE_FINAL: it waits for the next
// unit's slot).
GB300_HD int span_piece(int64_t &g, int64_t g_end, int num_kb, int unit, Work &w) {
    const int t = (int)(g / num_kb);
    const int k0 = (int)(g - (int64_t)t * num_kb);
    const int k1 = (int64_t)k0 + (g_end - g) < (int64_t)num_kb ? (int)((int64_t)k0 + (g_end - g)) : num_kb;
    w.kb0 = k0;
    w.kb1 = k1;
    w.role = (k0 == 0 && k1 == num_kb) ? ROLE_TILE : (k0 > 0 ? ROLE_EARLY : ROLE_FINAL);
    w.slot = k0 > 0 ? unit : unit + 1;
    g += k1 - k0;
    return t;
}

// The pieces one unit (CTA or CTA pair) processes, in order; every role of the kernel
// walks the same sequence.  Without stream-K: units tile0, tile0 + step, ... of the
// (tile x split) list.  With stream-K: first the whole tiles tile0, tile0 + step, ...
// below sk_dp_tiles, then the unit's span of the remaining tiles' k-blocks.
struct WorkIter {
    int unit, step, u;
    int64_t g, g_end;
    GB300_HD WorkIter(const KParams &p, int unit0, int step0) : unit(unit0), step(step0), u(unit0) {
        g = g_end = 0;
        if (p.sk) span_of(unit0, p.num_tiles, p.sk_dp_tiles, p.num_kb, p.sk_units, g, g_end);
    }
    GB300_HD bool next(const KParams &p, Work &w) {
        if (!p.sk) {
            if (u >= p.num_tiles * p.splits) return false;
            unit_coords(u, p, w.tm, w.tn, w.kb0, w.kb1);
            w.role = ROLE_TILE;
            w.slot = 0;
            u += step;
            return true;
        }
        if (u < p.sk_dp_tiles) {
            tile_coords(u, p.tiles_m, p.group_m, w.tm, w.tn, p.tiles_n);
            w.kb0 = 0;
            w.kb1 = p.num_kb;
            w.role = ROLE_TILE;
            w.slot = 0;
            u += step;
            return true;
        }
        if (g >= g_end) return false;
        const int t = span_piece(g, g_end, p.num_kb, unit, w);
        tile_coords(t, p.tiles_m, p.group_m, w.tm, w.tn, p.tiles_n);
        return true;
    }
};

// The pieces one unit (CTA or CTA pair) of the two-product chain (gemm_chain.cu) processes,
// in order.  Tiles are 1-D (rows of D).  Without stream-K: whole tiles unit0, unit0 + step, ...
// With stream-K: the whole tiles below sk_dp_tiles the same way, then the unit's span of the
// remaining tiles' first-product k-blocks.  A ROLE_TILE or ROLE_FINAL piece ends with the
// rounding, the second product and D; a ROLE_EARLY piece only hands its partial T over.
struct ChainIter {
    int unit, step, u;
    int64_t g, g_end;
    GB300_HD ChainIter(const ChainParams &p, int unit0, int step0) : unit(unit0), step(step0), u(unit0) {
        g = g_end = 0;
        if (p.sk) span_of(unit0, p.tiles, p.sk_dp_tiles, p.num_kb1, p.sk_units, g, g_end);
    }
    GB300_HD bool next(const ChainParams &p, Work &w) {
        if (u < (p.sk ? p.sk_dp_tiles : p.tiles)) {
            w.tm = u;
            w.tn = 0;
            w.kb0 = 0;
            w.kb1 = p.num_kb1;
            w.role = ROLE_TILE;
            w.slot = 0;
            u += step;
            return true;
        }
        if (!p.sk || g >= g_end) return false;
        w.tm = span_piece(g, g_end, p.num_kb1, unit, w);
        w.tn = 0;
        return true;
    }
};

// The bounded part of a barrier wait, out of line: reached only when the first probe
// found the phase still open.  Kept out of the inlined fast path, a completed wait costs
// the waiting thread ~86 clocks instead of ~200 (measured on GB300), which matters on the
// MMA issuer's path between k-blocks.
template <bool CLUSTER>
__device__ __noinline__ bool mbar_wait_slow(uint32_t a, uint32_t parity, bool honor_abort, volatile int *abort_flag,
                                            int *status, uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (CLUSTER ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity)) return true;
        if ((it & 15) == 0) {
            if (honor_abort && *abort_flag) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                *abort_flag = 1;
                atomicCAS(status, 0, (int)GEMM_ERR_TIMEOUT);   // the first error recorded stands
                return false;
            }
        }
    }
}

struct Waiter {
    volatile int *abort_flag;
    int *status;
    uint64_t timeout_ns;

    // wait for phase `parity` of `bar`; false if the kernel is giving up
    // (another role aborted, unless honor_abort is false, or the limit ran out).
    // CLUSTER: acquire at cluster scope (a barrier other CTAs' threads release-arrive on)
    template <bool CLUSTER = false>
    __device__ __forceinline__ bool wait(uint64_t *bar, uint32_t parity, bool honor_abort = true) const {
        const uint32_t a = smem_addr(bar);
        if (CLUSTER ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity)) return true;
        return mbar_wait_slow<CLUSTER>(a, parity, honor_abort, abort_flag, status, timeout_ns);
    }

    // wait until the global flag *f holds v (acquire); false if the kernel is giving up
    __device__ __forceinline__ bool wait_flag(const int *f, int v) const {
        if (ld_acquire_gpu(f) == v) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 1;; ++it) {
            __nanosleep(64);
            if (ld_acquire_gpu(f) == v) return true;
            if ((it & 15) == 0) {
                if (*abort_flag) return false;
                if (globaltimer_ns() - t0 > timeout_ns) {
                    *abort_flag = 1;
                    atomicCAS(status, 0, (int)GEMM_ERR_TIMEOUT);   // the first error recorded stands
                    return false;
                }
            }
        }
    }
};

// Per-role clock accounting of a GB300_TRACE=1 build (off by default): a role keeps its
// counters in registers (RoleClock laps between its waits) and adds them to its CTA's
// TRACE_SLOTS counters in KParams::trace when it ends.  In other builds every mark and
// lap compiles to nothing and the counters are dead code.
#ifndef GB300_TRACE
#define GB300_TRACE 0
#endif
struct RoleClock {
#if GB300_TRACE
    long long t = 0;
    __device__ __forceinline__ void mark() { t = clock64(); }
    __device__ __forceinline__ void lap(unsigned long long &acc) {
        const long long n = clock64();
        acc += (unsigned long long)(n - t);
        t = n;
    }
#else
    __device__ __forceinline__ void mark() {}
    __device__ __forceinline__ void lap(unsigned long long &) {}
#endif
};

__device__ __forceinline__ void trace_add(const KParams &p, int slot, unsigned long long v) {
#if GB300_TRACE
    if (p.trace) atomicAdd(p.trace + (size_t)blockIdx.x * TRACE_SLOTS + slot, v);
#endif
}

__device__ __forceinline__ void trace_max(const KParams &p, int slot, unsigned long long v) {
#if GB300_TRACE
    if (p.trace) atomicMax(p.trace + (size_t)blockIdx.x * TRACE_SLOTS + slot, v);
#endif
}

// clock64() at some point of this thread minus its value at kernel entry (trace builds)
__device__ __forceinline__ unsigned long long since(long long t_entry) {
#if GB300_TRACE
    return (unsigned long long)(clock64() - t_entry);
#else
    return 0ull;
#endif
}

// On-device checks of a GB300_CHECKS=1 build (the "checks" library variant; other builds
// compile them out).  Every TMA coordinate the kernels compute is checked against the
// tiling it comes from: the innermost coordinate starts on a 16-byte boundary (the
// copy is illegal otherwise), no coordinate is negative, and each lies inside the
// operand's extent rounded up to whole tiles (a copy beyond it only reads the fill
// value, so such a coordinate means a wrong tile or k-block index).  A failed check
// records GEMM_ERR_CHECK as the run's status (the first error recorded stands) and the
// coordinate is clamped to a legal value, so that the copy can neither fault nor hang.
#ifndef GB300_CHECKS
#define GB300_CHECKS 0
#endif
__device__ __forceinline__ void check_fail(int *status) {
#if GB300_CHECKS
    atomicCAS(status, 0, (int)GEMM_ERR_CHECK);
#endif
}

// innermost coordinate x (elements of ELEM_BYTES bytes) of a copy inside [0, limit)
template <int ELEM_BYTES>
__device__ __forceinline__ int checked_x(int *status, int x, int limit) {
#if GB300_CHECKS
    constexpr int ALIGN = ELEM_BYTES >= 16 ? 1 : 16 / ELEM_BYTES;
    if (x < 0 || x % ALIGN != 0 || x >= limit) {
        check_fail(status);
        x = x < 0 ? 0 : x - x % ALIGN;
    }
#endif
    return x;
}

// outer coordinate y of a copy inside [0, limit)
__device__ __forceinline__ int checked_y(int *status, int y, int limit) {
#if GB300_CHECKS
    if (y < 0 || y >= limit) {
        check_fail(status);
        if (y < 0) y = 0;
    }
#endif
    return y;
}

// Byte offset of 16-byte chunk c of staging row `row` under the TMA swizzle whose span is
// the row (128-, 64- or 32-byte rows: the 128B, 64B or 32B mode, which XOR address bits
// 4.. with bits 7..): for a warp whose lane i owns row i, each 8-lane phase of a 128-bit
// access then covers all 32 banks once.
template <int ROW_BYTES>
__device__ __forceinline__ uint32_t swz_off(int row, int c) {
    static_assert(ROW_BYTES == 128 || ROW_BYTES == 64 || ROW_BYTES == 32, "swizzle span");
    const int x = ROW_BYTES == 128 ? (row & 7) : (ROW_BYTES == 64 ? ((row >> 1) & 3) : ((row >> 2) & 1));
    return (uint32_t)(row * ROW_BYTES + ((c ^ x) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// SMEM -> TMEM copies of stage s's scales, each 512-byte SMEM block (32 lanes x 16
// bytes: one word of 128 rows) replicated to the 4 lane windows: SFA word w in columns
// sfa_t + 4w.., SFB (word w, column group h) in sfb_t + 4(w*HALVES + h)..  The stage's
// blocks are numbered SFA first, then SFB; with NPART issuing threads, part `part`
// issues the blocks whose number is part modulo NPART.
template <class Cfg, int NPART = 1>
__device__ __forceinline__ void copy_scales(uint8_t *smem, int s, uint32_t sfa_t, uint32_t sfb_t, int part = 0) {
    const uint32_t sf_src = smem_addr(smem + Cfg::OFF_SF + s * (Cfg::SFA_BYTES + Cfg::SFB_BYTES));
#pragma unroll
    for (int i = 0; i < Cfg::SF_WORDS; ++i)
        if (i % NPART == part)
            tmem_cp_32x128b_warpx4<Cfg::CG>(sfa_t + 4 * i, smem_desc(sf_src + 512 * i, 512, 128, SWZ_NONE));
#pragma unroll
    for (int i = 0; i < Cfg::SF_WORDS * Cfg::HALVES; ++i)
        if ((Cfg::SF_WORDS + i) % NPART == part)
            tmem_cp_32x128b_warpx4<Cfg::CG>(sfb_t + 4 * i,
                                            smem_desc(sf_src + Cfg::SFA_BYTES + 512 * i, 512, 128, SWZ_NONE));
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                   const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                   const KParams p) {
    constexpr int CG = Cfg::CG;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int BN = Cfg::BN;
    const long long t_entry = clock64();             // this thread's entry (clock meter, trace)
    const uint64_t ns_entry = threadIdx.x == 0 ? globaltimer_ns() : 0ull;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *tfull = bars + 2 * STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *cload = tempty + 2;
    uint64_t *drain = cload + 2 * Cfg::EPI_WARPS;
    uint64_t *epi_sync = drain + 1;                       // every epilogue warp stored its part of a partial sum
    uint64_t *cdrain = epi_sync + 1;                      // COPIER only
    uint64_t *sffull = cdrain + 1;                        // COPIER only
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::OFF_MISC + 4);
    const Waiter W{abort_flag, p.status, p.timeout_ns};

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (p.has_c) prefetch_tensormap(&tmC);
        prefetch_tensormap(&tmD);
        if constexpr (Cfg::SCALED) {
            prefetch_tensormap(&tmSFA);
            prefetch_tensormap(&tmSFB);
        }
        for (int s = 0; s < STAGES; ++s) {
            // the producer's arrival (with the operands' transaction bytes) and, with COPIER,
            // one commit per copier warp once the stage's scales are in TMEM
            mbar_init(&full[s], 1 + Cfg::COPIERS);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], Cfg::EPI_WARPS * CG);   // every epilogue warp of the pair
        }
        for (int i = 0; i < 2 * Cfg::EPI_WARPS; ++i) mbar_init(&cload[i], 1);
        mbar_init(drain, 1);
        mbar_init(epi_sync, Cfg::EPI_WARPS);
        if constexpr (Cfg::COPIER) {
            for (int i = 0; i < STAGES; ++i) mbar_init(&sffull[i], 1);
            mbar_init(cdrain, Cfg::COPIERS);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_addr(tmem_slot), 512);
        tmem_relinquish<CG>();
    }
    tc_fence_before_sync();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    const int tile0 = blockIdx.x / CG;
    const int tile_step = gridDim.x / CG;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            uint32_t round = 0;
            RoleClock rc;
            unsigned long long tr_wait = 0, tr_issue = 0, tr_stages = 0;
            WorkIter it(p, tile0, tile_step);
            Work wk;
            for (; ok && it.next(p, wk); ++round) {
                const int tm = wk.tm, tn = wk.tn, kb0 = wk.kb0, kb1 = wk.kb1;
                const int m0 = tm * TILE_M * CG + (int)rank * TILE_M;
                const int n0 = tn * BN + (int)rank * Cfg::B_ROWS;
                for (int j = 0; j < kb1 - kb0; ++j) {
                    const int kb = kb_at(j, kb0, kb1, round);
                    rc.mark();
                    if (!W.wait(&empty[s], ph ^ 1u)) { ok = false; break; }
                    rc.lap(tr_wait);
                    const bool withhold = p.fault == 1 && round == 0 && j == 0;
                    if (rank == 0 && Cfg::COPIER) mbar_arrive_expect_tx(&sffull[s], Cfg::TX_SF);
                    if (rank == 0 && !withhold) mbar_arrive_expect_tx(&full[s], Cfg::COPIER ? Cfg::TX_AB : Cfg::TX_BYTES);
                    const uint32_t a_dst = smem_addr(smem + Cfg::OFF_A + s * Cfg::A_BYTES);
                    const uint32_t b_dst = smem_addr(smem + Cfg::OFF_B + s * Cfg::B_BYTES);
                    const uint32_t fb = smem_addr(&full[s]);
                    // packed scale factors of this (128-row block, k-block) and (tile column, k-block):
                    // 512-byte blocks, viewed by their tensor maps as rows of 128 bytes
                    const uint32_t sf_dst = smem_addr(smem + Cfg::OFF_SF + s * (Cfg::SFA_BYTES + Cfg::SFB_BYTES));
                    const int sfa_row = ((tm * CG + (int)rank) * p.num_kb + kb) * (Cfg::SFA_BYTES / 128);
                    const int sfb_row = (tn * p.num_kb + kb) * (Cfg::SFB_BYTES / 128);
                    // the completion of every copy of the stage counts on the leader's full[s]
                    // (the scales' on its sffull[s] when a copier warp moves them)
                    const uint32_t bar = CG == 1 ? fb : mapa_shared(fb, 0);
                    uint32_t sbar = bar;
                    if constexpr (Cfg::COPIER) {
                        const uint32_t sfb = smem_addr(&sffull[s]);
                        sbar = CG == 1 ? sfb : mapa_shared(sfb, 0);
                    }
                    auto load_on = [&](uint32_t dst, const CUtensorMap *m, int c0, int c1, uint32_t mb) {
                        if constexpr (CG == 1) tma_load_2d(dst, m, mb, c0, c1);
                        else tma_load_2d_pair(dst, m, mb, c0, c1);
                    };
                    auto load = [&](uint32_t dst, const CUtensorMap *m, int c0, int c1) { load_on(dst, m, c0, c1, bar); };
                    // an operand tile: K-major, one box of BK x rows; MN-major, rows / ATOM_MN
                    // boxes of ATOM_MN x BK, one per 128-byte atom column
                    // (row_lim: the operand's rows rounded up to whole tiles; checks builds only)
                    auto load_operand = [&](uint32_t dst, const CUtensorMap *m, int row0, int rows, bool mn,
                                            int row_lim) {
                        constexpr int EB = Cfg::ELEM_BITS == 16 ? 2 : 1;   // bytes of a tensor-map element
                        if (!Cfg::MN_OK || !mn) {
                            load(dst, m, checked_x<EB>(p.status, kb * Cfg::TMA_BK, p.num_kb * Cfg::TMA_BK),
                                 checked_y(p.status, row0, row_lim));
                        } else {
                            for (int i = 0; i < rows / Cfg::ATOM_MN; ++i)
                                load(dst + i * Cfg::ATOM_BYTES, m, checked_x<EB>(p.status, row0 + i * Cfg::ATOM_MN, row_lim),
                                     checked_y(p.status, kb * Cfg::BK, p.num_kb * Cfg::BK));
                        }
                    };
                    if constexpr (Cfg::SCALED) {    // the scales first: the copier warp starts on them
                        load_on(sf_dst, &tmSFA, 0,
                                checked_y(p.status, sfa_row, p.tiles_m * CG * p.num_kb * (Cfg::SFA_BYTES / 128)), sbar);
                        load_on(sf_dst + Cfg::SFA_BYTES, &tmSFB, 0,
                                checked_y(p.status, sfb_row, p.tiles_n * p.num_kb * (Cfg::SFB_BYTES / 128)), sbar);
                    }
                    // test hook (fault 2): A rows shifted past the tiled extent, which only reads the
                    // fill value (wrong D, no fault) and which a checks build reports
                    const int a_row = m0 + (p.fault == 2 ? p.tiles_m * TILE_M * CG : 0);
                    load_operand(a_dst, &tmA, a_row, TILE_M, p.a_mn != 0, p.tiles_m * TILE_M * CG);
                    load_operand(b_dst, &tmB, n0, Cfg::B_ROWS, p.b_mn != 0, p.tiles_n * BN);
                    rc.lap(tr_issue);
                    ++tr_stages;
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
            }
            trace_add(p, TR_PROD_WAIT, tr_wait);
            trace_add(p, TR_PROD_ISSUE, tr_issue);
            trace_add(p, TR_PROD_STAGES, tr_stages);
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issue
        if (rank == 0 && lane == 0) {
            // shared-memory descriptors (128-byte swizzle).  K-major: 8-row groups 1024 B
            // apart, the leading offset unused (encoded 1), an MMA's K step = 32 bytes.
            // MN-major: 8-row K groups 1024 B apart, atom columns ATOM_BYTES apart (the
            // leading offset), an MMA's K step = MMA_K rows of 128 bytes.
            const uint32_t a_lbo = p.a_mn ? Cfg::ATOM_BYTES : 16, b_lbo = p.b_mn ? Cfg::ATOM_BYTES : 16;
            const uint32_t a_step = p.a_mn ? (Cfg::MMA_K * 128) >> 4 : 2, b_step = p.b_mn ? (Cfg::MMA_K * 128) >> 4 : 2;
            int s = 0;
            uint32_t ph = 0, acc_it = 0;
            bool ok = true;
            RoleClock rc;
            unsigned long long tr_wacc = 0, tr_wab = 0, tr_wsf = 0, tr_issue = 0, tr_kb = 0, tr_first = 0;
            WorkIter it(p, tile0, tile_step);
            Work wk;
            for (; ok && it.next(p, wk); ++acc_it) {
                const int kb0 = wk.kb0, kb1 = wk.kb1;
                const uint32_t b = Cfg::ACC_BUFS == 2 ? (acc_it & 1u) : 0u;
                const uint32_t aph = Cfg::ACC_BUFS == 2 ? ((acc_it >> 1) & 1u) : (acc_it & 1u);
                rc.mark();
                // the peer CTA's epilogue warps release-arrive on tempty: cluster-scope acquire
                if (!W.wait<CG == 2>(&tempty[b], aph ^ 1u)) { ok = false; break; }
                rc.lap(tr_wacc);
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * BN;
                for (int j = 0; j < kb1 - kb0; ++j) {
                    if (!W.wait(&full[s], ph)) { ok = false; break; }
                    rc.lap(tr_wab);
                    if (GB300_TRACE && tr_kb == 0) tr_first = since(t_entry);
                    tc_fence_after_sync();
                    const uint64_t ad = smem_desc(smem_addr(smem + Cfg::OFF_A + s * Cfg::A_BYTES), a_lbo, 1024, SWZ_128B);
                    const uint64_t bd = smem_desc(smem_addr(smem + Cfg::OFF_B + s * Cfg::B_BYTES), b_lbo, 1024, SWZ_128B);
                    if constexpr (Cfg::SCALED) {
                        // stage s's scale slot (filled here, or by the copier warps before their
                        // commits completed full[s])
                        const uint32_t sfa_t = tmem_base + Cfg::SF_COL0 + s * Cfg::SF_SLOT;
                        const uint32_t sfb_t = sfa_t + 4 * Cfg::SF_WORDS;
                        if constexpr (!Cfg::COPIER) copy_scales<Cfg>(smem, s, sfa_t, sfb_t);
                        // MMA step k reads scales k*SF_PER_MMA.. of the stage: word w, from byte id
                        // (1X: byte k; 2X: half-word 0 or 2; 4X: the whole word, id 0)
#pragma unroll
                        for (int k = 0; k < Cfg::BK / Cfg::MMA_K; ++k) {
                            const uint32_t w = (uint32_t)(k * Cfg::SF_PER_MMA) / 4u, id = (uint32_t)(k * Cfg::SF_PER_MMA) % 4u;
                            mma_scaled<Cfg::KIND, CG>(d_tmem, ad + a_step * k, bd + b_step * k,
                                                      p.idesc | (id << 4) | (id << 29), sfa_t + 4 * w,
                                                      sfb_t + 4 * Cfg::HALVES * w, (j != 0) | (k != 0));
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < Cfg::BK / Cfg::MMA_K; ++k)   // 32 bytes of K = 2 descriptor units
                            mma_f16<CG>(d_tmem, ad + a_step * k, bd + b_step * k, p.idesc, (j != 0) | (k != 0));
                    }
                    if constexpr (CG == 1) tc_commit<1>(smem_addr(&empty[s]));
                    else tc_commit_pair(smem_addr(&empty[s]), 0x3);
                    rc.lap(tr_issue);
                    ++tr_kb;
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                if constexpr (CG == 1) tc_commit<1>(smem_addr(&tfull[b]));
                else tc_commit_pair(smem_addr(&tfull[b]), 0x3);
            }
            // every MMA this thread issued has finished before teardown (also
            // after an abort: this wait is bounded by time only)
            tc_commit<CG>(smem_addr(drain));
            W.wait(drain, 0, false);
            trace_add(p, TR_MMA_WAIT_ACC, tr_wacc);
            trace_add(p, TR_MMA_WAIT_AB, tr_wab);
            trace_add(p, TR_MMA_WAIT_SF, tr_wsf);
            trace_add(p, TR_MMA_ISSUE, tr_issue);
            trace_add(p, TR_MMA_KBLOCKS, tr_kb);
            trace_add(p, TR_MMA_PIECES, acc_it);
            trace_add(p, TR_MMA_FIRST, tr_first);
            trace_add(p, TR_MMA_END, since(t_entry));
        }
    } else if (Cfg::COPIER && warp >= Cfg::COPY_WARP) {
        // ---------------------------------------------------------- scale copies
        if constexpr (Cfg::COPIER) {
            const int part = warp - Cfg::COPY_WARP;      // this warp's share of each stage's copies
            if (rank == 0 && lane == 0) {
                // stage s's slot is rewritten only after sffull[s] of the next round, i.e. after
                // the producer saw empty[s]: the MMAs that read the slot have completed
                int s = 0;
                uint32_t ph = 0;
                bool ok = true;
                RoleClock rc;
                unsigned long long tr_wait = 0, tr_issue = 0;
                WorkIter it(p, tile0, tile_step);
                Work wk;
                while (ok && it.next(p, wk)) {
                    for (int kb = wk.kb0; kb < wk.kb1; ++kb) {
                        rc.mark();
                        if (!W.wait(&sffull[s], ph)) { ok = false; break; }
                        rc.lap(tr_wait);
                        tc_fence_after_sync();
                        const uint32_t sfa_t = tmem_base + Cfg::SF_COL0 + s * Cfg::SF_SLOT;
                        copy_scales<Cfg, Cfg::COPIERS>(smem, s, sfa_t, sfa_t + 4 * Cfg::SF_WORDS, part);
                        // full[s] of the leader: the MMA issuer's one wait covers the copies
                        if constexpr (CG == 1) tc_commit<1>(smem_addr(&full[s]));
                        else tc_commit_pair(smem_addr(&full[s]), 0x1);
                        rc.lap(tr_issue);
                        if (++s == STAGES) { s = 0; ph ^= 1u; }
                    }
                }
                trace_add(p, TR_CP_WAIT, tr_wait);
                trace_add(p, TR_CP_ISSUE, tr_issue);
                // every copy this thread issued has finished before teardown
                if constexpr (CG == 1) tc_commit<1>(smem_addr(cdrain));
                else tc_commit_pair(smem_addr(cdrain), 0x1);
                W.wait(cdrain, 0, false);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int e = warp - 2;                           // epilogue warp index
        const int q = warp & 3;                           // TMEM lane window of this warp
        const int h = e / 4;                              // which WCOLS-wide column slice of the tile
        uint8_t *ebuf = smem + Cfg::OFF_EPI + e * Cfg::EPI_BUFS * Cfg::EPI_BUF;
        uint64_t *cb = cload + 2 * e;
        // C is read once and D written once: let them leave L2 before the operand tiles
        const uint64_t stream_pol = l2_policy_evict_first();
        // ec counts the 32 x 32 boxes this warp has stored (box ec is staged in buffer
        // ec % EPI_BUFS);
        // lc[i] counts the loads issued into buffer i (the phases of cb[i]); n_early counts the
        // stream-K partial sums this CTA has published (the phases of epi_sync)
        uint32_t acc_it = 0, ec = 0, n_early = 0;
        uint32_t lc0 = 0, lc1 = 0;                    // the lc[i] of the comment, kept in registers
        bool ok = true;
        RoleClock rc;
        unsigned long long tr_wacc = 0, tr_ld = 0, tr_wc = 0, tr_store = 0, tr_end = 0;
        // a TMA load of one 32 x EPI_BOX fp32 box into staging buffer i (issued by lane 0, counted by all)
        auto issue = [&](uint32_t i, const CUtensorMap *m, int c0, int c1) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&cb[i], Cfg::EPI_BUF);
                tma_load_2d_hint(smem_addr(ebuf + i * Cfg::EPI_BUF), m, smem_addr(&cb[i]),
                                 checked_x<4>(p.status, c0, p.N), checked_y(p.status, c1, p.M), stream_pol);
            }
            if (i) ++lc1; else ++lc0;
        };
        auto landed = [&](uint32_t i) -> bool {
            return __all_sync(0xffffffffu, W.wait(&cb[i], ((i ? lc1 : lc0) - 1u) & 1u));
        };
        // add the fp32 box in staging buffer i (row `lane` of EPI_BOX * 4 bytes, swizzled)
        auto add_box = [&](uint32_t i, float (&v)[Cfg::EPI_BOX]) {
            const uint32_t bb = smem_addr(ebuf + i * Cfg::EPI_BUF);
#pragma unroll
            for (int c = 0; c < Cfg::EPI_BOX / 4; ++c) {
                const float4 cv = ld_shared_v4f(bb + swz_off<Cfg::EPI_BOX * 4>(lane, c));
                v[4 * c + 0] += cv.x;
                v[4 * c + 1] += cv.y;
                v[4 * c + 2] += cv.z;
                v[4 * c + 3] += cv.w;
            }
        };
        // hand accumulator bb back to the MMA (all 32 lanes have read it)
        auto release = [&](uint32_t bb) {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 1) mbar_arrive(&tempty[bb]);
                else mbar_arrive_remote(mapa_shared(smem_addr(&tempty[bb]), 0));
            }
        };
        WorkIter it(p, tile0, tile_step);
        Work wk;
        for (; ok && it.next(p, wk); ++acc_it) {
            const uint32_t b = Cfg::ACC_BUFS == 2 ? (acc_it & 1u) : 0u;
            const uint32_t aph = Cfg::ACC_BUFS == 2 ? ((acc_it >> 1) & 1u) : (acc_it & 1u);
            const int m_warp = wk.tm * TILE_M * CG + (int)rank * TILE_M + 32 * q;
            const int n_warp = wk.tn * BN + h * Cfg::WCOLS;
            // 32 x EPI_BOX boxes that lie wholly outside D are neither loaded nor stored
            const int boxes_in = m_warp < p.M ? max(0, min(Cfg::WCHUNKS * Cfg::BOXES,
                                                           (p.N - n_warp + Cfg::EPI_BOX - 1) / Cfg::EPI_BOX))
                                              : 0;
            // every piece but a partial sum (ROLE_EARLY) adds C, loaded box by box
            const bool use_c = wk.role != ROLE_EARLY && p.has_c && boxes_in > 0;
            if (use_c) {                   // the piece's first C box loads while its accumulator is computed
                if (lane == 0) bulk_wait_group_read0();
                issue(ec % Cfg::EPI_BUFS, &tmC, n_warp, m_warp);
            }
            rc.mark();
            if (!__all_sync(0xffffffffu, W.wait(&tfull[b], aph))) break;
            rc.lap(tr_wacc);
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + b * BN + h * Cfg::WCOLS;

            auto release_accumulator = [&]() { release(b); };
            // a stream-K piece that starts its tile waits until its tile's other piece has
            // stored its partial sum into D and published it (the flag carries this run's
            // epoch); this one then adds into D
            if (GB300_CHECKS && wk.role != ROLE_TILE && (wk.slot < 0 || wk.slot >= p.sk_units)) {
                check_fail(p.status);           // a stream-K flag outside the plan's flag buffer
                ok = false;
                break;
            }
            auto await_partial = [&]() -> bool {
                if (wk.role != ROLE_FINAL) return true;
                const bool got = W.wait_flag(p.sk_flags + wk.slot * CG + (int)rank, p.epoch);
                if (got && lane == 0) fence_proxy_async_global();   // the flag before TMA traffic to D
                return __all_sync(0xffffffffu, got);
            };
            // box jb of the warp's slice (columns EPI_BOX * jb.., sub-box u of a 32-column
            // chunk whose registers are acc): add C, convert, stage in shared memory, then
            // TMA-store it to D (reduce-add for split-K slices and for stream-K pieces that
            // finish a tile)
            auto store_box = [&](int jb, const uint32_t (&acc)[32], int u) -> bool {
                const uint32_t cur = ec % Cfg::EPI_BUFS;
                uint8_t *buf = ebuf + cur * Cfg::EPI_BUF;
                if (Cfg::EPI_BUFS == 2 && use_c && jb + 1 < boxes_in) {
                    if (lane == 0) bulk_wait_group_read0();   // the store from the other buffer has read it
                    issue(cur ^ 1u, &tmC, n_warp + Cfg::EPI_BOX * (jb + 1), m_warp);
                }
                if (jb >= boxes_in) return true;
                if (Cfg::EPI_BUFS == 1 && use_c && jb > 0) {  // one buffer: this box's C loads now
                    if (lane == 0) bulk_wait_group_read0();   // the last store has read the buffer
                    issue(0, &tmC, n_warp + Cfg::EPI_BOX * jb, m_warp);
                }
                float v[Cfg::EPI_BOX];
#pragma unroll
                for (int i = 0; i < Cfg::EPI_BOX; ++i) v[i] = __uint_as_float(acc[u * Cfg::EPI_BOX + i]);
                if (use_c) {
                    rc.lap(tr_store);
                    if (!landed(cur)) return false;
                    rc.lap(tr_wc);
                    add_box(cur, v);
                } else if (lane == 0) {
                    // the store that last used this buffer (one or two boxes back) has read it
                    if (Cfg::EPI_BUFS == 2) bulk_wait_group_read1();
                    else bulk_wait_group_read0();
                }
                __syncwarp();
                const uint32_t sb = smem_addr(buf);
                if constexpr (Cfg::OUT_BF16) {
                    // rows of EPI_BOX * 2 bytes (64 or 32), swizzled over the row
#pragma unroll
                    for (int c = 0; c < Cfg::EPI_BOX / 8; ++c)
                        st_shared_v4(sb + swz_off<Cfg::EPI_BOX * 2>(lane, c), pack_bf16x2(v[8 * c + 0], v[8 * c + 1]),
                                     pack_bf16x2(v[8 * c + 2], v[8 * c + 3]), pack_bf16x2(v[8 * c + 4], v[8 * c + 5]),
                                     pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
                } else {
                    // rows of EPI_BOX * 4 bytes (128 or 64), swizzled over the row
#pragma unroll
                    for (int c = 0; c < Cfg::EPI_BOX / 4; ++c)
                        st_shared_v4(sb + swz_off<Cfg::EPI_BOX * 4>(lane, c), __float_as_uint(v[4 * c + 0]),
                                     __float_as_uint(v[4 * c + 1]), __float_as_uint(v[4 * c + 2]),
                                     __float_as_uint(v[4 * c + 3]));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    // a store must not start at a negative coordinate
                    const int dx = checked_x<Cfg::OUT_BF16 ? 2 : 4>(p.status, n_warp + Cfg::EPI_BOX * jb, p.N);
                    const int dy = checked_y(p.status, m_warp, p.M);
                    if (wk.role == ROLE_EARLY) {
                        tma_store_2d(&tmD, smem_addr(buf), dx, dy);
                    } else if (p.splits > 1 || wk.role == ROLE_FINAL) {
                        tma_reduce_add_2d(&tmD, smem_addr(buf), dx, dy);
                    } else {
                        tma_store_2d_hint(&tmD, smem_addr(buf), dx, dy, stream_pol);
                    }
                    bulk_commit_group();
                }
                ++ec;
                rc.lap(tr_store);
                return true;
            };

            if constexpr (Cfg::ACC_BUFS == 1) {
                // copy the whole slice to registers first so that the MMA can start the
                // next tile while this one is converted and stored
                uint32_t acc[Cfg::WCHUNKS][32];
#pragma unroll
                for (int j = 0; j < Cfg::WCHUNKS; ++j) tmem_ld_32x32b_x32(taddr + EPI_COLS * j, acc[j]);
                tmem_ld_wait_all();
#pragma unroll
                for (int j = 0; j < Cfg::WCHUNKS; ++j) tie_registers(acc[j]);
                release_accumulator();
                rc.lap(tr_ld);
                if (!await_partial()) { ok = false; break; }
                rc.lap(tr_wc);
#pragma unroll
                for (int j = 0; j < Cfg::WCHUNKS; ++j)
#pragma unroll
                    for (int u = 0; u < Cfg::BOXES; ++u)
                        if (ok) ok = store_box(j * Cfg::BOXES + u, acc[j], u);
            } else {
                if (!await_partial()) { ok = false; break; }
                rc.lap(tr_wc);
                for (int j = 0; j < Cfg::WCHUNKS && ok; ++j) {
                    uint32_t acc[32];
                    tmem_ld_32x32b_x32(taddr + EPI_COLS * j, acc);
                    tmem_ld_wait(acc);
                    if (j == Cfg::WCHUNKS - 1) release_accumulator();
                    rc.lap(tr_ld);
#pragma unroll
                    for (int u = 0; u < Cfg::BOXES; ++u)
                        if (ok) ok = store_box(j * Cfg::BOXES + u, acc, u);
                }
            }
            if (GB300_TRACE) tr_end = since(t_entry);
            if (ok && wk.role == ROLE_EARLY) {
                // publish the partial sum once every epilogue warp's stores have completed
                if (lane == 0) {
                    bulk_wait_group0();
                    fence_proxy_async_global();
                    mbar_arrive(epi_sync);
                }
                if (e == 0) {
                    ok = __all_sync(0xffffffffu, W.wait(epi_sync, n_early & 1u));
                    if (ok && lane == 0) {
                        __threadfence();
                        st_release_gpu(p.sk_flags + wk.slot * CG + (int)rank, p.epoch);
                    }
                }
                ++n_early;
            }
        }
        if (lane == 0) {
            bulk_wait_group0();
            trace_add(p, TR_EPI_WAIT_ACC, tr_wacc);
            trace_add(p, TR_EPI_TMEM_LD, tr_ld);
            trace_add(p, TR_EPI_WAIT_C, tr_wc);
            trace_add(p, TR_EPI_STORE, tr_store);
            trace_add(p, TR_EPI_PIECES, acc_it);
            trace_max(p, TR_EPI_END, tr_end);
        }
    }

    // ----------------------------------------------------------------- teardown
    __syncwarp();
    if (*abort_flag) {
        // give copies that were already in flight time to land before the
        // shared memory they target is released
        for (int i = 0; i < 64; ++i) __nanosleep(1000);
    }
    tc_fence_before_sync();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem_base, 512);
    }
    if (threadIdx.x == 0 && (p.clk_meter != nullptr || GB300_TRACE)) {
        const unsigned long long dclk = (unsigned long long)(clock64() - t_entry);
        const unsigned long long dns = globaltimer_ns() - ns_entry;
        if (p.clk_meter) {
            atomicAdd(p.clk_meter, dclk);
            atomicAdd(p.clk_meter + 1, dns);
        }
        trace_add(p, TR_KERNEL_CLK, dclk);
        trace_add(p, TR_KERNEL_NS, dns);
    }
}

// Launch with a cluster of Cfg::CG CTAs.
template <class Cfg>
cudaError_t launch_tc(const LaunchShape &shape, const CUtensorMap *maps, const KParams &p, cudaStream_t stream) {
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute attr[1];
    lc.gridDim = dim3(shape.grid, 1, 1);
    lc.blockDim = dim3(Cfg::THREADS, 1, 1);
    lc.dynamicSmemBytes = shape.smem;
    lc.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = shape.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    void *args[7] = {(void *)&maps[0], (void *)&maps[1], (void *)&maps[2], (void *)&maps[3],
                     (void *)&maps[4], (void *)&maps[5], (void *)&p};
    return cudaLaunchKernelExC(&lc, reinterpret_cast<const void *>(&gemm_tc_kernel<Cfg>), args);
}

template <class Cfg>
cudaError_t prepare_tc() {
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(&gemm_tc_kernel<Cfg>),
                                cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
}

template <class Cfg>
cudaError_t max_active_clusters_tc(int *clusters) {
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute attr[1];
    lc.gridDim = dim3(2 * 1024, 1, 1);
    lc.blockDim = dim3(Cfg::THREADS, 1, 1);
    lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = Cfg::CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, reinterpret_cast<const void *>(&gemm_tc_kernel<Cfg>), &lc);
}

// The instances (CTA group 1 / 2, D fp32 / bf16, and optionally a narrow pair form) of a
// block-scaled family
template <class C1F, class C1B, class C2F, class C2B, class C2NF = C2F, class C2NB = C2B>
struct ScaledInstances {
    static constexpr bool HAS_NARROW = !std::is_same<C2NF, C2F>::value;
    template <class C>
    static ScaledShape shape_of() {
        return ScaledShape{C::BN, C::STAGES, C::SMEM_BYTES, C::BK, C::SFA_BYTES, C::SFB_BYTES, C::EPI_BOX};
    }
    static ScaledShape shape(int cta_group, bool narrow) {
        if (cta_group == 1) return shape_of<C1F>();
        return narrow ? shape_of<C2NF>() : shape_of<C2F>();
    }
    static cudaError_t prepare(int cta_group, int out_bf16, bool narrow) {
        if (cta_group == 1) return out_bf16 ? prepare_tc<C1B>() : prepare_tc<C1F>();
        if (narrow) return out_bf16 ? prepare_tc<C2NB>() : prepare_tc<C2NF>();
        return out_bf16 ? prepare_tc<C2B>() : prepare_tc<C2F>();
    }
    static cudaError_t max_active_clusters(int cta_group, int out_bf16, bool narrow, int *clusters) {
        if (cta_group == 1)
            return out_bf16 ? max_active_clusters_tc<C1B>(clusters) : max_active_clusters_tc<C1F>(clusters);
        if (narrow) return out_bf16 ? max_active_clusters_tc<C2NB>(clusters) : max_active_clusters_tc<C2NF>(clusters);
        return out_bf16 ? max_active_clusters_tc<C2B>(clusters) : max_active_clusters_tc<C2F>(clusters);
    }
    static cudaError_t launch(int cta_group, int out_bf16, bool narrow, const LaunchShape &shape,
                              const CUtensorMap *maps, const KParams &p, cudaStream_t stream) {
        if (cta_group == 1)
            return out_bf16 ? launch_tc<C1B>(shape, maps, p, stream) : launch_tc<C1F>(shape, maps, p, stream);
        if (narrow)
            return out_bf16 ? launch_tc<C2NB>(shape, maps, p, stream) : launch_tc<C2NF>(shape, maps, p, stream);
        return out_bf16 ? launch_tc<C2B>(shape, maps, p, stream) : launch_tc<C2F>(shape, maps, p, stream);
    }
    static const ScaledFamily &family() {
        static const ScaledFamily f{&shape, &prepare, &max_active_clusters, &launch, HAS_NARROW};
        return f;
    }
    static_assert(C1F::CG == 1 && C1B::CG == 1 && C2F::CG == 2 && C2B::CG == 2 && C2NF::CG == 2 && C2NB::CG == 2,
                  "CTA groups");
    static_assert(!C1F::OUT_BF16 && C1B::OUT_BF16 && !C2F::OUT_BF16 && C2B::OUT_BF16 && !C2NF::OUT_BF16 &&
                      C2NB::OUT_BF16,
                  "D types");
    static_assert(C1F::SF_WORDS == C2F::SF_WORDS && C1F::BK == C2F::BK && C2NF::SF_WORDS == C2F::SF_WORDS &&
                      C2NF::BK == C2F::BK,
                  "one packed scale layout per family");
    static_assert(C1F::EPI_BOX == C1B::EPI_BOX && C2F::EPI_BOX == C2B::EPI_BOX && C2NF::EPI_BOX == C2NB::EPI_BOX,
                  "one C / D box per CTA group");
    static_assert(!HAS_NARROW || C2NF::BN == MXF8_NARROW_N, "narrow pair tile");
};

}  // namespace gb300
