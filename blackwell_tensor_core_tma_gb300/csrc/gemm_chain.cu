// Two chained tensor-core products with the intermediate kept in tensor memory
// ("Tensor Core 数据布局的演进", section "TMEM 中的累加器": some tcgen05.mma forms
// read A from TMEM instead of shared memory):
//     T = A·B        128 x N1 per CTA, fp32 accumulator in TMEM columns [0, 256)
//     P = round(T)   to the operand type, written back over T's first columns: two
//                    16-bit elements per 32-bit column, the lower K index in the low half
//     D = C + P·E    tcgen05.mma with A = P read from TMEM and E from shared memory,
//                    fp32 accumulator in TMEM columns [256, 512)
// so the intermediate never leaves the SM (except, with stream-K, which plans take on
// request only, the partial T of a tile cut between two units, which goes through
// global memory once).  One CTA (CG = 1) or one CTA pair (CG = 2, cta_group::2: 256
// rows, each CTA holding its 128 rows of A, T, P and D and half of B's and E's rows)
// owns a tile at a time and walks the tiles persistently.  Pairs halve the B and E bytes each SM takes in per row of A: the
// chain's main loop is bound by what one SM can take in (B is re-read by every
// tile), not by the L2.  Warp roles (192 threads per CTA):
//   warp 0     TMA producer (each CTA): per tile the K blocks of A and B, then the
//              K blocks of E, through one STAGES-deep ring (a stage holds A 128 x 64
//              and N1/CG rows of B, or N2/CG rows of E; 128-byte swizzled rows); a
//              pair's copies count on the leader's full[s].
//   warp 1     allocates the 512 TMEM columns; lane 0 (of the leader) issues both
//              products' MMAs.
//   warps 2-5  per tile: round T into P (tcgen05.ld, cvt, tcgen05.st), then the D
//              epilogue (tcgen05.ld, + C, convert, TMA store), each warp in its own
//              32-lane TMEM window.
// Every wait is bounded: when one runs out the kernel records GEMM_ERR_TIMEOUT,
// its roles stop, and it still frees its tensor memory.
#include "gemm_kernel.cuh"

namespace gb300 {
namespace {

template <bool OUT_BF16_, int CG_>
struct ChainCfg {
    static constexpr bool OUT_BF16 = OUT_BF16_;
    static constexpr int CG = CG_;
    static constexpr int THREADS = 192;
    static constexpr int BK = 64;                                     // 16-bit K elements per stage
    static constexpr int A_BYTES = TILE_M * 128;                      // 16 KiB
    // A and this CTA's rows of B, or of E: 48 KiB (single CTAs), 32 KiB (pairs)
    static constexpr int STAGE_BYTES = A_BYTES + CHAIN_MAX_N / CG * 128;
    static constexpr int STAGES = CG == 1 ? 4 : 6;
    static constexpr int EPI_BUF = 32 * EPI_COLS * 4;                 // one 32 x 32 fp32 box
    static constexpr int OFF_EPI = STAGES * STAGE_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + 4 * 2 * EPI_BUF;
    // full[STAGES], empty[STAGES], tfull, pready, dfull, dempty, cload[4][2], drain, epi_sync
    static constexpr int NBAR = 2 * STAGES + 4 + 8 + 2;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;               // tmem base slot, abort flag
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;           // + alignment slack
    static constexpr uint32_t T_COL = 0, D_COL = 256;
    static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0 && OFF_EPI % 1024 == 0, "1024-byte aligned");
    static_assert(SMEM_BYTES <= 232448, "shared-memory budget");
    static_assert(CG == 1 || CG == 2, "CTA group");
};

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    chain_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                 const __grid_constant__ CUtensorMap tmE, const ChainParams p) {
    constexpr int STAGES = Cfg::STAGES;
    constexpr int CG = Cfg::CG;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *tfull = bars + 2 * STAGES;   // first product complete (MMA -> epilogue)
    uint64_t *pready = tfull + 1;          // P written into TMEM (epilogue warps of the pair -> MMA)
    uint64_t *dfull = tfull + 2;           // second product complete (MMA -> epilogue, MMA)
    uint64_t *dempty = tfull + 3;          // D read out of TMEM (epilogue warps of the pair -> MMA)
    uint64_t *cload = tfull + 4;
    uint64_t *drain = cload + 8;
    uint64_t *epi_sync = drain + 1;        // every epilogue warp stored its rows of a partial T
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::OFF_MISC + 4);
    const Waiter W{abort_flag, p.status, p.timeout_ns};

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmE);
        prefetch_tensormap(&tmD);
        if (p.has_c) prefetch_tensormap(&tmC);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(pready, 4 * CG);
        mbar_init(dfull, 1);
        mbar_init(dempty, 4 * CG);
        for (int i = 0; i < 8; ++i) mbar_init(&cload[i], 1);
        mbar_init(drain, 1);
        mbar_init(epi_sync, 4);
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
    const int tile0 = blockIdx.x / CG, tile_step = gridDim.x / CG;
    // an epilogue warp's arrival on a barrier the leader's MMA thread waits for
    auto arrive_leader = [&](uint64_t *bar) {
        if constexpr (CG == 1) mbar_arrive(bar);
        else mbar_arrive_remote(mapa_shared(smem_addr(bar), 0));
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            // a pair's copies land in each CTA's own ring and count on the leader's full[s]
            auto load = [&](uint32_t dst, const CUtensorMap *m, uint32_t fb, int c0, int c1) {
                if constexpr (CG == 1) tma_load_2d(dst, m, fb, c0, c1);
                else tma_load_2d_pair(dst, m, mapa_shared(fb, 0), c0, c1);
            };
            ChainIter itr(p, tile0, tile_step);
            Work wk;
            bool first_piece = true;
            while (ok && itr.next(p, wk)) {
                const int m0 = wk.tm * TILE_M * CG + (int)rank * TILE_M;
                // the piece's first-product k-blocks, then (unless it only hands a partial T
                // over) the second product's
                const int n1 = wk.kb1 - wk.kb0, n = n1 + (wk.role == ROLE_EARLY ? 0 : p.num_kb2);
                for (int i = 0; i < n; ++i) {
                    if (!W.wait(&empty[s], ph ^ 1u)) { ok = false; break; }
                    const bool withhold = p.fault == 1 && first_piece && i == 0;
                    uint8_t *st = smem + s * Cfg::STAGE_BYTES;
                    const uint32_t fb = smem_addr(&full[s]);
                    const int kb = i < n1 ? wk.kb0 + i : p.num_kb1 + (i - n1);
                    if (kb < p.num_kb1) {         // A rows m0.., this CTA's n1p/CG rows of B, K block kb
                        if (rank == 0 && !withhold) mbar_arrive_expect_tx(&full[s], CG * Cfg::A_BYTES + p.n1p * 128);
                        const int x = checked_x<2>(p.status, kb * Cfg::BK, p.num_kb1 * Cfg::BK);
                        load(smem_addr(st), &tmA, fb, x, checked_y(p.status, m0, p.tiles * TILE_M * CG));
                        load(smem_addr(st + Cfg::A_BYTES), &tmB, fb, x,
                             checked_y(p.status, (int)rank * (p.n1p / CG), p.n1p));
                    } else {                      // this CTA's n2p/CG rows of E, K block kb - num_kb1
                        if (rank == 0) mbar_arrive_expect_tx(&full[s], p.n2p * 128);
                        load(smem_addr(st), &tmE, fb, checked_x<2>(p.status, (kb - p.num_kb1) * Cfg::BK, p.num_kb2 * Cfg::BK),
                             checked_y(p.status, (int)rank * (p.n2p / CG), p.n2p));
                    }
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
                first_piece = false;
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issue
        if (rank == 0 && lane == 0) {
            const uint32_t t_tmem = tmem_base + Cfg::T_COL;
            const uint32_t d_tmem = tmem_base + Cfg::D_COL;
            int s = 0;
            // it counts pieces (the phases of tfull, pready and dfull), nd the pieces with a
            // second product (the phases of dempty: a piece that only hands its partial T over
            // has no D, and its epilogue does not arrive on dempty)
            uint32_t ph = 0, it = 0, nd = 0;
            bool ok = true;
            // completion of a stage (both CTAs' rings) and of each product (both CTAs' epilogues)
            auto commit_all = [&](uint64_t *bar) {
                if constexpr (CG == 1) tc_commit<1>(smem_addr(bar));
                else tc_commit_pair(smem_addr(bar), 0x3);
            };
            ChainIter itr(p, tile0, tile_step);
            Work wk;
            for (; ok && itr.next(p, wk); ++it) {
                // T's columns are free once the previous piece's second product (which read
                // P from them) has completed, or its partial T has been read out
                if (it > 0 && !W.wait(dfull, (it - 1) & 1u)) break;
                tc_fence_after_sync();
                for (int kb = wk.kb0; kb < wk.kb1; ++kb) {
                    if (!W.wait(&full[s], ph)) { ok = false; break; }
                    tc_fence_after_sync();
                    const uint32_t st = smem_addr(smem + s * Cfg::STAGE_BYTES);
                    const uint64_t ad = smem_desc(st, 16, 1024, SWZ_128B);
                    const uint64_t bd = smem_desc(st + Cfg::A_BYTES, 16, 1024, SWZ_128B);
#pragma unroll
                    for (int k = 0; k < Cfg::BK / 16; ++k)   // 32 bytes of K = 2 descriptor units
                        mma_f16<CG>(t_tmem, ad + 2 * k, bd + 2 * k, p.idesc1, (kb != wk.kb0) | (k != 0));
                    commit_all(&empty[s]);
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                commit_all(tfull);
                // P is in TMEM, and the previous tile's D has been read out (in both CTAs: the
                // peer's epilogue warps release-arrive, so acquire at cluster scope)
                if (!W.wait<CG == 2>(pready, it & 1u)) break;
                if (wk.role != ROLE_EARLY && !W.wait<CG == 2>(dempty, (nd++ & 1u) ^ 1u)) break;
                tc_fence_after_sync();
                for (int j = 0; j < (wk.role == ROLE_EARLY ? 0 : p.num_kb2); ++j) {
                    if (!W.wait(&full[s], ph)) { ok = false; break; }
                    tc_fence_after_sync();
                    const uint64_t ed = smem_desc(smem_addr(smem + s * Cfg::STAGE_BYTES), 16, 1024, SWZ_128B);
#pragma unroll
                    for (int k = 0; k < Cfg::BK / 16; ++k) {
                        const int kk = j * Cfg::BK + 16 * k;   // K index of the second product
                        if (kk < p.n1p) mma_f16_ts<CG>(d_tmem, t_tmem + kk / 2, ed + 2 * k, p.idesc2, kk != 0);
                    }
                    commit_all(&empty[s]);
                    if (++s == STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                commit_all(dfull);
            }
            // every MMA this thread issued has finished before teardown
            tc_commit<CG>(smem_addr(drain));
            W.wait(drain, 0, false);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int e = warp - 2;                           // epilogue warp index
        const int q = warp & 3;                           // TMEM lane window of this warp
        const uint32_t lanes = (uint32_t)(32 * q) << 16;
        uint8_t *ebuf = smem + Cfg::OFF_EPI + e * 2 * Cfg::EPI_BUF;
        uint64_t *cb = cload + 2 * e;
        const uint64_t stream_pol = l2_policy_evict_first();
        const int t_chunks = (p.n1p + 31) / 32;
        const int d_chunks = (p.n2p + EPI_COLS - 1) / EPI_COLS;
        // ec counts the 32 x 32 boxes this warp has stored; box ec uses staging buffer
        // ec % 2, and its C load is that buffer's (ec / 2)-th
        // n_early counts the partial T this CTA has published (the phases of epi_sync)
        uint32_t it = 0, ec = 0, n_early = 0;
        bool ok = true;
        ChainIter itr(p, tile0, tile_step);
        Work wk;
        for (; ok && itr.next(p, wk); ++it) {
            const int m_warp = wk.tm * TILE_M * CG + (int)rank * TILE_M + 32 * q;
            if (!__all_sync(0xffffffffu, W.wait(tfull, it & 1u))) break;
            tc_fence_after_sync();
            // stream-K: the partial T of slot wk.slot, this CTA's 128 rows stored column by column
            // (t_chunks * 32 columns), so that a warp's 32 rows of one column are 128
            // consecutive bytes; `part` points at this thread's row of column 0
            float *part = wk.role == ROLE_TILE ? nullptr
                                               : p.sk_part + (size_t)(wk.slot * CG + (int)rank) * TILE_M * (32 * t_chunks) +
                                                     32 * q + lane;
            if (wk.role == ROLE_EARLY) {
                // hand the partial T over: store it, then publish it once every epilogue
                // warp's stores are visible
                for (int c = 0; c < t_chunks; ++c) {
                    uint32_t acc[32];
                    tmem_ld_32x32b_x32(tmem_base + lanes + Cfg::T_COL + 32 * c, acc);
                    tmem_ld_wait(acc);
#pragma unroll
                    for (int i = 0; i < 32; ++i) part[(size_t)(32 * c + i) * TILE_M] = __uint_as_float(acc[i]);
                }
                __threadfence();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    arrive_leader(pready);                 // T's columns have been read
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
                if (!__all_sync(0xffffffffu, W.wait(dfull, it & 1u))) break;
                continue;
            }
            if (wk.role == ROLE_FINAL) {
                // the rest of this tile's first product, from the unit whose span starts inside it
                const bool got = W.wait_flag(p.sk_flags + wk.slot * CG + (int)rank, p.epoch);
                if (!__all_sync(0xffffffffu, got)) break;
            }
            // P = round(T): chunk c of 32 fp32 columns becomes 16 columns of packed pairs at
            // column 16c, over columns whose T values this warp has already read
            for (int c = 0; c < t_chunks; ++c) {
                uint32_t acc[32];
                tmem_ld_32x32b_x32(tmem_base + lanes + Cfg::T_COL + 32 * c, acc);
                tmem_ld_wait(acc);
                if (wk.role == ROLE_FINAL) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)   // __ldcg: from L2, not a stale L1 line
                        acc[i] = __float_as_uint(__uint_as_float(acc[i]) + __ldcg(part + (size_t)(32 * c + i) * TILE_M));
                }
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float lo = __uint_as_float(acc[2 * i]), hi = __uint_as_float(acc[2 * i + 1]);
                    pk[i] = p.f16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
                }
                tmem_st_32x32b_x16(tmem_base + lanes + Cfg::T_COL + 16 * c, pk);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) arrive_leader(pready);

            // D = C + P·E: 32 x 32 boxes that lie wholly outside D are neither loaded nor stored
            const int chunks_in = m_warp < p.M ? (p.N2 + EPI_COLS - 1) / EPI_COLS : 0;
            const bool use_c = p.has_c && chunks_in > 0;
            if (use_c && lane == 0) {      // the first C box loads while the second product runs
                bulk_wait_group_read0();
                mbar_arrive_expect_tx(&cb[ec & 1u], Cfg::EPI_BUF);
                tma_load_2d_hint(smem_addr(ebuf + (ec & 1u) * Cfg::EPI_BUF), &tmC, smem_addr(&cb[ec & 1u]), 0,
                                 checked_y(p.status, m_warp, p.M), stream_pol);
            }
            if (!__all_sync(0xffffffffu, W.wait(dfull, it & 1u))) break;
            tc_fence_after_sync();
            for (int j = 0; j < d_chunks && ok; ++j) {
                uint32_t acc[32];
                tmem_ld_32x32b_x32(tmem_base + lanes + Cfg::D_COL + EPI_COLS * j, acc);
                tmem_ld_wait(acc);
                if (j == d_chunks - 1) {      // D's columns are free once every chunk is in registers
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) arrive_leader(dempty);
                }
                if (j >= chunks_in) continue;
                const uint32_t cur = ec & 1u;
                uint8_t *buf = ebuf + cur * Cfg::EPI_BUF;
                if (use_c && j + 1 < chunks_in && lane == 0) {
                    const uint32_t nx = cur ^ 1u;
                    bulk_wait_group_read0();                  // the store from buffer nx has read it
                    mbar_arrive_expect_tx(&cb[nx], Cfg::EPI_BUF);
                    tma_load_2d_hint(smem_addr(ebuf + nx * Cfg::EPI_BUF), &tmC, smem_addr(&cb[nx]),
                                     checked_x<4>(p.status, EPI_COLS * (j + 1), p.N2), checked_y(p.status, m_warp, p.M),
                                     stream_pol);
                }
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(acc[i]);
                if (use_c) {
                    if (!__all_sync(0xffffffffu, W.wait(&cb[cur], (ec >> 1) & 1u))) { ok = false; break; }
                    // row `lane` of the 128-byte-swizzled fp32 box: 16-byte chunk c at (c ^ (row % 8))
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float4 cv = ld_shared_v4f(smem_addr(buf + lane * 128 + ((c ^ (lane & 7)) << 4)));
                        v[4 * c + 0] += cv.x;
                        v[4 * c + 1] += cv.y;
                        v[4 * c + 2] += cv.z;
                        v[4 * c + 3] += cv.w;
                    }
                } else if (lane == 0) {
                    bulk_wait_group_read1();                  // the store two boxes back has read this buffer
                }
                __syncwarp();
                if constexpr (Cfg::OUT_BF16) {
                    // 64-byte rows, 64-byte swizzle: chunk c at (c ^ ((row / 2) % 4))
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        st_shared_v4(smem_addr(buf + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)),
                                     pack_bf16x2(v[8 * c + 0], v[8 * c + 1]), pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                                     pack_bf16x2(v[8 * c + 4], v[8 * c + 5]), pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        st_shared_v4(smem_addr(buf + lane * 128 + ((c ^ (lane & 7)) << 4)), __float_as_uint(v[4 * c + 0]),
                                     __float_as_uint(v[4 * c + 1]), __float_as_uint(v[4 * c + 2]),
                                     __float_as_uint(v[4 * c + 3]));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d_hint(&tmD, smem_addr(buf), checked_x<Cfg::OUT_BF16 ? 2 : 4>(p.status, EPI_COLS * j, p.N2),
                                      checked_y(p.status, m_warp, p.M), stream_pol);
                    bulk_commit_group();
                }
                ++ec;
            }
        }
        if (lane == 0) bulk_wait_group0();
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
}

template <class Cfg>
cudaError_t launch_chain(int grid, const CUtensorMap *maps, const ChainParams &p, cudaStream_t stream) {
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute attr[1];
    lc.gridDim = dim3(grid, 1, 1);
    lc.blockDim = dim3(Cfg::THREADS, 1, 1);
    lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
    lc.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = Cfg::CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    void *args[6] = {(void *)&maps[0], (void *)&maps[1], (void *)&maps[2], (void *)&maps[3], (void *)&maps[4],
                     (void *)&p};
    return cudaLaunchKernelExC(&lc, reinterpret_cast<const void *>(&chain_kernel<Cfg>), args);
}

template <class Cfg>
const void *chain_fn() {
    return reinterpret_cast<const void *>(&chain_kernel<Cfg>);
}

const void *chain_fn(int out_bf16, int cta_group) {
    if (cta_group == 2) return out_bf16 ? chain_fn<ChainCfg<true, 2>>() : chain_fn<ChainCfg<false, 2>>();
    return out_bf16 ? chain_fn<ChainCfg<true, 1>>() : chain_fn<ChainCfg<false, 1>>();
}

}  // namespace

int chain_smem_bytes(int cta_group) {
    return cta_group == 2 ? ChainCfg<false, 2>::SMEM_BYTES : ChainCfg<false, 1>::SMEM_BYTES;
}

int chain_stages(int cta_group) { return cta_group == 2 ? ChainCfg<false, 2>::STAGES : ChainCfg<false, 1>::STAGES; }

cudaError_t chain_prepare(int out_bf16, int cta_group) {
    return cudaFuncSetAttribute(chain_fn(out_bf16, cta_group), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                chain_smem_bytes(cta_group));
}

cudaError_t chain_max_active_clusters(int out_bf16, int cta_group, int *clusters) {
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute attr[1];
    lc.gridDim = dim3(2 * 1024, 1, 1);
    lc.blockDim = dim3(192, 1, 1);
    lc.dynamicSmemBytes = chain_smem_bytes(cta_group);
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cta_group;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, chain_fn(out_bf16, cta_group), &lc);
}

cudaError_t chain_launch(int out_bf16, int cta_group, int grid, const CUtensorMap *maps, const ChainParams &p,
                         cudaStream_t stream) {
    if (cta_group == 2)
        return out_bf16 ? launch_chain<ChainCfg<true, 2>>(grid, maps, p, stream)
                        : launch_chain<ChainCfg<false, 2>>(grid, maps, p, stream);
    return out_bf16 ? launch_chain<ChainCfg<true, 1>>(grid, maps, p, stream)
                    : launch_chain<ChainCfg<false, 1>>(grid, maps, p, stream);
}

}  // namespace gb300
