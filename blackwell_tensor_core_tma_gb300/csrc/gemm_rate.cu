// Tensor-pipe rate probe: the dense MMA throughput one SM sustains, in FLOP per SM
// clock, for each instruction shape the GEMM kernels issue.
//
// The GEMM's roofline needs a per-clock peak as well as a measured one: the SM clock
// under a dense tensor load sits well below its maximum (the power limit), so a
// fraction of a FLOP/s figure mixes kernel quality with the clock the run happened to
// get.  This kernel removes everything but the MMA stream: one CTA (or CTA pair) per
// SM, operands resident in shared memory (and scales in TMEM) before the clock starts,
// one thread issuing `iters` groups of four back-to-back tcgen05.mma into one TMEM
// accumulator — the instruction shape, operand layout and accumulate chain of the
// GEMM's own main loop ("Tensor Core 数据布局的演进", section on Blackwell: A and B from
// shared memory, the accumulator in TMEM; "Tensor Memory（TMEM）", allocation) — and a commit that marks
// the end.  Each CTA records the SM clocks and the globaltimer nanoseconds between its
// first issue and the commit's arrival; the ratio of the two is the SM clock of the
// run.  Operand values do not enter the per-clock rate, but they do enter the power the
// tensor pipe draws and so the clock the SM holds: the tiles hold hashed values of
// ordinary magnitude (|x| < 1, finite, both signs) and unit scales, like real data.
#include <algorithm>
#include <vector>

#include "gemm_internal.h"
#include "gemm_kernel.cuh"

namespace gb300 {
namespace {

constexpr int RATE_THREADS = 128;
constexpr int RATE_A_BYTES = 128 * 128;          // 128 rows x 128 bytes of K (one swizzle atom wide)
constexpr int RATE_B_BYTES = 256 * 128;          // up to 256 rows of B
constexpr int RATE_SF_BYTES = 512 * 3;           // one scale word: SFA (128 rows), SFB (2 x 128 columns)
constexpr int RATE_OFF_B = RATE_A_BYTES;
constexpr int RATE_OFF_SF = RATE_OFF_B + RATE_B_BYTES;
constexpr int RATE_OFF_BAR = RATE_OFF_SF + RATE_SF_BYTES;
// more than half an SM's shared memory, so that no two probe CTAs share an SM (and its TMEM)
constexpr int RATE_SMEM = 120 * 1024;
static_assert(RATE_OFF_BAR + 64 + 1024 <= RATE_SMEM, "probe shared memory");

struct RateParams {
    int iters;                      // groups of four MMAs
    uint32_t idesc;                 // instruction descriptor of the probed shape
    uint32_t fill_and, fill_or;     // operand word = (hash & fill_and) | fill_or
    uint32_t sf_word;               // four unit scale codes
    unsigned long long *clk;        // per CTA: SM clocks, globaltimer ns (leaders only)
    int *status;
    uint64_t timeout_ns;
};

// KIND 0: kind::f16 (bf16); 1..3: the block-scaled kinds of mma_scaled.  K bytes per MMA = 32.
template <int KIND, int CG>
__global__ void __launch_bounds__(RATE_THREADS, 1) tc_rate_kernel(const RateParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + RATE_OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + RATE_OFF_BAR + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + RATE_OFF_BAR + 12);
    const int warp = threadIdx.x >> 5;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;

    uint32_t *words = reinterpret_cast<uint32_t *>(smem);
    for (uint32_t i = threadIdx.x; i < RATE_OFF_SF / 4; i += RATE_THREADS) {
        uint32_t h = (i + 0x9E3779B9u * (blockIdx.x + 1)) * 0x85EBCA6Bu;   // an integer hash of the word index
        h ^= h >> 13;
        h *= 0xC2B2AE35u;
        h ^= h >> 16;
        words[i] = (h & p.fill_and) | p.fill_or;
    }
    for (uint32_t i = RATE_OFF_SF / 4 + threadIdx.x; i < RATE_OFF_BAR / 4; i += RATE_THREADS) words[i] = p.sf_word;
    fence_proxy_async_smem();                    // the tiles, visible to the tensor core
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0) {
        tmem_alloc<CG>(smem_addr(tmem_slot), 512);
        tmem_relinquish<CG>();
    }
    tc_fence_before_sync();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const Waiter W{abort_flag, p.status, p.timeout_ns};

    if (threadIdx.x == 0 && rank == 0) {
        const uint64_t ad = smem_desc(smem_addr(smem), 16, 1024, SWZ_128B);
        const uint64_t bd = smem_desc(smem_addr(smem + RATE_OFF_B), 16, 1024, SWZ_128B);
        const uint32_t sfa_t = tmem_base + 256, sfb_t = tmem_base + 260;
        if constexpr (KIND != 0) {
            const uint32_t sf = smem_addr(smem + RATE_OFF_SF);
            tmem_cp_32x128b_warpx4<CG>(sfa_t, smem_desc(sf, 512, 128, SWZ_NONE));
            tmem_cp_32x128b_warpx4<CG>(sfb_t, smem_desc(sf + 512, 512, 128, SWZ_NONE));
            tmem_cp_32x128b_warpx4<CG>(sfb_t + 4, smem_desc(sf + 1024, 512, 128, SWZ_NONE));
        }
        const unsigned long long c0 = clock64();
        const uint64_t g0 = globaltimer_ns();
        for (int i = 0; i < p.iters; ++i) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {           // a stage of the GEMM: 4 x 32 bytes of K
                if constexpr (KIND == 0)
                    mma_f16<CG>(tmem_base, ad + 2 * k, bd + 2 * k, p.idesc, (i | k) != 0);
                else
                    mma_scaled<KIND, CG>(tmem_base, ad + 2 * k, bd + 2 * k, p.idesc, sfa_t, sfb_t, (i | k) != 0);
            }
        }
        if constexpr (CG == 1) tc_commit<1>(smem_addr(bar));
        else tc_commit_pair(smem_addr(bar), 0x3);
        const bool ok = W.wait(bar, 0, false);
        const unsigned long long c1 = clock64();
        const uint64_t g1 = globaltimer_ns();
        p.clk[2 * (blockIdx.x / CG)] = ok ? c1 - c0 : 0ull;
        p.clk[2 * (blockIdx.x / CG) + 1] = ok ? g1 - g0 : 0ull;
    } else if (threadIdx.x == 0) {
        W.wait(bar, 0, false);                   // the pair's MMAs also write this CTA's TMEM
    }
    __syncwarp();
    tc_fence_before_sync();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem_base, 512);
    }
}

template <int KIND, int CG>
cudaError_t rate_launch(int grid, const RateParams &p, cudaStream_t stream, bool query, int *clusters) {
    const void *fn = reinterpret_cast<const void *>(&tc_rate_kernel<KIND, CG>);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, RATE_SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute attr[1];
    lc.gridDim = dim3(query ? 2 * 1024 : grid, 1, 1);    // the occupancy query wants a real grid
    lc.blockDim = dim3(RATE_THREADS, 1, 1);
    lc.dynamicSmemBytes = RATE_SMEM;
    lc.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    if (query) return cudaOccupancyMaxActiveClusters(clusters, fn, &lc);
    void *args[1] = {(void *)&p};
    return cudaLaunchKernelExC(&lc, fn, args);
}

template <int KIND>
cudaError_t rate_dispatch(int cg, int grid, const RateParams &p, cudaStream_t stream, bool query, int *clusters) {
    return cg == 1 ? rate_launch<KIND, 1>(grid, p, stream, query, clusters)
                   : rate_launch<KIND, 2>(grid, p, stream, query, clusters);
}

cudaError_t rate_call(int kind, int cg, int grid, const RateParams &p, cudaStream_t stream, bool query,
                      int *clusters) {
    switch (kind) {
    case 0: return rate_dispatch<0>(cg, grid, p, stream, query, clusters);
    case 1: return rate_dispatch<1>(cg, grid, p, stream, query, clusters);
    case 2: return rate_dispatch<2>(cg, grid, p, stream, query, clusters);
    default: return rate_dispatch<3>(cg, grid, p, stream, query, clusters);
    }
}

double median(std::vector<double> v) {
    std::sort(v.begin(), v.end());
    const size_t n = v.size();
    return n == 0 ? 0.0 : (n % 2 ? v[n / 2] : 0.5 * (v[n / 2 - 1] + v[n / 2]));
}

}  // namespace
}  // namespace gb300

using namespace gb300;

extern "C" gemm_status gemm_measure_tensor_rate(gemm_dtype ab, int block_scaled, int cta_group, int64_t iters,
                                                gemm_tensor_rate *out) {
    if (out == nullptr || (cta_group != 1 && cta_group != 2) || iters < 1 || iters > (1 << 20))
        return GEMM_ERR_INVALID_ARG;
    int kind;
    if ((ab == GEMM_BF16 || ab == GEMM_F16) && block_scaled == GEMM_SCALE_NONE) kind = 0;
    else if (ab == GEMM_E4M3 && block_scaled == GEMM_SCALE_UE8M0_32) kind = 1;
    else if (ab == GEMM_E2M1 && block_scaled == GEMM_SCALE_UE8M0_32) kind = 2;
    else if (ab == GEMM_E2M1 && block_scaled == GEMM_SCALE_UE4M3_16) kind = 3;
    else return block_scaled < 0 || block_scaled > 2 ? GEMM_ERR_INVALID_ARG : GEMM_ERR_UNSUPPORTED;

    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return GEMM_ERR_UNSUPPORTED;

    const uint32_t M = 128u * (uint32_t)cta_group, N = 256u;
    const int mma_k = kind == 0 ? 16 : (kind == 1 ? 32 : 64);
    RateParams p = {};
    p.iters = (int)iters;
    p.idesc = kind == 0 ? idesc_f16(ab == GEMM_BF16 ? 1u : 0u, M, N)
                        : (kind == 1 ? idesc_mxf8(M, N, 0, 0) : idesc_mxf4(M, N, kind == 3));
    p.timeout_ns = 2000000000ull;
    // |x| in [0.5, 1) for bf16 / fp16 (exponent fixed, sign and mantissa hashed); e4m3 with
    // exponent fields 0, 2, 4, 6 (never the NaN code); any e2m1 code (all finite)
    if (kind == 0 && ab == GEMM_BF16) { p.fill_and = 0x807F807Fu; p.fill_or = 0x3F003F00u; }
    else if (kind == 0) { p.fill_and = 0x83FF83FFu; p.fill_or = 0x38003800u; }
    else if (kind == 1) { p.fill_and = 0xB7B7B7B7u; p.fill_or = 0u; }
    else { p.fill_and = 0xFFFFFFFFu; p.fill_or = 0u; }
    p.sf_word = kind == 3 ? 0x38383838u : 0x7F7F7F7Fu;   // UE4M3 1.0 = 0x38, UE8M0 1.0 = 127

    if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;   // the SMs to itself
    int clusters = 0;
    if (rate_call(kind, cta_group, 0, p, nullptr, true, &clusters) != cudaSuccess || clusters < 1)
        clusters = prop.multiProcessorCount / cta_group;   // one CTA per SM: shared memory allows no second
    const int grid = clusters * cta_group;

    cudaStream_t stream = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    void *dbuf = nullptr;
    gemm_status st = GEMM_OK;
    std::vector<unsigned long long> clk((size_t)2 * clusters);
    const size_t clk_bytes = clk.size() * sizeof(unsigned long long);
    int dev_status = 0;
    float ms = 0.f;
    do {
        if (cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess ||
            cudaMalloc(&dbuf, clk_bytes + 16) != cudaSuccess ||
            cudaMemsetAsync(dbuf, 0, clk_bytes + 16, stream) != cudaSuccess) {
            st = GEMM_ERR_CUDA;
            break;
        }
        p.clk = static_cast<unsigned long long *>(dbuf);
        p.status = reinterpret_cast<int *>(static_cast<char *>(dbuf) + clk_bytes);
        if (cudaEventRecord(e0, stream) != cudaSuccess || rate_call(kind, cta_group, grid, p, stream, false, nullptr) != cudaSuccess ||
            cudaEventRecord(e1, stream) != cudaSuccess || cudaStreamSynchronize(stream) != cudaSuccess ||
            cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess ||
            cudaMemcpy(clk.data(), dbuf, clk_bytes, cudaMemcpyDeviceToHost) != cudaSuccess ||
            cudaMemcpy(&dev_status, p.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
            st = GEMM_ERR_CUDA;
            break;
        }
        if (dev_status != 0) {
            st = (gemm_status)dev_status;
            break;
        }
        const double flop_per_group = 4.0 * 2.0 * M * N * mma_k * (double)iters;   // one CTA (pair)
        std::vector<double> per_clk, mhz;
        for (int i = 0; i < clusters; ++i) {
            if (clk[2 * i] == 0 || clk[2 * i + 1] == 0) continue;
            per_clk.push_back(flop_per_group / cta_group / (double)clk[2 * i]);
            mhz.push_back((double)clk[2 * i] / (double)clk[2 * i + 1] * 1e3);
        }
        if ((int)per_clk.size() != clusters) {
            st = GEMM_ERR_TIMEOUT;
            break;
        }
        out->flop_per_clk_per_sm = median(per_clk);
        out->sm_mhz = median(mhz);
        out->tflops = flop_per_group * clusters / (ms * 1e-3) / 1e12;
        out->ms = ms;
        out->sms = grid;
    } while (0);
    if (dbuf) cudaFree(dbuf);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (stream) cudaStreamDestroy(stream);
    return st;
}
