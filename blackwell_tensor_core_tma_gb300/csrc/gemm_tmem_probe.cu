// Test-only probes (include/gb300gemm_testing.h).
//
// TMEM data movement (gemm_testing_tmem_ld_probe): runs the pages' own tcgen05.ld example shapes on the
// GPU so that their register counts and lane windows can be checked against the
// oracle's layout maps ("Tensor Memory（TMEM）", sections "每个 warp 能访问哪些 TMEM
// lanes" and "Shape 和 Repeat Factor": a .16x128b access moves 16 lanes x 128 bits
// per repeat, .num repeats along the columns, and the warp's 32 threads share the
// cells evenly; warp w of a warpgroup reaches lanes 32w..32w+31 only).
//
// One CTA of one warpgroup allocates 512 columns; each warp writes, with
// tcgen05.st.32x32b, the code (lane << 16) | column into every cell of its own
// 32-lane window, then reads its window back with .16x128b.x1 / .x2 / .x4 / .x8
// (at the window's first lane, columns 0, 32, 64 and 128) and with .32x32b.x32
// (column 256), and writes every register to global memory.
#include <cstdint>

#include "gemm_internal.h"
#include "ptx.cuh"

namespace gb300 {
namespace {

constexpr int PROBE_REGS = 2 + 4 + 8 + 16 + 32;   // registers one thread receives over the five loads

template <int N>
__device__ __forceinline__ void tmem_ld_16x128b(uint32_t taddr, uint32_t (&r)[2 * N]) {
    static_assert(N == 1 || N == 2 || N == 4 || N == 8, "repeat factor");
    if constexpr (N == 1)
        asm volatile("tcgen05.ld.sync.aligned.16x128b.x1.b32 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(taddr));
    else if constexpr (N == 2)
        asm volatile("tcgen05.ld.sync.aligned.16x128b.x2.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(taddr));
    else if constexpr (N == 4)
        asm volatile("tcgen05.ld.sync.aligned.16x128b.x4.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                       "=r"(r[7])
                     : "r"(taddr));
    else
        asm volatile(
            "tcgen05.ld.sync.aligned.16x128b.x8.b32 "
            "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr));
}

__global__ void __launch_bounds__(128, 1) tmem_probe_kernel(uint32_t *out) {
    __shared__ uint32_t tmem_slot;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        tmem_alloc<1>(smem_addr(&tmem_slot), 512);
        tmem_relinquish<1>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t base = tmem_slot;
    const uint32_t window = (uint32_t)(32 * warp) << 16;    // lane field of this warp's window
    // every cell of the window: (lane << 16) | column, this thread's lane = 32 * warp + lane
    for (int c0 = 0; c0 < 512; c0 += 16) {
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = ((uint32_t)(32 * warp + lane) << 16) | (uint32_t)(c0 + i);
        tmem_st_32x32b_x16(base + window + (uint32_t)c0, v);
    }
    tmem_st_wait();
    uint32_t r1[2], r2[4], r4[8], r8[16], r32[32];
    tmem_ld_16x128b<1>(base + window + 0, r1);
    tmem_ld_16x128b<2>(base + window + 32, r2);
    tmem_ld_16x128b<4>(base + window + 64, r4);
    tmem_ld_16x128b<8>(base + window + 128, r8);
    tmem_ld_32x32b_x32(base + window + 256, r32);
    tmem_ld_wait_all();
    uint32_t *o = out + ((size_t)warp * 32 + lane) * PROBE_REGS;
    int k = 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) o[k++] = r1[i];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[k++] = r2[i];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[k++] = r4[i];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[k++] = r8[i];
#pragma unroll
    for (int i = 0; i < 32; ++i) o[k++] = r32[i];
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc<1>(base, 512);
    }
}

// Epilogue staging patterns (test-only, gemm_testing_staging_probe): each of four warps
// issues `iters` rounds of 128-bit shared-memory accesses in one pattern, in its own
// 4 KiB buffer, and thread 0 of each warp records the SM clocks the rounds took.
//   0  bf16 D staging: row `lane` of 64 bytes, 16-byte chunk c at c ^ ((lane / 2) % 4)
//   1  fp32 C / D staging: row `lane` of 128 bytes, chunk c at c ^ (lane % 8)
//   2  linear: chunk c of lane at c * 512 + lane * 16 (a warp writes 512 contiguous bytes)
//   3  bf16 rows without the swizzle (chunk c at c)
//   4  fp32 rows without the swizzle
template <int P, bool LOAD>
__global__ void __launch_bounds__(128, 1) staging_probe_kernel(int iters, unsigned long long *clk, uint32_t *sink) {
    __shared__ __align__(1024) uint8_t buf[4 * 4096];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t base = smem_addr(buf + warp * 4096);
    constexpr int CHUNKS = (P == 0 || P == 3) ? 4 : 8;
    uint32_t acc = 0;
    __syncwarp();
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c) {
            uint32_t off;
            if constexpr (P == 0) off = lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4);
            else if constexpr (P == 1) off = lane * 128 + ((c ^ (lane & 7)) << 4);
            else if constexpr (P == 2) off = c * 512 + lane * 16;
            else if constexpr (P == 3) off = lane * 64 + c * 16;
            else off = lane * 128 + c * 16;
            if constexpr (LOAD) {
                const float4 v = ld_shared_v4f(base + off);
                acc += __float_as_uint(v.x) ^ __float_as_uint(v.w);
            } else {
                st_shared_v4(base + off, (uint32_t)it, (uint32_t)c, (uint32_t)lane, acc);
            }
        }
    }
    __syncwarp();
    const long long t1 = clock64();
    if (lane == 0) clk[warp] = (unsigned long long)(t1 - t0);
    if (acc == 0x9E3779B9u) sink[threadIdx.x] = acc;   // keeps the loads
}

template <int P>
cudaError_t staging_launch(int load, int iters, unsigned long long *clk, uint32_t *sink) {
    if (load) staging_probe_kernel<P, true><<<1, 128>>>(iters, clk, sink);
    else staging_probe_kernel<P, false><<<1, 128>>>(iters, clk, sink);
    return cudaGetLastError();
}

}  // namespace
}  // namespace gb300

using namespace gb300;

// Test hook (declared in include/gb300gemm_testing.h).
extern "C" gemm_status gemm_testing_staging_probe(int pattern, int load, int64_t iters, double *clk_per_access) {
    if (!clk_per_access || pattern < 0 || pattern > 4 || (load != 0 && load != 1) || iters < 1 || iters > (1 << 20))
        return GEMM_ERR_INVALID_ARG;
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return GEMM_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return GEMM_ERR_UNSUPPORTED;
    void *d = nullptr;
    if (cudaMalloc(&d, 4 * sizeof(unsigned long long) + 128 * sizeof(uint32_t)) != cudaSuccess) return GEMM_ERR_CUDA;
    unsigned long long *clk = static_cast<unsigned long long *>(d);
    uint32_t *sink = reinterpret_cast<uint32_t *>(clk + 4);
    cudaError_t e;
    switch (pattern) {
    case 0: e = staging_launch<0>(load, (int)iters, clk, sink); break;
    case 1: e = staging_launch<1>(load, (int)iters, clk, sink); break;
    case 2: e = staging_launch<2>(load, (int)iters, clk, sink); break;
    case 3: e = staging_launch<3>(load, (int)iters, clk, sink); break;
    default: e = staging_launch<4>(load, (int)iters, clk, sink); break;
    }
    unsigned long long h[4] = {0, 0, 0, 0};
    gemm_status st = GEMM_OK;
    if (e != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(h, clk, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess)
        st = GEMM_ERR_CUDA;
    cudaFree(d);
    if (st != GEMM_OK) return st;
    const int chunks = (pattern == 0 || pattern == 3) ? 4 : 8;
    unsigned long long mx = 0;
    for (unsigned long long v : h) mx = v > mx ? v : mx;
    *clk_per_access = (double)mx / ((double)iters * chunks);
    return GEMM_OK;
}

// Test hook (declared in include/gb300gemm_testing.h).
extern "C" gemm_status gemm_testing_tmem_ld_probe(uint32_t *host_out, int64_t n_words) {
    const int64_t words = (int64_t)128 * PROBE_REGS;
    if (!host_out || n_words < words) return GEMM_ERR_INVALID_ARG;
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return GEMM_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return GEMM_ERR_UNSUPPORTED;
    uint32_t *d = nullptr;
    if (cudaMalloc(&d, (size_t)words * sizeof(uint32_t)) != cudaSuccess) return GEMM_ERR_CUDA;
    gemm_status st = GEMM_OK;
    tmem_probe_kernel<<<1, 128>>>(d);
    if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(host_out, d, (size_t)words * sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        st = GEMM_ERR_CUDA;
    cudaFree(d);
    return st;
}
