// Host/device shared declarations of the GEMM library (not part of the C ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "gb300gemm.h"

namespace gb300 {

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
};
int f16_stages(int cta_group);
int f16_smem_bytes(int cta_group);
cudaError_t f16_prepare(const F16Config &cfg);   // set the kernel's shared-memory limit
cudaError_t f16_max_active_clusters(const F16Config &cfg, int *clusters);
cudaError_t f16_launch(const F16Config &cfg, const LaunchShape &shape, const CUtensorMap *maps,
                       const KParams &p, cudaStream_t stream);

// split-K preparation (gemm_f16.cu): D = C, or D = 0 without C (fp32, n elements, n % 4 == 0)
cudaError_t init_d_launch(float *D, const float *C, size_t n, int sm_count, cudaStream_t stream);

// block-scaled e4m3 kernel family (gemm_mxf8.cu)
int mxf8_tile_n(int cta_group);
int mxf8_stages(int cta_group);
int mxf8_smem_bytes(int cta_group);
size_t mxf8_workspace_a(int row_blocks, int num_kb);
size_t mxf8_workspace_b(int tiles_n, int num_kb);
int mxf8_sfb_block_bytes();
cudaError_t mxf8_prepare(int cta_group, int out_bf16);
cudaError_t mxf8_max_active_clusters(int cta_group, int out_bf16, int *clusters);
cudaError_t mxf8_pack(const uint8_t *sfa, const uint8_t *sfb, uint8_t *out_a, uint8_t *out_b, int M, int N, int K,
                      int row_blocks, int tiles_n, int tile_n, int num_kb, int sm_count, cudaStream_t stream);
cudaError_t mxf8_launch(int cta_group, int out_bf16, const LaunchShape &shape, const CUtensorMap *maps,
                        const KParams &p, cudaStream_t stream);

constexpr int TILE_M = 128;   // rows of D per CTA
constexpr int TILE_N = 256;   // columns of D per CTA (and per CTA pair)
constexpr int TILE_K16 = 64;  // 16-bit K elements per stage (one 128-byte swizzle row)
constexpr int EPI_COLS = 32;  // epilogue chunk width (columns)

}  // namespace gb300
