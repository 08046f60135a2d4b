// fp16 / bf16 instances of the tensor-core GEMM (gemm_kernel.cuh):
//   cta_group::1  128 x 256 tiles, 4-stage ring
//   cta_group::2  256 x 256 tiles per CTA pair, 6-stage ring
// each with fp32 or bf16 D, and for pairs with fp32 D a wide-epilogue form: 8 epilogue
// warps (two per TMEM lane window, each half of the tile's columns) and 5 stages, for
// short K, where storing a tile (C in, D out, 512 KiB per pair) takes longer than the
// next tile's main loop (measured: +14 % at 4096x4096x1024, +3.5 % at 4000x3000x2056,
// -2 % at 4096^3, so the plan chooses it for at most 40 k-blocks); and for pairs a
// 256 x 224 tile (6 stages, 4 epilogue warps) that a plan takes when its tiles fill the
// persistent waves clearly better than 256 x 256 ones (4096^3: 304 tiles = 4 waves of 76
// pairs instead of 256 = 3.4; measured +6 %; at 8192^3 the extra operand bytes per FLOP
// cost 3.5 %); and for single CTAs that each take at most one short tile (small problems,
// whose run is mostly the one tile's epilogue) a wide-epilogue form with 8 epilogue warps
// and 3 stages, either D type.
#include "gemm_kernel.cuh"

// ring depths (tuning knobs; the defaults fill shared memory)
#ifndef GB300_F16_CG1_STAGES
#define GB300_F16_CG1_STAGES 4
#endif
#ifndef GB300_F16_CG2_STAGES
#define GB300_F16_CG2_STAGES 6
#endif

namespace gb300 {
namespace {

template <int CG, bool OUT_BF16>
using F16Cfg = TileCfg<CG, OUT_BF16, KIND_F16, TILE_N, CG == 1 ? GB300_F16_CG1_STAGES : GB300_F16_CG2_STAGES>;
using F16Wide = TileCfg<2, false, KIND_F16, TILE_N, 5, 2, 8>;
template <bool OUT_BF16>
using F16Wide1 = TileCfg<1, OUT_BF16, KIND_F16, TILE_N, 3, 2, 8>;
template <bool OUT_BF16>
using F16Narrow = TileCfg<2, OUT_BF16, KIND_F16, F16_NARROW_N, GB300_F16_CG2_STAGES>;
bool narrow(const F16Config &cfg) { return cfg.cta_group == 2 && cfg.tile_n == F16_NARROW_N; }
bool wide(const F16Config &cfg) { return !narrow(cfg) && cfg.wide_epi && cfg.cta_group == 2 && !cfg.out_bf16; }
bool wide1(const F16Config &cfg) { return cfg.wide_epi && cfg.cta_group == 1; }

// D = C (or 0): the starting value split-K slices add their partial products to
__global__ void init_d_kernel(float4 *__restrict__ D, const float4 *__restrict__ C, size_t n4) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
        D[i] = C ? C[i] : make_float4(0.f, 0.f, 0.f, 0.f);
}

}  // namespace

cudaError_t init_d_launch(float *D, const float *C, size_t n, int sm_count, cudaStream_t stream) {
    const size_t n4 = n / 4;
    size_t blocks = (n4 + 255) / 256;
    if (blocks > (size_t)sm_count * 8) blocks = (size_t)sm_count * 8;
    if (blocks == 0) blocks = 1;
    init_d_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<float4 *>(D),
                                                         reinterpret_cast<const float4 *>(C), n4);
    return cudaGetLastError();
}

int f16_stages(const F16Config &cfg) {
    if (narrow(cfg)) return F16Narrow<false>::STAGES;
    if (wide(cfg)) return F16Wide::STAGES;
    if (wide1(cfg)) return F16Wide1<false>::STAGES;
    return cfg.cta_group == 1 ? F16Cfg<1, false>::STAGES : F16Cfg<2, false>::STAGES;
}

int f16_smem_bytes(const F16Config &cfg) {
    if (narrow(cfg)) return F16Narrow<false>::SMEM_BYTES;
    if (wide(cfg)) return F16Wide::SMEM_BYTES;
    if (wide1(cfg)) return F16Wide1<false>::SMEM_BYTES;
    return cfg.cta_group == 1 ? F16Cfg<1, false>::SMEM_BYTES : F16Cfg<2, false>::SMEM_BYTES;
}

cudaError_t f16_prepare(const F16Config &cfg) {
    if (narrow(cfg)) return cfg.out_bf16 ? prepare_tc<F16Narrow<true>>() : prepare_tc<F16Narrow<false>>();
    if (wide(cfg)) return prepare_tc<F16Wide>();
    if (wide1(cfg)) return cfg.out_bf16 ? prepare_tc<F16Wide1<true>>() : prepare_tc<F16Wide1<false>>();
    if (cfg.cta_group == 1) return cfg.out_bf16 ? prepare_tc<F16Cfg<1, true>>() : prepare_tc<F16Cfg<1, false>>();
    return cfg.out_bf16 ? prepare_tc<F16Cfg<2, true>>() : prepare_tc<F16Cfg<2, false>>();
}

cudaError_t f16_max_active_clusters(const F16Config &cfg, int *clusters) {
    if (narrow(cfg))
        return cfg.out_bf16 ? max_active_clusters_tc<F16Narrow<true>>(clusters)
                            : max_active_clusters_tc<F16Narrow<false>>(clusters);
    if (wide(cfg)) return max_active_clusters_tc<F16Wide>(clusters);
    if (wide1(cfg))
        return cfg.out_bf16 ? max_active_clusters_tc<F16Wide1<true>>(clusters)
                            : max_active_clusters_tc<F16Wide1<false>>(clusters);
    if (cfg.cta_group == 1)
        return cfg.out_bf16 ? max_active_clusters_tc<F16Cfg<1, true>>(clusters)
                            : max_active_clusters_tc<F16Cfg<1, false>>(clusters);
    return cfg.out_bf16 ? max_active_clusters_tc<F16Cfg<2, true>>(clusters)
                        : max_active_clusters_tc<F16Cfg<2, false>>(clusters);
}

cudaError_t f16_launch(const F16Config &cfg, const LaunchShape &shape, const CUtensorMap *maps, const KParams &p,
                       cudaStream_t stream) {
    if (narrow(cfg))
        return cfg.out_bf16 ? launch_tc<F16Narrow<true>>(shape, maps, p, stream)
                            : launch_tc<F16Narrow<false>>(shape, maps, p, stream);
    if (wide(cfg)) return launch_tc<F16Wide>(shape, maps, p, stream);
    if (wide1(cfg))
        return cfg.out_bf16 ? launch_tc<F16Wide1<true>>(shape, maps, p, stream)
                            : launch_tc<F16Wide1<false>>(shape, maps, p, stream);
    if (cfg.cta_group == 1)
        return cfg.out_bf16 ? launch_tc<F16Cfg<1, true>>(shape, maps, p, stream)
                            : launch_tc<F16Cfg<1, false>>(shape, maps, p, stream);
    return cfg.out_bf16 ? launch_tc<F16Cfg<2, true>>(shape, maps, p, stream)
                        : launch_tc<F16Cfg<2, false>>(shape, maps, p, stream);
}

}  // namespace gb300
