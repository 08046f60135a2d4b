// fp16 / bf16 instances of the tensor-core GEMM (gemm_kernel.cuh):
//   cta_group::1  128 x 256 tiles, 4-stage ring
//   cta_group::2  256 x 256 tiles per CTA pair, 6-stage ring
// each with fp32 or bf16 D.
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
using F16Cfg = TileCfg<CG, OUT_BF16, false, TILE_N, CG == 1 ? GB300_F16_CG1_STAGES : GB300_F16_CG2_STAGES>;

}  // namespace

int f16_stages(int cta_group) { return cta_group == 1 ? F16Cfg<1, false>::STAGES : F16Cfg<2, false>::STAGES; }

int f16_smem_bytes(int cta_group) {
    return cta_group == 1 ? F16Cfg<1, false>::SMEM_BYTES : F16Cfg<2, false>::SMEM_BYTES;
}

cudaError_t f16_prepare(const F16Config &cfg) {
    if (cfg.cta_group == 1) return cfg.out_bf16 ? prepare_tc<F16Cfg<1, true>>() : prepare_tc<F16Cfg<1, false>>();
    return cfg.out_bf16 ? prepare_tc<F16Cfg<2, true>>() : prepare_tc<F16Cfg<2, false>>();
}

cudaError_t f16_max_active_clusters(const F16Config &cfg, int *clusters) {
    if (cfg.cta_group == 1)
        return cfg.out_bf16 ? max_active_clusters_tc<F16Cfg<1, true>>(clusters)
                            : max_active_clusters_tc<F16Cfg<1, false>>(clusters);
    return cfg.out_bf16 ? max_active_clusters_tc<F16Cfg<2, true>>(clusters)
                        : max_active_clusters_tc<F16Cfg<2, false>>(clusters);
}

cudaError_t f16_launch(const F16Config &cfg, const LaunchShape &shape, const CUtensorMap *maps, const KParams &p,
                       cudaStream_t stream) {
    if (cfg.cta_group == 1)
        return cfg.out_bf16 ? launch_tc<F16Cfg<1, true>>(shape, maps, p, stream)
                            : launch_tc<F16Cfg<1, false>>(shape, maps, p, stream);
    return cfg.out_bf16 ? launch_tc<F16Cfg<2, true>>(shape, maps, p, stream)
                        : launch_tc<F16Cfg<2, false>>(shape, maps, p, stream);
}

}  // namespace gb300
