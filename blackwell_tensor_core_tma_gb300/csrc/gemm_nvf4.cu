// Block-scaled 4-bit instances of the tensor-core GEMM (gemm_kernel.cuh):
// e2m1 operands with one UE4M3 scale per 16 K elements: an MMA step of 64 K
// reads a whole four-scale TMEM word (scale_vec::4X, kind::mxf4nvf4).
//
// Operands are OCP E2M1 values packed two per byte along K (element 2t in the
// low nibble of byte t), K-major only; a 128-byte shared-memory row holds 256 K
// elements, so a stage spans 256 K and four MMA steps of 64.  The stage's scales
// arrive packed by sf_pack (gemm_sfpack.cu) and take 16 SFA + 32 SFB columns of the pair's slot (16 + 16 for single CTAs).
#include "gemm_kernel.cuh"

namespace gb300 {
namespace {

// single CTAs: 128 x 128 tiles, two accumulators, five stages, 4 epilogue warps.
// CTA pairs: 256 x 256 tiles, one 256-column accumulator drained to registers by
// 8 epilogue warps, five stages (one epilogue staging buffer per warp), and a copier
// warp that issues the scale copies so that they overlap the MMAs (measured on
// 8192^3: +6 % with two scales per step, +19 % with four).
template <bool OUT_BF16>
using Cfg1 = TileCfg<1, OUT_BF16, KIND_NVF4, 128, 5, 2, 4>;
// pair ring depth and epilogue staging buffers per warp (tuning knobs): one buffer per
// warp frees the shared memory of a fifth stage (measured on 8192^3: e4m3 +3 %, e2m1 +13 %)
#ifndef GB300_NVF4_PAIR_STAGES
#define GB300_NVF4_PAIR_STAGES 5
#endif
#ifndef GB300_NVF4_PAIR_EPI_BUFS
#define GB300_NVF4_PAIR_EPI_BUFS 1
#endif
// warps sharing the scale copies (two: e2m1 with UE4M3 scales +16 % per clock at 8192^3, e4m3 +1 %)
#ifndef GB300_NVF4_PAIR_COPIERS
#define GB300_NVF4_PAIR_COPIERS 2
#endif
template <bool OUT_BF16>
using Cfg2 = TileCfg<2, OUT_BF16, KIND_NVF4, 256, GB300_NVF4_PAIR_STAGES, 1, 8, true, GB300_NVF4_PAIR_EPI_BUFS,
                     32, GB300_NVF4_PAIR_COPIERS>;
using Family = ScaledInstances<Cfg1<false>, Cfg1<true>, Cfg2<false>, Cfg2<true>>;

}  // namespace

const ScaledFamily &family_nvf4() { return Family::family(); }

}  // namespace gb300
