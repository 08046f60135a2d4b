// Block-scaled e4m3 instances of the tensor-core GEMM (gemm_kernel.cuh).
//
// Block scaling ("Tensor Core 数据布局的演进", section "Block-Scaled MMA 的
// Scale Factors"): SFA[m][sfk] scales row m of A inside K block sfk, SFB[n][sfk]
// column n of B; one UE8M0 scale per 32 K elements, so an MMA step of 32 K reads
// one scale byte of a four-scale TMEM word (scale_vec::1X).  The scales arrive
// packed by sf_pack (gemm_sfpack.cu); each stage's scales take a 12-column TMEM
// slot (4 SFA + 8 SFB columns).  In a CTA pair each CTA holds the SFA of its own
// 128 rows and the SFB of all the tile's columns.
#include "gemm_kernel.cuh"

namespace gb300 {
namespace {

// single CTAs: 128 x 224 tiles, two accumulators (448 TMEM columns) and four
// stages of 12-column scale slots, 4 epilogue warps.
// CTA pairs: 256 x 256 tiles (the fewest operand bytes per FLOP that TMEM allows
// alongside the scale slots), one 256-column accumulator that 8 epilogue warps
// copy to registers and free at once, the other 256 TMEM columns for the stages'
// scale slots, and a copier warp that issues the scale copies (measured on 8192^3:
// +8.5 % over copies issued by the MMA thread).
template <bool OUT_BF16>
using Mx1 = TileCfg<1, OUT_BF16, KIND_MXF8, 224, 4, 2, 4>;
// pair ring depth and epilogue staging buffers per warp (tuning knobs): one buffer per
// warp frees the shared memory of a fifth stage (measured on 8192^3: e4m3 +3 %, e2m1 +13 %)
#ifndef GB300_MXF8_PAIR_STAGES
#define GB300_MXF8_PAIR_STAGES 6
#endif
#ifndef GB300_MXF8_PAIR_EPI_BUFS
#define GB300_MXF8_PAIR_EPI_BUFS 1
#endif
// columns of the epilogue's staging boxes: 16 halves the staging (8 warps x 2 KiB) so that
// a sixth stage fits
#ifndef GB300_MXF8_PAIR_EPI_BOX
#define GB300_MXF8_PAIR_EPI_BOX 16
#endif
// warps sharing the scale copies (two: e2m1 with UE4M3 scales +16 % per clock at 8192^3, e4m3 +1 %)
#ifndef GB300_MXF8_PAIR_COPIERS
#define GB300_MXF8_PAIR_COPIERS 2
#endif
template <bool OUT_BF16>
using Mx2 = TileCfg<2, OUT_BF16, KIND_MXF8, 256, GB300_MXF8_PAIR_STAGES, 1, 8, true, GB300_MXF8_PAIR_EPI_BUFS,
                    GB300_MXF8_PAIR_EPI_BOX, GB300_MXF8_PAIR_COPIERS>;
// narrow CTA pairs: 256 x 224 tiles with two accumulators (448 TMEM columns, five stages of
// 12-column scale slots) drained by 4 epilogue warps while the next tile accumulates, for
// shapes whose 256-wide tiles fill the persistent rounds badly or run short K (the plan's
// rule, e4m3_pair_tile_n; measured on 4096^3: +16 %, 4096 x 4096 x 8192: +6 %)
#ifndef GB300_MXF8_NARROW_STAGES
#define GB300_MXF8_NARROW_STAGES 5
#endif
template <bool OUT_BF16>
using Mx2N = TileCfg<2, OUT_BF16, KIND_MXF8, MXF8_NARROW_N, GB300_MXF8_NARROW_STAGES, 2, 4, true, 2, 32, 2>;
using MxF8 = ScaledInstances<Mx1<false>, Mx1<true>, Mx2<false>, Mx2<true>, Mx2N<false>, Mx2N<true>>;

}  // namespace

const ScaledFamily &family_mxf8() { return MxF8::family(); }

}  // namespace gb300
