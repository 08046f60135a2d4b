// Block-scaled e4m3 instance of the tensor-core GEMM (gemm_kernel.cuh) and
// the kernel that packs its scale factors.
//
// Block scaling ("Tensor Core 数据布局的演进", section "Block-Scaled MMA 的
// Scale Factors"): SFA[m][sfk] scales row m of A inside K block sfk, SFB[n][sfk]
// column n of B; one UE8M0 scale per 32 K elements (scale_vec::1X).
//
// The MMA reads its scales from TMEM.  The same page gives their TMEM layout
// for 128 rows and 4 K blocks (section "tcgen05.cp 如何写入 TMEM"):
//   S[(4, 32, 4) : (4@TCol, 1@TLane, 1@TCol)] + R[4 : 32@TLane]
// i.e. row m = 32*Mgroup + lane sits in TMEM lane `lane` (replicated to the
// four 32-lane windows by tcgen05.cp .32x128b.warpx4), 32-bit column Mgroup,
// byte sfk.  tcgen05.cp copies 32 rows x 16 bytes from shared memory, so the
// SMEM block for one (128-row block, 4-K-block group) is 512 bytes with byte
//   lane*16 + Mgroup*4 + sfk.
// sf_pack_kernel writes the caller's row-major SFA (M x SFK) and SFB (N x SFK)
// in exactly that order into the plan's workspace, one 512-byte block per
// (128-row block, k-block of 128 elements), so that the producer copies a
// stage's scales with one TMA copy per operand (the workspace is viewed as
// rows of 128 bytes).  Rows or K blocks past the
// matrix get scale code 127 (2^0): they multiply the zero-filled operand
// elements of the edge tiles.
//
// Each stage's scales take a 12-column TMEM slot (4 SFA + 8 SFB columns).  In
// a CTA pair each CTA holds the SFA of its own 128 rows and the SFB of all the
// tile's columns.
#include <type_traits>

#include "gemm_kernel.cuh"

namespace gb300 {
namespace {

// single CTAs: 128 x 224 tiles, two accumulators (448 TMEM columns) and four
// stages of 12-column scale slots, 4 epilogue warps.
// CTA pairs: 256 x 256 tiles (an MMA of N = 256 keeps the tensor pipe busiest),
// one 256-column accumulator that 8 epilogue warps copy to registers and free
// at once, the other 256 TMEM columns for the stages' scale slots.
template <int CG, bool OUT_BF16>
using MxCfg = typename std::conditional<CG == 1, TileCfg<1, OUT_BF16, true, 224, 4, 2, 4>,
                                        TileCfg<2, OUT_BF16, true, 256, 4, 1, 8>>::type;

constexpr uint8_t kUnitScale = 127;

// one thread per 16-byte row of a 512-byte block
__global__ void sf_pack_kernel(const uint8_t *__restrict__ sfa, const uint8_t *__restrict__ sfb,
                               uint8_t *__restrict__ out_a, uint8_t *__restrict__ out_b, int M, int N, int sfk,
                               int tiles_m, int tiles_n, int num_kb, int tile_n) {
    const int64_t a_rows = (int64_t)tiles_m * num_kb * 32;
    const int64_t halves = (tile_n + 127) / 128;
    const int64_t b_rows = (int64_t)tiles_n * num_kb * halves * 32;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < a_rows + b_rows;
         i += (int64_t)gridDim.x * blockDim.x) {
        const bool is_a = i < a_rows;
        const int64_t r = is_a ? i : i - a_rows;
        const int lane = (int)(r & 31);
        const int64_t blk = r >> 5;                     // 512-byte block index
        uint32_t w[4];
        if (is_a) {
            const int kb = (int)(blk % num_kb);
            const int mb = (int)(blk / num_kb);
            for (int mg = 0; mg < 4; ++mg) {
                const int row = mb * 128 + mg * 32 + lane;
                uint32_t word = 0;
                for (int s = 0; s < 4; ++s) {
                    const int col = kb * 4 + s;
                    const uint32_t v = (row < M && col < sfk) ? sfa[(int64_t)row * sfk + col] : kUnitScale;
                    word |= v << (8 * s);
                }
                w[mg] = word;
            }
        } else {
            const int h = (int)(blk % halves);
            const int kb = (int)((blk / halves) % num_kb);
            const int tn = (int)(blk / halves / num_kb);
            for (int mg = 0; mg < 4; ++mg) {
                const int in_tile = h * 128 + mg * 32 + lane;
                const int row = tn * tile_n + in_tile;
                uint32_t word = 0;
                for (int s = 0; s < 4; ++s) {
                    const int col = kb * 4 + s;
                    const uint32_t v =
                        (in_tile < tile_n && row < N && col < sfk) ? sfb[(int64_t)row * sfk + col] : kUnitScale;
                    word |= v << (8 * s);
                }
                w[mg] = word;
            }
        }
        uint8_t *dst = (is_a ? out_a : out_b) + blk * 512 + lane * 16;
        *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace

int mxf8_stages(int cta_group) { return cta_group == 1 ? MxCfg<1, false>::STAGES : MxCfg<2, false>::STAGES; }

int mxf8_smem_bytes(int cta_group) {
    return cta_group == 1 ? MxCfg<1, false>::SMEM_BYTES : MxCfg<2, false>::SMEM_BYTES;
}

size_t mxf8_workspace_a(int row_blocks, int num_kb) { return (size_t)row_blocks * num_kb * MxCfg<1, false>::SFA_BYTES; }

size_t mxf8_workspace_b(int tiles_n, int num_kb) { return (size_t)tiles_n * num_kb * MxCfg<1, false>::SFB_BYTES; }

int mxf8_sfb_block_bytes() { return MxCfg<1, false>::SFB_BYTES; }

int mxf8_tile_n(int cta_group) { return cta_group == 1 ? MxCfg<1, false>::BN : MxCfg<2, false>::BN; }

cudaError_t mxf8_prepare(int cta_group, int out_bf16) {
    if (cta_group == 1) return out_bf16 ? prepare_tc<MxCfg<1, true>>() : prepare_tc<MxCfg<1, false>>();
    return out_bf16 ? prepare_tc<MxCfg<2, true>>() : prepare_tc<MxCfg<2, false>>();
}

cudaError_t mxf8_max_active_clusters(int cta_group, int out_bf16, int *clusters) {
    if (cta_group == 1)
        return out_bf16 ? max_active_clusters_tc<MxCfg<1, true>>(clusters)
                        : max_active_clusters_tc<MxCfg<1, false>>(clusters);
    return out_bf16 ? max_active_clusters_tc<MxCfg<2, true>>(clusters)
                    : max_active_clusters_tc<MxCfg<2, false>>(clusters);
}

cudaError_t mxf8_pack(const uint8_t *sfa, const uint8_t *sfb, uint8_t *out_a, uint8_t *out_b, int M, int N, int K,
                      int row_blocks, int tiles_n, int tile_n, int num_kb, int sm_count, cudaStream_t stream) {
    const int sfk = (K + 31) / 32;
    const int64_t rows = ((int64_t)row_blocks * num_kb + (int64_t)tiles_n * num_kb * ((tile_n + 127) / 128)) * 32;
    int blocks = (int)((rows + 255) / 256);
    if (blocks > 8 * sm_count) blocks = 8 * sm_count;
    sf_pack_kernel<<<blocks, 256, 0, stream>>>(sfa, sfb, out_a, out_b, M, N, sfk, row_blocks, tiles_n, num_kb,
                                               tile_n);
    return cudaGetLastError();
}

cudaError_t mxf8_launch(int cta_group, int out_bf16, const LaunchShape &shape, const CUtensorMap *maps,
                        const KParams &p, cudaStream_t stream) {
    if (cta_group == 1)
        return out_bf16 ? launch_tc<MxCfg<1, true>>(shape, maps, p, stream)
                        : launch_tc<MxCfg<1, false>>(shape, maps, p, stream);
    return out_bf16 ? launch_tc<MxCfg<2, true>>(shape, maps, p, stream)
                    : launch_tc<MxCfg<2, false>>(shape, maps, p, stream);
}

}  // namespace gb300
