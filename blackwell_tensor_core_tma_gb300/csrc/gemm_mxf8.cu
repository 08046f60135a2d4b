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
#include <cstring>
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

// One CTA packs one 128-row block of scales for 16 consecutive k-blocks: it reads
// the 128 x 64-byte slab of the row-major scale matrix (rows of the block, scale
// columns 64*g .. 64*g+63) into shared memory with coalesced loads, then writes the
// 16 resulting 512-byte blocks (byte lane*16 + Mgroup*4 + sfk) with coalesced
// 16-byte stores.  Blocks of SFA: one per 128 rows of A; blocks of SFB: one per
// 128-row half of each tile_n-wide tile column.  Rows outside the matrix (or
// beyond tile_n in a tile column) and scale columns beyond SFK read as 127.
constexpr int PACK_KB = 16;                 // k-blocks per CTA
constexpr int PACK_COLS = PACK_KB * 4;      // scale bytes per row per CTA

__global__ void __launch_bounds__(256) sf_pack_kernel(const uint8_t *__restrict__ sfa, const uint8_t *__restrict__ sfb,
                                                      uint8_t *__restrict__ out_a, uint8_t *__restrict__ out_b, int M,
                                                      int N, int sfk, int row_blocks, int tiles_n, int num_kb,
                                                      int tile_n) {
    __shared__ __align__(16) uint8_t slab[128][PACK_COLS];
    const int kb_groups = (num_kb + PACK_KB - 1) / PACK_KB;
    const int halves = (tile_n + 127) / 128;
    const int a_ctas = row_blocks * kb_groups;
    int cta = blockIdx.x;
    const bool is_a = cta < a_ctas;
    if (!is_a) cta -= a_ctas;
    const int g = cta % kb_groups;                  // k-block group
    const int blk_row = cta / kb_groups;            // SFA: 128-row block; SFB: tn * halves + h
    const uint8_t *src = is_a ? sfa : sfb;
    // rows of this block in the scale matrix and how many of them are real
    int row0, valid;
    if (is_a) {
        row0 = blk_row * 128;
        valid = min(128, M - row0);
    } else {
        const int tn = blk_row / halves, h = blk_row % halves;
        row0 = tn * tile_n + h * 128;
        valid = min(min(128, tile_n - h * 128), N - row0);
    }
    const int col0 = g * PACK_COLS;
    const bool vec = (sfk % 16 == 0) && ((reinterpret_cast<uintptr_t>(src) & 15) == 0) && col0 + PACK_COLS <= sfk;
    // load: 128 rows x 64 bytes = 512 chunks of 16 bytes, two per thread
    for (int c = threadIdx.x; c < 128 * (PACK_COLS / 16); c += blockDim.x) {
        const int r = c / (PACK_COLS / 16), q = c % (PACK_COLS / 16);
        uint4 v;
        if (r < valid && vec) {
            v = *reinterpret_cast<const uint4 *>(src + (int64_t)(row0 + r) * sfk + col0 + 16 * q);
        } else {
            uint8_t b[16];
            for (int e = 0; e < 16; ++e) {
                const int col = col0 + 16 * q + e;
                b[e] = (r < valid && col < sfk) ? src[(int64_t)(row0 + r) * sfk + col] : kUnitScale;
            }
            memcpy(&v, b, 16);
        }
        *reinterpret_cast<uint4 *>(&slab[r][16 * q]) = v;
    }
    __syncthreads();
    // store: PACK_KB blocks of 512 bytes = 32 lanes x 16 bytes each
    uint8_t *dst_base = is_a ? out_a : out_b;
    for (int u = threadIdx.x; u < PACK_KB * 32; u += blockDim.x) {
        const int kbl = u / 32, lane = u % 32;
        const int kb = g * PACK_KB + kbl;
        if (kb >= num_kb) continue;
        uint32_t w[4];
        for (int mg = 0; mg < 4; ++mg) w[mg] = *reinterpret_cast<const uint32_t *>(&slab[mg * 32 + lane][4 * kbl]);
        int64_t blk;
        if (is_a) {
            blk = (int64_t)blk_row * num_kb + kb;
        } else {
            const int tn = blk_row / halves, h = blk_row % halves;
            blk = ((int64_t)tn * num_kb + kb) * halves + h;
        }
        *reinterpret_cast<uint4 *>(dst_base + blk * 512 + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
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
    (void)sm_count;
    const int sfk = (K + 31) / 32;
    const int kb_groups = (num_kb + PACK_KB - 1) / PACK_KB;
    const int64_t ctas = (int64_t)(row_blocks + tiles_n * ((tile_n + 127) / 128)) * kb_groups;
    sf_pack_kernel<<<(unsigned)ctas, 256, 0, stream>>>(sfa, sfb, out_a, out_b, M, N, sfk, row_blocks, tiles_n, num_kb,
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
