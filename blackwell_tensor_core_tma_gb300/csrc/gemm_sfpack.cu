// Packing of block scales for the block-scaled tensor-core kernels.
//
// The MMA reads its scales from TMEM ("Tensor Core 数据布局的演进", section
// "tcgen05.cp 如何写入 TMEM"), in the layout the page gives for 128 rows and four
// scales per row:
//   S[(4, 32, 4) : (4@TCol, 1@TLane, 1@TCol)] + R[4 : 32@TLane]
// i.e. row m = 32*Mgroup + lane sits in TMEM lane `lane` (replicated to the four
// 32-lane windows by tcgen05.cp .32x128b.warpx4), 32-bit column Mgroup, byte =
// scale index within the word.  tcgen05.cp copies 32 rows x 16 bytes from shared
// memory, so the SMEM block for one (128-row block, word of four scales) is 512
// bytes with byte lane*16 + Mgroup*4 + j.  A kernel stage consumes SF_WORDS such
// words per row (1 for e4m3 with one scale per 32 K, 2 for e2m1 with one per 32, 4
// for e2m1 with one per 16: section "scale_vec 的 Word 内复制").
//
// sf_pack_kernel writes the caller's row-major SFA (M x sfk) and SFB (N x sfk) in
// that order into a plan's workspace, so that the producer copies a stage's scales
// with one TMA copy per operand (the workspace viewed as rows of 128 bytes).  Rows
// or scale columns past the matrix get the scale format's 1.0: they multiply the
// zero-filled operand elements of the edge tiles.
#include <cstring>

#include "gemm_internal.h"

namespace gb300 {
namespace {

// One CTA packs one 128-row block of scales for 16 consecutive word groups (four
// scale columns each): it reads the 128 x 64-byte slab of the row-major scale
// matrix (rows of the block, scale columns 64*g .. 64*g+63) into shared memory with
// coalesced loads, then writes the 16 resulting 512-byte blocks (byte
// lane*16 + Mgroup*4 + column-in-group) with coalesced 16-byte stores.  Blocks of
// SFA: one per (128 rows of A, word group); blocks of SFB: one per (tile column,
// word group, 128-row group of the tile column), so that a stage's words follow
// each other.  Rows outside the matrix (or beyond tile_n in a tile column) and
// scale columns beyond sfk read as `pad`.
constexpr int PACK_WG = 16;                 // word groups per CTA
constexpr int PACK_COLS = PACK_WG * 4;      // scale bytes per row per CTA

__global__ void __launch_bounds__(256) sf_pack_kernel(const uint8_t *__restrict__ sfa, const uint8_t *__restrict__ sfb,
                                                      uint8_t *__restrict__ out_a, uint8_t *__restrict__ out_b, int M,
                                                      int N, int sfk, int row_blocks, int tiles_n, int n_wg,
                                                      int tile_n, uint8_t pad) {
    __shared__ __align__(16) uint8_t slab[128][PACK_COLS];
    const int wg_groups = (n_wg + PACK_WG - 1) / PACK_WG;
    const int halves = (tile_n + 127) / 128;
    const int a_ctas = row_blocks * wg_groups;
    int cta = blockIdx.x;
    const bool is_a = cta < a_ctas;
    if (!is_a) cta -= a_ctas;
    const int g = cta % wg_groups;                  // group of PACK_WG word groups
    const int blk_row = cta / wg_groups;            // SFA: 128-row block; SFB: tn * halves + h
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
                b[e] = (r < valid && col < sfk) ? src[(int64_t)(row0 + r) * sfk + col] : pad;
            }
            memcpy(&v, b, 16);
        }
        *reinterpret_cast<uint4 *>(&slab[r][16 * q]) = v;
    }
    __syncthreads();
    // store: PACK_WG blocks of 512 bytes = 32 lanes x 16 bytes each
    uint8_t *dst_base = is_a ? out_a : out_b;
    for (int u = threadIdx.x; u < PACK_WG * 32; u += blockDim.x) {
        const int wl = u / 32, lane = u % 32;
        const int wg = g * PACK_WG + wl;
        if (wg >= n_wg) continue;
        uint32_t w[4];
        for (int mg = 0; mg < 4; ++mg) w[mg] = *reinterpret_cast<const uint32_t *>(&slab[mg * 32 + lane][4 * wl]);
        int64_t blk;
        if (is_a) {
            blk = (int64_t)blk_row * n_wg + wg;
        } else {
            const int tn = blk_row / halves, h = blk_row % halves;
            blk = ((int64_t)tn * n_wg + wg) * halves + h;
        }
        *reinterpret_cast<uint4 *>(dst_base + blk * 512 + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace

cudaError_t sf_pack(const uint8_t *sfa, const uint8_t *sfb, uint8_t *out_a, uint8_t *out_b, int M, int N, int sfk,
                    int row_blocks, int tiles_n, int tile_n, int n_wg, uint8_t pad, cudaStream_t stream) {
    const int wg_groups = (n_wg + PACK_WG - 1) / PACK_WG;
    const int64_t ctas = (int64_t)(row_blocks + tiles_n * ((tile_n + 127) / 128)) * wg_groups;
    sf_pack_kernel<<<(unsigned)ctas, 256, 0, stream>>>(sfa, sfb, out_a, out_b, M, N, sfk, row_blocks, tiles_n, n_wg,
                                                       tile_n, pad);
    return cudaGetLastError();
}

}  // namespace gb300
