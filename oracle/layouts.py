"""Layout maps the pages print — TEST INFRASTRUCTURE ONLY (part of the oracle).

Each function restates one mapping in the notation of its page, so that the
tests can pin it to the page's worked examples and bijection properties, and
so that GPU tests can check a kernel's data placement against it.

Sources (page title, section):
  * "Tensor Core 数据布局的演进", "一个具体的 fragment 映射": the
    mma.sync.m16n8k16 register fragments of A, B and C/D, and the 8x8 atom
    S[(8, 4, 2) : (4@laneid, 1@laneid, 1@reg)].
  * same page, "ldmatrix：从 shared memory 构造 fragment": ldmatrix .m8n8.
  * "Tensor Memory（TMEM）" / "Tensor Memory (TMEM)": allocation sizes and
    ordering rule, per-warp lane windows, tcgen05.ld/st register counts.
  * "Tensor Core 数据布局的演进", "tcgen05.cp 如何写入 TMEM" and
    "scale_vec 的 Word 内复制": scale factors in TMEM.
  * "(二) CUTLASS —— 掌握 Tensor Memory Accelerator（TMA）": CTA tiling of a
    row-major matrix and the prefetch distance of a num_stages pipeline.
"""

from __future__ import annotations


# ------------------------------------------------ mma.sync.m16n8k16 fragments

def group_and_thread(lane: int) -> tuple[int, int]:
    """g = lane // 4 (4-lane group), t = lane % 4 (position in the group)."""
    if not 0 <= lane < 32:
        raise ValueError("lane out of range")
    return lane // 4, lane % 4


def mma_m16n8k16_cd(lane: int) -> list[tuple[int, int]]:
    """(row, col) of the four fp32 accumulators lane holds, in slot order.

    Group g covers rows g and g + 8; lane t of the group holds columns 2t and 2t + 1.
    """
    g, t = group_and_thread(lane)
    return [(g, 2 * t), (g, 2 * t + 1), (g + 8, 2 * t), (g + 8, 2 * t + 1)]


def mma_m16n8k16_a(lane: int) -> list[tuple[int, int]]:
    """(m, k) of the eight 16-bit A elements of a lane: 4 registers x 2 halves."""
    g, t = group_and_thread(lane)
    out = []
    for m_off, k_off in [(0, 0), (8, 0), (0, 8), (8, 8)]:      # registers 0..3
        out += [(g + m_off, 2 * t + k_off), (g + m_off, 2 * t + k_off + 1)]
    return out


def mma_m16n8k16_b(lane: int) -> list[tuple[int, int]]:
    """(k, n) of the four 16-bit B elements of a lane: 2 registers x 2 halves."""
    g, t = group_and_thread(lane)
    out = []
    for k_off in (0, 8):                                        # registers 0, 1
        out += [(2 * t + k_off, g), (2 * t + k_off + 1, g)]
    return out


def atom8x8_coord(row: int, col: int) -> tuple[int, int, int]:
    """Atom coordinate (row, column_pair, element_in_pair) of an 8x8 C/D element."""
    return row, col // 2, col % 2


def atom8x8_lane_slot(row: int, col: int) -> tuple[int, int]:
    """S[(8, 4, 2) : (4@laneid, 1@laneid, 1@reg)] evaluated at (row, col)."""
    r, p, e = atom8x8_coord(row, col)
    return 4 * r + 1 * p, 1 * e


# ---------------------------------------------------------- ldmatrix .m8n8

def ldmatrix_address_lane(matrix: int, row: int) -> int:
    """Lane that supplies the start address of row ``row`` of matrix ``matrix``."""
    return matrix * 8 + row


def ldmatrix_address_lanes(num: int) -> range:
    """Lanes that supply addresses for .x1 / .x2 / .x4 (num = 1, 2, 4)."""
    if num not in (1, 2, 4):
        raise ValueError("num must be 1, 2 or 4")
    return range(8 * num)


def ldmatrix_x1_received(lane: int) -> tuple[int, list[int]]:
    """(row, [cols]) of the two 16-bit elements lane receives from one 8x8 block."""
    return lane // 4, [2 * (lane % 4), 2 * (lane % 4) + 1]


# ----------------------------------------------------------------- TMEM

TMEM_LANES = 128
TMEM_MAX_COLS = 512
TMEM_CELL_BITS = 32
TMEM_ALLOC_SIZES = (32, 64, 128, 256, 512)


def tmem_alloc_size_ok(n_cols: int) -> bool:
    return n_cols in TMEM_ALLOC_SIZES


def tmem_alloc_sequence_ok(sizes: list[int]) -> bool:
    """A CTA's successive allocations may not request more columns than the previous one."""
    return all(tmem_alloc_size_ok(s) for s in sizes) and all(b <= a for a, b in zip(sizes, sizes[1:]))


def tmem_lane_window(warp_in_warpgroup: int) -> range:
    """TMEM lanes a warp may reach with tcgen05.ld/st: 32 * (warp id in its warpgroup) + 0..31."""
    if not 0 <= warp_in_warpgroup < 4:
        raise ValueError("warp id in a warpgroup is 0..3")
    return range(32 * warp_in_warpgroup, 32 * warp_in_warpgroup + 32)


def tcgen05_ld_16x128b_cells(num: int) -> int:
    """32-bit TMEM cells one .16x128b.x{num} access moves: 16 lanes x num x 4 cells."""
    if num not in (1, 2, 4, 8, 16, 32, 64, 128):
        raise ValueError("bad .num")
    return 16 * num * (128 // TMEM_CELL_BITS)


def tcgen05_ld_16x128b_regs(num: int) -> int:
    """32-bit registers per thread for .16x128b.x{num}: cells / 32 threads."""
    return tcgen05_ld_16x128b_cells(num) // 32


# ------------------------------------------------ scale factors in TMEM

def sf_tmem_position(mgroup: int, lane: int, sfk: int) -> tuple[int, int]:
    """S[(4, 32, 4) : (4@TCol, 1@TLane, 1@TCol)] for 8-bit scales, M = 128, SFK = 4.

    Returns (hardware_TCol, byte_in_word): the logical byte column
    4*Mgroup + sfk packed four to a 32-bit cell.  The TMEM lane is ``lane``
    (plus the replication below).
    """
    if not (0 <= mgroup < 4 and 0 <= lane < 32 and 0 <= sfk < 4):
        raise ValueError("coordinate out of range")
    logical = 4 * mgroup + sfk
    return logical // 4, logical % 4


def sf_replicated_lanes(lane: int) -> list[int]:
    """R[4 : 32@TLane]: the four TMEM lanes that hold a copy (.32x128b.warpx4)."""
    return [lane + 32 * w for w in range(4)]


def sf_row(mgroup: int, lane: int) -> int:
    """Matrix row m = 32 * Mgroup + lane whose scales sit at (Mgroup, lane, :)."""
    return 32 * mgroup + lane


def scale_vec_word(kind: str, sf: list[int]) -> list[int]:
    """Bytes 0..3 of a 32-bit scale word for scale_vec::1X / 2X / 4X."""
    if kind == "1X":
        return [sf[0]] * 4
    if kind == "2X":
        return [sf[0], sf[1], sf[0], sf[1]]
    if kind == "4X":
        return list(sf[:4])
    raise ValueError(kind)


def scale_id_choices(kind: str) -> list[int]:
    """Byte offsets an SFA_ID / SFB_ID may select for each scale_vec kind."""
    return {"1X": [0, 1, 2, 3], "2X": [0, 2], "4X": [0]}[kind]


# ------------------------------------------------------------------ TMA

def cta_tile(M: int, N: int, CTA_M: int, CTA_N: int, i: int, j: int) -> tuple[slice, slice]:
    """Rows and columns of CTA tile (i, j) of a row-major M x N matrix.

    The page's numpy sketch reshapes to (M // CTA_M, CTA_M, N // CTA_N, CTA_N)
    (its last extent is printed as N, read as CTA_N) and takes [i, :, j, :].
    """
    return slice(i * CTA_M, (i + 1) * CTA_M), slice(j * CTA_N, (j + 1) * CTA_N)


def prefetch_batch(compute_batch: int, num_stages: int) -> int:
    """fetch_batch = compute_batch + num_stages."""
    return compute_batch + num_stages
