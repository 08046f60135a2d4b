"""Pins of the oracle's layout maps to the values the pages print
(tests/golden/*.json, each citing its page and section) and to the
bijection properties the pages state."""
import itertools

import pytest

from oracle import layouts as L
from tests.conftest import golden


def test_cd_fragment_lane5_printed_example():
    g = golden("fragments.json")["cd_lane5"]
    assert L.group_and_thread(g["lane"]) == (g["g"], g["t"])
    assert L.mma_m16n8k16_cd(g["lane"]) == [tuple(e) for e in g["elements"]]


def test_cd_fragment_groups_and_bijection():
    g = golden("fragments.json")["cd_groups"]
    assert {r for l in range(4) for r, _ in L.mma_m16n8k16_cd(l)} == set(g["lanes_0_3_rows"])
    assert {r for l in range(4, 8) for r, _ in L.mma_m16n8k16_cd(l)} == set(g["lanes_4_7_rows"])
    cells = [e for l in range(32) for e in L.mma_m16n8k16_cd(l)]
    assert sorted(cells) == sorted(itertools.product(range(16), range(8)))


def test_atom_examples():
    for ex in golden("fragments.json")["atom_examples"]:
        assert L.atom8x8_coord(ex["row"], ex["col"]) == tuple(ex["atom"])
        assert L.atom8x8_lane_slot(ex["row"], ex["col"]) == (ex["lane"], ex["slot"])


def test_atom_agrees_with_cd_fragment():
    # rows 0..7 of the C/D fragment are the 8x8 atom: slot s of the atom = fragment slot s
    for r in range(8):
        for c in range(8):
            lane, slot = L.atom8x8_lane_slot(r, c)
            assert L.mma_m16n8k16_cd(lane)[slot] == (r, c)


def test_a_and_b_fragments():
    f = golden("fragments.json")
    a0 = L.mma_m16n8k16_a(0)
    for reg in range(4):
        assert a0[2 * reg:2 * reg + 2] == [tuple(e) for e in f["a_registers"][f"reg{reg}"]]
    b0 = L.mma_m16n8k16_b(0)
    for reg in range(2):
        assert b0[2 * reg:2 * reg + 2] == [tuple(e) for e in f["b_registers"][f"reg{reg}"]]
    # each fragment covers its tile exactly once over the 32 lanes
    a_cells = [e for l in range(32) for e in L.mma_m16n8k16_a(l)]
    assert sorted(a_cells) == sorted(itertools.product(range(16), range(16)))
    b_cells = [e for l in range(32) for e in L.mma_m16n8k16_b(l)]
    assert sorted(b_cells) == sorted(itertools.product(range(16), range(8)))
    # A and B use the same (g, t): lane 5 holds k = 2, 3, 10, 11 of row 1 / column 1
    assert {k for m, k in L.mma_m16n8k16_a(5) if m == 1} == {2, 3, 10, 11}
    assert {k for k, n in L.mma_m16n8k16_b(5)} == {2, 3, 10, 11} and {n for _, n in L.mma_m16n8k16_b(5)} == {1}


def test_ldmatrix():
    f = golden("fragments.json")["ldmatrix"]
    for name, num in [("x1", 1), ("x2", 2), ("x4", 4)]:
        lanes = L.ldmatrix_address_lanes(num)
        assert (lanes[0], lanes[-1]) == tuple(f["address_lanes"][name])
    assert [l for l in range(32) if L.ldmatrix_x1_received(l)[0] == 0] == f["row0_receivers"]
    assert L.ldmatrix_x1_received(0)[1] == f["lane0_cols"]
    assert L.ldmatrix_x1_received(1)[1] == f["lane1_cols"]
    got = sorted((r, c) for l in range(32) for r, cs in [L.ldmatrix_x1_received(l)] for c in cs)
    assert got == sorted(itertools.product(range(8), range(8)))
    assert L.ldmatrix_address_lane(3, 5) == 29


def test_tmem_facts():
    t = golden("tmem.json")
    assert (L.TMEM_LANES, L.TMEM_MAX_COLS, L.TMEM_CELL_BITS) == (t["lanes"], t["max_cols"], t["cell_bits"])
    assert list(L.TMEM_ALLOC_SIZES) == t["alloc_sizes"]
    assert not L.tmem_alloc_size_ok(96) and not L.tmem_alloc_size_ok(1024)
    for ex in t["alloc_order_examples"]:
        assert L.tmem_alloc_sequence_ok(ex["seq"]) == ex["legal"]
    for w, (lo, hi) in t["lane_windows"].items():
        win = L.tmem_lane_window(int(w))
        assert (win[0], win[-1]) == (lo, hi)
    for num, regs in t["ld_16x128b_regs"].items():
        assert L.tcgen05_ld_16x128b_regs(int(num)) == regs
    assert L.tcgen05_ld_16x128b_cells(4) == t["ld_16x128b_x4_cells"]
    assert L.tcgen05_ld_16x128b_cells(1) == t["ld_16x128b_x1_cells"]
    with pytest.raises(ValueError):
        L.tmem_lane_window(4)


def test_scale_factor_layout():
    s = golden("scale_factors.json")
    shape = s["layout_shape"]
    seen = {}
    for mg, lane, sfk in itertools.product(*(range(n) for n in shape)):
        col, byte = L.sf_tmem_position(mg, lane, sfk)
        assert col == (4 * mg + sfk) // 4 and byte == (4 * mg + sfk) % 4
        key = (lane, col, byte)
        assert key not in seen                          # injective: one scale per byte
        seen[key] = (L.sf_row(mg, lane), sfk)
    assert len(seen) == 128 * 4                         # 128 rows x 4 K blocks fill 32 lanes x 4 words
    assert sorted(r for r, _ in seen.values())[::4] == list(range(128))
    assert len(L.sf_replicated_lanes(5)) == s["replication"]
    assert L.sf_replicated_lanes(5) == [5, 37, 69, 101]


def test_scale_vec_words():
    s = golden("scale_factors.json")
    names = {"SF0": 10, "SF1": 11, "SF2": 12, "SF3": 13}
    for kind, pattern in s["scale_vec"].items():
        assert L.scale_vec_word(kind, [10, 11, 12, 13]) == [names[p] for p in pattern]
        assert L.scale_id_choices(kind) == s["sf_id"][kind]


def test_tma_tiling_and_prefetch():
    import numpy as np
    M, N, CM, CN = 8, 12, 4, 3
    A = np.arange(M * N).reshape(M, N)
    tiles = A.reshape(M // CM, CM, N // CN, CN)
    for i in range(M // CM):
        for j in range(N // CN):
            rs, cs = L.cta_tile(M, N, CM, CN, i, j)
            assert np.array_equal(A[rs, cs], tiles[i, :, j, :])
    # num_stages = 2: computing batch 0 prefetches batch 2, batch 1 prefetches 3
    assert [L.prefetch_batch(b, 2) for b in range(3)] == [2, 3, 4]
