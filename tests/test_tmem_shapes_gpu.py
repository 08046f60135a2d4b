"""The pages' tcgen05.ld example shapes on the GPU ("Tensor Memory（TMEM）", sections
"每个 warp 能访问哪些 TMEM lanes" and "Shape 和 Repeat Factor"), checked against the
oracle's layout maps and the values the pages print (tests/golden/tmem.json).

Every TMEM cell holds the code (lane << 16) | column.  Each warp of one warpgroup reads
its window back with .16x128b.x1 / .x2 / .x4 / .x8 and .32x32b.x32.  The pages fix the
register count per thread (2, 4, 8, 16), the cells one access moves (16 lanes x 4 cells
x num) and the lanes a warp reaches (32w..32w+31); they leave the cell-to-register
assignment to the instruction, so for .16x128b the test checks that the warp's registers
hold exactly those cells, each once, and for .32x32b (the kernels' own shape) that thread
t holds lane 32w + t, columns in order."""
import json
import os

import numpy as np
import pytest

from blackwell_tensor_core_tma_gb300 import gemm
from oracle import layouts

pytestmark = pytest.mark.gpu

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tmem.json")))
# (repeat factor, first register, first column) of the probe's .16x128b loads
LOADS = [(1, 0, 0), (2, 2, 32), (4, 6, 64), (8, 14, 128)]


@pytest.fixture(scope="module")
def regs():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return gemm.gemm_testing_tmem_ld_probe()


@pytest.mark.parametrize("num,first,col0", LOADS)
def test_16x128b_moves_16_lanes_of_the_window_num_times(regs, num, first, col0):
    n_regs = layouts.tcgen05_ld_16x128b_regs(num)
    assert n_regs == GOLDEN["ld_16x128b_regs"][str(num)] == 2 * num
    cells = layouts.tcgen05_ld_16x128b_cells(num)
    if num == 4:
        assert cells == GOLDEN["ld_16x128b_x4_cells"]
    if num == 1:
        assert cells == GOLDEN["ld_16x128b_x1_cells"]
    for w in range(4):
        vals = regs[w, :, first:first + n_regs].ravel()
        lanes, cols = vals >> 16, vals & 0xFFFF
        lo, hi = GOLDEN["lane_windows"][str(w)]
        assert list(layouts.tmem_lane_window(w)) == list(range(lo, hi + 1))
        assert lanes.min() >= lo and lanes.max() <= hi            # nothing outside the warp's window
        assert vals.size == cells and np.unique(vals).size == cells   # every cell exactly once
        assert set(lanes.tolist()) == set(range(lo, lo + 16))     # 16 lanes from the address's lane
        assert set(cols.tolist()) == set(range(col0, col0 + 4 * num))   # 128 bits = 4 cells per repeat
        for lane in range(lo, lo + 16):                          # each lane gives 4 * num cells
            assert int((lanes == lane).sum()) == 4 * num


def test_32x32b_gives_thread_t_lane_t_of_the_window(regs):
    """The epilogue's shape: thread t of warp w holds lane 32w + t, 32 consecutive columns."""
    for w in range(4):
        for t in range(32):
            want = ((32 * w + t) << 16) | np.arange(256, 288, dtype=np.uint32)
            assert np.array_equal(regs[w, t, 30:62], want)


@pytest.mark.parametrize("load", [False, True])
def test_epilogue_staging_patterns_cost_no_more_than_linear(load):
    """The epilogue's swizzled staging rows (bf16 D: 64-byte rows, fp32: 128-byte rows) take
    no longer per warp-wide 128-bit access than a linear pattern; 128-byte rows without the
    swizzle pay bank conflicts, so the probe does see them (64-byte rows without it were
    measured slower for stores but not for loads, so they are only reported)."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lin = gemm.gemm_testing_staging_probe(2, load)
    bf16_rows, f32_rows = gemm.gemm_testing_staging_probe(0, load), gemm.gemm_testing_staging_probe(1, load)
    plain_bf16, plain_f32 = gemm.gemm_testing_staging_probe(3, load), gemm.gemm_testing_staging_probe(4, load)
    assert bf16_rows <= 1.1 * lin and f32_rows <= 1.1 * lin, (bf16_rows, f32_rows, lin)
    assert plain_f32 > 1.5 * lin, (plain_bf16, plain_f32, lin)
    print(f"clocks per access ({'load' if load else 'store'}): linear {lin:.2f}, bf16 rows {bf16_rows:.2f}, "
          f"fp32 rows {f32_rows:.2f}, unswizzled bf16 rows {plain_bf16:.2f}, unswizzled fp32 rows {plain_f32:.2f}")
