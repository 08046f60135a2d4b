"""The wide-epilogue forms of the fp16/bf16 kernel (8 epilogue warps): for CTA pairs (5 stages),
which a plan chooses for fp32 D, 256-column tiles, whole tiles (no split-K or stream-K: the shapes
below fill the pairs or have fewer than 8 k-blocks) and at most 40 k-blocks; and for single CTAs
(3 stages) that take at most one tile of at most 40 k-blocks each, without split-K.  The choice
itself (seen as the plan's ring depth) and parity with the oracle over ragged shapes, C present
and absent, both storage orders of A and B, and several tiles per CTA pair."""
import dataclasses

import pytest

from blackwell_tensor_core_tma_gb300 import gemm, synth
from tests import gpucase

pytestmark = pytest.mark.gpu

F16_NORM = synth.WORKLOADS["f16_4000x3000x2056_f32out"]
BF16_UNI = synth.WORKLOADS["bf16_4096x4096x4096_f32out"]
PAIRS = gemm.GEMM_FLAG_FORCE_2CTA


@pytest.mark.parametrize("base,M,N,K,a_row,b_row,c_none", [
    (F16_NORM, 2000, 2300, 392, True, False, False),      # ragged M, N, K (K % 64 == 8), one wave
    (BF16_UNI, 2048, 2304, 2560, True, False, False),     # 40 k-blocks: the longest K that takes it
    (F16_NORM, 4000, 1000, 1032, True, False, True),      # C absent
    (BF16_UNI, 1536, 1024, 264, False, True, False),      # column-major A, row-major B
    (F16_NORM, 4096, 4608, 192, True, False, False),      # 288 tiles: several per pair, 3 k-blocks
])
def test_wide_epilogue_parity(base, M, N, K, a_row, b_row, c_none):
    w = dataclasses.replace(synth.scaled(base, M, N, K), a_row_major=a_row, b_row_major=b_row)
    x, D, info, st, intact = gpucase.run(w, flags=PAIRS, c_none=c_none, guard=1024)
    assert st == gemm.GEMM_OK and intact
    assert info["cta_group"] == 2 and info["tile_n"] == 256
    assert info["stages"] == 5 and info["splits"] == 1 and info["stream_k"] == 0
    gpucase.check_full(w, x, D, c_none=c_none)


@pytest.mark.parametrize("M,N,K,d,stages", [
    (2048, 2048, 2560, "f32", 5),      # 40 k-blocks, fp32 D: wide
    (2048, 2048, 2624, "f32", 6),      # 41 k-blocks: the default kernel
    (2048, 2048, 1024, "bf16", 6),     # bf16 D keeps four epilogue warps
])
def test_wide_epilogue_choice(M, N, K, d, stages):
    with gemm.Plan(M, N, K, "bf16", d, flags=PAIRS) as plan:
        assert plan.info["stages"] == stages


@pytest.mark.parametrize("base,M,N,K,d,a_row,b_row,c_none", [
    (BF16_UNI, 256, 256, 256, "f32", True, False, False),      # the first workload's shape: 2 tiles, 4 k-blocks
    (F16_NORM, 300, 520, 200, "bf16", True, False, False),     # bf16 D (never split along K), ragged
    (F16_NORM, 1000, 904, 448, "bf16", False, True, True),     # 32 tiles, MN-major A and B, C absent
    (BF16_UNI, 129, 8, 32, "f32", True, False, False),         # one k-block, one column group
])
def test_single_cta_wide_epilogue_parity(base, M, N, K, d, a_row, b_row, c_none):
    w = dataclasses.replace(synth.scaled(base, M, N, K, d=d), a_row_major=a_row, b_row_major=b_row)
    x, D, info, st, intact = gpucase.run(w, flags=gemm.GEMM_FLAG_FORCE_1CTA, c_none=c_none, guard=1024)
    assert st == gemm.GEMM_OK and intact
    assert info["cta_group"] == 1 and info["stages"] == 3 and info["splits"] == 1
    gpucase.check_full(w, x, D, c_none=c_none)


@pytest.mark.parametrize("M,N,K,d,stages", [
    (256, 256, 256, "f32", 3),         # one tile per CTA, 4 k-blocks: wide
    (512, 512, 640, "f32", 4),         # 10 k-blocks and few tiles: split along K instead
    (1000, 904, 2624, "bf16", 4),      # 41 k-blocks: the default single-CTA kernel
    (8192, 512, 512, "bf16", 3),       # 128 tiles on 152 CTAs: one each, wide
    (8192, 1024, 512, "bf16", 4),      # 256 tiles: more than one per CTA, the default kernel
])
def test_single_cta_wide_epilogue_choice(M, N, K, d, stages):
    with gemm.Plan(M, N, K, "bf16", d, flags=gemm.GEMM_FLAG_FORCE_1CTA) as plan:
        assert plan.info["stages"] == stages
