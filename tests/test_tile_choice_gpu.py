"""The fp16/bf16 pair plans' choice between 256 x 256 and 256 x 224 tiles (whichever fills
the persistent rounds better, 224 discounted for its extra operand bytes per FLOP; an
N-contiguous B keeps 256), and oracle parity of the 256 x 224 kernel over ragged shapes,
bf16 D, C absent and a column-major A."""
import dataclasses

import pytest

from blackwell_tensor_core_tma_gb300 import gemm, synth
from tests import gpucase

pytestmark = pytest.mark.gpu

F16_NORM = synth.WORKLOADS["f16_4000x3000x2056_f32out"]
BF16_UNI = synth.WORKLOADS["bf16_4096x4096x4096_f32out"]


def expected_tile_n(M, N, K, d, units=76):
    """The plan's rule, restated: column share x round share (0.89 under stream-K) x 0.965
    for 224, or x the wide epilogue's gain for 256 with fp32 D and at most 40 k-blocks."""
    tiles_m, kb = -(-M // 256), -(-K // 64)

    def eff(bn):
        tn = -(-N // bn)
        tiles = tiles_m * tn
        rounds = -(-tiles // units)
        sk = d == "f32" and kb >= 64 and tiles >= units and tiles % units != 0 and tiles < 4 * units
        e = N / (tn * bn) * (0.89 if sk else tiles / (rounds * units))
        if bn == 224:
            e *= 0.965
        elif d == "f32" and kb <= 40 and 2 * tiles > units:
            e *= 1.0 + 0.1 * (40 - kb) / 24.0
        return e
    return 224 if eff(224) > 1.02 * eff(256) else 256


@pytest.mark.parametrize("M,N,K,d,b_row", [
    (4096, 4096, 4096, "f32", False),      # 224: 304 tiles = 4 whole rounds; 256 needs stream-K
    (4000, 3000, 2056, "f32", False),      # 224: 2.95 rounds (256: 2.5, even with the wide epilogue)
    (8192, 8192, 8192, "bf16", False),     # 256: 1024 tiles; 224 gains no round and costs feed
    (2048, 2560, 4096, "f32", False),      # both need stream-K: 256 keeps every column busy
    (4096, 4096, 1024, "f32", False),      # 256 with the wide epilogue (16 k-blocks)
    (4096, 4096, 4096, "f32", True),       # N-contiguous B: 112-row halves are not whole atoms
])
def test_tile_choice(M, N, K, d, b_row):
    with gemm.Plan(M, N, K, "bf16", d, b_row_major=b_row) as plan:
        info = plan.info
    assert info["cta_group"] == 2
    if info["grid"] == 152:                 # 76 pairs co-resident, as the rule's figures assume
        assert info["tile_n"] == (256 if b_row else expected_tile_n(M, N, K, d))


@pytest.mark.parametrize("base,M,N,K,d,a_row,c_none", [
    (F16_NORM, 4000, 3000, 2632, "f32", True, False),     # ragged M, N and K
    (BF16_UNI, 4096, 2904, 1032, "bf16", True, False),    # bf16 D (rows of 16-byte multiples)
    (F16_NORM, 2000, 3000, 2632, "f32", True, True),      # C absent
    (BF16_UNI, 2048, 3000, 2704, "f32", False, False),    # column-major A
])
def test_narrow_tile_parity(base, M, N, K, d, a_row, c_none):
    w = dataclasses.replace(synth.scaled(base, M, N, K, d=d), a_row_major=a_row)
    x, D, info, st, intact = gpucase.run(w, flags=gemm.GEMM_FLAG_FORCE_2CTA, c_none=c_none, guard=1024)
    assert st == gemm.GEMM_OK and intact
    if info["grid"] == 152:
        assert info["tile_n"] == 224 == expected_tile_n(M, N, K, d)
    gpucase.check_full(w, x, D, c_none=c_none)
