"""The tensor-pipe rate probe: every MMA shape the GEMM kernels issue reports a per-SM,
per-clock rate below the dense rate of its kind and a clock the device can run at, and
the whole-GPU rate agrees with the per-SM rate at that clock."""
import pytest

from blackwell_tensor_core_tma_gb300 import gemm

pytestmark = pytest.mark.gpu

# dense FLOP per SM clock of kind::f16 (a 128 x 256 x 16 MMA per 64 clocks); the other
# kinds at most the multiple of it that their per-GPU dense figures state
F16_PER_CLK = 8192
CASES = [("bf16", gemm.GEMM_SCALE_NONE, 1, 1), ("bf16", gemm.GEMM_SCALE_NONE, 2, 1),
         ("f16", gemm.GEMM_SCALE_NONE, 2, 1), ("e4m3", gemm.GEMM_SCALE_UE8M0_32, 1, 2),
         ("e4m3", gemm.GEMM_SCALE_UE8M0_32, 2, 2), ("e2m1", gemm.GEMM_SCALE_UE8M0_32, 2, 6),
         ("e2m1", gemm.GEMM_SCALE_UE4M3_16, 2, 6)]


@pytest.mark.parametrize("ab,scale,cg,mult", CASES)
def test_rate_is_plausible(ab, scale, cg, mult):
    r = gemm.gemm_measure_tensor_rate(ab, scale, cg, 2048)
    assert r["sms"] >= 100 and r["sms"] % cg == 0
    # at least half the kind::f16 rate, at most the dense rate of the kind (+5 % for clock noise)
    assert 0.5 * F16_PER_CLK <= r["flop_per_clk_per_sm"] <= 1.05 * mult * F16_PER_CLK, r
    assert 300.0 <= r["sm_mhz"] <= 2200.0, r
    # whole-GPU TFLOP/s = SMs x FLOP/clk x clock, within the spread of the CTAs' clocks
    expect = r["sms"] * r["flop_per_clk_per_sm"] * r["sm_mhz"] * 1e6 / 1e12
    assert 0.8 * expect <= r["tflops"] <= 1.1 * expect, (r, expect)


def test_pairs_match_single_ctas_per_sm():
    one = gemm.gemm_measure_tensor_rate("bf16", gemm.GEMM_SCALE_NONE, 1, 2048)
    two = gemm.gemm_measure_tensor_rate("bf16", gemm.GEMM_SCALE_NONE, 2, 2048)
    assert 0.8 <= two["flop_per_clk_per_sm"] / one["flop_per_clk_per_sm"] <= 1.25, (one, two)
