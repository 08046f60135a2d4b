"""The plan's SM clock meter: counted runs give a plausible mean SM clock, reading clears
the counter, and a disabled meter counts nothing."""
import pytest

from blackwell_tensor_core_tma_gb300 import gemm, synth
from tests import gpucase

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gemm.lib()


def test_clock_meter_reads_the_sm_clock():
    import torch
    w = synth.scaled(synth.WORKLOADS["bf16_8192x8192x8192_bf16out"], 2048, 2048, 2048)
    x = synth.make_inputs(w)
    A, B, C = gpucase.to_device(x["A"]), gpucase.to_device(x["B"]), gpucase.to_device(x["C"])
    D = torch.empty((w.M, w.N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream()
    with gemm.Plan(w.M, w.N, w.K, w.ab, w.d) as plan:
        assert plan.read_clock_meter() == {"sm_mhz": 0.0, "cta_seconds": 0.0}   # never enabled
        plan.set_clock_meter(True)
        for _ in range(5):
            plan.run(A, B, C, D, None, None, s)
        m = plan.read_clock_meter()
        assert 300.0 < m["sm_mhz"] < 2500.0, m
        assert m["cta_seconds"] > 0.0
        assert plan.read_clock_meter()["cta_seconds"] == 0.0                    # reading clears
        plan.set_clock_meter(False)
        plan.run(A, B, C, D, None, None, s)
        assert plan.read_clock_meter()["cta_seconds"] == 0.0
        assert plan.last_status() == gemm.GEMM_OK
    gpucase.check_full(w, x, gpucase.decode_d(D, w.d))
