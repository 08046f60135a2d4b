"""Failure detection without a GPU fault: the test-only hook makes the
producer withhold one arrival, so the MMA issuer's bounded wait runs out.
The run must report GEMM_ERR_TIMEOUT, and the same plan (same context) must
then produce a correct result."""
import numpy as np
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


def test_withheld_arrival_times_out_and_context_survives():
    import torch
    w = synth.scaled(synth.WORKLOADS["bf16_4096x4096x4096_f32out"], 512, 512, 512)
    x = synth.make_inputs(w)
    A, B, C = gpucase.to_device(x["A"]), gpucase.to_device(x["B"]), gpucase.to_device(x["C"])
    D = torch.zeros((w.M, w.N), dtype=torch.float32, device="cuda")
    with gemm.Plan(w.M, w.N, w.K, w.ab, w.d) as plan:
        plan.set_timeout(20_000_000)                        # 20 ms per wait
        gemm.gemm_testing_set_fault(plan.handle, 1)
        plan.run(A, B, C, D, None, None, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert plan.last_status() == gemm.GEMM_ERR_TIMEOUT
        assert plan.last_status() == gemm.GEMM_OK          # reading resets the word
        gemm.gemm_testing_set_fault(plan.handle, 0)
        plan.set_timeout(1_000_000_000)
        plan.run(A, B, C, D, None, None, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert plan.last_status() == gemm.GEMM_OK
    gpucase.check_full(w, x, gpucase.decode_d(D, w.d))


def test_sync_flag_returns_kernel_status():
    import torch
    w = synth.scaled(synth.WORKLOADS["bf16_4096x4096x4096_f32out"], 256, 256, 128)
    x = synth.make_inputs(w)
    A, B, C = gpucase.to_device(x["A"]), gpucase.to_device(x["B"]), gpucase.to_device(x["C"])
    D = torch.zeros((w.M, w.N), dtype=torch.float32, device="cuda")
    with gemm.Plan(w.M, w.N, w.K, w.ab, w.d, flags=gemm.GEMM_FLAG_SYNC) as plan:
        plan.set_timeout(20_000_000)
        gemm.gemm_testing_set_fault(plan.handle, 1)
        with pytest.raises(gemm.GemmError) as e:
            plan.run(A, B, C, D, None, None, torch.cuda.current_stream())
        assert e.value.status == gemm.GEMM_ERR_TIMEOUT
        gemm.gemm_testing_set_fault(plan.handle, 0)
        assert plan.run(A, B, C, D, None, None, torch.cuda.current_stream()) == gemm.GEMM_OK
    gpucase.check_full(w, x, gpucase.decode_d(D, w.d))
