"""Split-K (TMA reduce-add of K slices into D = C) against the oracle, and the
plan's choice of slices."""
import numpy as np
import pytest

from blackwell_tensor_core_tma_gb300 import gemm, synth
from tests import gpucase

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
FORCE = {"1cta": gemm.GEMM_FLAG_FORCE_1CTA, "2cta": gemm.GEMM_FLAG_FORCE_2CTA}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gemm.lib()


def _run(w, flags, splits, c_none=False):
    import torch
    x = synth.make_inputs(w)
    A, B = gpucase.to_device(x["A"]), gpucase.to_device(x["B"])
    C = None if c_none else gpucase.to_device(x["C"])
    SFA = gpucase.to_device(x["SFA"]) if w.block_scaled else None
    SFB = gpucase.to_device(x["SFB"]) if w.block_scaled else None
    D = torch.full((w.M, w.N), float("nan"), dtype=torch.float32, device="cuda")
    with gemm.Plan(w.M, w.N, w.K, w.ab, w.d, w.block_scaled, flags, a_row_major=w.a_row_major,
                   b_row_major=w.b_row_major) as plan:
        if splits is not None:
            plan.set_split_k(splits)
        info = plan.info
        plan.run(A, B, C, D, SFA, SFB, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert plan.last_status() == gemm.GEMM_OK
    return x, gpucase.decode_d(D, w.d), info


@pytest.mark.parametrize("variant", ["1cta", "2cta"])
@pytest.mark.parametrize("name,M,N,K,splits", [
    ("bf16_4096x4096x4096_f32out", 256, 512, 8192, 8),
    ("f16_4000x3000x2056_f32out", 200, 300, 2056, 5),        # ragged, K slices of unequal length
    ("bf16_4096x4096x4096_f32out", 130, 264, 1032, 17),      # splits clamped to the 17 k-blocks
])
def test_split_k_matches_oracle(variant, name, M, N, K, splits):
    w = synth.scaled(W[name], M, N, K)
    x, D, info = _run(w, FORCE[variant], splits)
    assert info["splits"] == min(splits, -(-K // 64)) and info["launches_per_run"] == 2
    gpucase.check_full(w, x, D)


def test_split_k_without_c_and_column_major():
    w = synth.scaled(W["bf16_4096x4096x4096_f32out"], 264, 136, 4096, a_row_major=False, b_row_major=True)
    x, D, info = _run(w, gemm.GEMM_FLAG_FORCE_1CTA, 7, c_none=True)
    assert info["splits"] == 7
    gpucase.check_full(w, x, D, c_none=True)


@pytest.mark.parametrize("variant", ["1cta", "2cta"])
def test_split_k_block_scaled(variant):
    w = synth.scaled(W["mxf8e4m3_8192x8192x8192_c0_f32out"], 256, 512, 4096, c="normal")
    x, D, info = _run(w, FORCE[variant], 6)
    assert info["splits"] == 6 and info["launches_per_run"] == 3
    gpucase.check_full(w, x, D)


def test_automatic_choice():
    # 512 x 512 output tiles cannot fill the GPU; K = 16384 gives 256 k-blocks to share
    w = synth.scaled(W["bf16_4096x4096x4096_f32out"], 512, 512, 16384)
    x, D, info = _run(w, 0, None)
    assert info["splits"] > 1 and info["grid"] > info["tiles"]
    gpucase.check_full(w, x, D)
    # a problem that fills the GPU is not split; bf16 D is never split
    with gemm.Plan(4096, 4096, 4096, "bf16", "f32") as plan:
        assert plan.info["splits"] == 1
    with gemm.Plan(512, 512, 16384, "bf16", "f32", flags=gemm.GEMM_FLAG_DETERMINISTIC) as plan:
        assert plan.info["splits"] == 1
        with pytest.raises(gemm.GemmError) as e:
            plan.set_split_k(4)
        assert e.value.status == gemm.GEMM_ERR_UNSUPPORTED
    with gemm.Plan(512, 512, 16384, "bf16", "bf16") as plan:
        assert plan.info["splits"] == 1
        with pytest.raises(gemm.GemmError) as e:
            plan.set_split_k(4)
        assert e.value.status == gemm.GEMM_ERR_UNSUPPORTED
