"""Stream-K (the last waves' tiles shared out as equal spans of K blocks; a cut tile's
first piece stores its partial sum into D and publishes it, the piece that finishes
the tile adds into D) against the oracle and against the whole-tile schedule, for
every kernel family and both CTA modes, and the plan's choice of it."""
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


def _run(w, flags, stream_k=True, c_none=False, reps=1):
    import torch
    x = synth.make_inputs(w)
    A, B = gpucase.to_device(x["A"]), gpucase.to_device(x["B"])
    C = None if c_none else gpucase.to_device(x["C"])
    SFA = gpucase.to_device(x["SFA"]) if w.block_scaled else None
    SFB = gpucase.to_device(x["SFB"]) if w.block_scaled else None
    tdt = torch.bfloat16 if w.d == "bf16" else torch.float32
    outs = []
    with gemm.Plan(w.M, w.N, w.K, w.ab, w.d, w.block_scaled, flags, a_row_major=w.a_row_major,
                   b_row_major=w.b_row_major) as plan:
        plan.set_stream_k(stream_k)
        info = plan.info
        for _ in range(reps):
            D = torch.full((w.M, w.N), float("nan"), dtype=tdt, device="cuda")
            plan.run(A, B, C, D, SFA, SFB, torch.cuda.current_stream())
            torch.cuda.synchronize()
            assert plan.last_status() == gemm.GEMM_OK
            outs.append(gpucase.decode_d(D, w.d))
    return x, outs, info


@pytest.mark.parametrize("variant", ["1cta", "2cta"])
@pytest.mark.parametrize("name,M,N,K,d", [
    # 2cta: 8 x 10 = 80 pair tiles over 76 pairs (every tile in a span); 1cta: 160 tiles, 152 CTAs
    ("bf16_4096x4096x4096_f32out", 2048, 2560, 4096, "f32"),
    # ragged edges, a K tail; 1cta: 16 x 11 = 176 tiles (one whole round, then spans)
    ("f16_4000x3000x2056_f32out", 2000, 2700, 4104, "f32"),
])
def test_stream_k_matches_oracle(variant, name, M, N, K, d):
    w = synth.scaled(W[name], M, N, K, d=d)
    x, (D,), info = _run(w, FORCE[variant])
    assert info["stream_k"] == 1 and info["splits"] == 1
    gpucase.check_full(w, x, D)


def test_stream_k_whole_rounds_then_spans_pairs():
    # 10 x 20 = 200 pair tiles: 76 whole tiles per unit round, then 124 tiles in spans
    w = synth.scaled(W["bf16_4096x4096x4096_f32out"], 2560, 5120, 4104, c="normal")
    x, (D,), info = _run(w, FORCE["2cta"])
    assert info["stream_k"] == 1 and info["tiles"] == 200
    rows, cols = gpucase.sample_entries(w.M, w.N, info["tile_m"], info["tile_n"], n_random=8192)
    gpucase.check_entries(w, x, D, rows, cols)


@pytest.mark.parametrize("name", ["mxf8e4m3_8192x8192x8192_c0_f32out", "mxf4e2m1_8192x8192x8192_c0_f32out",
                                  "nvf4e2m1_8192x8192x8192_c0_f32out"])
def test_stream_k_block_scaled(name):
    w = synth.scaled(W[name], 2048, 2560, 16384, c="normal")
    x, (D,), info = _run(w, FORCE["2cta"])
    assert info["stream_k"] == 1
    rows, cols = gpucase.sample_entries(w.M, w.N, info["tile_m"], info["tile_n"], n_random=2048)
    gpucase.check_entries(w, x, D, rows, cols)


def test_stream_k_is_deterministic_and_close_to_whole_tiles():
    w = synth.scaled(W["bf16_4096x4096x4096_f32out"], 2048, 2560, 4096)
    x, outs, info = _run(w, gemm.GEMM_FLAG_DETERMINISTIC, reps=3)
    assert info["stream_k"] == 1
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    x, (D0,), info0 = _run(w, gemm.GEMM_FLAG_DETERMINISTIC, stream_k=False)
    assert info0["stream_k"] == 0
    rows, cols = gpucase.sample_entries(w.M, w.N, info["tile_m"], info["tile_n"], n_random=4096)
    gpucase.check_entries(w, x, outs[0], rows, cols)
    gpucase.check_entries(w, x, D0, rows, cols)


def test_stream_k_c_none():
    w = synth.scaled(W["bf16_4096x4096x4096_f32out"], 2048, 2560, 4096)
    x, (D,), info = _run(w, FORCE["2cta"], c_none=True)
    assert info["stream_k"] == 1
    gpucase.check_full(w, x, D, c_none=True)


def test_stream_k_rule():
    # short tiles (16 k-blocks), many waves or bf16 D: whole tiles only
    with gemm.Plan(2048, 2560, 1024, "bf16", "f32") as plan:
        assert plan.info["stream_k"] == 0
    with gemm.Plan(8192, 8192, 8192, "bf16", "f32") as plan:
        assert plan.info["stream_k"] == 0
    with gemm.Plan(4096, 4096, 4096, "bf16", "bf16") as plan:
        assert plan.info["stream_k"] == 0
    # 4096^3 with 256 x 224 pair tiles: 304 tiles are 4 whole rounds of 76 pairs, no spans needed
    with gemm.Plan(4096, 4096, 4096, "bf16", "f32") as plan:
        if plan.info["grid"] == 152:
            assert plan.info["tile_n"] == 224 and plan.info["stream_k"] == 0


def test_stream_k_not_used_for_whole_waves():
    # 76 pair tiles exactly fill the GPU: no spans needed
    with gemm.Plan(256 * 4, 256 * 19, 512, "bf16", "f32") as plan:
        info = plan.info
    assert info["tiles"] == 76 and info["cta_group"] == 2
    if info["grid"] == 152:                 # 76 pairs run at once: one whole wave
        assert info["stream_k"] == 0
