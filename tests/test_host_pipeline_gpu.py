"""gemm_run_host with host buffers: the pipelined form (row chunks copied up, multiplied
and copied back on three streams) against the oracle, for ragged chunk counts, both D
types and C present or absent, and the plain form for shapes it does not apply to."""
import numpy as np
import pytest

from blackwell_tensor_core_tma_gb300 import gemm, synth
from tests import gpucase

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gemm.lib()


def _host_run(w, c_none=False, flags=0, reps=1):
    import torch
    x = synth.make_inputs(w)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).pin_memory()
    hA, hB = pin(x["A"]), pin(x["B"])
    hC = None if c_none else pin(x["C"])
    hSFA = pin(x["SFA"]) if w.block_scaled else None
    hSFB = pin(x["SFB"]) if w.block_scaled else None
    tdt = torch.bfloat16 if w.d == "bf16" else torch.float32
    outs = []
    with gemm.Plan(w.M, w.N, w.K, w.ab, w.d, w.block_scaled, flags, a_row_major=w.a_row_major,
                   b_row_major=w.b_row_major) as plan:
        for _ in range(reps):
            hD = torch.full((w.M, w.N), float("nan"), dtype=tdt).pin_memory()
            assert plan.run_host(hA, hB, hC, hD, hSFA, hSFB, torch.cuda.current_stream()) == gemm.GEMM_OK
            outs.append(gpucase.decode_d(hD, w.d))
        info = plan.info
    return x, outs, info


@pytest.mark.parametrize("M,N,K,d", [
    (4096, 1024, 512, "f32"),     # four chunks of 1024 rows
    (3500, 776, 264, "bf16"),     # three whole chunks and a ragged one; ragged N and K
    (2048, 512, 1024, "f32"),     # exactly two chunks
    (4096, 2904, 1032, "bf16"),   # CTA pairs with 256 x 224 tiles in every chunk
    (4096, 1024, 512, "bf16"),    # CTA pairs with 256 x 256 tiles, bf16 D
])
def test_pipelined_host_run_matches_oracle(M, N, K, d):
    w = synth.scaled(W["bf16_4096x4096x4096_f32out"], M, N, K, d=d)
    x, (D,), info = _host_run(w)
    if (M, N) == (4096, 2904) and info["grid"] == 152:
        assert info["cta_group"] == 2 and info["tile_n"] == 224
    rows, cols = gpucase.sample_entries(w.M, w.N, info["tile_m"], info["tile_n"], n_random=8192)
    gpucase.check_entries(w, x, D, rows, cols)


def test_pipelined_host_run_c_none_and_repeat():
    w = synth.scaled(W["f16_4000x3000x2056_f32out"], 4000, 520, 520)
    x, outs, info = _host_run(w, c_none=True, reps=2)
    assert np.array_equal(outs[0], outs[1])
    gpucase.check_full(w, x, outs[0], c_none=True)


@pytest.mark.parametrize("case", ["small", "col-major-A", "block-scaled"])
def test_plain_host_run_where_the_pipeline_does_not_apply(case):
    if case == "small":
        w = synth.scaled(W["bf16_4096x4096x4096_f32out"], 1000, 512, 256)
    elif case == "col-major-A":
        w = synth.scaled(W["bf16_4096x4096x4096_f32out"], 4096, 512, 256, a_row_major=False)
    else:                                   # below two chunks of rows
        w = synth.scaled(W["mxf8e4m3_8192x8192x8192_c0_f32out"], 1000, 512, 256, c="normal")
    x, (D,), info = _host_run(w)
    rows, cols = gpucase.sample_entries(w.M, w.N, info["tile_m"], info["tile_n"], n_random=4096)
    gpucase.check_entries(w, x, D, rows, cols)


@pytest.mark.parametrize("name,M,N,K", [
    ("mxf8e4m3_8192x8192x8192_c0_f32out", 4096, 512, 256),     # four chunks, single CTAs
    ("mxf8e4m3_8192x8192x8192_c0_f32out", 3000, 1280, 512),    # CTA pairs, a ragged last chunk
    ("mxf4e2m1_8192x8192x8192_c0_f32out", 2048, 1024, 1024),   # UE8M0 / 32, exactly two chunks
    ("nvf4e2m1_8192x8192x8192_c0_f32out", 4096, 1536, 512),    # UE4M3 / 16
])
def test_pipelined_block_scaled_host_run(name, M, N, K):
    """Block-scaled plans from host buffers run as the row-chunk pipeline: each chunk's SFA
    rows go up with its A and C rows and are packed before its kernel; SFB goes up once."""
    w = synth.scaled(W[name], M, N, K, c="normal")
    x, (D,), info = _host_run(w)
    rows, cols = gpucase.sample_entries(w.M, w.N, info["tile_m"], info["tile_n"], n_random=4096)
    gpucase.check_entries(w, x, D, rows, cols)
