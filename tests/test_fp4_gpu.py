"""GPU parity of the 4-bit block-scaled kernels (E2M1 operands; UE8M0 scales per
32 K with scale_vec::2X, UE4M3 scales per 16 K with scale_vec::4X) through the
C ABI against the oracle: ragged M, N and K in both CTA modes, both D types,
C present or absent, and the full-size workloads on sampled entries."""
import pytest

from blackwell_tensor_core_tma_gb300 import gemm, synth
from tests import gpucase

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
FP4 = ["mxf4e2m1_8192x8192x8192_c0_f32out", "nvf4e2m1_8192x8192x8192_c0_f32out"]
FORCE = {"1cta": gemm.GEMM_FLAG_FORCE_1CTA, "2cta": gemm.GEMM_FLAG_FORCE_2CTA}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gemm.lib()


@pytest.mark.parametrize("name", FP4, ids=["mxf4", "nvf4"])
@pytest.mark.parametrize("variant", ["1cta", "2cta"])
@pytest.mark.parametrize("M,N,K,d,c", [
    (128, 128, 256, "f32", "zero"),        # one tile, one stage
    (300, 260, 544, "f32", "normal"),      # ragged M and N, a K tail of 32 inside the third stage
    (1048, 776, 1056, "bf16", "normal"),   # several tiles, bf16 D
    (64, 40, 32, "f32", "normal"),         # smaller than one tile, one scale block of K
])
def test_fp4_parity(name, variant, M, N, K, d, c):
    w = synth.scaled(W[name], M, N, K, d=d, c=c)
    x, D, info, st, intact = gpucase.run(w, flags=FORCE[variant], guard=512)
    assert st == gemm.GEMM_OK and intact
    assert info["cta_group"] == (1 if variant == "1cta" else 2)
    assert info["tile_k"] == 256
    gpucase.check_full(w, x, D)


@pytest.mark.parametrize("name", FP4, ids=["mxf4", "nvf4"])
def test_fp4_c_none_and_repeat(name):
    w = synth.scaled(W[name], 520, 392, 800, c="normal")
    x, D, info, st, intact = gpucase.run(w, c_none=True, guard=256, reps=3)
    assert st == gemm.GEMM_OK and intact
    gpucase.check_full(w, x, D, c_none=True)


@pytest.mark.parametrize("name", FP4, ids=["mxf4", "nvf4"])
def test_fp4_full_size_sampled(name):
    w = W[name]
    x, D, info, st, intact = gpucase.run(w, guard=1024)
    assert st == gemm.GEMM_OK and intact
    assert info["cta_group"] == 2 and info["tile_n"] == 256
    rows, cols = gpucase.sample_entries(w.M, w.N, info["tile_m"], info["tile_n"], n_random=2048)
    gpucase.check_entries(w, x, D, rows, cols)


def test_fp4_split_k():
    # fp32 D with few tiles: the plan splits K and the slices add into D
    w = synth.scaled(W["nvf4e2m1_8192x8192x8192_c0_f32out"], 256, 256, 16384, c="normal")
    x = synth.make_inputs(w)
    with gemm.Plan(w.M, w.N, w.K, w.ab, w.d, w.block_scaled) as plan:
        splits = plan.info["splits"]
    assert splits > 1
    x, D, info, st, intact = gpucase.run(w, guard=256, inputs=x)
    assert st == gemm.GEMM_OK and intact
    gpucase.check_full(w, x, D)
