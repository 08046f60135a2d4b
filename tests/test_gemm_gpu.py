"""GPU parity of the tensor-core GEMM against the fp64 oracle, through the C ABI.

Small cases compare every element; the full-size workloads (in the launch
configuration the benchmark times, i.e. the default plan) compare tile
corners and edges, a full row and column, and random entries."""
import numpy as np
import pytest

from tests import rules
from blackwell_tensor_core_tma_gb300 import gemm, synth
from tests import gpucase

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
BF16_UNI = W["bf16_4096x4096x4096_f32out"]
F16_NORM = W["f16_4000x3000x2056_f32out"]
BF16_OUT = W["bf16_8192x8192x8192_bf16out"]
MXF8 = W["mxf8e4m3_8192x8192x8192_c0_f32out"]

FORCE = {"1cta": gemm.GEMM_FLAG_FORCE_1CTA, "2cta": gemm.GEMM_FLAG_FORCE_2CTA}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gemm.lib()


def test_first_workload_full():
    """bf16 256^3, C = 0 passed as a zero buffer, fp32 D: every element."""
    w = W["bf16_256x256x256_c0_f32out"]
    x, D, info, st, intact = gpucase.run(w, guard=4096)
    assert st == gemm.GEMM_OK and intact
    gpucase.check_full(w, x, D)


@pytest.mark.parametrize("variant", ["1cta", "2cta"])
@pytest.mark.parametrize("base,M,N,K", [
    (BF16_UNI, 640, 768, 512),        # several whole tiles
    (F16_NORM, 1000, 600, 520),       # ragged M, N and K (K % 64 == 8)
    (BF16_OUT, 1100, 1048, 1032),     # bf16 D, ragged
    (F16_NORM, 129, 260, 72),         # one row and a few columns past a tile
])
def test_parity_small(variant, base, M, N, K):
    w = synth.scaled(base, M, N, K)
    x, D, info, st, intact = gpucase.run(w, flags=FORCE[variant], guard=1024)
    assert st == gemm.GEMM_OK and intact
    assert info["cta_group"] == (1 if variant == "1cta" else 2)
    gpucase.check_full(w, x, D)


@pytest.mark.parametrize("variant", ["1cta", "2cta"])
def test_c_null_means_zero(variant):
    w = synth.scaled(F16_NORM, 300, 520, 264)
    x, D, info, st, intact = gpucase.run(w, flags=FORCE[variant], c_none=True, guard=512)
    assert st == gemm.GEMM_OK and intact
    gpucase.check_full(w, x, D, c_none=True)


@pytest.mark.parametrize("M,N,K", [(1, 4, 8), (1, 8, 8), (7, 12, 24), (128, 256, 64), (257, 264, 8)])
def test_degenerate_shapes(M, N, K):
    base = BF16_OUT if N % 8 == 0 else BF16_UNI
    w = synth.scaled(base, M, N, K)
    x, D, info, st, intact = gpucase.run(w, guard=256)
    assert st == gemm.GEMM_OK and intact
    gpucase.check_full(w, x, D)


def test_long_k_and_many_tiles_per_cta():
    """K = 16384 stresses the ring over many wraps; 2 x 32 tiles per CTA for the scheduler."""
    w = synth.scaled(BF16_UNI, 256, 512, 16384)
    x, D, info, st, _ = gpucase.run(w, flags=gemm.GEMM_FLAG_FORCE_1CTA)
    assert st == gemm.GEMM_OK
    gpucase.check_full(w, x, D)
    for M, N, K, flags in [(4096, 4096, 64, gemm.GEMM_FLAG_FORCE_1CTA), (8192, 4096, 64, 0)]:
        w2 = synth.scaled(BF16_UNI, M, N, K)
        x, D, info, st, _ = gpucase.run(w2, flags=flags)
        assert st == gemm.GEMM_OK and info["tiles"] > 2 * info["grid"] // info["cta_group"]
        gpucase.check_full(w2, x, D)


def test_repeated_runs_identical():
    """A deterministic plan gives bitwise-identical results run after run (this
    shape would otherwise be split along K)."""
    w = synth.scaled(BF16_UNI, 512, 512, 640)
    det = gemm.GEMM_FLAG_DETERMINISTIC
    x, D1, info, st1, _ = gpucase.run(w, flags=det, reps=1)
    _, D3, _, st3, _ = gpucase.run(w, flags=det, inputs=x, reps=3)
    assert st1 == st3 == gemm.GEMM_OK and info["splits"] == 1
    assert np.array_equal(D1, D3)


@pytest.mark.parametrize("M,N,K,d,c", [
    (640, 448, 512, "f32", "zero"),      # two whole 128 x 224 tiles across, 4 k-blocks
    (1000, 600, 528, "f32", "normal"),   # ragged M, N; K = 4 k-blocks + 16 (last scale block partial)
    (300, 232, 96, "bf16", "normal"),    # bf16 D; one k-block, 3 scale blocks
    (129, 8, 32, "f32", "zero"),         # one scale block
])
@pytest.mark.parametrize("variant", ["1cta", "2cta"])
def test_block_scaled_small(variant, M, N, K, d, c):
    """e4m3 x e4m3 with one UE8M0 scale per 32 K, distinct per (row, block): a wrong
    scale byte or block shows as errors of up to 2^8."""
    w = synth.scaled(MXF8, M, N, K, d=d, c=c)
    x, D, info, st, intact = gpucase.run(w, flags=FORCE[variant], guard=512)
    assert st == gemm.GEMM_OK and intact
    # single CTAs: 128 x 224 tiles; pairs: the plan's rule (256, or 224 with two accumulators)
    assert info["tile_n"] == (224 if variant == "1cta" else rules.e4m3_tile_rule(M, N, K, d == "f32"))
    assert info["launches_per_run"] == 2
    assert info["cta_group"] == (1 if variant == "1cta" else 2)
    gpucase.check_full(w, x, D)


@pytest.mark.parametrize("M,N,K,d,c_none,b_row", [
    (4096, 4096, 4096, "f32", False, False),   # 304 narrow tiles: four whole rounds (+16 % measured)
    (1100, 1504, 2080, "bf16", False, False),  # ragged M, N and K, bf16 D
    (2000, 1300, 1024, "f32", True, False),    # C absent
    (1536, 2048, 1024, "f32", False, True),    # N-contiguous B: 112 rows are not whole atoms, 256 kept
])
def test_e4m3_pair_tile_forms(M, N, K, d, c_none, b_row):
    """CTA pairs with 256 x 224 tiles and two accumulators (the narrow form), where the plan's
    rule picks them, against the oracle."""
    w = synth.scaled(MXF8, M, N, K, d=d, c="normal", b_row_major=b_row)
    x, D, info, st, intact = gpucase.run(w, c_none=c_none, guard=512)
    assert st == gemm.GEMM_OK and intact and info["cta_group"] == 2
    assert info["tile_n"] == (256 if b_row else rules.e4m3_tile_rule(M, N, K, d == "f32"))
    if not b_row:
        assert info["tile_n"] == 224
    if M * N * K > 2 ** 34:                    # sampled entries (C present)
        rows, cols = gpucase.sample_entries(w.M, w.N, info["tile_m"], info["tile_n"], n_random=4096)
        gpucase.check_entries(w, x, D, rows, cols)
    else:
        gpucase.check_full(w, x, D, c_none=c_none)


def test_block_scaled_c_null():
    w = synth.scaled(MXF8, 384, 480, 256, c="normal")
    x, D, info, st, intact = gpucase.run(w, c_none=True, guard=512)
    assert st == gemm.GEMM_OK and intact
    gpucase.check_full(w, x, D, c_none=True)


@pytest.mark.parametrize("name", ["bf16_4096x4096x4096_f32out", "f16_4000x3000x2056_f32out",
                                  "bf16_8192x8192x8192_bf16out", "mxf8e4m3_8192x8192x8192_c0_f32out"])
def test_full_size_sampled(name):
    w = W[name]
    x, D, info, st, intact = gpucase.run(w, guard=4096)
    assert st == gemm.GEMM_OK and intact
    rows, cols = gpucase.sample_entries(w.M, w.N, info["tile_m"], info["tile_n"])
    gpucase.check_entries(w, x, D, rows, cols)
    assert np.isfinite(D).all()
