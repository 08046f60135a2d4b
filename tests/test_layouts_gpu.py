"""GPU parity for every storage order of A and B (row- / column-major), through
the C ABI, against the oracle.  K-major operands (row-major A, column-major B)
and M/N-major ones reach the tensor core through different shared-memory
layouts and descriptors, so each combination runs in both CTA modes, with
ragged edges in M, N and K."""
import pytest

from blackwell_tensor_core_tma_gb300 import gemm, synth
from tests import gpucase

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
LAYOUTS = [(True, False), (True, True), (False, False), (False, True)]
IDS = ["A_row-B_col", "A_row-B_row", "A_col-B_col", "A_col-B_row"]
FORCE = {"1cta": gemm.GEMM_FLAG_FORCE_1CTA, "2cta": gemm.GEMM_FLAG_FORCE_2CTA}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gemm.lib()


@pytest.mark.parametrize("layout", LAYOUTS, ids=IDS)
@pytest.mark.parametrize("variant", ["1cta", "2cta"])
@pytest.mark.parametrize("name,M,N,K", [
    ("bf16_4096x4096x4096_f32out", 520, 392, 264),     # several 64-element atoms, ragged M/N/K
    ("f16_4000x3000x2056_f32out", 136, 264, 72),       # one row and a few columns past a tile
    ("bf16_8192x8192x8192_bf16out", 1048, 776, 520),   # bf16 D
])
def test_layouts_16bit(layout, variant, name, M, N, K):
    a_rm, b_rm = layout
    w = synth.scaled(W[name], M, N, K, a_row_major=a_rm, b_row_major=b_rm)
    x, D, info, st, intact = gpucase.run(w, flags=FORCE[variant], guard=512)
    assert st == gemm.GEMM_OK and intact
    gpucase.check_full(w, x, D)


@pytest.mark.parametrize("layout", LAYOUTS, ids=IDS)
@pytest.mark.parametrize("variant", ["1cta", "2cta"])
@pytest.mark.parametrize("M,N,K,d", [(528, 400, 272, "f32"), (272, 512, 144, "bf16")])
def test_layouts_block_scaled(layout, variant, M, N, K, d):
    a_rm, b_rm = layout
    w = synth.scaled(W["mxf8e4m3_8192x8192x8192_c0_f32out"], M, N, K, d=d, c="normal",
                     a_row_major=a_rm, b_row_major=b_rm)
    if b_rm and variant == "1cta":
        with pytest.raises(gemm.GemmError) as e:
            gemm.Plan(M, N, K, "e4m3", d, True, FORCE[variant], a_row_major=a_rm, b_row_major=b_rm)
        assert e.value.status == gemm.GEMM_ERR_UNSUPPORTED
        return
    x, D, info, st, intact = gpucase.run(w, flags=FORCE[variant], guard=512)
    assert st == gemm.GEMM_OK and intact
    gpucase.check_full(w, x, D)


def test_column_major_alignment_rule():
    # column-major A: its rows hold M elements, so M (not K) must give 16-byte rows
    with pytest.raises(gemm.GemmError) as e:
        gemm.Plan(260, 256, 256, "bf16", "f32", a_row_major=False)
    assert e.value.status == gemm.GEMM_ERR_ALIGNMENT
    with pytest.raises(gemm.GemmError) as e:
        gemm.Plan(256, 264, 256, "e4m3", "f32", True, b_row_major=True)       # 264 e4m3 = 264 bytes
    assert e.value.status == gemm.GEMM_ERR_ALIGNMENT
    gemm.Plan(256, 256, 260, "bf16", "f32", a_row_major=False, b_row_major=True).close()   # K is free then


@pytest.mark.parametrize("layout", LAYOUTS[1:], ids=IDS[1:])
def test_layouts_full_size_sampled(layout):
    a_rm, b_rm = layout
    w = synth.scaled(W["bf16_4096x4096x4096_f32out"], 4096, 4096, 4096, a_row_major=a_rm, b_row_major=b_rm)
    x, D, info, st, intact = gpucase.run(w, guard=1024)
    assert st == gemm.GEMM_OK and intact
    rows, cols = gpucase.sample_entries(w.M, w.N, info["tile_m"], info["tile_n"], n_random=2048)
    gpucase.check_entries(w, x, D, rows, cols)
