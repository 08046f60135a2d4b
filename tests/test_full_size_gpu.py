"""Every element of every full-size workload against the oracle.

The GEMM workloads (bf16 4096^3 fp32 D; fp16 4000 x 3000 x 2056 fp32 D; bf16 8192^3 bf16 D;
block-scaled e4m3 8192^3 fp32 D) run through the plan the library chooses, as the
benchmark runs them, and all M x N entries are compared with the fp64 oracle under
|D - D_ref| <= 1e-5 * sum_k |a b| + 1e-6 * |c| (+ one bf16 ulp for bf16 D).  The
two-product chain (A 32768 x 4096, N1 = N2 = 256, bf16 D) is compared on all of its
rows under its derived bound.  The oracle's full products take about half a minute
each for the 8192^3 workloads on 16 host cores; setting GB300GEMM_ORACLE_CACHE to a
directory keeps them there, keyed by a checksum of the inputs and the oracle source.
The largest error / tolerance ratio of each workload is printed."""
import pytest

from blackwell_tensor_core_tma_gb300 import gemm, synth
from tests import gpucase

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gemm.lib()


@pytest.mark.parametrize("name", ["bf16_4096x4096x4096_f32out", "f16_4000x3000x2056_f32out",
                                  "bf16_8192x8192x8192_bf16out", "mxf8e4m3_8192x8192x8192_c0_f32out"])
def test_every_element_of_the_full_size_workload(name):
    w = synth.WORKLOADS[name]
    x, D, info, status, intact = gpucase.run(w, guard=1024)
    assert status == gemm.GEMM_OK and intact
    ratio = gpucase.full_ratio(w, x, D)
    print(f"{name}: {w.M * w.N} entries, max err/tol {ratio:.4f} (plan: cta_group {info['cta_group']}, "
          f"tile {info['tile_m']}x{info['tile_n']}, splits {info['splits']}, stream_k {info['stream_k']})")


def test_every_row_of_the_full_size_chain():
    w = synth.CHAIN_WORKLOADS["chain_bf16_32768x4096_256x256_bf16out"]
    x, D, info, status, intact = gpucase.run_chain(w, guard=1024)
    assert status == gemm.GEMM_OK and intact
    ratio = gpucase.check_chain(w, x, D)
    print(f"{w.name}: {w.M} rows x {w.N2}, max err/tol {ratio:.4f}")
