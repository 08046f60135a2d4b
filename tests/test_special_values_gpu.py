"""Special values the seeded workloads never produce, compared element by element with
the oracle: infinities and NaN in C; fp16 operands whose products overflow fp16 but not
fp32 (the accumulation is fp32), fp16 infinities and NaN in A and B; e4m3 operands at their
saturation limit +-448 and the e4m3 NaN code; the UE8M0 NaN scale code 255.

Where the oracle's value is NaN the GPU's must be NaN, where it is an infinity the GPU's must
be the same infinity, and every finite entry meets the usual bound
|D - D_ref| <= 1e-5 * sum_k |a b| + 1e-6 * |c| (+ one bf16 ulp for bf16 D)."""
import numpy as np
import pytest

import oracle
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


def _compare(w, x, D):
    D_ref, S = oracle.gemm(x["A"], x["B"], x["C"], w.M, w.N, w.K, w.ab, SFA=x.get("SFA"), SFB=x.get("SFB"),
                           block_scaled=w.block_scaled)
    nan_ref, inf_ref = np.isnan(D_ref), np.isinf(D_ref)
    assert np.array_equal(np.isnan(D), nan_ref), (int(np.isnan(D).sum()), int(nan_ref.sum()))
    assert np.array_equal(np.isinf(D), inf_ref), (int(np.isinf(D).sum()), int(inf_ref.sum()))
    assert np.array_equal(np.sign(D[inf_ref]), np.sign(D_ref[inf_ref]))
    fin = np.isfinite(D_ref)
    c = x["C"].astype(np.float64)
    gpucase._assert_within(w, D[fin], D_ref[fin], S[fin], c[fin], "finite entries")
    return int(nan_ref.sum()), int(inf_ref.sum())


def _run(w, x):
    _, D, _, status, _ = gpucase.run(w, inputs=x)
    assert status == gemm.GEMM_OK
    return D


@pytest.mark.parametrize("M,N,K,d", [(384, 320, 256, "f32"), (384, 320, 256, "bf16"), (1024, 1280, 192, "bf16"),
                                     (1024, 1024, 320, "f32")])
def test_infinities_and_nan_in_c(M, N, K, d):
    w = synth.scaled(W["bf16_4096x4096x4096_f32out"], M, N, K, d=d)
    x = synth.make_inputs(w)
    C = x["C"]
    rng = np.random.default_rng(M + N + K)
    for val in (np.inf, -np.inf, np.nan):
        r, c = rng.integers(0, M, 40), rng.integers(0, N, 40)
        C[r, c] = val
    n_nan, n_inf = _compare(w, x, _run(w, x))
    assert n_nan > 0 and n_inf > 0


@pytest.mark.parametrize("M,N,K", [(512, 512, 512), (1024, 1024, 256)])
def test_fp16_operands_beyond_the_fp16_range_and_fp16_infinities_and_nan(M, N, K):
    w = synth.scaled(W["f16_4000x3000x2056_f32out"], M, N, K)
    x = synth.make_inputs(w)
    A, B = x["A"], x["B"]                      # A (M, K) codes; B stored (N, K): B[j, k] is element (k, j)
    f16 = lambda v: np.float16(v).view(np.uint16)
    A[3, :] = f16(60000.0)                     # row 3 x column 5: products 2.4e5, beyond fp16's 65504
    B[5, :] = f16(4.0)
    A[7, :] = f16(65504.0)                     # the largest fp16 in both: products 4.3e9, sums 2e12
    B[9, :] = f16(-65504.0)
    A[10, 20] = f16(np.inf)                    # row 10: +-inf where b[20, j] != 0, NaN where it is 0
    B[11, 20] = f16(0.0)
    A[12, 30] = f16(-np.inf)
    B[40, 33] = f16(np.nan)                    # column 40: NaN everywhere
    n_nan, n_inf = _compare(w, x, _run(w, x))
    assert n_nan >= M and n_inf > 0


@pytest.mark.parametrize("M,N,K", [(512, 512, 512), (1024, 1024, 512)])
def test_e4m3_saturation_nan_code_and_nan_scale(M, N, K):
    w = synth.scaled(W["mxf8e4m3_8192x8192x8192_c0_f32out"], M, N, K, c="normal")
    x = synth.make_inputs(w)
    A, B, SFA, SFB = x["A"], x["B"], x["SFA"], x["SFB"]
    A[2, :] = 0x7E                             # +448, the largest e4m3
    B[3, :] = 0xFE                             # -448
    A[4, 64:96] = 0x7E
    B[6, 64:96] = 0x7E
    A[5, 7] = 0x7F                             # the e4m3 NaN code: row 5 NaN
    B[8, 100] = 0xFF                           # -NaN: column 8 NaN
    SFA[9, 2] = 255                            # UE8M0 NaN: row 9 NaN
    SFB[11, 1] = 255                           # column 11 NaN
    n_nan, n_inf = _compare(w, x, _run(w, x))
    assert n_nan >= 4 * M - 8
