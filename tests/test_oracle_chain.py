"""Pins of the oracle's two-product chain D = C + round(A·B)·E: the rounding
against torch's conversions, exact integer chains, hand-derived ties of the
round-to-nearest-even step, and row selection."""
import numpy as np
import pytest
import torch

from blackwell_tensor_core_tma_gb300 import synth


def _bits(vals, dtype):
    vals = np.asarray(vals, dtype=np.float32)
    return synth.f32_to_bf16_bits(vals) if dtype == "bf16" else synth.f32_to_f16_bits(vals)


@pytest.mark.parametrize("dtype,tdt", [("bf16", torch.bfloat16), ("f16", torch.float16)])
def test_rounding_matches_torch(oracle_mod, dtype, tdt):
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(20000) * np.exp2(rng.integers(-30, 30, 20000))).astype(np.float32)
    if dtype == "f16":
        x = x[np.abs(x) < 65504]
    ties = (np.float32(1.0) + np.float32(2.0 ** -8) * np.arange(1, 64, 2, dtype=np.float32))
    x = np.concatenate([x, ties, -ties])
    ours = oracle_mod.round_to(x.astype(np.float64), dtype)
    ref = torch.from_numpy(x).to(tdt).double().numpy()
    assert np.array_equal(ours, ref)


def test_rounding_overflow_and_ties(oracle_mod):
    assert oracle_mod.round_to([65519.0, 65520.0, -70000.0], "f16").tolist() == [65504.0, np.inf, -np.inf]
    assert oracle_mod.round_to([2.0 ** -25, 3 * 2.0 ** -26], "f16").tolist() == [0.0, 2.0 ** -24]


def _chain_inputs(a, b, e, dtype):
    """Logical a (M,K), b (K,N1), e (N1,N2) -> the chain's storage (A row-major, B and E column-major)."""
    return _bits(a, dtype), _bits(b.T, dtype), _bits(e.T, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_exact_integer_chain(oracle_mod, dtype):
    # |T| <= 4 * 3 * 3 * K = 36 * 7: exact in both formats (256 = 2^8 bounds bf16's exact integers)
    rng = np.random.default_rng(5)
    M, K, N1, N2 = 9, 7, 12, 5
    a = rng.integers(-3, 4, (M, K))
    b = rng.integers(-3, 4, (K, N1))
    e = rng.integers(-4, 5, (N1, N2))
    c = rng.integers(-50, 50, (M, N2)).astype(np.float32)
    A, B, E = _chain_inputs(a, b, e, dtype)
    T, S1, D, S2 = oracle_mod.chain(A, B, E, c, M, N1, N2, K, dtype)
    t = a @ b
    assert np.abs(t).max() <= 256
    assert np.array_equal(T, t) and np.array_equal(S1, np.abs(a) @ np.abs(b))
    assert np.array_equal(D, t @ e + c) and np.array_equal(S2, np.abs(t) @ np.abs(e))


@pytest.mark.parametrize("dtype,base,t,p", [
    # bf16: spacing 2 on [256, 512), 4 on [512, 1024)
    ("bf16", [256, 256, 256, 256, 512, 512, 512], [257, 259, 261, 263, 513, 514, 518], [256, 260, 260, 264, 512, 512, 520]),
    # fp16: spacing 2 on [2048, 4096), 4 on [4096, 8192)
    ("f16", [2048, 2048, 2048, 4096, 4096, 4096], [2049, 2051, 2053, 4097, 4098, 4102], [2048, 2052, 2052, 4096, 4096, 4104]),
])
def test_intermediate_rounds_half_to_even(oracle_mod, dtype, base, t, p):
    # row i of A is [base_i, t_i - base_i] (both exact in the format), B = [[1], [1]]: T = t
    # exactly; E = identity, so D = round(T)
    M, K, N1 = len(t), 2, 1
    a = np.array([[bi, ti - bi] for bi, ti in zip(base, t)], dtype=np.float64)
    b = np.array([[1.0], [1.0]])
    e = np.eye(1)
    A, B, E = _chain_inputs(a, b, e, dtype)
    T, _, D, _ = oracle_mod.chain(A, B, E, None, M, N1, 1, K, dtype)
    assert T[:, 0].tolist() == t
    assert D[:, 0].tolist() == p


def test_rows_select_and_bounds(oracle_mod):
    w = synth.scaled(synth.WORKLOADS["bf16_4096x4096x4096_f32out"], 40, 24, 96)
    x = synth.make_inputs(w)
    E = synth.f32_to_bf16_bits(synth.uniform_pm1(3, 7, 16 * 24)).reshape(16, 24)   # N2 = 16 rows of N1 = 24
    T, S1, D, S2 = oracle_mod.chain(x["A"], x["B"], E, x["C"][:, :16], 40, 24, 16, 96, "bf16")
    rows = np.array([39, 0, 17])
    Tr, S1r, Dr, S2r = oracle_mod.chain(x["A"], x["B"], E, x["C"][:, :16], 40, 24, 16, 96, "bf16", rows=rows)
    assert np.array_equal(Tr, T[rows]) and np.array_equal(Dr, D[rows]) and np.array_equal(S2r, S2[rows])
    # T equals the plain product, and |D - C| <= S2
    Dg, Sg = oracle_mod.gemm(x["A"], x["B"], None, 40, 24, 96, "bf16")
    assert np.array_equal(T, Dg) and np.array_equal(S1, Sg)
    assert np.all(np.abs(D - x["C"][:, :16].astype(np.float64)) <= S2 * (1 + 1e-12))
    with pytest.raises(ValueError):
        oracle_mod.chain(x["A"], x["B"], E, None, 40, 24, 16, 96, "bf16", rows=[40])
