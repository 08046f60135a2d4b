"""Pins of the fp64 GEMM oracle against closed forms, exact integer brute
force and exact rational arithmetic — nothing here re-derives the oracle's
own loop.  Each case is built so that a dropped term (C, a product, a scale),
a wrong sign, a wrong index or a transposed operand changes the result."""
from fractions import Fraction

import numpy as np
import pytest

from blackwell_tensor_core_tma_gb300 import synth


def _bits(vals, dtype):
    vals = np.asarray(vals, dtype=np.float32)
    return {"bf16": synth.f32_to_bf16_bits, "f16": synth.f32_to_f16_bits,
            "e4m3": synth.f32_to_e4m3_bits}[dtype](vals)


def _store_a(a, row_major):
    return a if row_major else np.ascontiguousarray(a.T)       # (M,K) or (K,M)


def _store_b(b, row_major):
    return b if row_major else np.ascontiguousarray(b.T)       # (K,N) or (N,K)


def test_identity_gives_b_plus_c(oracle_mod):
    M = K = 48
    N = 40
    eye = _bits(np.eye(M), "bf16")
    b = synth.f32_to_bf16_bits(synth.uniform_pm1(5, 1, K * N)).reshape(K, N)
    c = synth.normal(5, 2, M * N).reshape(M, N)
    bval = oracle_mod.decode(b, "bf16")
    for a_rm in (True, False):
        for b_rm in (True, False):
            D, S = oracle_mod.gemm(_store_a(eye, a_rm), _store_b(b, b_rm), c, M, N, K, "bf16",
                                   a_row_major=a_rm, b_row_major=b_rm)
            assert np.array_equal(D, bval + c.astype(np.float64))
            assert np.array_equal(S, np.abs(bval))


def test_rank_one(oracle_mod):
    M, N, K = 33, 27, 70
    rng = np.random.default_rng(1)
    u = synth.f32_to_bf16_bits(synth.uniform_pm1(6, 0, M))
    a = np.repeat(u[:, None], K, axis=1)                       # A = u 1^T
    bint = rng.integers(-9, 10, (K, N))
    b = _bits(bint, "bf16")
    c = synth.normal(6, 2, M * N).reshape(M, N)
    colsum = bint.sum(axis=0)                                  # exact integers
    uval = oracle_mod.decode(u, "bf16")
    expect = uval[:, None] * colsum[None, :] + c.astype(np.float64)
    D, S = oracle_mod.gemm(a, _store_b(b, False), c, M, N, K, "bf16")
    assert np.array_equal(D, expect)
    assert np.array_equal(S, np.abs(uval)[:, None] * np.abs(bint).sum(axis=0)[None, :])


@pytest.mark.parametrize("dtype", ["bf16", "f16", "e4m3"])
def test_all_ones_and_alternating(oracle_mod, dtype):
    M, N, K = 17, 9, 131
    ones_a = _bits(np.ones((M, K)), dtype)
    ones_b = _bits(np.ones((N, K)), dtype)
    c = synth.normal(7, 2, M * N).reshape(M, N)
    D, S = oracle_mod.gemm(ones_a, ones_b, c, M, N, K, dtype)
    assert np.array_equal(D, K + c.astype(np.float64)) and np.all(S == K)
    alt = _bits(np.tile((-1.0) ** np.arange(K), (M, 1)), dtype)  # a[i][k] = (-1)^k
    D, S = oracle_mod.gemm(alt, ones_b, c, M, N, K, dtype)
    assert np.array_equal(D, (K % 2) + c.astype(np.float64)) and np.all(S == K)
    D, S = oracle_mod.gemm(alt, ones_b, None, M, N, K, dtype)  # C = NULL means 0
    assert np.all(D == K % 2)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "e4m3"])
@pytest.mark.parametrize("a_rm,b_rm", [(True, False), (True, True), (False, False), (False, True)])
def test_integer_brute_force(oracle_mod, dtype, a_rm, b_rm):
    rng = np.random.default_rng(hash((dtype, a_rm, b_rm)) & 0xFFFF)
    M, N, K = 13, 21, 37                                       # nothing square, nothing aligned
    ai = rng.integers(-8, 9, (M, K))
    bi = rng.integers(-8, 9, (K, N))
    ci = rng.integers(-1000, 1000, (M, N))
    expect = ci + ai @ bi                                      # exact int64
    D, S = oracle_mod.gemm(_store_a(_bits(ai, dtype), a_rm), _store_b(_bits(bi, dtype), b_rm),
                           ci.astype(np.float32), M, N, K, dtype, a_row_major=a_rm, b_row_major=b_rm)
    assert np.array_equal(D, expect.astype(np.float64))
    assert np.array_equal(S, (np.abs(ai) @ np.abs(bi)).astype(np.float64))
    assert np.all(S >= np.abs(D - ci))


def test_4x4x4_exact_rationals(oracle_mod):
    for seed in range(8):
        w = synth.scaled(synth.WORKLOADS["bf16_4096x4096x4096_f32out"], 4, 4, 4)
        w = synth.dataclasses.replace(w, seed=100 + seed)
        x = synth.make_inputs(w)
        a = oracle_mod.decode(x["A"], "bf16")                  # (M,K)
        b = oracle_mod.decode(x["B"], "bf16").T                # stored (N,K) -> (K,N)
        c = x["C"].astype(np.float64)
        D, S = oracle_mod.gemm(x["A"], x["B"], x["C"], 4, 4, 4, "bf16")
        for i in range(4):
            for j in range(4):
                exact = Fraction(c[i, j]) + sum(Fraction(a[i, k]) * Fraction(b[k, j]) for k in range(4))
                sabs = sum(abs(Fraction(a[i, k]) * Fraction(b[k, j])) for k in range(4))
                assert abs(Fraction(D[i, j]) - exact) <= Fraction(2.0 ** -50) * (sabs + abs(Fraction(c[i, j])))
                assert abs(Fraction(S[i, j]) - sabs) <= Fraction(2.0 ** -50) * sabs


def test_block_scales_per_32_k(oracle_mod):
    rng = np.random.default_rng(3)
    M, N, K = 9, 7, 80                                         # 3 scale blocks, the last one partial
    sfk = 3
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    a = rng.choice(codes, (M, K))
    b = rng.choice(codes, (N, K))                              # column-major B: (N, K)
    sfa = rng.integers(123, 132, (M, sfk)).astype(np.uint8)
    sfb = rng.integers(123, 132, (N, sfk)).astype(np.uint8)
    av = oracle_mod.decode(a, "e4m3")
    bv = oracle_mod.decode(b, "e4m3")
    c = synth.normal(8, 2, M * N).reshape(M, N)
    D, S = oracle_mod.gemm(a, b, c, M, N, K, "e4m3", SFA=sfa, SFB=sfb, block_scaled=True)
    for i in range(M):
        for j in range(N):
            exact = Fraction(float(c[i, j]))
            sabs = Fraction(0)
            for k in range(K):
                p = Fraction(av[i, k]) * 2 ** (int(sfa[i, k // 32]) - 127) * \
                    Fraction(bv[j, k]) * 2 ** (int(sfb[j, k // 32]) - 127)
                exact += p
                sabs += abs(p)
            assert abs(Fraction(D[i, j]) - exact) <= Fraction(2.0 ** -50) * sabs
            assert abs(Fraction(S[i, j]) - sabs) <= Fraction(2.0 ** -50) * sabs
    # unit scales (code 127) give the unscaled product
    one = np.full((M, sfk), 127, np.uint8), np.full((N, sfk), 127, np.uint8)
    D1, _ = oracle_mod.gemm(a, b, c, M, N, K, "e4m3", SFA=one[0], SFB=one[1], block_scaled=True)
    D0, _ = oracle_mod.gemm(a, b, c, M, N, K, "e4m3")
    assert np.array_equal(D0, D1)


def test_entries_and_row_slabs_match_full(oracle_mod):
    w = synth.scaled(synth.WORKLOADS["f16_4000x3000x2056_f32out"], 70, 50, 90)
    x = synth.make_inputs(w)
    D, S = oracle_mod.gemm(x["A"], x["B"], x["C"], 70, 50, 90, "f16")
    rng = np.random.default_rng(0)
    r = rng.integers(0, 70, 200)
    c = rng.integers(0, 50, 200)
    De, Se = oracle_mod.gemm_entries(x["A"], x["B"], x["C"], 70, 50, 90, "f16", r, c)
    assert np.array_equal(De, D[r, c]) and np.array_equal(Se, S[r, c])
    Ds, Ss = oracle_mod.gemm(x["A"], x["B"], x["C"], 70, 50, 90, "f16", rows=(13, 40))
    assert np.array_equal(Ds, D[13:40]) and np.array_equal(Ss, S[13:40])


def test_rejects_bad_arguments(oracle_mod):
    a = np.zeros((4, 4), np.uint16)
    with pytest.raises(ValueError):
        oracle_mod.gemm(a, a, None, 4, 4, 5, "bf16")
    with pytest.raises(ValueError):
        oracle_mod.gemm(a, a, None, 4, 4, 4, "bf16", SFA=np.zeros(4, np.uint8), SFB=np.zeros(4, np.uint8),
                        block_scaled=True)
    with pytest.raises(ValueError):
        oracle_mod.gemm_entries(a, a, None, 4, 4, 4, "bf16", [4], [0])


# ------------------------------------------------------------- 4-bit operands
# OCP MX FP4 E2M1 magnitudes of codes 0..7 (bit 3 is the sign)
E2M1_TABLE = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
              Fraction(4), Fraction(6)]


def _e2m1_value(code):
    v = E2M1_TABLE[int(code) & 7]
    return -v if int(code) & 8 else v


def _scale_values(codes, mode):
    """Exact scale values: UE8M0 2^(c-127); UE4M3 through torch's float8_e4m3fn."""
    import torch
    codes = np.asarray(codes, np.uint8)
    if mode == 1:
        return [[Fraction(2) ** (int(c) - 127) for c in row] for row in codes]
    vals = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()
    return [[Fraction(float(v)) for v in row] for row in vals]


def _pack_store(codes, row_major_of_logical):
    """Logical (R, C) codes -> packed storage: rows of C when row_major, else rows of R."""
    s = codes if row_major_of_logical else np.ascontiguousarray(codes.T)
    return synth.pack_e2m1(s)


@pytest.mark.parametrize("mode,K", [(1, 72), (2, 72), (2, 32)])
@pytest.mark.parametrize("a_rm,b_rm", [(True, False), (True, True), (False, False), (False, True)])
def test_e2m1_block_scaled_exact_rationals(oracle_mod, mode, K, a_rm, b_rm):
    # every product and partial sum is a short dyadic (or, with UE4M3 scales,
    # a short multiple of 2^-20) rational: compare with exact arithmetic
    rng = np.random.default_rng(11 + mode + K)
    M, N = 6, 4                                                # even, so column-wise packing works
    blk = 32 if mode == 1 else 16
    sfk = -(-K // blk)
    a = rng.integers(0, 16, (M, K)).astype(np.uint8)           # logical a[i][k]
    b = rng.integers(0, 16, (K, N)).astype(np.uint8)           # logical b[k][j]
    if mode == 1:
        sfa = rng.integers(122, 133, (M, sfk)).astype(np.uint8)
        sfb = rng.integers(122, 133, (N, sfk)).astype(np.uint8)
    else:
        sfa = synth.ue4m3_codes(3, 3, M * sfk).reshape(M, sfk)
        sfb = synth.ue4m3_codes(3, 4, N * sfk).reshape(N, sfk)
    c = synth.normal(9, 2, M * N).reshape(M, N)
    A = _pack_store(a, a_rm)                                   # (M, K/2) or (K, M/2)
    B = _pack_store(b, b_rm)                                   # (K, N/2) or (N, K/2)
    D, S = oracle_mod.gemm(A, B, c, M, N, K, "e2m1", a_row_major=a_rm, b_row_major=b_rm,
                           SFA=sfa, SFB=sfb, block_scaled=mode)
    sa, sb = _scale_values(sfa, mode), _scale_values(sfb, mode)
    for i in range(M):
        for j in range(N):
            terms = [_e2m1_value(a[i, k]) * sa[i][k // blk] * _e2m1_value(b[k, j]) * sb[j][k // blk]
                     for k in range(K)]
            exact = Fraction(float(c[i, j])) + sum(terms)
            sabs = sum(abs(t) for t in terms)
            assert abs(Fraction(D[i, j]) - exact) <= Fraction(2.0 ** -50) * (sabs + abs(Fraction(float(c[i, j]))))
            assert abs(Fraction(S[i, j]) - sabs) <= Fraction(2.0 ** -50) * sabs


def test_e2m1_low_nibble_is_the_even_element(oracle_mod):
    # A row 0 = [0, 1, 0, 0, ...]: only element k = 1 (high nibble of byte 0) is set
    M, N, K = 2, 2, 32
    a = np.zeros((M, K), np.uint8)
    a[0, 1] = 0x2                                              # 1.0
    b = np.zeros((K, N), np.uint8)
    b[0, 0], b[1, 0] = 0x4, 0x5                                # b[0][0] = 2, b[1][0] = 3
    one = np.full((M, 1), 127, np.uint8), np.full((N, 1), 127, np.uint8)
    D, _ = oracle_mod.gemm(synth.pack_e2m1(a), synth.pack_e2m1(np.ascontiguousarray(b.T)), None, M, N, K,
                           "e2m1", SFA=one[0], SFB=one[1], block_scaled=1)
    assert D[0, 0] == 3.0 and D[1, 0] == 0.0


@pytest.mark.parametrize("mode,unit", [(1, 127), (2, 0x38)])
def test_e2m1_unit_scales_give_unscaled_product(oracle_mod, mode, unit):
    w = synth.scaled(synth.WORKLOADS["nvf4e2m1_8192x8192x8192_c0_f32out"], 20, 12, 96, c="normal")
    x = synth.make_inputs(w)
    sfk = 96 // (32 if mode == 1 else 16)
    D1, S1 = oracle_mod.gemm(x["A"], x["B"], x["C"], 20, 12, 96, "e2m1", SFA=np.full((20, sfk), unit, np.uint8),
                             SFB=np.full((12, sfk), unit, np.uint8), block_scaled=mode)
    D0, S0 = oracle_mod.gemm(x["A"], x["B"], x["C"], 20, 12, 96, "e2m1")
    assert np.array_equal(D0, D1) and np.array_equal(S0, S1)


def test_scale_mode_pairing_is_checked(oracle_mod):
    a = np.zeros((4, 32), np.uint8)
    sf = np.zeros((4, 2), np.uint8)
    with pytest.raises(ValueError):                            # UE4M3 scales are for 4-bit operands only
        oracle_mod.gemm(a, a, None, 4, 4, 32, "e4m3", SFA=sf, SFB=sf, block_scaled=2)
    with pytest.raises(ValueError):                            # packed sizes: K/2 bytes per row
        oracle_mod.gemm(a, a, None, 4, 4, 32, "e2m1", SFA=sf[:, :1], SFB=sf[:, :1], block_scaled=1)
