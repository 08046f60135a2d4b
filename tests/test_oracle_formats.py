"""Pins of the oracle's operand decoders and of the shared input rounding.

Decoders are checked exhaustively against independent conversions (torch and
numpy) and against fixed points of the format definitions (IEEE 754 binary16,
bf16 = upper half of binary32, OCP FP8 E4M3, OCP UE8M0, the OCP MX FP4 E2M1
value table).  The generator's
encoders are pinned by decode -> encode identity on every finite code.
"""
import numpy as np
import pytest
import torch

from blackwell_tensor_core_tma_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _same(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.array_equal(a, b, equal_nan=True) and np.array_equal(np.signbit(a), np.signbit(b))


def test_bf16_decode_exhaustive(oracle_mod):
    codes = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle_mod.decode(codes, "bf16")
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert _same(ours, ref)


def test_f16_decode_exhaustive(oracle_mod):
    codes = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle_mod.decode(codes, "f16")
    ref = codes.view(np.float16).astype(np.float64)
    assert _same(ours, ref)


def test_e4m3_decode_exhaustive(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle_mod.decode(codes, "e4m3")
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert _same(ours, ref)


def test_e4m3_definition_points(oracle_mod):
    # OCP 8-bit floating point spec, E4M3: bias 7, max normal S.1111.110 = 448,
    # NaN S.1111.111, no infinities, min subnormal 2^-9, min normal 2^-6
    d = lambda c: float(oracle_mod.decode(np.array([c], dtype=np.uint8), "e4m3")[0])
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert d(0x78) == 256.0                       # exponent field 15 is a normal binade
    assert d(0x01) == 2.0 ** -9 and d(0x07) == 7 * 2.0 ** -9
    assert d(0x08) == 2.0 ** -6
    assert d(0x38) == 1.0 and d(0x39) == 1.125 and d(0xB8) == -1.0
    assert d(0x00) == 0.0 and np.signbit(d(0x80))


def test_f16_definition_points(oracle_mod):
    d = lambda c: float(oracle_mod.decode(np.array([c], dtype=np.uint16), "f16")[0])
    assert d(0x3C00) == 1.0 and d(0x7BFF) == 65504.0 and d(0x0001) == 2.0 ** -24
    assert d(0x0400) == 2.0 ** -14 and d(0x7C00) == np.inf and np.isnan(d(0x7E00))
    assert d(0xC000) == -2.0


def test_bf16_definition_points(oracle_mod):
    d = lambda c: float(oracle_mod.decode(np.array([c], dtype=np.uint16), "bf16")[0])
    assert d(0x3F80) == 1.0 and d(0x3F81) == 1.0 + 2.0 ** -7 and d(0xBF80) == -1.0
    assert d(0x0001) == 2.0 ** -133 and d(0x0080) == 2.0 ** -126


def test_ue8m0_decode(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    v = oracle_mod.decode(codes, "ue8m0")
    assert np.isnan(v[255])
    assert np.array_equal(v[:255], np.ldexp(1.0, np.arange(255) - 127))
    assert v[127] == 1.0 and v[131] == 16.0 and v[123] == 1.0 / 16


def test_bf16_encode_roundtrip(oracle_mod):
    codes = np.arange(1 << 16, dtype=np.uint16)
    vals = oracle_mod.decode(codes, "bf16")
    fin = np.isfinite(vals)
    back = synth.f32_to_bf16_bits(vals[fin].astype(np.float32))
    assert np.array_equal(back, codes[fin])


def test_f16_encode_roundtrip(oracle_mod):
    codes = np.arange(1 << 16, dtype=np.uint16)
    vals = oracle_mod.decode(codes, "f16")
    fin = np.isfinite(vals)
    back = synth.f32_to_f16_bits(vals[fin].astype(np.float32))
    assert np.array_equal(back, codes[fin])


def test_e4m3_encode_roundtrip(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle_mod.decode(codes, "e4m3")
    fin = np.isfinite(vals)
    back = synth.f32_to_e4m3_bits(vals[fin].astype(np.float32))
    # -0 and +0 keep their sign
    assert np.array_equal(back, codes[fin])


def test_bf16_ulp_is_grid_spacing(oracle_mod):
    # for every positive finite bf16 below the largest, the next code is one ulp away
    codes = np.arange(1, 0x7F7F, dtype=np.uint16)
    v = oracle_mod.decode(codes, "bf16")
    nxt = oracle_mod.decode(codes + 1, "bf16")
    assert np.array_equal(nxt - v, oracle_mod.bf16_ulp(v))
    assert oracle_mod.bf16_ulp(1.0) == 2.0 ** -7
    assert oracle_mod.bf16_ulp(-3.0) == 2.0 ** -6
    assert oracle_mod.bf16_ulp(0.0) == 2.0 ** -133


# OCP Microscaling Formats (MX) v1.0, FP4 E2M1: the eight magnitudes of codes
# 0b0000 .. 0b0111 (bias 1; 0b0001 is the one subnormal), bit 3 the sign
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_exhaustive(oracle_mod):
    codes = np.arange(16, dtype=np.uint8)
    ours = oracle_mod.decode(codes, "e2m1")
    ref = np.array(E2M1_TABLE + [-v for v in E2M1_TABLE])
    assert _same(ours, ref)
    # only the low nibble is the code
    assert _same(oracle_mod.decode(codes | np.uint8(0xA0), "e2m1"), ref)


def test_ue4m3_decode_exhaustive(oracle_mod):
    codes = np.arange(128, dtype=np.uint8)
    ours = oracle_mod.decode(codes, "ue4m3")
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert _same(ours, ref)                      # 0x7F (exponent and mantissa all ones) is NaN
    assert float(oracle_mod.decode(np.array([0x38], np.uint8), "ue4m3")[0]) == 1.0
    assert np.all(np.isnan(oracle_mod.decode(np.arange(128, 256, dtype=np.uint8), "ue4m3")))


def test_e2m1_encode_is_nearest_ties_to_even(oracle_mod):
    # brute force: the nearest representable magnitude, on a tie the one with an
    # even code (mantissa bit 0), beyond 6 the largest (satfinite)
    rng = np.random.default_rng(4)
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 1e9]
    x = np.concatenate([rng.uniform(-8, 8, 20000), rng.standard_normal(20000), ties]).astype(np.float32)
    x = np.concatenate([x, -x])
    table = np.array(E2M1_TABLE)
    a = np.abs(x.astype(np.float64))
    dist = np.abs(a[:, None] - table[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    even = cand & (np.arange(8)[None, :] % 2 == 0)
    code = np.where(even.any(axis=1), np.argmax(even, axis=1), np.argmax(cand, axis=1))
    code = np.where(a > 6.0, 7, code)
    expect = code.astype(np.uint8) | (np.signbit(x).astype(np.uint8) << 3)
    assert np.array_equal(synth.f32_to_e2m1_bits(x), expect)
    # decode -> encode identity on every code
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(synth.f32_to_e2m1_bits(oracle_mod.decode(codes, "e2m1").astype(np.float32)), codes)


def test_e2m1_packing():
    codes = np.arange(16, dtype=np.uint8).reshape(2, 8)
    packed = synth.pack_e2m1(codes)
    assert packed.shape == (2, 4)
    assert packed[0, 0] == 0x10 and packed[0, 3] == 0x76 and packed[1, 0] == 0x98
    assert np.array_equal(synth.unpack_e2m1(packed), codes)
