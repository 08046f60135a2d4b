"""Pins of the oracle's operand decoders and of the shared input rounding.

Decoders are checked exhaustively against independent conversions (torch and
numpy) and against fixed points of the format definitions (IEEE 754 binary16,
bf16 = upper half of binary32, OCP FP8 E4M3, OCP UE8M0).  The generator's
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
