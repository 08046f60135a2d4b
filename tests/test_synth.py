"""The seeded input generator: published splitmix64 values, rounding against
torch's conversions, determinism, and the distributions of the recipes."""
import numpy as np
import pytest
import torch

from blackwell_tensor_core_tma_gb300 import synth


def test_splitmix64_published_sequence():
    # splitmix64 started from state 0 (Vigna's reference generator): first outputs
    expect = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F,
              0xF88BB8A8724C81EC, 0x1B39896A51A8749B]
    with np.errstate(over="ignore"):
        got = synth.mix64(np.arange(1, 6, dtype=np.uint64) * synth.GAMMA)
    assert [int(x) for x in got] == expect


def test_stream_is_counter_based():
    full = synth.stream(7, 3, 0, 100)
    assert np.array_equal(full[40:60], synth.stream(7, 3, 40, 20))
    assert not np.array_equal(full, synth.stream(7, 4, 0, 100))
    assert not np.array_equal(full, synth.stream(8, 3, 0, 100))


def _probe_values(n=1 << 20, seed=11):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))
    # add exact ties of each format
    ties = np.float32(1.0) + np.float32(2.0 ** -8) * np.arange(1, 64, 2, dtype=np.float32)
    return np.concatenate([x.astype(np.float32), ties, -ties])


def test_bf16_rounding_matches_torch():
    x = _probe_values()
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f16_rounding_matches_torch():
    x = _probe_values()
    x = x[np.abs(x) < 65504]
    ours = synth.f32_to_f16_bits(x)
    ref = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_e4m3_rounding_matches_torch():
    x = _probe_values()
    x = x[np.abs(x) <= 448]
    ours = synth.f32_to_e4m3_bits(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturates():
    x = np.array([449.0, 463.9, 464.0, 1e6, -500.0], dtype=np.float32)
    assert list(synth.f32_to_e4m3_bits(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE]


def test_uniform_range_and_moments():
    u = synth.uniform_pm1(0, 0, 1 << 20).astype(np.float64)
    assert u.min() >= -1.0 and u.max() < 1.0
    assert abs(u.mean()) < 3e-3 and abs(u.var() - 1.0 / 3.0) < 3e-3
    assert np.all(np.ldexp(u, 23) == np.round(np.ldexp(u, 23)))      # 2^-23 grid


def test_normal_moments():
    z = synth.normal(2, 0, 1 << 20, sigma=0.5).astype(np.float64)
    assert abs(z.mean()) < 3e-3 and abs(z.std() - 0.5) < 3e-3
    # Box-Muller tails: P(|z| > 3 sigma) ~ 0.0027
    assert 0.0020 < np.mean(np.abs(z) > 1.5) < 0.0034


def test_ue8m0_codes():
    c = synth.ue8m0_codes(4, 3, 1 << 18)
    assert c.min() == 123 and c.max() == 131
    counts = np.bincount(c, minlength=256)[123:132]
    assert np.all(np.abs(counts / c.size - 1.0 / 9) < 0.01)


def test_make_inputs_shapes_and_determinism():
    w = synth.scaled(synth.WORKLOADS["mxf8e4m3_8192x8192x8192_c0_f32out"], 64, 48, 96)
    a = synth.make_inputs(w)
    b = synth.make_inputs(w)
    assert a["A"].shape == (64, 96) and a["A"].dtype == np.uint8
    assert a["B"].shape == (48, 96)
    assert a["SFA"].shape == (64, 3) and a["SFB"].shape == (48, 3)
    assert not a["C"].any()
    for k in a:
        assert np.array_equal(a[k], b[k])
    w2 = synth.scaled(synth.WORKLOADS["f16_4000x3000x2056_f32out"], 40, 30, 24)
    c = synth.make_inputs(w2)
    assert c["A"].dtype == np.uint16 and c["C"].dtype == np.float32 and c["C"].std() > 0.5


def test_workload_table():
    w = synth.WORKLOADS[synth.HEADLINE]
    assert (w.M, w.N, w.K, w.ab, w.d, w.seed) == (8192, 8192, 8192, "bf16", "bf16", 3)
    assert w.flops == 2 * 8192 ** 3


def test_ue4m3_codes():
    c = synth.ue4m3_codes(5, 3, 1 << 18)
    e, m = c >> 3, c & 7
    assert c.max() < 0x80                                      # no sign bit
    assert e.min() == 3 and e.max() == 11                      # 2^-4 .. 2^4
    assert np.all(np.abs(np.bincount(e, minlength=16)[3:12] / c.size - 1.0 / 9) < 0.01)
    assert np.all(np.abs(np.bincount(m, minlength=8) / c.size - 1.0 / 8) < 0.01)


def test_make_inputs_e2m1():
    w = synth.scaled(synth.WORKLOADS["nvf4e2m1_8192x8192x8192_c0_f32out"], 64, 48, 96)
    x = synth.make_inputs(w)
    assert x["A"].shape == (64, 48) and x["A"].dtype == np.uint8      # K/2 bytes per row
    assert x["B"].shape == (48, 48)
    assert x["SFA"].shape == (64, 6) and x["SFB"].shape == (48, 6)    # one scale per 16 K
    codes = synth.unpack_e2m1(x["A"])
    # N(0, 1) rounded to E2M1: zero is the most common code, 6 the saturated tail
    assert set(np.unique(codes & 7)) <= set(range(8)) and (codes & 7).max() >= 5
    w1 = synth.scaled(synth.WORKLOADS["mxf4e2m1_8192x8192x8192_c0_f32out"], 64, 48, 96)
    x1 = synth.make_inputs(w1)
    assert x1["SFA"].shape == (64, 3) and 123 <= x1["SFA"].min() and x1["SFA"].max() <= 131


def test_chain_inputs():
    w = synth.CHAIN_WORKLOADS["chain_bf16_32768x4096_256x256_bf16out"]
    assert (w.M, w.K, w.N1, w.N2, w.ab, w.d) == (32768, 4096, 256, 256, "bf16", "bf16")
    assert w.flops == 2 * 32768 * 256 * (4096 + 256)
    s = synth.scaled_chain(w, 100, 24, 16, 64)
    x = synth.make_chain_inputs(s)
    assert x["A"].shape == (100, 64) and x["B"].shape == (24, 64) and x["E"].shape == (16, 24)
    assert x["C"].shape == (100, 16) and x["A"].dtype == np.uint16
    # E has its own stream: it is not a copy of a slice of A or B
    assert not np.array_equal(x["E"].ravel(), x["B"].ravel()[:x["E"].size])
    assert np.array_equal(synth.make_chain_inputs(s)["E"], x["E"])
