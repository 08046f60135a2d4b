"""The C-ABI library builds, loads without a GPU, exports every symbol the
headers declare, and rejects bad plans before touching a device."""
import os
import re

import pytest

from tests import rules
from blackwell_tensor_core_tma_gb300 import build, gemm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in ("gb300gemm.h", "gb300gemm_testing.h"):
        text = open(os.path.join(ROOT, "include", h)).read()
        names |= set(re.findall(r"^\s*(?:gemm_status|const char \*|int)\s*\**(gemm_\w+)\s*\(", text, re.M))
    return names


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gemm.lib()


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert declared == set(gemm.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_enum_values_match_header():
    text = open(os.path.join(ROOT, "include", "gb300gemm.h")).read()
    for name in ("GEMM_F16", "GEMM_BF16", "GEMM_E4M3", "GEMM_F32", "GEMM_E2M1"):
        assert int(re.search(rf"\b{name} = (\d+)", text).group(1)) == getattr(gemm, name)
    for name in ("GEMM_SCALE_NONE", "GEMM_SCALE_UE8M0_32", "GEMM_SCALE_UE4M3_16"):
        assert int(re.search(rf"#define {name}\s+(\d+)", text).group(1)) == getattr(gemm, name)


def test_status_strings(lib):
    for s in range(6):
        assert gemm.gemm_status_string(s)
    assert "unknown" in gemm.gemm_status_string(99)


@pytest.mark.parametrize("args,status", [
    ((0, 256, 256), gemm.GEMM_ERR_INVALID_ARG),
    ((256, -1, 256), gemm.GEMM_ERR_INVALID_ARG),
    ((256, 256, 0), gemm.GEMM_ERR_INVALID_ARG),
    ((256, 256, 2057), gemm.GEMM_ERR_ALIGNMENT),     # 16-bit K-major rows of 4114 bytes
    ((256, 258, 256), gemm.GEMM_ERR_ALIGNMENT),      # fp32 C rows of 1032 bytes
])
def test_plan_rejects_before_device(lib, args, status):
    with pytest.raises(gemm.GemmError) as e:
        gemm.gemm_plan_create(*args)
    assert e.value.status == status


def test_plan_rejects_unsupported_combinations(lib):
    cases = [
        dict(ab="f32"), dict(c="bf16"), dict(d="f16"),
        dict(ab="e4m3", block_scaled=0), dict(ab="bf16", block_scaled=1),
        dict(ab="e2m1", block_scaled=0), dict(ab="e4m3", block_scaled=2), dict(ab="bf16", block_scaled=2),
        dict(ab="e2m1", block_scaled=1, a_row_major=0), dict(ab="e2m1", block_scaled=2, b_row_major=1),
    ]
    for kw in cases:
        with pytest.raises(gemm.GemmError) as e:
            gemm.gemm_plan_create(256, 256, 256, **kw)
        assert e.value.status == gemm.GEMM_ERR_UNSUPPORTED, kw
    with pytest.raises(gemm.GemmError) as e:
        gemm.gemm_plan_create(256, 256, 256, flags=gemm.GEMM_FLAG_FORCE_1CTA | gemm.GEMM_FLAG_FORCE_2CTA)
    assert e.value.status == gemm.GEMM_ERR_INVALID_ARG
    for mode in (-1, 3):
        with pytest.raises(gemm.GemmError) as e:
            gemm.gemm_plan_create(256, 256, 256, ab="e2m1", block_scaled=mode)
        assert e.value.status == gemm.GEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("K", [16, 48, 272])
def test_e2m1_rows_must_hold_16_bytes(lib, K):
    # packed 4-bit K-major rows of K/2 bytes: K must be a multiple of 32
    with pytest.raises(gemm.GemmError) as e:
        gemm.gemm_plan_create(256, 256, K, ab="e2m1", block_scaled=2)
    assert e.value.status == gemm.GEMM_ERR_ALIGNMENT


def test_null_plan_calls(lib):
    assert lib.gemm_run(None, None, None, None, None, None, None, None) == gemm.GEMM_ERR_INVALID_ARG
    assert lib.gemm_plan_last_status(None) == gemm.GEMM_ERR_INVALID_ARG
    assert lib.gemm_plan_destroy(None) == gemm.GEMM_OK
    assert lib.gemm_plan_set_timeout(None, 10) == gemm.GEMM_ERR_INVALID_ARG
    assert lib.gemm_testing_set_fault(None, 1) == gemm.GEMM_ERR_INVALID_ARG


def test_no_cpu_fallback_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(build, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(gemm, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU path"):
        gemm.lib()


@pytest.mark.parametrize("args,kw,status", [
    ((0, 64, 64, 64), {}, gemm.GEMM_ERR_INVALID_ARG),
    ((128, 264, 64, 64), {}, gemm.GEMM_ERR_UNSUPPORTED),                    # N1 > 256
    ((128, 64, 272, 64), {}, gemm.GEMM_ERR_UNSUPPORTED),                    # N2 > 256
    ((128, 64, 64, 64), {"ab": "e4m3"}, gemm.GEMM_ERR_UNSUPPORTED),
    ((128, 64, 48, 64), {"flags": gemm.GEMM_FLAG_FORCE_2CTA}, gemm.GEMM_ERR_UNSUPPORTED),  # pair N2 not % 32
    ((128, 40, 64, 64), {"flags": gemm.GEMM_FLAG_FORCE_2CTA}, gemm.GEMM_ERR_UNSUPPORTED),  # pair N1 pads to 48
    ((128, 64, 64, 60), {}, gemm.GEMM_ERR_ALIGNMENT),                       # K rows of 120 bytes
    ((128, 60, 64, 64), {}, gemm.GEMM_ERR_ALIGNMENT),                       # E rows of N1 = 60
    ((128, 64, 12, 64), {"d": "bf16"}, gemm.GEMM_ERR_ALIGNMENT),            # bf16 D rows of 24 bytes
])
def test_chain_plan_rejects_before_device(lib, args, kw, status):
    with pytest.raises(gemm.GemmError) as e:
        gemm.gemm_chain_plan_create(*args, **kw)
    assert e.value.status == status


def test_chain_calls_reject_null(lib):
    assert lib.gemm_chain_run(None, None, None, None, None, None, None) == gemm.GEMM_ERR_INVALID_ARG
    assert lib.gemm_chain_run_host(None, None, None, None, None, None, None) == gemm.GEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("args,status", [
    ((gemm.GEMM_BF16, 0, 3, 64), gemm.GEMM_ERR_INVALID_ARG),        # cta_group 3
    ((gemm.GEMM_BF16, 0, 2, 0), gemm.GEMM_ERR_INVALID_ARG),         # no iterations
    ((gemm.GEMM_BF16, 0, 2, (1 << 20) + 1), gemm.GEMM_ERR_INVALID_ARG),
    ((gemm.GEMM_BF16, 5, 2, 64), gemm.GEMM_ERR_INVALID_ARG),        # block_scaled out of range
    ((gemm.GEMM_F32, 0, 2, 64), gemm.GEMM_ERR_UNSUPPORTED),
    ((gemm.GEMM_E4M3, gemm.GEMM_SCALE_UE4M3_16, 2, 64), gemm.GEMM_ERR_UNSUPPORTED),
    ((gemm.GEMM_BF16, gemm.GEMM_SCALE_UE8M0_32, 1, 64), gemm.GEMM_ERR_UNSUPPORTED),
])
def test_tensor_rate_probe_rejects_before_device(lib, args, status):
    out = gemm.TensorRate()
    import ctypes
    assert lib.gemm_measure_tensor_rate(*args, ctypes.byref(out)) == status
    assert lib.gemm_measure_tensor_rate(gemm.GEMM_BF16, 0, 2, 64, None) == gemm.GEMM_ERR_INVALID_ARG


def _tile_rule(M, N, K, f32, units=76):
    """The pair tile-width rule restated from its definition (column share x round share, 0.89
    under stream-K, x 0.965 for 224 or the wide-epilogue gain for 256; 224 must win by 2 %)."""
    tiles_m, kb = -(-M // 256), -(-K // 64)

    def eff(bn):
        tn = -(-N // bn)
        tiles = tiles_m * tn
        rounds = -(-tiles // units)
        sk = f32 and kb >= 64 and tiles >= units and tiles % units != 0 and tiles < 4 * units
        e = N / (tn * bn) * (0.89 if sk else tiles / (rounds * units))
        if bn == 224:
            e *= 0.965
        elif f32 and kb <= 40 and 2 * tiles > units:
            e *= 1.0 + 0.1 * (40 - kb) / 24.0
        return e
    return 224 if eff(224) > 1.02 * eff(256) else 256


def test_pair_tile_rule_without_device(lib):
    import ctypes
    import numpy as np
    out = ctypes.c_int()
    # the measured cases: 4096^3 and 4000x3000x2056 take 224; 8192^3, 2048x2560x4096 (both
    # tilings need stream-K) and 4096x4096x1024 (the wide epilogue) keep 256
    for (M, N, K, d), want in [((4096, 4096, 4096, gemm.GEMM_F32), 224), ((4000, 3000, 2056, gemm.GEMM_F32), 224),
                               ((8192, 8192, 8192, gemm.GEMM_BF16), 256), ((2048, 2560, 4096, gemm.GEMM_F32), 256),
                               ((4096, 4096, 1024, gemm.GEMM_F32), 256), ((4096, 4096, 4096, gemm.GEMM_BF16), 224)]:
        assert lib.gemm_testing_pair_tile_n(M, N, K, d, 76, ctypes.byref(out)) == gemm.GEMM_OK
        assert out.value == want, (M, N, K, d)
    rng = np.random.default_rng(7)
    for _ in range(2000):
        M, N, K = (int(v) for v in rng.integers(1, 20000, 3))
        d = gemm.GEMM_F32 if rng.integers(2) else gemm.GEMM_BF16
        units = int(rng.integers(1, 160))
        assert lib.gemm_testing_pair_tile_n(M, N, K, d, units, ctypes.byref(out)) == gemm.GEMM_OK
        assert out.value == _tile_rule(M, N, K, d == gemm.GEMM_F32, units), (M, N, K, d, units)
    assert lib.gemm_testing_pair_tile_n(0, 1, 1, gemm.GEMM_F32, 76, ctypes.byref(out)) == gemm.GEMM_ERR_INVALID_ARG
    assert lib.gemm_testing_pair_tile_n(1, 1, 1, gemm.GEMM_F16, 76, ctypes.byref(out)) == gemm.GEMM_ERR_INVALID_ARG
    assert lib.gemm_testing_pair_tile_n(1, 1, 1, gemm.GEMM_F32, 76, None) == gemm.GEMM_ERR_INVALID_ARG


def test_e4m3_pair_tile_rule_without_device(lib):
    import ctypes
    import numpy as np
    out = ctypes.c_int()
    # the measured cases: 224 won at 4096^3 (+16 %) and 4096 x 4096 x 8192 (+6 %, against
    # 256-wide tiles under stream-K) and lost at 8192^3, 6144^3 and 3072 x 3072 x 8192
    for (M, N, K), want in [((4096, 4096, 4096), 224), ((4096, 4096, 8192), 224), ((8192, 8192, 8192), 256),
                            ((6144, 6144, 6144), 256), ((3072, 3072, 8192), 256)]:
        assert lib.gemm_testing_e4m3_pair_tile_n(M, N, K, gemm.GEMM_F32, 76, ctypes.byref(out)) == gemm.GEMM_OK
        assert out.value == want, (M, N, K)
    rng = np.random.default_rng(9)
    for _ in range(2000):
        M, N, K = (int(v) for v in rng.integers(1, 20000, 3))
        d = gemm.GEMM_F32 if rng.integers(2) else gemm.GEMM_BF16
        units = int(rng.integers(1, 160))
        assert lib.gemm_testing_e4m3_pair_tile_n(M, N, K, d, units, ctypes.byref(out)) == gemm.GEMM_OK
        assert out.value == rules.e4m3_tile_rule(M, N, K, d == gemm.GEMM_F32, units), (M, N, K, d, units)
    assert lib.gemm_testing_e4m3_pair_tile_n(0, 1, 1, gemm.GEMM_F32, 76, ctypes.byref(out)) == gemm.GEMM_ERR_INVALID_ARG
    assert lib.gemm_testing_e4m3_pair_tile_n(1, 1, 1, gemm.GEMM_F32, 76, None) == gemm.GEMM_ERR_INVALID_ARG


def test_product_code_does_not_reach_the_oracle():
    """The package (binding, builders, CUDA sources) neither imports nor links the CPU oracle;
    only tests, smoke() and the bench's CPU legs may use it."""
    pkg = os.path.join(ROOT, "blackwell_tensor_core_tma_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if not f.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                continue
            text = open(os.path.join(dirpath, f), encoding="utf-8").read()
            assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
            assert "liboracle" not in text and "gemm_oracle" not in text, f


def test_trace_is_compiled_out_of_the_default_library(lib):
    """The default build keeps no per-role trace: no counters, and setting one is refused."""
    assert lib.gemm_testing_trace_slots() == 0
    assert gemm.gemm_testing_trace_slots() == 0


def test_trace_counter_names_follow_the_kernel_slots():
    """The binding's counter names are the kernel's trace slots, in order (parsed from the
    internal header), and the trace build reports that many slots per CTA."""
    text = open(os.path.join(ROOT, "blackwell_tensor_core_tma_gb300", "csrc", "gemm_internal.h")).read()
    body = re.search(r"enum TraceSlot : int \{(.*?)\};", text, re.S).group(1)
    names = re.findall(r"^\s*TR_(\w+)", body, re.M)
    slots = int(re.search(r"TRACE_SLOTS = (\d+)", body).group(1))
    assert [n.lower() for n in names] == gemm.TRACE_FIELDS
    assert len(names) <= slots
    import ctypes
    L = ctypes.CDLL(build.build(variant="trace"))
    L.gemm_testing_trace_slots.restype = ctypes.c_int
    assert L.gemm_testing_trace_slots() == slots
