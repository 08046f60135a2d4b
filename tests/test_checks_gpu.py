"""The checks build of the library (variant "checks": the kernels' on-device checks of every
computed TMA coordinate, and ring depths other than the default ones).

A child process loads the checks variant (GB300GEMM_VARIANT=checks) and runs one case of
every kernel family and mode: CTA pairs and single CTAs, ragged edges, MN-major operands,
split-K, stream-K, the three block-scaled kinds, and the two-product chain in both tile
forms.  Every run must end GEMM_OK (no check fired) with D within the oracle's bound, and,
where the order of the sums does not depend on the launch (no split-K, asked for or chosen by
the plan for few tiles, whose slices reduce-add in L2 in any order), bit-equal to the default
library's D although the rings are of other depths.  A planted error (test hook fault 2: A rows one tiled extent too far,
which only reads the fill value) must come back as GEMM_ERR_CHECK from the checks build and
pass unreported through the default one, where the checks are compiled out."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

from blackwell_tensor_core_tma_gb300 import build, gemm, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
W = synth.WORKLOADS
F1, F2 = gemm.GEMM_FLAG_FORCE_1CTA, gemm.GEMM_FLAG_FORCE_2CTA

# (name, workload, M, N, K, flags, splits, a_row_major, b_row_major)
GEMM_CASES = [
    ("pair_bf16_ragged", "bf16_8192x8192x8192_bf16out", 1100, 1048, 1032, 0, 0, True, False),
    ("single_f16_ragged", "f16_4000x3000x2056_f32out", 1000, 600, 520, F1, 0, True, False),
    ("pair_mn_major", "bf16_4096x4096x4096_f32out", 520, 776, 648, F2, 0, False, True),
    ("single_mn_major", "bf16_4096x4096x4096_f32out", 264, 392, 520, F1, 0, False, True),
    ("pair_stream_k", "bf16_4096x4096x4096_f32out", 2048, 2560, 4096, F2, 0, True, False),
    ("single_split_k", "bf16_4096x4096x4096_f32out", 264, 136, 4096, F1, 7, True, False),
    ("pair_e4m3", "mxf8e4m3_8192x8192x8192_c0_f32out", 1000, 1040, 1056, F2, 0, True, False),
    ("single_e4m3_mn", "mxf8e4m3_8192x8192x8192_c0_f32out", 528, 400, 640, F1, 0, False, False),
    ("pair_e2m1_ue8m0", "mxf4e2m1_8192x8192x8192_c0_f32out", 1048, 776, 1056, F2, 0, True, False),
    ("pair_e2m1_ue4m3", "nvf4e2m1_8192x8192x8192_c0_f32out", 1048, 776, 1056, F2, 0, True, False),
]
# (name, M, K, N1, N2, flags)
CHAIN_CASES = [
    ("chain_pair", 777, 1000, 160, 224, 0),
    ("chain_single", 300, 520, 200, 136, 0),
]
PLANTED = ("pair_bf16_ragged", "single_f16_ragged")
# cases whose kernel instance takes its ring depth from the knobs the checks build sets
OTHER_DEPTH = ("pair_bf16_ragged", "single_f16_ragged", "pair_stream_k", "pair_e4m3", "pair_e2m1_ue8m0",
               "pair_e2m1_ue4m3")


def _values(bits, d):
    """fp64 values of D's raw codes (bf16 codes widened exactly)."""
    if d == "bf16":
        return (bits.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return bits.view(np.float32).astype(np.float64)


def _gemm_w(case):
    _, name, M, N, K, flags, splits, a_rm, b_rm = case
    return synth.scaled(W[name], M, N, K, c="normal", a_row_major=a_rm, b_row_major=b_rm)


def _run_gemm(case, fault=0):
    import torch
    from tests import gpucase
    w = _gemm_w(case)
    flags, splits = case[5], case[6]
    x = synth.make_inputs(w)
    A, B, C = gpucase.to_device(x["A"]), gpucase.to_device(x["B"]), gpucase.to_device(x["C"])
    SFA = gpucase.to_device(x["SFA"]) if w.block_scaled else None
    SFB = gpucase.to_device(x["SFB"]) if w.block_scaled else None
    D = torch.full((w.M, w.N), float("nan"), dtype=torch.bfloat16 if w.d == "bf16" else torch.float32,
                   device="cuda")
    with gemm.Plan(w.M, w.N, w.K, w.ab, w.d, w.block_scaled, flags, a_row_major=w.a_row_major,
                   b_row_major=w.b_row_major) as plan:
        if splits:
            plan.set_split_k(splits)
        if fault:
            gemm.gemm_testing_set_fault(plan.handle, fault)
        plan.run(A, B, C, D, SFA, SFB, torch.cuda.current_stream())
        torch.cuda.synchronize()
        status, info = plan.last_status(), plan.info
    return D.view(torch.int16 if w.d == "bf16" else torch.int32).cpu().numpy(), status, info


def _run_chain(case):
    from tests import gpucase
    name, M, K, N1, N2, flags = case
    w = synth.scaled_chain(synth.CHAIN_WORKLOADS["chain_bf16_32768x4096_256x256_bf16out"], M, N1, N2, K)
    x, D, info, status, intact = gpucase.run_chain(w, flags=flags, guard=64)
    assert intact
    return D, status, info


def _child(out_dir):
    """Child process (checks variant loaded): D, status and plan of every case."""
    res = {}
    for case in GEMM_CASES:
        bits, st, info = _run_gemm(case)
        np.save(os.path.join(out_dir, case[0] + ".npy"), bits)
        res[case[0]] = {"status": st, "stages": info["stages"], "splits": info["splits"]}
    for case in CHAIN_CASES:
        D, st, info = _run_chain(case)
        np.save(os.path.join(out_dir, case[0] + ".npy"), D)
        res[case[0]] = {"status": st, "stages": info["stages"], "cta_group": info["cta_group"]}
    for name in PLANTED:
        _, st, _ = _run_gemm(next(c for c in GEMM_CASES if c[0] == name), fault=2)
        res["planted_" + name] = {"status": st}
    with open(os.path.join(out_dir, "res.json"), "w") as f:
        json.dump(res, f)


def test_checks_variant_is_a_known_build():
    assert "checks" in build.VARIANTS and "-DGB300_CHECKS=1" in build.VARIANTS["checks"]
    assert build.lib_path("checks").endswith("libgb300gemm_checks.so")


def test_check_status_code():
    import ctypes
    L = ctypes.CDLL(build.build())
    L.gemm_status_string.restype = ctypes.c_char_p
    assert gemm.GEMM_ERR_CHECK == 6
    assert L.gemm_status_string(gemm.GEMM_ERR_CHECK) == b"an on-device check of a copy coordinate failed"


@pytest.mark.gpu
def test_checks_build_passes_every_family_and_catches_a_planted_error(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tests import gpucase
    build.build(variant="checks")
    env = dict(os.environ, GB300GEMM_VARIANT="checks")
    r = subprocess.run([sys.executable, "-m", "tests.test_checks_gpu", str(tmp_path)], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.load(open(tmp_path / "res.json"))
    for case in GEMM_CASES:
        name = case[0]
        assert res[name]["status"] == gemm.GEMM_OK, name
        bits, st, info = _run_gemm(case)
        assert st == gemm.GEMM_OK
        if name in OTHER_DEPTH:
            assert res[name]["stages"] != info["stages"], f"{name}: the checks build runs another ring depth"
        w = _gemm_w(case)
        checked = np.load(tmp_path / f"{name}.npy")
        gpucase.check_full(w, synth.make_inputs(w), _values(checked, w.d))
        if info["splits"] == 1 and res[name]["splits"] == 1:
            assert np.array_equal(checked, bits), f"{name}: checks build differs from the default build"
    for case in CHAIN_CASES:
        name = case[0]
        assert res[name]["status"] == gemm.GEMM_OK, name
        D, st, info = _run_chain(case)
        assert st == gemm.GEMM_OK and res[name]["cta_group"] == info["cta_group"]
        assert np.array_equal(np.load(tmp_path / f"{name}.npy"), D), f"{name}: checks build differs"
    for name in PLANTED:
        assert res["planted_" + name]["status"] == gemm.GEMM_ERR_CHECK, name
        _, st, _ = _run_gemm(next(c for c in GEMM_CASES if c[0] == name), fault=2)
        assert st == gemm.GEMM_OK          # the default build compiles the checks out


if __name__ == "__main__":
    _child(sys.argv[1])
