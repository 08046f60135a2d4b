"""The allocation-free entry point gemm_run_noalloc, for callers that cannot
call cudaMalloc (a host program whose allocator owns all device memory, a
latency-critical loop that cannot take cudaMalloc's device-wide
synchronisation, a plug-in on a fixed memory budget).

Two calls in a row, each through the C ABI, are compared with the plan entry
point gemm_run on the same inputs, under the accept rule the other GPU tests
use.  This file is collected last so that a run stopping at its first failure
has already run every other test; it also passes alone in a fresh process
(its first call does the one-time device set-up)."""
import numpy as np
import pytest

import oracle
from blackwell_tensor_core_tma_gb300 import gemm, synth
from tests import gpucase

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gemm.lib()


def _setup(w, c_none):
    import torch
    x = synth.make_inputs(w)
    A, B = gpucase.to_device(x["A"]), gpucase.to_device(x["B"])
    C = None if c_none else gpucase.to_device(x["C"])
    tdt = torch.bfloat16 if w.d == "bf16" else torch.float32
    D_plan = torch.full((w.M, w.N), float("nan"), dtype=tdt, device="cuda")
    D_free = torch.full((w.M, w.N), float("nan"), dtype=tdt, device="cuda")
    with gemm.Plan(w.M, w.N, w.K, w.ab, w.d) as plan:
        plan.run(A, B, C, D_plan, None, None, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert plan.last_status() == gemm.GEMM_OK
    return dict(w=w, c_none=c_none, x=x, A=A, B=B, C=C, D_plan=D_plan, D_free=D_free)


def test_two_calls_in_a_row_match_gemm_run():
    import torch
    cases = [
        _setup(synth.scaled(synth.WORKLOADS["f16_4000x3000x2056_f32out"], 1000, 600, 520), False),
        _setup(synth.scaled(synth.WORKLOADS["bf16_8192x8192x8192_bf16out"], 1100, 1048, 1032), True),
    ]
    stream = torch.cuda.current_stream()
    for k in cases:                                   # two allocation-free calls back to back
        w = k["w"]
        st = gemm.gemm_run_noalloc(w.M, w.N, w.K, w.ab, w.d, k["A"], k["B"], k["C"], k["D_free"], stream, wait=1)
        assert st == gemm.GEMM_OK
    for k in cases:
        w, x, c_none = k["w"], k["x"], k["c_none"]
        D_plan = gpucase.decode_d(k["D_plan"], w.d)
        D_free = gpucase.decode_d(k["D_free"], w.d)
        D_ref, S = oracle.gemm(x["A"], x["B"], None if c_none else x["C"], w.M, w.N, w.K, w.ab)
        c = np.zeros_like(S) if c_none else x["C"].astype(np.float64)
        tol = gpucase.tolerance(w, D_ref, S, c)
        assert np.all(np.abs(D_free - D_plan) <= tol)
        assert np.all(np.abs(D_free - D_ref) <= tol)


def test_enqueue_only_call_then_waiting_call_on_one_stream():
    """A caller on a latency-critical path enqueues without waiting (wait = 0); the next call
    on the same stream waits.  Its clearing of the shared status word is ordered after the
    first kernel by the stream, so both products come out right and the second call reports
    the status of its own kernel."""
    import torch
    cases = [
        _setup(synth.scaled(synth.WORKLOADS["bf16_4096x4096x4096_f32out"], 1040, 1280, 776), False),
        _setup(synth.scaled(synth.WORKLOADS["f16_4000x3000x2056_f32out"], 700, 264, 1112), True),
    ]
    stream = torch.cuda.current_stream()
    for k, wait in zip(cases, (0, 1)):
        w = k["w"]
        st = gemm.gemm_run_noalloc(w.M, w.N, w.K, w.ab, w.d, k["A"], k["B"], k["C"], k["D_free"], stream,
                                   wait=wait)
        assert st == gemm.GEMM_OK
    torch.cuda.synchronize()
    for k in cases:
        w, x, c_none = k["w"], k["x"], k["c_none"]
        D_plan = gpucase.decode_d(k["D_plan"], w.d)
        D_free = gpucase.decode_d(k["D_free"], w.d)
        D_ref, S = oracle.gemm(x["A"], x["B"], None if c_none else x["C"], w.M, w.N, w.K, w.ab)
        c = np.zeros_like(S) if c_none else x["C"].astype(np.float64)
        tol = gpucase.tolerance(w, D_ref, S, c)
        assert np.all(np.abs(D_free - D_plan) <= tol)
        assert np.all(np.abs(D_free - D_ref) <= tol)


def test_waiting_call_is_refused_on_a_capturing_stream():
    """Synchronising inside a graph capture would break the capture: a waiting call on a
    capturing stream is refused before anything is enqueued, and the capture stays valid."""
    import torch
    w = synth.scaled(synth.WORKLOADS["bf16_4096x4096x4096_f32out"], 256, 256, 256)
    x = synth.make_inputs(w)
    A, B = gpucase.to_device(x["A"]), gpucase.to_device(x["B"])
    D = torch.empty((w.M, w.N), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    # the device's one-time set-up happens outside the capture
    assert gemm.gemm_run_noalloc(w.M, w.N, w.K, w.ab, w.d, A, B, None, D, s, wait=1) == gemm.GEMM_OK
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        g.capture_begin()
        try:
            with pytest.raises(gemm.GemmError) as e:
                gemm.gemm_run_noalloc(w.M, w.N, w.K, w.ab, w.d, A, B, None, D, s, wait=1)
        finally:
            g.capture_end()
    assert e.value.status == gemm.GEMM_ERR_INVALID_ARG


def test_rejects_bad_arguments_without_launching():
    with pytest.raises(gemm.GemmError) as e:
        gemm.gemm_run_noalloc(0, 256, 256, "bf16", "f32", 16, 16, None, 16)
    assert e.value.status == gemm.GEMM_ERR_INVALID_ARG
    with pytest.raises(gemm.GemmError) as e:
        gemm.gemm_run_noalloc(256, 256, 2057, "bf16", "f32", 16, 16, None, 16)
    assert e.value.status == gemm.GEMM_ERR_ALIGNMENT
    with pytest.raises(gemm.GemmError) as e:
        gemm.gemm_run_noalloc(256, 256, 256, "e4m3", "f32", 16, 16, None, 16)
    assert e.value.status == gemm.GEMM_ERR_UNSUPPORTED
