"""The per-role clock trace (library variant built with GB300_TRACE=1) leaves results
unchanged and counts what it should.

A child process loads the trace variant (GB300GEMM_VARIANT=trace), runs each case with a
trace buffer attached and saves D and the counters; this process runs the same inputs
through the default library.  The two D must agree bit for bit (the cases use neither
split-K nor stream-K, so each tile's sums are formed in the same order), and the counters
must add up: every k-block of every tile consumed once by the MMA issuer, filled once by
each CTA's producer, waits and issue time within the issuer's lifetime."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

from blackwell_tensor_core_tma_gb300 import build, gemm, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (workload, M, N, K): a bf16 CTA-pair plan, a block-scaled e4m3 pair plan (copier warp) and a
# single-CTA plan, all with a D type or tile count that rules out split-K and stream-K
CASES = [
    ("bf16_8192x8192x8192_bf16out", 2048, 2048, 1024),
    ("mxf8e4m3_8192x8192x8192_c0_f32out", 2048, 2304, 1024),
    ("bf16_8192x8192x8192_bf16out", 512, 768, 640),
]


def _run(case, traced):
    import torch
    from tests import gpucase
    name, M, N, K = case
    w = synth.scaled(synth.WORKLOADS[name], M, N, K)
    x = synth.make_inputs(w)
    A, B, C = gpucase.to_device(x["A"]), gpucase.to_device(x["B"]), gpucase.to_device(x["C"])
    SFA = gpucase.to_device(x["SFA"]) if w.block_scaled else None
    SFB = gpucase.to_device(x["SFB"]) if w.block_scaled else None
    D = torch.empty((M, N), dtype=torch.bfloat16 if w.d == "bf16" else torch.float32, device="cuda")
    with gemm.Plan(M, N, K, w.ab, w.d, w.block_scaled) as plan:
        info = plan.info
        tr = None
        if traced:
            slots = gemm.gemm_testing_trace_slots()
            tr = torch.zeros(info["grid"] * slots, dtype=torch.int64, device="cuda")
            gemm.gemm_testing_set_trace(plan.handle, tr, tr.numel() * 8)
        plan.run(A, B, C, D, SFA, SFB, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert plan.last_status() == gemm.GEMM_OK
    bits = D.view(torch.int16 if w.d == "bf16" else torch.int32).cpu().numpy()
    return bits, info, (tr.cpu().numpy().reshape(info["grid"], -1) if traced else None)


def _child(out_dir):
    """Child process (trace variant loaded): D bits and counters of every case."""
    for i, case in enumerate(CASES):
        bits, info, tr = _run(case, traced=True)
        np.save(os.path.join(out_dir, f"d{i}.npy"), bits)
        np.save(os.path.join(out_dir, f"t{i}.npy"), tr)
        with open(os.path.join(out_dir, f"i{i}.json"), "w") as f:
            json.dump(info, f)


@pytest.mark.gpu
def test_trace_build_matches_default_build_and_counts_add_up(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build(variant="trace")
    env = dict(os.environ, GB300GEMM_VARIANT="trace")
    r = subprocess.run([sys.executable, "-m", "tests.test_trace_gpu", str(tmp_path)], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    F = {n: i for i, n in enumerate(gemm.TRACE_FIELDS)}
    for i, case in enumerate(CASES):
        bits, info, _ = _run(case, traced=False)
        assert np.array_equal(bits, np.load(tmp_path / f"d{i}.npy")), f"{case}: traced D differs"
        tr = np.load(tmp_path / f"t{i}.npy").astype(np.float64)
        assert json.load(open(tmp_path / f"i{i}.json")) == info
        kb_total = info["tiles"] * -(-case[3] // info["tile_k"])
        cg = info["cta_group"]
        assert tr[:, F["mma_kblocks"]].sum() == kb_total
        assert tr[:, F["prod_stages"]].sum() == cg * kb_total
        assert (tr[:, F["kernel_clk"]] > 0).all() and (tr[:, F["kernel_ns"]] > 0).all()
        mhz = tr[:, F["kernel_clk"]] / tr[:, F["kernel_ns"]] * 1e3
        assert ((mhz > 200) & (mhz < 2500)).all(), mhz
        lead = tr[:, F["mma_kblocks"]] > 0
        assert lead.sum() == info["grid"] // cg
        parts = tr[:, [F["mma_wait_acc"], F["mma_wait_ab"], F["mma_wait_sf"], F["mma_issue"]]].sum(axis=1)
        assert (parts[lead] <= tr[lead, F["mma_end"]]).all()
        assert (tr[lead, F["mma_end"]] <= 1.01 * tr[lead, F["kernel_clk"]]).all()
        assert (tr[lead, F["mma_first"]] < tr[lead, F["mma_end"]]).all()
        assert tr[:, F["mma_pieces"]].sum() == info["tiles"]
        assert tr[:, F["epi_pieces"]].sum() > 0
        if case[0].startswith("mxf8") and cg == 2:
            assert (tr[lead, F["cp_issue"]] > 0).all()          # the copier warp moved the scales


if __name__ == "__main__":
    _child(sys.argv[1])
