"""GPU parity of the two-product chain D = C + round(A·B)·E, whose intermediate
stays in tensor memory and feeds the second product as its A operand (the
tcgen05.mma form that reads A from TMEM), through the C ABI against the
oracle: ragged M, K, N1 and N2, fp16 and bf16 operands, fp32 and bf16 D, C
present or absent, repeated runs, the full-size workload on sampled rows, and
the bounded-wait timeout."""
import numpy as np
import pytest

from blackwell_tensor_core_tma_gb300 import gemm, synth
from tests import gpucase

pytestmark = pytest.mark.gpu

CW = synth.CHAIN_WORKLOADS["chain_bf16_32768x4096_256x256_bf16out"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gemm.lib()


def _pads_to_32(n):
    return (n + 15) // 16 * 16 % 32 == 0


@pytest.mark.parametrize("flags", [0, gemm.GEMM_FLAG_FORCE_1CTA], ids=["default", "1cta"])
@pytest.mark.parametrize("M,K,N1,N2,ab,d", [
    (128, 64, 16, 8, "bf16", "f32"),          # one tile, one K block, the smallest N1 and N2
    (300, 520, 200, 136, "bf16", "f32"),      # ragged M and K, N1 and N2 not multiples of 32
    (1000, 2048, 256, 256, "bf16", "bf16"),   # the full TMEM split, bf16 D
    (260, 1024, 72, 40, "f16", "f32"),        # fp16 operands and intermediate
    (512, 136, 248, 256, "f16", "bf16"),      # N1 rounds up to 256 inside the kernel
    (300, 520, 192, 96, "bf16", "f32"),       # pairs: the last pair tile holds 44 rows, its second CTA none
    (1000, 264, 32, 64, "f16", "bf16"),       # pairs: the narrowest products (16 and 32 rows of B and E per CTA)
    (777, 1000, 160, 224, "bf16", "f32"),     # pairs: ragged M and K, N1 and N2 multiples of 32
])
def test_chain_parity(M, K, N1, N2, ab, d, flags):
    """Both tile forms: CTA pairs (the default when M spans more than one 128-row tile and N1 and
    N2 pad to multiples of 32) and single CTAs."""
    w = synth.scaled_chain(CW, M, N1, N2, K, ab=ab, d=d)
    x, D, info, st, intact = gpucase.run_chain(w, flags=flags, guard=512)
    assert st == gemm.GEMM_OK and intact
    pair = flags == 0 and M > 128 and _pads_to_32(N1) and _pads_to_32(N2)
    assert info["cta_group"] == (2 if pair else 1) and info["launches_per_run"] == 1
    gpucase.check_chain(w, x, D)


@pytest.mark.parametrize("M,K,N1,N2", [(128, 64, 64, 32), (100, 200, 256, 256), (64, 128, 96, 128)])
def test_chain_forced_pairs_on_one_tile(M, K, N1, N2):
    """A pair forced onto rows that fit one CTA tile: the second CTA's rows all lie outside D."""
    w = synth.scaled_chain(CW, M, N1, N2, K)
    x, D, info, st, intact = gpucase.run_chain(w, flags=gemm.GEMM_FLAG_FORCE_2CTA, guard=256)
    assert st == gemm.GEMM_OK and intact and info["cta_group"] == 2
    gpucase.check_chain(w, x, D)


@pytest.mark.parametrize("M,K,N1,N2,ab,d,flags", [
    (20480, 1024, 256, 256, "bf16", "bf16", 0),                            # 80 pair tiles on 76 pairs
    (20000, 1000, 192, 96, "f16", "f32", 0),                               # ragged M and K, 79 pair tiles
    (20480, 1024, 128, 64, "bf16", "f32", gemm.GEMM_FLAG_FORCE_1CTA),      # 160 single tiles on 152 CTAs
    (45000, 2048, 64, 160, "bf16", "bf16", 0),                             # 176 pair tiles: two whole rounds first
])
def test_chain_stream_k(M, K, N1, N2, ab, d, flags):
    """Stream-K over the first product (on request: chain plans default to whole tiles): a tile
    cut between two units is finished by the one that computed its first k-blocks, after adding
    the other's partial T (the oracle's bound covers the different grouping of the fp32 sums);
    the same shapes without stream-K agree within it too."""
    w = synth.scaled_chain(CW, M, N1, N2, K, ab=ab, d=d)
    x = synth.make_chain_inputs(w)
    for sk in (1, 0):
        _, D, info, st, intact = gpucase.run_chain(w, flags=flags, guard=256, inputs=x, stream_k=sk, reps=2)
        assert st == gemm.GEMM_OK and intact and info["stream_k"] == sk
        gpucase.check_chain(w, x, D)


def test_chain_c_none_and_repeat():
    w = synth.scaled_chain(CW, 640, 128, 96, 384)
    x, D, info, st, intact = gpucase.run_chain(w, c_none=True, guard=256, reps=3)
    assert st == gemm.GEMM_OK and intact
    gpucase.check_chain(w, x, D, c_none=True)


def test_chain_full_size_sampled_rows():
    w = CW
    x, D, info, st, intact = gpucase.run_chain(w, guard=1024)
    assert st == gemm.GEMM_OK and intact and info["cta_group"] == 2 and info["stream_k"] == 0
    rng = np.random.default_rng(0)
    edges = [r for t in range(0, w.M, 128 * 37) for r in (t, t + 31, t + 32, t + 127) if r < w.M]
    rows = np.unique(np.concatenate([edges, [w.M - 1], rng.integers(0, w.M, 160)]))
    gpucase.check_chain(w, x, D, rows=rows)


def test_chain_rejected_by_gemm_run():
    import torch
    with gemm.ChainPlan(128, 64, 64, 64) as plan:
        z = torch.zeros(128 * 128, dtype=torch.float32, device="cuda")
        with pytest.raises(gemm.GemmError) as e:
            gemm.gemm_run(plan.handle, z, z, None, z)
        assert e.value.status == gemm.GEMM_ERR_INVALID_ARG


def test_chain_timeout_and_recovery():
    import torch
    w = synth.scaled_chain(CW, 384, 128, 64, 256)
    x = synth.make_chain_inputs(w)
    A, B, E, C = (gpucase.to_device(x[k]) for k in ("A", "B", "E", "C"))
    D = torch.zeros((w.M, w.N2), dtype=torch.bfloat16, device="cuda")
    with gemm.ChainPlan(w.M, w.N1, w.N2, w.K, w.ab, w.d) as plan:
        plan.set_timeout(20_000_000)
        gemm.gemm_testing_set_fault(plan.handle, 1)
        plan.run(A, B, E, C, D, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert plan.last_status() == gemm.GEMM_ERR_TIMEOUT
        gemm.gemm_testing_set_fault(plan.handle, 0)
        plan.set_timeout(1_000_000_000)
        plan.run(A, B, E, C, D, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert plan.last_status() == gemm.GEMM_OK
    gpucase.check_chain(w, x, gpucase.decode_d(D, w.d))


@pytest.mark.parametrize("M,K,N1,N2,d,c_none", [
    (1000, 520, 200, 136, "bf16", False),     # ragged, bf16 D (single CTAs)
    (640, 1024, 256, 256, "f32", True),       # C absent (CTA pairs)
])
def test_chain_host_run(M, K, N1, N2, d, c_none):
    """gemm_chain_run_host: the same result from pinned host buffers as from device buffers."""
    import torch
    w = synth.scaled_chain(CW, M, N1, N2, K, d=d)
    x, D_dev, info, st, intact = gpucase.run_chain(w, c_none=c_none)
    assert st == gemm.GEMM_OK
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int16) if a.dtype == np.uint16 else a)).pin_memory()
    hD = torch.full((M, N2), float("nan"), dtype=torch.bfloat16 if d == "bf16" else torch.float32).pin_memory()
    with gemm.ChainPlan(M, N1, N2, K, w.ab, d) as plan:
        assert plan.run_host(pin(x["A"]), pin(x["B"]), pin(x["E"]), None if c_none else pin(x["C"]), hD,
                             torch.cuda.current_stream()) == gemm.GEMM_OK
    D_host = gpucase.decode_d(hD, d)
    assert np.array_equal(D_host, D_dev)
    gpucase.check_chain(w, x, D_host, c_none=c_none)
