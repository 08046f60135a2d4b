"""Randomised parity sweep: seeded random shapes (from a single row up to a few tiles,
every ragged edge), every operand kind, every storage order it allows, both D types,
C present or absent and both CTA modes, each checked in full against the oracle."""
import numpy as np
import pytest

from blackwell_tensor_core_tma_gb300 import gemm, synth
from tests import gpucase

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
# recipe, K granule (contiguous-K rows of 16 bytes), contiguous-M/N granule, storage orders allowed
KINDS = {
    "bf16": ("bf16_4096x4096x4096_f32out", 8, 8, True),
    "f16": ("f16_4000x3000x2056_f32out", 8, 8, True),
    "e4m3": ("mxf8e4m3_8192x8192x8192_c0_f32out", 16, 16, True),
    "mxf4": ("mxf4e2m1_8192x8192x8192_c0_f32out", 32, None, False),
    "nvf4": ("nvf4e2m1_8192x8192x8192_c0_f32out", 32, None, False),
}


def _cases(n=150, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    fixed = [("bf16", 1, 8, 8, True, False, "f32", True, 0), ("f16", 1, 8, 8, True, False, "bf16", False, 0),
             ("e4m3", 1, 16, 16, True, False, "f32", True, 0), ("mxf4", 3, 8, 32, True, False, "f32", True, 0),
             ("nvf4", 2, 16, 32, True, False, "bf16", True, 0)]
    out += fixed
    kinds = list(KINDS)
    for _ in range(n - len(fixed)):
        kind = kinds[rng.integers(len(kinds))]
        _, kg, mg, any_order = KINDS[kind]
        a_rm = True if not any_order else bool(rng.integers(2))
        b_rm = False if not any_order else bool(rng.integers(2))
        d = "bf16" if rng.integers(2) else "f32"
        M = int(rng.integers(1, 700))
        N = int(rng.integers(1, 600))
        K = int(rng.integers(1, 1100))
        ng = 8 if d == "bf16" else 4
        if b_rm:
            ng = int(np.lcm(ng, mg))
        N = max(ng, N // ng * ng)
        if a_rm or not b_rm:                    # some operand has K-contiguous rows
            K = max(kg, K // kg * kg)
        if not a_rm:
            M = max(mg, M // mg * mg)
        cta = int(rng.integers(3))              # 0 plan's choice, 1 single CTAs, 2 pairs
        if kind == "e4m3" and b_rm and cta == 1:
            cta = 2                             # row-major B needs CTA pairs for e4m3
        out.append((kind, M, N, K, a_rm, b_rm, d, bool(rng.integers(2)), cta))
    return out


CASES = _cases()


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gemm.lib()


@pytest.mark.parametrize("kind,M,N,K,a_rm,b_rm,d,with_c,cta", CASES,
                         ids=[f"{c[0]}-{c[1]}x{c[2]}x{c[3]}-{'A' if c[4] else 'At'}{'Bt' if c[5] else 'B'}-{c[6]}"
                              f"-{'C' if c[7] else 'noC'}-cg{c[8]}" for c in CASES])
def test_random_shape(kind, M, N, K, a_rm, b_rm, d, with_c, cta):
    recipe = KINDS[kind][0]
    w = synth.scaled(W[recipe], M, N, K, d=d, c="normal", a_row_major=a_rm, b_row_major=b_rm)
    flags = {0: 0, 1: gemm.GEMM_FLAG_FORCE_1CTA, 2: gemm.GEMM_FLAG_FORCE_2CTA}[cta]
    x, D, info, st, intact = gpucase.run(w, flags=flags, c_none=not with_c, guard=128)
    assert st == gemm.GEMM_OK and intact
    gpucase.check_full(w, x, D, c_none=not with_c)


def _chain_cases(n=20, seed=7):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        d = "bf16" if rng.integers(2) else "f32"
        ab = "bf16" if rng.integers(2) else "f16"
        M = int(rng.integers(1, 600))
        K = int(rng.integers(1, 800)) // 8 * 8 or 8
        N1 = int(rng.integers(1, 257)) // 8 * 8 or 8
        N2 = int(rng.integers(1, 257)) // 8 * 8 or 8
        out.append((M, K, N1, N2, ab, d, bool(rng.integers(2))))
    return out


CHAIN_CASES = _chain_cases()


def _chain_pair_cases(n=12, seed=8):
    """Shapes the plan runs as CTA pairs: more than 128 rows, N1 and N2 multiples of 32."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        d = "bf16" if rng.integers(2) else "f32"
        ab = "bf16" if rng.integers(2) else "f16"
        M = int(rng.integers(129, 1400))
        K = int(rng.integers(1, 1200)) // 8 * 8 or 8
        N1 = 32 * int(rng.integers(1, 9))
        N2 = 32 * int(rng.integers(1, 9))
        out.append((M, K, N1, N2, ab, d, bool(rng.integers(2))))
    return out


CHAIN_PAIR_CASES = _chain_pair_cases()


@pytest.mark.parametrize("M,K,N1,N2,ab,d,with_c", CHAIN_CASES,
                         ids=[f"{c[0]}x{c[1]}-{c[2]}x{c[3]}-{c[4]}-{c[5]}-{'C' if c[6] else 'noC'}" for c in CHAIN_CASES])
def test_random_chain(M, K, N1, N2, ab, d, with_c):
    cw = synth.scaled_chain(synth.CHAIN_WORKLOADS["chain_bf16_32768x4096_256x256_bf16out"], M, N1, N2, K, ab=ab, d=d)
    x, D, info, st, intact = gpucase.run_chain(cw, c_none=not with_c, guard=128)
    assert st == gemm.GEMM_OK and intact
    gpucase.check_chain(cw, x, D, c_none=not with_c)


@pytest.mark.parametrize("M,K,N1,N2,ab,d,with_c", CHAIN_PAIR_CASES,
                         ids=[f"{c[0]}x{c[1]}-{c[2]}x{c[3]}-{c[4]}-{c[5]}-{'C' if c[6] else 'noC'}"
                              for c in CHAIN_PAIR_CASES])
def test_random_chain_pairs(M, K, N1, N2, ab, d, with_c):
    cw = synth.scaled_chain(synth.CHAIN_WORKLOADS["chain_bf16_32768x4096_256x256_bf16out"], M, N1, N2, K, ab=ab, d=d)
    x, D, info, st, intact = gpucase.run_chain(cw, c_none=not with_c, guard=128)
    assert st == gemm.GEMM_OK and intact and info["cta_group"] == 2
    gpucase.check_chain(cw, x, D, c_none=not with_c)
