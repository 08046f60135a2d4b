"""Shared helpers of the GPU parity tests: run one workload through the C ABI
and compare it with the oracle under the accept rule

    |D_gpu - D_ref| <= 1e-5 * sum_k |a b| + 1e-6 * |c|   (+ 1 bf16 ulp of D_ref for bf16 D)

The operands are the seeded synthetic inputs both sides share; the reference
values come from the oracle only."""
from __future__ import annotations

import numpy as np

import oracle
from blackwell_tensor_core_tma_gb300 import gemm, synth

REL_S = 1e-5
REL_C = 1e-6


def to_device(x: np.ndarray):
    import torch
    if x.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16))
    else:
        t = torch.from_numpy(np.ascontiguousarray(x))
    return t.cuda()


def decode_d(t, d: str) -> np.ndarray:
    """fp64 values of a device D (fp32, or bf16 codes widened exactly)."""
    import torch
    if d == "bf16":
        bits = t.view(torch.int16).cpu().numpy().view(np.uint16)
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def run(w: synth.Workload, flags: int = 0, c_none: bool = False, guard: int = 0, inputs=None, reps: int = 1):
    """Run w through gemm_run; returns (inputs, D as fp64, plan info, status, guard intact)."""
    import torch
    x = inputs if inputs is not None else synth.make_inputs(w)
    A, B = to_device(x["A"]), to_device(x["B"])
    C = None if c_none else to_device(x["C"])
    SFA = to_device(x["SFA"]) if w.block_scaled else None
    SFB = to_device(x["SFB"]) if w.block_scaled else None
    tdt = torch.bfloat16 if w.d == "bf16" else torch.float32
    n = w.M * w.N
    g = guard
    buf = torch.full((n + 2 * g,), float("nan"), dtype=tdt, device="cuda")
    D = buf[g:g + n].view(w.M, w.N)
    with gemm.Plan(w.M, w.N, w.K, w.ab, w.d, w.block_scaled, flags, a_row_major=w.a_row_major,
                   b_row_major=w.b_row_major) as plan:
        for _ in range(reps):
            plan.run(A, B, C, D, SFA, SFB, torch.cuda.current_stream())
        torch.cuda.synchronize()
        status = plan.last_status()
        info = plan.info
    intact = True
    if g:
        intact = bool(torch.isnan(buf[:g]).all().item()) and bool(torch.isnan(buf[g + n:]).all().item())
    return x, decode_d(D, w.d), info, status, intact


def tolerance(w, D_ref, S, c):
    tol = REL_S * S + REL_C * np.abs(c)
    if w.d == "bf16":
        tol = tol + oracle.bf16_ulp(D_ref)
    return tol


def check_full(w, x, D, c_none=False):
    C = None if c_none else x["C"]
    D_ref, S = oracle.gemm(x["A"], x["B"], C, w.M, w.N, w.K, w.ab, a_row_major=w.a_row_major,
                           b_row_major=w.b_row_major, SFA=x.get("SFA"), SFB=x.get("SFB"),
                           block_scaled=w.block_scaled)
    c = np.zeros_like(D_ref) if c_none else x["C"].astype(np.float64)
    _assert_within(w, D, D_ref, S, c, "full")


def _input_key(w, x, extra=()) -> str:
    """Checksum of everything a full oracle product depends on: the input bytes, the problem's
    shape, types and layouts, and the oracle's own C source."""
    import hashlib
    import os
    h = hashlib.sha256()
    for k in sorted(x):
        if x[k] is not None:
            h.update(k.encode())
            h.update(np.ascontiguousarray(x[k]).tobytes())
    h.update(repr((type(w).__name__, sorted(vars(w).items()), extra)).encode())
    with open(os.path.join(os.path.dirname(oracle.__file__), "gemm_oracle.c"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:32]


def cached(key: str, compute):
    """compute() (a tuple of arrays), kept on disk under $GB300GEMM_ORACLE_CACHE/<key>.npz when
    that variable names a directory; without it nothing is written."""
    import os
    d = os.environ.get("GB300GEMM_ORACLE_CACHE")
    path = os.path.join(d, key + ".npz") if d else None
    if path and os.path.exists(path):
        with np.load(path) as z:
            return tuple(z[f"a{i}"] for i in range(len(z.files)))
    out = compute()
    if path:
        os.makedirs(d, exist_ok=True)
        tmp = path + ".tmp.npz"
        np.savez(tmp, **{f"a{i}": a for i, a in enumerate(out)})
        os.replace(tmp, path)
    return out


def full_ratio(w, x, D) -> float:
    """Every element of D against the oracle's full product (fp64; cached by input checksum):
    asserts the accept rule and returns the largest error / tolerance ratio."""
    D_ref, S = cached(_input_key(w, x), lambda: oracle.gemm(
        x["A"], x["B"], x["C"], w.M, w.N, w.K, w.ab, a_row_major=w.a_row_major, b_row_major=w.b_row_major,
        SFA=x.get("SFA"), SFB=x.get("SFB"), block_scaled=w.block_scaled))
    c = x["C"].astype(np.float64)
    _assert_within(w, D, D_ref, S, c, "every element")
    tol = tolerance(w, D_ref, S, c)
    return float(np.max(np.abs(D - D_ref) / np.maximum(tol, 1e-300)))


def sample_entries(M: int, N: int, tile_m: int, tile_n: int, n_random: int = 4096, seed: int = 0):
    """Tile corners and edges, one full row and column, and random entries."""
    rng = np.random.default_rng(seed)
    rows, cols = [], []
    rm = sorted({r for t in range(0, M, tile_m) for r in (t, t + 31, t + 32, t + tile_m // 2, t + tile_m - 1)
                 if r < M} | {M - 1})
    cn = sorted({c for t in range(0, N, tile_n) for c in (t, t + 31, t + 32, t + tile_n // 2, t + tile_n - 1)
                 if c < N} | {N - 1})
    for r in rm[:: max(1, len(rm) // 64)]:
        for c in cn[:: max(1, len(cn) // 64)]:
            rows.append(r)
            cols.append(c)
    r0 = int(rng.integers(0, M))
    c0 = int(rng.integers(0, N))
    rows += [r0] * N + list(range(M))
    cols += list(range(N)) + [c0] * M
    rows += list(rng.integers(0, M, n_random))
    cols += list(rng.integers(0, N, n_random))
    return np.array(rows, np.int64), np.array(cols, np.int64)


def check_entries(w, x, D, rows, cols):
    D_ref, S = oracle.gemm_entries(x["A"], x["B"], x["C"], w.M, w.N, w.K, w.ab, rows, cols,
                                   a_row_major=w.a_row_major, b_row_major=w.b_row_major,
                                   SFA=x.get("SFA"), SFB=x.get("SFB"), block_scaled=w.block_scaled)
    c = x["C"][rows, cols].astype(np.float64)
    _assert_within(w, D[rows, cols], D_ref, S, c, f"{rows.size} sampled entries")


def _assert_within(w, D, D_ref, S, c, what):
    tol = tolerance(w, D_ref, S, c)
    err = np.abs(D - D_ref)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.flatnonzero(bad.ravel())
        k = idx[np.argmax((err.ravel()[idx]) / np.maximum(tol.ravel()[idx], 1e-300))] if idx.size else 0
        raise AssertionError(
            f"{w.name} ({what}): {idx.size} of {err.size} entries outside tolerance; worst flat index {k}: "
            f"gpu {D.ravel()[k]!r} ref {D_ref.ravel()[k]!r} tol {tol.ravel()[k]!r}")


# ------------------------------------------------------------ two-product chain

def run_chain(w, flags: int = 0, c_none: bool = False, guard: int = 0, inputs=None, reps: int = 1,
              stream_k=None):
    """Run a ChainWorkload through gemm_chain_run; returns (inputs, D as fp64, plan info, status, guard intact).
    stream_k: None keeps the plan's choice, 0 or 1 is passed to gemm_plan_set_stream_k."""
    import torch
    x = inputs if inputs is not None else synth.make_chain_inputs(w)
    A, B, E = to_device(x["A"]), to_device(x["B"]), to_device(x["E"])
    C = None if c_none else to_device(x["C"])
    tdt = torch.bfloat16 if w.d == "bf16" else torch.float32
    n = w.M * w.N2
    g = guard
    buf = torch.full((n + 2 * g,), float("nan"), dtype=tdt, device="cuda")
    D = buf[g:g + n].view(w.M, w.N2)
    with gemm.ChainPlan(w.M, w.N1, w.N2, w.K, w.ab, w.d, flags) as plan:
        if stream_k is not None:
            plan.set_stream_k(stream_k)
        for _ in range(reps):
            plan.run(A, B, E, C, D, torch.cuda.current_stream())
        torch.cuda.synchronize()
        status = plan.last_status()
        info = plan.info
    intact = True
    if g:
        intact = bool(torch.isnan(buf[:g]).all().item()) and bool(torch.isnan(buf[g + n:]).all().item())
    return x, decode_d(D, w.d), info, status, intact


def format_ulp(x, dtype: str) -> np.ndarray:
    """Spacing of the bf16 / fp16 grid at |x| (subnormal spacing below the smallest normal)."""
    p, emin = (8, -126) if dtype == "bf16" else (11, -14)
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(a)
    ex = np.where(a > 0, np.maximum(e - 1, emin), emin)
    return np.ldexp(1.0, ex - (p - 1))


def check_chain(w, x, D, rows=None, c_none=False):
    """D against the oracle's chain on the listed rows (all by default).

    The intermediate is rounded from the exact sum by the oracle and from an fp32 sum by
    the GPU, so an element of P may differ by one unit of the format at |T| plus the
    first product's accumulation error; the bound carries that through E:
        |dD| <= REL_S * S2 + REL_C * |c| + sum_j (ulp(|T| + REL_S * S1) + REL_S * S1)_ij * |e_jn|
    (+ one bf16 ulp of D for bf16 D).
    """
    rows = np.arange(w.M) if rows is None else np.asarray(rows, dtype=np.int64)
    C = None if c_none else x["C"]
    T, S1, D_ref, S2 = oracle.chain(x["A"], x["B"], x["E"], C, w.M, w.N1, w.N2, w.K, w.ab, rows=rows)
    e_abs = np.abs(oracle.decode(x["E"], w.ab)).T                   # (N1, N2)
    slack = (format_ulp(np.abs(T) + REL_S * S1, w.ab) + REL_S * S1) @ e_abs
    c = np.zeros_like(D_ref) if c_none else x["C"][rows].astype(np.float64)
    tol = REL_S * S2 + REL_C * np.abs(c) + slack
    if w.d == "bf16":
        tol = tol + oracle.bf16_ulp(D_ref)
    err = np.abs(D[rows] - D_ref)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{w.name}: {int(bad.sum())} of {bad.size} entries out of tolerance; worst "
                           f"err/tol {float(np.max(err / np.maximum(tol, 1e-300))):.3g}")
    return float(np.max(err / np.maximum(tol, 1e-300)))
