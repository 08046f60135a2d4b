"""CPU oracle for D = A·B + C — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The CUDA library never links, loads or
calls it, and it imports nothing from the CUDA package.

``gemm`` / ``gemm_entries`` wrap the plain fp64 triple loop in
``gemm_oracle.c`` (the definition D[i][j] = C[i][j] + sum_k a[i][k] b[k][j]
from "Tensor Core 数据布局的演进", overview, with the block-scaling rule of its
section "Block-Scaled MMA 的 Scale Factors": one scale per 32 K elements
(UE8M0, e4m3 or e2m1 operands) or per 16 (UE4M3, e2m1 operands)).  ``chain``
is the two-product chain D = C + round(A·B)·E whose intermediate a tensor-core
kernel keeps in tensor memory (same page, section "TMEM 中的累加器": some MMA
forms read A from TMEM).
``layouts`` holds the pages' register-fragment and TMEM layout maps.

Parity pins (tests/test_oracle_*.py): exhaustive format decodes against
torch/numpy conversions and the OCP/IEEE tables; A = I, rank-1, all-ones and
sign-alternating closed forms; brute force in exact integer arithmetic on
small problems in every storage order; block scales against a per-block
exact evaluation; the pages' printed fragment and TMEM examples.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

DTYPES = {"f16": 0, "bf16": 1, "e4m3": 2, "e2m1": 3}

# scale modes: none; UE8M0 per 32 K elements; UE4M3 per 16 K elements
SCALE_NONE, SCALE_UE8M0_32, SCALE_UE4M3_16 = 0, 1, 2
SCALE_BLOCK = {SCALE_UE8M0_32: 32, SCALE_UE4M3_16: 16}

_lib = None


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c with gcc (OpenMP, no fp contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
        L.oracle_gemm.argtypes = [i64, i64, i64, ctypes.c_int, vp, ctypes.c_int, vp, ctypes.c_int,
                                  vp, vp, vp, ctypes.c_int, i64, i64, dp, dp, ctypes.c_int]
        L.oracle_gemm.restype = ctypes.c_int
        L.oracle_gemm_entries.argtypes = [i64, i64, i64, ctypes.c_int, vp, ctypes.c_int, vp, ctypes.c_int,
                                          vp, vp, vp, ctypes.c_int, i64, vp, vp, dp, dp, ctypes.c_int]
        L.oracle_gemm_entries.restype = ctypes.c_int
        for name, arg in [("oracle_decode_bf16", ctypes.c_uint16), ("oracle_decode_f16", ctypes.c_uint16),
                          ("oracle_decode_e4m3", ctypes.c_uint8), ("oracle_decode_ue8m0", ctypes.c_uint8),
                          ("oracle_decode_e2m1", ctypes.c_uint8), ("oracle_decode_ue4m3", ctypes.c_uint8)]:
            f = getattr(L, name)
            f.argtypes = [arg]
            f.restype = ctypes.c_double
        L.oracle_chain.argtypes = [i64, i64, i64, i64, ctypes.c_int, vp, vp, vp, vp, i64, vp, dp, dp, dp, dp,
                                   ctypes.c_int]
        L.oracle_chain.restype = ctypes.c_int
        for name in ("oracle_round_bf16", "oracle_round_f16"):
            f = getattr(L, name)
            f.argtypes = [ctypes.c_double]
            f.restype = ctypes.c_double
        L.oracle_threads.argtypes = [ctypes.c_int]
        L.oracle_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def threads(nthreads: int = 0) -> int:
    return lib().oracle_threads(nthreads)


def decode(codes, dtype: str) -> np.ndarray:
    """fp64 values of bf16 / f16 / e4m3 / ue8m0 / ue4m3 codes, or of e2m1 codes
    given one per element in the low 4 bits (element by element)."""
    f = getattr(lib(), "oracle_decode_" + dtype)
    flat = np.asarray(codes).ravel()
    return np.array([f(int(c)) for c in flat], dtype=np.float64).reshape(np.shape(codes))


def _ptr(a):
    return None if a is None else a.ctypes.data


def _packed_bytes(n: int, dtype: str) -> int:
    """Bytes holding n elements: e2m1 two per byte (element 2t in the low nibble of byte t)."""
    return (n + 1) // 2 if dtype == "e2m1" else n


def _check_operands(A, B, C, SFA, SFB, M, N, K, dtype, block_scaled):
    width = np.uint8 if dtype in ("e4m3", "e2m1") else np.uint16
    A = np.ascontiguousarray(A, dtype=width)
    B = np.ascontiguousarray(B, dtype=width)
    if A.size != _packed_bytes(M * K, dtype) or B.size != _packed_bytes(K * N, dtype):
        raise ValueError("operand sizes do not match M, N, K")
    if C is not None:
        C = np.ascontiguousarray(C, dtype=np.float32)
        if C.size != M * N:
            raise ValueError("C size does not match M, N")
    mode = int(block_scaled)
    if mode:
        sfk = -(-K // SCALE_BLOCK[mode])
        SFA = np.ascontiguousarray(SFA, dtype=np.uint8)
        SFB = np.ascontiguousarray(SFB, dtype=np.uint8)
        if SFA.size != M * sfk or SFB.size != N * sfk:
            raise ValueError("scale-factor sizes do not match M, N, ceil(K/block)")
    else:
        SFA = SFB = None
    return A, B, C, SFA, SFB


def gemm(A, B, C, M: int, N: int, K: int, dtype: str, a_row_major: bool = True,
         b_row_major: bool = False, SFA=None, SFB=None, block_scaled: int = 0,
         rows: tuple | None = None, nthreads: int = 0):
    """(D, S) as fp64 arrays of shape (rows, N): D = C + sum_k a b, S = sum_k |a b|.

    ``block_scaled``: 0 (or False) none, 1 (or True) UE8M0 per 32 K, 2 UE4M3
    per 16 K.  ``rows`` = (row0, row1) restricts the work to a row slab
    (default: all).
    """
    A, B, C, SFA, SFB = _check_operands(A, B, C, SFA, SFB, M, N, K, dtype, block_scaled)
    r0, r1 = rows if rows is not None else (0, M)
    D = np.empty((r1 - r0, N), dtype=np.float64)
    S = np.empty((r1 - r0, N), dtype=np.float64)
    rc = lib().oracle_gemm(M, N, K, DTYPES[dtype], _ptr(A), int(a_row_major), _ptr(B), int(b_row_major),
                           _ptr(C), _ptr(SFA), _ptr(SFB), int(block_scaled), r0, r1,
                           D.ctypes.data, S.ctypes.data, nthreads)
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return D, S


def gemm_entries(A, B, C, M: int, N: int, K: int, dtype: str, rows, cols, a_row_major: bool = True,
                 b_row_major: bool = False, SFA=None, SFB=None, block_scaled: int = 0,
                 nthreads: int = 0):
    """(D, S) at the listed (row, col) entries, each computed on its own."""
    A, B, C, SFA, SFB = _check_operands(A, B, C, SFA, SFB, M, N, K, dtype, block_scaled)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    n = rows.size
    D = np.empty(n, dtype=np.float64)
    S = np.empty(n, dtype=np.float64)
    rc = lib().oracle_gemm_entries(M, N, K, DTYPES[dtype], _ptr(A), int(a_row_major), _ptr(B),
                                   int(b_row_major), _ptr(C), _ptr(SFA), _ptr(SFB), int(block_scaled),
                                   n, rows.ctypes.data, cols.ctypes.data, D.ctypes.data, S.ctypes.data,
                                   nthreads)
    if rc != 0:
        raise ValueError("oracle_gemm_entries rejected its arguments")
    return D, S


def round_to(x, dtype: str) -> np.ndarray:
    """fp64 values rounded to bf16 / f16 (nearest, ties to even; overflow to infinity)."""
    f = getattr(lib(), "oracle_round_" + dtype)
    flat = np.asarray(x, dtype=np.float64).ravel()
    return np.array([f(float(v)) for v in flat], dtype=np.float64).reshape(np.shape(x))


def chain(A, B, E, C, M: int, N1: int, N2: int, K: int, dtype: str, rows=None, nthreads: int = 0):
    """Two chained products: T = A·B, P = round(T) to ``dtype``, D = C + P·E.

    A is (M, K) row-major, B (N1, K) (column-major K x N1), E (N2, N1) (column-major
    N1 x N2), C (M, N2) fp32 or None.  Returns (T, S1, D, S2) for the listed rows
    (default: all): T, S1 = sum_k |a b| of shape (rows, N1); D, S2 = sum_j |P e| of
    shape (rows, N2).
    """
    width = np.uint16
    A = np.ascontiguousarray(A, dtype=width)
    B = np.ascontiguousarray(B, dtype=width)
    E = np.ascontiguousarray(E, dtype=width)
    if A.size != M * K or B.size != K * N1 or E.size != N1 * N2:
        raise ValueError("operand sizes do not match M, N1, N2, K")
    if C is not None:
        C = np.ascontiguousarray(C, dtype=np.float32)
        if C.size != M * N2:
            raise ValueError("C size does not match M, N2")
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.size
    T = np.empty((n, N1)); S1 = np.empty((n, N1)); D = np.empty((n, N2)); S2 = np.empty((n, N2))
    rc = lib().oracle_chain(M, N1, N2, K, DTYPES[dtype], _ptr(A), _ptr(B), _ptr(E), _ptr(C), n,
                            rows.ctypes.data, T.ctypes.data, S1.ctypes.data, D.ctypes.data, S2.ctypes.data,
                            nthreads)
    if rc != 0:
        raise ValueError("oracle_chain rejected its arguments")
    return T, S1, D, S2


def bf16_ulp(x) -> np.ndarray:
    """Spacing of the bf16 grid (8 significant bits) at |x|: 2**(floor(log2|x|) - 7).

    Below the smallest normal (2**-126) the spacing is the subnormal one, 2**-133.
    """
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(a)                              # a = m * 2**e, m in [0.5, 1); e = 0 at 0
    ex = np.where(a > 0, np.maximum(e - 1, -126), -126)
    return np.ldexp(1.0, ex - 7)
