"""Seeded synthetic inputs for D = A·B + C.

This module is shared by the CUDA path and the CPU oracle: it produces the
operand *bit patterns* (bf16 / fp16 / e4m3 / e2m1 codes, UE8M0 and UE4M3
scale codes, fp32 C) and nothing else.  It contains none of the multiply-accumulate arithmetic.

Random numbers
    A counter-based splitmix64 stream (Steele, Lea & Flood, "Fast splittable
    pseudorandom number generators", OOPSLA 2014; the finaliser constants are
    Vigna's published splitmix64).  Output i of stream (seed, tensor) is
    ``mix64(base + (i + 1) * GAMMA)`` with ``base = mix64(seed << 32 | tensor)``.

Distributions
    uniform[-1, 1): the top 24 bits of an output, ``u * 2**-23 - 1`` (exact
    in fp32).
    N(0, sigma): Box & Muller (1958), two stream outputs per sample, evaluated
    in fp64 and rounded to fp32 (sigma is the standard deviation).
    UE8M0 scale 2**e with e uniform over {-4, ..., 4}: code = e + 127.
    UE4M3 scale (1 + m/8) * 2**e with e uniform over {-4, ..., 4} and m over
    {0, ..., 7}: code = (e + 7) << 3 | m (two stream outputs per code).

Rounding of operands (round to nearest, ties to even, from an fp32 sample)
    bf16 : the upper half of the binary32 pattern after RNE on bit 16.
    fp16 : IEEE binary16 (numpy's correctly rounded conversion).
    e4m3 : OCP 8-bit floating point (E4M3: bias 7, no infinities, max 448,
           S.1111.111 is NaN), saturating to +-448.
    e2m1 : OCP 4-bit floating point (E2M1: bias 1, values 0, 0.5, 1, 1.5, 2,
           3, 4, 6 and their negatives), saturating to +-6; stored two per
           byte, element 2t in the low nibble of byte t of the storage order.
"""

from __future__ import annotations

import dataclasses
import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream ids of the tensors of one problem
T_A, T_B, T_C, T_SFA, T_SFB = 0, 1, 2, 3, 4

_CHUNK = 1 << 22


def mix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _base(seed: int, tensor: int) -> np.uint64:
    key = np.array([((seed & 0xFFFFFFFF) << 32) | (tensor & 0xFFFFFFFF)], dtype=np.uint64)
    return mix64(key)[0]


def stream(seed: int, tensor: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the (seed, tensor) stream."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return mix64(_base(seed, tensor) + i * GAMMA)


def uniform_pm1(seed: int, tensor: int, n: int) -> np.ndarray:
    """n fp32 samples of uniform[-1, 1) on a 2**-23 grid."""
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        x = stream(seed, tensor, s, c) >> np.uint64(40)
        out[s:s + c] = (x.astype(np.float64) * 2.0 ** -23 - 1.0).astype(np.float32)
    return out


def normal(seed: int, tensor: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """n fp32 samples of N(0, sigma**2) by Box-Muller (outputs 2i and 2i+1)."""
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        x = stream(seed, tensor, 2 * s, 2 * c)
        u1 = ((x[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (x[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        out[s:s + c] = (sigma * z).astype(np.float32)
    return out


def ue8m0_codes(seed: int, tensor: int, n: int, lo: int = -4, hi: int = 4) -> np.ndarray:
    """n UE8M0 codes (biased exponents) of 2**e, e uniform over {lo..hi}."""
    span = np.uint64(hi - lo + 1)
    out = np.empty(n, dtype=np.uint8)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        x = stream(seed, tensor, s, c) >> np.uint64(32)
        e = ((x * span) >> np.uint64(32)).astype(np.int64) + lo
        out[s:s + c] = (e + 127).astype(np.uint8)
    return out


def ue4m3_codes(seed: int, tensor: int, n: int, lo: int = -4, hi: int = 4) -> np.ndarray:
    """n UE4M3 codes of (1 + m/8) * 2**e, e uniform over {lo..hi}, m over {0..7}."""
    span = np.uint64(hi - lo + 1)
    out = np.empty(n, dtype=np.uint8)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        x = stream(seed, tensor, 2 * s, 2 * c) >> np.uint64(32)
        e = ((x[0::2] * span) >> np.uint64(32)).astype(np.int64) + lo
        m = ((x[1::2] * np.uint64(8)) >> np.uint64(32)).astype(np.int64)
        out[s:s + c] = ((e + 7) << 3 | m).astype(np.uint8)
    return out


# ---------------------------------------------------------------- rounding

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """RNE fp32 -> bf16 codes (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """RNE fp32 -> IEEE binary16 codes."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """RNE fp32 -> OCP E4M3 codes, saturating finite values to +-448."""
    x = np.ascontiguousarray(x, dtype=np.float32).astype(np.float64)
    sign = (np.signbit(x)).astype(np.uint8) << np.uint8(7)
    a = np.abs(x)
    _, e2 = np.frexp(np.where(a > 0, a, 1.0))        # a = m * 2**e2, m in [0.5, 1)
    ex = np.maximum(e2 - 1, -6)                        # unbiased exponent, subnormals share -6
    q = np.ldexp(1.0, ex - 3)                          # spacing of the 3-bit mantissa grid
    r = np.rint(a / q) * q                             # ties to even (a/q is exact)
    r = np.minimum(r, 448.0)                           # satfinite
    _, er = np.frexp(np.where(r > 0, r, 1.0))
    er = er - 1
    normal_ = r >= 2.0 ** -6
    e_field = np.where(normal_, er + 7, 0)
    m_field = np.where(normal_, r / np.ldexp(1.0, er - 3) - 8.0, r / 2.0 ** -9)
    code = (e_field.astype(np.int64) << 3) | m_field.astype(np.int64)
    code = np.where(r == 0, 0, code)
    return (code.astype(np.uint8) | sign).astype(np.uint8)


E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def f32_to_e2m1_bits(x: np.ndarray) -> np.ndarray:
    """RNE fp32 -> OCP E2M1 codes (one per uint8, low 4 bits), saturating to +-6."""
    x = np.ascontiguousarray(x, dtype=np.float32).astype(np.float64)
    sign = (np.signbit(x)).astype(np.uint8) << np.uint8(3)
    a = np.abs(x)
    _, e2 = np.frexp(np.where(a > 0, a, 1.0))          # a = m * 2**e2, m in [0.5, 1)
    ex = np.maximum(e2 - 1, 0)                          # unbiased exponent, the subnormal shares 0
    q = np.ldexp(1.0, ex - 1)                           # spacing of the 1-bit mantissa grid
    r = np.minimum(np.rint(a / q) * q, 6.0)             # ties to even, then satfinite
    code = np.searchsorted(E2M1_MAGNITUDES, r)          # r is one of the magnitudes
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """Pack E2M1 codes two per byte along the last axis (even element in the low nibble)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    if c.shape[-1] % 2:
        raise ValueError("the packed axis needs an even length")
    return (c[..., 0::2] & np.uint8(0xF)) | ((c[..., 1::2] & np.uint8(0xF)) << np.uint8(4))


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """Inverse of pack_e2m1: one code per uint8."""
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & np.uint8(0xF)
    out[..., 1::2] = p >> np.uint8(4)
    return out


# ---------------------------------------------------------------- workloads

# scale modes (the C ABI's block_scaled argument)
SCALE_NONE, SCALE_UE8M0_32, SCALE_UE4M3_16 = 0, 1, 2

@dataclasses.dataclass(frozen=True)
class Workload:
    """One GEMM problem D = A·B + C and the recipe of its inputs.

    A is M x K, row-major when ``a_row_major`` (else column-major); B is K x N,
    column-major unless ``b_row_major`` (column-major K x N = N rows of K).
    ``ab`` is "bf16", "f16", "e4m3" or "e2m1"; ``dist`` "uniform" or "normal"
    with ``sigma``; ``c`` "zero" or "normal"; ``d`` "f32" or "bf16".
    ``block_scaled`` is a scale mode: 0 none, 1 (or True) UE8M0 per 32 K
    elements, 2 UE4M3 per 16.
    """
    name: str
    M: int
    N: int
    K: int
    ab: str
    dist: str
    sigma: float
    c: str
    d: str
    seed: int
    block_scaled: int = SCALE_NONE
    a_row_major: bool = True
    b_row_major: bool = False

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def sf_block(self) -> int:
        return 16 if int(self.block_scaled) == SCALE_UE4M3_16 else 32

    @property
    def sfk(self) -> int:
        return -(-self.K // self.sf_block)


WORKLOADS = {
    w.name: w for w in [
        Workload("bf16_256x256x256_c0_f32out", 256, 256, 256, "bf16", "uniform", 1.0, "zero", "f32", 0),
        Workload("bf16_4096x4096x4096_f32out", 4096, 4096, 4096, "bf16", "uniform", 1.0, "normal", "f32", 1),
        Workload("f16_4000x3000x2056_f32out", 4000, 3000, 2056, "f16", "normal", 0.5, "normal", "f32", 2),
        Workload("bf16_8192x8192x8192_bf16out", 8192, 8192, 8192, "bf16", "uniform", 1.0, "normal", "bf16", 3),
        Workload("mxf8e4m3_8192x8192x8192_c0_f32out", 8192, 8192, 8192, "e4m3", "normal", 1.0, "zero", "f32", 4,
                 block_scaled=SCALE_UE8M0_32),
        # 4-bit operands with two (UE8M0 per 32) or four (UE4M3 per 16) scales per 64-element MMA step
        Workload("mxf4e2m1_8192x8192x8192_c0_f32out", 8192, 8192, 8192, "e2m1", "normal", 1.0, "zero", "f32", 5,
                 block_scaled=SCALE_UE8M0_32),
        Workload("nvf4e2m1_8192x8192x8192_c0_f32out", 8192, 8192, 8192, "e2m1", "normal", 1.0, "zero", "f32", 6,
                 block_scaled=SCALE_UE4M3_16),
    ]
}

HEADLINE = "bf16_8192x8192x8192_bf16out"


@dataclasses.dataclass(frozen=True)
class ChainWorkload:
    """Two chained products D = C + round(A·B)·E and the recipe of their inputs.

    A is M x K row-major, B is K x N1 column-major (N1 rows of K), E is N1 x N2
    column-major (N2 rows of N1), C is M x N2 fp32, D is M x N2; ``ab`` ("bf16"
    or "f16") is the type of A, B, E and of the rounded intermediate.
    """
    name: str
    M: int
    N1: int
    N2: int
    K: int
    ab: str
    dist: str
    sigma: float
    c: str
    d: str
    seed: int

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N1 * (self.K + self.N2)


T_E = 5   # stream id of E

CHAIN_WORKLOADS = {
    w.name: w for w in [
        ChainWorkload("chain_bf16_32768x4096_256x256_bf16out", 32768, 256, 256, 4096, "bf16", "uniform", 1.0,
                      "normal", "bf16", 7),
    ]
}


def scaled_chain(w: ChainWorkload, M: int, N1: int, N2: int, K: int, **kw) -> ChainWorkload:
    return dataclasses.replace(w, name=f"{w.name}@{M}x{K}_{N1}x{N2}", M=M, N1=N1, N2=N2, K=K, **kw)


def make_chain_inputs(w: ChainWorkload) -> dict:
    """Bit patterns of A (M, K), B (N1, K), E (N2, N1) and fp32 C (M, N2)."""
    A = _operand(w, T_A, w.M * w.K).reshape(w.M, w.K)
    B = _operand(w, T_B, w.K * w.N1).reshape(w.N1, w.K)
    E = _operand(w, T_E, w.N1 * w.N2).reshape(w.N2, w.N1)
    if w.c == "zero":
        C = np.zeros((w.M, w.N2), dtype=np.float32)
    else:
        C = normal(w.seed, T_C, w.M * w.N2, 1.0).reshape(w.M, w.N2)
    return {"A": A, "B": B, "E": E, "C": C}


def scaled(w: Workload, M: int, N: int, K: int, name: str | None = None, **kw) -> Workload:
    """The same recipe at other sizes (parity cases the oracle finishes quickly)."""
    return dataclasses.replace(w, name=name or f"{w.name}@{M}x{N}x{K}", M=M, N=N, K=K, **kw)


def _operand(w: Workload, tensor: int, n: int) -> np.ndarray:
    if w.dist == "uniform":
        x = uniform_pm1(w.seed, tensor, n)
    else:
        x = normal(w.seed, tensor, n, w.sigma)
    if w.ab == "bf16":
        return f32_to_bf16_bits(x)
    if w.ab == "f16":
        return f32_to_f16_bits(x)
    if w.ab == "e4m3":
        return f32_to_e4m3_bits(np.clip(x, -448.0, 448.0))
    if w.ab == "e2m1":
        return f32_to_e2m1_bits(x)
    raise ValueError(w.ab)


def make_inputs(w: Workload) -> dict:
    """Bit patterns of A, B, C (and SFA, SFB) for workload w.

    Shapes follow the memory layout: A is (M, K) when row-major, else (K, M);
    B is (N, K) when column-major, else (K, N); C is (M, N) fp32 row-major;
    SFA is (M, sfk) and SFB is (N, sfk), sfk = ceil(K / block), both row-major
    u8.  e2m1 operands are packed two per byte along the contiguous axis, which
    halves its length (K must then be even for a K-major operand, M or N for an
    M- or N-major one).
    """
    M, N, K = w.M, w.N, w.K

    def operand(tensor, shape):
        x = _operand(w, tensor, shape[0] * shape[1]).reshape(shape)
        return pack_e2m1(x) if w.ab == "e2m1" else x

    A = operand(T_A, (M, K) if w.a_row_major else (K, M))
    B = operand(T_B, (K, N) if w.b_row_major else (N, K))
    if w.c == "zero":
        C = np.zeros((M, N), dtype=np.float32)
    else:
        C = normal(w.seed, T_C, M * N, 1.0).reshape(M, N)
    out = {"A": A, "B": B, "C": C}
    mode = int(w.block_scaled)
    if mode:
        codes = ue4m3_codes if mode == SCALE_UE4M3_16 else ue8m0_codes
        out["SFA"] = codes(w.seed, T_SFA, M * w.sfk).reshape(M, w.sfk)
        out["SFB"] = codes(w.seed, T_SFB, N * w.sfk).reshape(N, w.sfk)
    return out
