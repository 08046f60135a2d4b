"""ctypes binding of libgb300gemm.so (include/gb300gemm.h), same entry-point names.

Argument marshalling only: every step of D = A·B + C runs in the CUDA
library.  Pointers may be passed as ints or as torch tensors (their
``data_ptr()``); streams as ints or torch streams (their ``cuda_stream``).
There is no fallback: if the library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os

from . import build as _build

GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_UNSUPPORTED, GEMM_ERR_ALIGNMENT, GEMM_ERR_CUDA, GEMM_ERR_TIMEOUT, \
    GEMM_ERR_CHECK = range(7)
GEMM_F16, GEMM_BF16, GEMM_E4M3, GEMM_F32, GEMM_E2M1 = range(5)
GEMM_SCALE_NONE, GEMM_SCALE_UE8M0_32, GEMM_SCALE_UE4M3_16 = range(3)
GEMM_FLAG_SYNC, GEMM_FLAG_FORCE_1CTA, GEMM_FLAG_FORCE_2CTA, GEMM_FLAG_DETERMINISTIC = 0x1, 0x2, 0x4, 0x8

DTYPE = {"f16": GEMM_F16, "bf16": GEMM_BF16, "e4m3": GEMM_E4M3, "f32": GEMM_F32, "e2m1": GEMM_E2M1}

# every symbol include/gb300gemm.h and include/gb300gemm_testing.h declare
EXPORTS = ["gemm_plan_create", "gemm_run", "gemm_run_host", "gemm_plan_last_status", "gemm_plan_get_info",
           "gemm_plan_set_timeout", "gemm_plan_destroy", "gemm_status_string", "gemm_testing_set_fault",
           "gemm_run_noalloc", "gemm_plan_set_split_k", "gemm_chain_plan_create", "gemm_chain_run",
           "gemm_chain_run_host", "gemm_plan_set_stream_k", "gemm_measure_tensor_rate",
           "gemm_testing_pair_tile_n", "gemm_plan_set_clock_meter", "gemm_plan_read_clock_meter",
           "gemm_testing_trace_slots", "gemm_testing_set_trace", "gemm_testing_tmem_ld_probe",
           "gemm_testing_staging_probe", "gemm_testing_schedule", "gemm_testing_e4m3_pair_tile_n"]

# the per-role trace counters of one CTA, in slot order (a GB300_TRACE=1 library:
# gemm_testing_set_trace); SM clock cycles unless the name says otherwise
TRACE_FIELDS = ["kernel_clk", "kernel_ns", "prod_wait", "prod_issue", "prod_stages", "mma_wait_acc",
                "mma_wait_ab", "mma_wait_sf", "mma_issue", "mma_kblocks", "mma_pieces", "mma_first", "mma_end",
                "cp_wait", "cp_issue", "epi_wait_acc", "epi_tmem_ld", "epi_wait_c", "epi_store", "epi_pieces",
                "epi_end"]


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gemm_status_string(status)} (status {status})")


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("cta_group", "tile_m", "tile_n", "tile_k", "stages", "grid", "tiles",
                                            "smem_bytes", "launches_per_run", "sm_count", "splits",
                                            "stream_k")]


class TensorRate(ctypes.Structure):
    _fields_ = [("flop_per_clk_per_sm", ctypes.c_double), ("sm_mhz", ctypes.c_double), ("tflops", ctypes.c_double),
                ("ms", ctypes.c_double), ("sms", ctypes.c_int)]


_lib = None


def library_variant() -> str:
    """The build variant this process loads: GB300GEMM_VARIANT ("" = the default library)."""
    return os.environ.get("GB300GEMM_VARIANT", "")


def library_path() -> str:
    return _build.lib_path(library_variant())


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first (python -m "
                               "blackwell_tensor_core_tma_gb300.build); there is no CPU path")
        L = ctypes.CDLL(path)
        vp, i64, st = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.gemm_plan_create.argtypes = [ctypes.POINTER(vp), i64, i64, i64, st, st, st, st, st, st, ctypes.c_uint]
        L.gemm_plan_create.restype = st
        for name in ("gemm_run", "gemm_run_host"):
            f = getattr(L, name)
            f.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
            f.restype = st
        L.gemm_plan_last_status.argtypes = [vp]
        L.gemm_plan_last_status.restype = st
        L.gemm_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
        L.gemm_plan_get_info.restype = st
        L.gemm_plan_set_timeout.argtypes = [vp, ctypes.c_uint64]
        L.gemm_plan_set_timeout.restype = st
        L.gemm_plan_destroy.argtypes = [vp]
        L.gemm_plan_destroy.restype = st
        L.gemm_status_string.argtypes = [st]
        L.gemm_status_string.restype = ctypes.c_char_p
        L.gemm_testing_set_fault.argtypes = [vp, st]
        L.gemm_testing_set_fault.restype = st
        L.gemm_plan_set_split_k.argtypes = [vp, st]
        L.gemm_plan_set_split_k.restype = st
        L.gemm_plan_set_stream_k.argtypes = [vp, st]
        L.gemm_plan_set_stream_k.restype = st
        L.gemm_run_noalloc.argtypes = [i64, i64, i64, st, st, vp, vp, vp, vp, vp, st]
        L.gemm_run_noalloc.restype = st
        L.gemm_testing_pair_tile_n.argtypes = [i64, i64, i64, st, st, ctypes.POINTER(ctypes.c_int)]
        L.gemm_testing_pair_tile_n.restype = st
        L.gemm_testing_e4m3_pair_tile_n.argtypes = [i64, i64, i64, st, st, ctypes.POINTER(ctypes.c_int)]
        L.gemm_testing_e4m3_pair_tile_n.restype = st
        ip = ctypes.POINTER(ctypes.c_int)
        L.gemm_testing_schedule.argtypes = [st] * 10 + [ip, st, ip]
        L.gemm_testing_schedule.restype = st
        L.gemm_measure_tensor_rate.argtypes = [st, st, st, i64, ctypes.POINTER(TensorRate)]
        L.gemm_measure_tensor_rate.restype = st
        L.gemm_plan_set_clock_meter.argtypes = [vp, st]
        L.gemm_plan_set_clock_meter.restype = st
        L.gemm_plan_read_clock_meter.argtypes = [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
        L.gemm_plan_read_clock_meter.restype = st
        L.gemm_testing_trace_slots.argtypes = []
        L.gemm_testing_trace_slots.restype = st
        L.gemm_testing_set_trace.argtypes = [vp, vp, i64]
        L.gemm_testing_set_trace.restype = st
        L.gemm_testing_tmem_ld_probe.argtypes = [vp, i64]
        L.gemm_testing_tmem_ld_probe.restype = st
        L.gemm_testing_staging_probe.argtypes = [st, st, i64, ctypes.POINTER(ctypes.c_double)]
        L.gemm_testing_staging_probe.restype = st
        L.gemm_chain_plan_create.argtypes = [ctypes.POINTER(vp), i64, i64, i64, i64, st, st, ctypes.c_uint]
        L.gemm_chain_plan_create.restype = st
        for name in ("gemm_chain_run", "gemm_chain_run_host"):
            f = getattr(L, name)
            f.argtypes = [vp, vp, vp, vp, vp, vp, vp]
            f.restype = st
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):                       # numpy array (host buffers)
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str):
    if status != GEMM_OK:
        raise GemmError(status, where)


def gemm_status_string(status: int) -> str:
    return lib().gemm_status_string(status).decode()


def gemm_plan_create(M: int, N: int, K: int, ab="bf16", c="f32", d="f32", a_row_major: int = 1,
                     b_row_major: int = 0, block_scaled: int = 0, flags: int = 0) -> int:
    out = ctypes.c_void_p()
    st = lib().gemm_plan_create(ctypes.byref(out), M, N, K, DTYPE.get(ab, ab), DTYPE.get(c, c), DTYPE.get(d, d),
                                int(a_row_major), int(b_row_major), int(block_scaled), flags)
    _check(st, "gemm_plan_create")
    return out.value


def gemm_run(plan: int, A, B, C, D, SFA=None, SFB=None, stream=None) -> int:
    st = lib().gemm_run(plan, _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(SFA), _ptr(SFB), _stream(stream))
    _check(st, "gemm_run")
    return st


def gemm_run_host(plan: int, A, B, C, D, SFA=None, SFB=None, stream=None) -> int:
    st = lib().gemm_run_host(plan, _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(SFA), _ptr(SFB), _stream(stream))
    _check(st, "gemm_run_host")
    return st


def gemm_chain_plan_create(M: int, N1: int, N2: int, K: int, ab="bf16", d="f32", flags: int = 0) -> int:
    out = ctypes.c_void_p()
    st = lib().gemm_chain_plan_create(ctypes.byref(out), M, N1, N2, K, DTYPE.get(ab, ab), DTYPE.get(d, d), flags)
    _check(st, "gemm_chain_plan_create")
    return out.value


def gemm_chain_run(plan: int, A, B, E, C, D, stream=None) -> int:
    st = lib().gemm_chain_run(plan, _ptr(A), _ptr(B), _ptr(E), _ptr(C), _ptr(D), _stream(stream))
    _check(st, "gemm_chain_run")
    return st


def gemm_chain_run_host(plan: int, A, B, E, C, D, stream=None) -> int:
    st = lib().gemm_chain_run_host(plan, _ptr(A), _ptr(B), _ptr(E), _ptr(C), _ptr(D), _stream(stream))
    _check(st, "gemm_chain_run_host")
    return st


def gemm_plan_last_status(plan: int) -> int:
    return lib().gemm_plan_last_status(plan)


def gemm_plan_get_info(plan: int) -> dict:
    info = PlanInfo()
    _check(lib().gemm_plan_get_info(plan, ctypes.byref(info)), "gemm_plan_get_info")
    return {n: getattr(info, n) for n, _ in PlanInfo._fields_}


def gemm_plan_set_timeout(plan: int, ns: int):
    _check(lib().gemm_plan_set_timeout(plan, ns), "gemm_plan_set_timeout")


def gemm_plan_set_split_k(plan: int, splits: int):
    _check(lib().gemm_plan_set_split_k(plan, splits), "gemm_plan_set_split_k")


def gemm_plan_set_stream_k(plan: int, enable: int):
    _check(lib().gemm_plan_set_stream_k(plan, int(enable)), "gemm_plan_set_stream_k")


def gemm_plan_set_clock_meter(plan: int, enable: int):
    _check(lib().gemm_plan_set_clock_meter(plan, int(enable)), "gemm_plan_set_clock_meter")


def gemm_plan_read_clock_meter(plan: int) -> dict:
    """Mean SM clock (MHz) over the CTA lifetimes counted since the meter was last read."""
    mhz, sec = ctypes.c_double(), ctypes.c_double()
    _check(lib().gemm_plan_read_clock_meter(plan, ctypes.byref(mhz), ctypes.byref(sec)), "gemm_plan_read_clock_meter")
    return {"sm_mhz": mhz.value, "cta_seconds": sec.value}


def gemm_testing_trace_slots() -> int:
    return lib().gemm_testing_trace_slots()


def gemm_testing_set_trace(plan: int, buf, nbytes: int):
    _check(lib().gemm_testing_set_trace(plan, _ptr(buf), int(nbytes)), "gemm_testing_set_trace")


def gemm_testing_tmem_ld_probe():
    """Registers of the TMEM probe's five loads: uint32 array [warp 4][thread 32][62]."""
    import numpy as np
    out = np.zeros(128 * 62, dtype=np.uint32)
    _check(lib().gemm_testing_tmem_ld_probe(out.ctypes.data, out.size), "gemm_testing_tmem_ld_probe")
    return out.reshape(4, 32, 62)


def gemm_testing_staging_probe(pattern: int, load: bool, iters: int = 4096) -> float:
    """SM clocks per warp-wide 128-bit shared-memory access of an epilogue staging pattern."""
    out = ctypes.c_double()
    _check(lib().gemm_testing_staging_probe(int(pattern), int(load), int(iters), ctypes.byref(out)),
           "gemm_testing_staging_probe")
    return out.value


def gemm_plan_destroy(plan: int):
    _check(lib().gemm_plan_destroy(plan), "gemm_plan_destroy")


def gemm_testing_set_fault(plan: int, fault: int):
    _check(lib().gemm_testing_set_fault(plan, fault), "gemm_testing_set_fault")


def gemm_run_noalloc(M: int, N: int, K: int, ab, d, A, B, C, D, stream=None, wait: int = 0) -> int:
    """Allocation-free run (no plan): the kernel's status word lives in a static device array."""
    st = lib().gemm_run_noalloc(M, N, K, DTYPE.get(ab, ab), DTYPE.get(d, d), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                _stream(stream), int(wait))
    _check(st, "gemm_run_noalloc")
    return st


def gemm_measure_tensor_rate(ab, block_scaled: int = GEMM_SCALE_NONE, cta_group: int = 2,
                             iters: int = 4096) -> dict:
    """The tensor-pipe rate probe: FLOP per SM clock of the GEMM's MMA shape, the SM clock
    during the probe, and the whole-GPU TFLOP/s it reached (blocks until done)."""
    out = TensorRate()
    _check(lib().gemm_measure_tensor_rate(DTYPE.get(ab, ab), int(block_scaled), int(cta_group), int(iters),
                                          ctypes.byref(out)), "gemm_measure_tensor_rate")
    return {n: getattr(out, n) for n, _ in TensorRate._fields_}


class Plan:
    """Owning wrapper of a gemm_plan_t (destroyed on close / context exit)."""

    def __init__(self, M, N, K, ab="bf16", d="f32", block_scaled=GEMM_SCALE_NONE, flags=0, c="f32",
                 a_row_major=True, b_row_major=False):
        """``block_scaled``: GEMM_SCALE_NONE / GEMM_SCALE_UE8M0_32 (True) / GEMM_SCALE_UE4M3_16."""
        self.M, self.N, self.K, self.ab, self.d = M, N, K, ab, d
        self.block_scaled = int(block_scaled)
        self.handle = None
        self.handle = gemm_plan_create(M, N, K, ab, c, d, int(a_row_major), int(b_row_major), int(block_scaled), flags)

    @property
    def info(self) -> dict:
        return gemm_plan_get_info(self.handle)

    def run(self, A, B, C, D, SFA=None, SFB=None, stream=None):
        return gemm_run(self.handle, A, B, C, D, SFA, SFB, stream)

    def run_host(self, A, B, C, D, SFA=None, SFB=None, stream=None):
        return gemm_run_host(self.handle, A, B, C, D, SFA, SFB, stream)

    def last_status(self) -> int:
        return gemm_plan_last_status(self.handle)

    def set_timeout(self, ns: int):
        gemm_plan_set_timeout(self.handle, ns)

    def set_split_k(self, splits: int):
        gemm_plan_set_split_k(self.handle, splits)

    def set_stream_k(self, enable: bool):
        gemm_plan_set_stream_k(self.handle, int(enable))

    def set_clock_meter(self, enable: bool):
        gemm_plan_set_clock_meter(self.handle, int(enable))

    def read_clock_meter(self) -> dict:
        return gemm_plan_read_clock_meter(self.handle)

    def close(self):
        if self.handle:
            gemm_plan_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class ChainPlan(Plan):
    """Owning wrapper of a two-product chain plan: D = C + round(A·B)·E."""

    def __init__(self, M, N1, N2, K, ab="bf16", d="f32", flags=0):
        self.M, self.N1, self.N2, self.K, self.ab, self.d = M, N1, N2, K, ab, d
        self.handle = None
        self.handle = gemm_chain_plan_create(M, N1, N2, K, ab, d, flags)

    def run(self, A, B, E, C, D, stream=None):
        return gemm_chain_run(self.handle, A, B, E, C, D, stream)

    def run_host(self, A, B, E, C, D, stream=None):
        return gemm_chain_run_host(self.handle, A, B, E, C, D, stream)


def gemm_testing_schedule(chain: bool, tiles_m: int, tiles_n: int, group_m: int, num_kb: int, splits: int,
                          sk_dp_tiles: int, sk_units: int, unit: int, units: int) -> list:
    """The pieces (tm, tn, kb0, kb1, role, slot) one unit of the persistent grid processes, from
    the kernels' own schedule code run on the host (no device needed)."""
    n = ctypes.c_int()
    args = (int(bool(chain)), tiles_m, tiles_n, group_m, num_kb, splits, sk_dp_tiles, sk_units, unit, units)
    cap = 64
    while True:
        buf = (ctypes.c_int * (6 * cap))()
        st = lib().gemm_testing_schedule(*args, buf, cap, ctypes.byref(n))
        if st != GEMM_OK:
            raise GemmError(st, "gemm_testing_schedule")
        if n.value <= cap:
            return [tuple(buf[6 * i:6 * i + 6]) for i in range(n.value)]
        cap = n.value
