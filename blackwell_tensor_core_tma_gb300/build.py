"""Build libgb300gemm.so (the CUDA library) in-tree with nvcc for sm_103a.

Each translation unit under csrc/ compiles in parallel to an object file,
then nvcc links them (with the static CUDA runtime) into a shared library
next to this file.  Nothing is installed anywhere else.

Variant "trace" (libgb300gemm_trace.so, compiled with GB300_TRACE=1) keeps the
kernels' per-role clock counters (gemm_testing_set_trace); variant "checks"
(libgb300gemm_checks.so) keeps the kernels' on-device coordinate checks and uses
other ring depths; the default library compiles both out.  The binding loads the variant named by the environment
variable GB300GEMM_VARIANT (unset: the default library).
"""

from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libgb300gemm.so")
# "checks": the kernels' on-device coordinate checks (GEMM_ERR_CHECK), with ring depths other
# than the default ones so that a run of the tests on it also exercises other ring phases
VARIANTS = {
    "": [],
    "trace": ["-DGB300_TRACE=1"],
    "checks": ["-DGB300_CHECKS=1", "-DGB300_F16_CG1_STAGES=3", "-DGB300_F16_CG2_STAGES=5",
               "-DGB300_MXF8_PAIR_STAGES=5", "-DGB300_MXF8_NARROW_STAGES=4", "-DGB300_MXF4_PAIR_STAGES=4",
               "-DGB300_NVF4_PAIR_STAGES=4"],
}


def lib_path(variant: str = "") -> str:
    if variant not in VARIANTS:
        raise ValueError(f"unknown library variant {variant!r} (known: {sorted(VARIANTS)})")
    return LIB if not variant else os.path.join(HERE, f"libgb300gemm_{variant}.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return path


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))


def up_to_date(variant: str = "") -> bool:
    out = lib_path(variant)
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None, variant: str = "") -> str:
    target = lib_path(variant)
    if not force and up_to_date(variant):
        return target
    cc = nvcc()
    extra = VARIANTS[variant] + list(extra or [])
    with tempfile.TemporaryDirectory(prefix="gb300gemm_") as tmp:
        def compile_one(src):
            obj = os.path.join(tmp, os.path.basename(src) + ".o")
            cmd = [cc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
            if verbose and r.stderr:
                print(r.stderr)
            return obj

        with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(sources()))) as ex:
            objs = list(ex.map(compile_one, sources()))
        out = os.path.join(tmp, "libgb300gemm.so")
        cmd = [cc, *ARCH, "-shared", "-o", out, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
        staged = target + ".tmp"
        shutil.copyfile(out, staged)
        os.replace(staged, target)
    return target


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra=["-Xptxas", "-v"] if "--ptxas" in sys.argv else None,
                variant="trace" if "--trace" in sys.argv else ""))
