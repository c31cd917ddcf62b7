"""Build the in-tree C-ABI library ``libmoe_gb300.so`` with nvcc for sm_103a.

Each ``csrc/*.cu`` translation unit compiles in parallel to an object under
``_build/``; the objects link into one shared library next to this file.
Rebuilds only what changed (source or header newer than the object).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build", "moe")
LIB = os.path.join(PKG, "libmoe_gb300.so")
# Phase-trace variant of the library (decode kernel with global-timer stamps,
# see trace_phases.py); never loaded by the package unless asked for.
TRACE_BUILD = os.path.join(ROOT, "_build", "moe_trace")
TRACE_LIB = os.path.join(PKG, "libmoe_gb300_trace.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _cuda_lib_dir() -> str:
    nvcc = os.path.realpath(_nvcc())
    return os.path.join(os.path.dirname(os.path.dirname(nvcc)), "lib64")


def _newest_dep() -> float:
    deps = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]
    return max(os.path.getmtime(d) for d in deps)


def _compile(src: str, extra: list[str], build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), _newest_dep()):
        return obj
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    os.replace(obj + ".tmp", obj)
    return obj


def build(verbose: bool = False, extra: list[str] | None = None, trace: bool = False) -> str:
    """Compile every CUDA source and link the shared library; returns its path.
    ``trace=True`` builds the phase-trace variant (``-DMOE_PHASE_TRACE``) into
    its own directory and library instead."""
    build_dir, lib = (TRACE_BUILD, TRACE_LIB) if trace else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    extra = list(extra or []) + (["-DMOE_PHASE_TRACE"] if trace else [])
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), srcs))
    newest = max(os.path.getmtime(o) for o in objs)
    if not os.path.exists(lib) or os.path.getmtime(lib) < newest:
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "shared",
               "-Xlinker", "-rpath," + _cuda_lib_dir()]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    if verbose:
        print(lib)
    return lib


def ptxas_report() -> str:
    """Registers / spills / shared memory per kernel (``-Xptxas -v``)."""
    out = []
    for src in sorted(glob.glob(os.path.join(CSRC, "*.cu"))):
        cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, "-Xptxas", "-v", "-c", src, "-o", os.devnull]
        r = subprocess.run(cmd, capture_output=True, text=True)
        out.append(f"== {os.path.basename(src)}\n{r.stderr}")
    return "\n".join(out)


if __name__ == "__main__":
    build(verbose=True)
