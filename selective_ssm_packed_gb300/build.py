"""Builds libvarlen_ssm.so in-tree for sm_103a (GB300) with nvcc.

Each .cu file compiles in parallel to an object in ``_build/``; the objects
link into ``_build/libvarlen_ssm.so`` (CUDA runtime linked statically).  A
rebuild happens only when a source or header is newer than the library.
Set VSSM_PTXAS_VERBOSE=1 to print register / spill / shared-memory usage.

``build(checks=True)`` (or VSSM_CHECKS=1 in the environment) builds the
checked variant instead, ``_build_checks/libvarlen_ssm_checks.so``: the same
sources with -DVSSM_CHECKS=1, whose kernels verify the indices that input
data can push out of range and report a failure in the call's status word
(VSSM_ERR_DEVICE_CHECK) instead of making the access; the calls also verify
caller-supplied position indices against cu_seqlens.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libvarlen_ssm.so")
CHECKS_BUILD_DIR = os.path.join(HERE, "_build_checks")
CHECKS_LIB_PATH = os.path.join(CHECKS_BUILD_DIR, "libvarlen_ssm_checks.so")

SOURCES = ["api.cu", "misc.cu", "conv.cu", "scan_fwd.cu", "scan_bwd.cu", "noalloc.cu", "packer.cu"]
HEADERS = [os.path.join(CSRC, "common.cuh"), os.path.join(CSRC, "kernels.h"),
           os.path.join(INCLUDE, "varlen_ssm.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"),
                 os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc"),
                 shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or CUDA_HOME)")


def checks_requested() -> bool:
    """Whether the environment asks for the checked build (VSSM_CHECKS=1)."""
    return os.environ.get("VSSM_CHECKS", "0") not in ("", "0")


def lib_path(checks: bool | None = None) -> str:
    if checks is None:
        checks = checks_requested()
    return CHECKS_LIB_PATH if checks else LIB_PATH


def _flags(checks: bool = False):
    f = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]
    if checks:
        f.append("-DVSSM_CHECKS=1")
    if os.environ.get("VSSM_PTXAS_VERBOSE"):
        f += ["-Xptxas", "-v"]
    return f


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, checks: bool | None = None) -> str:
    """Builds the library (the checked variant when checks is true, or when it
    is None and VSSM_CHECKS=1 is set) and returns its path."""
    if checks is None:
        checks = checks_requested()
    build_dir, out_path = (CHECKS_BUILD_DIR, CHECKS_LIB_PATH) if checks else (BUILD_DIR, LIB_PATH)
    os.makedirs(build_dir, exist_ok=True)
    nvcc = nvcc_path()
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s, *HEADERS]):
            jobs.append([nvcc, *_flags(checks), "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    if jobs:
        with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
            for cmd, r in ex.map(run, jobs):
                if verbose or os.environ.get("VSSM_PTXAS_VERBOSE"):
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if force or jobs or _stale(out_path, objs):
        tmp = out_path + f".tmp{os.getpid()}"
        r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out_path)
    return out_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, checks="--checks" in sys.argv or None))
