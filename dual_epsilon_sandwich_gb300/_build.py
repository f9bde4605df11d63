"""Build libmrn.so in-tree with nvcc for sm_103a (GB300).

One translation unit per operation plus the C-ABI layer, compiled in parallel,
then linked into ``dual_epsilon_sandwich_gb300/libmrn.so`` (the CUDA runtime is
linked statically).  No fast-math: sqrt and division stay IEEE-rounded.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIBRARY = os.path.join(PKG, "libmrn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-I", INCLUDE, "-I", CSRC]
SOURCES = ["mrn_api.cpp", "mrn_ops_rmsnorm.cu", "mrn_ops_then_add.cu", "mrn_ops_sandwich.cu",
           "mrn_ops_add_rmsnorm.cu", "mrn_ops_then_add_scale.cu", "mrn_ops_rmsnorm_q8_1.cu",
           "mrn_ops_seam_f16.cu", "mrn_ops_seam_bf16.cu", "mrn_seam_scale.cu"]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH") or "/usr/local/cuda"
    cand = os.path.join(home, "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: set CUDA_HOME or put nvcc on PATH")
    return found


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "mrn.h"))
    return files


def is_stale() -> bool:
    if not os.path.exists(LIBRARY):
        return True
    t = os.path.getmtime(LIBRARY)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _compile(src: str, ptxas_verbose: bool) -> tuple[str, str]:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    if ptxas_verbose and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    return obj, res.stderr


def build(force: bool = False, ptxas_verbose: bool = False, log=None) -> str:
    """Compile and link libmrn.so; returns its path.  ``log`` receives compiler
    diagnostics (e.g. ``-Xptxas -v`` register reports) when given."""
    if not force and not ptxas_verbose and not is_stale():
        return LIBRARY
    os.makedirs(BUILD_DIR, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
        results = list(pool.map(lambda s: _compile(s, ptxas_verbose), SOURCES))
    if log is not None:
        for _, diag in results:
            log(diag)
    tmp = LIBRARY + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    import sys
    verbose = "-v" in sys.argv
    print(build(force=True, ptxas_verbose=verbose, log=(print if verbose else None)))
