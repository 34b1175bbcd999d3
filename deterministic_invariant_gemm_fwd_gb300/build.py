"""Build the carbon_gemm CUDA library in-tree (nvcc, sm_103a only).

Produces ``libcarbon_gemm.so`` next to this file.  The CUDA runtime is
linked statically, so the library needs only the NVIDIA driver at run time;
the driver's tensor-map encoder is looked up through the runtime's
driver-entry-point query, so there is no link-time dependency on libcuda.

Usage: ``python deterministic_invariant_gemm_fwd_gb300/build.py [--force]`` (run as a
file: importing the package itself loads the library).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(HERE, "libcarbon_gemm.so")
BUILD_DIR = os.path.join(HERE, "_build")
SOURCES = ["api.cu", "exact_kbn.cu", "exact_int.cu", "exact_tc.cu", "superacc.cu", "tc_gemm.cu",
           "measure.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xptxas", "-v", *ARCH]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, nvcc: str) -> tuple[str, str]:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    # the exact tier's float64 arithmetic is written with explicit *_rn
    # intrinsics; forbid any contraction the compiler might add on top
    if src in ("exact_kbn.cu", "exact_int.cu", "exact_tc.cu"):
        cmd.insert(1, "-fmad=false")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit (in parallel) and link the library."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, nvcc), SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", *ARCH, "-cudart", "static", "-o", tmp,
           *[o for o, _ in results], "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
