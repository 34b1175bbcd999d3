"""Build the carbon_gemm CUDA library in-tree (nvcc, sm_103a only).

Produces ``libcarbon_gemm.so`` next to this file.  The CUDA runtime is
linked statically, so the library needs only the NVIDIA driver at run time;
the driver's tensor-map encoder is looked up through the runtime's
driver-entry-point query, so there is no link-time dependency on libcuda.

A second library, ``libcarbon_gemm_bounds.so``, is the bounds-checked debug
build (``-DCARBON_DEBUG_BOUNDS``): every global-memory access the kernels
index themselves is checked against its buffer, an access out of range is
skipped and reported as CARBON_ERR_OUT_OF_BOUNDS by
carbon_get_device_status().  The package loads it instead of the regular
library when the environment variable CARBON_GEMM_LIBRARY names it.

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
LIB_BOUNDS = os.path.join(HERE, "libcarbon_gemm_bounds.so")
BUILD_DIR = os.path.join(HERE, "_build")
# variant -> (library, object folder, extra flags)
VARIANTS = {"regular": (LIB, BUILD_DIR, []),
            "bounds": (LIB_BOUNDS, os.path.join(HERE, "_build_bounds"), ["-DCARBON_DEBUG_BOUNDS"])}
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


def _compile(src: str, nvcc: str, variant: str) -> tuple[str, str]:
    _, build_dir, extra = VARIANTS[variant]
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    # the exact tier's float64 arithmetic is written with explicit *_rn
    # intrinsics; forbid any contraction the compiler might add on top
    if src in ("exact_kbn.cu", "exact_int.cu", "exact_tc.cu"):
        cmd.insert(1, "-fmad=false")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src} ({variant}):\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _link(nvcc: str, lib: str, objs: list) -> None:
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", *ARCH, "-cudart", "static", "-o", tmp, *objs,
           "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False, variants=("regular", "bounds")) -> str:
    """Compile every translation unit of each variant (all in parallel) and
    link the libraries; returns the regular library's path."""
    todo = [v for v in variants
            if force or not os.path.exists(VARIANTS[v][0]) or os.path.getmtime(VARIANTS[v][0]) < _deps_mtime()]
    if not todo:
        return LIB
    nvcc = _nvcc()
    jobs = [(v, src) for v in todo for src in SOURCES]
    for v in todo:
        os.makedirs(VARIANTS[v][1], exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 8))) as ex:
        results = list(ex.map(lambda job: _compile(job[1], nvcc, job[0]), jobs))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    for v in todo:
        _link(nvcc, VARIANTS[v][0], [o for (vv, _), (o, _) in zip(jobs, results) if vv == v])
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
