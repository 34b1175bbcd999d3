"""CPU oracle for the deterministic linear-layer GEMM (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library it wraps (``oracle.c``)
is plain C: products in float64, Kahan-Babushka-Neumaier accumulation in
256-wide chunks left to right, chunk values combined left to right with KBN,
bias added in float64, one round-to-nearest-even to the output type (Carbon
README, "How It Works"; sgemm-bi "Determinism contracts" for the downcast).
It shares nothing with the CUDA library.  ``gemm_superacc`` computes the
correctly rounded tier (README "Roadmap": superaccumulators): the exact dot
product plus the bias, rounded once.

Every function of the oracle has pins in ``tests/test_oracle.py``: closed
forms, exact rational sums within the KBN error bound, exact rounding, and
the batch/permutation/transposition invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
CFLAGS = ["-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared", "-pthread"]

PASSES = {"fwd": 0, "dx": 1, "dw": 2}
DTYPES = {"f32": 0, "bf16": 1, "f16": 2}
CHUNK = 256

_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (gcc, no GPU needed)."""
    if (force or not os.path.exists(_LIB)
            or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_gemm.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp,
                                    i64, i64, i64, vp, vp, ctypes.c_int]
        lib.oracle_gemm.restype = ctypes.c_int
        lib.oracle_gemm_at.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp,
                                       i64, i64, i64, vp, vp, i64, vp, vp,
                                       ctypes.c_int]
        lib.oracle_gemm_at.restype = ctypes.c_int
        lib.oracle_gemm_superacc.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp,
                                             i64, i64, i64, vp, vp, i64, vp, ctypes.c_int]
        lib.oracle_gemm_superacc.restype = ctypes.c_int
        lib.oracle_round.argtypes = [ctypes.c_int, vp, vp, i64]
        lib.oracle_round.restype = None
        lib.oracle_chunk_width.restype = ctypes.c_int
        _lib = lib
    return _lib


def _np_dtype(dtype: str):
    return np.float32 if dtype == "f32" else np.uint16


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _prep(a, dtype):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != _np_dtype(dtype):
        raise TypeError(f"expected {_np_dtype(dtype).__name__} storage for {dtype}")
    return a


def out_shape(pass_: str, M: int, K: int, N: int):
    return {"fwd": (M, N), "dx": (M, K), "dw": (K, N)}[pass_]


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def gemm(pass_: str, dtype: str, A, B, bias, M: int, K: int, N: int,
         threads: int | None = None):
    """Dense pass.  A, B = (X, W) fwd; (dY, W) dX; (X, dY) dW.

    Returns (out, y64): the rounded output (fp32 array, or uint16 bf16 bits)
    and the float64 value before rounding.
    """
    lib = _load()
    A, B, bias = _prep(A, dtype), _prep(B, dtype), _prep(bias, dtype)
    shape = out_shape(pass_, M, K, N)
    out = np.empty(shape, dtype=_np_dtype(dtype))
    y64 = np.empty(shape, dtype=np.float64)
    rc = lib.oracle_gemm(PASSES[pass_], DTYPES[dtype], _ptr(A), _ptr(B),
                         _ptr(bias), M, K, N, _ptr(out), _ptr(y64),
                         threads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_gemm failed ({rc})")
    return out, y64


def gemm_at(pass_: str, dtype: str, A, B, bias, M: int, K: int, N: int,
            rows, cols, threads: int | None = None):
    """Selected outputs (rows[k], cols[k]) only; returns (out, y64) vectors."""
    lib = _load()
    A, B, bias = _prep(A, dtype), _prep(B, dtype), _prep(bias, dtype)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    R, C = out_shape(pass_, M, K, N)
    if rows.shape != cols.shape or rows.ndim != 1:
        raise ValueError("rows/cols must be 1-D and of equal length")
    if rows.size and (rows.min() < 0 or rows.max() >= R or cols.min() < 0 or cols.max() >= C):
        raise ValueError("sample coordinates out of range")
    out = np.empty(rows.shape, dtype=_np_dtype(dtype))
    y64 = np.empty(rows.shape, dtype=np.float64)
    rc = lib.oracle_gemm_at(PASSES[pass_], DTYPES[dtype], _ptr(A), _ptr(B),
                            _ptr(bias), M, K, N, _ptr(rows), _ptr(cols),
                            rows.size, _ptr(out), _ptr(y64),
                            threads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_gemm_at failed ({rc})")
    return out, y64


def gemm_superacc(pass_: str, dtype: str, A, B, bias, M: int, K: int, N: int,
                  rows=None, cols=None, threads: int | None = None):
    """Correctly rounded tier: RNE of the exact dot product (+ bias for fwd),
    every output (dense) or the outputs (rows[k], cols[k]).  Returns the
    rounded outputs (fp32 array, or uint16 bits of bf16 / fp16)."""
    lib = _load()
    A, B, bias = _prep(A, dtype), _prep(B, dtype), _prep(bias, dtype)
    if rows is None:
        out = np.empty(out_shape(pass_, M, K, N), dtype=_np_dtype(dtype))
        rc = lib.oracle_gemm_superacc(PASSES[pass_], DTYPES[dtype], _ptr(A), _ptr(B),
                                      _ptr(bias), M, K, N, None, None, 0, _ptr(out),
                                      threads or default_threads())
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        R, C = out_shape(pass_, M, K, N)
        if rows.shape != cols.shape or rows.ndim != 1:
            raise ValueError("rows/cols must be 1-D and of equal length")
        if rows.size and (rows.min() < 0 or rows.max() >= R or cols.min() < 0 or cols.max() >= C):
            raise ValueError("sample coordinates out of range")
        out = np.empty(rows.shape, dtype=_np_dtype(dtype))
        rc = lib.oracle_gemm_superacc(PASSES[pass_], DTYPES[dtype], _ptr(A), _ptr(B),
                                      _ptr(bias), M, K, N, _ptr(rows), _ptr(cols), rows.size,
                                      _ptr(out), threads or default_threads())
    if rc:
        raise RuntimeError(f"oracle_gemm_superacc failed ({rc})")
    return out


def round_out(dtype: str, y64) -> np.ndarray:
    """The oracle's output rounding alone (float64 -> fp32 or bf16 bits)."""
    lib = _load()
    y = np.ascontiguousarray(y64, dtype=np.float64)
    out = np.empty(y.shape, dtype=_np_dtype(dtype))
    lib.oracle_round(DTYPES[dtype], _ptr(y), _ptr(out), y.size)
    return out


def chunk_width() -> int:
    return int(_load().oracle_chunk_width())
