"""Thin ctypes binding of the carbon_gemm C ABI (include/carbon_gemm.h).

Argument marshalling only: every step of the GEMMs runs in the library's
CUDA kernels.  Functions take torch tensors (or raw integer device pointers)
and the same arguments as the C entry points, and raise ``CarbonError`` on a
status other than CARBON_OK.  The library is loaded on the first call (or the
first access to ``lib``), so importing the package maps no CUDA code; there
is no fallback: if the compiled library is missing, that first call raises
``ImportError``.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
# CARBON_GEMM_LIBRARY may name another build of the library (the
# bounds-checked libcarbon_gemm_bounds.so); default: the regular one.
LIB_PATH = os.environ.get("CARBON_GEMM_LIBRARY") or os.path.join(HERE, "libcarbon_gemm.so")
HEADERS = [os.path.join(os.path.dirname(HERE), "include", h)
           for h in ("carbon_gemm.h", "carbon_gemm_debug.h")]

F32, BF16, F16 = 0, 1, 2
TIER_EXACT, TIER_TC, TIER_SUPERACC = 0, 1, 2
PASS_FWD, PASS_DX, PASS_DW = 0, 1, 2
STATUS = {0: "CARBON_OK", 1: "CARBON_ERR_INVALID_ARG", 2: "CARBON_ERR_UNSUPPORTED",
          3: "CARBON_ERR_MISALIGNED", 4: "CARBON_ERR_CUDA", 5: "CARBON_ERR_TIMEOUT",
          6: "CARBON_ERR_SCRATCH_LIMIT", 7: "CARBON_ERR_OUT_OF_BOUNDS"}
DTYPES = {"f32": F32, "bf16": BF16, "f16": F16}
TIERS = {"exact": TIER_EXACT, "tc": TIER_TC, "superacc": TIER_SUPERACC}
PASSES = {"fwd": PASS_FWD, "dx": PASS_DX, "dw": PASS_DW}


class CarbonError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"carbon_gemm CUDA library not built ({LIB_PATH} missing); run "
            "`python deterministic_invariant_gemm_fwd_gb300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, dp = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    sig = {
        "carbon_gemm_fwd": [vp, vp, vp, vp, i64, i64, i64, i32, i32, vp],
        "carbon_gemm_dx": [vp, vp, vp, i64, i64, i64, i32, i32, vp],
        "carbon_gemm_dw": [vp, vp, vp, i64, i64, i64, i32, i32, vp],
        "carbon_gemm_dw_f32": [vp, vp, vp, i64, i64, i64, i32, vp],
        "carbon_get_device_status": [vp],
        "carbon_gemm_exact_bf16_noalloc": [i32, vp, vp, vp, vp, i64, i64, i64, vp],
        "carbon_gemm_chunk_values": [i32, vp, vp, vp, i64, i64, i64, i32, vp],
        "carbon_chunk_values_combine": [vp, vp, i64, i64, i64, vp, i32, vp],
        "carbon_debug_exact_y64": [i32, vp, vp, vp, vp, i64, i64, i64, i32, vp],
        "carbon_debug_tc_f32": [i32, vp, vp, vp, vp, i64, i64, i64, vp],
        "carbon_debug_round": [i32, vp, vp, i64, vp],
        "carbon_debug_timeout_probe": [i64, vp],
        "carbon_measure_fp64_rate": [ctypes.POINTER(dp), ctypes.POINTER(dp), vp],
        "carbon_measure_int_mac_rate": [ctypes.POINTER(dp), vp],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.carbon_status_string.argtypes = [i32]
    lib.carbon_status_string.restype = ctypes.c_char_p
    lib.carbon_last_cuda_error.argtypes = []
    lib.carbon_last_cuda_error.restype = ctypes.c_char_p
    lib.carbon_abi_version.argtypes = []
    lib.carbon_abi_version.restype = ctypes.c_int
    lib.carbon_debug_launch_count.argtypes = []
    lib.carbon_debug_launch_count.restype = ctypes.c_int64
    lib.carbon_debug_kernel_timing.argtypes = [ctypes.c_int]
    lib.carbon_debug_kernel_timing.restype = None
    lib.carbon_debug_kernel_time.argtypes = [ctypes.POINTER(ctypes.c_double),
                                             ctypes.POINTER(ctypes.c_int64),
                                             ctypes.POINTER(ctypes.c_int64)]
    lib.carbon_debug_kernel_time.restype = ctypes.c_int
    lib.carbon_debug_exact_phase_time.argtypes = [ctypes.POINTER(ctypes.c_double)] * 3
    lib.carbon_debug_exact_phase_time.restype = ctypes.c_int
    lib.carbon_debug_exact_path_counts.argtypes = [ctypes.POINTER(ctypes.c_int64),
                                                   ctypes.POINTER(ctypes.c_int64)]
    lib.carbon_debug_exact_path_counts.restype = ctypes.c_int
    return lib


_LIB = None


def _lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def __getattr__(name):
    # ``_binding.lib`` loads the library on first access.
    if name == "lib":
        return _lib()
    raise AttributeError(name)


def declared_functions() -> list:
    """Names of every function declared in include/*.h."""
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(carbon_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != 0:
        detail = _lib().carbon_last_cuda_error().decode() if status == 4 else ""
        raise CarbonError(status, where, detail)


def _code(table, v):
    return table[v] if isinstance(v, str) else int(v)


def carbon_gemm_fwd(Y, X, W, bias, M, K, N, dtype, tier, stream=None) -> None:
    _check(_lib().carbon_gemm_fwd(_ptr(Y), _ptr(X), _ptr(W), _ptr(bias), M, K, N,
                               _code(DTYPES, dtype), _code(TIERS, tier), _stream(stream)),
           "carbon_gemm_fwd")


def carbon_gemm_dx(dX, dY, W, M, K, N, dtype, tier, stream=None) -> None:
    _check(_lib().carbon_gemm_dx(_ptr(dX), _ptr(dY), _ptr(W), M, K, N,
                              _code(DTYPES, dtype), _code(TIERS, tier), _stream(stream)),
           "carbon_gemm_dx")


def carbon_gemm_dw(dW, X, dY, M, K, N, dtype, tier, stream=None) -> None:
    _check(_lib().carbon_gemm_dw(_ptr(dW), _ptr(X), _ptr(dY), M, K, N,
                              _code(DTYPES, dtype), _code(TIERS, tier), _stream(stream)),
           "carbon_gemm_dw")


def carbon_gemm_dw_f32(dW, X, dY, M, K, N, tier, stream=None) -> None:
    """dW (fp32) = X^T.dY of bf16 operands: the exact tier's float64 value
    rounded once to fp32, or the tensor-core tier's fp32 accumulator."""
    _check(_lib().carbon_gemm_dw_f32(_ptr(dW), _ptr(X), _ptr(dY), M, K, N, _code(TIERS, tier),
                                  _stream(stream)), "carbon_gemm_dw_f32")


def carbon_gemm_exact_bf16_noalloc(pass_, out, A, B, bias, M, K, N, stream=None) -> None:
    """Exact-tier bf16 GEMM that allocates no device memory (fixed 64 MiB
    library workspace); same bits as carbon_gemm_fwd/dx/dw with the exact tier."""
    _check(_lib().carbon_gemm_exact_bf16_noalloc(_code(PASSES, pass_), _ptr(out), _ptr(A), _ptr(B),
                                              _ptr(bias), M, K, N, _stream(stream)),
           "carbon_gemm_exact_bf16_noalloc")


def carbon_gemm_chunk_values(pass_, P, A, B, M, K, N, dtype, stream=None) -> None:
    """Exact-tier chunk values of one rank's share of a reduction:
    P[q][i][j] = fl(s + c) of chunk q, float64 [ceil(R/256)][rows][cols]."""
    _check(_lib().carbon_gemm_chunk_values(_code(PASSES, pass_), _ptr(P), _ptr(A), _ptr(B),
                                           M, K, N, _code(DTYPES, dtype), _stream(stream)),
           "carbon_gemm_chunk_values")


def carbon_chunk_values_combine(out, P, nchunks, rows, cols, bias, dtype, stream=None) -> None:
    """Outer KBN over chunk values in chunk order, the bias, one rounding."""
    _check(_lib().carbon_chunk_values_combine(_ptr(out), _ptr(P), nchunks, rows, cols, _ptr(bias),
                                              _code(DTYPES, dtype), _stream(stream)),
           "carbon_chunk_values_combine")


def carbon_get_device_status(stream=None) -> int:
    """Synchronises the stream; returns the status code (does not raise)."""
    return int(_lib().carbon_get_device_status(_stream(stream)))


def carbon_debug_exact_y64(pass_, y64, A, B, bias, M, K, N, dtype, stream=None) -> None:
    _check(_lib().carbon_debug_exact_y64(_code(PASSES, pass_), _ptr(y64), _ptr(A), _ptr(B),
                                      _ptr(bias), M, K, N, _code(DTYPES, dtype),
                                      _stream(stream)), "carbon_debug_exact_y64")


def carbon_debug_tc_f32(pass_, acc, A, B, bias, M, K, N, stream=None) -> None:
    _check(_lib().carbon_debug_tc_f32(_code(PASSES, pass_), _ptr(acc), _ptr(A), _ptr(B),
                                   _ptr(bias), M, K, N, _stream(stream)),
           "carbon_debug_tc_f32")


def carbon_debug_round(dtype, out, inp, n, stream=None) -> None:
    _check(_lib().carbon_debug_round(_code(DTYPES, dtype), _ptr(out), _ptr(inp), n,
                                  _stream(stream)), "carbon_debug_round")


def carbon_debug_timeout_probe(budget_ns: int, stream=None) -> None:
    _check(_lib().carbon_debug_timeout_probe(budget_ns, _stream(stream)),
           "carbon_debug_timeout_probe")


def carbon_measure_fp64_rate(stream=None) -> tuple:
    """(DFMA lane-ops/s, DADD lane-ops/s) measured on the current device."""
    a, b = ctypes.c_double(), ctypes.c_double()
    _check(_lib().carbon_measure_fp64_rate(ctypes.byref(a), ctypes.byref(b), _stream(stream)),
           "carbon_measure_fp64_rate")
    return a.value, b.value


def carbon_measure_int_mac_rate(stream=None) -> float:
    """32x32->64-bit integer multiply-adds per second on the current device."""
    a = ctypes.c_double()
    _check(_lib().carbon_measure_int_mac_rate(ctypes.byref(a), _stream(stream)),
           "carbon_measure_int_mac_rate")
    return a.value


def carbon_status_string(status: int) -> str:
    return _lib().carbon_status_string(status).decode()


def carbon_abi_version() -> int:
    return int(_lib().carbon_abi_version())


def carbon_debug_launch_count() -> int:
    return int(_lib().carbon_debug_launch_count())


def carbon_debug_kernel_timing(enable: bool) -> None:
    """Start (and clear) or stop event timing of the exact tier's tensor-core kernel."""
    _lib().carbon_debug_kernel_timing(1 if enable else 0)


def carbon_debug_kernel_time():
    """(milliseconds, launches, plane products) recorded since timing was enabled."""
    ms, n, kg = ctypes.c_double(), ctypes.c_int64(), ctypes.c_int64()
    _check(_lib().carbon_debug_kernel_time(ctypes.byref(ms), ctypes.byref(n), ctypes.byref(kg)),
           "carbon_debug_kernel_time")
    return ms.value, int(n.value), int(kg.value)


def carbon_debug_exact_phase_time():
    """(pre-pass, tensor-core kernel, post-pass) milliseconds of the bf16 exact
    tier's calls recorded since timing was enabled."""
    a, b, c = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    _check(_lib().carbon_debug_exact_phase_time(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
           "carbon_debug_exact_phase_time")
    return a.value, b.value, c.value


def carbon_debug_exact_path_counts():
    """(chunk repairs, whole-output fix-ups) recorded since timing was enabled."""
    r, f = ctypes.c_int64(), ctypes.c_int64()
    _check(_lib().carbon_debug_exact_path_counts(ctypes.byref(r), ctypes.byref(f)),
           "carbon_debug_exact_path_counts")
    return int(r.value), int(f.value)
