"""Deterministic, batch-invariant linear-layer GEMM for GB300 (sm_103a).

The C ABI (``include/carbon_gemm.h``) is exposed with the same names by
``_binding``; the torch-tensor helpers below only allocate the output tensor
and call it.  Weights are stored [in, out] (sgemm-bi page, "Use").

    from deterministic_invariant_gemm_fwd_gb300 import linear_fwd, linear_dx, linear_dw
    Y  = linear_fwd(X, W, b, tier="exact")   # Y  = X.W + b
    dX = linear_dx(dY, W, tier="exact")      # dX = dY.W^T
    dW = linear_dw(X, dY, tier="exact")      # dW = X^T.dY

``deterministic_invariant_gemm_fwd_gb300.nn`` wraps them in an autograd
``Linear`` / ``deterministic_linear`` (with a deterministic bias gradient).
"""
from __future__ import annotations

from ._binding import (CarbonError, carbon_abi_version, carbon_debug_exact_y64,  # noqa: F401
                       carbon_debug_exact_path_counts, carbon_debug_exact_phase_time,
                       carbon_debug_kernel_time,
                       carbon_debug_kernel_timing,
                       carbon_debug_launch_count, carbon_debug_round,
                       carbon_debug_tc_f32, carbon_debug_timeout_probe,
                       carbon_chunk_values_combine, carbon_gemm_chunk_values,
                       carbon_gemm_dw, carbon_gemm_dw_f32, carbon_gemm_dx, carbon_gemm_fwd,
                       carbon_get_device_status, carbon_measure_fp64_rate,
                       carbon_measure_int_mac_rate,
                       carbon_status_string)


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return "f32"
    if t.dtype == torch.bfloat16:
        return "bf16"
    if t.dtype == torch.float16:
        return "f16"
    raise TypeError(f"unsupported dtype {t.dtype}; expected float32, bfloat16 or float16")


def _check2d(name, t):
    if t.dim() != 2 or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name} must be a contiguous 2-D CUDA tensor")


def linear_fwd(X, W, bias=None, tier="exact", stream=None):
    """Y[M,N] = X[M,K] . W[K,N] + bias[N]."""
    import torch
    _check2d("X", X)
    _check2d("W", W)
    M, K = X.shape
    if W.shape[0] != K:
        raise ValueError("X and W disagree on K")
    N = W.shape[1]
    if bias is not None and (bias.numel() != N or not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous [N] tensor")
    Y = torch.empty((M, N), dtype=X.dtype, device=X.device)
    carbon_gemm_fwd(Y, X, W, bias, M, K, N, _dtype_code(X), tier, stream)
    return Y


def linear_dx(dY, W, tier="exact", stream=None):
    """dX[M,K] = dY[M,N] . W[K,N]^T."""
    import torch
    _check2d("dY", dY)
    _check2d("W", W)
    M, N = dY.shape
    K = W.shape[0]
    if W.shape[1] != N:
        raise ValueError("dY and W disagree on N")
    dX = torch.empty((M, K), dtype=dY.dtype, device=dY.device)
    carbon_gemm_dx(dX, dY, W, M, K, N, _dtype_code(dY), tier, stream)
    return dX


def linear_dw(X, dY, tier="exact", stream=None):
    """dW[K,N] = X[M,K]^T . dY[M,N]."""
    import torch
    _check2d("X", X)
    _check2d("dY", dY)
    M, K = X.shape
    if dY.shape[0] != M:
        raise ValueError("X and dY disagree on M")
    N = dY.shape[1]
    dW = torch.empty((K, N), dtype=X.dtype, device=X.device)
    carbon_gemm_dw(dW, X, dY, M, K, N, _dtype_code(X), tier, stream)
    return dW


def linear_dw_f32(X, dY, tier="exact", stream=None):
    """dW[K,N] in fp32 = X[M,K]^T . dY[M,N] for bf16 X and dY."""
    import torch
    _check2d("X", X)
    _check2d("dY", dY)
    if X.dtype != torch.bfloat16 or dY.dtype != torch.bfloat16:
        raise TypeError("linear_dw_f32 takes bfloat16 operands")
    M, K = X.shape
    if dY.shape[0] != M:
        raise ValueError("X and dY disagree on M")
    N = dY.shape[1]
    dW = torch.empty((K, N), dtype=torch.float32, device=X.device)
    carbon_gemm_dw_f32(dW, X, dY, M, K, N, tier, stream)
    return dW
