"""Autograd linear layer over the carbon_gemm C ABI.

A drop-in linear layer whose three GEMMs run in this library's kernels, as
the sgemm-bi page describes its ``Linear`` module and functional form
("Use": weights stored [in, out], ``Linear.from_torch`` converting a
``torch.nn.Linear``; the tensor-core switch there is the ``tier`` argument
here) and as the Carbon README describes its ``DeterministicLinear`` ("How
It Works").

    forward   Y  = X.W + b       carbon_gemm_fwd
    backward  dX = dY.W^T        carbon_gemm_dx
              dW = X^T.dY        carbon_gemm_dw
              db = sum_t dY[t]   carbon_gemm_dw with a column of ones for X,
                                 on the exact tier (on the correctly
                                 rounded tier when the layer uses it)

The bias gradient is the one piece the sgemm-bi page leaves to a plain
PyTorch column sum ("Determinism contracts"); here it is the exact tier's
fixed-order sum over tokens (256-token chunks summed with KBN, the chunk
values combined with KBN, one rounding), so it is bit-identical run to run,
for every batch split into the same tokens, and to the CPU oracle.  A layer
on the correctly rounded tier ("superacc") takes db from that tier too: the
exact column sum rounded once.

Leading dimensions of the input are flattened into the token dimension.
There is no CPU path: inputs must be CUDA tensors (float32, bfloat16 or
float16; the tensor-core tier takes bfloat16 or float16).
"""
from __future__ import annotations

import math

import torch

from . import _dtype_code, carbon_gemm_dw, linear_dw, linear_dx, linear_fwd


def bias_grad(dY, stream=None, tier="exact"):
    """db[N] = sum over tokens t of dY[t, :]: the GEMM dW = X^T.dY with X a
    column of ones (every product is exact), in dY's dtype, on the exact tier
    (fixed-order KBN) or, with tier="superacc", correctly rounded."""
    if tier not in ("exact", "superacc"):
        raise ValueError("the bias gradient runs on the exact or the superacc tier")
    if dY.dim() != 2 or not dY.is_contiguous() or not dY.is_cuda:
        raise ValueError("dY must be a contiguous 2-D CUDA tensor")
    M, N = dY.shape
    ones = torch.ones((M, 1), dtype=dY.dtype, device=dY.device)
    db = torch.empty((1, N), dtype=dY.dtype, device=dY.device)
    carbon_gemm_dw(db, ones, dY, M, 1, N, _dtype_code(dY), tier, stream)
    return db.view(N)


class _LinearFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight, bias, tier):
        K, N = weight.shape
        if x.shape[-1] != K:
            raise ValueError(f"input has {x.shape[-1]} features, weight expects {K}")
        x2 = x.reshape(-1, K).contiguous()
        y = linear_fwd(x2, weight, bias, tier)
        ctx.save_for_backward(x2, weight)
        ctx.tier = tier
        ctx.has_bias = bias is not None
        ctx.x_shape = x.shape
        return y.view(*x.shape[:-1], N)

    @staticmethod
    def backward(ctx, grad_y):
        x2, weight = ctx.saved_tensors
        g2 = grad_y.reshape(-1, weight.shape[1]).contiguous()
        dx = dw = db = None
        if ctx.needs_input_grad[0]:
            dx = linear_dx(g2, weight, ctx.tier).view(ctx.x_shape)
        if ctx.needs_input_grad[1]:
            dw = linear_dw(x2, g2, ctx.tier)
        if ctx.has_bias and ctx.needs_input_grad[2]:
            db = bias_grad(g2, tier="superacc" if ctx.tier == "superacc" else "exact")
        return dx, dw, db, None


def deterministic_linear(x, weight, bias=None, tier="exact"):
    """y = x.weight + bias with weight [in, out]; differentiable in x, weight
    and bias (the gradients come from the same library)."""
    return _LinearFunction.apply(x, weight, bias, tier)


class Linear(torch.nn.Module):
    """Linear layer with weight [in_features, out_features] and the library's
    kernels for the forward and backward GEMMs."""

    def __init__(self, in_features, out_features, bias=True, tier="exact", device=None,
                 dtype=None):
        super().__init__()
        self.in_features, self.out_features, self.tier = in_features, out_features, tier
        self.weight = torch.nn.Parameter(torch.empty((in_features, out_features), device=device,
                                                     dtype=dtype))
        self.bias = (torch.nn.Parameter(torch.empty(out_features, device=device, dtype=dtype))
                     if bias else None)
        self.reset_parameters()

    def reset_parameters(self):
        # torch.nn.Linear's initialisation, applied to the [out, in] view
        torch.nn.init.kaiming_uniform_(self.weight.t(), a=math.sqrt(5))
        if self.bias is not None:
            bound = 1.0 / math.sqrt(self.in_features) if self.in_features > 0 else 0.0
            torch.nn.init.uniform_(self.bias, -bound, bound)

    @classmethod
    def from_torch(cls, linear: torch.nn.Linear, tier="exact"):
        """The same layer with its weight stored [in, out] (a copy)."""
        out = cls(linear.in_features, linear.out_features, bias=linear.bias is not None,
                  tier=tier, device=linear.weight.device, dtype=linear.weight.dtype)
        with torch.no_grad():
            out.weight.copy_(linear.weight.t())
            if linear.bias is not None:
                out.bias.copy_(linear.bias)
        return out

    def forward(self, x):
        return deterministic_linear(x, self.weight, self.bias, self.tier)

    def extra_repr(self):
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"bias={self.bias is not None}, tier={self.tier!r}")
