"""Data-parallel weight gradient, bit-identical to a single device (exact tier).

The Carbon README ("How It Works") replaces the all-reduce of gradients
across data-parallel ranks with an all-gather followed by a reduction in rank
order, and its "Roadmap" lists a deterministic multi-GPU all-reduce.  With
the exact tier's fixed summation order the reduction over tokens can be
split so that the result does not depend on the number of ranks at all:

* the M tokens are split into contiguous ranges whose boundaries are
  multiples of 256 (``token_ranges``), so every 256-token chunk of the
  single-device reduction belongs to exactly one rank;
* each rank computes the chunk values fl(s + c) of its own chunks
  (``carbon_gemm_chunk_values``): the same doubles the single-device call
  forms for those chunks;
* the chunk values are all-gathered in rank order, which is chunk order;
* every rank runs the outer KBN over all chunk values, left to right, and the
  one rounding (``carbon_chunk_values_combine``).

The combined dW is then bit-identical to ``carbon_gemm_dw`` over all M tokens
on one device, on every rank.  The gathered volume is 8 bytes per output per
chunk (for GPT-2's 768 x 3072 weight over 8192 tokens, 32 chunks: 604 MB).

The collective runs on the process group's backend: device tensors for NCCL,
host copies for gloo.
"""
from __future__ import annotations

import torch

from . import _binding, _dtype_code

CHUNK = 256


def token_ranges(M: int, world: int):
    """[(m_0, m_1), (m_1, m_2), ...] for ranks 0 .. world-1: contiguous, in rank
    order, covering [0, M), every boundary a multiple of 256 except M itself;
    the ranks get the 256-token chunks as evenly as possible (a rank may get
    none when there are fewer chunks than ranks)."""
    if M < 0 or world < 1:
        raise ValueError("need M >= 0 and world >= 1")
    nq = (M + CHUNK - 1) // CHUNK
    bounds = [min(M, CHUNK * (nq * r // world)) for r in range(world + 1)]
    return [(bounds[r], bounds[r + 1]) for r in range(world)]


def chunk_values(X, dY, stream=None):
    """Chunk values of dW = X^T.dY over this rank's tokens: float64
    [ceil(m / 256), K, N] on X's device (X [m, K], dY [m, N], same dtype)."""
    if X.dim() != 2 or dY.dim() != 2 or X.shape[0] != dY.shape[0]:
        raise ValueError("X [m, K] and dY [m, N] must share their token count")
    if not (X.is_cuda and dY.is_cuda and X.is_contiguous() and dY.is_contiguous()):
        raise ValueError("X and dY must be contiguous CUDA tensors")
    m, K = X.shape
    N = dY.shape[1]
    P = torch.empty(((m + CHUNK - 1) // CHUNK, K, N), dtype=torch.float64, device=X.device)
    if m > 0:
        _binding.carbon_gemm_chunk_values("dw", P, X, dY, m, K, N, _dtype_code(X), stream)
    return P


def combine(P, dtype: str, bias=None, stream=None):
    """RNE(outer KBN over P[0], P[1], ... in order (+ bias)) in `dtype`
    ("f32", "bf16" or "f16"): [rows, cols] on P's device."""
    nq, rows, cols = P.shape
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    out = torch.empty((rows, cols), dtype=tdt, device=P.device)
    _binding.carbon_chunk_values_combine(out, P.contiguous(), nq, rows, cols, bias, dtype, stream)
    return out


def gather_in_rank_order(P_local, counts, group=None):
    """All-gather every rank's chunk values and concatenate them in rank order.
    counts[r] = chunks of rank r.  Tensors travel as device tensors on NCCL and
    as host copies on other backends; the result is on P_local's device."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    if len(counts) != world:
        raise ValueError("one chunk count per rank")
    _, rows, cols = P_local.shape
    cmax = max(counts) if counts else 0
    on_device = dist.get_backend(group) == "nccl"
    send = P_local if on_device else P_local.cpu()
    if send.shape[0] < cmax:                           # equal shapes for the collective
        pad = torch.zeros((cmax - send.shape[0], rows, cols), dtype=send.dtype, device=send.device)
        send = torch.cat([send, pad])
    recv = [torch.empty_like(send) for _ in range(world)]
    dist.all_gather(recv, send.contiguous(), group=group)
    full = torch.cat([recv[r][:counts[r]] for r in range(world)])
    return full.to(P_local.device)


def linear_dw_data_parallel(X_local, dY_local, M: int, group=None, stream=None,
                            chunk_values_fn=chunk_values, combine_fn=combine):
    """dW[K, N] = X^T.dY over all M tokens, with this rank holding the tokens
    ``token_ranges(M, world)[rank]`` of X and dY; bit-identical to the
    single-device exact-tier ``carbon_gemm_dw`` on every rank.
    (``chunk_values_fn`` and ``combine_fn`` exist so that the orchestration can
    be exercised on CPU ranks.)"""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    ranges = token_ranges(M, world)
    lo, hi = ranges[rank]
    if X_local.shape[0] != hi - lo or dY_local.shape[0] != hi - lo:
        raise ValueError(f"rank {rank} must hold tokens [{lo}, {hi}) of {M}")
    P_local = chunk_values_fn(X_local, dY_local, stream)
    counts = [(b - a + CHUNK - 1) // CHUNK for a, b in ranges]
    P = gather_in_rank_order(P_local, counts, group)
    return combine_fn(P, _dtype_code(X_local), None, stream)
