"""Seeded synthetic inputs for the deterministic linear-layer GEMM.

This module only draws and encodes random operands.  It holds none of the
method's arithmetic (no products, no sums, no output rounding) and imports
neither the CUDA binding nor the oracle, so both sides of every parity test
can take their inputs from here.

Workloads (shapes follow the Carbon README, "The Proof" section, and the
sgemm-bi page, "Use" section; the pages' own training runs need code,
weights and data that are not available, so these synthetic operands of the
same shapes stand in for them):

* ``single``   - one fp32 forward GEMM, M=64, K=128, N=96; X, W ~ U(-1, 1),
                 bias ~ U(-0.1, 0.1).
* ``toy_mlp``  - the three linear layers of a ~500K-parameter MLP (Carbon
                 README, "Toy Model (500K params ...)"), fp32, M=512 tokens,
                 (K, N) in {(256,512), (512,512), (512,256)}; X ~ N(0,1),
                 W ~ N(0, 0.02), bias ~ N(0, 0.02), dY ~ N(0, 1e-3).
* ``gpt2``     - GPT-2-124M linear shapes (Carbon README, "GPT-2 124M
                 Fine-Tune"), bf16, M = 8 x 1024 = 8192 tokens, (K, N) in
                 {(768,2304), (768,768), (768,3072), (3072,768)}; X ~ N(0,1),
                 W ~ N(0, 0.02), bias ~ N(0, 0.02), dY ~ N(0, 1e-4).
* ``stress``   - a dW GEMM over 65536 tokens with K=768, N=3072 in fp32 whose
                 entries are +-2^e (e uniform in [-20, 20], random sign) and
                 whose second half of token rows are exact negated duplicates
                 (in X) of the first half, rows shuffled jointly.

The second parameter of N(mu, sigma) is the standard deviation.  Normal
draws are made in float64 and rounded to nearest-even into fp32; bf16 operands
are rounded to nearest-even from that fp32 value (fp16 operands likewise, to
IEEE binary16).  bf16 and fp16 tensors are carried as ``numpy.uint16`` bit
patterns.

Seeds 42, 123, 7, 999 and 2024 are the five seeds of the Carbon README's
"Toy Model" table.
"""
from __future__ import annotations

import numpy as np

SEEDS = (42, 123, 7, 999, 2024)

TOY_MLP_LAYERS = ((256, 512), (512, 512), (512, 256))
GPT2_LAYERS = ((768, 2304), (768, 768), (768, 3072), (3072, 768))
GPT2_TOKENS = 8 * 1024
TOY_TOKENS = 512


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even) and return the bits.

    NaNs become the canonical quiet NaN.  This is the input encoding step of
    the data recipe, not part of the GEMM.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        r = r.copy()
        r[nan] = np.uint16(0x7FC0)
    return r


def f32_to_f16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to IEEE binary16 (nearest, ties to even; numpy's
    conversion) and return the bits.  Values beyond 65504 become infinities.
    This is the input encoding step of the data recipe, not part of the GEMM."""
    return np.ascontiguousarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def f16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen binary16 bit patterns to fp32 values (exact)."""
    return np.ascontiguousarray(b, dtype=np.uint16).view(np.float16).astype(np.float32)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 values (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_f32(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    return (rng.standard_normal(size=shape) * std).astype(np.float32)


def _uniform_f32(rng: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    return rng.uniform(lo, hi, size=shape).astype(np.float32)


def _encode(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(a, dtype=np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(a)
    if dtype == "f16":
        return f32_to_f16_bits(a)
    raise ValueError(f"unknown dtype {dtype!r}")


def single_gemm(seed: int = 42, M: int = 64, K: int = 128, N: int = 96) -> dict:
    """One fp32 forward GEMM: X, W ~ U(-1,1), bias ~ U(-0.1,0.1)."""
    rng = np.random.default_rng(seed)
    X = _uniform_f32(rng, (M, K), -1.0, 1.0)
    W = _uniform_f32(rng, (K, N), -1.0, 1.0)
    b = _uniform_f32(rng, (N,), -0.1, 0.1)
    return {"dtype": "f32", "M": M, "K": K, "N": N, "X": X, "W": W, "b": b}


def linear_layer(rng: np.random.Generator, M: int, K: int, N: int, dtype: str,
                 dy_std: float) -> dict:
    """One linear layer's operands, drawn in the order X, W, b, dY."""
    X = _normal_f32(rng, (M, K), 1.0)
    W = _normal_f32(rng, (K, N), 0.02)
    b = _normal_f32(rng, (N,), 0.02)
    dY = _normal_f32(rng, (M, N), dy_std)
    return {"dtype": dtype, "M": M, "K": K, "N": N,
            "X": _encode(X, dtype), "W": _encode(W, dtype),
            "b": _encode(b, dtype), "dY": _encode(dY, dtype)}


def toy_mlp(seed: int = 42, M: int = TOY_TOKENS, layers=TOY_MLP_LAYERS) -> list:
    """fp32 operands for the toy MLP's linear layers (fwd, dX and dW)."""
    rng = np.random.default_rng(seed)
    return [linear_layer(rng, M, K, N, "f32", 1e-3) for (K, N) in layers]


def gpt2(seed: int = 42, M: int = GPT2_TOKENS, layers=GPT2_LAYERS) -> list:
    """bf16 operands for the GPT-2-124M-shaped linear layers."""
    rng = np.random.default_rng(seed)
    return [linear_layer(rng, M, K, N, "bf16", 1e-4) for (K, N) in layers]


def toy_param_count(layers=TOY_MLP_LAYERS) -> int:
    """Weights of the toy MLP's linear layers (K*N summed)."""
    return int(sum(K * N for (K, N) in layers))


def stress_dw(seed: int = 42, M: int = 65536, K: int = 768, N: int = 3072,
              emin: int = -20, emax: int = 20) -> dict:
    """Cancellation stress operands for one fp32 dW GEMM (reduction over M).

    Entries are sign * 2**e with e uniform in [emin, emax].  Rows M/2..M-1 are
    copies of rows 0..M/2-1 taken in a random order: the X copy is negated, the
    dY copy is not, so every exact dW entry is zero.  One joint permutation of
    the token rows is applied at the end.
    """
    if M % 2:
        raise ValueError("M must be even")
    rng = np.random.default_rng(seed)
    half = M // 2

    def pm_pow2(shape):
        e = rng.integers(emin, emax + 1, size=shape, dtype=np.int32)
        s = rng.integers(0, 2, size=shape, dtype=np.int32) * 2 - 1
        return (np.ldexp(np.float32(1.0), e) * s).astype(np.float32)

    X = np.empty((M, K), dtype=np.float32)
    dY = np.empty((M, N), dtype=np.float32)
    X[:half] = pm_pow2((half, K))
    dY[:half] = pm_pow2((half, N))
    src = rng.permutation(half)
    X[half:] = -X[src]
    dY[half:] = dY[src]
    perm = rng.permutation(M)
    X = np.ascontiguousarray(X[perm])
    dY = np.ascontiguousarray(dY[perm])
    return {"dtype": "f32", "M": M, "K": K, "N": N, "X": X, "dY": dY}


def sample_indices(seed: int, rows: int, cols: int, count: int,
                   corners: bool = True) -> tuple:
    """Pick output coordinates to compare at full size.

    Returns (row_idx, col_idx) int64 arrays: the four corners and the last
    row/column (ragged tiles) plus ``count`` uniform draws.
    """
    rng = np.random.default_rng(seed ^ 0x5EED)
    r = rng.integers(0, rows, size=count, dtype=np.int64)
    c = rng.integers(0, cols, size=count, dtype=np.int64)
    if corners:
        er = np.array([0, 0, rows - 1, rows - 1, rows // 2], dtype=np.int64)
        ec = np.array([0, cols - 1, 0, cols - 1, cols // 2], dtype=np.int64)
        r = np.concatenate([er, r])
        c = np.concatenate([ec, c])
    return r, c
