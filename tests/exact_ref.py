"""Exact rational arithmetic used to pin the oracle (tests only).

Nothing here follows the oracle's algorithm.  The exact result of a matrix
product is taken with Python's unbounded rationals and numpy's object-array
matmul (the mathematical definition, no rounding anywhere); rounding to fp32,
bf16 or fp16 is done from the definition of round-to-nearest-even on the
exact rational value.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

U = Fraction(1, 2 ** 53)          # unit roundoff of binary64

FORMATS = {
    # significand bits (incl. hidden), min normal exponent, max exponent
    "f32": (24, -126, 127),
    "bf16": (8, -126, 127),
    "f16": (11, -14, 15),
}


def to_fractions(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact rational values of fp32 arrays or bf16 / fp16 bit arrays."""
    if dtype == "f16":
        a = np.asarray(a, dtype=np.uint16).view(np.float16).astype(np.float64)
        flat = [Fraction(float(v)) for v in a.ravel()]
        out = np.empty(len(flat), dtype=object)
        out[:] = flat
        return out.reshape(np.shape(a))
    if dtype == "bf16":
        a = (np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    flat = [Fraction(float(v)) for v in np.asarray(a, dtype=np.float32).ravel()]
    out = np.empty(len(flat), dtype=object)
    out[:] = flat
    return out.reshape(np.shape(a))


def exact_product(pass_: str, A, B, dtype: str) -> np.ndarray:
    """Exact Y = A.B (fwd), dY.W^T (dX) or X^T.dY (dW) as Fractions."""
    a = to_fractions(A, dtype)
    b = to_fractions(B, dtype)
    if pass_ == "fwd":
        return a @ b
    if pass_ == "dx":
        return a @ b.T
    if pass_ == "dw":
        return a.T @ b
    raise ValueError(pass_)


def term_matrices(pass_: str, A, B, dtype: str):
    """For each output, the exact products in reduction order (list of lists).

    Returns an object array of shape out x R holding Fractions.
    """
    a = to_fractions(A, dtype)
    b = to_fractions(B, dtype)
    if pass_ == "fwd":
        return a[:, None, :] * b.T[None, :, :]
    if pass_ == "dx":
        return a[:, None, :] * b[None, :, :]
    return a.T[:, None, :] * b.T[None, :, :]


def kbn_bound(terms, chunk: int = 256) -> Fraction:
    """Error bound for the two-level fixed-order KBN sum of ``terms``.

    Neumaier's bound for n terms (Higham, Accuracy and Stability of Numerical
    Algorithms, 2nd ed., section 4.3) is |S_hat - S| <= 2u|S| + O(n^2 u^2)
    * sum|x|.  It is applied to every chunk (n <= chunk) and then to the
    outer sum of the chunk values; constants are taken generously.
    """
    terms = list(terms)
    n = len(terms)
    if n == 0:
        return Fraction(0)
    total = sum(terms, Fraction(0))
    abs_all = sum((abs(t) for t in terms), Fraction(0))
    nchunks = (n + chunk - 1) // chunk
    chunk_abs_exact = Fraction(0)
    for q in range(nchunks):
        chunk_abs_exact += abs(sum(terms[q * chunk:(q + 1) * chunk], Fraction(0)))
    return (3 * U * (abs(total) + chunk_abs_exact)
            + 8 * (chunk ** 2 + nchunks ** 2) * U * U * abs_all)


def floor_log2(q: Fraction) -> int:
    """floor(log2(q)) for q > 0, exactly."""
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    elif Fraction(2) ** (e + 1) <= q:
        e += 1
    return e


def rne(q: Fraction, fmt: str):
    """Round an exact rational to the nearest value of ``fmt`` (ties to even).

    Returns a Fraction, or +-inf (as a float) on overflow.
    """
    p, emin, emax = FORMATS[fmt]
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = max(floor_log2(a), emin)
    quantum = Fraction(2) ** (e - (p - 1))
    scaled = a / quantum
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = n * quantum
    largest = (2 - Fraction(2) ** (1 - p)) * Fraction(2) ** emax
    if r > largest:
        return sign * float("inf")
    return sign * r


def near_midpoint(q: Fraction, fmt: str, tol: Fraction) -> bool:
    """True if q lies within tol of a rounding midpoint of ``fmt``."""
    p, emin, _ = FORMATS[fmt]
    a = abs(q)
    exps = {emin} if a - tol <= 0 else set()
    for cand in (a - tol, a, a + tol):
        if cand > 0:
            exps.add(max(floor_log2(cand), emin))
    for e in exps:
        quantum = Fraction(2) ** (e - (p - 1))
        k = (a / quantum).numerator // (a / quantum).denominator
        for kk in (k - 1, k, k + 1):
            if abs((kk + Fraction(1, 2)) * quantum - a) <= tol:
                return True
    return False


def value_bits(v, fmt: str) -> int:
    """Bit pattern of a value (Fraction or +-inf) that is exact in ``fmt``."""
    if fmt == "f16":
        return int(np.array([float(v)], dtype=np.float16).view(np.uint16)[0])
    f = np.float32(float(v))
    u = int(np.array([f], dtype=np.float32).view(np.uint32)[0])
    return u if fmt == "f32" else (u >> 16)
