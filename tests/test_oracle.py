"""Pins for the CPU oracle (no GPU).

Each test ties the oracle to something other than its own code:
closed forms derived by hand (tests/golden/closed_form.json), exact rational
sums within the KBN error bound, exact round-to-nearest-even from the
definition, and invariants of the matrix products (row/column permutation,
independence of the batch size, the transposition identities between the
three passes).
"""
import json
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
import seeded_inputs as inputs
from tests import exact_ref as ex

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form.json")


def _enc(values, dtype):
    a = np.array(values, dtype=np.float64).astype(np.float32)
    if dtype == "f16":
        return inputs.f32_to_f16_bits(a)
    return a if dtype == "f32" else inputs.f32_to_bf16_bits(a)


def _as_f64(out, dtype):
    if dtype == "f32":
        return out.astype(np.float64)
    if dtype == "f16":
        return inputs.f16_bits_to_f32(out).astype(np.float64)
    return inputs.bf16_bits_to_f32(out).astype(np.float64)


def _case_operands(case, pass_, dtype):
    R = case["K"]
    x = [0.0] * R
    w = [1.0] * R
    for k, v in case["x"].items():
        x[int(k)] = float.fromhex(v)
    for k, v in case["w"].items():
        w[int(k)] = float.fromhex(v)
    xa, wa = _enc(x, dtype), _enc(w, dtype)
    bias = _enc([float.fromhex(case["bias"])], dtype) if "bias" in case else None
    if pass_ == "fwd":
        return xa.reshape(1, R), wa.reshape(R, 1), bias, (1, R, 1)
    if pass_ == "dx":
        return xa.reshape(1, R), wa.reshape(1, R), None, (1, 1, R)
    return xa.reshape(R, 1), wa.reshape(R, 1), None, (R, 1, 1)


def _golden_params():
    cases = json.load(open(GOLDEN))["cases"]
    for case in cases:
        for dtype in case["dtypes"]:
            for pass_ in case.get("passes", ["fwd", "dx", "dw"]):
                yield pytest.param(case, dtype, pass_, id=f"{case['name']}-{dtype}-{pass_}")


@pytest.mark.parametrize("case,dtype,pass_", list(_golden_params()))
def test_closed_form(case, dtype, pass_):
    A, B, bias, (M, K, N) = _case_operands(case, pass_, dtype)
    out, y64 = oracle.gemm(pass_, dtype, A, B, bias, M, K, N)
    expect = float.fromhex(case["expect"])
    got = float(_as_f64(out, dtype).ravel()[0])
    assert got == expect, (got, expect)
    if "expect_sign_bit" in case:
        assert np.signbit(got) == bool(case["expect_sign_bit"])
        assert np.signbit(y64.ravel()[0]) == bool(case["expect_sign_bit"])


def test_chunk_width_is_256():
    assert oracle.chunk_width() == 256


# --------------------------------------------------------------------------
# Exact rationals: y64 within the KBN bound of the exact sum, and the output
# equal to RNE(exact) unless the exact value sits within that bound of a
# rounding midpoint.

SMALL_SHAPES = [
    # (M, K, N): reduction lengths that cross 0, 1, 2 chunk boundaries
    (3, 1, 4), (2, 255, 3), (3, 256, 2), (2, 257, 3), (2, 513, 2), (1, 600, 1),
]


def _random_operands(rng, pass_, M, K, N, dtype, scale_a=1.0, scale_b=0.02):
    def draw(shape, s):
        return (rng.standard_normal(size=shape) * s).astype(np.float32)
    if pass_ == "fwd":
        A, B = draw((M, K), scale_a), draw((K, N), scale_b)
    elif pass_ == "dx":
        A, B = draw((M, N), scale_a), draw((K, N), scale_b)
    else:
        A, B = draw((M, K), scale_a), draw((M, N), scale_b)
    bias = draw((N,), scale_b) if pass_ == "fwd" else None
    if dtype == "bf16":
        A, B = inputs.f32_to_bf16_bits(A), inputs.f32_to_bf16_bits(B)
        bias = None if bias is None else inputs.f32_to_bf16_bits(bias)
    if dtype == "f16":
        A, B = inputs.f32_to_f16_bits(A), inputs.f32_to_f16_bits(B)
        bias = None if bias is None else inputs.f32_to_f16_bits(bias)
    return A, B, bias


@pytest.mark.parametrize("seed", inputs.SEEDS)
@pytest.mark.parametrize("pass_", ["fwd", "dx", "dw"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_exact_rational(seed, pass_, dtype):
    rng = np.random.default_rng(seed)
    shapes = SMALL_SHAPES[seed % 3::2] if pass_ != "fwd" else SMALL_SHAPES
    for (M, K, N) in shapes:
        A, B, bias = _random_operands(rng, pass_, M, K, N, dtype)
        out, y64 = oracle.gemm(pass_, dtype, A, B, bias, M, K, N)
        exact = ex.exact_product(pass_, A, B, dtype)
        terms = ex.term_matrices(pass_, A, B, dtype)
        bvals = ex.to_fractions(bias, dtype) if bias is not None else None
        outv = _as_f64(out, dtype)
        for idx in np.ndindex(exact.shape):
            e = exact[idx]
            bound = ex.kbn_bound(terms[idx])
            if bvals is not None:
                e = e + bvals[idx[1]]
                bound = bound + 2 * ex.U * (abs(e) + bound)   # the bias addition
            err = abs(Fraction(float(y64[idx])) - e)
            assert err <= bound, (pass_, M, K, N, idx, float(err), float(bound))
            if not ex.near_midpoint(e, dtype, bound):
                assert Fraction(float(outv[idx])) == ex.rne(e, dtype), (idx, float(e))


def test_kbn_beats_plain_sum_on_ill_conditioned_rows():
    """Sums with heavy cancellation: KBN stays within its bound of the exact
    value, while a plain float64 left-to-right sum of the same products does
    not (shows the compensation term is in use, not just the plain sum)."""
    rng = np.random.default_rng(7)
    big = np.ldexp(1.0, rng.integers(0, 31, size=90)) * rng.choice([-1.0, 1.0], size=90)
    small = np.ldexp(1.0, rng.integers(-30, -19, size=20)) * rng.choice([-1.0, 1.0], size=20)
    x = rng.permutation(np.concatenate([big, -big, small])).astype(np.float32)
    K = x.size                  # one chunk; big terms cancel in pairs
    w = np.ones(K, dtype=np.float32)
    out, y64 = oracle.gemm("fwd", "f32", x.reshape(1, K), w.reshape(K, 1), None, 1, K, 1)
    exact = sum((Fraction(float(v)) for v in x), Fraction(0))
    terms = [Fraction(float(v)) for v in x]
    plain = 0.0
    for v in x:
        plain += float(v)
    assert abs(Fraction(float(y64[0, 0])) - exact) <= ex.kbn_bound(terms)
    assert abs(Fraction(plain) - exact) > ex.kbn_bound(terms)


# --------------------------------------------------------------------------
# Output rounding against RNE from the definition.

def _f64_bits_to_float(u):
    return struct.unpack("<d", struct.pack("<Q", int(u)))[0]


def _rounding_corpus(rng, n=20000):
    vals = list(rng.standard_normal(n) * np.ldexp(1.0, rng.integers(-140, 130, n)))
    # midpoints and their neighbours, for fp32 (24 bits) and bf16 (8 bits)
    for p in (24, 8):
        for e in (-130, -127, -126, -100, -1, 0, 1, 50, 126, 127):
            for k in (0, 1, 2, 3, 2 ** (p - 1) - 1, 2 ** p - 1):
                mid = (2 ** (p - 1) + k + 0.5) * 2.0 ** (e - (p - 1))
                for d in (0.0, 1.0, -1.0):
                    v = np.nextafter(mid, np.inf) if d > 0 else (
                        np.nextafter(mid, -np.inf) if d < 0 else mid)
                    vals += [v, -v]
    # overflow boundary: largest finite, the midpoint above it, 2^128
    for p in (24, 8):
        largest = (2 - 2.0 ** (1 - p)) * 2.0 ** 127
        mid = largest + 2.0 ** (127 - p)
        vals += [largest, mid, np.nextafter(mid, 0), np.nextafter(mid, np.inf), 2.0 ** 128]
    # subnormal bf16/fp32 region and zeros
    vals += [2.0 ** -133, 1.5 * 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135, 2.0 ** -149,
             2.0 ** -150, 1.5 * 2.0 ** -149, 0.0, -0.0, 5e-324]
    # binary16: midpoints across its exponent range, the overflow boundary
    # (65504, the midpoint 65520 above it) and the subnormal region (quantum 2^-24)
    vals += list(rng.standard_normal(n // 4) * np.ldexp(1.0, rng.integers(-30, 18, n // 4)))
    for e in (-16, -15, -14, -13, -1, 0, 1, 10, 14, 15):
        for k in (0, 1, 2, 3, 1023, 2047 - 1024):
            mid = (1024 + k + 0.5) * 2.0 ** (e - 10)
            for d in (0.0, 1.0, -1.0):
                v = np.nextafter(mid, np.inf) if d > 0 else (
                    np.nextafter(mid, -np.inf) if d < 0 else mid)
                vals += [v, -v]
    vals += [65504.0, 65519.99, 65520.0, np.nextafter(65520.0, 0), 65536.0, 1e6,
             2.0 ** -24, 2.0 ** -25, np.nextafter(2.0 ** -25, 1), 3 * 2.0 ** -26, 2.0 ** -26,
             1.5 * 2.0 ** -24, 2.5 * 2.0 ** -24, 1023.5 * 2.0 ** -24, 2.0 ** -14]
    return np.array(vals, dtype=np.float64)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_output_rounding_is_rne(dtype):
    y = _rounding_corpus(np.random.default_rng(2024))
    got = oracle.round_out(dtype, y)
    if dtype == "f32":
        got = got.view(np.uint32)
    inf_bits = {"f32": 0x7F800000, "bf16": 0x7F80, "f16": 0x7C00}[dtype]
    sign_bit = 0x80000000 if dtype == "f32" else 0x8000
    for v, g in zip(y, got):
        r = ex.rne(Fraction(float(v)), dtype)
        if isinstance(r, float):                      # overflow
            want = inf_bits | (sign_bit if v < 0 else 0)
        else:
            want = ex.value_bits(r, dtype)
            if r == 0 and np.signbit(v):
                want |= sign_bit
        assert int(g) == want, (v.hex(), hex(int(g)), hex(want))


def test_rounding_special_values():
    y = np.array([np.inf, -np.inf, np.nan], dtype=np.float64)
    b = oracle.round_out("bf16", y)
    assert list(b[:2]) == [0x7F80, 0xFF80]
    assert (int(b[2]) & 0x7F80) == 0x7F80 and (int(b[2]) & 0x7F) != 0
    h = oracle.round_out("f16", y)
    assert list(h[:2]) == [0x7C00, 0xFC00]
    assert (int(h[2]) & 0x7C00) == 0x7C00 and (int(h[2]) & 0x3FF) != 0


def test_f16_decoding_is_exact():
    """Every binary16 bit pattern decodes to its value: the oracle's sums of
    one product x * 1 return x itself, for all finite patterns."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = bits[(bits & 0x7C00) != 0x7C00]
    K = finite.size
    one = inputs.f32_to_f16_bits(np.ones((1, 1), dtype=np.float32))
    _, y = oracle.gemm("fwd", "f16", finite.reshape(K, 1), one, None, K, 1, 1)
    want = finite.view(np.float16).astype(np.float64)
    assert np.array_equal(y.reshape(K), want)


# --------------------------------------------------------------------------
# Invariants of the matrix products (bit-identical).

def test_row_permutation_and_batch_independence():
    d = inputs.single_gemm(42)
    X, W, b = d["X"], d["W"], d["b"]
    M, K, N = d["M"], d["K"], d["N"]
    Y, _ = oracle.gemm("fwd", "f32", X, W, b, M, K, N)
    perm = np.random.default_rng(1).permutation(M)
    Yp, _ = oracle.gemm("fwd", "f32", X[perm], W, b, M, K, N)
    assert np.array_equal(Yp.view(np.uint32), Y[perm].view(np.uint32))
    for m in (1, 7, 8):
        Ym, _ = oracle.gemm("fwd", "f32", X[:m], W, b, m, K, N)
        assert np.array_equal(Ym.view(np.uint32), Y[:m].view(np.uint32))


def test_column_permutation():
    d = inputs.single_gemm(123)
    X, W, b = d["X"], d["W"], d["b"]
    M, K, N = d["M"], d["K"], d["N"]
    Y, _ = oracle.gemm("fwd", "f32", X, W, b, M, K, N)
    perm = np.random.default_rng(2).permutation(N)
    Yp, _ = oracle.gemm("fwd", "f32", X, np.ascontiguousarray(W[:, perm]), b[perm], M, K, N)
    assert np.array_equal(Yp.view(np.uint32), Y[:, perm].view(np.uint32))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_pass_transposition_identities(dtype):
    rng = np.random.default_rng(999)
    M, K, N = 37, 300, 29       # R spans two chunks for fwd/dX; dW R=37
    layer = inputs.linear_layer(rng, M, K, N, dtype, 1e-3)
    X, W, dY = layer["X"], layer["W"], layer["dY"]
    # dX(dY, W) == fwd(dY, W^T) with no bias
    dX, _ = oracle.gemm("dx", dtype, dY, W, None, M, K, N)
    ref, _ = oracle.gemm("fwd", dtype, dY, np.ascontiguousarray(W.T), None, M, N, K)
    assert np.array_equal(dX.view(np.uint8), ref.view(np.uint8))
    # dW(X, dY) == fwd(X^T, dY) with no bias
    dW, _ = oracle.gemm("dw", dtype, X, dY, None, M, K, N)
    ref, _ = oracle.gemm("fwd", dtype, np.ascontiguousarray(X.T), dY, None, K, M, N)
    assert np.array_equal(dW.view(np.uint8), ref.view(np.uint8))


def test_sampled_matches_dense():
    rng = np.random.default_rng(5)
    M, K, N = 20, 513, 17
    layer = inputs.linear_layer(rng, M, K, N, "bf16", 1e-4)
    for pass_, A, B, bias in (("fwd", layer["X"], layer["W"], layer["b"]),
                              ("dx", layer["dY"], layer["W"], None),
                              ("dw", layer["X"], layer["dY"], None)):
        dense, y64 = oracle.gemm(pass_, "bf16", A, B, bias, M, K, N)
        R, C = dense.shape
        rows, cols = inputs.sample_indices(3, R, C, 50)
        s_out, s_y = oracle.gemm_at(pass_, "bf16", A, B, bias, M, K, N, rows, cols)
        assert np.array_equal(s_out, dense[rows, cols])
        assert np.array_equal(s_y.view(np.uint64), y64[rows, cols].view(np.uint64))


def test_thread_count_does_not_change_bits():
    layer = inputs.toy_mlp(42, M=64)[1]
    a, _ = oracle.gemm("dw", "f32", layer["X"], layer["dY"], None, 64, 512, 512, threads=1)
    b, _ = oracle.gemm("dw", "f32", layer["X"], layer["dY"], None, 64, 512, 512, threads=5)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


# --------------------------------------------------------------------------
# Workload facts.

def test_toy_mlp_has_about_500k_parameters():
    # Carbon README, "Toy Model (500K params ...)"
    assert inputs.toy_param_count() == 524288


def test_stress_rows_cancel_exactly_and_oracle_is_within_bound():
    d = inputs.stress_dw(2024, M=2048, K=6, N=5)
    X, dY = d["X"], d["dY"]
    # every product is +-2^e with |e| <= 40: scaled by 2^40 it is an integer
    xi = np.rint(np.ldexp(X.astype(np.float64), 20)).astype(np.int64)
    yi = np.rint(np.ldexp(dY.astype(np.float64), 20)).astype(np.int64)
    exact = xi.T.astype(object) @ yi.astype(object)
    assert all(v == 0 for v in exact.ravel())
    out, y64 = oracle.gemm("dw", "f32", X, dY, None, d["M"], d["K"], d["N"])
    terms = ex.term_matrices("dw", X, dY, "f32")
    for idx in np.ndindex(y64.shape):
        assert abs(Fraction(float(y64[idx]))) <= ex.kbn_bound(terms[idx])


# --------------------------------------------------------------------------
# The pins fail on plausible mistakes.  Each mutant is a copy of the oracle's
# source with one planted mistake, compiled on the CPU into a temporary
# folder; at least one closed form must reject it.

MUTANTS = {
    "inner_chunk_right_to_left": (
        "for (r = q0; r < q1; ++r) {",
        "for (r = q1 - 1; r >= q0; --r) {"),
    "chunks_right_to_left": (
        "for (q0 = 0; q0 < R; q0 += ORACLE_CHUNK) {",
        "for (q0 = R > 0 ? ((R - 1) / ORACLE_CHUNK) * ORACLE_CHUNK : -1; q0 >= 0;"
        " q0 -= ORACLE_CHUNK) {"),
    "chunk_width_128": ("#define ORACLE_CHUNK 256", "#define ORACLE_CHUNK 128"),
    "chunk_width_512": ("#define ORACLE_CHUNK 256", "#define ORACLE_CHUNK 512"),
    "no_compensation_in_chunk": (
        "kbn_step(&S, &C, s + c);", "kbn_step(&S, &C, s);"),
    "pair_passed_to_outer_level": (
        "kbn_step(&S, &C, s + c);", "kbn_step(&S, &C, s); kbn_step(&S, &C, c);"),
    "kbn_branch_swapped": (
        "if (fabs(*sum) >= fabs(x))", "if (fabs(*sum) < fabs(x))"),
    "output_rounded_before_bias": (
        "y = y + decode(jb->bias, jb->dtype, j);",
        "y = (double)(float)y + decode(jb->bias, jb->dtype, j);"),
    "bf16_rounded_through_fp32": (
        "round_to_f16_bits(y) : round_to_bf16_bits(y);",
        "round_to_f16_bits(y) : round_to_bf16_bits((double)(float)y);"),
    "bf16_ties_away_from_zero": (
        "n = nearbyint(a / quantum);         /* default mode: ties to even */\n    r = n * quantum;\n    if (r >= 0x1p128)",
        "n = round(a / quantum);\n    r = n * quantum;\n    if (r >= 0x1p128)"),
}


def _mutant_rejected(lib_path):
    import ctypes
    lib = ctypes.CDLL(lib_path)
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_gemm.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp,
                                i64, i64, i64, vp, vp, ctypes.c_int]
    lib.oracle_gemm.restype = ctypes.c_int
    failed = []
    for case, dtype, pass_ in (p.values for p in _golden_params()):
        A, B, bias, (M, K, N) = _case_operands(case, pass_, dtype)
        out = np.empty(oracle.out_shape(pass_, M, K, N),
                       dtype=np.float32 if dtype == "f32" else np.uint16)
        ptr = (lambda a: None if a is None else a.ctypes.data_as(vp))
        rc = lib.oracle_gemm(oracle.PASSES[pass_], oracle.DTYPES[dtype], ptr(A), ptr(B),
                             ptr(bias), M, K, N, ptr(out), None, 1)
        assert rc == 0
        if float(_as_f64(out, dtype).ravel()[0]) != float.fromhex(case["expect"]):
            failed.append(case["name"])
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name, tmp_path):
    import subprocess
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = str(tmp_path / f"lib{name}.so")
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", lib, str(path), "-lm"], check=True)
    assert _mutant_rejected(lib), f"no closed form rejects the mutant {name}"


# --------------------------------------------------------------------------
# The correctly rounded tier (superaccumulator; Carbon README, "Roadmap"):
# RNE of the exact dot product plus the bias.  Pinned to the closed forms'
# expect_superacc values and to exact rationals (no midpoint exception: the
# value is defined exactly).

@pytest.mark.parametrize("case,dtype,pass_", list(_golden_params()))
def test_superacc_closed_form(case, dtype, pass_):
    A, B, bias, (M, K, N) = _case_operands(case, pass_, dtype)
    out = oracle.gemm_superacc(pass_, dtype, A, B, bias, M, K, N)
    got = float(_as_f64(out, dtype).ravel()[0])
    expect = float.fromhex(case["expect_superacc"])
    assert got == expect, (got, expect)
    if expect == 0:
        assert not np.signbit(got)


def _superacc_want(exact, dtype):
    r = ex.rne(exact, dtype)
    if isinstance(r, float):            # overflow
        inf_bits = {"f32": 0x7F800000, "bf16": 0x7F80, "f16": 0x7C00}[dtype]
        return inf_bits | ((0x80000000 if dtype == "f32" else 0x8000) if r < 0 else 0)
    return ex.value_bits(r, dtype)


@pytest.mark.parametrize("seed", inputs.SEEDS)
@pytest.mark.parametrize("pass_", ["fwd", "dx", "dw"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_superacc_exact_rational(seed, pass_, dtype):
    rng = np.random.default_rng(seed + 77)
    shapes = SMALL_SHAPES[seed % 3::2] if pass_ != "fwd" else SMALL_SHAPES
    for (M, K, N) in shapes:
        A, B, bias = _random_operands(rng, pass_, M, K, N, dtype)
        out = oracle.gemm_superacc(pass_, dtype, A, B, bias, M, K, N)
        exact = ex.exact_product(pass_, A, B, dtype)
        bvals = ex.to_fractions(bias, dtype) if bias is not None else None
        got = out.view(np.uint32) if dtype == "f32" else out
        for idx in np.ndindex(exact.shape):
            e = exact[idx] + (bvals[idx[1]] if bvals is not None else 0)
            assert int(got[idx]) == _superacc_want(e, dtype), (pass_, M, K, N, idx)


def test_superacc_wide_range_and_cancellation():
    """Values spread over 2^+-60 with exact cancellation between them: the
    result is the exact sum rounded once, and the same for any order of the
    reduction index."""
    rng = np.random.default_rng(3)
    K = 700
    x = (rng.choice([-1.0, 1.0], K) * np.ldexp(1.0, rng.integers(-60, 61, K))).astype(np.float32)
    x[350:] = -x[:350][rng.permutation(350)]          # cancels the first half exactly...
    x[699] = np.float32(2.0 ** -70)                     # ...but for a tiny residue
    w = np.ones(K, dtype=np.float32)
    for perm in (np.arange(K), rng.permutation(K), np.arange(K)[::-1]):
        xa, wa = np.ascontiguousarray(x[perm]), np.ascontiguousarray(w[perm])
        out = oracle.gemm_superacc("fwd", "f32", xa.reshape(1, K), wa.reshape(K, 1), None, 1, K, 1)
        exact = sum((Fraction(float(v)) for v in x), Fraction(0))
        assert int(out.view(np.uint32)[0, 0]) == _superacc_want(exact, "f32")


def test_superacc_non_finite_and_overflow():
    big = np.float32(2.0 ** 127)
    cases = [  # (x, w, expected fp32 bits)
        ([big, big, -big], [big, big, big], 0x7F800000),          # exact 2^254: overflows to +inf
        ([np.inf, 1.0], [1.0, 1.0], 0x7F800000),                   # +inf
        ([np.inf, -np.inf], [1.0, 1.0], None),                     # NaN
        ([np.nan, 1.0], [1.0, 1.0], None),
        ([-big, -big], [big, big], 0xFF800000),                    # -inf
    ]
    for xv, wv, want in cases:
        K = len(xv)
        x = np.array(xv, dtype=np.float32).reshape(1, K)
        w = np.array(wv, dtype=np.float32).reshape(K, 1)
        got = int(oracle.gemm_superacc("fwd", "f32", x, w, None, 1, K, 1).view(np.uint32)[0, 0])
        if want is None:
            assert (got & 0x7F800000) == 0x7F800000 and (got & 0x7FFFFF) != 0
        else:
            assert got == want, hex(got)


SUPERACC_MUTANTS = {
    "no_sticky_bit": ("sticky = sa_bit(a, k);", "sticky = 0;"),
    "ties_away_from_zero": ("if (half && (sticky || (n & 1)))", "if (half)"),
    "bias_left_out": ("    if (bias)\n        sa_add(&acc, decode(bias, dtype, j));", "    (void)bias;"),
    "sign_of_negative_sums_lost": ("            neg = 1;\n", ""),
    "rounded_through_float64": (
        "        v = ldexp((double)n, q - SA_OFFSET);   /* exact; may reach the overflow bound */",
        "        { double hi = 0; for (k = 32 * SA_DIGITS - 1; k >= 0; --k) hi = 2 * hi + sa_bit(a, k);"
        " v = ldexp(hi, -SA_OFFSET); (void)n; }"),
}


def _superacc_mutant_rejected(lib_path):
    import ctypes
    lib = ctypes.CDLL(lib_path)
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_gemm_superacc.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp,
                                         i64, i64, i64, vp, vp, i64, vp, ctypes.c_int]
    failed = []
    ptr = (lambda a: None if a is None else a.ctypes.data_as(vp))
    for case, dtype, pass_ in (p.values for p in _golden_params()):
        A, B, bias, (M, K, N) = _case_operands(case, pass_, dtype)
        out = np.empty(oracle.out_shape(pass_, M, K, N),
                       dtype=np.float32 if dtype == "f32" else np.uint16)
        assert lib.oracle_gemm_superacc(oracle.PASSES[pass_], oracle.DTYPES[dtype], ptr(A),
                                        ptr(B), ptr(bias), M, K, N, None, None, 0, ptr(out), 1) == 0
        if float(_as_f64(out, dtype).ravel()[0]) != float.fromhex(case["expect_superacc"]):
            failed.append(case["name"])
    return failed


@pytest.mark.parametrize("name", sorted(SUPERACC_MUTANTS))
def test_superacc_pins_catch_planted_mistakes(name, tmp_path):
    import subprocess
    src = open(oracle._SRC).read()
    old, new = SUPERACC_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = str(tmp_path / f"lib{name}.so")
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", lib, str(path), "-lm"], check=True)
    assert _superacc_mutant_rejected(lib), f"no closed form rejects the mutant {name}"
