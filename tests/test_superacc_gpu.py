"""The correctly rounded tier (CARBON_TIER_SUPERACC) on the GPU, through the
C ABI, against the oracle's superaccumulator.

The tier's result is the exact dot product plus the bias, rounded once to the
output type (Carbon README, "Roadmap": superaccumulators, exact summation
that needs no fixed order).  The bar is bit-identity with the oracle, on
every pass and dtype, on ragged shapes, and on operands built to drive each
path of the bf16 tensor-core kernel: chunk sums at or above 2^53 (which the
KBN tier would round and this tier must not), lines too wide for the digit
planes (chunk repair), running sums out of the 64-bit range and inf/NaN
operands (the warp-per-output superaccumulator), biases far from the output
grain.  No order of the reduction may show in the result: permuting the
reduction index leaves every output's bits unchanged.
"""
import json
import os

import numpy as np
import pytest

import oracle
import seeded_inputs as inputs
from tests.gpu_util import dev, host_bits, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import deterministic_invariant_gemm_fwd_gb300 as cg  # noqa: E402


def run(pass_, dtype, A, B, bias, M, K, N, tier="superacc"):
    shape = oracle.out_shape(pass_, M, K, N)
    f16 = dtype == "f16"
    tA, tB = dev(A, f16=f16), dev(B, f16=f16)
    tb = dev(bias, f16=f16) if bias is not None else None
    out = torch.empty(shape, dtype=torch_dtype(dtype), device="cuda")
    {"fwd": lambda: cg.carbon_gemm_fwd(out, tA, tB, tb, M, K, N, dtype, tier),
     "dx": lambda: cg.carbon_gemm_dx(out, tA, tB, M, K, N, dtype, tier),
     "dw": lambda: cg.carbon_gemm_dw(out, tA, tB, M, K, N, dtype, tier)}[pass_]()
    torch.cuda.synchronize()
    assert cg.carbon_get_device_status() == 0
    return host_bits(out)


def want_bits(pass_, dtype, A, B, bias, M, K, N):
    out = oracle.gemm_superacc(pass_, dtype, A, B, bias, M, K, N)
    return out.view(np.uint32) if dtype == "f32" else out


def check(pass_, dtype, A, B, bias, M, K, N):
    got = run(pass_, dtype, A, B, bias, M, K, N)
    want = want_bits(pass_, dtype, A, B, bias, M, K, N)
    assert np.array_equal(got, want), \
        f"{pass_} {dtype} {M}x{K}x{N}: {np.count_nonzero(got != want)} mismatches"
    return got


def bf16(a):
    return inputs.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def spread(rng, shape, lo, hi, sign=True):
    v = np.ldexp(1.0 + rng.integers(0, 128, shape) / 128.0, rng.integers(lo, hi + 1, shape))
    return v * rng.choice([-1.0, 1.0], shape) if sign else v


def operands(L, pass_):
    return {"fwd": (L["X"], L["W"], L["b"]), "dx": (L["dY"], L["W"], None),
            "dw": (L["X"], L["dY"], None)}[pass_]


GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form.json")


def test_closed_forms():
    from tests.test_oracle import _case_operands
    for case in json.load(open(GOLDEN))["cases"]:
        for dtype in case["dtypes"]:
            for pass_ in case.get("passes", ["fwd", "dx", "dw"]):
                A, B, bias, (M, K, N) = _case_operands(case, pass_, dtype)
                got = int(run(pass_, dtype, A, B, bias, M, K, N).ravel()[0])
                w = np.float32(float.fromhex(case["expect_superacc"])).view(np.uint32)
                w = int(w) >> 16 if dtype == "bf16" else int(w)
                assert got == w, (case["name"], dtype, pass_, hex(got), hex(w))


@pytest.mark.parametrize("pass_", ["fwd", "dx", "dw"])
def test_gpt2_shapes_reduced_batch(pass_):
    for L in inputs.gpt2(7, M=600):
        M, K, N = L["M"], L["K"], L["N"]
        check(pass_, "bf16", *operands(L, pass_), M, K, N)


EDGE = [(1, 1, 1), (7, 255, 3), (129, 256, 65), (1, 257, 65), (7, 513, 1),
        (3, 0, 5), (129, 1, 3), (33, 31, 33)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("M,K,N", EDGE)
def test_edge_shapes_all_passes(dtype, M, K, N):
    rng = np.random.default_rng(M * 1000 + K * 10 + N + 5)
    L = inputs.linear_layer(rng, M, K, N, dtype, 1e-3)
    for pass_ in ("fwd", "dx", "dw"):
        check(pass_, dtype, *operands(L, pass_), M, K, N)
    check("fwd", dtype, L["X"], L["W"], None, M, K, N)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_toy_mlp_all_passes(dtype):
    for L in inputs.toy_mlp(42, M=256):
        M, K, N = L["M"], L["K"], L["N"]
        if dtype == "f16":
            L = {k: (inputs.f32_to_f16_bits(v) if isinstance(v, np.ndarray) else v) for k, v in L.items()}
        for pass_ in ("fwd", "dx", "dw"):
            check(pass_, dtype, *operands(L, pass_), M, K, N)


def test_chunk_sums_above_2_53_are_not_rounded():
    """Same-sign operands of width ~30: chunk sums far above 2^53 grain units,
    which the KBN tier rounds to 53 bits and this tier keeps whole; each tier
    equals its own oracle (where the bf16 outputs of the two differ is rare:
    the closed forms hold a case that shows it)."""
    rng = np.random.default_rng(11)
    M, K, N = 140, 600, 70
    X = bf16(spread(rng, (M, K), -11, 11, sign=False))
    W = bf16(spread(rng, (K, N), -11, 11, sign=False))
    b = bf16(rng.standard_normal(N))
    check("fwd", "bf16", X, W, b, M, K, N)
    kbn = run("fwd", "bf16", X, W, b, M, K, N, tier="exact")
    assert np.array_equal(kbn, oracle.gemm("fwd", "bf16", X, W, b, M, K, N)[0])


@pytest.mark.parametrize("pass_", ["fwd", "dw"])
def test_wide_lines_chunk_repair(pass_):
    rng = np.random.default_rng(12)
    M, K, N = 200, 520, 100
    L = inputs.linear_layer(rng, M, K, N, "bf16", 1e-3)
    X = inputs.bf16_bits_to_f32(L["X"]).copy()
    W = inputs.bf16_bits_to_f32(L["W"]).copy()
    X[[3, 77, 150], [10, 300, 511]] = np.float32(2.0 ** -40)
    W[[5, 260], [7, 64]] = np.float32(-(2.0 ** -50))
    if pass_ == "fwd":
        check("fwd", "bf16", bf16(X), bf16(W), L["b"], M, K, N)
    else:
        check("dw", "bf16", bf16(X), L["dY"], None, M, K, N)


def test_outer_sum_out_of_range_and_non_finite():
    """Tiny and huge chunks in one row (the sum needs far more than 64 bits of
    the output grain), inf in a row, 2^-120 and 2^120 in another: those
    outputs take the warp-per-output superaccumulator."""
    rng = np.random.default_rng(13)
    M, K, N = 130, 512, 65
    X = rng.standard_normal((M, K))
    X[0, :256] = np.ldexp(1.0, -90) * (1 + rng.integers(0, 128, 256) / 128.0)
    X[0, 256:] = np.ldexp(1.0, 60) * (1 + rng.integers(0, 128, 256) / 128.0)
    X[5, 17] = np.inf
    X[9, 3] = 2.0 ** -120
    X[9, 200] = 2.0 ** 120
    X[11, 40] = np.nan
    W = rng.standard_normal((K, N)) * 0.02
    W[100, 3] = 0.0                                   # inf * 0 in output (5, 3)? only if X[5,100] is inf
    W[17, 4] = 0.0                                    # inf * 0 = NaN for output (5, 4)
    b = bf16(rng.standard_normal(N) * 0.02)
    got = run("fwd", "bf16", bf16(X), bf16(W), b, M, K, N)
    want = want_bits("fwd", "bf16", bf16(X), bf16(W), b, M, K, N)
    nan_w = (want & 0x7F80) == 0x7F80
    nan_w &= (want & 0x7F) != 0
    nan_g = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
    assert np.array_equal(nan_g, nan_w)
    assert np.array_equal(got[~nan_w], want[~nan_w])
    assert nan_w[5, 4] and nan_w[11].all()


def test_bias_far_from_the_grain():
    rng = np.random.default_rng(15)
    M, K, N = 130, 300, 66
    X = rng.standard_normal((M, K))
    W = rng.standard_normal((K, N)) * 0.02
    b = rng.standard_normal(N) * 0.02
    b[:10] = np.ldexp(1.0, -110) * (1 + rng.integers(0, 128, 10) / 128.0)
    b[10:20] = np.ldexp(1.0, 50) * (1 + rng.integers(0, 128, 10) / 128.0)
    b[20] = 0.0
    b[21] = -0.0
    b[22] = 2.0 ** -133                                # smallest subnormal
    check("fwd", "bf16", bf16(X), bf16(W), bf16(b), M, K, N)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_no_order_shows(dtype):
    """Permuting the reduction index (columns of X with rows of W) leaves every
    output's bits unchanged, across chunk boundaries and pieces; so does
    computing rows alone (any M)."""
    rng = np.random.default_rng(21)
    M, K, N = 96, 1100, 130
    L = inputs.linear_layer(rng, M, K, N, dtype, 1e-3)
    X, W, b = L["X"], L["W"], L["b"]
    base = check("fwd", dtype, X, W, b, M, K, N)
    perm = rng.permutation(K)
    Xp, Wp = np.ascontiguousarray(X[:, perm]), np.ascontiguousarray(W[perm])
    assert np.array_equal(run("fwd", dtype, Xp, Wp, b, M, K, N), base)
    assert np.array_equal(run("fwd", dtype, X[:5], W, b, 5, K, N), base[:5])


@pytest.mark.parametrize("seed", [42])
def test_gpt2_full_size_sampled(seed):
    for li, L in enumerate(inputs.gpt2(seed)):
        M, K, N = L["M"], L["K"], L["N"]
        for pass_ in ("fwd", "dx", "dw"):
            A, B, bias = operands(L, pass_)
            out = run(pass_, "bf16", A, B, bias, M, K, N)
            rows, cols = inputs.sample_indices(seed + li, out.shape[0], out.shape[1], 200)
            want = oracle.gemm_superacc(pass_, "bf16", A, B, bias, M, K, N, rows, cols)
            assert np.array_equal(out[rows, cols], want), (li, pass_)


def test_bias_gradient_layer_tier():
    """The autograd layer accepts the tier (bias gradient: the correctly
    rounded column sum over tokens)."""
    from deterministic_invariant_gemm_fwd_gb300 import nn
    rng = np.random.default_rng(3)
    L = inputs.linear_layer(rng, 300, 128, 64, "bf16", 1e-3)
    X, W, b, dY = (dev(L[k]) for k in ("X", "W", "b", "dY"))
    X.requires_grad_(True)
    W.requires_grad_(True)
    b.requires_grad_(True)
    Y = nn.deterministic_linear(X, W, b, tier="superacc")
    Y.backward(dY)
    ones = inputs.f32_to_bf16_bits(np.ones((300, 1), dtype=np.float32))
    want_db = oracle.gemm_superacc("dw", "bf16", ones, L["dY"], None, 300, 1, 64)
    assert np.array_equal(host_bits(b.grad).reshape(1, 64), want_db)
    assert np.array_equal(host_bits(Y), want_bits("fwd", "bf16", L["X"], L["W"], L["b"], 300, 128, 64))
