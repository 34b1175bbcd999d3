"""Exact tier on the GPU, through the C ABI, against the CPU oracle.

The bar is bit-identity: the rounded outputs and the float64 values before
rounding must equal the oracle's bits exactly (Carbon README, "How It
Works": a fixed summation order makes the result a function of the inputs
alone).
"""
import json
import os

import numpy as np
import pytest

import oracle
import seeded_inputs as inputs
from tests.gpu_util import bits, dev, host_bits, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import deterministic_invariant_gemm_fwd_gb300 as cg  # noqa: E402

PASS_OPERANDS = {"fwd": ("X", "W", "b"), "dx": ("dY", "W", None), "dw": ("X", "dY", None)}


def gpu_pass(pass_, dtype, A, B, bias, M, K, N, tier="exact", f64=False):
    """Run one pass on the GPU; returns the output tensor."""
    oshape = oracle.out_shape(pass_, M, K, N)
    tA, tB = dev(A), dev(B)
    tb = dev(bias) if bias is not None else None
    if f64:
        out = torch.empty(oshape, dtype=torch.float64, device="cuda")
        cg.carbon_debug_exact_y64(pass_, out, tA, tB, tb, M, K, N, dtype)
    else:
        out = torch.empty(oshape, dtype=torch_dtype(dtype), device="cuda")
        if pass_ == "fwd":
            cg.carbon_gemm_fwd(out, tA, tB, tb, M, K, N, dtype, tier)
        elif pass_ == "dx":
            cg.carbon_gemm_dx(out, tA, tB, M, K, N, dtype, tier)
        else:
            cg.carbon_gemm_dw(out, tA, tB, M, K, N, dtype, tier)
    torch.cuda.synchronize()
    assert cg.carbon_get_device_status() == 0
    return out


def check_dense(pass_, dtype, A, B, bias, M, K, N):
    ref, ref64 = oracle.gemm(pass_, dtype, A, B, bias, M, K, N)
    got = host_bits(gpu_pass(pass_, dtype, A, B, bias, M, K, N))
    got64 = host_bits(gpu_pass(pass_, dtype, A, B, bias, M, K, N, f64=True))
    assert np.array_equal(got64, bits(ref64)), \
        f"{pass_} {dtype} {M}x{K}x{N}: {np.count_nonzero(got64 != bits(ref64))} float64 mismatches"
    assert np.array_equal(got, bits(ref)), \
        f"{pass_} {dtype} {M}x{K}x{N}: {np.count_nonzero(got != bits(ref))} output mismatches"


def layer_operands(layer, pass_):
    a, b_, c = PASS_OPERANDS[pass_]
    return layer[a], layer[b_], (layer[c] if c else None)


# ---------------------------------------------------------------- single GEMM

def test_single_gemm_bit_exact_and_batch_invariant():
    d = inputs.single_gemm(42)
    X, W, b, M, K, N = d["X"], d["W"], d["b"], d["M"], d["K"], d["N"]
    check_dense("fwd", "f32", X, W, b, M, K, N)
    full = host_bits(gpu_pass("fwd", "f32", X, W, b, M, K, N))
    part = host_bits(gpu_pass("fwd", "f32", X[:8], W, b, 8, K, N))
    assert np.array_equal(part, full[:8])


# ------------------------------------------------------------------- toy MLP

@pytest.mark.parametrize("seed", inputs.SEEDS)
def test_toy_mlp_all_passes_bit_exact(seed):
    for layer in inputs.toy_mlp(seed):
        M, K, N = layer["M"], layer["K"], layer["N"]
        for pass_ in ("fwd", "dx", "dw"):
            A, B, bias = layer_operands(layer, pass_)
            check_dense(pass_, "f32", A, B, bias, M, K, N)


# ------------------------------------------------- GPT-2 shapes, reduced batch

def test_gpt2_shapes_reduced_batch_bit_exact():
    """All four GPT-2 layer shapes at M=600 (dW reduces over three chunks,
    the last one ragged), every element."""
    for layer in inputs.gpt2(7, M=600):
        M, K, N = layer["M"], layer["K"], layer["N"]
        for pass_ in ("fwd", "dx", "dw"):
            A, B, bias = layer_operands(layer, pass_)
            check_dense(pass_, "bf16", A, B, bias, M, K, N)


# --------------------------------------------------- GPT-2 shapes, full batch

@pytest.mark.parametrize("seed", [42, 2024])
def test_gpt2_full_size_sampled(seed):
    """M = 8192, every output computed on the GPU, a sample of outputs
    (corners, last row/column, random) recomputed by the oracle."""
    for li, layer in enumerate(inputs.gpt2(seed)):
        M, K, N = layer["M"], layer["K"], layer["N"]
        for pass_ in ("fwd", "dx", "dw"):
            A, B, bias = layer_operands(layer, pass_)
            out = host_bits(gpu_pass(pass_, "bf16", A, B, bias, M, K, N))
            rows, cols = inputs.sample_indices(seed + li, out.shape[0], out.shape[1], 150)
            ref, _ = oracle.gemm_at(pass_, "bf16", A, B, bias, M, K, N, rows, cols)
            assert np.array_equal(out[rows, cols], ref), (li, pass_)


@pytest.mark.slow
def test_gpt2_full_size_dense():
    """M = 8192, seed 42: every output of all 12 GEMMs (rounded and float64
    before rounding) against the oracle.  The kernel's paths that depend on
    the batch (row regrouping in 1024-row groups, the chunk range cut into
    pieces, run-time work units) only run at sizes like these."""
    for li, layer in enumerate(inputs.gpt2(42)):
        M, K, N = layer["M"], layer["K"], layer["N"]
        for pass_ in ("fwd", "dx", "dw"):
            A, B, bias = layer_operands(layer, pass_)
            ref, ref64 = oracle.gemm(pass_, "bf16", A, B, bias, M, K, N)
            got = host_bits(gpu_pass(pass_, "bf16", A, B, bias, M, K, N))
            assert np.array_equal(got, bits(ref)), \
                (li, pass_, int(np.count_nonzero(got != bits(ref))))
            got64 = host_bits(gpu_pass(pass_, "bf16", A, B, bias, M, K, N, f64=True))
            assert np.array_equal(got64, bits(ref64)), \
                (li, pass_, int(np.count_nonzero(got64 != bits(ref64))))


# ---------------------------------------------------------- stress (dW only)

def test_stress_dw_full_size_sampled():
    d = inputs.stress_dw(42)
    M, K, N = d["M"], d["K"], d["N"]
    out = gpu_pass("dw", "f32", d["X"], d["dY"], None, M, K, N)
    out64 = gpu_pass("dw", "f32", d["X"], d["dY"], None, M, K, N, f64=True)
    rows, cols = inputs.sample_indices(5, K, N, 300)
    ref, ref64 = oracle.gemm_at("dw", "f32", d["X"], d["dY"], None, M, K, N, rows, cols)
    assert np.array_equal(host_bits(out)[rows, cols], bits(ref))
    assert np.array_equal(host_bits(out64)[rows, cols], bits(ref64))


@pytest.mark.slow
def test_stress_dw_full_size_dense():
    """65536 tokens, K = 768, N = 3072: every output against the oracle."""
    d = inputs.stress_dw(42)
    M, K, N = d["M"], d["K"], d["N"]
    ref, ref64 = oracle.gemm("dw", "f32", d["X"], d["dY"], None, M, K, N)
    got = host_bits(gpu_pass("dw", "f32", d["X"], d["dY"], None, M, K, N))
    assert np.array_equal(got, bits(ref)), int(np.count_nonzero(got != bits(ref)))
    got64 = host_bits(gpu_pass("dw", "f32", d["X"], d["dY"], None, M, K, N, f64=True))
    assert np.array_equal(got64, bits(ref64)), int(np.count_nonzero(got64 != bits(ref64)))


def test_stress_dw_reduced_dense():
    d = inputs.stress_dw(999, M=4096, K=48, N=40)
    check_dense("dw", "f32", d["X"], d["dY"], None, d["M"], d["K"], d["N"])


# ------------------------------------------------------------- edge shapes

EDGE = [(1, 1, 1), (7, 255, 3), (129, 256, 65), (1, 257, 65), (7, 513, 1),
        (3, 0, 5), (129, 1, 3), (33, 31, 33)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,K,N", EDGE)
def test_edge_shapes_all_passes(dtype, M, K, N):
    rng = np.random.default_rng(M * 1000 + K * 10 + N)
    layer = inputs.linear_layer(rng, M, K, N, dtype, 1e-3)
    for pass_ in ("fwd", "dx", "dw"):
        A, B, bias = layer_operands(layer, pass_)
        check_dense(pass_, dtype, A, B, bias, M, K, N)
    # forward without bias
    check_dense("fwd", dtype, layer["X"], layer["W"], None, M, K, N)


def test_empty_output_is_no_op():
    X = torch.zeros((0, 4), device="cuda")
    W = torch.zeros((4, 3), device="cuda")
    Y = torch.empty((0, 3), device="cuda")
    cg.carbon_gemm_fwd(Y, X, W, None, 0, 4, 3, "f32", "exact")
    assert cg.carbon_get_device_status() == 0


def test_zero_reduction_gives_bias_or_zero():
    b = np.array([0.375, -2.0, 1e-3], dtype=np.float32)
    X = np.zeros((4, 0), dtype=np.float32)
    W = np.zeros((0, 3), dtype=np.float32)
    Y = host_bits(gpu_pass("fwd", "f32", X, W, b, 4, 0, 3))
    assert np.array_equal(Y, np.tile(bits(b), (4, 1)))
    Y0 = host_bits(gpu_pass("fwd", "f32", X, W, None, 4, 0, 3))
    assert not Y0.any()


# -------------------------------------------------------- closed-form cases

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form.json")


def test_closed_form_cases_on_gpu():
    from tests.test_oracle import _case_operands
    for case in json.load(open(GOLDEN))["cases"]:
        for dtype in case["dtypes"]:
            for pass_ in case.get("passes", ["fwd", "dx", "dw"]):
                A, B, bias, (M, K, N) = _case_operands(case, pass_, dtype)
                out = host_bits(gpu_pass(pass_, dtype, A, B, bias, M, K, N)).ravel()[0]
                want = np.float32(float.fromhex(case["expect"]))
                wbits = int(want.view(np.uint32))
                if dtype == "bf16":
                    wbits >>= 16
                assert int(out) == wbits, (case["name"], dtype, pass_, hex(int(out)), hex(wbits))


# ------------------------------------------------------------- rounding

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_device_rounding_matches_rne(dtype):
    from tests.test_oracle import _rounding_corpus
    y = _rounding_corpus(np.random.default_rng(11))
    ref = bits(oracle.round_out(dtype, y))
    ty = torch.from_numpy(y).cuda()
    out = torch.empty(y.shape, dtype=torch_dtype(dtype), device="cuda")
    cg.carbon_debug_round(dtype, out, ty, y.size)
    torch.cuda.synchronize()
    got = host_bits(out)
    nan = np.isnan(y)
    assert np.array_equal(got[~nan], ref[~nan])


def test_non_finite_inputs_agree_on_nan():
    X = np.array([[1.0, np.inf, 2.0], [1.0, 2.0, 3.0]], dtype=np.float32)
    W = np.array([[1.0], [0.5], [2.0]], dtype=np.float32)
    ref, _ = oracle.gemm("fwd", "f32", X, W, None, 2, 3, 1)
    got = gpu_pass("fwd", "f32", X, W, None, 2, 3, 1).cpu().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert got[1, 0] == ref[1, 0]


# ------------------------------------------------------ determinism / status

def test_repeat_runs_and_batch_sweep_bit_identical():
    layer = inputs.gpt2(123, M=513, layers=((768, 768),))[0]
    X, W, b = layer["X"], layer["W"], layer["b"]
    full = host_bits(gpu_pass("fwd", "bf16", X, W, b, 513, 768, 768))
    for _ in range(2):
        assert np.array_equal(host_bits(gpu_pass("fwd", "bf16", X, W, b, 513, 768, 768)), full)
    for m in (1, 7, 64):
        part = host_bits(gpu_pass("fwd", "bf16", X[:m], W, b, m, 768, 768))
        assert np.array_equal(part, full[:m])
    dX = host_bits(gpu_pass("dx", "bf16", layer["dY"], W, None, 513, 768, 768))
    for m in (1, 7, 64):
        part = host_bits(gpu_pass("dx", "bf16", layer["dY"][:m], W, None, m, 768, 768))
        assert np.array_equal(part, dX[:m])


def test_timeout_probe_reports_and_clears():
    assert cg.carbon_get_device_status() == 0
    cg.carbon_debug_timeout_probe(2_000_000)      # 2 ms budget, nothing arrives
    assert cg.carbon_get_device_status() == 5     # CARBON_ERR_TIMEOUT
    assert cg.carbon_get_device_status() == 0     # cleared
    d = inputs.single_gemm(7)
    check_dense("fwd", "f32", d["X"], d["W"], d["b"], d["M"], d["K"], d["N"])


def test_fp64_rate_microbenchmark_is_sane():
    dfma, dadd = cg.carbon_measure_fp64_rate()
    # GB300: a few lanes per SM per clock; nominal 1.25 TFLOP/s = 0.6e12 DFMA/s
    assert 1e11 < dfma < 5e12
    assert 1e11 < dadd < 5e12


# ------------------------------------------- fast path / full step boundary

def _adversarial(kind, rng, shape):
    """Operands that make some KBN steps round and others not (the kernel
    proves exactness per 32-deep slice and falls back to the full step)."""
    if kind == "wide":        # bf16 values spread over 2^-60 .. 2^60
        v = np.ldexp(1.0, rng.integers(-60, 61, shape)) * (1 + rng.integers(0, 128, shape) / 128.0)
        return v * rng.choice([-1.0, 1.0], shape)
    if kind == "rare_tiny":   # normal data with rare tiny entries
        v = rng.standard_normal(shape)
        flat = v.reshape(-1)
        flat[rng.integers(0, flat.size, max(1, flat.size // 500))] *= 2.0 ** -45
        return v
    if kind == "growing":     # magnitudes growing along the reduction
        v = rng.standard_normal(shape)
        return v * np.ldexp(1.0, (np.arange(v.size) % 97 // 6).reshape(shape))
    if kind == "integers":    # small integers: every step exact
        return rng.integers(-8, 9, shape).astype(np.float64)
    raise ValueError(kind)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("kind", ["wide", "rare_tiny", "growing", "integers"])
def test_exactness_proof_boundaries(kind, dtype):
    rng = np.random.default_rng(hash(kind) % 1000 + (dtype == "f32"))
    M, K, N = 70, 600, 45
    enc = (lambda a: a.astype(np.float32)) if dtype == "f32" else \
        (lambda a: inputs.f32_to_bf16_bits(a.astype(np.float32)))
    X = enc(_adversarial(kind, rng, (M, K)))
    W = enc(_adversarial(kind, rng, (K, N)) * 0.02)
    dY = enc(_adversarial(kind, rng, (M, N)) * 1e-3)
    b = enc(rng.standard_normal(N) * 0.02)
    check_dense("fwd", dtype, X, W, b, M, K, N)
    check_dense("dx", dtype, dY, W, None, M, K, N)
    check_dense("dw", dtype, X, dY, None, M, K, N)


def test_int_mac_rate_microbenchmark_is_sane():
    rate = cg.carbon_measure_int_mac_rate()
    # GB300: tens of 32x32->64 multiply-adds per SM per clock over 152 SMs
    assert 1e12 < rate < 1e14


@pytest.mark.parametrize("pass_", ["fwd", "dx", "dw"])
def test_bf16_outlier_rows_and_columns(pass_):
    """bf16 operands with a few huge-range rows/columns: the integer path must
    route those (row, column, chunk) groups through the precise check or the
    float64 step, and every other group through the integer sum, with the
    oracle's bits everywhere."""
    rng = np.random.default_rng(31)
    M, K, N = 130, 700, 70
    L = inputs.linear_layer(rng, M, K, N, "bf16", 1e-3)
    for key, axis in (("X", 0), ("W", 1), ("dY", 0)):
        a = inputs.bf16_bits_to_f32(L[key]).copy()
        idx = rng.integers(0, a.shape[axis], 3)
        if axis == 0:
            a[idx, rng.integers(0, a.shape[1], 3)] *= np.float32(2.0 ** -40)
            a[idx[:1], :5] *= np.float32(2.0 ** 30)
        else:
            a[rng.integers(0, a.shape[0], 3), idx] *= np.float32(2.0 ** -40)
        L[key] = inputs.f32_to_bf16_bits(a)
    A, B, bias = layer_operands(L, pass_)
    check_dense(pass_, "bf16", A, B, bias, M, K, N)
