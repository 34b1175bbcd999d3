"""Tensor-core tier on the GPU, through the C ABI.

Bars (sgemm-bi "Determinism contracts", tensor-core tier):
  * bit-identical across repeated runs;
  * fwd and dX rows bit-identical for every batch size M;
  * fp32 accumulator within 2e-4 * sum_k |x_ik * w_kj| of the oracle's
    float64 value, bf16 output within that plus one bf16 ulp;
  * exact on inputs whose fp32 accumulation cannot round (small integers),
    which pins operand layout and indexing independently of any tolerance.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as inputs
from tests.gpu_util import dev, host_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import deterministic_invariant_gemm_fwd_gb300 as cg  # noqa: E402

TOL = 2e-4
OPERANDS = {"fwd": ("X", "W", "b"), "dx": ("dY", "W", None), "dw": ("X", "dY", None)}


def run_tc(pass_, A, B, bias, M, K, N, f32=False):
    shape = oracle.out_shape(pass_, M, K, N)
    tA, tB = dev(A), dev(B)
    tb = dev(bias) if bias is not None else None
    if f32:
        out = torch.empty(shape, dtype=torch.float32, device="cuda")
        cg.carbon_debug_tc_f32(pass_, out, tA, tB, tb, M, K, N)
    else:
        out = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        if pass_ == "fwd":
            cg.carbon_gemm_fwd(out, tA, tB, tb, M, K, N, "bf16", "tc")
        elif pass_ == "dx":
            cg.carbon_gemm_dx(out, tA, tB, M, K, N, "bf16", "tc")
        else:
            cg.carbon_gemm_dw(out, tA, tB, M, K, N, "bf16", "tc")
    torch.cuda.synchronize()
    assert cg.carbon_get_device_status() == 0
    return out


def f64(a):
    return inputs.bf16_bits_to_f32(a).astype(np.float64)


def abs_dot(pass_, A, B):
    a, b = np.abs(f64(A)), np.abs(f64(B))
    return {"fwd": lambda: a @ b, "dx": lambda: a @ b.T, "dw": lambda: a.T @ b}[pass_]()


def check_tolerance(pass_, A, B, bias, M, K, N, rows=None, cols=None):
    """fp32 accumulator and bf16 output against the oracle's float64 value."""
    acc = run_tc(pass_, A, B, bias, M, K, N, f32=True).cpu().numpy().astype(np.float64)
    out = run_tc(pass_, A, B, bias, M, K, N).float().cpu().numpy().astype(np.float64)
    if rows is None:
        _, y64 = oracle.gemm(pass_, "bf16", A, B, bias, M, K, N)
        ad = abs_dot(pass_, A, B)
        acc_s, out_s = acc, out
    else:
        _, y64 = oracle.gemm_at(pass_, "bf16", A, B, bias, M, K, N, rows, cols)
        ad = abs_dot(pass_, A, B)[rows, cols]
        acc_s, out_s = acc[rows, cols], out[rows, cols]
    bound = TOL * ad
    if bias is not None:
        bb = np.abs(f64(bias))
        bound = bound + 2.0 ** -23 * (np.abs(y64) + (bb[cols] if rows is not None else bb))
    err = np.abs(acc_s - y64)
    assert np.all(err <= bound), f"{pass_}: acc err {err.max():.3g} > bound"
    ulp = np.spacing(np.abs(out_s).astype(np.float32)).astype(np.float64) * 65536.0
    assert np.all(np.abs(out_s - y64) <= bound + ulp), f"{pass_}: bf16 output out of tolerance"
    # the bf16 output is the fp32 accumulator rounded once (RNE)
    want = torch.from_numpy(acc_s.astype(np.float32)).to(torch.bfloat16).float().numpy()
    assert np.array_equal(out_s.astype(np.float32), want)


def test_small_integer_inputs_accumulate_exactly():
    """Products and partial sums of small integers are exact in fp32, so any
    operand-layout or indexing error shows up as a wrong integer."""
    rng = np.random.default_rng(3)
    M, K, N = 200, 320, 136
    X = inputs.f32_to_bf16_bits(rng.integers(-4, 5, size=(M, K)).astype(np.float32))
    W = inputs.f32_to_bf16_bits(rng.integers(-4, 5, size=(K, N)).astype(np.float32))
    dY = inputs.f32_to_bf16_bits(rng.integers(-4, 5, size=(M, N)).astype(np.float32))
    b = inputs.f32_to_bf16_bits(rng.integers(-8, 9, size=(N,)).astype(np.float32))
    for pass_, A, B, bias in (("fwd", X, W, b), ("dx", dY, W, None), ("dw", X, dY, None)):
        acc = run_tc(pass_, A, B, bias, M, K, N, f32=True).cpu().numpy().astype(np.float64)
        a, bb = f64(A), f64(B)
        exact = {"fwd": lambda: a @ bb, "dx": lambda: a @ bb.T, "dw": lambda: a.T @ bb}[pass_]()
        if bias is not None:
            exact = exact + f64(bias)
        assert np.array_equal(acc, exact), f"{pass_}: {np.count_nonzero(acc != exact)} wrong"


@pytest.mark.parametrize("M,K,N", [(2048, 256, 256), (4000, 384, 200), (1100, 128, 1024), (2048, 768, 2304),
                                   (2048, 768, 768), (2048, 3072, 768), (2048, 768, 1024), (2048, 512, 1024),
                                   (2048, 512, 128)])
def test_dw_token_split_accumulates_exactly(M, K, N):
    """dW shapes with few output tiles take the cluster split of the token
    range; with small-integer operands every partial and their in-order sum
    are exact, so the result must equal the exact product.  Tile width and
    piece count: 768 x 2304 192 columns in two pieces, 768 x 768 192 in four,
    the first three 192 in eight; 3072 x 768 256 in two, 768 x 1024 256 in
    four, 512 x 1024 256 in eight, 512 x 128 128 in eight."""
    rng = np.random.default_rng(M)
    X = inputs.f32_to_bf16_bits(rng.integers(-4, 5, size=(M, K)).astype(np.float32))
    dY = inputs.f32_to_bf16_bits(rng.integers(-4, 5, size=(M, N)).astype(np.float32))
    acc = run_tc("dw", X, dY, None, M, K, N, f32=True).cpu().numpy().astype(np.float64)
    exact = f64(X).T @ f64(dY)
    assert np.array_equal(acc, exact), f"{np.count_nonzero(acc != exact)} wrong"
    out = host_bits(run_tc("dw", X, dY, None, M, K, N))
    again = host_bits(run_tc("dw", X, dY, None, M, K, N))
    assert np.array_equal(out, again)


@pytest.mark.parametrize("M,K,N", [(128, 64, 128), (7, 768, 768), (513, 256, 2304),
                                   (300, 3072, 136), (64, 1000, 264)])
def test_tolerance_all_passes(M, K, N):
    rng = np.random.default_rng(M + K + N)
    L = inputs.linear_layer(rng, M, K, N, "bf16", 1e-4)
    for pass_ in ("fwd", "dx", "dw"):
        a, b_, c = OPERANDS[pass_]
        check_tolerance(pass_, L[a], L[b_], L[c] if c else None, M, K, N)
    check_tolerance("fwd", L["X"], L["W"], None, M, K, N)


@pytest.mark.parametrize("seed", [42, 999])
def test_gpt2_full_size_tolerance_sampled(seed):
    for li, L in enumerate(inputs.gpt2(seed)):
        M, K, N = L["M"], L["K"], L["N"]
        for pass_ in ("fwd", "dx", "dw"):
            a, b_, c = OPERANDS[pass_]
            R, C = oracle.out_shape(pass_, M, K, N)
            rows, cols = inputs.sample_indices(seed * 10 + li, R, C, 200)
            check_tolerance(pass_, L[a], L[b_], L[c] if c else None, M, K, N, rows, cols)


def test_batch_invariance_and_repeatability():
    """Rows of fwd and dX are bit-identical for M in {1,7,64,513,2048,8192}
    and across 5 repeated runs (all four GPT-2 shapes)."""
    Ms = (1, 7, 64, 513, 2048, 8192)
    for L in inputs.gpt2(2024):
        K, N = L["K"], L["N"]
        X, W, b, dY = L["X"], L["W"], L["b"], L["dY"]
        full_y = host_bits(run_tc("fwd", X, W, b, 8192, K, N))
        full_dx = host_bits(run_tc("dx", dY, W, None, 8192, K, N))
        for _ in range(4):
            assert np.array_equal(host_bits(run_tc("fwd", X, W, b, 8192, K, N)), full_y)
            assert np.array_equal(host_bits(run_tc("dx", dY, W, None, 8192, K, N)), full_dx)
        for m in Ms[:-1]:
            y = host_bits(run_tc("fwd", X[:m], W, b, m, K, N))
            assert np.array_equal(y, full_y[:m]), (K, N, m)
            dx = host_bits(run_tc("dx", dY[:m], W, None, m, K, N))
            assert np.array_equal(dx, full_dx[:m]), (K, N, m)
        dw = host_bits(run_tc("dw", X, dY, None, 8192, K, N))
        for _ in range(4):
            assert np.array_equal(host_bits(run_tc("dw", X, dY, None, 8192, K, N)), dw)


def test_rows_are_independent_of_their_neighbours():
    """Changing other rows of X does not change row 0 of Y."""
    L = inputs.gpt2(7, M=256, layers=((768, 768),))[0]
    X2 = L["X"].copy()
    X2[1:] = inputs.f32_to_bf16_bits(np.random.default_rng(1).standard_normal((255, 768)).astype(np.float32))
    y1 = host_bits(run_tc("fwd", L["X"], L["W"], L["b"], 256, 768, 768))
    y2 = host_bits(run_tc("fwd", X2, L["W"], L["b"], 256, 768, 768))
    assert np.array_equal(y1[0], y2[0])


def test_empty_reduction_and_empty_output():
    b = inputs.f32_to_bf16_bits(np.array([0.5, -1.0, 2.0, 0.25, 1, 2, 3, 4], dtype=np.float32))
    X = np.zeros((3, 0), dtype=np.uint16)
    W = np.zeros((0, 8), dtype=np.uint16)
    y = host_bits(run_tc("fwd", X, W, b, 3, 0, 8))
    assert np.array_equal(y, np.tile(b, (3, 1)))
    Y = torch.empty((0, 8), dtype=torch.bfloat16, device="cuda")
    cg.carbon_gemm_fwd(Y, dev(X), dev(W), None, 0, 0, 8, "bf16", "tc")


def test_rejections():
    X = torch.zeros((16, 12), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((12, 16), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((16, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cg.CarbonError) as e:        # K not a multiple of 8
        cg.carbon_gemm_fwd(Y, X, W, None, 16, 12, 16, "bf16", "tc")
    assert e.value.status == 3
    Xf = torch.zeros((16, 16), device="cuda")
    Wf = torch.zeros((16, 16), device="cuda")
    Yf = torch.empty((16, 16), device="cuda")
    with pytest.raises(cg.CarbonError) as e:
        cg.carbon_gemm_fwd(Yf, Xf, Wf, None, 16, 16, 16, "f32", "tc")
    assert e.value.status == 2
    Xb = torch.zeros((16 * 16 + 8,), dtype=torch.bfloat16, device="cuda")[1:257].view(16, 16)
    Wb = torch.zeros((16, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cg.CarbonError) as e:         # base not 16-byte aligned
        cg.carbon_gemm_fwd(Y, Xb, Wb, None, 16, 16, 16, "bf16", "tc")
    assert e.value.status == 3
