"""fp16 operands (IEEE binary16) on both tiers, against the CPU oracle.

The sgemm-bi page lists float16 among its engine's dtypes ("Use").  The exact
tier computes the same fixed-order KBN sum of float64 products as for fp32
and bf16 (Carbon README, "How It Works") and rounds once to fp16; it must be
bit-identical to the oracle.  The tensor-core tier multiplies fp16 x fp16
into fp32 accumulators; it must be deterministic, batch-invariant and within
the tolerance of the oracle's float64 value plus one fp16 rounding.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as inputs
from tests.gpu_util import bits, dev, host_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import deterministic_invariant_gemm_fwd_gb300 as cg  # noqa: E402


def _operands(layer, pass_):
    if pass_ == "fwd":
        return layer["X"], layer["W"], layer["b"]
    if pass_ == "dx":
        return layer["dY"], layer["W"], None
    return layer["X"], layer["dY"], None


def _call(pass_, A, B, bias, M, K, N, tier):
    tA, tB = dev(A, f16=True), dev(B, f16=True)
    tb = dev(bias, f16=True) if bias is not None else None
    shape = oracle.out_shape(pass_, M, K, N)
    out = torch.empty(shape, dtype=torch.float16, device="cuda")
    {"fwd": lambda: cg.carbon_gemm_fwd(out, tA, tB, tb, M, K, N, "f16", tier),
     "dx": lambda: cg.carbon_gemm_dx(out, tA, tB, M, K, N, "f16", tier),
     "dw": lambda: cg.carbon_gemm_dw(out, tA, tB, M, K, N, "f16", tier)}[pass_]()
    torch.cuda.synchronize()
    assert cg.carbon_get_device_status() == 0
    return out


@pytest.mark.parametrize("M,K,N", [(1, 1, 1), (7, 255, 3), (129, 256, 65), (33, 513, 33),
                                   (96, 320, 72), (260, 600, 70)])
@pytest.mark.parametrize("pass_", ["fwd", "dx", "dw"])
def test_exact_tier_bit_exact(M, K, N, pass_):
    # dY ~ N(0, 1e-3) puts many fp16 operands in the subnormal range
    layer = inputs.linear_layer(np.random.default_rng(M + 7 * K + 13 * N), M, K, N, "f16", 1e-3)
    A, B, bias = _operands(layer, pass_)
    ref, ref64 = oracle.gemm(pass_, "f16", A, B, bias, M, K, N)
    got = host_bits(_call(pass_, A, B, bias, M, K, N, "exact"))
    assert np.array_equal(got, bits(ref)), f"{np.count_nonzero(got != bits(ref))} mismatches"
    y64 = torch.empty(ref64.shape, dtype=torch.float64, device="cuda")
    cg.carbon_debug_exact_y64(pass_, y64, dev(A, f16=True), dev(B, f16=True),
                              dev(bias, f16=True) if bias is not None else None, M, K, N, "f16")
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(y64), bits(ref64))


def test_device_rounding_matches_the_oracle():
    rng = np.random.default_rng(16)
    y = np.concatenate([rng.standard_normal(20000) * np.ldexp(1.0, rng.integers(-30, 18, 20000)),
                        [65504.0, 65519.99, 65520.0, 65536.0, 2.0 ** -24, 2.0 ** -25,
                         3 * 2.0 ** -26, 2.0 ** -14, 0.0, -0.0, np.inf, -np.inf]])
    out = torch.empty(y.size, dtype=torch.float16, device="cuda")
    cg.carbon_debug_round("f16", out, torch.from_numpy(y).cuda(), y.size)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(out), oracle.round_out("f16", y))


@pytest.mark.parametrize("M,K,N", [(200, 256, 192), (513, 768, 768), (1100, 128, 1024)])
@pytest.mark.parametrize("pass_", ["fwd", "dx", "dw"])
def test_tc_tier_tolerance_and_determinism(M, K, N, pass_):
    layer = inputs.linear_layer(np.random.default_rng(3 * M + K + N), M, K, N, "f16", 1e-2)
    A, B, bias = _operands(layer, pass_)
    y1 = _call(pass_, A, B, bias, M, K, N, "tc")
    y2 = _call(pass_, A, B, bias, M, K, N, "tc")
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    _, y64 = oracle.gemm(pass_, "f16", A, B, bias, M, K, N)
    a = inputs.f16_bits_to_f32(A).astype(np.float64)
    b = inputs.f16_bits_to_f32(B).astype(np.float64)
    absdot = {"fwd": lambda: np.abs(a) @ np.abs(b), "dx": lambda: np.abs(a) @ np.abs(b).T,
              "dw": lambda: np.abs(a).T @ np.abs(b)}[pass_]()
    yt = y1.float().cpu().numpy().astype(np.float64)
    ulp = np.spacing(np.abs(yt).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(yt - y64) <= 2e-4 * absdot + ulp + 2.0 ** -24)


def test_tc_tier_rows_do_not_depend_on_the_batch():
    layer = inputs.linear_layer(np.random.default_rng(77), 513, 256, 192, "f16", 1e-2)
    full = _call("fwd", layer["X"], layer["W"], layer["b"], 513, 256, 192, "tc")
    for m in (1, 7, 64):
        part = _call("fwd", layer["X"][:m], layer["W"], layer["b"], m, 256, 192, "tc")
        assert torch.equal(full[:m].view(torch.int16), part.view(torch.int16))
