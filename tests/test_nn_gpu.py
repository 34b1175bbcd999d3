"""The autograd linear layer on the GPU: its forward and backward results
are the library's GEMMs bit for bit, its bias gradient is the exact tier's
fixed-order sum over tokens (bit-identical to the CPU oracle), and rows do
not depend on the batch they are computed in."""
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
from deterministic_invariant_gemm_fwd_gb300 import nn as cnn  # noqa: E402


def _layer(dtype, M, K, N, seed):
    L = inputs.linear_layer(np.random.default_rng(seed), M, K, N, dtype, 1e-3)
    return L, {k: dev(L[k]) for k in ("X", "W", "b", "dY")}


@pytest.mark.parametrize("dtype,tier", [("f32", "exact"), ("bf16", "exact"), ("bf16", "tc")])
def test_autograd_matches_the_abi_calls(dtype, tier):
    M, K, N = 2 * 96, 320, 72
    L, t = _layer(dtype, M, K, N, 5)
    x = t["X"].view(2, 96, K).clone().requires_grad_(True)
    w = t["W"].clone().requires_grad_(True)
    b = t["b"].clone().requires_grad_(True)
    y = cnn.deterministic_linear(x, w, b, tier)
    y.backward(t["dY"].view(2, 96, N))
    torch.cuda.synchronize()
    assert cg.carbon_get_device_status() == 0
    assert torch.equal(y.detach().view(M, N), cg.linear_fwd(t["X"], t["W"], t["b"], tier=tier))
    assert torch.equal(x.grad.view(M, K), cg.linear_dx(t["dY"], t["W"], tier=tier))
    assert torch.equal(w.grad, cg.linear_dw(t["X"], t["dY"], tier=tier))
    # the bias gradient: the exact tier's fixed-order KBN sum over the tokens
    ones = np.ones((M, 1), dtype=np.float32)
    if dtype == "bf16":
        ones = inputs.f32_to_bf16_bits(ones)
    ref, _ = oracle.gemm("dw", dtype, ones, L["dY"], None, M, 1, N)
    assert np.array_equal(host_bits(b.grad), bits(ref).reshape(N))


def test_bias_grad_long_token_range_is_exact():
    """1000 tokens (4 chunks, the last short) of values spread over 2^+-20:
    the column sums are the oracle's, bit for bit."""
    rng = np.random.default_rng(9)
    M, N = 1000, 130
    v = np.ldexp(rng.integers(1, 256, (M, N)).astype(np.float64), rng.integers(-20, 20, (M, N)))
    dY = inputs.f32_to_bf16_bits((v * rng.choice([-1.0, 1.0], (M, N))).astype(np.float32))
    db = cnn.bias_grad(dev(dY))
    ones = inputs.f32_to_bf16_bits(np.ones((M, 1), dtype=np.float32))
    ref, _ = oracle.gemm("dw", "bf16", ones, dY, None, M, 1, N)
    assert np.array_equal(host_bits(db), bits(ref).reshape(N))


@pytest.mark.parametrize("tier", ["exact", "tc"])
def test_module_rows_do_not_depend_on_the_batch(tier):
    torch.manual_seed(0)
    ref = torch.nn.Linear(256, 192).to(torch.bfloat16).cuda()
    lin = cnn.Linear.from_torch(ref, tier=tier)
    x = torch.randn(513, 256, device="cuda").to(torch.bfloat16)
    full = lin(x)
    part = lin(x[:7].contiguous())
    again = lin(x)
    torch.cuda.synchronize()
    assert torch.equal(full[:7], part)
    assert torch.equal(full, again)
    # the weight is the torch layer's, transposed: same product up to rounding
    assert torch.allclose(full.float(), ref(x).float(), atol=0.05, rtol=0.05)
