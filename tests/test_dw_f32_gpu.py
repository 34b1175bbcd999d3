"""Weight gradient of bf16 operands into an fp32 output (sgemm-bi: dW is
f32-accumulated).  Exact tier: the fixed-order KBN float64 value, rounded
once to fp32, bit-identical to the oracle's float64 value rounded to fp32.
Tensor-core tier: the fp32 accumulator, the same bits as the inspection
path, within the tolerance of the oracle."""
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


@pytest.mark.parametrize("M,K,N", [(3, 5, 7), (129, 1, 3), (600, 200, 264), (1000, 130, 70)])
def test_exact_tier_is_the_float64_value_rounded_to_fp32(M, K, N):
    L = inputs.linear_layer(np.random.default_rng(M + K + N), M, K, N, "bf16", 1e-3)
    _, y64 = oracle.gemm("dw", "bf16", L["X"], L["dY"], None, M, K, N)
    got = cg.linear_dw_f32(dev(L["X"]), dev(L["dY"]), tier="exact")
    torch.cuda.synchronize()
    assert cg.carbon_get_device_status() == 0
    want = y64.astype(np.float32)                  # numpy's conversion rounds to nearest even
    assert np.array_equal(host_bits(got), want.view(np.uint32))


@pytest.mark.parametrize("M,K,N", [(2048, 256, 256), (1100, 128, 1024)])
def test_tc_tier_is_the_fp32_accumulator(M, K, N):
    L = inputs.linear_layer(np.random.default_rng(5 * M + N), M, K, N, "bf16", 1e-2)
    X, dY = dev(L["X"]), dev(L["dY"])
    got = cg.linear_dw_f32(X, dY, tier="tc")
    acc = torch.empty((K, N), dtype=torch.float32, device="cuda")
    cg.carbon_debug_tc_f32("dw", acc, X, dY, None, M, K, N)
    torch.cuda.synchronize()
    assert cg.carbon_get_device_status() == 0
    assert torch.equal(got, acc)
    _, y64 = oracle.gemm("dw", "bf16", L["X"], L["dY"], None, M, K, N)
    a = inputs.bf16_bits_to_f32(L["X"]).astype(np.float64)
    b = inputs.bf16_bits_to_f32(L["dY"]).astype(np.float64)
    absdot = np.abs(a).T @ np.abs(b)
    assert np.all(np.abs(got.cpu().numpy().astype(np.float64) - y64) <= 2e-4 * absdot)
