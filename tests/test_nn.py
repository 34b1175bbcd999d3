"""The autograd linear layer's host side: parameter layout ([in, out]),
conversion from torch.nn.Linear, initialisation bounds, and that it has no
CPU path (a CPU input is rejected before any library call)."""
import math

import pytest

torch = pytest.importorskip("torch")

from deterministic_invariant_gemm_fwd_gb300 import nn as cnn  # noqa: E402


def test_weight_is_stored_in_out():
    lin = cnn.Linear(24, 40)
    assert lin.weight.shape == (24, 40) and lin.bias.shape == (40,)
    bound = 1.0 / math.sqrt(24)
    assert float(lin.weight.detach().abs().max()) <= bound + 1e-7
    assert float(lin.bias.detach().abs().max()) <= bound + 1e-7
    assert "tier='exact'" in repr(lin)


def test_from_torch_transposes_the_weight():
    ref = torch.nn.Linear(24, 40)
    lin = cnn.Linear.from_torch(ref, tier="tc")
    assert lin.tier == "tc"
    assert torch.equal(lin.weight, ref.weight.t())
    assert torch.equal(lin.bias, ref.bias)
    nob = cnn.Linear.from_torch(torch.nn.Linear(8, 16, bias=False))
    assert nob.bias is None


def test_cpu_inputs_are_rejected():
    lin = cnn.Linear(8, 16)
    with pytest.raises(ValueError):
        lin(torch.zeros(4, 8))
    with pytest.raises(ValueError):
        cnn.bias_grad(torch.zeros(4, 8))


def test_feature_mismatch_is_rejected():
    with pytest.raises(ValueError):
        cnn.deterministic_linear(torch.zeros(4, 9), torch.zeros(8, 16))
