"""The exact tier's no-allocation entry point, through the C ABI.

carbon_gemm_exact_bf16_noalloc exists for callers that cannot allocate device
memory while they run (a framework allocator that owns the whole GPU, a
latency-critical loop that must never wait on or fail in an allocator, a
process without the stream-ordered pool).  It takes its workspace from a
fixed 64 MiB device array that CUDA reserves when the library's module for
this entry point loads on the device (its first call there), so it must give
the same bits as the regular bf16 exact-tier entry points (the exact tier's
tolerance is bit-identity), also when called twice in a row with different
inputs (the array keeps the previous call's contents).  Its kernels are the
integer-pipe exact kernels, which no other entry point runs, so the outputs
are also compared with the CPU oracle element by element.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

import oracle
import seeded_inputs as inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import deterministic_invariant_gemm_fwd_gb300 as cg  # noqa: E402
from deterministic_invariant_gemm_fwd_gb300 import _binding  # noqa: E402


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _operands(L, pass_):
    if pass_ == "fwd":
        return L["X"], L["W"], L["b"]
    if pass_ == "dx":
        return L["dY"], L["W"], None
    return L["X"], L["dY"], None


def _regular(pass_, A, B, bias, M, K, N):
    shape = {"fwd": (M, N), "dx": (M, K), "dw": (K, N)}[pass_]
    out = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    if pass_ == "fwd":
        cg.carbon_gemm_fwd(out, _dev(A), _dev(B), None if bias is None else _dev(bias),
                           M, K, N, "bf16", "exact")
    elif pass_ == "dx":
        cg.carbon_gemm_dx(out, _dev(A), _dev(B), M, K, N, "bf16", "exact")
    else:
        cg.carbon_gemm_dw(out, _dev(A), _dev(B), M, K, N, "bf16", "exact")
    return out


def _noalloc(pass_, A, B, bias, M, K, N):
    shape = {"fwd": (M, N), "dx": (M, K), "dw": (K, N)}[pass_]
    out = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    # keep the operand tensors alive until the kernels have run
    tA, tB = _dev(A), _dev(B)
    tb = None if bias is None else _dev(bias)
    # straight through the C entry point (ctypes), raw device pointers
    st = _binding.lib.carbon_gemm_exact_bf16_noalloc(
        _binding.PASSES[pass_], out.data_ptr(), tA.data_ptr(), tB.data_ptr(),
        None if tb is None else tb.data_ptr(), M, K, N,
        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0, _binding.STATUS.get(st, st)
    return out


@pytest.mark.parametrize("pass_", ["fwd", "dx", "dw"])
def test_noalloc_matches_regular_entry_point_twice_in_a_row(pass_):
    rng = np.random.default_rng(2024)
    shapes = [(600, 768, 640), (257, 300, 129)]   # second call: other sizes and data
    for (M, K, N) in shapes:
        L = inputs.linear_layer(rng, M, K, N, "bf16", 1e-4)
        A, B, bias = _operands(L, pass_)
        ref = _regular(pass_, A, B, bias, M, K, N)
        torch.cuda.synchronize()
        got = _noalloc(pass_, A, B, bias, M, K, N)
        assert cg.carbon_get_device_status() == 0
        assert np.array_equal(_bits(got), _bits(ref)), (pass_, M, K, N)
        want, _ = oracle.gemm(pass_, "bf16", A, B, bias, M, K, N)
        assert np.array_equal(_bits(got), want), (pass_, M, K, N, "oracle")


def test_noalloc_rejects_problems_beyond_its_workspace():
    M, K, N = 8192, 3072, 768            # fwd needs ~110 MB of workspace > 64 MiB
    X = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    st = _binding.lib.carbon_gemm_exact_bf16_noalloc(
        _binding.PASSES["fwd"], Y.data_ptr(), X.data_ptr(), W.data_ptr(), None, M, K, N,
        torch.cuda.current_stream().cuda_stream)
    assert _binding.STATUS[st] == "CARBON_ERR_SCRATCH_LIMIT"
    assert cg.carbon_status_string(st) == "CARBON_ERR_SCRATCH_LIMIT"
