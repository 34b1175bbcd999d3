"""Reductions split across ranks on the GPU: chunk values and their combine
through the C ABI, bit-identical to the single-device exact tier and to the
oracle (Carbon README, "How It Works": all-gather and a reduction in rank
order; the fixed chunk order makes the split invisible).

* one process emulating the ranks' shares in turn (token ranges of
  dp.token_ranges), every pass and dtype, ragged sizes, the GPT-2 dW shape
  and the cancellation stress input;
* two processes on the one GPU with a gloo process group (host copies of the
  chunk values), each running dp.linear_dw_data_parallel on its own tokens.
  Their kernels never wait on one another; only the host collective joins
  them.
"""
import os
import socket

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
from deterministic_invariant_gemm_fwd_gb300 import dp  # noqa: E402


def single_dw(X, dY, M, K, N, dtype):
    out = torch.empty((K, N), dtype=torch_dtype(dtype), device="cuda")
    cg.carbon_gemm_dw(out, X, dY, M, K, N, dtype, "exact")
    torch.cuda.synchronize()
    return host_bits(out)


def split_dw(X, dY, M, K, N, dtype, world):
    parts = [dp.chunk_values(X[a:b].contiguous(), dY[a:b].contiguous())
             for a, b in dp.token_ranges(M, world)]
    P = torch.cat(parts)
    assert P.shape[0] == (M + 255) // 256
    out = dp.combine(P, dtype)
    torch.cuda.synchronize()
    assert cg.carbon_get_device_status() == 0
    return host_bits(out)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("world", [2, 3, 5])
def test_split_dw_equals_single_device_and_oracle(dtype, world):
    rng = np.random.default_rng(world * 10 + len(dtype))
    M, K, N = 1100, 70, 45
    L = inputs.linear_layer(rng, M, K, N, dtype, 1e-3)
    f16 = dtype == "f16"
    X, dY = dev(L["X"], f16=f16), dev(L["dY"], f16=f16)
    got = split_dw(X, dY, M, K, N, dtype, world)
    assert np.array_equal(got, single_dw(X, dY, M, K, N, dtype))
    want, _ = oracle.gemm("dw", dtype, L["X"], L["dY"], None, M, K, N)
    assert np.array_equal(got, bits(want))


def test_chunk_values_are_the_oracle_chunk_values():
    """One chunk per call: the chunk value of a 256-token share is the oracle's
    whole float64 value of that share (one chunk, outer KBN of one value)."""
    rng = np.random.default_rng(3)
    M, K, N = 256, 33, 20
    L = inputs.linear_layer(rng, M, K, N, "bf16", 1e-3)
    P = dp.chunk_values(dev(L["X"]), dev(L["dY"]))
    _, y64 = oracle.gemm("dw", "bf16", L["X"], L["dY"], None, M, K, N)
    assert np.array_equal(host_bits(P[0]), bits(y64))


@pytest.mark.parametrize("pass_", ["fwd", "dx"])
def test_split_reduction_other_passes_with_bias(pass_):
    """The same split along K (fwd) or N (dX), the bias joining at the combine."""
    rng = np.random.default_rng(9)
    M, K, N = 64, 800, 300
    L = inputs.linear_layer(rng, M, K, N, "f32", 1e-3)
    X, W, b, dY = (dev(L[k]) for k in ("X", "W", "b", "dY"))
    R = K if pass_ == "fwd" else N
    parts = []
    for a, c in dp.token_ranges(R, 3):
        if pass_ == "fwd":
            A, B = X[:, a:c].contiguous(), W[a:c].contiguous()
            P = torch.empty(((c - a + 255) // 256, M, N), dtype=torch.float64, device="cuda")
            if c > a:
                cg.carbon_gemm_chunk_values("fwd", P, A, B, M, c - a, N, "f32")
        else:
            A, B = dY[:, a:c].contiguous(), W[:, a:c].contiguous()
            P = torch.empty(((c - a + 255) // 256, M, K), dtype=torch.float64, device="cuda")
            if c > a:
                cg.carbon_gemm_chunk_values("dx", P, A, B, M, K, c - a, "f32")
        parts.append(P)
    got = host_bits(dp.combine(torch.cat(parts), "f32", bias=b if pass_ == "fwd" else None))
    want, _ = oracle.gemm(pass_, "f32", L["X"] if pass_ == "fwd" else L["dY"], L["W"],
                          L["b"] if pass_ == "fwd" else None, M, K, N)
    assert np.array_equal(got, bits(want))


def test_gpt2_dw_shape_split_over_four_ranks():
    L = inputs.gpt2(42, layers=((768, 3072),))[0]
    M, K, N = L["M"], L["K"], L["N"]
    X, dY = dev(L["X"]), dev(L["dY"])
    got = split_dw(X, dY, M, K, N, "bf16", 4)
    assert np.array_equal(got, single_dw(X, dY, M, K, N, "bf16"))
    rows, cols = inputs.sample_indices(1, K, N, 300)
    want, _ = oracle.gemm_at("dw", "bf16", L["X"], L["dY"], None, M, K, N, rows, cols)
    assert np.array_equal(got[rows, cols], want)


def test_stress_dw_split_over_three_ranks():
    d = inputs.stress_dw(7, M=8192, K=96, N=80)
    M, K, N = d["M"], d["K"], d["N"]
    X, dY = dev(d["X"]), dev(d["dY"])
    got = split_dw(X, dY, M, K, N, "f32", 3)
    want, _ = oracle.gemm("dw", "f32", d["X"], d["dY"], None, M, K, N)
    assert np.array_equal(got, bits(want))
    assert np.array_equal(got, single_dw(X, dY, M, K, N, "f32"))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        L = inputs.gpt2(2024, M=2000, layers=((768, 768),))[0]
        M, K, N = L["M"], L["K"], L["N"]
        lo, hi = dp.token_ranges(M, world)[rank]
        X, dY = dev(L["X"]), dev(L["dY"])
        got = dp.linear_dw_data_parallel(X[lo:hi].contiguous(), dY[lo:hi].contiguous(), M)
        torch.cuda.synchronize()
        ok = cg.carbon_get_device_status() == 0
        same = np.array_equal(host_bits(got), single_dw(X, dY, M, K, N, "bf16"))
        out.put((rank, bool(ok and same)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_processes_on_one_gpu():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert got == [(0, True), (1, True)]
