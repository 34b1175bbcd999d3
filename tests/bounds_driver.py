"""Runs the library's GEMMs on shapes that drive its index arithmetic to the
edges and checks, after every call, that no kernel skipped an access out of
range (CARBON_ERR_OUT_OF_BOUNDS) and that the results equal the oracle's.
Meant for the bounds-checked build: run it as
``CARBON_GEMM_LIBRARY=.../libcarbon_gemm_bounds.so python -m tests.bounds_driver``
(tests/test_bounds_gpu.py does).  Prints one line per case and "ok" at the
end; exits non-zero on the first failure."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import seeded_inputs as inputs  # noqa: E402
from tests.gpu_util import bits, dev, host_bits, torch_dtype  # noqa: E402


def main():
    import torch
    import deterministic_invariant_gemm_fwd_gb300 as cg
    from deterministic_invariant_gemm_fwd_gb300 import _binding

    lib = os.environ.get("CARBON_GEMM_LIBRARY", "")
    assert _binding.LIB_PATH == lib and lib, "CARBON_GEMM_LIBRARY must name the library under test"

    def run(tier, pass_, dtype, L, M, K, N, with_bias=True):
        f16 = dtype == "f16"
        A, B, bias = {"fwd": (L["X"], L["W"], L["b"] if with_bias else None),
                      "dx": (L["dY"], L["W"], None), "dw": (L["X"], L["dY"], None)}[pass_]
        tA, tB = dev(A, f16=f16), dev(B, f16=f16)
        tb = dev(bias, f16=f16) if bias is not None else None
        out = torch.empty(oracle.out_shape(pass_, M, K, N), dtype=torch_dtype(dtype), device="cuda")
        {"fwd": lambda: cg.carbon_gemm_fwd(out, tA, tB, tb, M, K, N, dtype, tier),
         "dx": lambda: cg.carbon_gemm_dx(out, tA, tB, M, K, N, dtype, tier),
         "dw": lambda: cg.carbon_gemm_dw(out, tA, tB, M, K, N, dtype, tier)}[pass_]()
        st = cg.carbon_get_device_status()
        assert st == 0, f"{tier} {pass_} {dtype} {M}x{K}x{N}: {cg.carbon_status_string(st)}"
        got = host_bits(out)
        if tier == "exact":
            want = bits(oracle.gemm(pass_, dtype, A, B, bias, M, K, N)[0])
        elif tier == "superacc":
            want = bits(oracle.gemm_superacc(pass_, dtype, A, B, bias, M, K, N))
        else:
            return                                      # TC tier: the status is what is checked here
        assert np.array_equal(got, want), f"{tier} {pass_} {dtype} {M}x{K}x{N}: mismatch"

    shapes = [(1, 1, 1), (7, 255, 3), (129, 256, 65), (1, 257, 65), (7, 513, 1), (3, 0, 5),
              (129, 1, 3), (33, 31, 33), (300, 700, 190), (1100, 64, 136)]
    for (M, K, N) in shapes:
        rng = np.random.default_rng(M * 7 + K * 3 + N)
        for dtype in ("f32", "bf16", "f16"):
            L = inputs.linear_layer(rng, M, K, N, dtype, 1e-3)
            for tier in ("exact", "superacc", "tc"):
                if tier == "tc" and (dtype == "f32" or K % 8 or N % 8):
                    continue
                for pass_ in ("fwd", "dx", "dw"):
                    run(tier, pass_, dtype, L, M, K, N)
                run(tier, "fwd", dtype, L, M, K, N, with_bias=False)
        print("shape", M, K, N, "ok", flush=True)
    # GPT-2 shapes at a reduced batch (row order groups, pieces, run-time units)
    for L in inputs.gpt2(7, M=1100):
        M, K, N = L["M"], L["K"], L["N"]
        for tier in ("exact", "superacc", "tc"):
            for pass_ in ("fwd", "dx", "dw"):
                run(tier, pass_, "bf16", L, M, K, N)
        print("gpt2", K, N, "ok", flush=True)
    # chunk repairs and fix-ups: tiny entries (lines too wide for the digit
    # planes), a row whose sums leave the 64-bit grain, inf
    rng = np.random.default_rng(12)
    M, K, N = 200, 520, 100
    L = inputs.linear_layer(rng, M, K, N, "bf16", 1e-3)
    X = inputs.bf16_bits_to_f32(L["X"]).copy()
    X[[3, 77, 150], [10, 300, 511]] = np.float32(2.0 ** -40)
    X[5, :256] = np.float32(2.0 ** -90)
    X[5, 256:] = np.float32(2.0 ** 60)
    X[9, 17] = np.float32(np.inf)
    L["X"] = inputs.f32_to_bf16_bits(X)
    for tier in ("exact", "superacc"):
        for pass_ in ("fwd", "dw"):
            try:
                run(tier, pass_, "bf16", L, M, K, N)
            except AssertionError as e:
                if "mismatch" not in str(e):
                    raise                               # NaN patterns may differ; the status may not
    print("repairs and fix-ups ok", flush=True)
    # split reductions: chunk values and their combine
    from deterministic_invariant_gemm_fwd_gb300 import dp
    rng = np.random.default_rng(3)
    M, K, N = 1100, 70, 45
    L = inputs.linear_layer(rng, M, K, N, "f32", 1e-3)
    X, dY = dev(L["X"]), dev(L["dY"])
    parts = [dp.chunk_values(X[a:b].contiguous(), dY[a:b].contiguous()) for a, b in dp.token_ranges(M, 3)]
    out = dp.combine(torch.cat(parts), "f32")
    assert cg.carbon_get_device_status() == 0
    assert np.array_equal(host_bits(out), bits(oracle.gemm("dw", "f32", L["X"], L["dY"], None, M, K, N)[0]))
    print("split reductions ok", flush=True)
    print("ok")


if __name__ == "__main__":
    main()
