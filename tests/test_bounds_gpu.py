"""The bounds-checked build on the GPU: the same GEMMs as the regular build,
every global-memory access the kernels index themselves checked against its
buffer (CARBON_DEBUG_BOUNDS; an access out of range is skipped and reported
as CARBON_ERR_OUT_OF_BOUNDS).  Edge shapes, all tiers, passes and dtypes,
GPT-2 shapes at a reduced batch, repair and fix-up paths and split
reductions must run with a clean status and give the oracle's bits.  The
driver runs in a child process so that it loads the bounds-checked library
instead of the regular one."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "deterministic_invariant_gemm_fwd_gb300", "libcarbon_gemm_bounds.so")


def test_bounds_checked_build_runs_clean():
    assert os.path.exists(LIB), "build() builds the bounds-checked library"
    env = dict(os.environ, CARBON_GEMM_LIBRARY=LIB)
    r = subprocess.run([sys.executable, "-m", "tests.bounds_driver"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert r.stdout.strip().endswith("ok")
