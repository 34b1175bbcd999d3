"""The public headers are plain C and the library is usable from a C program:
tests/c/abi_from_c.c is compiled with gcc as C99 against include/*.h, linked
against the in-tree libcarbon_gemm.so and run.  It exercises only paths that
answer without a GPU (versions, status strings, argument errors, fault
injection)."""
import os
import shutil
import subprocess

import pytest

from deterministic_invariant_gemm_fwd_gb300 import _binding as b

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_uses_the_abi(tmp_path):
    exe = tmp_path / "abi_from_c"
    libdir = os.path.dirname(b.LIB_PATH)
    cmd = ["gcc", "-std=c99", "-D_POSIX_C_SOURCE=200112L", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c", "abi_from_c.c"),
           "-o", str(exe), f"-L{libdir}", "-l:libcarbon_gemm.so", f"-Wl,-rpath,{libdir}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    env = dict(os.environ)
    env.pop("CARBON_FAULT", None)
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
