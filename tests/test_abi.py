"""The C-ABI library on a machine without a GPU: it loads, exports every
function its headers declare, and rejects bad arguments before touching the
device."""
import ctypes
import os

import pytest

from deterministic_invariant_gemm_fwd_gb300 import _binding as b

INVALID, UNSUPPORTED, MISALIGNED = 1, 2, 3


def test_every_declared_symbol_is_exported():
    names = b.declared_functions()
    for must in ("carbon_gemm_fwd", "carbon_gemm_dx", "carbon_gemm_dw",
                 "carbon_get_device_status", "carbon_status_string",
                 "carbon_abi_version"):
        assert must in names
    raw = ctypes.CDLL(b.LIB_PATH)
    for name in names:
        assert hasattr(raw, name), name


def test_abi_version_and_status_names():
    assert b.carbon_abi_version() == (1 << 16) | 2    # minor 2: superacc tier, chunk values
    for code, name in b.STATUS.items():
        assert b.carbon_status_string(code) == name


FAKE = 0x1000   # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("fn", ["fwd", "dx", "dw"])
def test_negative_sizes_rejected(fn):
    for M, K, N in ((-1, 2, 3), (2, -1, 3), (2, 3, -1)):
        if fn == "fwd":
            st = b.lib.carbon_gemm_fwd(FAKE, FAKE, FAKE, None, M, K, N, 0, 0, None)
        elif fn == "dx":
            st = b.lib.carbon_gemm_dx(FAKE, FAKE, FAKE, M, K, N, 0, 0, None)
        else:
            st = b.lib.carbon_gemm_dw(FAKE, FAKE, FAKE, M, K, N, 0, 0, None)
        assert st == INVALID


def test_overflowing_sizes_rejected():
    big = 1 << 40
    assert b.lib.carbon_gemm_fwd(FAKE, FAKE, FAKE, None, big, big, 4, 0, 0, None) == INVALID
    assert b.lib.carbon_gemm_dw(FAKE, FAKE, FAKE, 4, big, 1 << 30, 0, 0, None) == INVALID


def test_bad_dtype_and_tier_rejected():
    assert b.lib.carbon_gemm_fwd(FAKE, FAKE, FAKE, None, 2, 3, 4, 7, 0, None) == INVALID
    assert b.lib.carbon_gemm_fwd(FAKE, FAKE, FAKE, None, 2, 3, 4, 0, 9, None) == INVALID
    assert b.lib.carbon_debug_exact_y64(5, FAKE, FAKE, FAKE, None, 2, 3, 4, 0, None) == INVALID


def test_tc_tier_rejects_f32():
    assert b.lib.carbon_gemm_fwd(FAKE, FAKE, FAKE, None, 2, 8, 8, 0, 1, None) == UNSUPPORTED


def test_null_pointers_rejected():
    assert b.lib.carbon_gemm_fwd(None, FAKE, FAKE, None, 2, 3, 4, 0, 0, None) == INVALID
    assert b.lib.carbon_gemm_fwd(FAKE, None, FAKE, None, 2, 3, 4, 0, 0, None) == INVALID
    assert b.lib.carbon_gemm_dx(FAKE, FAKE, None, 2, 3, 4, 0, 0, None) == INVALID
    assert b.lib.carbon_gemm_dw(FAKE, None, FAKE, 2, 3, 4, 1, 0, None) == INVALID


def test_empty_outputs_are_a_no_op():
    # no output elements: OK without touching the device or any pointer
    assert b.lib.carbon_gemm_fwd(None, None, None, None, 0, 3, 4, 0, 0, None) == 0
    assert b.lib.carbon_gemm_fwd(None, None, None, None, 5, 3, 0, 1, 0, None) == 0
    assert b.lib.carbon_gemm_dx(None, None, None, 5, 0, 4, 0, 0, None) == 0
    assert b.lib.carbon_gemm_dw(None, None, None, 5, 0, 4, 0, 0, None) == 0


def test_debug_round_validation():
    assert b.lib.carbon_debug_round(3, FAKE, FAKE, 4, None) == INVALID
    assert b.lib.carbon_debug_round(0, None, FAKE, 4, None) == INVALID
    assert b.lib.carbon_debug_round(0, None, None, 0, None) == 0
    assert b.lib.carbon_debug_timeout_probe(0, None) == INVALID


def test_import_maps_no_cuda_library():
    """Importing the package and the input generator loads no CUDA code: the
    library is mapped on the first call only (so the oracle-only benchmark
    arm never loads it)."""
    import subprocess
    import sys
    code = ("import deterministic_invariant_gemm_fwd_gb300, seeded_inputs\n"
            "maps = open('/proc/self/maps').read()\n"
            "assert 'libcarbon_gemm' not in maps, 'library mapped at import'\n"
            "from deterministic_invariant_gemm_fwd_gb300 import _binding\n"
            "_binding.carbon_abi_version()\n"
            "assert 'libcarbon_gemm' in open('/proc/self/maps').read()\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    subprocess.run([sys.executable, "-c", code], check=True, cwd=root)


def test_superacc_tier_argument_checks():
    SUPERACC = 2
    # accepted as a tier: argument errors still come first, empty outputs are no-ops
    assert b.lib.carbon_gemm_fwd(FAKE, FAKE, FAKE, None, -1, 3, 4, 0, SUPERACC, None) == INVALID
    assert b.lib.carbon_gemm_dw(None, None, None, 5, 0, 4, 2, SUPERACC, None) == 0
    assert b.lib.carbon_gemm_dx(FAKE, None, FAKE, 2, 3, 4, 1, SUPERACC, None) == INVALID
    # no fp32 staging variant of the weight gradient on this tier
    assert b.lib.carbon_gemm_dw_f32(FAKE, FAKE, FAKE, 16, 16, 16, SUPERACC, None) == UNSUPPORTED
    assert b.lib.carbon_gemm_fwd(FAKE, FAKE, FAKE, None, 2, 3, 4, 0, 3, None) == INVALID


def test_bounds_checked_library_exports_the_same_symbols():
    """build() also builds the bounds-checked library (CARBON_DEBUG_BOUNDS)."""
    path = os.path.join(os.path.dirname(b.LIB_PATH), "libcarbon_gemm_bounds.so")
    if not os.path.exists(path):
        pytest.skip("bounds-checked library not built")
    raw = ctypes.CDLL(path)
    for name in b.declared_functions():
        assert hasattr(raw, name), name
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    raw.carbon_gemm_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, i32, vp]
    raw.carbon_gemm_fwd.restype = i32
    assert raw.carbon_gemm_fwd(None, None, None, None, 0, 3, 4, 0, 0, None) == 0
    assert raw.carbon_gemm_fwd(None, None, None, None, -1, 3, 4, 0, 0, None) == INVALID
