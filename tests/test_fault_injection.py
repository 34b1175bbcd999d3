"""Host-side fault injection (CARBON_FAULT=launch): the GEMM entry points fail
after their argument checks with CARBON_ERR_CUDA, as a failed launch would,
without touching any device, so a caller's error handling can be tested on
a machine without a GPU.  No GPU is faulted; the fake pointers below are
never dereferenced."""
import pytest

import deterministic_invariant_gemm_fwd_gb300 as cg
from deterministic_invariant_gemm_fwd_gb300 import _binding as b

FAKE = 0x1000
CUDA_ERR, INVALID = 4, 1


@pytest.fixture
def injected(monkeypatch):
    monkeypatch.setenv("CARBON_FAULT", "other,launch")
    yield


@pytest.mark.parametrize("fn", ["fwd", "dx", "dw"])
@pytest.mark.parametrize("tier", ["exact", "tc"])
def test_injected_launch_failure_is_reported(injected, fn, tier):
    call = {"fwd": lambda: cg.carbon_gemm_fwd(FAKE, FAKE, FAKE, None, 16, 16, 16, "bf16", tier, 0),
            "dx": lambda: cg.carbon_gemm_dx(FAKE, FAKE, FAKE, 16, 16, 16, "bf16", tier, 0),
            "dw": lambda: cg.carbon_gemm_dw(FAKE, FAKE, FAKE, 16, 16, 16, "bf16", tier, 0)}[fn]
    with pytest.raises(cg.CarbonError) as err:
        call()
    assert err.value.status == CUDA_ERR
    assert "injected launch failure" in str(err.value)
    assert "CARBON_FAULT" in b.lib.carbon_last_cuda_error().decode()


def test_argument_errors_and_empty_outputs_come_first(injected):
    # a bad size is still INVALID_ARG, an empty output still succeeds
    assert b.lib.carbon_gemm_fwd(FAKE, FAKE, FAKE, None, -1, 16, 16, 1, 0, None) == INVALID
    assert b.lib.carbon_gemm_fwd(FAKE, FAKE, FAKE, None, 0, 16, 16, 1, 0, None) == 0


def test_only_the_named_fault_is_injected(monkeypatch):
    monkeypatch.setenv("CARBON_FAULT", "launchpad,lunch")
    # no injection: on a machine without a GPU the call now fails at the
    # device query with a real CUDA error, not the injected one; with a GPU
    # it would run, so only the message is checked where there is none
    import torch
    if torch.cuda.is_available():
        pytest.skip("without injection this call would reach the device")
    st = b.lib.carbon_gemm_fwd(FAKE, FAKE, FAKE, None, 16, 16, 16, 1, 0, None)
    assert st != 0
    assert "injected" not in b.lib.carbon_last_cuda_error().decode()


@pytest.mark.parametrize("tier", ["exact", "tc"])
def test_dw_f32_injected_failure_is_reported(injected, tier):
    with pytest.raises(cg.CarbonError) as err:
        cg.carbon_gemm_dw_f32(FAKE, FAKE, FAKE, 16, 16, 16, tier, 0)
    assert err.value.status == CUDA_ERR and "injected launch failure" in str(err.value)


def test_dw_f32_argument_errors():
    assert b.lib.carbon_gemm_dw_f32(FAKE, FAKE, FAKE, -1, 16, 16, 0, None) == INVALID
    assert b.lib.carbon_gemm_dw_f32(FAKE, FAKE, FAKE, 16, 16, 16, 9, None) == INVALID
    assert b.lib.carbon_gemm_dw_f32(None, FAKE, FAKE, 16, 16, 16, 0, None) == INVALID
    assert b.lib.carbon_gemm_dw_f32(FAKE, FAKE, FAKE, 16, 0, 16, 0, None) == 0     # empty output


def test_noalloc_injected_failure_is_reported(injected):
    st = b.lib.carbon_gemm_exact_bf16_noalloc(0, FAKE, FAKE, FAKE, None, 16, 16, 16, None)
    assert st == CUDA_ERR
    assert "CARBON_FAULT" in b.lib.carbon_last_cuda_error().decode()


def test_noalloc_argument_errors_and_limit_come_first(injected):
    SCRATCH_LIMIT = 6
    assert b.lib.carbon_gemm_exact_bf16_noalloc(0, FAKE, FAKE, FAKE, None, -1, 16, 16, None) == INVALID
    assert b.lib.carbon_gemm_exact_bf16_noalloc(3, FAKE, FAKE, FAKE, None, 16, 16, 16, None) == INVALID
    assert b.lib.carbon_gemm_exact_bf16_noalloc(0, None, FAKE, FAKE, None, 16, 16, 16, None) == INVALID
    # byte counts that overflow int64
    big = 1 << 31
    assert b.lib.carbon_gemm_exact_bf16_noalloc(0, FAKE, FAKE, FAKE, None, big, big, 4, None) == INVALID
    # beyond the fixed workspace: rejected before the injected failure
    assert b.lib.carbon_gemm_exact_bf16_noalloc(
        0, FAKE, FAKE, FAKE, None, 8192, 3072, 768, None) == SCRATCH_LIMIT
    assert b.lib.carbon_gemm_exact_bf16_noalloc(0, FAKE, FAKE, FAKE, None, 0, 16, 16, None) == 0


def test_chunk_value_entry_points_injected_failure(injected):
    assert b.lib.carbon_gemm_chunk_values(2, FAKE, FAKE, FAKE, 300, 16, 16, 1, None) == CUDA_ERR
    assert b.lib.carbon_chunk_values_combine(FAKE, FAKE, 2, 16, 16, None, 1, None) == CUDA_ERR
    # argument errors first, empty outputs are no-ops
    assert b.lib.carbon_gemm_chunk_values(5, FAKE, FAKE, FAKE, 300, 16, 16, 1, None) == INVALID
    assert b.lib.carbon_gemm_chunk_values(2, None, FAKE, FAKE, 300, 16, 16, 1, None) == INVALID
    assert b.lib.carbon_chunk_values_combine(FAKE, None, 2, 16, 16, None, 1, None) == INVALID
    assert b.lib.carbon_chunk_values_combine(FAKE, FAKE, -1, 16, 16, None, 1, None) == INVALID
    assert b.lib.carbon_chunk_values_combine(None, None, 2, 0, 16, None, 1, None) == 0
