"""The benchmark's multi-rank path on CPU: two gloo ranks in separate
processes, the way torchrun starts one process per GPU.

Each rank runs its own replica of the step (weak scaling, no collective on
the data path); the only collective is the max of the ranks' step times, and
the whole-job throughput is world x the per-rank flops over that time.  The
reference arm runs on rank 0 alone.  No GPU is needed.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")

import bench  # noqa: E402


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        ms = bench.max_over_ranks(times[rank], dist, "cpu")
        out.put((r, w, local, ms, bench.whole_job_gflops(2.0e12, w, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [12.5, 20.0]
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, w, local, ms, gflops) in enumerate(got):
        assert (r, w, local) == (rank, 2, rank)
        assert ms == max(times)
        assert gflops == pytest.approx(2 * 2.0e12 / (max(times) * 1e-3) / 1e9)


def test_single_process_is_its_own_max():
    assert bench.max_over_ranks(7.25) == 7.25
    assert bench.whole_job_gflops(1.0e12, 1, 10.0) == pytest.approx(1.0e5)


def test_reference_arm_prints_on_rank_zero_only(capsys):
    class Args:
        steps, warmup, gpus = 1, 3, 2
    assert bench.reference_arm(Args, 2, 1) is None
    assert capsys.readouterr().out == ""


def test_recorded_traffic_needs_matching_sources(tmp_path, monkeypatch):
    """A traffic figure is reported only with the hash of the kernel's
    sources it was taken on."""
    files = bench.KERNEL_SOURCES["exact_tc_kernel"]
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "k.md").write_text(
        f"traffic exact_tc_kernel bytes_per_launch=1234 sources_sha256={bench.sources_sha256(files)}\n"
        "traffic tc_tier bytes_per_launch=99 sources_sha256=0000\n")
    csrc = os.path.join(bench.ROOT, "deterministic_invariant_gemm_fwd_gb300", "csrc")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "deterministic_invariant_gemm_fwd_gb300").mkdir()
    os.symlink(csrc, tmp_path / "deterministic_invariant_gemm_fwd_gb300" / "csrc")
    assert bench.recorded_traffic("exact_tc_kernel") == 1234
    assert bench.recorded_traffic("tc_tier") is None
    assert bench.recorded_traffic("missing") is None
    # one changed byte in one of the kernel's files changes the hash
    assert bench.sources_sha256(files, lambda n: b"x") != bench.sources_sha256(files)
