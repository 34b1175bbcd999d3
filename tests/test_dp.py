"""The data-parallel weight gradient's host side on CPU ranks (no GPU).

``dp.linear_dw_data_parallel`` splits the tokens on 256-token chunk
boundaries, computes each rank's chunk values, all-gathers them in rank
order and combines them once (Carbon README, "How It Works": all-gather and a
reduction in rank order instead of an all-reduce).  Here two and three gloo
ranks in separate processes run it with stand-ins for the two CUDA steps (a
per-chunk float64 sum and an ordered combine, both plain numpy): the chunks
each rank contributes, the padding of the collective and the rank order must
put every chunk value where the single-device computation has it, so the
combined result equals the stand-in's single-device result bit for bit.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from deterministic_invariant_gemm_fwd_gb300 import dp  # noqa: E402


def test_token_ranges_are_chunk_aligned_and_cover():
    for M in (0, 1, 255, 256, 257, 1000, 8192, 65536, 70000):
        for world in (1, 2, 3, 4, 7, 8):
            rs = dp.token_ranges(M, world)
            assert len(rs) == world
            assert rs[0][0] == 0 and rs[-1][1] == M
            for (a, b), (c, _) in zip(rs, rs[1:]):
                assert b == c                                  # contiguous, rank order
            for a, b in rs:
                assert a <= b and a % 256 == 0
                assert b % 256 == 0 or b == M
            sizes = [(b - a + 255) // 256 for a, b in rs]
            assert max(sizes) - min(sizes) <= 1
            assert sum(sizes) == (M + 255) // 256


def _fake_chunk_values(X, dY, stream=None):
    """Stand-in: per 256-token chunk, a plain float64 sum of x * dy."""
    x = X.numpy().astype(np.float64)
    y = dY.numpy().astype(np.float64)
    m = x.shape[0]
    out = [x[q:q + 256].T @ y[q:q + 256] for q in range(0, m, 256)]
    if not out:
        return torch.zeros((0, x.shape[1], y.shape[1]), dtype=torch.float64)
    return torch.from_numpy(np.stack(out))


def _fake_combine(P, dtype, bias=None, stream=None):
    """Stand-in: left-to-right float64 sum over chunks, to float32."""
    acc = np.zeros(P.shape[1:], dtype=np.float64)
    for q in range(P.shape[0]):
        acc = acc + P[q].numpy()
    return torch.from_numpy(acc.astype(np.float32))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, M, K, N, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(5)
        X = rng.standard_normal((M, K)).astype(np.float32)
        dY = rng.standard_normal((M, N)).astype(np.float32)
        lo, hi = dp.token_ranges(M, world)[rank]
        got = dp.linear_dw_data_parallel(torch.from_numpy(X[lo:hi].copy()),
                                         torch.from_numpy(dY[lo:hi].copy()), M,
                                         chunk_values_fn=_fake_chunk_values,
                                         combine_fn=_fake_combine)
        want = _fake_combine(_fake_chunk_values(torch.from_numpy(X), torch.from_numpy(dY)), "f32")
        out.put((rank, bool(np.array_equal(got.numpy().view(np.uint32),
                                           want.numpy().view(np.uint32)))))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,M", [(2, 1000), (3, 700), (2, 200)])
def test_gloo_ranks_gather_chunk_values_in_order(world, M):
    """(2, 1000): ranks of 2 chunks each, the last one ragged; (3, 700): 3
    chunks over 3 ranks; (2, 200): one chunk, rank 1 holds no tokens."""
    K, N = 5, 7
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, M, K, N, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(r, True) for r in range(world)]


def test_token_ranges_reject_bad_sizes():
    with pytest.raises(ValueError):
        dp.token_ranges(-1, 2)
    with pytest.raises(ValueError):
        dp.token_ranges(10, 0)
