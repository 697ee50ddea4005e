"""The benchmark's multi-rank logic on CPU ranks (gloo, world size 2): every rank projects its
own batch of rows against its own replica of W (no collective on the data path); the
timing is the maximum over ranks and the value counts the rows of all ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = [0.25, 0.31][rank]
        mx = bench.max_over_ranks(ms, "cpu")
        q.put((rank, mx, bench.job_rows_per_s(world, 16, mx), bench.rank_rows_seed(rank)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_all_rows():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [0.31, 0.31]
    assert res[0][2] == pytest.approx(2 * 16 / 0.31e-3)
    assert res[0][3] != res[1][3]  # each rank draws its own batch of rows


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(1.5, "cpu") == 1.5
    assert bench.job_rows_per_s(1, 16, 0.25) == pytest.approx(64000.0)
