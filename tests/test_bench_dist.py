"""The multi-rank path of bench.py on CPU: world-size-2 gloo ranks run the
same timing aggregation the GPU ranks use (max over ranks, whole-job rows/s).
Rows are independent, so ranks are replicas and exchange nothing else."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    dist = bench.init_dist(world, "gloo")
    try:
        seconds = [0.5, 0.8][rank]
        mx = bench.reduce_max(dist, seconds)
        value = bench.aggregate_rows_per_s(32, world, mx)
        dist.barrier()
        q.put((rank, mx, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("rank hung")
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, mx, value in got:
        assert mx == 0.8
        assert value == pytest.approx(32 * 2 / 0.8)


def test_single_process_needs_no_group():
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.reduce_max(None, 1.5) == 1.5
    assert bench.aggregate_rows_per_s(10, 1, 0.5) == 20.0
