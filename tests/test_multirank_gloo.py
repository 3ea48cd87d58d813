"""Multi-rank host logic of bench.py on CPU with the gloo backend (world size 2): rank
set-up from the torchrun environment, the max of the per-rank time over ranks, and the
whole-job throughput (units of all ranks over the slowest rank's time)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier()
    elapsed = 2.0 if rank == 0 else 3.0          # seconds; rank 1 is the slow one
    worst = bench.max_over_ranks(elapsed)
    value = bench.aggregate_throughput(100.0, w, worst)
    q.put((rank, worst, value))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_all_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, worst, value in res:
        assert worst == 3.0
        assert value == pytest.approx(100.0 * 2 / 3.0)


def test_single_process_needs_no_group():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    assert bench.max_over_ranks(1.5) == 1.5
    assert bench.aggregate_throughput(10.0, 1, 2.0) == 5.0
