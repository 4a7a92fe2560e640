"""The N > 1 path of bench.py on CPU: two gloo ranks run independent
replicas; the job value is all ranks' units over the slowest rank's time, and
the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local_ms = [100.0, 250.0][rank]  # rank 1 is the slow one
    value, slowest = bench.job_throughput(local_ms, units_per_rank=4096, steps=10, dist=dist)
    rc = bench.run_reference(bench.parse_args(["--impl", "reference"])) if rank == 1 else None
    out.put((rank, value, slowest, rc))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_and_reference_rank_gating():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        rank, value, slowest, rc = q.get(timeout=120)
        res[rank] = (value, slowest, rc)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        value, slowest, _ = res[rank]
        assert slowest == 250.0  # max over ranks
        assert value == pytest.approx(2 * 4096 * 10 / 0.25)
    assert res[1][2] == 0  # non-zero ranks of the reference arm exit 0 without work


def test_single_process_throughput():
    sys.path.insert(0, ROOT)
    import bench

    value, slowest = bench.job_throughput(50.0, 100, 4)
    assert slowest == 50.0 and value == pytest.approx(100 * 4 / 0.05)
