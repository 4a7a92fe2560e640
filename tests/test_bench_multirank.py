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


def test_reference_arm_json_line(capsys):
    """The reference arm (the oracle on host cores) prints one JSON line with
    the contract's keys, its own cpu_baseline and a zero-copy e2e."""
    import json

    sys.path.insert(0, ROOT)
    import bench

    rc = bench.run_reference(bench.parse_args(["--impl", "reference", "--workload", "tiny",
                                               "--steps", "2", "--warmup", "3"]))
    assert rc == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_cpu_model_is_reported():
    sys.path.insert(0, ROOT)
    import bench

    m = bench.cpu_model()
    assert isinstance(m, str) and m and m != "unknown"


def test_batch_override_reduces_the_workload():
    import bench

    wl = bench.make_workload(bench.parse_args(["--bs", "16", "--quant-mode", "0"]))
    assert wl.cfg["max_bs"] == 16 and wl.cfg["quant_mode"] == 0
    assert wl.x.shape[:2] == (32, 16)
    with pytest.raises(SystemExit):
        bench.make_workload(bench.parse_args(["--workload", "perf8", "--bs", "16"]))


def test_kernels_per_step_follows_the_dispatch_path():
    """The launch count the bench line claims: two kernels for a batch small
    enough for the one-kernel dispatch, four (five with per-expert smooth
    rows) otherwise."""
    import bench
    import combine_quant_gb300 as cq
    from combine_quant_gb300 import build as cqbuild
    from combine_quant_gb300 import workloads

    cqbuild.build()  # the decision is the library's (cq_dispatch_one_kernel, host only)

    def n(wl):
        cfg = cq.Config.from_dict(wl.cfg)
        return bench.kernels_per_step(cfg, wl.smooth is not None and cfg.quant_mode in (1, 2, 3))

    assert n(workloads.tiny()) == 2 and n(workloads.perf_table(8)) == 2
    assert n(workloads.dsv3()) == 4 and n(workloads.special()) == 4
    assert n(workloads.skew()) == 5
    assert n(workloads.mxfp8(W=4, BS=8, M=16, K=4, H=1024)) == 2
    # the one-kernel dispatch's limits: 2048 (token, slot) pairs, and with one
    # smooth row per expert 2^23 values quantised row by row
    assert n(workloads.perf_table(32)) == 2 and n(workloads.perf_table(64)) == 4
    assert n(workloads.skew(BS=4)) == 2 and n(workloads.skew(BS=8)) == 5
