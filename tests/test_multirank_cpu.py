"""The bench's multi-rank path on the CPU: two gloo ranks (no GPU), each with
its own replica time; the job's time per step is the slowest rank's and its
throughput counts every rank's bytes (weak scaling, no collective on the data
path)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = [0.250, 0.262][rank]  # rank 1 is the slower replica
        dist.barrier()
        ms_max = bench.max_over_ranks(ms, "cpu", world)
        results[rank] = (ms_max, bench.job_throughput_gbs(1_638_400_000, world, ms_max))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        got = dict(results)
    assert got[0][0] == pytest.approx(0.262) and got[1][0] == pytest.approx(0.262)
    assert got[0][1] == pytest.approx(2 * 1_638_400_000 / 0.262e-3 / 1e9)
    assert got[0] == got[1]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(0.3, "cpu", 1) == 0.3
    assert bench.job_throughput_gbs(1000, 1, 1.0) == pytest.approx(1e-3)


def test_reference_arm_under_two_ranks_prints_one_line():
    """bench.py --impl reference under torchrun with two ranks on the CPU: rank 0
    alone times the oracle and prints the one JSON line (carrying the launch's
    N); the other rank exits 0 without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny_d64", "--steps", "1", "--warmup", "3",
           "--reference-budget-s", "2"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
