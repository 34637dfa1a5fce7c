"""The multi-rank side of bench.py, on CPU with the gloo backend.

The decode path shards by sequence: every rank holds its own replica of the
workload and no collective runs on the data path.  What does cross ranks is
the timing: the whole-job value is the units all ranks processed divided by
the slowest rank's time.  These tests run that aggregation in two gloo
ranks, and launch the reference arm under torchrun with two ranks (rank 0
alone does the work and prints the one JSON line)."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, per_rank, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    bench.dist_init(world, "gloo")
    t_ms, units = per_rank[rank]
    bench.barrier(world)
    value, t_max = bench.aggregate(t_ms, units, world)
    q.put((rank, value, t_max))
    dist.destroy_process_group()


def run_ranks(per_rank):
    world = len(per_rank)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, per_rank, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return sorted(q.get(timeout=5) for _ in range(world))


def test_aggregate_two_ranks_max_time_sum_units():
    # rank 1 is slower and did more work: value = (1000 + 3000) / 0.2 s
    res = run_ranks([(100.0, 1000.0), (200.0, 3000.0)])
    for rank, value, t_max in res:
        assert t_max == pytest.approx(200.0)
        assert value == pytest.approx(4000.0 / 0.2)


def test_aggregate_single_rank_is_local():
    sys.path.insert(0, ROOT)
    import bench
    value, t_max = bench.aggregate(50.0, 500.0, 1)
    assert (value, t_max) == (pytest.approx(10000.0), 50.0)


def test_reference_arm_under_torchrun_two_ranks():
    """Only rank 0 runs the oracle and prints; rank 1 exits 0 without work."""
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "tiny", "--steps", "1", "--warmup", "0",
           "--cpu-tokens", "2000"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
