"""The N > 1 path of bench.py on the CPU: two gloo ranks (no GPU).

bench.py runs one process per GPU and scales by replicas only (every rank runs
the whole workload; there is no data-path exchange). What crosses ranks is the
timing protocol: a barrier around the timed region, the maximum elapsed time
over ranks, and the job's images/s from all ranks' images over that time. The
reference arm under torchrun runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    bench.init_dist(world, rank)
    try:
        assert dist.get_backend() == "gloo"
        bench.barrier(world)
        # each rank "timed" a different duration: everyone gets the slowest
        m = bench.allreduce_max(1.0 + rank, world)
        value, s_max = bench.weak_scaling_value(1000, 2.0 if rank == 0 else 4.0, world)
        q.put((rank, m, value, s_max))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_timing_protocol_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, m, value, s_max in res:
        assert m == 2.0                       # max over ranks of 1 + rank
        assert s_max == 4.0                   # the slowest rank's time
        assert value == pytest.approx(2 * 1000 / 4.0)   # all ranks' images over that time


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    bench.init_dist(1, 0)
    bench.barrier(1)
    assert bench.allreduce_max(3.5, 1) == 3.5
    assert bench.weak_scaling_value(100, 0.5, 1) == (200.0, 0.5)


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_once_from_rank_zero():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3", "--config", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, OMP_NUM_THREADS="4"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2 and out["value"] > 0
    assert out["cpu_baseline"]["kind"] == "oracle"
