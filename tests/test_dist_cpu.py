"""Replica-mode multi-process logic of bench.py on CPU (gloo, world size 2).

The method's per-step path has no data exchange between GPUs: N ranks are N
independent replicas, each timing its own steps.  What the N>1 path adds is
host-side: process-group set-up, a barrier around the timed region, the
maximum of the elapsed times over ranks, the whole-job throughput built from
it, and rank 0 alone printing the result line."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, elapsed: list, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    try:
        r, w = bench.dist_init("gloo")
        bench.barrier()
        value, slowest = bench.aggregate(elapsed[rank], 1000.0, w)
        q.put((r, w, value, slowest))
    finally:
        import torch.distributed as dist

        if dist.is_initialized():
            dist.destroy_process_group()


def test_aggregate_takes_the_slowest_rank():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    elapsed = [0.5, 2.0]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, elapsed, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, world, value, slowest) in enumerate(out):
        assert (rank, world) == (r, 2)
        assert slowest == 2.0                    # max over ranks, seen by every rank
        assert value == pytest.approx(2 * 1000.0 / 2.0)   # all ranks' units / slowest time


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    value, slowest = bench.aggregate(0.25, 10.0, 1)
    assert (value, slowest) == (40.0, 0.25)


def test_torchrun_two_ranks_print_one_line():
    """The reference arm under torchrun: rank 0 alone works and prints."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env={**os.environ, "OMP_NUM_THREADS": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 2
    assert d["value"] > 0 and d["unit"] == "layers/s"
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
