"""Multi-process paths of bench.py on the CPU (gloo, world size 2).

The layer over one graph is one problem, so N processes run N independent
replicas: the only cross-rank steps are the barriers around the timed region
and the maximum of the ranks' times.  These tests run that host logic with
the gloo backend and launch the reference arm under torchrun, where rank 0
alone prints the JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _max_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ws, r, _ = bench.dist_setup()
    assert (ws, r) == (world, rank)
    bench.barrier(ws)
    # each rank reports its own time; every rank must see the largest
    m = bench.max_over_ranks(10.0 + 5.0 * rank, ws, torch.device("cpu"))
    out[rank] = m
    bench.barrier(ws)
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    with mp.get_context("spawn").Manager() as mgr:   # no fork of a threaded process
        out = mgr.dict()
        mp.spawn(_max_worker, args=(world, free_port(), out), nprocs=world, join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, 1, torch.device("cpu")) == 3.0
    bench.barrier(1)   # no-op


def test_reference_arm_under_torchrun_prints_once():
    """bench.py --impl reference launched as the driver launches N > 1 runs:
    rank 0 prints one line, the other rank exits 0 without output."""
    import oracle
    oracle.build()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py",
           "--impl", "reference", "--config", "1", "--steps", "1", "--warmup", "1", "--gpus", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


@pytest.mark.parametrize("argv", [["--impl", "reference", "--config", "1"]])
def test_bench_arguments_parse(argv):
    sys.path.insert(0, ROOT)
    import bench
    a = bench.parse_args(argv)
    assert a.gpus == 1 and a.steps > 0 and a.warmup >= 3
