"""Host-side multi-rank logic of bench.py on CPU (gloo, world size 2).

The path shards by sequences with no collective on the data path; the only cross-rank steps are
the barriers around the timed region and the final reduction (units summed, time maxed), which
these tests run as real gloo process groups on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _aggregate_worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    bench.dist_init(world, "gloo")
    bench.barrier(world)
    units, secs = bench.aggregate(1000.0 * (rank + 1), 0.25 * (rank + 1), world)
    bench.barrier(world)
    out[rank] = (units, secs)
    torch.distributed.destroy_process_group()


def test_aggregate_sums_units_and_takes_slowest_rank():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_aggregate_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        got = dict(out)
    # units: 1000 + 2000; time: max(0.25, 0.5); every rank sees the same whole-job numbers
    assert got == {0: (3000.0, 0.5), 1: (3000.0, 0.5)}


def test_single_rank_aggregate_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(123.0, 4.5, 1) == (123.0, 4.5)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--config", "1",
           "--steps", "2", "--warmup", "3", "--ref-budget", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
