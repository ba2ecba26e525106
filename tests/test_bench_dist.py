"""The multi-process (N > 1) host logic of bench.py on CPU with gloo."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world)})
    sys.path.insert(0, ROOT)
    import torch.distributed as tdist
    import bench
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    out[rank] = bench.max_over_ranks(1.5 + rank)
    tdist.barrier()
    tdist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, 29611, out), nprocs=world, join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25


def test_reference_arm_two_ranks_prints_one_line():
    """Under torchrun the oracle reference arm runs on rank 0 only; the other
    rank exits 0 without work and exactly one JSON line is printed."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", "29613", "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "2", "--warmup", "3", "--ref-budget-s", "0.2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
