"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the replicas
path has no data-path collective, only the max of the step times over ranks,
and the reference arm runs on rank 0 alone."""
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _max_worker(rank, world, port, values, out):
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(values[rank], dist, torch.device("cpu"))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    values = [1.25, 3.5]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_max_worker, args=(2, _free_port(), values, out), nprocs=2, join=True)
        assert dict(out) == {0: 3.5, 1: 3.5}


def test_max_over_ranks_without_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(2.0, None, torch.device("cpu")) == 2.0


@pytest.mark.timeout(600)
def test_reference_arm_two_ranks_prints_one_line():
    """torchrun with 2 CPU ranks: rank 0 times the oracle and prints one JSON
    line, rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
