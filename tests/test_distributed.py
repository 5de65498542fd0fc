"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

The attention path shards by (sequence, KV head) with no exchange, so several GPUs run
independent replicas; what needs checking without GPUs is the job-level reduction (the slowest
rank sets the time) and that only rank 0 reports.
"""
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


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    v = bench.max_over_ranks(1.5 + rank, world, torch.device("cpu"))
    dist.barrier()
    out[rank] = v
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_reports_on_rank0_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "c0", "--steps", "1", "--warmup", "0", "--gpus", "2"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank == 0:
        assert len(lines) == 1
        rec = json.loads(lines[0])
        assert rec["impl"] == "reference" and rec["unit"] == "ms" and rec["value"] > 0
        assert rec["cpu_baseline"]["kind"] == "oracle" and rec["n_gpus"] == 2
    else:
        assert lines == []
