"""The benchmark's multi-rank host logic on CPU (gloo, world size 2): the
timing is the maximum over ranks, the value counts every rank's bytes, and
under a launcher only rank 0 prints (the reference arm: the other ranks exit
without work)."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, out):
    import torch
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=2)
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, torch.device("cpu"), 2)
    out[rank] = (ms, bench.job_gbs(2, 1e9, 4, ms))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value_with_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1] == (15.0, 2 * 1e9 * 4 / 0.015 / 1e9)


def test_reference_arm_prints_on_rank_zero_only():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "gauss_1k",
           "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r1 = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    env.update(RANK="0", LOCAL_RANK="0")
    r0 = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600)
    assert r0.returncode == 0
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
