"""The N > 1 host path of bench.py on CPU ranks (gloo, world size 2).

Multi-GPU runs are independent replicas: every rank times its own copy of the
workload, the ranks meet at a barrier on both sides of the timed region, and
the step time is the maximum over ranks.  These tests drive those helpers and
the reference arm's rank-0-only output through real process groups.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup(argparse.Namespace(impl="reference"))
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    got = bench.max_over_ranks(w, 10.0 * rank + 0.25)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": got}, f)
    bench.barrier(w)
    dist.destroy_process_group()


def test_barrier_and_max_over_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        got = json.load(open(tmp_path / f"rank{r}.json"))["max"]
        assert got == 10.0 * (world - 1) + 0.25


@pytest.mark.timeout(300)
def test_reference_arm_prints_one_line_from_rank_zero():
    env = dict(os.environ, PYTHONPATH=ROOT, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload",
           "single_head_3bit", "--cpu-budget", "1.0"]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=280)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [json.loads(l) for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
