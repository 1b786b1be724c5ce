"""Host-side logic of bench.py on CPU: the multi-rank reduction and seeds
(two gloo ranks), and the reference arm's JSON line on a small workload."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 3.0 + rank * 1.5
        out[rank] = (bench.max_over_ranks(local_ms, world), bench.rank_seeds(rank))
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_and_share_weights():
    world, port = 2, 29517
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 4.5
    (w0, t0), (w1, t1) = res[0][1], res[1][1]
    assert w0 == w1 and t0 != t1


def test_single_rank_max_is_identity():
    assert bench.max_over_ranks(7.25, 1) == 7.25


def test_reference_arm_prints_its_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "c3s", "--steps", "2", "--warmup", "3", "--ref-tokens", "4"],
                       capture_output=True, text=True, cwd=ROOT, timeout=600,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in line
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "c3s", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, cwd=ROOT, timeout=300, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""
