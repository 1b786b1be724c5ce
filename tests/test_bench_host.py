"""Host-side logic of bench.py on CPU: the multi-rank reduction and seeds
(two gloo ranks), and the reference arm's JSON line on a small workload."""
import json
import os
import subprocess
import sys

import numpy as np
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


def test_covering_tokens_reach_every_expert():
    import synth
    rng = np.random.default_rng(3)
    T, E, k = 4096, 384, 6
    ids = np.argsort(rng.random((T, E)) ** np.linspace(0.2, 3, E), axis=1)[:, :k]
    rows = synth.covering_tokens(ids, E, 512, 256)
    assert len(rows) == 768 and np.all(np.diff(rows) > 0)
    assert np.unique(ids[rows]).size == np.unique(ids).size
    assert np.array_equal(rows, synth.covering_tokens(ids, E, 512, 256))  # seeded
    few = synth.covering_tokens(ids[:10], E, 4)
    assert np.array_equal(few, np.arange(10))  # 10 tokens cannot reach 60 experts with fewer


def test_cpu_baseline_reports_all_cores_and_one_core():
    import synth
    dd = synth.make_inputs_torch("c3s", device="cpu")
    before = bench._blas_threads()
    b = bench.cpu_baseline(dd, 64, 16)
    assert bench._blas_threads() == before  # restored
    for key in ("value", "unit", "cores", "kind", "cores_all", "value_all", "value_1core", "sample"):
        assert key in b
    assert b["extrapolated"] is True and b["cores"] == os.cpu_count()
    assert b["value"] > 0 and b["value_1core"] > 0 and "every routed expert" in b["sample"]


def test_reference_step_models_the_layer_from_one_expert():
    # the bounded step of the reference arm: one expert's FFN on its rows and
    # on one row, the layer's FFN time modelled from the two (decode per
    # active expert + cost per routed row); step 0 takes the most loaded
    # expert, on all its rows up to the cap
    import oracle
    import synth
    dd = synth.make_inputs_torch("c3s", device="cpu")
    r = bench.OracleRunner(dd)
    v, t_route, t_dec, per_row, n = bench.oracle_expert_leg(r, 0, n_cap=64)
    assert v > 0 and t_route >= 0 and t_dec > 0 and per_row >= 0 and 2 <= n <= 64
    ids, _ = r.route()
    counts = np.bincount(ids.ravel(), minlength=r.c["E"])
    assert n == min(64, int(counts.max()))  # the most loaded expert first
    e = int(np.argmax(counts))
    rows = np.nonzero((ids == e).any(axis=1))[0][:n]
    X64 = oracle.bf16_to_f64(r.X[rows])
    W1, W2 = r.bits(dd["W1"][e]), r.bits(dd["W2"][e])
    assert oracle.swiglu_expert(X64, W1, W2).shape == (n, r.c["H"])
