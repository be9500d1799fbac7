"""Runs over N > 1 ranks, checked with two gloo ranks on the CPU.

The unified step shards by request and KV head with no exchange step, so a
run on N GPUs is N replicas: each rank times its own seeded replica of the
workload, the ranks meet only at the timing barriers, and the whole-job
value divides the slowest rank's time by the layer-steps of all ranks.  These
checks drive the helpers bench.py uses for that through a real gloo process
group (world size 2), and the rank rules of both bench arms.
"""
import argparse
import contextlib
import io
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, elapsed, steps, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        dist.barrier()
        m = bench.max_over_ranks(elapsed[rank], world, "cpu")
        dist.barrier()
        q.put((rank, m, bench.whole_job_us(m, steps, world), bench.dist_env()))
    finally:
        dist.destroy_process_group()


def _run_two_ranks(elapsed, steps):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, elapsed, steps, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=180) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    return res


def test_two_gloo_ranks_report_the_slowest_rank_over_all_layer_steps():
    elapsed = [3.25, 5.5]  # ms: rank 1 is the slower replica
    res = _run_two_ranks(elapsed, steps=10)
    assert [r[0] for r in res] == [0, 1]
    for rank, m, us, env in res:
        assert m == 5.5                                # every rank holds the maximum
        assert us == pytest.approx(5.5e3 / (10 * 2))  # 20 layer-steps in the slowest rank's 5.5 ms
        assert env[0] == rank and env[1] == 2


def test_a_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(7.0, 1, "cpu") == 7.0
    assert bench.whole_job_us(7.0, 14, 1) == pytest.approx(500.0)


def test_replicas_are_the_same_shape_with_distinct_seeds():
    import bench
    import workloads as W
    args = argparse.Namespace(workload="qwen3_8b", length_scale=1.0, batch=None)
    r0, r1, r2 = (bench.replica_recipe(args, r) for r in range(3))
    assert r0 is W.RECIPES["qwen3_8b"]  # rank 0 times the named workload itself
    for r in (r1, r2):
        for f in ("B", "Hq", "Hkv", "D", "k", "s_num", "s_den", "lengths", "pillar_frac", "pool_min", "mode_rule"):
            assert getattr(r, f) == getattr(r0, f), f
    assert len({r0.seed, r1.seed, r2.seed}) == 3


def test_small_replicas_generate_distinct_data_of_one_shape():
    import numpy as np
    import bench
    import workloads as W
    args = argparse.Namespace(workload="tiny", length_scale=1.0, batch=None)
    w0, w1 = (W.generate(bench.replica_recipe(args, r)) for r in range(2))
    assert w0.q.shape == w1.q.shape and w0.B == w1.B
    assert not np.array_equal(w0.q, w1.q)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(workload="qwen3_8b", gpus=2, steps=3, warmup=3)
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        assert bench.run_reference(args) == 0
    assert out.getvalue() == ""  # the other ranks exit without work and print nothing


def test_reference_arm_line_on_rank_zero(monkeypatch):
    """The reference arm (the fp64 oracle on the host cores) prints one JSON
    line with the keys the bench contract asks of it."""
    import json
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    args = argparse.Namespace(workload="tiny", gpus=1, steps=2, warmup=1)
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        assert bench.run_reference(args) == 0
    line = json.loads(out.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["value"] > 0 and line["higher_is_better"] is False and line["steps"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "tiny"
