"""Multi-rank plumbing of bench.py on the CPU (gloo, world size 2).

The path runs as independent replicas, one per GPU, with no collective on the
data path; the only cross-rank steps are the barrier around the timed region
and the maximum of the per-rank times. These tests run those helpers in two
gloo processes and check the whole-job aggregation and that only rank 0 runs
the reference arm.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    os.environ["CUDA_VISIBLE_DEVICES"] = ""  # the gloo path, also on a machine with a GPU
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    w, r, _ = bench.dist_setup(None)
    bench.barrier(w)
    t = bench.max_over_ranks(times[r], w)
    bench.barrier(w)
    q.put((r, w, t))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    times = [1.25, 3.5]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == world for g in got)
    # every rank sees the maximum, so rank 0's whole-job figure is
    # units * world / slowest time
    assert all(g[2] == max(times) for g in got)


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(2.5, 1) == 2.5
    bench.barrier(1)  # no-op


def test_reference_arm_runs_on_rank_zero_only():
    # a non-zero rank of the reference arm exits 0 at once and prints nothing
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_line_keeps_the_bench_contract():
    """Rank 0 of the reference arm (the fp64 oracle on the host cores) prints
    one JSON line with the keys the bench contract names, the oracle
    described as its CPU baseline and an end-to-end entry without copies."""
    import json
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["higher_is_better"] is True
    assert d["config"]["workload"] and d["config"]["tokens_per_step"] == [1, 8, 32]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
