"""The benchmark's multi-rank plumbing on CPU: two ranks over gloo.

The layer has no exchange step, so `bench.py --gpus N` runs N independent replicas; the only
cross-rank logic is the barrier around the timed region, the maximum of the ranks' step times
and the whole-job throughput computed from it.  These tests run that logic as two gloo
processes (no GPU), and check that the reference arm leaves the work to rank 0.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, step_ms, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench._DIST["on"] = True
    try:
        bench.barrier()
        ms = bench.reduce_max(step_ms[rank])
        value = bench.replica_value(world, 2048, ms)
        bench.barrier()
        out_q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def _run_ranks(step_ms):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    world = len(step_ms)
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, step_ms, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(got)


def test_two_replicas_are_timed_by_the_slowest_rank():
    got = _run_ranks([0.75, 1.25])
    assert [r for r, _, _ in got] == [0, 1]
    for _, ms, value in got:
        assert ms == 1.25                                  # every rank sees the maximum
        assert value == pytest.approx(2 * 2048 / 1.25e-3)  # all ranks' tokens over that time


def test_one_process_reduces_to_itself():
    sys.path.insert(0, ROOT)
    import bench
    assert not bench._DIST["on"]
    assert bench.reduce_max(0.5) == 0.5
    assert bench.replica_value(1, 2048, 0.5) == pytest.approx(2048 / 0.5e-3)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""     # rank 1 prints nothing and does no work


def test_reference_arm_line_on_rank_zero():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
