"""The N > 1 replica path of bench.py on CPU: two gloo ranks, one process each.

bench.py runs one independent replica of the layer per GPU (the layer has no exchange step) and reports the
slowest rank's time with every rank's routes.  Here each rank reports made-up figures and the aggregation must
return max(time) and sum(routes) on both ranks; the reference arm must print from rank 0 only.
"""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, routes = bench.aggregate_over_ranks(10.0 + 5.0 * rank, 100 * (rank + 1), world, "cpu")
        out.put((rank, ms, routes))
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_aggregation_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(out.get(timeout=5) for _ in range(2))
    for rank, ms, routes in res:
        assert ms == 15.0            # the slowest rank's time
        assert routes == 300.0       # every rank's routes


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_over_ranks(7.5, 42, 1, "cpu") == (7.5, 42.0)


def test_replica_launch_plan():
    """--gpus N: one rank of a launch of N runs as is; without a launcher bench.py starts N local ranks; a
    launcher whose world size differs from --gpus is refused."""
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    a1, a4 = argparse.Namespace(gpus=1), argparse.Namespace(gpus=4)
    assert bench.replica_launch(a1, {}) is None
    assert bench.replica_launch(a4, {"WORLD_SIZE": "4"}) is None
    with pytest.raises(SystemExit):
        bench.replica_launch(a4, {"WORLD_SIZE": "2"})
    cmd = bench.replica_launch(a4, {})
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"] and "--nproc-per-node=4" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert any(c.endswith("bench.py") for c in cmd)


@pytest.mark.slow
def test_bench_gpus_2_starts_its_own_ranks():
    """`bench.py --gpus 2` without a launcher starts two local ranks (torchrun); on the reference arm rank 0
    alone prints, so exactly one JSON line comes out."""
    env = dict(os.environ, PYTHONPATH=ROOT)
    env.pop("WORLD_SIZE", None)
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--workload", "tiny"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    assert json.loads(lines[0])["impl"] == "reference"


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_once():
    """--impl reference under torchrun with two ranks (gloo is enough: no collective is used): one JSON line."""
    env = dict(os.environ, PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
