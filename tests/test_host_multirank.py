"""Host-side multi-rank logic of bench.py on CPU ranks (gloo, world size 2), no GPU.

The benchmark's N > 1 path runs independent replicas; the only cross-rank steps are a barrier
around the timed region and the max over ranks of the elapsed time.  These run here as two
gloo ranks on 127.0.0.1.  The reference arm prints from rank 0 only.
"""
import importlib.util
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


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _bench()
        assert bench.dist_env() == (rank, world, rank)
        bench.barrier(world)
        got = bench.reduce_max(1.5 + rank * 10.0, world)
        bench.barrier(world)
        got_neg = bench.reduce_max(-3.0 - rank, world)
        out.put((rank, got, got_neg))
    finally:
        dist.destroy_process_group()


def test_reduce_max_and_barrier_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert res == [(0, 11.5, -3.0), (1, 11.5, -3.0)]


def test_reduce_max_is_identity_on_one_rank():
    bench = _bench()
    assert bench.reduce_max(2.25, 1) == 2.25
    bench.barrier(1)   # no process group needed


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_on_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "single_1m", "--steps", "1", "--warmup", "3",
                        "--ref-sample-elems", "65536"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank != 0:
        assert lines == []
    else:
        line = json.loads(lines[-1])
        assert line["impl"] == "reference" and line["n_gpus"] == 2
        assert line["unit"] == "GB/s" and line["value"] > 0
        assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
        assert line["e2e"]["h2d_bytes_per_step"] == 0
