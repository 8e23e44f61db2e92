"""The benchmark's multi-rank path on CPU: world size 2 over gloo.

bench.py under torchrun shares one N^2 problem among the ranks (each owns a
range of targets), takes the slowest rank's step time (max over ranks) and
reports the whole problem's pairs over it; only rank 0 prints.  No GPU is
needed for these checks.
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    slowest = bench.max_over_ranks(100.0 + 50.0 * rank, world, device="cpu")
    bench.barrier(world)
    value = bench.whole_job_value(1e12, slowest)
    q.put((rank, slowest, value))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [150.0, 150.0]            # both ranks see the slowest time
    assert all(abs(g[2] - 1e12 / 0.150) < 1 for g in got)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_on_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "smallcube1024", "--steps", "1", "--warmup", "0",
                        "--cpu-seconds", "0.2", "--gpus", "2"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank == 0:
        line = json.loads(lines[-1])
        assert line["impl"] == "reference" and line["value"] > 0
        assert line["cpu_baseline"]["kind"] == "oracle"
        assert line["e2e"]["h2d_bytes_per_step"] == 0
    else:
        assert lines == []
