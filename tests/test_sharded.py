"""Target sharding over ranks (all_pairs_gravitational_gb300.sharded).

CPU: the partition of the targets, and the gather of every rank's bodies
over gloo with world size 2 and 3 and uneven shares; the oracle evaluated per
rank's range and concatenated is the whole-problem oracle.  GPU: two ranks
over gloo sharing one GPU (their kernels never wait on each other; the
exchange happens on the host between launches) reproduce the single-process
target/source call bit for bit and match the oracle.
"""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from all_pairs_gravitational_gb300 import sharded  # noqa: E402


@pytest.mark.parametrize("n", [0, 1, 2, 7, 1000, 20011, 2 ** 20 + 3])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_shard_ranges_cover_the_targets_once(n, world):
    ranges = [sharded.shard_range(n, r, world) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == n
    for (a, b), (c, d) in zip(ranges, ranges[1:]):
        assert b == c and a <= b
    sizes = [b - a for a, b in ranges]
    assert max(sizes) - min(sizes) <= 1 and sum(sizes) == n
    with pytest.raises(ValueError):
        sharded.shard_range(n, world, world)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _cpu_worker(rank, world, port, n, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import oracle
    from all_pairs_gravitational_gb300 import sharded as S
    from all_pairs_gravitational_gb300 import workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = W.clumps(n, seed=n)
    lo, hi = S.shard_range(n, rank, world)
    local = torch.from_numpy(w.pos_mass[lo:hi].copy())
    full = S.gather_bodies(local, n)
    ok_gather = bool(np.array_equal(full.numpy(), w.pos_mass))
    part = oracle.forces_ts(full.numpy()[lo:hi], full.numpy(), w.eps2)
    q.put((rank, ok_gather, part))
    dist.destroy_process_group()


@pytest.mark.parametrize("world,n", [(2, 1001), (3, 2000), (2, 1)])
def test_gather_and_partition_gloo(world, n):
    import torch.multiprocessing as mp
    import oracle
    from all_pairs_gravitational_gb300 import workloads as W
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_cpu_worker, args=(r, world, port, n, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=180) for _ in procs), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(g[1] for g in got)
    w = W.clumps(n, seed=n)
    whole = oracle.forces(w.pos_mass, w.eps2)
    assert np.array_equal(np.concatenate([g[2] for g in got]), whole)


def _gpu_worker(rank, world, port, n, steps, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import all_pairs_gravitational_gb300 as apg
    from all_pairs_gravitational_gb300 import sharded as S
    from all_pairs_gravitational_gb300 import workloads as W
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        dev = torch.device("cuda:0")
        w = W.plummer(n, seed=n, eps=0.01)
        lo, hi = S.shard_range(n, rank, world)
        pm = torch.from_numpy(w.pos_mass[lo:hi].copy()).to(dev)
        vel = torch.from_numpy(w.vel[lo:hi].copy()).to(dev)
        acc = S.forces_sharded(pm, n, float(w.eps2))
        # the same range through one process's target/source call
        full = torch.from_numpy(w.pos_mass).to(dev)
        ref = apg.nbody_forces_ts(full[lo:hi].contiguous(), full, float(w.eps2))
        torch.cuda.synchronize()
        same = bool(torch.equal(acc, ref))
        ws = torch.empty(apg.nbody_forces_workspace_bytes(n) + 16, dtype=torch.uint8, device=dev)
        S.simulate_sharded(pm, vel, acc, n, float(w.eps2), float(w.dt), steps, workspace=ws)
        torch.cuda.synchronize()
        q.put((rank, same, acc.cpu().numpy(), pm.cpu().numpy(), vel.cpu().numpy(), None))
        dist.destroy_process_group()
    except Exception as e:          # reported to the parent
        q.put((rank, False, None, None, None, repr(e)))


@pytest.mark.gpu
def test_two_ranks_on_one_gpu_reproduce_one_process():
    """n = 20011 split 10006 / 10005: each rank's forces equal the
    single-process target/source call on its range bit for bit, the union
    matches the oracle, and three sharded steps equal three steps of the same
    per-range calls made in one process."""
    import torch
    import torch.multiprocessing as mp
    import __graft_entry__
    __graft_entry__.build()
    import all_pairs_gravitational_gb300 as apg
    import oracle
    from all_pairs_gravitational_gb300 import workloads as W
    n, world, steps = 20011, 2, 3
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gpu_worker, args=(r, world, port, n, steps, q))
             for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=600) for _ in procs), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=120)
    assert all(g[5] is None for g in got), [g[5] for g in got]
    assert all(g[1] for g in got)
    # the sharded trajectory against the per-range calls in one process
    w = W.plummer(n, seed=n, eps=0.01)
    dev = torch.device("cuda:0")
    pm = torch.from_numpy(w.pos_mass).to(dev)
    vel = torch.from_numpy(w.vel).to(dev)
    acc = torch.empty_like(pm)
    ranges = [sharded.shard_range(n, r, world) for r in range(world)]
    first = None
    for step in range(steps + 1):
        parts = [apg.nbody_forces_ts(pm[lo:hi].contiguous(), pm, float(w.eps2)) for lo, hi in ranges]
        acc = torch.cat(parts)
        if step == 0:
            first = acc.cpu().numpy()
        if step == steps:
            break
        apg.nbody_euler_step(pm, vel, acc, float(w.dt))
    torch.cuda.synchronize()
    ref0 = oracle.forces(w.pos_mass, w.eps2)
    rng = np.random.default_rng(1)
    rows = rng.choice(n, 1500, replace=False)
    got0 = first[rows].astype(np.float64)
    assert np.linalg.norm(got0[:, :3] - ref0[rows, :3]) / np.linalg.norm(ref0[rows, :3]) <= 1e-5
    pm_all = np.concatenate([g[3] for g in got])
    vel_all = np.concatenate([g[4] for g in got])
    assert np.array_equal(pm_all, pm.cpu().numpy()) and np.array_equal(vel_all, vel.cpu().numpy())
