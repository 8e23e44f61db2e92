"""The caller-owned workspace, the bounded pool and the passes of the
symmetric and tiled paths, through the C ABI (needs a GPU).

A workspace that holds at least one group of the decomposition gives the
same partial sums, added in the same order, whatever the number of passes:
the results are bit-identical across budgets.  Smaller workspaces run a
decomposition without partials, still within the parity bounds.
"""
import numpy as np
import pytest
import torch

import all_pairs_gravitational_gb300 as apg
import oracle
from all_pairs_gravitational_gb300 import workloads as W

pytestmark = pytest.mark.gpu

L2_TOL = 1e-5
BODY_TOL = 1e-4
SYM = apg.NBODY_PATH_SYMMETRIC


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"


def dev():
    return torch.device("cuda:0")


def sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def assert_parity(got, ref, rows=None, potential=True):
    got = np.asarray(got, np.float64)
    if rows is not None:
        got = got[rows]
    ea = np.linalg.norm(got[:, :3] - ref[:, :3]) / np.linalg.norm(ref[:, :3])
    ba = (np.linalg.norm(got[:, :3] - ref[:, :3], axis=1) / np.linalg.norm(ref[:, :3], axis=1)).max()
    assert ea <= L2_TOL and ba <= BODY_TOL, (ea, ba)
    if potential:
        ep = np.linalg.norm(got[:, 3] - ref[:, 3]) / np.linalg.norm(ref[:, 3])
        bp = (np.abs(got[:, 3] - ref[:, 3]) / np.abs(ref[:, 3])).max()
        assert ep <= L2_TOL and bp <= BODY_TOL, (ep, bp)


def workspace(nbytes):
    return torch.empty(int(nbytes), dtype=torch.uint8, device=dev())


def rows_of(n, k, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.choice(n, size=min(k, n), replace=False),
                                     np.arange(max(0, n - 64), n)]))


# ------------------------------------------------------------ size queries

@pytest.mark.parametrize("n", [1, 1000, 8192, 20011, 65536, 200003, 1048576])
def test_size_query_is_the_default_plan(n):
    plan = apg.nbody_plan_forces(n, sm_count())
    assert apg.nbody_forces_workspace_bytes(n) == plan["scratch_bytes"]
    assert plan["scratch_bytes"] <= apg.NBODY_DEFAULT_WORKSPACE_BYTES
    sim = apg.nbody_simulate_workspace_bytes(n)
    extra = 16 * n if plan["path"] in (apg.NBODY_PATH_CLUSTER, apg.NBODY_PATH_ROWS) else 0
    assert sim == plan["scratch_bytes"] + extra


# ------------------------------------------------------------ bit-identity across budgets

@pytest.mark.parametrize("n,dists", [(20011, 3), (65537, 5), (130003, 0)])
def test_symmetric_budgets_give_the_same_bits(n, dists):
    """Forced distances per group give several groups; workspaces of one
    group, two groups, all groups and the default pool all produce the same
    bits, and match the oracle."""
    w = W.clumps(n, seed=n % 1000)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    base = apg.nbody_plan_forces(n, sm_count(), path=SYM, dists=dists)
    assert base["groups"] > 1 or dists == 0
    ref = apg.nbody_forces_ex(pm, float(w.eps2), path=SYM, dists=dists)
    lo = base["scratch_min_bytes"]
    one = apg.nbody_plan_forces(n, sm_count(), path=SYM, dists=dists, workspace_bytes=1 << 40)
    seen = set()
    for budget in (lo, lo + 16 * n * (base["splits"] + base["dists"]), one["scratch_bytes"]):
        plan = apg.nbody_plan_forces(n, sm_count(), path=SYM, dists=dists, workspace_bytes=budget)
        seen.add(plan["passes"])
        out = torch.full_like(pm, float("nan"))
        apg.nbody_forces_ws(pm, float(w.eps2), out, workspace=workspace(budget), path=SYM,
                            dists=dists)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), (budget, plan["passes"])
    if base["groups"] > 1:
        assert len(seen) >= 2
    rows = rows_of(n, 1500, 3)
    assert_parity(ref.cpu().numpy(), oracle.forces(w.pos_mass, w.eps2, rows=rows), rows)


def test_tiled_budgets_give_the_same_bits():
    n = 200003
    w = W.clumps(n, seed=4)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    ref = apg.nbody_forces_ex(pm, float(w.eps2), path=apg.NBODY_PATH_TILED)
    base = apg.nbody_plan_forces(n, sm_count(), path=apg.NBODY_PATH_TILED)
    assert base["splits"] > 2
    for budget in (2 * 16 * n, 3 * 16 * n, 16 * n * base["splits"]):
        out = apg.nbody_forces_ws(pm, float(w.eps2), workspace=workspace(budget),
                                  path=apg.NBODY_PATH_TILED)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), budget
    rows = rows_of(n, 1000, 5)
    assert_parity(ref.cpu().numpy(), oracle.forces(w.pos_mass, w.eps2, rows=rows), rows)


@pytest.mark.parametrize("n", [5003, 20011, 70001])
def test_no_workspace_runs_without_partials(n):
    """A workspace of 0 bytes: the automatic choice needs no partials (one
    piece per target block) and stays within the parity bounds."""
    w = W.clumps(n, seed=n)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    out = apg.nbody_forces_ws(pm, float(w.eps2), workspace=torch.empty(0, device=dev()))
    torch.cuda.synchronize()
    # below 10240 bodies the automatic choice (row-split) has no partials anyway
    ref = apg.nbody_forces_ex(pm, float(w.eps2), path=apg.NBODY_PATH_TILED if n >= 10240 else 0,
                              splits=1 if n >= 10240 else 0)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    rows = rows_of(n, 1000, 6)
    assert_parity(out.cpu().numpy(), oracle.forces(w.pos_mass, w.eps2, rows=rows), rows)


def test_forced_symmetric_path_rejects_a_too_small_workspace():
    w = W.clumps(65536, seed=1)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    out = torch.full_like(pm, 7.0)
    with pytest.raises(apg.NbodyError) as e:
        apg.nbody_forces_ws(pm, float(w.eps2), out, workspace=workspace(1 << 20), path=SYM)
    assert e.value.status == 8
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)            # nothing launched


@pytest.mark.slow
def test_plummer1048576_one_pass_equals_the_default_passes():
    """The benchmark workload: the default call (several passes within the
    default budget) and one pass in a caller's workspace give the same bits."""
    w = W.named("plummer1048576")
    pm = torch.from_numpy(w.pos_mass).to(dev())
    plan = apg.nbody_plan_forces(w.n, sm_count())
    assert plan["passes"] > 1
    one = apg.nbody_plan_forces(w.n, sm_count(), workspace_bytes=1 << 40)
    assert one["passes"] == 1 and one["splits"] == plan["splits"]
    ref = apg.nbody_forces(pm, float(w.eps2))
    ws = workspace(one["scratch_bytes"])
    out = apg.nbody_forces_ws(pm, float(w.eps2), workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


# ------------------------------------------------------------ simulate

def _separate_steps(w, steps):
    pm = torch.from_numpy(w.pos_mass).to(dev())
    vel = torch.from_numpy(w.vel).to(dev())
    acc = torch.empty_like(pm)
    for _ in range(steps):
        apg.nbody_forces(pm, float(w.eps2), acc)
        apg.nbody_euler_step(pm, vel, acc, float(w.dt))
    torch.cuda.synchronize()
    return pm, vel, acc


@pytest.mark.parametrize("name,steps", [("smallcube1024", 5), ("smallcube8192", 3),
                                        ("plummer65536", 3)])
def test_simulate_ws_is_the_separate_calls(name, steps):
    w = W.named(name)
    ref = _separate_steps(w, steps)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    vel = torch.from_numpy(w.vel).to(dev())
    acc = torch.empty_like(pm)
    ws = workspace(max(16, apg.nbody_simulate_workspace_bytes(w.n)))
    apg.nbody_simulate_ws(pm, vel, acc, float(w.eps2), float(w.dt), steps, ws)
    torch.cuda.synchronize()
    for got, exp in zip((pm, vel, acc), ref):
        assert torch.equal(got, exp)
    apg.nbody_release_cached()      # the graph no longer refers to ws


@pytest.mark.parametrize("name,steps", [("smallcube2048", 5), ("smallcube4096", 18)])
def test_simulate_ws_without_room_for_the_fused_steps(name, steps):
    """A workspace too small for the second position buffer: the row-split
    path's steps run as a force launch and an Euler launch each (no fused
    pairs), with the same bits as the separate calls."""
    w = W.named(name)
    assert apg.nbody_simulate_workspace_bytes(w.n) == 16 * w.n
    ref = _separate_steps(w, steps)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    vel = torch.from_numpy(w.vel).to(dev())
    acc = torch.empty_like(pm)
    apg.nbody_simulate_ws(pm, vel, acc, float(w.eps2), float(w.dt), steps, workspace(16))
    torch.cuda.synchronize()
    for got, exp in zip((pm, vel, acc), ref):
        assert torch.equal(got, exp)
    apg.nbody_release_cached()


def test_simulate_same_problem_from_two_streams():
    """Two streams replay the same cached graph back to back without any
    host synchronisation: the library orders the second call after the
    first on the GPU, so the result is that of the steps in sequence."""
    w = W.plummer(30011, seed=8, eps=0.01)
    ref = _separate_steps(w, 6)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    vel = torch.from_numpy(w.vel).to(dev())
    acc = torch.empty_like(pm)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    apg.nbody_simulate(pm, vel, acc, float(w.eps2), float(w.dt), 3, stream=s1)
    apg.nbody_simulate(pm, vel, acc, float(w.eps2), float(w.dt), 3, stream=s2)
    torch.cuda.synchronize()
    assert torch.equal(pm, ref[0]) and torch.equal(vel, ref[1]) and torch.equal(acc, ref[2])


# ------------------------------------------------------------ memory held by the library

def test_release_returns_the_library_memory():
    """After the pool-based calls and nbody_release_cached, the device has
    the free memory it had before them (up to a few MiB of driver
    bookkeeping)."""
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    w = W.named("plummer65536")
    pm = torch.from_numpy(w.pos_mass).to(dev())
    vel = torch.from_numpy(w.vel).to(dev())
    acc = torch.empty_like(pm)
    apg.nbody_forces(pm, float(w.eps2), acc)            # warm the library up first
    apg.nbody_release_cached()
    free0, _ = torch.cuda.mem_get_info()
    big = W.clumps(400009, seed=2)
    bpm = torch.from_numpy(big.pos_mass).to(dev())
    bacc = torch.empty_like(bpm)
    apg.nbody_forces(bpm, float(big.eps2), bacc)       # hundreds of MB of partials
    apg.nbody_simulate(pm, vel, acc, float(w.eps2), float(w.dt), 2)
    torch.cuda.synchronize()
    del bpm, bacc
    torch.cuda.empty_cache()
    apg.nbody_release_cached()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 >= free0 - (8 << 20), (free0, free1)


def test_pool_shortage_falls_back_to_a_plan_without_partials():
    """With almost no device memory left, nbody_forces cannot take its
    partials from the pool: it re-plans without them (the tiled kernel, one
    piece per target block) instead of failing."""
    n = 200003
    w = W.clumps(n, seed=3)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    out = torch.empty_like(pm)
    no_partials = apg.nbody_forces_ex(pm, float(w.eps2), path=apg.NBODY_PATH_TILED, splits=1)
    apg.nbody_release_cached()
    torch.cuda.synchronize()
    need = apg.nbody_plan_forces(n, sm_count())["scratch_bytes"]
    free, _ = torch.cuda.mem_get_info()
    hog = None
    try:
        # leave less than the partials need (and much less than is free now)
        hog = torch.empty(free - need // 4, dtype=torch.uint8, device=dev())
        apg.nbody_forces(pm, float(w.eps2), out)
        torch.cuda.synchronize()
    finally:
        del hog
        torch.cuda.empty_cache()
    assert torch.equal(out, no_partials)
    rows = rows_of(n, 800, 9)
    assert_parity(out.cpu().numpy(), oracle.forces(w.pos_mass, w.eps2, rows=rows), rows)


# ------------------------------------------------------------ randomized shapes

def _random_cases(count=24, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for k in range(count):
        n = int(rng.integers(1, 30000))
        path = int(rng.choice([0, 1, 2, 3, 4]))
        if path in (2, 4) and n > 12000:   # the cluster and row-split paths serve small n
            path = 0
        dists = int(rng.choice([0, 1, 2, 5])) if path == 3 else 0
        splits = int(rng.choice([0, 1, 3, 17])) if path in (1, 3, 4) else 0
        cases.append((k, n, path, dists, splits))
    return cases


@pytest.mark.parametrize("k,n,path,dists,splits", _random_cases())
def test_random_shapes_budgets_and_paths(k, n, path, dists, splits):
    """Seeded random sizes, paths, distances per group and pieces: the
    result within a workspace of the least size that keeps the plan, and
    within the default, agree bit for bit and match the oracle."""
    w = W.clumps(n, seed=k + 7) if k % 2 else W.cube(n, seed=k + 7)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    kw = dict(path=path, dists=dists, splits=splits)
    plan = apg.nbody_plan_forces(n, sm_count(), **kw)
    ref = apg.nbody_forces_ex(pm, float(w.eps2), **kw)
    lo = max(plan["scratch_min_bytes"], 16)
    out = apg.nbody_forces_ws(pm, float(w.eps2), workspace=workspace(lo), **kw)
    torch.cuda.synchronize()
    assert torch.equal(out, ref), plan
    rows = rows_of(n, 300, k)
    assert_parity(ref.cpu().numpy(), oracle.forces(w.pos_mass, w.eps2, rows=rows), rows)


def test_target_source_workspace_on_one_array_is_the_symmetric_call():
    """nbody_forces_ts_ws with the same array as targets and sources takes
    the symmetric path within the caller's workspace: the bits of
    nbody_forces."""
    w = W.clumps(30011, seed=31)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    ref = apg.nbody_forces(pm, float(w.eps2))
    ws = workspace(apg.nbody_forces_workspace_bytes(w.n))
    out = apg.nbody_forces_ts_ws(pm, pm, float(w.eps2), workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
