"""Parity of the CUDA path with the oracle, through the C ABI (needs a GPU).

Tolerances: relative L2 error of the accelerations (all 3N components) and
of the potentials <= 1e-5; largest per-body relative error <= 1e-4 for |a|
and for |p|; the Euler step bit-identical given the same accelerations.
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


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"


def dev():
    return torch.device("cuda:0")


def _rel(diff, scale):
    """diff / scale, where a zero reference must be matched exactly."""
    diff = np.asarray(diff, np.float64)
    scale = np.asarray(scale, np.float64)
    exact = np.where(diff == 0, 0.0, np.inf)
    with np.errstate(divide="ignore", invalid="ignore"):
        return np.where(scale > 0, diff / np.where(scale > 0, scale, 1.0), exact)


def errors(got, ref, rows=None, potential=True):
    got = np.asarray(got, np.float64)
    if rows is not None:
        got = got[rows]
    ea = float(_rel(np.linalg.norm(got[:, :3] - ref[:, :3]), np.linalg.norm(ref[:, :3])))
    na = np.linalg.norm(ref[:, :3], axis=1)
    ba = float(_rel(np.linalg.norm(got[:, :3] - ref[:, :3], axis=1), na).max())
    out = {"l2_a": ea, "body_a": ba}
    if potential:
        out["l2_p"] = np.linalg.norm(got[:, 3] - ref[:, 3]) / np.linalg.norm(ref[:, 3])
        out["body_p"] = (np.abs(got[:, 3] - ref[:, 3]) / np.abs(ref[:, 3])).max()
    return out


def assert_parity(got, ref, rows=None, potential=True):
    e = errors(got, ref, rows, potential)
    assert e["l2_a"] <= L2_TOL and e["body_a"] <= BODY_TOL, e
    if potential:
        assert e["l2_p"] <= L2_TOL and e["body_p"] <= BODY_TOL, e
    return e


def gpu_forces(pm_np, eps2, **kw):
    pm = torch.from_numpy(np.ascontiguousarray(pm_np)).to(dev())
    acc = apg.nbody_forces_ex(pm, float(eps2), **kw)
    torch.cuda.synchronize()
    return acc.cpu().numpy()


def sample_rows(n, k, seed):
    rng = np.random.default_rng(seed)
    rows = rng.choice(n, size=min(k, n), replace=False)
    return np.unique(np.concatenate([rows, [0, n - 1]]))


def _hard_rows(w, k, seed, core=4096, block=2048):
    """Rows where the per-body bound is most likely to fail, plus a random
    sample: the `core` bodies nearest the centre of mass (densest region,
    largest near-neighbour terms and cancellation), every body of the first,
    a middle and the last `block`-body block (edges of the symmetric
    decomposition), the ragged tail, and k random rows."""
    n = w.n
    x = w.pos_mass[:, :3].astype(np.float64)
    m = w.pos_mass[:, 3].astype(np.float64)
    com = (m[:, None] * x).sum(0) / m.sum()
    r = np.linalg.norm(x - com, axis=1)
    dense = np.argsort(r, kind="stable")[:min(core, n)]
    mid = (n // block // 2) * block
    edges = np.concatenate([np.arange(0, min(block, n)), np.arange(mid, min(mid + block, n)),
                            np.arange(max(0, n - block), n)])
    return np.unique(np.concatenate([sample_rows(n, k, seed), dense, edges]))


# ------------------------------------------------------------ configurations

def test_disk4096_acceleration_and_euler():
    w = W.named("disk4096")
    acc = gpu_forces(w.pos_mass, w.eps2)
    ref = oracle.forces(w.pos_mass, w.eps2)
    assert_parity(acc, ref, potential=False)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    vel = torch.from_numpy(w.vel).to(dev())
    a = torch.from_numpy(acc).to(dev())
    apg.nbody_euler_step(pm, vel, a, float(w.dt))
    torch.cuda.synchronize()
    pm_ref, v_ref = oracle.euler(w.pos_mass, w.vel, acc, w.dt)
    assert np.array_equal(pm.cpu().numpy(), pm_ref)
    assert np.array_equal(vel.cpu().numpy(), v_ref)


def test_cube16384_full():
    w = W.named("cube16384")
    assert_parity(gpu_forces(w.pos_mass, w.eps2), oracle.forces(w.pos_mass, w.eps2))


def test_plummer65536_ten_steps():
    """Ten force + Euler steps on the GPU's own state; parity on sampled rows
    at every step and the Euler step bit-exact every step."""
    w = W.named("plummer65536")
    pm = torch.from_numpy(w.pos_mass).to(dev())
    vel = torch.from_numpy(w.vel).to(dev())
    acc = torch.empty_like(pm)
    for step in range(w.steps):
        apg.nbody_forces(pm, float(w.eps2), acc)
        torch.cuda.synchronize()
        pm_np, v_np, a_np = pm.cpu().numpy(), vel.cpu().numpy(), acc.cpu().numpy()
        rows = sample_rows(w.n, 1024, step)
        ref = oracle.forces(pm_np, w.eps2, rows=rows)
        assert_parity(a_np, ref, rows)
        apg.nbody_euler_step(pm, vel, acc, float(w.dt))
        torch.cuda.synchronize()
        pm_ref, v_ref = oracle.euler(pm_np, v_np, a_np, w.dt)
        assert np.array_equal(pm.cpu().numpy(), pm_ref), step
        assert np.array_equal(vel.cpu().numpy(), v_ref), step


@pytest.mark.slow
def test_plummer65536_trajectory_against_fp64():
    """The ten GPU steps of the Plummer workload against the same ten Euler
    steps kept in fp64 throughout (the oracle's fp64 forces and fp64
    updates): the fp32 trajectory drifts from it only by rounding."""
    w = W.named("plummer65536")
    pm = torch.from_numpy(w.pos_mass).to(dev())
    vel = torch.from_numpy(w.vel).to(dev())
    acc = torch.empty_like(pm)
    apg.nbody_simulate(pm, vel, acc, float(w.eps2), float(w.dt), w.steps)
    torch.cuda.synchronize()
    pm64, v64 = oracle.trajectory_f64(w.pos_mass, w.vel, float(np.float32(w.eps2)),
                                      float(np.float32(w.dt)), w.steps)
    dx = np.abs(pm.cpu().numpy()[:, :3].astype(np.float64) - pm64[:, :3])
    dv = np.abs(vel.cpu().numpy()[:, :3].astype(np.float64) - v64[:, :3])
    rx = dx.max() / np.abs(pm64[:, :3]).max()
    rv = dv.max() / np.abs(v64[:, :3]).max()
    print(f"fp64 trajectory drift after {w.steps} steps: max |dx| {dx.max():.3e} "
          f"(rms {np.sqrt((dx ** 2).mean()):.3e}), max |dv| {dv.max():.3e} "
          f"(rms {np.sqrt((dv ** 2).mean()):.3e})")
    assert rx < 1e-6 and rv < 1e-5, (rx, rv)


def test_clumps200003_every_body():
    """Every one of the 200003 bodies against the oracle (about 4e10 fp64
    pairs on the host); the per-body maxima are printed."""
    w = W.named("clumps200003")
    acc = gpu_forces(w.pos_mass, w.eps2)
    e = assert_parity(acc, oracle.forces(w.pos_mass, w.eps2))
    print(f"clumps200003, all bodies: {e}")


@pytest.mark.parametrize("name", ["clumps200003", "plummer65536"])
def test_tiled_path_at_large_n(name):
    """The ordered-pair tiled kernel forced at sizes the automatic choice
    sends to the symmetric path (it still serves the compensated precision,
    the target/source form and n beyond the symmetric partials' cap)."""
    w = W.named(name)
    acc = gpu_forces(w.pos_mass, w.eps2, path=apg.NBODY_PATH_TILED)
    rows = np.unique(np.concatenate([sample_rows(w.n, 1024, 6), np.arange(w.n - 100, w.n)]))
    assert_parity(acc, oracle.forces(w.pos_mass, w.eps2, rows=rows), rows)


@pytest.mark.slow
def test_plummer1048576_in_bench_configuration():
    """The full-size workload in the launch configuration the benchmark times
    (default plan, several passes), checked on more than 16384 rows: the 4096
    bodies of the dense core, every body of the first, a middle and the last
    2048-body block, and 8192 random rows.  The per-body maxima are printed."""
    w = W.named("plummer1048576")
    plan = apg.nbody_plan_forces(w.n, torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["path"] == apg.NBODY_PATH_SYMMETRIC and plan["passes"] > 1
    assert plan["scratch_bytes"] <= apg.NBODY_DEFAULT_WORKSPACE_BYTES
    acc = gpu_forces(w.pos_mass, w.eps2)
    rows = _hard_rows(w, 8192, seed=2)
    assert rows.size >= 16384
    e = assert_parity(acc, oracle.forces(w.pos_mass, w.eps2, rows=rows), rows)
    print(f"plummer1048576, {rows.size} rows: {e}")


@pytest.mark.parametrize("n", W.SMALL_SWEEP)
def test_small_cube_sweep(n):
    w = W.small_cube(n)
    assert_parity(gpu_forces(w.pos_mass, w.eps2), oracle.forces(w.pos_mass, w.eps2))


# ------------------------------------------------------------ edges and plans

@pytest.mark.parametrize("n", [1, 2, 3, 31, 33, 127, 129, 255, 257, 511, 513, 1000, 1025, 4097])
def test_ragged_sizes(n):
    w = W.cube(n, seed=n + 17)
    assert_parity(gpu_forces(w.pos_mass, w.eps2), oracle.forces(w.pos_mass, w.eps2))


def test_single_body_self_term():
    pm = np.array([[0.25, -1.5, 3.0, 2.0]], np.float32)
    out = gpu_forces(pm, 0.0625)
    assert out[0, :3].tolist() == [0.0, 0.0, 0.0]
    assert out[0, 3] == pytest.approx(-8.0, rel=1e-6)


@pytest.mark.parametrize("path", [1, 2, 3, 4])
def test_smallest_accepted_softening(path):
    """eps^2 = NBODY_MIN_EPS2: the self term m (eps^2)^(-3/2) * 0 stays 0
    (finite in fp32 for masses up to 10), on every path; a lone body has
    a = 0 and p = -m / eps."""
    eps2 = apg.NBODY_MIN_EPS2
    one = gpu_forces(np.array([[0.25, -0.5, 0.75, 10.0]], np.float32), eps2,
                     path=path if path != 3 else 0)
    assert np.all(one[0, :3] == 0.0)
    np.testing.assert_allclose(one[0, 3], -10.0 / np.sqrt(np.float64(np.float32(eps2))), rtol=1e-6)
    w = W.cube(5003, seed=61)
    pm = w.pos_mass.copy()
    pm[:, 3] = np.random.default_rng(5).uniform(0.1, 10.0, w.n).astype(np.float32)
    got = gpu_forces(pm, eps2, path=path)
    assert np.all(np.isfinite(got))
    assert_parity(got, oracle.forces(pm, np.float32(eps2)))


def test_two_body_closed_form():
    pm = np.array([[0, 0, 0, 1], [4, 0, 0, 2]], np.float32)
    out = gpu_forces(pm, 9.0).astype(np.float64)
    np.testing.assert_allclose(out[:, 0], [8 / 125, -4 / 125], rtol=1e-6)
    np.testing.assert_allclose(out[:, 3], [-11 / 15, -13 / 15], rtol=1e-6)
    assert np.all(out[:, 1:3] == 0)


def _variant_count(path):
    v = 0
    while True:
        try:
            apg.nbody_plan_forces(1000, 152, path=path, variant=v)
        except apg.NbodyError:
            return v
        v += 1


@pytest.mark.parametrize("variant", range(_variant_count(apg.NBODY_PATH_TILED)))
@pytest.mark.parametrize("splits", [1, 2, 3, 7, 40])
def test_forced_plans(variant, splits):
    w = W.clumps(5003, seed=77)
    ref = oracle.forces(w.pos_mass, w.eps2)
    got = gpu_forces(w.pos_mass, w.eps2, path=apg.NBODY_PATH_TILED, variant=variant,
                     splits=splits)
    assert_parity(got, ref)


@pytest.mark.parametrize("path", [1, 2, 3, 4])
def test_disk_near_neighbours_all_paths(path):
    """The disk workload has bodies whose nearest neighbours contribute terms
    hundreds of times |a_i| (condition number ~1e3): the per-body bound holds."""
    w = W.named("disk4096")
    got = gpu_forces(w.pos_mass, w.eps2, path=path)
    assert_parity(got, oracle.forces(w.pos_mass, w.eps2), potential=False)


@pytest.mark.parametrize("variant", range(_variant_count(apg.NBODY_PATH_CLUSTER)))
@pytest.mark.parametrize("n", [1, 3, 100, 1000, 4096, 5003, 12000])
def test_cluster_path(variant, n):
    w = W.cube(n, seed=n + 3)
    got = gpu_forces(w.pos_mass, w.eps2, path=apg.NBODY_PATH_CLUSTER, variant=variant)
    assert_parity(got, oracle.forces(w.pos_mass, w.eps2))


def test_paths_agree_small_n():
    """Every small-N path on the same input: each within tolerance of the oracle."""
    w = W.small_cube(2048)
    ref = oracle.forces(w.pos_mass, w.eps2)
    for path in (apg.NBODY_PATH_TILED, apg.NBODY_PATH_CLUSTER, apg.NBODY_PATH_ROWS):
        assert_parity(gpu_forces(w.pos_mass, w.eps2, path=path), ref)


# ------------------------------------------------------------ row-split path

ROWS = apg.NBODY_PATH_ROWS


@pytest.mark.parametrize("variant", range(_variant_count(ROWS)))
@pytest.mark.parametrize("n", [1, 2, 3, 7, 100, 152, 153, 1000, 1064, 2048, 3071, 4096, 4865,
                               8192, 10239, 12000])
def test_rows_path(variant, n):
    """Each row-split shape on ragged sizes: targets per CTA not a multiple
    of K (phantom targets), sources not a multiple of 64 (zero padding),
    one to several pieces."""
    w = W.cube(n, seed=n + 11)
    got = gpu_forces(w.pos_mass, w.eps2, path=ROWS, variant=variant)
    assert_parity(got, oracle.forces(w.pos_mass, w.eps2))


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 40])
def test_rows_forced_pieces(splits):
    """Forced piece counts, including pieces longer than 2048 sources and
    pieces made only of padding."""
    w = W.clumps(5003, seed=78)
    got = gpu_forces(w.pos_mass, w.eps2, path=ROWS, splits=splits)
    assert_parity(got, oracle.forces(w.pos_mass, w.eps2))


def test_rows_path_deterministic_and_the_automatic_choice():
    w = W.small_cube(4096)
    a = gpu_forces(w.pos_mass, w.eps2, path=ROWS)
    for _ in range(3):
        assert np.array_equal(gpu_forces(w.pos_mass, w.eps2, path=ROWS), a)
    assert np.array_equal(gpu_forces(w.pos_mass, w.eps2), a)


@pytest.mark.parametrize("nt,ns", [(1, 1), (1, 5000), (5000, 1), (37, 10000), (10000, 37),
                                   (700, 4099), (20000, 3000), (100, 14400), (1000, 14000)])
def test_rows_target_source_form(nt, ns):
    """Separate target and source arrays: few sources against few or many
    targets (20000 targets: several items per warp), and the most sources
    shared memory holds (14400: 225 KB per CTA)."""
    t, s = _ts_bodies(nt, ns, nt * 5 + ns)
    eps2 = np.float32(1e-3)
    out = apg.nbody_forces_ts_ws(torch.from_numpy(t).to(dev()), torch.from_numpy(s).to(dev()),
                                 float(eps2), workspace=torch.empty(0, device=dev()), path=ROWS)
    torch.cuda.synchronize()
    assert_parity(out.cpu().numpy(), oracle.forces_ts(t, s, eps2))


def test_cluster_path_deterministic():
    w = W.small_cube(4096)
    a = gpu_forces(w.pos_mass, w.eps2, path=apg.NBODY_PATH_CLUSTER)
    for _ in range(3):
        assert np.array_equal(gpu_forces(w.pos_mass, w.eps2, path=apg.NBODY_PATH_CLUSTER), a)


def test_bitwise_deterministic():
    w = W.clumps(30011, seed=5)
    a = gpu_forces(w.pos_mass, w.eps2)
    for _ in range(3):
        assert np.array_equal(gpu_forces(w.pos_mass, w.eps2), a)


def test_newtons_third_law_on_gpu():
    w = W.clumps(20000, seed=8)
    acc = gpu_forces(w.pos_mass, w.eps2).astype(np.float64)
    m = w.pos_mass[:, 3].astype(np.float64)[:, None]
    total = np.abs((m * acc[:, :3]).sum(0)).max()
    assert total < 1e-6 * (m * np.abs(acc[:, :3])).sum()


def test_canaries_and_offsets_untouched():
    """Output written exactly in [0, n): records before and after are intact."""
    w = W.cube(3001, seed=3)
    n = w.n
    big = torch.full((n + 8, 4), 12345.0, device=dev())
    out = big[4:4 + n]
    pm = torch.from_numpy(w.pos_mass).to(dev())
    apg.nbody_forces(pm, float(w.eps2), out)
    torch.cuda.synchronize()
    b = big.cpu().numpy()
    assert np.all(b[:4] == 12345.0) and np.all(b[-4:] == 12345.0)
    assert_parity(b[4:4 + n], oracle.forces(w.pos_mass, w.eps2))
    assert np.array_equal(pm.cpu().numpy(), w.pos_mass)          # input untouched


def test_side_stream():
    w = W.cube(2000, seed=4)
    s = torch.cuda.Stream()
    pm = torch.from_numpy(w.pos_mass).to(dev())
    with torch.cuda.stream(s):
        acc = apg.nbody_forces(pm, float(w.eps2))
    s.synchronize()
    assert_parity(acc.cpu().numpy(), oracle.forces(w.pos_mass, w.eps2))


def test_empty_input_is_a_noop():
    pm = torch.empty((0, 4), device=dev())
    acc = apg.nbody_forces(pm, 1e-4)
    assert acc.shape == (0, 4)
    apg.nbody_euler_step(pm, torch.empty_like(pm), acc, 1e-3)


def test_host_rejections_on_gpu_tensors():
    pm = torch.zeros((17, 4), device=dev())
    flat = torch.zeros(17 * 4 + 1, device=dev())
    mis = flat[1:].view(17, 4)                                    # 4 bytes off alignment
    with pytest.raises(apg.NbodyError) as e:
        apg.nbody_forces(mis, 1e-4)
    assert e.value.status == 2
    with pytest.raises(apg.NbodyError) as e:
        apg.nbody_forces(pm, 1e-4, pm)
    assert e.value.status == 3
    with pytest.raises(apg.NbodyError) as e:
        apg.nbody_forces(pm, 0.0)
    assert e.value.status == 1


def test_euler_large_bit_exact():
    w = W.plummer(300007, seed=1)
    acc = np.zeros_like(w.pos_mass)
    acc[:, :3] = W.Stream(9).uniform(3 * w.n, -50, 50).reshape(w.n, 3)
    acc[:, 3] = 7.0
    pm = torch.from_numpy(w.pos_mass).to(dev())
    vel = torch.from_numpy(w.vel).to(dev())
    apg.nbody_euler_step(pm, vel, torch.from_numpy(acc).to(dev()), float(w.dt))
    torch.cuda.synchronize()
    pm_ref, v_ref = oracle.euler(w.pos_mass, w.vel, acc, w.dt)
    assert np.array_equal(pm.cpu().numpy(), pm_ref)
    assert np.array_equal(vel.cpu().numpy(), v_ref)


# ------------------------------------------------------------ symmetric path

SYM = 3   # NBODY_PATH_SYMMETRIC


def _sym_block(variant=0):
    plan = apg.nbody_plan_forces(4096, 152, path=SYM, variant=variant)
    return plan["threads"] * plan["i_per_thread"]


# T = 2048 for the default variant: one block, two (the even extra distance),
# three, five and eight blocks, each with a ragged last block.
@pytest.mark.parametrize("n", [1, 2, 33, 1000, 2048, 2049, 4095, 4096, 4097, 6144, 9000, 10240,
                               16383, 20011])
def test_symmetric_path_parity(n):
    w = W.clumps(n, seed=n + 101)
    got = gpu_forces(w.pos_mass, w.eps2, path=SYM)
    assert_parity(got, oracle.forces(w.pos_mass, w.eps2))


@pytest.mark.parametrize("variant", range(_variant_count(SYM)))
@pytest.mark.parametrize("splits", [0, 1, 2, 5, 17, 1000])
def test_symmetric_variants_and_splits(variant, splits):
    n = 3 * _sym_block(variant) + 77                      # four blocks (even), ragged
    w = W.cube(n, seed=variant * 100 + splits)
    got = gpu_forces(w.pos_mass, w.eps2, path=SYM, variant=variant, splits=splits)
    assert_parity(got, oracle.forces(w.pos_mass, w.eps2))


@pytest.mark.parametrize("n,splits", [(32768, 0), (65537, 0), (65537, 1), (131072, 0),
                                      (262147, 0), (1048576, 0)])
def test_symmetric_path_counts_every_pair_once(n, splits):
    """Unit masses and eps^2 = 2^40: |r|^2 < 12 vanishes against 2^40 in fp32,
    so every potential term is the same value t, the kernel's rsqrt(2^40)
    (2^-20 up to the hardware rsqrt's error).  Then -p_i / t counts the
    bodies that body i met, and a block pair skipped or evaluated twice moves
    that count by at least one for every body involved.  When t is exactly
    2^-20 every partial sum is exact and the count must be n exactly."""
    one = gpu_forces(np.array([[0.5, 0.5, 0.5, 1.0]], np.float32), 2.0 ** 40, path=SYM)
    t = -float(one[0, 3])
    assert abs(t * 2.0 ** 20 - 1.0) < 2.0 ** -21
    print(f"potential term t = 2^-20 * {t * 2.0 ** 20!r} (exact count: {t == 2.0 ** -20})")
    pm = np.zeros((n, 4), np.float32)
    pm[:, :3] = W.Stream(n).uniform(3 * n, -1.0, 1.0).reshape(n, 3)
    pm[:, 3] = 1.0
    got = gpu_forces(pm, 2.0 ** 40, path=SYM, splits=splits).astype(np.float64)
    assert np.isfinite(got).all()
    count = -got[:, 3] / t
    if t == 2.0 ** -20:
        assert np.array_equal(count, np.full(n, float(n))), (count.min(), count.max())
    else:   # fp32 sums of an inexact t: rounding well below one count
        assert np.abs(count - n).max() < 0.25, (count.min(), count.max())


@pytest.mark.slow
def test_symmetric_path_partials_past_2_34_bytes():
    """n = 2^21 + 7: 1025 blocks (odd) with a ragged last one.  With a
    caller's workspace large enough for every group in one pass, the partial
    offsets pass 2^34 bytes; the result is bit-identical to the default call
    (one group per pass, within the default budget), and every body met
    every body exactly once."""
    n = 2 ** 21 + 7
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    base = apg.nbody_plan_forces(n, sm)
    assert base["num_iblocks"] == 1025 and base["passes"] > 1
    one = apg.nbody_plan_forces(n, sm, workspace_bytes=1 << 40)
    assert one["passes"] == 1 and one["scratch_bytes"] > 2 ** 34
    pm = np.zeros((n, 4), np.float32)
    pm[:, :3] = W.Stream(n).uniform(3 * n, -1.0, 1.0).reshape(n, 3)
    pm[:, 3] = 1.0
    d_pm = torch.from_numpy(pm).to(dev())
    ws = torch.empty(one["scratch_bytes"], dtype=torch.uint8, device=dev())
    a = apg.nbody_forces_ws(d_pm, 2.0 ** 40, workspace=ws)
    del ws
    b = apg.nbody_forces(d_pm, 2.0 ** 40)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    test_symmetric_path_counts_every_pair_once(n, 0)


@pytest.mark.parametrize("n", [10239, 10240, 45055, 45056, 327679, 327680])
def test_planner_switch_points(n):
    """Either side of each automatic switch: row-split to symmetric at 10240,
    512- to 1024-body blocks at 45056, 1024- to 2048-body blocks at 327680."""
    w = W.clumps(n, seed=n % 997)
    acc = gpu_forces(w.pos_mass, w.eps2)
    rows = np.unique(np.concatenate([sample_rows(n, 600, 11), np.arange(n - 64, n)]))
    assert_parity(acc, oracle.forces(w.pos_mass, w.eps2, rows=rows), rows)


def test_symmetric_path_deterministic_and_ts_identical():
    w = W.clumps(70001, seed=9)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    a = apg.nbody_forces_ex(pm, float(w.eps2), path=SYM)
    for _ in range(2):
        assert torch.equal(apg.nbody_forces_ex(pm, float(w.eps2), path=SYM), a)
    assert torch.equal(apg.nbody_forces(pm, float(w.eps2)), a)        # automatic choice
    assert torch.equal(apg.nbody_forces_ts(pm, pm, float(w.eps2)), a)  # same array
    torch.cuda.synchronize()


def test_symmetric_path_needs_one_array():
    """The target/source form with distinct arrays never takes the symmetric
    path: with a copy of the bodies as sources it matches the oracle too."""
    w = W.clumps(40000, seed=12)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    out = apg.nbody_forces_ts(pm, pm.clone(), float(w.eps2))
    torch.cuda.synchronize()
    rows = sample_rows(w.n, 1500, 3)
    assert_parity(out.cpu().numpy()[rows], oracle.forces(w.pos_mass, w.eps2, rows=rows))


# ------------------------------------------------------------ target/source form

def _ts_bodies(nt, ns, seed):
    st = W.Stream(seed)
    t = np.zeros((nt, 4), np.float32)
    t[:, :3] = st.uniform(3 * nt, -1.5, 1.5).reshape(nt, 3)
    t[:, 3] = st.uniform(nt, 5.0, 9.0)             # never read
    s = np.zeros((ns, 4), np.float32)
    s[:, :3] = st.uniform(3 * ns, -1.0, 1.0).reshape(ns, 3)
    s[:, 3] = st.uniform(ns, 0.5, 1.5)
    return t, s


@pytest.mark.parametrize("nt,ns", [(1, 1), (1, 1000), (1000, 1), (100, 5000), (5000, 100),
                                   (3000, 20000), (20000, 3000), (77777, 1025), (1025, 77777)])
def test_target_source_form(nt, ns):
    t, s = _ts_bodies(nt, ns, nt * 7 + ns)
    eps2 = np.float32(1e-3)
    out = apg.nbody_forces_ts(torch.from_numpy(t).to(dev()), torch.from_numpy(s).to(dev()),
                              float(eps2))
    torch.cuda.synchronize()
    assert_parity(out.cpu().numpy(), oracle.forces_ts(t, s, eps2))


@pytest.mark.parametrize("path,splits", [(1, 7), (1, 1), (4, 3)])
def test_target_source_forced_launch_options(path, splits):
    """The target/source call within a workspace, with a forced path and
    piece count: tiled pieces through the workspace and the row-split path's
    pieces in shared memory."""
    t, s = _ts_bodies(3000, 9000, 41)
    eps2 = np.float32(1e-3)
    tt, st = torch.from_numpy(t).to(dev()), torch.from_numpy(s).to(dev())
    plan = apg.nbody_plan_forces_ts(3000, 9000, sm_count_of_device(), path=path, splits=splits)
    assert plan["path"] == path and plan["splits"] == splits
    ws = torch.empty(max(16, plan["scratch_bytes"]), dtype=torch.uint8, device=dev())
    out = apg.nbody_forces_ts_ws(tt, st, float(eps2), workspace=ws, path=path, splits=splits)
    torch.cuda.synchronize()
    assert_parity(out.cpu().numpy(), oracle.forces_ts(t, s, eps2))


def sm_count_of_device():
    return torch.cuda.get_device_properties(dev()).multi_processor_count


def test_target_source_golden_three_body():
    """The worked three-body example through the target/source form: target 0
    against the three bodies."""
    pm = np.array([[0, 0, 0, 1.5], [3, 4, 0, 2], [1, 4, 8, 0.25]], np.float32)
    tgt = torch.from_numpy(pm[:1].copy()).to(dev())
    out = apg.nbody_forces_ts(tgt, torch.from_numpy(pm).to(dev()), 144.0).cpu().numpy()
    exp = [6 / 2197 + 1 / 13500, 8 / 2197 + 1 / 3375, 2 / 3375, -2 / 13 - 1 / 60 - 1 / 8]
    np.testing.assert_allclose(out[0].astype(np.float64), exp, rtol=2e-6)


def test_target_source_no_sources_writes_zeros():
    t = torch.full((37, 4), 3.0, device=dev())
    out = torch.full_like(t, float("nan"))
    apg.nbody_forces_ts(t, torch.empty((0, 4), device=dev()), 1e-4, out)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


@pytest.mark.parametrize("n", [1000, 30011])
def test_target_source_equals_all_pairs_when_same_array(n):
    w = W.clumps(n, seed=n)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    a = apg.nbody_forces(pm, float(w.eps2))
    b = apg.nbody_forces_ts(pm, pm, float(w.eps2))
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# ------------------------------------------------------------ multi-step driver

def _separate_steps(w, steps):
    pm = torch.from_numpy(w.pos_mass).to(dev())
    vel = torch.from_numpy(w.vel).to(dev())
    acc = torch.empty_like(pm)
    for _ in range(steps):
        apg.nbody_forces(pm, float(w.eps2), acc)
        apg.nbody_euler_step(pm, vel, acc, float(w.dt))
    torch.cuda.synchronize()
    return pm, vel, acc


@pytest.mark.parametrize("name,steps", [("smallcube1024", 20), ("smallcube1024", 7),
                                        ("smallcube1024", 37), ("smallcube4096", 3),
                                        ("smallcube8192", 4), ("smallcube8192", 33),
                                        ("cube16384", 17), ("plummer65536", 10),
                                        ("clumps200003", 2)])
def test_simulate_is_the_separate_calls(name, steps):
    """Row-split path (1024, 4096, 8192: fused pairs of steps) and symmetric
    path (16384, 65536, 200003); 37, 33 and 17 steps run through the
    16-step batch graph and then the pair and single-step graphs."""
    w = W.named(name)
    ref = _separate_steps(w, steps)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    vel = torch.from_numpy(w.vel).to(dev())
    acc = torch.empty_like(pm)
    apg.nbody_simulate(pm, vel, acc, float(w.eps2), float(w.dt), steps)
    torch.cuda.synchronize()
    for got, exp in zip((pm, vel, acc), ref):
        assert torch.equal(got, exp)


def test_simulate_graph_cache_rebuilds():
    """Alternate between two problems (the cached graph is rebuilt each time)
    and repeat one (the cached graph is replayed): every result matches."""
    wa, wb = W.small_cube(2048), W.plummer(20000, seed=3, eps=0.01)
    bufs = {}
    for w in (wa, wb):
        pm = torch.from_numpy(w.pos_mass).to(dev())
        bufs[w.name] = (w, pm, torch.from_numpy(w.vel).to(dev()), torch.empty_like(pm))
    plan = [("smallcube2048", 3), ("plummer20000", 2), ("smallcube2048", 1), ("smallcube2048", 4)]
    done = {"smallcube2048": 0, "plummer20000": 0}
    for name, k in plan:
        w, pm, vel, acc = bufs[name]
        apg.nbody_simulate(pm, vel, acc, float(w.eps2), float(w.dt), k)
        done[name] += k
    torch.cuda.synchronize()
    for name, (w, pm, vel, acc) in bufs.items():
        ref = _separate_steps(w, done[name])
        assert torch.equal(pm, ref[0]) and torch.equal(vel, ref[1]) and torch.equal(acc, ref[2])


def test_simulate_zero_steps_is_a_noop():
    w = W.small_cube(1024)
    pm = torch.from_numpy(w.pos_mass).to(dev())
    vel = torch.from_numpy(w.vel).to(dev())
    acc = torch.zeros_like(pm)
    apg.nbody_simulate(pm, vel, acc, float(w.eps2), float(w.dt), 0)
    torch.cuda.synchronize()
    assert np.array_equal(pm.cpu().numpy(), w.pos_mass) and torch.count_nonzero(acc).item() == 0


# ------------------------------------------------------------ large arrays (64-bit offsets)

@pytest.mark.slow
def test_huge_source_array():
    """2^26 + 5 sources (1 GiB): source offsets past 2^31 bytes, a ragged last
    tile, hundreds of source splits; 300 targets checked against the oracle."""
    ns, nt = 2 ** 26 + 5, 300
    st = W.Stream(99)
    s = np.empty((ns, 4), np.float32)
    s[:, :3] = st.uniform(3 * ns, -1.0, 1.0).reshape(ns, 3)
    s[:, 3] = np.float32(1.0 / ns)
    t = np.zeros((nt, 4), np.float32)
    t[:, :3] = st.uniform(3 * nt, -0.5, 0.5).reshape(nt, 3)
    out = apg.nbody_forces_ts(torch.from_numpy(t).to(dev()), torch.from_numpy(s).to(dev()), 1e-4)
    torch.cuda.synchronize()
    assert_parity(out.cpu().numpy(), oracle.forces_ts(t, s, np.float32(1e-4)))


@pytest.mark.slow
def test_huge_target_array():
    """2^26 targets (1 GiB in, 1 GiB out) against 77 sources: target and
    output offsets past 2^31 bytes; sampled rows, the last ones included."""
    nt, ns = 2 ** 26, 77
    st = W.Stream(98)
    t = np.empty((nt, 4), np.float32)
    t[:, :3] = st.uniform(3 * nt, -2.0, 2.0).reshape(nt, 3)
    t[:, 3] = 0.0
    s = np.zeros((ns, 4), np.float32)
    s[:, :3] = st.uniform(3 * ns, -1.0, 1.0).reshape(ns, 3)
    s[:, 3] = st.uniform(ns, 0.5, 1.5)
    out = apg.nbody_forces_ts(torch.from_numpy(t).to(dev()), torch.from_numpy(s).to(dev()), 1e-3)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([sample_rows(nt, 4000, 7), np.arange(nt - 1100, nt)]))
    got = out[torch.from_numpy(rows).to(dev())].cpu().numpy()
    assert_parity(got, oracle.forces_ts(t[rows], s, np.float32(1e-3)))


# ------------------------------------------------------------ compensated precision

def test_compensated_precision_on_the_ill_conditioned_disk():
    """Body 1888 of the disk workload has near neighbours 380x |a_i|
    (condition number 1244): the compensated kernel cuts its error well
    below the default kernel's."""
    w = W.named("disk4096")
    ref = oracle.forces(w.pos_mass, w.eps2)
    base = errors(gpu_forces(w.pos_mass, w.eps2), ref, potential=False)
    comp = errors(gpu_forces(w.pos_mass, w.eps2, precision=apg.NBODY_PRECISION_COMPENSATED), ref,
                  potential=False)
    assert comp["body_a"] <= 3e-5 and comp["body_a"] < 0.6 * base["body_a"], (base, comp)
    assert comp["l2_a"] <= base["l2_a"]


@pytest.mark.parametrize("name", ["cube16384", "clumps200003"])
def test_compensated_precision_parity(name):
    w = W.named(name)
    got = gpu_forces(w.pos_mass, w.eps2, precision=apg.NBODY_PRECISION_COMPENSATED)
    rows = np.arange(w.n) if w.n <= 20000 else sample_rows(w.n, 1500, 4)
    e = assert_parity(got, oracle.forces(w.pos_mass, w.eps2, rows=rows), rows)
    assert e["l2_a"] <= 1e-6 and e["l2_p"] <= 1e-6, e


@pytest.mark.slow
def test_plummer1048576_properties_of_every_output():
    """All 2^20 outputs of the benchmark workload, through properties that hold
    at any size: Newton's third law over every body, and the binned radial
    acceleration and potential of the (r <= 10 truncated) Plummer profile."""
    w = W.named("plummer1048576")
    acc = gpu_forces(w.pos_mass, w.eps2).astype(np.float64)
    assert np.isfinite(acc).all()
    m = w.pos_mass[:, 3].astype(np.float64)
    x = w.pos_mass[:, :3].astype(np.float64)
    total = np.abs((m[:, None] * acc[:, :3]).sum(0)).max()
    assert total < 1e-6 * (m[:, None] * np.abs(acc[:, :3])).sum()
    r = np.linalg.norm(x, axis=1)
    ar = (acc[:, :3] * x).sum(1) / r
    mass = lambda rr: rr ** 3 / (1.0 + rr * rr) ** 1.5
    mtrunc = mass(10.0)
    for lo, hi in [(0.3, 0.6), (0.6, 1.0), (1.0, 2.0), (2.0, 4.0), (4.0, 8.0)]:
        sel = (r >= lo) & (r < hi)
        model = -(mass(r[sel]) / mtrunc) / r[sel] ** 2
        assert abs(ar[sel].mean() / model.mean() - 1.0) < 0.01, (lo, hi)
    # potential without the self term; the r <= 10 truncated profile has
    # phi(r) = -[(1 + r^2)^(-1/2) - 101^(-3/2)] / M(10) inside the cut
    pself = acc[:, 3] + m / np.sqrt(float(w.eps2))
    for lo, hi in [(0.3, 1.0), (1.0, 3.0), (3.0, 8.0)]:
        sel = (r >= lo) & (r < hi)
        model = -(1.0 / np.sqrt(1.0 + r[sel] ** 2) - 101.0 ** -1.5) / mtrunc
        assert abs(pself[sel].mean() / model.mean() - 1.0) < 0.01, (lo, hi)


# ------------------------------------------------------------ acceleration only

def gpu_forces_acc(pm_np, eps2, **kw):
    pm = torch.from_numpy(np.ascontiguousarray(pm_np)).to(dev())
    acc = apg.nbody_forces_ex(pm, float(eps2), quantities=apg.NBODY_QUANTITIES_ACC, **kw)
    torch.cuda.synchronize()
    return acc.cpu().numpy()


def test_disk4096_acceleration_only():
    """The disk workload checks the acceleration only: nbody_forces_acc
    against the oracle over every body, its .w exactly 0."""
    w = W.named("disk4096")
    pm = torch.from_numpy(w.pos_mass).to(dev())
    got = apg.nbody_forces_acc(pm, float(w.eps2))
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    assert np.all(got[:, 3] == 0.0)
    assert_parity(got, oracle.forces(w.pos_mass, w.eps2), potential=False)


@pytest.mark.parametrize("path", [1, 2, 3, 4])
@pytest.mark.parametrize("n", [1, 1000, 5003, 20011])
def test_acceleration_only_every_path(path, n):
    """Each kernel without its potential operations: the acceleration is the
    same arithmetic, so it matches the a + p call bit for bit; .w is 0."""
    if path == 4 and n > 12000:   # the row-split path holds every source in shared memory
        n = 12000
    w = W.clumps(n, seed=n + 5)
    if path == 2 and n > 4864:
        path = 1
    full = gpu_forces(w.pos_mass, w.eps2, path=path)
    acc = gpu_forces_acc(w.pos_mass, w.eps2, path=path)
    assert np.array_equal(acc[:, :3], full[:, :3])
    assert np.all(acc[:, 3] == 0.0)
    assert_parity(acc, oracle.forces(w.pos_mass, w.eps2), potential=False)


def test_acceleration_only_target_source_form():
    t, s = _ts_bodies(3000, 20000, 77)
    tt, ss = torch.from_numpy(t).to(dev()), torch.from_numpy(s).to(dev())
    ws = torch.empty(0, device=dev())
    out = apg.nbody_forces_ts_ws(tt, ss, 1e-3, workspace=ws, quantities=apg.NBODY_QUANTITIES_ACC)
    full = apg.nbody_forces_ts(tt, ss, 1e-3)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out[:, 3]).item() == 0
    # the same plan with the potential: identical accelerations
    assert torch.equal(out[:, :3], apg.nbody_forces_ts_ws(tt, ss, 1e-3, workspace=ws)[:, :3])
    assert_parity(out.cpu().numpy(), oracle.forces_ts(t, s, np.float32(1e-3)), potential=False)


@pytest.mark.slow
def test_plummer1048576_acceleration_only_sampled():
    """The full-size workload without the potential, in the default plan:
    sampled rows, the dense core included."""
    w = W.named("plummer1048576")
    acc = gpu_forces_acc(w.pos_mass, w.eps2)
    rows = _hard_rows(w, 2048, seed=12)
    assert_parity(acc, oracle.forces(w.pos_mass, w.eps2, rows=rows), rows, potential=False)
    assert np.all(acc[:, 3] == 0.0)


# ------------------------------------------------------------ concurrency

def test_concurrent_host_threads_and_streams():
    """Four host threads, each with its own stream and problem, call the
    library at the same time (the C calls run without the GIL): per-device
    set-up, the split scratch pool and the launches are thread-safe, and
    each result matches the same call made alone."""
    import threading
    sizes = [3001, 20011, 70001, 4096]
    work = [W.clumps(n, seed=40 + n) for n in sizes]
    alone = [gpu_forces(w.pos_mass, w.eps2) for w in work]
    outs = [None] * len(work)
    errs = []

    def run(k):
        try:
            st = torch.cuda.Stream()
            w = work[k]
            with torch.cuda.stream(st):
                pm = torch.from_numpy(w.pos_mass).to(dev(), non_blocking=False)
                acc = torch.empty_like(pm)
                for _ in range(3):
                    apg.nbody_forces(pm, float(w.eps2), acc)
            st.synchronize()
            outs[k] = acc.cpu().numpy()
        except Exception as e:                       # reported below
            errs.append(e)

    threads = [threading.Thread(target=run, args=(k,)) for k in range(len(work))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errs, errs
    for k in range(len(work)):
        assert np.array_equal(outs[k], alone[k]), sizes[k]


def test_simulate_from_two_threads_alternately():
    """nbody_simulate's per-device graph cache under two threads that take
    turns with different problems: every trajectory equals the separate
    calls."""
    import threading
    wa, wb = W.small_cube(1024), W.plummer(30000, seed=5, eps=0.01)
    ref = {w.name: _separate_steps(w, 6) for w in (wa, wb)}
    got = {}
    lock = threading.Lock()

    def run(w):
        pm = torch.from_numpy(w.pos_mass).to(dev())
        vel = torch.from_numpy(w.vel).to(dev())
        acc = torch.empty_like(pm)
        st = torch.cuda.Stream()
        for _ in range(3):
            with lock:                      # interleave the two problems' calls
                with torch.cuda.stream(st):
                    apg.nbody_simulate(pm, vel, acc, float(w.eps2), float(w.dt), 2)
        st.synchronize()
        got[w.name] = (pm, vel, acc)

    threads = [threading.Thread(target=run, args=(w,)) for w in (wa, wb)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    for name, (pm, vel, acc) in got.items():
        assert torch.equal(pm, ref[name][0]) and torch.equal(vel, ref[name][1])
        assert torch.equal(acc, ref[name][2])
