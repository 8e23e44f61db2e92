"""Pins for the oracle: each test ties it to something other than its own code.

A plausible slip anywhere in the oracle (a dropped term, a wrong sign, the
target's mass used for the source's, the exponent 1 for 3/2, eps for eps^2, a
transposed component, a missing self term in the potential, an FMA in the Euler
step, velocities advanced before positions) fails at least one test here.
"""
import json
import math
import os
import re
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

import oracle
from all_pairs_gravitational_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _q(expr: str) -> Fraction:
    """Exact value of a fixture expression such as '-2/13 - 1/60 - 1/8'."""
    terms = re.findall(r"[+-]?\d+(?:/\d+)?", expr.replace(" ", ""))
    assert "".join(terms) == expr.replace(" ", ""), expr
    return sum((Fraction(t) for t in terms), Fraction(0))


@pytest.mark.parametrize("name", ["two_body_collinear", "two_body_3d", "three_body_target",
                                  "single_body"])
def test_golden_worked_examples(name):
    with open(os.path.join(GOLDEN, name + ".json")) as f:
        fx = json.load(f)
    bodies = np.array([[float(_q(c)) for c in b] for b in fx["bodies"]], dtype=np.float32)
    # the fixtures use values that fp32 holds exactly
    for b, row in zip(fx["bodies"], bodies):
        assert all(Fraction(float(v)) == _q(c) for c, v in zip(b, row))
    eps2 = np.float32(float(_q(fx["eps2"])))
    got = oracle.forces(bodies, eps2, rows=fx["rows"])
    for r, exp_row in enumerate(fx["expected"]):
        for c, e in enumerate(exp_row):
            e = float(_q(e))
            assert got[r, c] == pytest.approx(e, rel=1e-14, abs=1e-300), (name, r, c)


def test_single_body_self_term_is_exact():
    pm = np.array([[0.3, -0.7, 0.1, 2.0]], dtype=np.float32)
    out = oracle.forces(pm, np.float32(0.0625))
    assert out[0, :3].tolist() == [0.0, 0.0, 0.0]
    assert out[0, 3] == -2.0 / 0.25


def _fib_sphere(n, radius=1.0):
    k = np.arange(n) + 0.5
    cz = 1.0 - 2.0 * k / n
    phi = np.pi * (1.0 + 5.0 ** 0.5) * k
    sz = np.sqrt(1.0 - cz * cz)
    return radius * np.stack([sz * np.cos(phi), sz * np.sin(phi), cz], axis=1)


def test_shell_theorem():
    """A thin uniform shell: no field inside, a point mass outside (Newton's
    shell theorem; holds only for the inverse-square law)."""
    n = 6000
    pm = np.zeros((n, 4), np.float32)
    pm[:, :3] = _fib_sphere(n)
    pm[:, 3] = np.float32(1.0 / n)
    M = float(pm[:, 3].astype(np.float64).sum())
    eps2 = np.float32(1e-12)
    inside = np.array([[0, 0, 0, 0], [0.3, -0.2, 0.1, 0], [0, 0.5, 0, 0], [-0.4, 0.1, -0.3, 0]],
                      np.float32)
    out = oracle.forces_ts(inside, pm, eps2)
    assert np.abs(out[:, :3]).max() < 2e-4 * M                 # field ~ 0 (scale M/R^2 = 1)
    np.testing.assert_allclose(out[:, 3], -M, rtol=2e-4)        # potential -M/R
    outside = np.array([[2, 0, 0, 0], [0, -3, 0, 0], [1.5, 1.5, 1.5, 0]], np.float32)
    out = oracle.forces_ts(outside, pm, eps2)
    for t, o in zip(outside.astype(np.float64), out):
        r = np.linalg.norm(t[:3])
        np.testing.assert_allclose(o[:3], -M * t[:3] / r ** 3, rtol=1e-4, atol=1e-6)
        assert o[3] == pytest.approx(-M / r, rel=1e-4)


def test_target_mass_is_not_used():
    """Targets' fourth lane is never read: only source masses enter."""
    src = W.cube(64, seed=7).pos_mass
    t = src[:5].copy()
    a = oracle.forces_ts(t, src, np.float32(1e-3))
    t[:, 3] = np.float32(123.0)
    b = oracle.forces_ts(t, src, np.float32(1e-3))
    assert np.array_equal(a, b)


def _brute_decimal(bodies, eps2):
    """Independent textbook loop in 60-digit decimal: sources j != i, then the
    target's own potential term added back separately."""
    getcontext().prec = 60
    B = [[Decimal(float(v)) for v in b] for b in bodies]
    e2 = Decimal(float(eps2))
    res = []
    for i, bi in enumerate(B):
        acc = [Decimal(0)] * 3
        pot = Decimal(0)
        for j, bj in enumerate(B):
            if j == i:
                continue
            r = [bj[c] - bi[c] for c in range(3)]
            d = r[0] * r[0] + r[1] * r[1] + r[2] * r[2] + e2
            root = d.sqrt()
            for c in range(3):
                acc[c] += bj[3] * r[c] / (d * root)
            pot -= bj[3] / root
        pot -= bi[3] / e2.sqrt()
        res.append([float(acc[0]), float(acc[1]), float(acc[2]), float(pot)])
    return np.array(res)


@pytest.mark.parametrize("n,seed", [(2, 1), (3, 2), (5, 3), (8, 4)])
def test_brute_force_small_n(n, seed):
    s = W.Stream(seed)
    pm = np.zeros((n, 4), np.float32)
    pm[:, :3] = s.uniform(3 * n, -1, 1).reshape(n, 3)
    pm[:, 3] = s.uniform(n, 0.1, 2.0)
    eps2 = np.float32(0.01)
    got = oracle.forces(pm, eps2)
    ref = _brute_decimal(pm, eps2)
    # scale: the sum of the magnitudes of the terms, per row
    scale = np.abs(ref).max()
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-13 * scale)


def test_newtons_third_law():
    """Pair forces are equal and opposite: sum_i m_i a_i = 0."""
    w = W.clumps(3001, seed=11)
    out = oracle.forces(w.pos_mass, w.eps2)
    m = w.pos_mass[:, 3].astype(np.float64)[:, None]
    total = (m * out[:, :3]).sum(axis=0)
    scale = (m * np.abs(out[:, :3])).sum()
    assert np.abs(total).max() < 1e-12 * scale


def test_potential_energy_symmetry():
    """phi_ij = phi_ji: sum_i m_i p_i is unchanged by reordering the bodies,
    and equals twice the pair energy plus the self terms."""
    w = W.cube(500, seed=5)
    eps2 = w.eps2
    out = oracle.forces(w.pos_mass, eps2)
    m = w.pos_mass[:, 3].astype(np.float64)
    e1 = (m * out[:, 3]).sum()
    perm = np.random.default_rng(0).permutation(w.n)
    out2 = oracle.forces(w.pos_mass[perm], eps2)
    e2 = (m[perm] * out2[:, 3]).sum()
    assert e1 == pytest.approx(e2, rel=1e-13)
    x = w.pos_mass[:, :3].astype(np.float64)
    d = np.sqrt(((x[:, None, :] - x[None, :, :]) ** 2).sum(-1) + float(eps2))
    iu = np.triu_indices(w.n, 1)
    pair = -(m[iu[0]] * m[iu[1]] / d[iu]).sum()
    self_terms = -(m * m).sum() / math.sqrt(float(eps2))
    assert e1 == pytest.approx(2 * pair + self_terms, rel=1e-12)


def test_permutation_equivariance():
    w = W.cube(300, seed=9)
    perm = np.random.default_rng(1).permutation(w.n)
    a = oracle.forces(w.pos_mass, w.eps2)
    b = oracle.forces(w.pos_mass[perm], w.eps2)
    np.testing.assert_allclose(b, a[perm], rtol=1e-12, atol=1e-12 * np.abs(a).max())


def test_scaling_laws():
    """a(lx, l^2 eps^2) = a/l^2, p(lx, l^2 eps^2) = p/l; a and p are linear in m.
    Powers of two keep the fp32 inputs exact."""
    w = W.clumps(400, seed=3)
    base = oracle.forces(w.pos_mass, w.eps2)
    lam = 4.0
    pm = w.pos_mass.copy()
    pm[:, :3] *= np.float32(lam)
    sc = oracle.forces(pm, np.float32(w.eps2 * np.float32(lam * lam)))
    np.testing.assert_allclose(sc[:, :3], base[:, :3] / lam ** 2, rtol=1e-12,
                               atol=1e-12 * np.abs(base[:, :3]).max())
    np.testing.assert_allclose(sc[:, 3], base[:, 3] / lam, rtol=1e-12)
    pm = w.pos_mass.copy()
    pm[:, 3] *= np.float32(8.0)
    ms = oracle.forces(pm, w.eps2)
    np.testing.assert_allclose(ms, base * 8.0, rtol=1e-12, atol=1e-12 * np.abs(base).max())


def test_rows_select_targets():
    w = W.cube(257, seed=2)
    full = oracle.forces(w.pos_mass, w.eps2)
    rows = [0, 5, 256, 100, 5]
    part = oracle.forces(w.pos_mass, w.eps2, rows=rows)
    assert np.array_equal(part, full[rows])


def _plummer_mass(r):
    return r ** 3 / (1.0 + r * r) ** 1.5


def test_plummer_mean_field():
    """Binned radial acceleration of a sampled Plummer sphere follows the
    analytic field of the (r <= 10 truncated) profile, -M(<r)/r^2."""
    w = W.plummer(40000, seed=123, eps=0.01)
    r = np.linalg.norm(w.pos_mass[:, :3].astype(np.float64), axis=1)
    rng = np.random.default_rng(0)
    rows = rng.choice(w.n, 1500, replace=False)
    out = oracle.forces(w.pos_mass, w.eps2, rows=rows)
    x = w.pos_mass[rows, :3].astype(np.float64)
    rr = r[rows]
    ar = (out[:, :3] * x).sum(1) / rr
    mtrunc = _plummer_mass(10.0)
    for lo, hi in [(0.5, 1.0), (1.0, 2.0), (2.0, 4.0)]:
        sel = (rr >= lo) & (rr < hi)
        model = -(_plummer_mass(rr[sel]) / mtrunc) / rr[sel] ** 2
        ratio = ar[sel].mean() / model.mean()
        assert abs(ratio - 1.0) < 0.03, (lo, hi, ratio)
    # potential minus the self term, at mid radii: -1/sqrt(1+r^2) up to truncation
    pself = out[:, 3] + w.pos_mass[rows, 3].astype(np.float64) / math.sqrt(float(w.eps2))
    sel = (rr > 0.5) & (rr < 2.0)
    model = -1.0 / np.sqrt(1.0 + rr[sel] ** 2)
    assert abs(pself[sel].mean() / model.mean() - 1.0) < 0.03


def test_empty_and_bad_arguments():
    out = oracle.forces(np.zeros((0, 4), np.float32), np.float32(1.0))
    assert out.shape == (0, 4)
    lib = oracle._load()
    assert lib.oracle_forces_ts(None, -1, None, 0, 1.0, None, 0) == -1
    assert lib.oracle_euler(None, None, None, -1, 1.0) == -1


# ---------------------------------------------------------------- Euler


def _rne_f32(q: Fraction) -> Fraction:
    """Round a rational to the nearest fp32 (ties to even), normal range only."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (e - 23)
    k = a / ulp
    fl = math.floor(k)
    rem = k - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * ulp


def test_euler_hand_values_and_order():
    """Exactly representable case: positions must move with the OLD velocity."""
    pm = np.array([[1.0, 2.0, -3.0, 7.0]], np.float32)
    v = np.array([[0.5, -0.25, 2.0, 9.0]], np.float32)
    a = np.array([[4.0, 8.0, -16.0, -1.0]], np.float32)
    pm2, v2 = oracle.euler(pm, v, a, np.float32(0.125))
    assert pm2.tolist() == [[1.0625, 1.96875, -2.75, 7.0]]
    assert v2.tolist() == [[1.0, 0.75, 0.0, 9.0]]


def euler_rounding_cases(count=200, seed=2024):
    """Seeded (x, v, dt) triples with the exact separately-rounded x + dt*v and
    the fused result, both by exact rational arithmetic rounded by hand. dt*v is
    of the same magnitude as x, so the product's rounding reaches the sum's."""
    s = W.Stream(seed)
    fq = lambda t: Fraction(float(t))
    cases = []
    for _ in range(count):
        x, v, dt = (np.float32(t) for t in s.uniform(3, 0.5, 2.0))
        sep = _rne_f32(fq(x) + _rne_f32(fq(dt) * fq(v)))
        fused = _rne_f32(fq(x) + fq(dt) * fq(v))
        cases.append((x, v, dt, sep, fused))
    return cases


def test_euler_rounds_product_and_sum_separately():
    """Each product dt*v is rounded to fp32 before the add (no fused multiply-add)."""
    found = 0
    for x, v, dt, sep, fused in euler_rounding_cases():
        pm = np.array([[x, x, x, 1]], np.float32)
        vel = np.array([[v, v, v, 0]], np.float32)
        acc = np.zeros((1, 4), np.float32)
        pm2, _ = oracle.euler(pm, vel, acc, dt)
        assert Fraction(float(pm2[0, 0])) == sep
        if sep != fused:
            found += 1
    assert found > 0   # at least one case where an FMA would have given another answer


def test_euler_velocity_uses_acceleration_and_keeps_w():
    w = W.disk(64, seed=3)
    acc = np.zeros((64, 4), np.float32)
    acc[:, :3] = W.Stream(5).uniform(192, -10, 10).reshape(64, 3)
    acc[:, 3] = -1.0
    dt = np.float32(1e-3)
    pm2, v2 = oracle.euler(w.pos_mass, w.vel, acc, dt)
    assert np.array_equal(pm2[:, 3], w.pos_mass[:, 3])
    assert np.array_equal(v2[:, 3], w.vel[:, 3])
    for i in range(0, 64, 7):
        for c in range(3):
            exp = _rne_f32(Fraction(float(w.vel[i, c])) +
                           _rne_f32(Fraction(float(dt)) * Fraction(float(acc[i, c]))))
            assert Fraction(float(v2[i, c])) == exp


# ---------------------------------------------------------------- fp64 trajectory

def test_forces_f64_is_the_pinned_definition_on_fp32_bodies():
    """On bodies fp32 holds exactly, the fp64-input entry point gives the bits
    of the pinned fp32-input one: the same arithmetic in the same order."""
    w = W.clumps(700, seed=31)
    eps2 = np.float32(w.eps2)
    got = oracle.forces_f64(w.pos_mass.astype(np.float64), float(eps2))
    assert np.array_equal(got, oracle.forces(w.pos_mass, eps2))


def test_trajectory_f64_free_body_moves_in_a_straight_line():
    """A lone body feels no force (its own term adds 0 to a): with dt a power
    of two and dyadic coordinates every fp64 step is exact."""
    pm = np.array([[0.5, -0.25, 2.0, 3.0]])
    v = np.array([[1.0, 0.5, -0.25, 0.0]])
    dt = 2.0 ** -10
    for k in (1, 7, 64):
        pm_k, v_k = oracle.trajectory_f64(pm, v, 1e-4, dt, k)
        assert np.array_equal(pm_k[:, :3], pm[:, :3] + k * dt * v[:, :3])
        assert np.array_equal(v_k, v) and pm_k[0, 3] == 3.0


def test_trajectory_f64_moves_positions_with_the_old_velocity():
    """From rest, one step leaves the positions where they were (they move
    with the velocity from before the step) and sets v = dt a; the next step
    moves them by dt^2 a."""
    pm = np.array([[0.0, 0.0, 0.0, 1.0], [3.0, 4.0, 0.0, 2.0]])
    v = np.zeros((2, 4))
    dt = 2.0 ** -4
    a0 = oracle.forces_f64(pm, 144.0)
    pm1, v1 = oracle.trajectory_f64(pm, v, 144.0, dt, 1)
    assert np.array_equal(pm1, pm)
    assert np.array_equal(v1[:, :3], dt * a0[:, :3])
    pm2, _ = oracle.trajectory_f64(pm, v, 144.0, dt, 2)
    assert np.array_equal(pm2[:, :3], pm[:, :3] + dt * (dt * a0[:, :3]))
    # the worked two-body value (distance 5, eps 12: |r|^2 + eps^2 = 13^2)
    assert a0[0, 0] == pytest.approx(2.0 * 3.0 / 13.0 ** 3, rel=1e-15)
