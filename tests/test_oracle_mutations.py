"""Planted mistakes: each mutant of the oracle must fail at least one pin.

Every mutant is a copy of ``oracle/nbody_oracle.c`` with one plausible slip,
compiled into a temporary library on the CPU. The checks below are the same
facts that ``test_oracle_pins.py`` holds the oracle to (worked examples, the
shell theorem, hand-rounded Euler values).
"""
import ctypes
import json
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

from test_oracle_pins import GOLDEN, _q, _fib_sphere

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "nbody_oracle.c")

MUTANTS = {
    "r_sign": ("(double)sources[4 * j + 0] - xi", "xi - (double)sources[4 * j + 0]"),
    "exponent_1": ("mj * inv * inv * inv", "mj * inv * inv"),
    "eps_not_squared": ("+ e2;", "+ sqrt(e2);"),
    "potential_sign": ("p -= mj * inv;", "p += mj * inv;"),
    "transposed_y_z": ("ay += s * ry;", "ay += s * rz;"),
    "target_mass": ("const double mj = (double)sources[4 * j + 3];",
                    "const double mj = (double)targets[4 * t + 3];"),
    "dropped_z": ("rx * rx + ry * ry + rz * rz + e2", "rx * rx + ry * ry + e2"),
    "skip_self_potential": ("p -= mj * inv;", "if (d2 != e2) p -= mj * inv;"),
    "euler_fma": ("pos_mass[4 * i + c] = pos_mass[4 * i + c] + step_x;",
                  "pos_mass[4 * i + c] = fmaf(dt, v_old, pos_mass[4 * i + c]);"),
    "euler_velocity_first": ("const float v_old = vel[4 * i + c];",
                             "const float v_old = vel[4 * i + c] + dt * acc_pot[4 * i + c];"),
}


def _build(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    str(path), "-o", str(so), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    lib.oracle_forces_ts.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                     ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int]
    lib.oracle_euler.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                 ctypes.c_int64, ctypes.c_float]
    return lib


def _forces(lib, targets, sources, eps2):
    t = np.ascontiguousarray(targets, np.float32)
    s = np.ascontiguousarray(sources, np.float32)
    out = np.empty((t.shape[0], 4))
    lib.oracle_forces_ts(t.ctypes.data, t.shape[0], s.ctypes.data, s.shape[0],
                         ctypes.c_float(eps2), out.ctypes.data, 1)
    return out


def _pins_hold(lib) -> bool:
    for name in ["two_body_collinear", "two_body_3d", "three_body_target", "single_body"]:
        fx = json.load(open(os.path.join(GOLDEN, name + ".json")))
        bodies = np.array([[float(_q(c)) for c in b] for b in fx["bodies"]], np.float32)
        got = _forces(lib, bodies[fx["rows"]], bodies, float(_q(fx["eps2"])))
        exp = np.array([[float(_q(e)) for e in r] for r in fx["expected"]])
        if not np.allclose(got, exp, rtol=1e-13, atol=1e-300):
            return False
    n = 2000
    shell = np.zeros((n, 4), np.float32)
    shell[:, :3] = _fib_sphere(n)
    shell[:, 3] = 1.0 / n
    probe = np.array([[0.2, -0.1, 0.3, 0], [2, 0, 0, 0]], np.float32)
    out = _forces(lib, probe, shell, 1e-12)
    if np.abs(out[0, :3]).max() > 1e-3 or not np.allclose(out[1, :3], [-0.25, 0, 0], atol=1e-3):
        return False
    # Euler: exactly representable step, then a case where rounding matters
    pm = np.array([[1.0, 2.0, -3.0, 7.0]], np.float32)
    v = np.array([[0.5, -0.25, 2.0, 9.0]], np.float32)
    a = np.array([[4.0, 8.0, -16.0, -1.0]], np.float32)
    lib.oracle_euler(pm.ctypes.data, v.ctypes.data, a.ctypes.data, 1, ctypes.c_float(0.125))
    if pm[0].tolist() != [1.0625, 1.96875, -2.75, 7.0] or v[0].tolist() != [1.0, 0.75, 0.0, 9.0]:
        return False
    from test_oracle_pins import euler_rounding_cases
    for x, v0, dt, sep, fused in euler_rounding_cases(40):
        pm = np.array([[x, x, x, 1]], np.float32)
        vel = np.array([[v0, v0, v0, 0]], np.float32)
        acc = np.zeros((1, 4), np.float32)
        lib.oracle_euler(pm.ctypes.data, vel.ctypes.data, acc.ctypes.data, 1, ctypes.c_float(dt))
        if Fraction(float(pm[0, 0])) != sep:
            return False
    return True


def test_unmutated_oracle_passes(tmp_path):
    src = open(SRC).read()
    lib = _build(tmp_path, "identity", src[:40], src[:40])
    assert _pins_hold(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _build(tmp_path, name, old, new)
    assert not _pins_hold(lib), f"mutant {name} slipped past the pins"
