"""The oracle: a plain CPU statement of the all-pairs softened gravity path.

TEST INFRASTRUCTURE ONLY. The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the library
``all_pairs_gravitational_gb300`` never does, and the two share no code.

The arithmetic lives in ``nbody_oracle.c`` (fp64 accumulation, libm ``sqrt``,
sum over sources in index order, fp32 Euler with every product and sum rounded
separately). This module only builds that file with gcc and marshals numpy
arrays into it.

Function pins: every function here is pinned by ``tests/test_oracle_pins.py``
(worked two- and three-body values, the shell theorem, the Plummer field,
Newton's third law, brute force in 60-digit decimal arithmetic, scaling and
permutation laws, hand-rounded Euler values).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nbody_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``nbody_oracle.c`` into ``liboracle.so`` next to it (gcc, OpenMP).

    ``-ffp-contract=off`` keeps every fp32 product of the Euler step rounded on
    its own, and no fast-math flag may reorder the fp64 sums.
    """
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_forces_ts.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                             ctypes.c_int64, ctypes.c_float, ctypes.c_void_p,
                                             ctypes.c_int]
            lib.oracle_forces_ts.restype = ctypes.c_int
            lib.oracle_forces_f64.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_double,
                                              ctypes.c_void_p, ctypes.c_int]
            lib.oracle_forces_f64.restype = ctypes.c_int
            lib.oracle_euler.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_int64, ctypes.c_float]
            lib.oracle_euler.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _bodies(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    if a.ndim != 2 or a.shape[1] != 4:
        raise ValueError(f"expected an [n, 4] float32 array, got shape {a.shape}")
    return a


def max_threads() -> int:
    """OpenMP threads a call with ``threads=0`` uses on this host."""
    return int(_load().oracle_max_threads())


def forces_ts(targets, sources, eps2, threads: int = 0) -> np.ndarray:
    """fp64 (ax, ay, az, p) at each target from every source; shape [nt, 4]."""
    lib = _load()
    t = _bodies(targets)
    s = _bodies(sources)
    out = np.empty((t.shape[0], 4), dtype=np.float64)
    rc = lib.oracle_forces_ts(t.ctypes.data, t.shape[0], s.ctypes.data, s.shape[0],
                              ctypes.c_float(np.float32(eps2)), out.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError("oracle_forces_ts rejected its arguments")
    return out


def forces(pos_mass, eps2, rows=None, threads: int = 0) -> np.ndarray:
    """All-pairs (ax, ay, az, p) in fp64 for the given target rows (default: all).

    Every body is a source, the target itself included (its own term adds 0 to
    a and -m_i/eps to p).
    """
    pm = _bodies(pos_mass)
    targets = pm if rows is None else pm[np.asarray(rows, dtype=np.int64)]
    return forces_ts(targets, pm, eps2, threads)


def euler(pos_mass, vel, acc_pot, dt):
    """One fp32 Euler step on copies; returns (pos_mass', vel')."""
    lib = _load()
    pm = _bodies(pos_mass).copy()
    v = _bodies(vel).copy()
    a = _bodies(acc_pot)
    if not (pm.shape == v.shape == a.shape):
        raise ValueError("pos_mass, vel and acc_pot must have the same shape")
    rc = lib.oracle_euler(pm.ctypes.data, v.ctypes.data, a.ctypes.data, pm.shape[0],
                          ctypes.c_float(np.float32(dt)))
    if rc != 0:
        raise ValueError("oracle_euler rejected its arguments")
    return pm, v


def forces_f64(bodies, eps2, threads: int = 0) -> np.ndarray:
    """All-pairs (ax, ay, az, p) of fp64 bodies [n, 4] (x, y, z, m), in fp64."""
    lib = _load()
    b = np.ascontiguousarray(bodies, dtype=np.float64)
    if b.ndim != 2 or b.shape[1] != 4:
        raise ValueError(f"expected an [n, 4] array, got shape {b.shape}")
    out = np.empty_like(b)
    rc = lib.oracle_forces_f64(b.ctypes.data, b.shape[0], float(eps2), out.ctypes.data,
                               int(threads))
    if rc != 0:
        raise ValueError("oracle_forces_f64 rejected its arguments")
    return out


def trajectory_f64(pos_mass, vel, eps2, dt, steps, threads: int = 0):
    """`steps` explicit Euler steps kept in fp64 throughout (the lecture's order:
    positions from the old velocities, then velocities from a); returns the
    fp64 (pos_mass, vel) after the last step."""
    pm = np.array(pos_mass, dtype=np.float64)
    v = np.array(vel, dtype=np.float64)
    dt = float(dt)
    for _ in range(int(steps)):
        a = forces_f64(pm, eps2, threads)
        pm[:, :3] = pm[:, :3] + dt * v[:, :3]
        v[:, :3] = v[:, :3] + dt * a[:, :3]
    return pm, v
