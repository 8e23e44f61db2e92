"""Seeded synthetic bodies for the all-pairs gravity path.

This module draws inputs only: it holds none of the force or integration
arithmetic, and both the CUDA path and the oracle are fed from it.

Random numbers come from splitmix64 (Steele, Lea & Flood 2014; the output
mixer as published by Vigna), used as a counter-based generator: output k of a
stream seeded with s is mix(s + (k+1) * 0x9E3779B97F4A7C15). That makes every
draw reproducible from (seed, position) alone and lets numpy evaluate it in
bulk. Uniforms take the top 53 bits; normals use the Box-Muller transform.
Everything is computed in fp64 and rounded to fp32 once.

The workloads follow the configurations the all-pairs method is measured on:

* ``disk``: the lecture's initial() (x, y, vx, vy uniform in [-1, 1], z = vz
  = 0, m = 1), seeded with N as the lecture's srand(N) is. glibc rand() itself
  is not reproduced.
* ``cube``: x, y, z uniform in [-1, 1]^3, masses uniform in [lo, hi], v = 0.
* ``plummer``: an equal-mass Plummer sphere (M = 1, scale radius 1, G = 1)
  by the Aarseth, Henon & Wielen (1974) construction: radius by the inverse
  cumulative mass X^(-2/3) - 1 = r^-2, redrawn when r > 10; speed q * v_esc
  with q drawn by von Neumann rejection from q^2 (1 - q^2)^(7/2); both
  directions isotropic.
* ``clumps``: 90% of the bodies in two Gaussian clumps (sigma 0.1) at
  (+1, 0, 0) and (-1, 0, 0), 10% uniform in [-3, 3]^3, masses lognormal
  (mu 0, sigma 0.5) normalised to a total of 1; stored clump+, clump-,
  uniform, unshuffled.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


class Stream:
    """Counter-based splitmix64 stream; each draw advances the counter."""

    def __init__(self, seed: int):
        self.seed = np.uint64(int(seed) & 0xFFFFFFFFFFFFFFFF)
        self.pos = 0

    def bits(self, count: int) -> np.ndarray:
        k = np.arange(self.pos + 1, self.pos + 1 + count, dtype=np.uint64)
        self.pos += count
        with np.errstate(over="ignore"):
            z = self.seed + k * _GAMMA
            z = (z ^ (z >> np.uint64(30))) * _M1
            z = (z ^ (z >> np.uint64(27))) * _M2
            z = z ^ (z >> np.uint64(31))
        return z

    def uniform(self, count: int, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
        """count doubles in [lo, hi)."""
        u = (self.bits(count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        return lo + (hi - lo) * u

    def normal(self, count: int) -> np.ndarray:
        """count standard normal doubles (Box-Muller, both outputs used)."""
        half = (count + 1) // 2
        u1 = 1.0 - self.uniform(half)          # in (0, 1]
        u2 = self.uniform(half)
        rad = np.sqrt(-2.0 * np.log(u1))
        out = np.empty(2 * half)
        out[0::2] = rad * np.cos(2.0 * np.pi * u2)
        out[1::2] = rad * np.sin(2.0 * np.pi * u2)
        return out[:count]

    def isotropic(self, count: int) -> np.ndarray:
        """count unit vectors, uniform on the sphere."""
        cz = self.uniform(count, -1.0, 1.0)
        phi = self.uniform(count, 0.0, 2.0 * np.pi)
        sz = np.sqrt(np.maximum(0.0, 1.0 - cz * cz))
        return np.stack([sz * np.cos(phi), sz * np.sin(phi), cz], axis=1)


@dataclass
class Workload:
    """One synthetic problem: bodies, velocities, softening and step size."""

    name: str
    pos_mass: np.ndarray          # float32 [n, 4]: x, y, z, m
    vel: np.ndarray               # float32 [n, 4]: vx, vy, vz, 0
    eps2: np.float32
    dt: np.float32
    steps: int = 1
    potential: bool = True        # whether p is part of what the workload checks
    recipe: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def n(self) -> int:
        return int(self.pos_mass.shape[0])


def _pack(pos: np.ndarray, mass: np.ndarray, vel: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    n = pos.shape[0]
    pm = np.zeros((n, 4), dtype=np.float32)
    pm[:, :3] = pos
    pm[:, 3] = mass
    v = np.zeros((n, 4), dtype=np.float32)
    v[:, :3] = vel
    return pm, v


def disk(n: int = 4096, seed: int | None = None) -> Workload:
    s = Stream(n if seed is None else seed)
    u = s.uniform(4 * n, -1.0, 1.0).reshape(n, 4)       # per body: x, y, vx, vy
    pos = np.zeros((n, 3))
    pos[:, 0], pos[:, 1] = u[:, 0], u[:, 1]
    vel = np.zeros((n, 3))
    vel[:, 0], vel[:, 1] = u[:, 2], u[:, 3]
    pm, v = _pack(pos, np.ones(n), vel)
    return Workload(f"disk{n}", pm, v, np.float32(1e-6), np.float32(1e-3), 1, False,
                    "x,y,vx,vy ~ U[-1,1], z=vz=0, m=1, seed N")


def cube(n: int = 16384, seed: int | None = None, mass=(0.5, 1.5), eps2: float = 1e-4,
         name: str | None = None) -> Workload:
    s = Stream(n if seed is None else seed)
    pos = s.uniform(3 * n, -1.0, 1.0).reshape(n, 3)
    if mass[0] == mass[1]:
        m = np.full(n, float(mass[0]))
    else:
        m = s.uniform(n, mass[0], mass[1])
    pm, v = _pack(pos, m, np.zeros((n, 3)))
    return Workload(name or f"cube{n}", pm, v, np.float32(eps2), np.float32(1e-3), 1, True,
                    f"x,y,z ~ U[-1,1]^3, m ~ U[{mass[0]},{mass[1]}], v=0, seed N")


def small_cube(n: int) -> Workload:
    """Small-N sweep: uniform cube, unit masses, eps^2 = 1e-4."""
    return cube(n, seed=n, mass=(1.0, 1.0), eps2=1e-4, name=f"smallcube{n}")


def _plummer_radii(s: Stream, n: int, rmax: float) -> np.ndarray:
    out = np.empty(0)
    while out.size < n:
        want = n - out.size
        x = s.uniform(want + want // 8 + 16)
        x = x[x > 0.0]
        r = 1.0 / np.sqrt(x ** (-2.0 / 3.0) - 1.0)
        out = np.concatenate([out, r[r <= rmax]])
    return out[:n]


def _plummer_q(s: Stream, n: int) -> np.ndarray:
    out = np.empty(0)
    while out.size < n:
        want = n - out.size
        k = 3 * want + 64
        q = s.uniform(k)
        y = s.uniform(k, 0.0, 0.1)                  # 0.1 bounds q^2 (1-q^2)^3.5 from above
        out = np.concatenate([out, q[y < q * q * (1.0 - q * q) ** 3.5]])
    return out[:n]


def plummer(n: int, seed: int | None = None, eps: float = 0.01, rmax: float = 10.0,
            dt: float = 1e-3, steps: int = 1) -> Workload:
    s = Stream(n if seed is None else seed)
    r = _plummer_radii(s, n, rmax)
    pos = r[:, None] * s.isotropic(n)
    q = _plummer_q(s, n)
    speed = q * np.sqrt(2.0) * (1.0 + r * r) ** -0.25
    vel = speed[:, None] * s.isotropic(n)
    pm, v = _pack(pos, np.full(n, 1.0 / n), vel)
    return Workload(f"plummer{n}", pm, v, np.float32(eps * eps), np.float32(dt), steps, True,
                    f"equal-mass Plummer sphere, m=1/N, a=1, r<={rmax}, eps={eps}, seed N",
                    {"eps": eps})


def clumps(n: int = 200003, seed: int | None = None) -> Workload:
    s = Stream(n if seed is None else seed)
    n_c = int(round(0.9 * n))
    n_plus = n_c // 2
    n_minus = n_c - n_plus
    n_u = n - n_c
    g = s.normal(3 * n_c).reshape(n_c, 3) * 0.1
    g[:n_plus, 0] += 1.0
    g[n_plus:, 0] -= 1.0
    u = s.uniform(3 * n_u, -3.0, 3.0).reshape(n_u, 3)
    pos = np.concatenate([g, u])
    m = np.exp(0.5 * s.normal(n))
    m = m / m.sum()
    pm, v = _pack(pos, m, np.zeros((n, 3)))
    return Workload(f"clumps{n}", pm, v, np.float32(1e-5), np.float32(1e-3), 1, True,
                    "90% in two N(+-1,0,0; 0.1^2) clumps, 10% U[-3,3]^3, m lognormal(0,0.5)/sum",
                    {"n_plus": n_plus, "n_minus": n_minus, "n_uniform": n_u})


def named(name: str) -> Workload:
    """The measured configurations, by name."""
    table = {
        "disk4096": lambda: disk(4096),
        "cube16384": lambda: cube(16384),
        "plummer65536": lambda: plummer(65536, eps=0.01, steps=10),
        "clumps200003": lambda: clumps(200003),
        "plummer1048576": lambda: plummer(1048576, eps=0.005),
    }
    if name in table:
        return table[name]()
    if name.startswith("smallcube"):
        return small_cube(int(name[len("smallcube"):]))
    raise KeyError(name)


CONFIG_NAMES = ["disk4096", "cube16384", "plummer65536", "clumps200003", "plummer1048576"]
SMALL_SWEEP = [1024, 2048, 4096, 8192]
