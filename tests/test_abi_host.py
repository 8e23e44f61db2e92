"""Host-side checks of the C ABI: no GPU and no compute call needed.

The library loads, exports every function include/nbody.h declares, rejects
bad arguments before touching CUDA, and plans launches that cover every
target and source exactly once.
"""
import ctypes
import os
import re

import pytest

import all_pairs_gravitational_gb300 as apg
from all_pairs_gravitational_gb300 import _binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "nbody.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return apg.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nbody_\w+)\s*\(", text)))


def test_header_and_binding_agree():
    assert _declared_functions() == sorted(apg.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in _binding.STATUS_NAMES.items():
        assert apg.nbody_status_string(code).startswith(name)
    assert "UNKNOWN" in apg.nbody_status_string(99)


P = 1 << 20          # a fake, 16-byte aligned "device" address: never dereferenced


def _forces(lib, pm, n, eps2, acc):
    return lib.nbody_forces(ctypes.c_void_p(pm), n, ctypes.c_float(eps2), ctypes.c_void_p(acc),
                            None)


def test_forces_argument_checks(lib):
    # nothing below reaches CUDA: each call is rejected (or is a no-op) on the host
    assert _forces(lib, P, 0, 1e-4, P + 4096) == 0                   # n == 0: no-op
    assert _forces(lib, 0, 0, 1e-4, 0) == 0
    assert _forces(lib, P, -1, 1e-4, P + 4096) == 1
    assert _forces(lib, P, 2 ** 31, 1e-4, P + 2 ** 36) == 1
    assert _forces(lib, 0, 10, 1e-4, P) == 1                         # null input
    assert _forces(lib, P, 10, 1e-4, 0) == 1                         # null output
    for bad in (0.0, -1e-4, float("nan"), float("inf"), 1e-40):      # 1e-40 is subnormal
        assert _forces(lib, P, 10, bad, P + 4096) == 1, bad
    assert _forces(lib, P + 4, 10, 1e-4, P + 4096) == 2              # misaligned input
    assert _forces(lib, P, 10, 1e-4, P + 4104) == 2                  # misaligned output
    assert _forces(lib, P, 10, 1e-4, P) == 3                         # same buffer
    assert _forces(lib, P, 10, 1e-4, P + 144) == 3                   # overlaps the last body
    assert _forces(lib, P + 144, 10, 1e-4, P) == 3


def test_forces_ts_argument_checks(lib):
    def call(t, nt, s, ns, eps2, out):
        return lib.nbody_forces_ts(ctypes.c_void_p(t), nt, ctypes.c_void_p(s), ns,
                                   ctypes.c_float(eps2), ctypes.c_void_p(out), None)
    t, s, o = P, P + 4096, P + 8192
    # every call below is rejected (or is a no-op) on the host
    assert call(t, 0, s, 5, 1e-4, o) == 0                 # no targets: no-op
    assert call(t, -1, s, 5, 1e-4, o) == 1
    assert call(t, 5, s, -1, 1e-4, o) == 1
    assert call(t, 5, s, 2 ** 31, 1e-4, o) == 1
    assert call(0, 5, s, 5, 1e-4, o) == 1
    assert call(t, 5, 0, 5, 1e-4, o) == 1                 # sources needed when ns > 0
    assert call(t, 5, s, 5, 1e-4, 0) == 1
    assert call(t, 5, s, 5, 0.0, o) == 1
    assert call(t, 5, s, 5, float("nan"), o) == 1
    assert call(t + 8, 5, s, 5, 1e-4, o) == 2
    assert call(t, 5, s + 4, 5, 1e-4, o) == 2
    assert call(t, 5, s, 5, 1e-4, o + 12) == 2
    assert call(t, 5, s, 5, 1e-4, t + 64) == 3            # out overlaps the targets
    assert call(t, 5, s, 300, 1e-4, s + 4000) == 3        # out overlaps the sources' tail
    assert call(t, 2, s, 5, 1e-4, s - 16) == 3            # out's tail overlaps the sources


def test_simulate_argument_checks(lib):
    def call(pm, v, a, n, eps2, dt, steps):
        return lib.nbody_simulate(ctypes.c_void_p(pm), ctypes.c_void_p(v), ctypes.c_void_p(a), n,
                                  ctypes.c_float(eps2), ctypes.c_float(dt), steps, None)
    a, b, c = P, P + 4096, P + 8192
    # every call below is rejected (or is a no-op) on the host
    assert call(a, b, c, 0, 1e-4, 1e-3, 5) == 0
    assert call(a, b, c, 5, 1e-4, 1e-3, 0) == 0
    assert call(a, b, c, 5, 1e-4, 1e-3, -1) == 1
    assert call(a, b, c, 5, 1e-4, float("nan"), 3) == 1
    assert call(a, b, c, 5, 0.0, 1e-3, 3) == 1
    assert call(a, 0, c, 5, 1e-4, 1e-3, 3) == 1
    assert call(a, b + 8, c, 5, 1e-4, 1e-3, 3) == 2
    assert call(a, a + 32, c, 5, 1e-4, 1e-3, 3) == 3
    assert call(a, b, a + 16, 5, 1e-4, 1e-3, 3) == 3
    assert call(a, c + 16, c, 5, 1e-4, 1e-3, 3) == 3


def test_euler_argument_checks(lib):
    def call(pm, v, a, n, dt):
        return lib.nbody_euler_step(ctypes.c_void_p(pm), ctypes.c_void_p(v), ctypes.c_void_p(a), n,
                                    ctypes.c_float(dt), None)
    a, b, c = P, P + 4096, P + 8192
    assert call(a, b, c, 0, 1e-3) == 0
    assert call(a, b, c, -5, 1e-3) == 1
    assert call(0, b, c, 5, 1e-3) == 1
    assert call(a, b, c, 5, float("nan")) == 1
    assert call(a, b, c, 5, float("inf")) == 1
    assert call(a + 8, b, c, 5, 1e-3) == 2
    assert call(a, b, c + 8, 5, 1e-3) == 2
    assert call(a, a + 64, c, 5, 1e-3) == 3       # pos and vel overlap
    assert call(a, b, b + 16, 5, 1e-3) == 3       # vel and acc overlap
    assert call(a, b, a, 5, 1e-3) == 3            # acc is pos


def _covers(plan, n):
    """Every target in exactly one target block, every source tile in exactly
    one piece of the source range."""
    ntiles = -(-n // plan["tile"])
    if plan["path"] == apg.NBODY_PATH_SYMMETRIC:
        _sym_covers(plan, n)
        return
    if plan["path"] == apg.NBODY_PATH_TILED:
        bi = plan["threads"] * plan["i_per_thread"]
        tps, s = plan["tiles_per_split"], plan["splits"]
        assert plan["grid"] == plan["num_iblocks"] * s
        assert plan["scratch_bytes"] == (16 * s * n if s > 1 else 0)
    else:
        assert plan["path"] == apg.NBODY_PATH_CLUSTER
        bi = 32 * plan["i_per_thread"]
        tps, s = plan["tiles_per_split"], plan["cluster"]
        assert s in (1, 2, 4, 8)
        assert plan["splits"] == s * plan["warps_j"]
        assert plan["threads"] == 32 * plan["warps_j"]
        assert plan["tile"] % plan["warps_j"] == 0 and plan["tile"] // plan["warps_j"] <= 32
        assert plan["grid"] == plan["num_iblocks"] * s
        assert plan["scratch_bytes"] == 0
    assert plan["num_iblocks"] * bi >= n > (plan["num_iblocks"] - 1) * bi
    assert s * tps >= ntiles > (s - 1) * tps
    assert plan["grid"] < 2 ** 31
    assert 0 < plan["fill"] <= 1.0


def _sym_units(nb):
    """Block pairs of the symmetric decomposition, as the header states it:
    row I takes its own block one way (d = 0) and blocks I + d (mod nb) both
    ways for 1 <= d <= (nb - 1) / 2, plus d = nb / 2 for I < nb / 2 when nb
    is even."""
    h = (nb - 1) // 2
    rows = []
    for i in range(nb):
        ds = list(range(0, h + 1)) + ([nb // 2] if nb % 2 == 0 and i < nb // 2 else [])
        rows.append([(i, (i + d) % nb, d) for d in ds])
    return rows


@pytest.mark.parametrize("nb", list(range(1, 40)) + [64, 127, 128, 512, 513])
def test_symmetric_decomposition_meets_every_pair_once(nb):
    seen = {}
    for row in _sym_units(nb):
        for i, j, d in row:
            if d == 0:
                assert i == j
                seen[(i, i)] = seen.get((i, i), 0) + 1
            else:
                for key in ((i, j), (j, i)):           # one evaluation, both ways
                    seen[key] = seen.get(key, 0) + 1
    assert len(seen) == nb * nb and set(seen.values()) == {1}
    # j-side slot d - 1 of every body is written by exactly one row
    slots = {}
    for row in _sym_units(nb):
        for i, j, d in row:
            if d:
                slots[(j, d - 1)] = slots.get((j, d - 1), 0) + 1
    assert set(slots.values()) <= {1}
    h = (nb - 1) // 2
    for j in range(nb):
        want = h + (1 if nb % 2 == 0 and j >= nb // 2 else 0)
        assert sorted(s for (b, s) in slots if b == j) == list(range(want))


def _sym_covers(plan, n):
    t = plan["threads"] * plan["i_per_thread"]
    nb = plan["num_iblocks"]
    assert nb == -(-n // t) and t % plan["tile"] == 0 and plan["tile"] % 32 == 0
    jslots = (nb - 1) // 2 + (1 if nb % 2 == 0 else 0)
    units = (1 + jslots) * (t // plan["tile"])
    s, upp = plan["splits"], plan["tiles_per_split"]
    assert 1 <= s <= units and upp == -(-units // s)
    assert plan["grid"] == nb * s < 2 ** 31
    want = 16 * (s + jslots) * n if (s > 1 or jslots > 0) else 0
    assert plan["scratch_bytes"] == want <= 24 << 30
    assert 0 < plan["fill"] <= 1.0


@pytest.mark.parametrize("n", [1, 2, 33, 2048, 2049, 4096, 4097, 20011, 32768, 65537, 200003,
                               1048576, 2 ** 21])
@pytest.mark.parametrize("splits", [0, 1, 3, 64])
def test_symmetric_plan(lib, n, splits):
    plan = apg.nbody_plan_forces(n, 152, path=apg.NBODY_PATH_SYMMETRIC, splits=splits)
    assert plan["path"] == apg.NBODY_PATH_SYMMETRIC
    _sym_covers(plan, n)
    if splits:
        units = plan["tiles_per_split"] * plan["splits"]
        assert plan["splits"] == min(splits, units) or plan["splits"] == splits


@pytest.mark.parametrize("sm", [1, 148, 160, 264])
@pytest.mark.parametrize("n", [10240, 45056, 163840, 1048576, 2097159])
@pytest.mark.parametrize("variant", [-1, 0, 1, 2, 3, 4, 5])
def test_symmetric_plan_other_gpus_and_variants(n, sm, variant):
    ref = apg.nbody_plan_forces(4096, 152, path=apg.NBODY_PATH_SYMMETRIC, variant=variant)
    t = ref["threads"] * ref["i_per_thread"]
    nb = -(-n // t)
    jslots = (nb - 1) // 2 + (1 if nb % 2 == 0 else 0)
    if variant >= 0 and 16 * (jslots + 1) * n > 24 << 30:   # partials beyond the cap
        with pytest.raises(apg.NbodyError):
            apg.nbody_plan_forces(n, sm, path=apg.NBODY_PATH_SYMMETRIC, variant=variant)
        return
    plan = apg.nbody_plan_forces(n, sm, path=apg.NBODY_PATH_SYMMETRIC, variant=variant)
    assert plan["path"] == apg.NBODY_PATH_SYMMETRIC
    if variant >= 0:
        assert plan["variant"] == variant
    _sym_covers(plan, n)


def test_symmetric_plan_forced_splits_stay_within_the_cap():
    plan = apg.nbody_plan_forces(2 ** 21, 152, path=apg.NBODY_PATH_SYMMETRIC, splits=1000)
    assert plan["scratch_bytes"] <= 24 << 30 and plan["splits"] < 1000
    _sym_covers(plan, 2 ** 21)


def test_symmetric_plan_limits():
    with pytest.raises(apg.NbodyError):      # j-side partials beyond 24 GiB
        apg.nbody_plan_forces(2 ** 23, 152, path=apg.NBODY_PATH_SYMMETRIC)
    with pytest.raises(apg.NbodyError):      # the compensated kernel is tiled only
        apg.nbody_plan_forces(65536, 152, path=apg.NBODY_PATH_SYMMETRIC,
                              precision=apg.NBODY_PRECISION_COMPENSATED)
    # automatic planning falls back to the tiled path where the partials do not fit
    assert apg.nbody_plan_forces(2 ** 23, 152)["path"] == apg.NBODY_PATH_TILED


@pytest.mark.parametrize("n", [1, 2, 3, 31, 33, 127, 128, 129, 255, 257, 1000, 1024, 4096,
                               16384, 65536, 200003, 1048576, 2 ** 24 + 3, 2 ** 31 - 1])
@pytest.mark.parametrize("sm", [1, 148, 152, 160])
def test_plan_covers_all_pairs(lib, n, sm):
    plan = apg.nbody_plan_forces(n, sm)
    _covers(plan, n)


def test_plan_fills_the_gpu_at_one_million():
    for path in (apg.NBODY_PATH_TILED, apg.NBODY_PATH_SYMMETRIC):
        plan = apg.nbody_plan_forces(1048576, 152, path=path)
        assert plan["fill"] > 0.97
        one = apg.nbody_plan_forces(1048576, 152, path=path, splits=1)
        assert one["splits"] == 1
        assert plan["fill"] > one["fill"]
    one = apg.nbody_plan_forces(1048576, 152, path=apg.NBODY_PATH_TILED, splits=1)
    assert one["scratch_bytes"] == 0


@pytest.mark.parametrize("n", [1, 2, 3, 33, 127, 129, 1000, 1024, 2048, 4096, 8192, 12288, 16384])
@pytest.mark.parametrize("variant", [-1, 0, 1, 2, 3])
def test_cluster_plan_covers_all_pairs(n, variant):
    plan = apg.nbody_plan_forces(n, 152, path=apg.NBODY_PATH_CLUSTER, variant=variant)
    _covers(plan, n)
    if variant >= 0:
        assert plan["variant"] == variant


def test_auto_path_choice():
    assert apg.nbody_plan_forces(1024, 152)["path"] == apg.NBODY_PATH_CLUSTER
    assert apg.nbody_plan_forces(4096, 152)["path"] == apg.NBODY_PATH_CLUSTER
    assert apg.nbody_plan_forces(8192, 152)["path"] == apg.NBODY_PATH_TILED
    assert apg.nbody_plan_forces(10239, 152)["path"] == apg.NBODY_PATH_TILED
    assert apg.nbody_plan_forces(10240, 152)["path"] == apg.NBODY_PATH_SYMMETRIC
    # the symmetric block size grows with n: 512, 1024, then 2048 bodies
    blocks = [apg.nbody_plan_forces(n, 152)["threads"] * apg.nbody_plan_forces(n, 152)["i_per_thread"]
              for n in (10240, 45055, 45056, 163839, 163840, 1048576)]
    assert blocks == [512, 512, 1024, 1024, 2048, 2048]
    assert apg.nbody_plan_forces(1048576, 152)["path"] == apg.NBODY_PATH_SYMMETRIC
    with pytest.raises(apg.NbodyError):
        apg.nbody_plan_forces(1000, 152, path=apg.NBODY_PATH_CLUSTER, splits=3)
    with pytest.raises(apg.NbodyError):
        apg.nbody_plan_forces(1000, 152, path=7)


def test_compensated_precision_plans_the_compensated_kernel():
    for n in (1, 1000, 4096, 1048576):
        plan = apg.nbody_plan_forces(n, 152, precision=apg.NBODY_PRECISION_COMPENSATED)
        assert plan["path"] == apg.NBODY_PATH_TILED and plan["variant"] == 7
        _covers(plan, n)
    with pytest.raises(apg.NbodyError):
        apg.nbody_plan_forces(1000, 152, path=apg.NBODY_PATH_CLUSTER,
                              precision=apg.NBODY_PRECISION_COMPENSATED)
    with pytest.raises(apg.NbodyError):
        apg.nbody_plan_forces(1000, 152, variant=0, precision=apg.NBODY_PRECISION_COMPENSATED)
    with pytest.raises(apg.NbodyError):
        apg.nbody_plan_forces(1000, 152, precision=2)


def test_plan_forced_splits_and_variants(lib):
    v = 0
    while True:
        try:
            apg.nbody_plan_forces(1000, 152, path=apg.NBODY_PATH_TILED, variant=v)
        except apg.NbodyError:
            break
        v += 1
    assert v >= 4
    for v in range(v):
        for s in (1, 2, 7, 64):
            plan = apg.nbody_plan_forces(200003, 152, path=apg.NBODY_PATH_TILED, variant=v,
                                         splits=s)
            _covers(plan, 200003)
            assert plan["variant"] == v
    with pytest.raises(apg.NbodyError):
        apg.nbody_plan_forces(1000, 152, variant=99)
    with pytest.raises(apg.NbodyError):
        apg.nbody_plan_forces(0, 152)
    with pytest.raises(apg.NbodyError):
        apg.nbody_plan_forces(1000, 0)
