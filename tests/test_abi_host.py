"""Host-side checks of the C ABI: no GPU and no compute call needed.

The library loads, exports every function include/nbody.h declares, rejects
bad arguments before touching CUDA, and plans launches that cover every
target and source exactly once.
"""
import ctypes
import os
import re

import numpy as np
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
    header = open(HEADER).read()
    assert re.search(r"#define NBODY_MIN_EPS2 1\.0e-25f", header)
    assert apg.NBODY_MIN_EPS2 == 1.0e-25
    # the self term's m (eps^2)^(-3/2) stays finite in fp32 for m up to 10
    assert 10.0 * np.float32(apg.NBODY_MIN_EPS2) ** -1.5 < np.finfo(np.float32).max


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
    for bad in (0.0, -1e-4, float("nan"), float("inf"), 1e-40,       # 1e-40 is subnormal
                1.17549435e-38, 1e-26, 9.9e-26):   # (eps2)^(-3/2) overflows fp32 below 2.05e-26
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


def _covers(plan, n, budget=None):
    """Every target in exactly one target block, every source tile in exactly
    one piece of the source range, and the workspace within the budget."""
    ntiles = -(-n // plan["tile"])
    if budget is not None and plan["scratch_min_bytes"] <= budget:
        assert plan["scratch_bytes"] <= budget
    if plan["path"] == apg.NBODY_PATH_SYMMETRIC:
        _sym_covers(plan, n)
        return
    if plan["path"] == apg.NBODY_PATH_ROWS:
        _rows_covers(plan, n, n)
        return
    if plan["path"] == apg.NBODY_PATH_TILED:
        bi = plan["threads"] * plan["i_per_thread"]
        tps, s = plan["tiles_per_split"], plan["splits"]
        g, passes = plan["groups_per_pass"], plan["passes"]
        assert plan["groups"] == s and 1 <= g <= s and passes == -(-s // g)
        assert plan["grid"] == plan["num_iblocks"] * g
        rec = 16 * n
        if s == 1:
            assert plan["scratch_bytes"] == plan["scratch_min_bytes"] == 0
        elif passes == 1:
            assert plan["scratch_bytes"] == s * rec and plan["scratch_min_bytes"] == min(s, 2) * rec
        else:   # g pieces and the carry slot
            assert plan["scratch_bytes"] == (g + 1) * rec and plan["scratch_min_bytes"] == 2 * rec
    else:
        assert plan["path"] == apg.NBODY_PATH_CLUSTER
        bi = 32 * plan["i_per_thread"]
        tps, s = plan["tiles_per_split"], plan["cluster"]
        assert s in (1, 2, 4, 8)
        assert plan["splits"] == s * plan["warps_j"]
        assert plan["threads"] == 32 * plan["warps_j"]
        assert plan["tile"] % plan["warps_j"] == 0 and plan["tile"] // plan["warps_j"] <= 32
        assert plan["grid"] == plan["num_iblocks"] * s
        assert plan["scratch_bytes"] == 0 and plan["passes"] == 1
    assert plan["num_iblocks"] * bi >= n > (plan["num_iblocks"] - 1) * bi
    assert s * tps >= ntiles > (s - 1) * tps
    assert plan["grid"] < 2 ** 31
    assert 0 < plan["fill"] <= 1.0


def _rows_items(plan, nt, ns):
    """The warp items of a row-split plan, as the header states them: CTA b
    takes targets [b tb, (b + 1) tb); its items are runs of K of them (the
    last run of a CTA may be short) against S pieces of `tile` sources."""
    tb, k, s, tile = (plan["tiles_per_split"], plan["i_per_thread"], plan["splits"],
                      plan["tile"])
    for b in range(plan["num_iblocks"]):
        t0, t1 = b * tb, min((b + 1) * tb, nt)
        for g in range(0, t1 - t0, k):
            for piece in range(s):
                yield (range(t0 + g, min(t0 + g + k, t1)),
                       range(piece * tile, min((piece + 1) * tile, ns)))


def _rows_covers(plan, nt, ns, sm=None):
    tb = plan["tiles_per_split"]
    assert plan["i_per_thread"] in (7, 6, 4, 2) and plan["threads"] in (256, 384)
    assert plan["num_iblocks"] == plan["grid"] == -(-nt // tb)
    if sm is not None:   # an equal share of the targets per SM
        assert tb == -(-nt // sm) and plan["grid"] <= sm
    assert plan["tile"] % 64 == 0 and plan["splits"] * plan["tile"] >= ns
    assert plan["scratch_bytes"] == plan["scratch_min_bytes"] == 0 and plan["passes"] == 1
    assert 0 < plan["fill"] <= 1.0
    # shared memory: the padded sources and the piece sums of the CTA's targets
    tb_pad = -(-tb // plan["i_per_thread"]) * plan["i_per_thread"]
    assert 16 * plan["splits"] * plan["tile"] + 16 * plan["splits"] * tb_pad <= 227 * 1024


@pytest.mark.parametrize("nt,ns", [(1, 1), (2, 2), (3, 3), (33, 33), (152, 152), (153, 153),
                                   (1000, 1000), (1024, 1024), (2047, 2047), (300, 5000),
                                   (5000, 300), (4097, 4097)])
def test_rows_decomposition_meets_every_pair_once(nt, ns):
    plan = apg.nbody_plan_forces_ts(nt, ns, 152, path=apg.NBODY_PATH_ROWS)
    _rows_covers(plan, nt, ns, 152)
    seen = np.zeros((nt, ns), dtype=np.int32)
    for ti, sj in _rows_items(plan, nt, ns):
        if len(ti) and len(sj):
            seen[ti.start:ti.stop, sj.start:sj.stop] += 1
    assert (seen == 1).all()


@pytest.mark.parametrize("n", [1, 7, 1000, 1024, 2048, 3072, 4096, 4864, 6144, 8192, 10239])
def test_rows_plan_bounds(n):
    """Automatic row-split plans: at most 2048 sources per piece (32 terms
    per lane half before the tree), and forced variants and piece counts are
    honoured."""
    plan = apg.nbody_plan_forces(n, 152)
    assert plan["path"] == apg.NBODY_PATH_ROWS and plan["tile"] <= 2048
    _rows_covers(plan, n, n, 152)
    for v in range(4):
        forced = apg.nbody_plan_forces(n, 152, path=apg.NBODY_PATH_ROWS, variant=v)
        assert forced["variant"] == v
        _rows_covers(forced, n, n)
    three = apg.nbody_plan_forces(n, 152, path=apg.NBODY_PATH_ROWS, splits=3)
    assert three["splits"] == 3
    _rows_covers(three, n, n)


def test_rows_plan_rejects_sources_beyond_shared_memory():
    # every source in shared memory: up to 14400 with few targets, not 14500
    plan = apg.nbody_plan_forces_ts(100, 14400, 152, path=apg.NBODY_PATH_ROWS)
    _rows_covers(plan, 100, 14400, 152)
    with pytest.raises(apg.NbodyError):
        apg.nbody_plan_forces_ts(100, 14500, 152, path=apg.NBODY_PATH_ROWS)
    with pytest.raises(apg.NbodyError):
        apg.nbody_plan_forces(20000, 152, path=apg.NBODY_PATH_ROWS)
    # the automatic choice then takes another path
    assert apg.nbody_plan_forces_ts(100, 20000, 152)["path"] == apg.NBODY_PATH_TILED


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


def _ndist(nb):
    return (nb - 1) // 2 + 1 + (1 if nb % 2 == 0 else 0)


def _jslots(nb, d_per_group):
    nd = _ndist(nb)
    groups = -(-nd // d_per_group)
    return max(min((g + 1) * d_per_group, nd) - max(g * d_per_group, 1)
               for g in range(min(groups, 2)))


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


def _simulate_slots(nb, spb, P, D, gpp):
    """The slot traffic of the symmetric path, restated from the header and
    the kernels' index rules at unit granularity (a unit = spb-th of a
    block): which (group, slot, block, unit) record each CTA writes, and
    which records the reduction pass reads for each body's block.  Returns
    the ordered block pairs each block's final sum covers, with the count."""
    nd = _ndist(nb)
    h = (nb - 1) // 2
    groups = -(-nd // D)
    covered = {x: {} for x in range(nb)}
    for g0 in range(0, groups, gpp):
        gp = min(gpp, groups - g0)
        written = {}   # (gl, slot, block, unit) -> (source block set of the partial)
        for gl in range(gp):
            dlo = (g0 + gl) * D
            jbase = max(dlo, 1)
            for row in range(nb):
                dmax = h + (1 if nb % 2 == 0 and row < nb // 2 else 0)
                dhi = min(dlo + D, dmax + 1)
                units = max(0, dhi - dlo) * spb
                for piece in range(P):
                    u0, u1 = units * piece // P, units * (piece + 1) // P
                    # the i-side slot `piece` of every unit of the row's block
                    for ub in range(spb):
                        key = (gl, piece, row, ub)
                        assert key not in written
                        written[key] = []
                    for u in range(u0, u1):
                        d = dlo + u // spb
                        sub = u % spb
                        jblk = (row + d) % nb
                        for ub in range(spb):     # the row's targets meet unit `sub` of J
                            written[(gl, piece, row, ub)].append((jblk, sub))
                        if d != 0:                # unit `sub` of J meets all the row's targets
                            key = (gl, P + d - jbase, jblk, sub)
                            assert key not in written, key
                            written[key] = [(row, ub) for ub in range(spb)]
        # the reduction pass
        for x in range(nb):
            upper = nb % 2 == 0 and x >= nb // 2
            for ub in range(spb):
                for gl in range(gp):
                    dlo = (g0 + gl) * D
                    jbase = max(dlo, 1)
                    reads = list(range(P))
                    dhi = min(dlo + D, nd)
                    if nb % 2 == 0 and not upper:
                        dhi = min(dhi, h + 1)
                    reads += [P + d - jbase for d in range(jbase, dhi)]
                    for slot in reads:
                        assert slot < P + _jslots(nb, D)
                        for src in written[(gl, slot, x, ub)]:
                            covered[x][(ub, src)] = covered[x].get((ub, src), 0) + 1
    return covered


@pytest.mark.parametrize("nb", [1, 2, 3, 4, 5, 6, 7, 8, 11, 16, 17])
@pytest.mark.parametrize("P,D", [(1, 1), (1, 2), (2, 1), (3, 2), (4, 3), (5, 7), (2, 64)])
@pytest.mark.parametrize("gpp", [1, 2, 3, 100])
def test_symmetric_groups_and_passes_cover_every_pair_once(nb, P, D, gpp):
    """Every (target unit, source unit) pair reaches the target's final sum
    exactly once, whatever the pieces, the distances per group and the
    groups per pass; no partial record is written twice in a pass, and every
    record the reduction reads was written in that pass."""
    spb = 3
    D = min(D, _ndist(nb))
    covered = _simulate_slots(nb, spb, P, D, gpp)
    every = {(ub, (j, us)) for ub in range(spb) for j in range(nb) for us in range(spb)}
    for x in range(nb):
        assert set(covered[x]) == every and set(covered[x].values()) == {1}, x


def _sym_covers(plan, n):
    t = plan["threads"] * plan["i_per_thread"]
    nb = plan["num_iblocks"]
    assert nb == -(-n // t) and t % plan["tile"] == 0 and plan["tile"] % 32 == 0
    spb = t // plan["tile"]
    nd = _ndist(nb)
    P, D, G = plan["splits"], plan["dists"], plan["groups"]
    g, passes = plan["groups_per_pass"], plan["passes"]
    assert 1 <= D <= nd and G == -(-nd // D)
    assert 1 <= P <= max(1, D * spb) and plan["tiles_per_split"] == -(-min(D, nd) * spb // P)
    assert 1 <= g <= G and passes == -(-G // g)
    assert plan["grid"] == nb * P * g < 2 ** 31
    rec = 16 * n
    per_group = (P + _jslots(nb, D)) * rec
    if nb == 1 and P == 1:
        assert plan["scratch_bytes"] == plan["scratch_min_bytes"] == 0
    elif passes == 1:
        assert plan["scratch_bytes"] == G * per_group
        assert plan["scratch_min_bytes"] == min(G * per_group, per_group + rec)
    else:
        assert plan["scratch_bytes"] == g * per_group + rec
        assert plan["scratch_min_bytes"] == per_group + rec
    assert 0 < plan["fill"] <= 1.0


@pytest.mark.parametrize("n", [1, 2, 33, 2048, 2049, 4096, 4097, 20011, 32768, 65537, 200003,
                               1048576, 2 ** 21])
@pytest.mark.parametrize("splits", [0, 1, 3, 64])
def test_symmetric_plan(lib, n, splits):
    plan = apg.nbody_plan_forces(n, 152, path=apg.NBODY_PATH_SYMMETRIC, splits=splits)
    assert plan["path"] == apg.NBODY_PATH_SYMMETRIC
    _sym_covers(plan, n)
    assert plan["scratch_bytes"] <= max(apg.NBODY_DEFAULT_WORKSPACE_BYTES, 48 * n)
    if splits:
        units = plan["dists"] * plan["threads"] * plan["i_per_thread"] // plan["tile"]
        assert plan["splits"] == min(splits, max(1, units)) or plan["splits"] <= splits


@pytest.mark.parametrize("sm", [1, 148, 160, 264])
@pytest.mark.parametrize("n", [10240, 45056, 163840, 327680, 1048576, 2097159])
@pytest.mark.parametrize("variant", [-1, 0, 1, 2])
def test_symmetric_plan_other_gpus_and_variants(n, sm, variant):
    plan = apg.nbody_plan_forces(n, sm, path=apg.NBODY_PATH_SYMMETRIC, variant=variant)
    assert plan["path"] == apg.NBODY_PATH_SYMMETRIC
    if variant >= 0:
        assert plan["variant"] == variant
    _sym_covers(plan, n)
    assert plan["scratch_bytes"] <= apg.NBODY_DEFAULT_WORKSPACE_BYTES


def test_symmetric_plan_forced_splits_stay_within_the_budget():
    plan = apg.nbody_plan_forces(2 ** 21, 152, path=apg.NBODY_PATH_SYMMETRIC, splits=1000)
    assert plan["scratch_bytes"] <= apg.NBODY_DEFAULT_WORKSPACE_BYTES and plan["splits"] < 1000
    _sym_covers(plan, 2 ** 21)


def test_symmetric_plan_limits():
    with pytest.raises(apg.NbodyError):      # the compensated kernel is tiled only
        apg.nbody_plan_forces(65536, 152, path=apg.NBODY_PATH_SYMMETRIC,
                              precision=apg.NBODY_PRECISION_COMPENSATED)
    with pytest.raises(apg.NbodyError) as e:  # a forced symmetric path without room for a group
        apg.nbody_plan_forces(65536, 152, path=apg.NBODY_PATH_SYMMETRIC, workspace_bytes=1 << 20)
    assert e.value.status == 8
    # the symmetric path serves every n: its workspace is bounded by a budget,
    # not by n^2 (the pool-based calls allow one group's minimum beyond it)
    for n in (2 ** 23, 2 ** 25, 2 ** 31 - 1):
        plan = apg.nbody_plan_forces(n, 152)
        assert plan["path"] == apg.NBODY_PATH_SYMMETRIC
        _sym_covers(plan, n)
        assert plan["scratch_bytes"] <= max(apg.NBODY_DEFAULT_WORKSPACE_BYTES, 48 * n)


def test_default_workspace_at_one_million():
    """The benchmark's call: the symmetric path within the default budget."""
    plan = apg.nbody_plan_forces(1048576, 152)
    assert plan["path"] == apg.NBODY_PATH_SYMMETRIC
    assert 0 < plan["scratch_bytes"] <= apg.NBODY_DEFAULT_WORKSPACE_BYTES
    assert plan["passes"] > 1 and plan["fill"] > 0.97


@pytest.mark.parametrize("n", [20011, 65536, 200003, 1048576])
def test_workspace_budget_changes_passes_not_the_decomposition(n):
    """Every workspace of at least one group keeps the pieces, the distances
    per group and therefore the partial sums and their order; only the
    groups per pass change."""
    base = apg.nbody_plan_forces(n, 152)
    lo = base["scratch_min_bytes"]
    seen_passes = set()
    for budget in (lo, lo + 1, lo + 16 * n * 50, 2 * lo, 10 * lo, 1 << 40):
        plan = apg.nbody_plan_forces(n, 152, workspace_bytes=budget)
        assert (plan["path"], plan["variant"], plan["splits"], plan["dists"], plan["groups"]) == \
               (base["path"], base["variant"], base["splits"], base["dists"], base["groups"])
        assert plan["scratch_bytes"] <= budget
        seen_passes.add(plan["passes"])
        if budget == 1 << 40:
            assert plan["passes"] == 1
    # below one group the automatic choice runs without partials
    none = apg.nbody_plan_forces(n, 152, workspace_bytes=0)
    assert none["scratch_bytes"] == 0 and none["splits"] == 1


def test_tiled_passes_within_a_workspace():
    n = 200003
    base = apg.nbody_plan_forces(n, 152, path=apg.NBODY_PATH_TILED)
    assert base["splits"] > 2
    for budget in (2 * 16 * n, 3 * 16 * n, 16 * n * base["splits"]):
        plan = apg.nbody_plan_forces(n, 152, path=apg.NBODY_PATH_TILED, workspace_bytes=budget)
        assert plan["splits"] == base["splits"] and plan["scratch_bytes"] <= budget
        _covers(plan, n, budget)
    small = apg.nbody_plan_forces(n, 152, path=apg.NBODY_PATH_TILED, workspace_bytes=16 * n)
    assert small["splits"] == 1 and small["scratch_bytes"] == 0


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
        if path == apg.NBODY_PATH_TILED:   # the symmetric path fills waves with groups too
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
    for n in (1, 1024, 4096, 4864, 8192, 10239):
        assert apg.nbody_plan_forces(n, 152)["path"] == apg.NBODY_PATH_ROWS
    assert apg.nbody_plan_forces(10240, 152)["path"] == apg.NBODY_PATH_SYMMETRIC
    # target/source calls: the row-split path for fewer than 10240 sources and
    # up to 131072 targets where its piece sums fit, the tiled path otherwise
    ts = lambda nt, ns: apg.nbody_plan_forces_ts(nt, ns, 152)["path"]
    assert ts(20000, 1000) == ts(131072, 2000) == ts(5000, 10239) == apg.NBODY_PATH_ROWS
    assert ts(131073, 2000) == ts(131072, 10000) == ts(100, 10240) == apg.NBODY_PATH_TILED
    assert ts(1000000, 1000) == apg.NBODY_PATH_TILED
    # the row-split variant by the cost model, the measured fastest: K = 7, except
    # K = 4 (12 warps) at 4864
    assert [apg.nbody_plan_forces(n, 152)["i_per_thread"] for n in (1024, 4096, 4864, 8192)] == \
        [7, 7, 4, 7]
    # the symmetric block size grows with n: 512, 1024, then 2048 bodies
    blocks = [apg.nbody_plan_forces(n, 152)["threads"] * apg.nbody_plan_forces(n, 152)["i_per_thread"]
              for n in (10240, 45055, 45056, 327679, 327680, 1048576)]
    assert blocks == [512, 512, 1024, 1024, 2048, 2048]
    assert apg.nbody_plan_forces(1048576, 152)["path"] == apg.NBODY_PATH_SYMMETRIC
    with pytest.raises(apg.NbodyError):
        apg.nbody_plan_forces(1000, 152, path=apg.NBODY_PATH_CLUSTER, splits=3)
    with pytest.raises(apg.NbodyError):
        apg.nbody_plan_forces(1000, 152, path=7)
    with pytest.raises(apg.NbodyError):      # distances per group belong to the symmetric path
        apg.nbody_plan_forces(20000, 152, path=apg.NBODY_PATH_TILED, dists=3)
    with pytest.raises(apg.NbodyError):
        apg.nbody_plan_forces(20000, 152, quantities=2)


def test_symmetric_finer_pieces():
    """From 16384 bodies the 512- and 1024-body blocks take 3x (else 2x) the
    wave model's pieces in one pass, pieces within 10 % of equal; the
    2048-body blocks and smaller n keep the model's count."""
    picks = {n: apg.nbody_plan_forces(n, 152)["splits"]
             for n in (12000, 16384, 20000, 45056, 65536, 100000, 200003, 1048576)}
    assert picks == {12000: 35, 16384: 68, 20000: 84, 45056: 39, 65536: 57, 100000: 18,
                     200003: 102, 1048576: 16}
    for n in (16384, 20000, 30000, 45055, 45056, 65536, 100000, 163839, 200003):
        plan = apg.nbody_plan_forces(n, 152)
        nb, d, p = plan["num_iblocks"], plan["dists"], plan["splits"]
        spb = plan["threads"] * plan["i_per_thread"] // plan["tile"]
        units = min(d, _ndist(nb)) * spb
        assert plan["passes"] == 1 and -(-units // p) * p <= 1.1 * units
        _covers(plan, n)


def test_acceleration_only_plans_like_the_default():
    for n in (1000, 8192, 20011, 1048576):
        a = apg.nbody_plan_forces(n, 152)
        b = apg.nbody_plan_forces(n, 152, quantities=apg.NBODY_QUANTITIES_ACC)
        assert a == b


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
    with pytest.raises(apg.NbodyError):
        apg.nbody_plan_forces(1000, 152, workspace_bytes=-1)


# ------------------------------------------------------------ workspace entry points

SZ = ctypes.c_size_t


def test_workspace_argument_checks(lib):
    """The *_ws calls check the workspace like the body arrays (nothing below
    reaches CUDA: each call is rejected on the host)."""
    a, o = P, P + 4096
    n = 10

    def ws_call(ws, nbytes, pm=a, acc=o):
        size = SZ(nbytes)
        return lib.nbody_forces_ws(ctypes.c_void_p(pm), n, ctypes.c_float(1e-4),
                                   ctypes.c_void_p(acc), None, ctypes.c_void_p(ws),
                                   ctypes.byref(size), None)
    assert ws_call(P + 8192 + 8, 1024) == 2            # misaligned workspace
    assert ws_call(a + 64, 1024) == 3                  # workspace overlaps the bodies
    assert ws_call(o - 512, 1024) == 3                 # workspace overlaps the output
    assert ws_call(P + 8192, 1024, pm=a + 4) == 2      # body checks still apply
    assert lib.nbody_forces_ws(ctypes.c_void_p(a), n, ctypes.c_float(1e-4), ctypes.c_void_p(o),
                               None, ctypes.c_void_p(P + 8192), None, None) == 1   # no size
    size = SZ(0)
    assert lib.nbody_forces_ws(None, -1, ctypes.c_float(1e-4), None, None, None,
                               ctypes.byref(size), None) == 1                    # bad n in a query
    assert lib.nbody_forces_ws(None, 5, ctypes.c_float(0.0), None, None, None,
                               ctypes.byref(size), None) == 1                    # bad eps2 in a query
    assert lib.nbody_forces_ws(None, 0, ctypes.c_float(1e-4), None, None, None,
                               ctypes.byref(size), None) == 0 and size.value == 0

    def ts_call(ws, nbytes):
        size = SZ(nbytes)
        return lib.nbody_forces_ts_ws(ctypes.c_void_p(P), 5, ctypes.c_void_p(P + 4096), 7,
                                      ctypes.c_float(1e-4), ctypes.c_void_p(P + 8192), None,
                                      ctypes.c_void_p(ws), ctypes.byref(size), None)
    assert ts_call(P + 4096 + 16, 64) == 3             # overlaps the sources
    assert ts_call(P + 12288 + 4, 64) == 2

    def sim_call(ws, nbytes):
        size = SZ(nbytes)
        return lib.nbody_simulate_ws(ctypes.c_void_p(a), ctypes.c_void_p(P + 4096),
                                     ctypes.c_void_p(P + 8192), n, ctypes.c_float(1e-4),
                                     ctypes.c_float(1e-3), 2, ctypes.c_void_p(ws),
                                     ctypes.byref(size), None)
    assert sim_call(P + 4096 + 32, 64) == 3            # overlaps the velocities
    assert sim_call(P + 12288 + 8, 64) == 2
