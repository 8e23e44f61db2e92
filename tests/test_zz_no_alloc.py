"""nbody_forces_noalloc, the entry point for callers that may not allocate
device memory (a host framework that owns all GPU memory, code under a hard
latency budget, a fixed memory budget): it keeps its split partials in a
fixed array inside the library.

Checked through the C ABI against nbody_forces and against the oracle, two
calls in a row (the second sees whatever the first left in the shared
array), with the parity tolerances of the other GPU tests; the calls after
the one-time set-up leave the device's free memory unchanged.  This file is
collected last.
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
    assert torch.cuda.is_available(), "this test needs a CUDA GPU"


def _close(got, ref):
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    l2a = np.linalg.norm(got[:, :3] - ref[:, :3]) / np.linalg.norm(ref[:, :3])
    l2p = np.linalg.norm(got[:, 3] - ref[:, 3]) / np.linalg.norm(ref[:, 3])
    ba = (np.linalg.norm(got[:, :3] - ref[:, :3], axis=1) / np.linalg.norm(ref[:, :3], axis=1)).max()
    bp = (np.abs(got[:, 3] - ref[:, 3]) / np.abs(ref[:, 3])).max()
    assert l2a <= L2_TOL and l2p <= L2_TOL and ba <= BODY_TOL and bp <= BODY_TOL, (l2a, l2p, ba, bp)


def _noalloc_splits(n, sm, occ):
    """The split count nbody_forces_noalloc chooses: the best predicted fill
    over S <= NBODY_NOALLOC_MAX_N / n (at most 256), on the tiled path."""
    best, best_fill = None, -1.0
    for s in range(1, min(apg.NBODY_NOALLOC_MAX_N // n, 256) + 1):
        p = apg.nbody_plan_forces(n, sm, occ, path=apg.NBODY_PATH_TILED, splits=s)
        if p["splits"] > apg.NBODY_NOALLOC_MAX_N // n:
            continue
        if best is None or p["fill"] > best_fill * (1.0 + 1e-3):
            best, best_fill = p["splits"], p["fill"]
    return best


def test_noalloc_matches_nbody_forces_and_the_oracle_on_two_calls_in_a_row():
    dev = torch.device("cuda:0")
    sm = torch.cuda.get_device_properties(dev).multi_processor_count
    # one-time set-up of the entry point on this device, and the first use
    # of its kernels (loading a kernel's code may take device memory)
    warm = torch.from_numpy(W.cube(20011, seed=1).pos_mass).to(dev)
    apg.nbody_forces_noalloc(warm, 1e-4, torch.empty_like(warm))
    torch.cuda.synchronize()
    # the larger problem first, so the second call runs over the first's leftovers
    for w in (W.clumps(65536, seed=21), W.cube(20011, seed=22)):
        # both sizes are split over several CTAs, i.e. through the fixed scratch
        # (the default tiled kernel holds 2 CTAs per SM)
        assert _noalloc_splits(w.n, sm, 2) > 1
        pm = torch.from_numpy(w.pos_mass).to(dev)
        ref = apg.nbody_forces(pm, float(w.eps2))
        out = torch.full_like(pm, float("nan"))
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        apg.nbody_forces_noalloc(pm, float(w.eps2), out)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert free1 == free0                       # nothing allocated by the call
        got = out.cpu().numpy()
        _close(got, ref.cpu().numpy())
        rng = np.random.default_rng(w.n)
        rows = np.unique(np.concatenate([rng.choice(w.n, 1000, replace=False),
                                         np.arange(w.n - 50, w.n)]))
        _close(got[rows], oracle.forces(w.pos_mass, w.eps2, rows=rows))


def test_noalloc_rejects_sizes_beyond_its_scratch():
    n = apg.NBODY_NOALLOC_MAX_N + 1
    pm = torch.zeros((n, 4), device="cuda:0")
    out = torch.zeros_like(pm)
    with pytest.raises(apg.NbodyError) as e:
        apg.nbody_forces_noalloc(pm, 1e-4, out)
    assert e.value.status == 7
