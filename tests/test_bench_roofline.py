"""bench.py's roofline arithmetic (CPU only): the fp32 lane operations per
interaction of each force path, counted by hand for small plans."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

LANES = 152 * 2070e6 * 128


def _plan(path, threads=256, k=8, nb=1):
    return {"path": path, "threads": threads, "i_per_thread": k, "num_iblocks": nb}


def test_ordered_pair_paths_cost_13_per_interaction():
    for path in (1, 2):
        r = bench.force_roofline(_plan(path), 5000, 152, 2070.0)
        assert r["ops_per_interaction"] == 13.0
        assert r["peak"] == pytest.approx(LANES / 13.0)
        assert r["ordered_pair_peak"] == pytest.approx(LANES / 13.0)


def test_symmetric_path_counts_diagonal_blocks_one_way():
    # n = 5000 in blocks of 2048: two full blocks and one of 904 bodies.
    # Off the diagonal blocks every unordered pair costs 18 (9 per
    # interaction); on them every ordered pair costs 13.
    n = 5000
    diag = 2 * 2048 ** 2 + 904 ** 2
    ops = 9.0 * (n * n - diag) + 13.0 * diag
    r = bench.force_roofline(_plan(3, nb=3), n, 152, 2070.0)
    assert r["ops_per_interaction"] == pytest.approx(ops / (n * n))
    assert r["peak"] == pytest.approx(LANES * n * n / ops)
    assert r["ordered_pair_peak"] == pytest.approx(LANES / 13.0)


def test_symmetric_bound_at_one_million():
    # 512 blocks of 2048: the diagonal is 0.2 % of the pairs
    n = 1 << 20
    r = bench.force_roofline(_plan(3, nb=512), n, 152, 2070.0)
    assert r["ops_per_interaction"] == pytest.approx(9.0078125)
    assert r["peak"] == pytest.approx(4.471e12, rel=1e-3)


def test_one_block_is_all_diagonal():
    r = bench.force_roofline(_plan(3, nb=1), 1000, 152, 2070.0)
    assert r["ops_per_interaction"] == 13.0


def test_kernel_source_hash_ignores_comments(tmp_path, monkeypatch):
    a = tmp_path / "a.cu"
    a.write_text("// one\nint f() { return 1; }  /* two */\n")
    monkeypatch.setitem(bench.KERNEL_SOURCES, "t", [str(a)])
    h1 = bench.kernel_source_hash("t")
    a.write_text("// changed comment\n\n  int f() {   return 1; }\n")
    assert bench.kernel_source_hash("t") == h1
    a.write_text("int f() { return 2; }\n")
    assert bench.kernel_source_hash("t") != h1
