"""Pins of the CPU oracle to things other than itself (no GPU needed).

* the grid size the page prints (432 x 496 = 214,272 pillars, "Fig. 2");
* a hand-derived boundary table, re-derived here with exact rational
  arithmetic ("Binning a point");
* points whose cell needs a correctly rounded division;
* a hand-worked example of the canonical layout;
* an O(N^2) brute force and a NumPy stable-sort restatement on random tiny
  clouds where both caps bind;
* invariants and the canonical order on the seeded workloads;
* the expected number of distinct pillars of a uniform cloud;
* planted mistakes: mutated copies of the oracle must fail at least one pin.
"""

from __future__ import annotations

import math
import os
import re
import shutil
import tempfile

import numpy as np
import pytest

import oracle
from lidar_point_cloud_gb300 import synth
from _helpers import (
    check_invariants, check_order_with_index_intensity, exact_cell, f32_of_bits, first_difference,
    random_tiny_case, read_division_points, read_edge_points, read_worked_example, same_bits,
    worked_expected,
)

KR, KV = synth.KITTI_RANGE, synth.KITTI_VOXEL


# ---------------------------------------------------------------- pin checks
# Each returns a list of failure strings so the mutant test can reuse them.

def pin_grid(lib):
    fails = []
    st, g = oracle.grid(KR, KV, lib)
    if st != 0 or g != (432, 496, 1) or g[0] * g[1] != 214_272:
        fails.append(f"KITTI grid {st} {g}")
    st, g = oracle.grid(synth.DENSE_RANGE, synth.DENSE_VOXEL, lib)
    if st != 0 or g != (1024, 1024, 1):
        fails.append(f"dense grid {st} {g}")
    return fails


def pin_edges(lib):
    fails = []
    for bits, exp in read_edge_points():
        p = [f32_of_bits(b) for b in bits]
        got = oracle.bin_point(p, KR, KV, lib)
        if got != exp:
            fails.append(f"edge {[hex(b) for b in bits]}: {got} != {exp}")
    return fails


def pin_division(lib):
    fails = []
    for b, cx in read_division_points():
        got = oracle.bin_point([f32_of_bits(b), 0.0, -1.0, 0.5], KR, KV, lib)
        if got != (cx, 248, 0):
            fails.append(f"division {hex(b)}: {got} != {cx}")
    return fails


def pin_worked(lib):
    fails = []
    rng, vox, pts, cases = read_worked_example()
    for case in cases:
        ev, ec, en, eV = worked_expected(pts, case)
        st, v, c, n, V = oracle.voxelize(pts, rng, vox, case["max_points"], case["max_voxels"], lib)
        if st != 0 or V != eV or not (same_bits(v, ev) and same_bits(c, ec) and same_bits(n, en)):
            fails.append(f"worked case {case['max_points']},{case['max_voxels']}: "
                         f"V {V} vs {eV}; vox {first_difference(v, ev)}; coords {first_difference(c, ec)}")
    return fails


def pin_grid3d(lib):
    fails = []
    st, g = oracle.grid3d(KR, (0.16, 0.16, 0.5), lib)
    if st != 0 or g != (432, 496, 8):  # 4 m slab / 0.5 m
        fails.append(f"KITTI 3-D grid {st} {g}")
    # A SECOND-style grid: [0, 70.4] x [-40, 40] x [-3, 1] at 0.05 x 0.05 x 0.1 m.
    st, g = oracle.grid3d((0.0, -40.0, -3.0, 70.4, 40.0, 1.0), (0.05, 0.05, 0.1), lib)
    if st != 0 or g != (1408, 1600, 40):
        fails.append(f"fine 3-D grid {st} {g}")
    st, g = oracle.grid3d(KR, KV, lib)  # one layer: the pillar grid
    if st != 0 or g != (432, 496, 1):
        fails.append(f"one-layer grid {st} {g}")
    return fails


def pin_worked3d(lib):
    fails = []
    rng, vox, pts, cases = read_worked_example("worked_example_3d.txt")
    for case in cases:
        ev, ec, en, eV = worked_expected(pts, case)
        st, v, c, n, V = oracle.voxelize3d(pts, rng, vox, case["max_points"], case["max_voxels"], lib)
        if st != 0 or V != eV or not (same_bits(v, ev) and same_bits(c, ec) and same_bits(n, en)):
            fails.append(f"3-D worked case {case['max_points']},{case['max_voxels']}: "
                         f"V {V} vs {eV}; vox {first_difference(v, ev)}; coords {first_difference(c, ec)}")
    return fails


def pin_bruteforce3d(lib, n_cases=80, seed=2025):
    fails = []
    rng = np.random.Generator(np.random.PCG64(seed))
    for t in range(n_cases):
        pts, r, v, K, M = random_tiny_case(rng, gz_max=5)
        st, ov, oc, on, oV = oracle.voxelize3d(pts, r, v, K, M, lib)
        bv, bc, bn, bV = oracle.voxelize_bruteforce(pts, r, v, K, M, three_d=True)
        if st != 0 or oV != bV or not (same_bits(ov, bv) and same_bits(oc, bc) and same_bits(on, bn)):
            fails.append(f"3-D case {t}: V {oV} vs {bV}; {first_difference(ov, bv)}; {first_difference(oc, bc)}")
            if len(fails) > 3:
                break
    return fails


def pin_bruteforce(lib, n_cases=120, seed=2024):
    fails = []
    rng = np.random.Generator(np.random.PCG64(seed))
    for t in range(n_cases):
        pts, r, v, K, M = random_tiny_case(rng)
        st, ov, oc, on, oV = oracle.voxelize(pts, r, v, K, M, lib)
        bv, bc, bn, bV = oracle.voxelize_bruteforce(pts, r, v, K, M)
        if st != 0 or oV != bV or not (same_bits(ov, bv) and same_bits(oc, bc) and same_bits(on, bn)):
            fails.append(f"case {t}: V {oV} vs {bV}; {first_difference(ov, bv)}")
            if len(fails) > 3:
                break
    return fails


ALL_PINS = (pin_grid, pin_edges, pin_division, pin_worked, pin_bruteforce, pin_grid3d, pin_worked3d, pin_bruteforce3d)


# ------------------------------------------------------------- the pins pass

def test_grid_matches_page():
    assert pin_grid(oracle.load()) == []
    assert oracle.grid_py(KR, KV) == (432, 496, 1)


def test_edge_table_is_exact_arithmetic():
    """The golden boundary table agrees with exact rational binary32 steps."""
    g = (432, 496, 1)
    for bits, exp in read_edge_points():
        if any((b & 0x7F800000) == 0x7F800000 for b in bits[:3]):
            assert exp is None
            continue
        cells = [exact_cell(bits[a], KR[a], KV[a], g[a]) for a in range(3)]
        derived = None if any(c is None for c in cells) else tuple(cells)
        assert derived == exp, ([hex(b) for b in bits], derived, exp)


def test_division_table_is_exact_arithmetic():
    for b, cx in read_division_points():
        assert exact_cell(b, KR[0], KV[0], 432) == cx
        # The same point under a rounded-reciprocal multiply lands one lower.
        x = np.float32(f32_of_bits(b))
        assert int(np.floor(x * (np.float32(1.0) / np.float32(KV[0])))) == cx - 1


def test_edge_points_oracle():
    assert pin_edges(oracle.load()) == []


def test_edge_points_numpy_restatement():
    pts = synth.edge_points()
    ok, cx, cy, g = oracle.bin_numpy(pts, KR, KV)
    for i, (bits, exp) in enumerate(read_edge_points()):
        got = (int(cx[i]), int(cy[i]), 0) if ok[i] else None
        assert got == exp, i


def test_edge_points_match_generator():
    """The boundary points the tiny workload appends are the table's points."""
    tbl = np.array([b for b, _ in read_edge_points()], dtype=np.uint32)
    assert np.array_equal(tbl, synth.EDGE_POINT_BITS)
    tiny = synth.tiny()
    assert np.array_equal(tiny[-16:].view(np.uint32), tbl)


def test_division_points_oracle():
    assert pin_division(oracle.load()) == []


def test_worked_example_all_three():
    assert pin_worked(oracle.load()) == []
    rng, vox, pts, cases = read_worked_example()
    for case in cases:
        ev, ec, en, eV = worked_expected(pts, case)
        for fn in (oracle.voxelize_numpy, oracle.voxelize_bruteforce):
            v, c, n, V = fn(pts, rng, vox, case["max_points"], case["max_voxels"])
            assert V == eV and same_bits(v, ev) and same_bits(c, ec) and same_bits(n, en), fn.__name__


def test_bruteforce_random_tiny():
    assert pin_bruteforce(oracle.load()) == []


def test_voxel3d_grid():
    assert pin_grid3d(oracle.load()) == []


def test_voxel3d_worked_example_all_three():
    assert pin_worked3d(oracle.load()) == []
    rng, vox, pts, cases = read_worked_example("worked_example_3d.txt")
    for case in cases:
        ev, ec, en, eV = worked_expected(pts, case)
        for fn in (oracle.voxelize_numpy, oracle.voxelize_bruteforce):
            v, c, n, V = fn(pts, rng, vox, case["max_points"], case["max_voxels"], three_d=True)
            assert V == eV and same_bits(v, ev) and same_bits(c, ec) and same_bits(n, en), fn.__name__


def test_voxel3d_bruteforce_random_tiny():
    assert pin_bruteforce3d(oracle.load()) == []


def test_voxel3d_numpy_restatement_random_tiny():
    rng = np.random.Generator(np.random.PCG64(78))
    lib = oracle.load()
    for _ in range(150):
        pts, r, v, K, M = random_tiny_case(rng, gz_max=5)
        st, ov, oc, on, oV = oracle.voxelize3d(pts, r, v, K, M, lib)
        nv, nc, nn, nV = oracle.voxelize_numpy(pts, r, v, K, M, three_d=True)
        assert st == 0 and oV == nV
        assert same_bits(ov, nv) and same_bits(oc, nc) and same_bits(on, nn)


@pytest.mark.parametrize("name", ["tiny", "kitti", "uniform_50000"])
def test_voxel3d_with_one_layer_is_the_pillar_oracle(name):
    pts, P = synth.make(name)
    a = oracle.voxelize(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)
    b = oracle.voxelize3d(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)
    assert a[0] == b[0] == 0 and a[4] == b[4]
    assert all(same_bits(x, y) for x, y in zip(a[1:4], b[1:4]))


def test_numpy_restatement_random_tiny():
    rng = np.random.Generator(np.random.PCG64(77))
    lib = oracle.load()
    for _ in range(200):
        pts, r, v, K, M = random_tiny_case(rng)
        st, ov, oc, on, oV = oracle.voxelize(pts, r, v, K, M, lib)
        nv, nc, nn, nV = oracle.voxelize_numpy(pts, r, v, K, M)
        assert st == 0 and oV == nV
        assert same_bits(ov, nv) and same_bits(oc, nc) and same_bits(on, nn)


def test_argument_errors():
    lib = oracle.load()
    pts = synth.uniform(10, 0)
    assert oracle.voxelize(pts, KR, (0.16, 0.16, 2.0), 32, 100, lib)[0] == oracle.ERR_UNSUPPORTED
    assert oracle.voxelize(pts, KR, (0.0, 0.16, 4.0), 32, 100, lib)[0] == oracle.ERR_INVALID
    assert oracle.voxelize(pts, (1, 0, 0, 0, 1, 1), (0.16, 0.16, 4.0), 32, 100, lib)[0] == oracle.ERR_INVALID
    assert oracle.voxelize(pts, KR, (float("nan"), 0.16, 4.0), 32, 100, lib)[0] == oracle.ERR_INVALID
    assert oracle.voxelize(pts, KR, KV, 0, 100, lib)[0] == oracle.ERR_INVALID
    assert oracle.voxelize(pts, KR, KV, 32, 0, lib)[0] == oracle.ERR_INVALID


def test_empty_cloud():
    st, v, c, n, V = oracle.voxelize(np.zeros((0, 4), np.float32), KR, KV, 32, 16, oracle.load())
    assert st == 0 and V == 0 and not v.any() and not c.any() and not n.any()


# ----------------------------------------------------- invariants on workloads

def _independent_keys(pts, r, v):
    ok, cx, cy, g = oracle.bin_numpy(pts, r, v)
    keys = np.where(ok, cy * g[0] + cx, -1)
    return ok, keys, (g[0], g[1])


@pytest.mark.parametrize("name", ["tiny", "kitti", "uniform_25000", "uniform_130000", "dense"])
def test_invariants_on_workloads(name):
    pts, P = synth.make(name)
    st, v, c, n, V = oracle.voxelize(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)
    assert st == 0
    ok, keys, gxy = _independent_keys(pts, P.point_cloud_range, P.voxel_size)
    check_invariants(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels, v, c, n, V,
                     ok, keys, gxy)


@pytest.mark.parametrize("name", ["tiny", "kitti", "uniform_130000"])
def test_order_with_index_intensity(name):
    pts, P = synth.make(name)
    pts = pts.copy()
    pts[:, 3] = np.arange(pts.shape[0], dtype=np.float32)  # exact below 2^24
    st, v, c, n, V = oracle.voxelize(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)
    ok, keys, _ = _independent_keys(pts, P.point_cloud_range, P.voxel_size)
    check_order_with_index_intensity(pts, v, n, V, ok, keys)
    # Kept points of each pillar are exactly its first min(n, K) points.
    vi = np.flatnonzero(ok)
    s = np.argsort(keys[vi], kind="stable")
    k_sorted = keys[vi][s]
    starts = np.r_[0, np.flatnonzero(np.diff(k_sorted)) + 1]
    first_of_group = vi[s][starts]
    order = np.argsort(first_of_group)[:V]
    for r in range(0, V, max(1, V // 300)):
        gstart = starts[order[r]]
        gend = starts[order[r] + 1] if order[r] + 1 < starts.size else k_sorted.size
        want = vi[s][gstart:gend][: P.max_points]
        assert np.array_equal(v[r, : n[r], 3].astype(np.int64), want)


def test_uniform_distinct_pillars_statistics():
    """Distinct pillars of n uniform points over C cells: C (1 - exp(-n / C))."""
    C = 432 * 496
    for n in synth.UNIFORM_SIZES:
        pts = synth.uniform(n, 2 + synth.UNIFORM_SIZES.index(n))
        ok, keys, _ = _independent_keys(pts, KR, KV)
        d = np.unique(keys[ok]).size
        mean = C * (1 - math.exp(-n / C))
        var = C * math.exp(-n / C) * (1 - (1 + n / C) * math.exp(-n / C))
        assert abs(d - mean) < 6 * math.sqrt(var) + 5, (n, d, mean)


# ------------------------------------------------------------ planted mistakes

MUTANTS = {
    "truncate_instead_of_floor": ("std::floor(q)", "std::trunc(q)"),
    "upper_bound_inclusive": ("f < static_cast<float>(cells)", "f <= static_cast<float>(cells)"),
    "reciprocal_multiply": ("float q = d / v;", "float q = d * (1.0f / v);"),
    "sign_of_offset": ("float d = c - lo;", "float d = c + lo;"),
    "coords_transposed": ("static_cast<int32_t>(id / grid[0]);\n        out_coords[3 * r + 2] = static_cast<int32_t>(id % grid[0]);",
                          "static_cast<int32_t>(id % grid[0]);\n        out_coords[3 * r + 2] = static_cast<int32_t>(id / grid[0]);"),
    "voxel_z_stride": ("(cell[2] * grid[1] + cell[1])", "(cell[2] * grid[0] + cell[1])"),
    "voxel_z_coordinate_zero": ("out_coords[3 * r + 0] = static_cast<int32_t>(cell[2]);",
                                "out_coords[3 * r + 0] = 0;"),
    "voxel_grid_keeps_pillar_check": ("  if (grid_out[0] * grid_out[1] * grid_out[2] >= (int64_t(1) << 31))\n    return kErrInvalid;\n  return kOk;",
                                      "  if (grid_out[0] * grid_out[1] * grid_out[2] >= (int64_t(1) << 31))\n    return kErrInvalid;\n  if (grid_out[2] != 1) return kErrUnsupported;\n  return kOk;"),
    "wrong_row_stride": ("cell[1] * grid[0] + cell[0]", "cell[1] * grid[1] + cell[0]"),
    "nan_check_on_intensity": ("!is_finite_bits(p[2])", "!is_finite_bits(p[3])"),
    # (Dropping the explicit NaN/Inf test is an equivalent mutant: the float
    # bounds test already rejects NaN and +-Inf, so it is not listed.)
    "keep_last_instead_of_first": (
        "if (k >= max_points) continue;",
        "if (k >= max_points) { std::memcpy(out_voxels + static_cast<size_t>(r) * row_floats"
        " + static_cast<size_t>(max_points - 1) * 4, p, 16); continue; }"),
    "point_cap_off_by_one": ("if (k >= max_points) continue;", "if (k + 1 >= max_points) continue;"),
    "grid_ceil": ("std::llround(len / static_cast<double>(v))", "std::ceil(len / static_cast<double>(v))"),
    "z_slab_unchecked": ("for (int a = 0; a < 3; ++a)\n    if (!bin_axis", "for (int a = 0; a < 2; ++a)\n    if (!bin_axis"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="pv_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, mutant_dir):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "pv_oracle.cpp")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path_src = os.path.join(mutant_dir, f"{name}.cpp")
    with open(path_src, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.load_path(oracle.build(src=path_src, out=os.path.join(mutant_dir, f"{name}.so")))
    failures = []
    for pin in ALL_PINS:
        try:
            failures += pin(lib) if pin is not pin_bruteforce else pin(lib, n_cases=60)
        except Exception as e:  # a crash in the mutant also counts as caught
            failures.append(f"{pin.__name__} raised {e!r}")
        if failures:
            break
    assert failures, f"mutant {name} passed every pin"


# ------------------------------------------------------------ stored digests

def _read_digests():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "oracle_digests.txt")
    out = {}
    for line in open(path):
        if line.strip() and not line.startswith("#"):
            name, V, d = line.split()
            out[name] = (int(V), d)
    return out


@pytest.mark.parametrize("name", ["tiny", "kitti", "uniform_25000", "uniform_130000", "dense", "adversarial"])
def test_oracle_digests_unchanged(name):
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "make_digests", os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "make_digests.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    assert mod.digest(name) == _read_digests()[name]
