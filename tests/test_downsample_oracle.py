"""Pins of the centroid-downsampling oracle (no GPU).

* a hand-worked example with exact means (tests/golden/downsample_example.txt);
* a restatement with exact sums (math.fsum) on random tiny clouds and on
  slices of the workloads: integer outputs equal, centroids within one
  float32 unit in the last place (the oracle sums in double in index order:
  its sum differs from the exact one by at most (n - 1) * 2^-53 of the sum
  of magnitudes, far below half a float32 ulp of a mean of values of one
  sign, so only a mean sitting next to a float32 rounding boundary can move,
  and then by one ulp);
* invariants: counts add up to the valid points, every centroid lies in its
  voxel's box;
* planted mistakes in the oracle are caught.
"""

from __future__ import annotations

import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle
from _helpers import random_tiny_case
from lidar_point_cloud_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_example():
    pts, cases = [], []
    for line in open(os.path.join(GOLDEN, "downsample_example.txt")):
        s = line.split("#", 1)[0].split()
        if not s:
            continue
        if s[0] == "range":
            rng = tuple(float(t) for t in s[1:7])
        elif s[0] == "voxel" and len(s) == 4:
            vox = tuple(float(t) for t in s[1:4])
        elif s[0] == "point":
            pts.append([float(t) for t in s[2:6]])
        elif s[0] == "case":
            kv = dict(t.split("=") for t in s[1:])
            cases.append({"M": int(kv["max_voxels"]), "V": int(kv["V"]), "rows": []})
        elif s[0] == "voxel":
            cases[-1]["rows"].append((int(s[1]), tuple(int(t) for t in s[3:6]), int(s[7]),
                                      tuple(float(t) for t in s[9:13])))
    return rng, vox, np.array(pts, np.float32), cases


def pin_example(lib):
    fails = []
    rng, vox, pts, cases = read_example()
    for case in cases:
        M = case["M"]
        ec = np.zeros((M, 4), np.float32)
        eco = np.zeros((M, 3), np.int32)
        en = np.zeros((M,), np.int32)
        for r, co, n, c in case["rows"]:
            ec[r], eco[r], en[r] = c, co, n
        st, c, co, n, V = oracle.downsample(pts, rng, vox, M, lib)
        if st != 0 or V != case["V"] or c.tobytes() != ec.tobytes() or co.tobytes() != eco.tobytes() \
                or n.tobytes() != en.tobytes():
            fails.append(f"example M={M}: V {V}; centroids {c[:case['V']].tolist()}")
    return fails


def pin_exact(lib, n_cases=80, seed=606):
    fails = []
    rng = np.random.Generator(np.random.PCG64(seed))
    for t in range(n_cases):
        pts, r, v, K, M = random_tiny_case(rng, gz_max=4)
        M = M * 3
        st, c, co, n, V = oracle.downsample(pts, r, v, M, lib)
        ec, eco, en, eV = oracle.downsample_exact(pts, r, v, M)
        if st != 0 or V != eV or co.tobytes() != eco.tobytes() or n.tobytes() != en.tobytes() \
                or oracle.ulp_distance32(c, ec).max(initial=0) > 1:
            fails.append(f"case {t}: V {V} vs {eV}")
            if len(fails) > 3:
                break
    return fails


PINS = (pin_example, pin_exact)


def test_hand_worked_example():
    assert pin_example(oracle.load()) == []


def test_exact_sums_random_tiny():
    assert pin_exact(oracle.load()) == []


@pytest.mark.parametrize("name", ["kitti3d", "dense3d"])
def test_exact_sums_on_workload_slices(name):
    pts, P = synth.make(name)
    part = pts[:30_000]
    st, c, co, n, V = oracle.downsample(part, P.point_cloud_range, P.voxel_size, P.max_voxels)
    ec, eco, en, eV = oracle.downsample_exact(part, P.point_cloud_range, P.voxel_size, P.max_voxels)
    assert st == 0 and V == eV and co.tobytes() == eco.tobytes() and n.tobytes() == en.tobytes()
    assert oracle.ulp_distance32(c, ec).max() <= 1


@pytest.mark.parametrize("name", ["kitti3d", "second", "dense3d"])
def test_invariants(name):
    pts, P = synth.make(name)
    st, c, co, n, V = oracle.downsample(pts, P.point_cloud_range, P.voxel_size, 10 ** 6)
    ok, *_ = oracle.cells_numpy(pts, P.point_cloud_range, P.voxel_size)
    assert st == 0 and n[:V].sum() == ok.sum() and np.all(n[:V] > 0)
    lo = np.array(P.point_cloud_range[:3], np.float64)
    vs = np.array(P.voxel_size, np.float64)
    cell = co[:V, ::-1].astype(np.float64)  # (x, y, z)
    a = lo + cell * vs
    b = a + vs
    slack = 1e-5 * np.maximum(1.0, np.abs(b))
    assert np.all(c[:V, :3] >= a - slack) and np.all(c[:V, :3] <= b + slack)


MUTANTS = {
    "float_sums": ("sum[4 * static_cast<size_t>(r) + c] += static_cast<double>(p[c]);",
                   "sum[4 * static_cast<size_t>(r) + c] = static_cast<double>(static_cast<float>("
                   "sum[4 * static_cast<size_t>(r) + c]) + p[c]);"),
    "count_plus_one": ("/ static_cast<double>(out_counts[r]));", "/ static_cast<double>(out_counts[r] + 1));"),
    "intensity_not_averaged": ("for (int c = 0; c < 4; ++c) sum[", "for (int c = 0; c < 3; ++c) sum["),
    "voxel_id_without_z": ("cell[0] + grid[0] * (cell[1] + grid[1] * cell[2]);", "cell[0] + grid[0] * cell[1];"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="pv_ds_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, mutant_dir):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "pv_oracle.cpp")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    path = os.path.join(mutant_dir, f"{name}.cpp")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.load_path(oracle.build(src=path, out=os.path.join(mutant_dir, f"{name}.so")))
    fails = []
    for pin in PINS:
        fails += pin(lib)
        if fails:
            break
    assert fails, f"mutant {name} passed every pin"
