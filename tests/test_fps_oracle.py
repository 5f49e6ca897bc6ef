"""Pins of the farthest-point-sampling oracle (no GPU).

* hand-worked sequences with ties (tests/golden/fps_examples.txt);
* a vectorised NumPy restatement (same float32 operation order) on random
  clouds, several sizes, sample counts and start points: identical indices;
* FPS invariants: the distance of each new sample to the earlier ones never
  grows, and samples are distinct while points remain uncovered;
* the restatement on the LiDAR-shaped benchmark cloud, whose near-ties
  expose a distance rounded once instead of per operation;
* planted mistakes in the oracle are caught.
"""

from __future__ import annotations

import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_examples():
    cases = []
    for line in open(os.path.join(GOLDEN, "fps_examples.txt")):
        s = line.split("#", 1)[0].split()
        if not s:
            continue
        if s[0] == "case":
            kv = dict(t.split("=") for t in s[2:])
            cases.append({"name": s[1], "start": int(kv["start"]),
                          "samples": [int(t) for t in kv["samples"].split(",")], "points": []})
        elif s[0] == "point":
            cases[-1]["points"].append([float(t) for t in s[1:4]] + [0.0])
    return cases


def pin_examples(lib):
    fails = []
    for c in read_examples():
        pts = np.array(c["points"], np.float32)
        st, idx = oracle.fps(pts, len(c["samples"]), c["start"], lib)
        if st != 0 or idx.tolist() != c["samples"]:
            fails.append(f"{c['name']}: {idx.tolist()} != {c['samples']}")
    return fails


def pin_restatement(lib, seed=808):
    fails = []
    rng = np.random.default_rng(seed)
    for t in range(12):
        n = int(rng.integers(1, 3000))
        m = int(rng.integers(1, 400))
        start = int(rng.integers(0, n))
        pts = (rng.random((n, 4)) * rng.choice([1.0, 30.0, 100.0])).astype(np.float32)
        if t % 3 == 0:  # duplicates and exact ties
            pts[: n // 2] = np.round(pts[: n // 2])
        st, idx = oracle.fps(pts, m, start, lib)
        ref = oracle.fps_numpy(pts, m, start)
        if st != 0 or not np.array_equal(idx, ref):
            fails.append(f"case {t}: first difference at {int(np.argmax(idx != ref))}")
    return fails


def pin_lidar_cloud(lib, samples=1600):
    """The restatement on the LiDAR-shaped benchmark cloud: its structured
    ranges put many points within an ulp of the farthest distance, so a
    distance rounded once instead of per operation (a fused multiply-add)
    picks a different sample within the first 1,600 (the first such sample of
    seed 1 is number 1,408)."""
    from lidar_point_cloud_gb300 import synth

    pts = synth.fps_cloud(1)
    st, idx = oracle.fps(pts, samples, 0, lib)
    ref = oracle.fps_numpy(pts, samples, 0)
    if st != 0 or not np.array_equal(idx, ref):
        return [f"lidar cloud: first difference at {int(np.argmax(idx != ref))}"]
    return []


PINS = (pin_examples, pin_restatement, pin_lidar_cloud)


def test_examples():
    assert pin_examples(oracle.load()) == []


def test_restatement():
    assert pin_restatement(oracle.load()) == []


def test_lidar_cloud():
    assert pin_lidar_cloud(oracle.load()) == []


def test_invariants():
    rng = np.random.default_rng(9)
    pts = (rng.random((5000, 4)) * 50).astype(np.float32)
    st, idx = oracle.fps(pts, 800, 17)
    assert st == 0 and idx[0] == 17 and np.unique(idx).size == 800
    p = pts[:, :3].astype(np.float64)
    prev = np.inf
    for k in range(1, 800):
        d = ((p[idx[:k]] - p[idx[k]]) ** 2).sum(axis=1).min()
        assert d <= prev * (1 + 1e-6)
        prev = d


def test_argument_errors():
    pts = np.zeros((4, 4), np.float32)
    assert oracle.fps(pts, 2, 4)[0] == oracle.ERR_INVALID
    assert oracle.fps(pts, 0, 0)[0] == oracle.ERR_INVALID
    bad = pts.copy()
    bad[2, 1] = np.nan
    assert oracle.fps(bad, 2, 0)[0] == oracle.ERR_INVALID


MUTANTS = {
    "tie_to_last": ("if (min_dist[i] > best_d) {", "if (min_dist[i] >= best_d) {"),
    "no_running_minimum": ("min_dist[i] = std::min(min_dist[i], d);", "min_dist[i] = d;"),
    "start_ignored": ("int64_t sel = start;", "int64_t sel = 0;"),
    "no_z_term": ("const float d = (dx * dx + dy * dy) + dz * dz;", "const float d = dx * dx + dy * dy;"),
    "fused_distance": ("const float d = (dx * dx + dy * dy) + dz * dz;",
                       "const float d = std::fma(dx, dx, dy * dy) + dz * dz;"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="pv_fps_mutants_")
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
