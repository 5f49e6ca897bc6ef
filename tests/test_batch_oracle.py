"""Pins of the batched oracle (several frames per call), no GPU.

* a hand-worked two-frame batch (tests/golden/batch_example.txt);
* one frame is the single-cloud oracle with a batch index column;
* the per-frame oracle against a restatement over the whole concatenated
  cloud (grouping key (frame, voxel id), per-frame budgets), on random tiny
  batches with empty frames, pillar and 3-D grids.
"""

from __future__ import annotations

import os

import numpy as np
import pytest

import oracle
from _helpers import first_difference, random_tiny_batch, read_worked_example, same_bits
from lidar_point_cloud_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_batch_example():
    off, case, frames = None, None, {}
    for line in open(os.path.join(GOLDEN, "batch_example.txt")):
        s = line.split("#", 1)[0].split()
        if not s:
            continue
        if s[0] == "offsets":
            off = [int(t) for t in s[1:]]
        elif s[0] == "case":
            kv = dict(t.split("=") for t in s[1:])
            case = (int(kv["max_points"]), int(kv["max_voxels"]))
        elif s[0] == "frame":
            cur = int(s[1])
            frames[cur] = {"V": int(s[2].split("=")[1]), "rows": []}
        elif s[0] == "row":
            frames[cur]["rows"].append((int(s[1]), tuple(int(t) for t in s[3:7]), int(s[8]),
                                        [int(t) for t in s[10:]]))
    return off, case, frames


def test_hand_worked_batch():
    rng, vox, pts, _ = read_worked_example()
    off, (K, M), frames = read_batch_example()
    B = len(off) - 1
    ev = np.zeros((B, M, K, 4), np.float32)
    ec = np.zeros((B, M, 4), np.int32)
    en = np.zeros((B, M), np.int32)
    eV = np.zeros(B, np.int32)
    for b, f in frames.items():
        eV[b] = f["V"]
        for r, c, n, idx in f["rows"]:
            ec[b, r], en[b, r] = c, n
            for p, i in enumerate(idx):
                ev.view(np.uint32)[b, r, p] = pts.view(np.uint32)[i]
    st, v, c, n, V = oracle.voxelize_batch(pts, off, rng, vox, K, M)
    assert st == 0 and np.array_equal(V, eV)
    assert same_bits(c, ec), first_difference(c, ec)
    assert same_bits(n, en) and same_bits(v, ev)
    v2, c2, n2, V2 = oracle.voxelize_batch_numpy(pts, off, rng, vox, K, M)
    assert np.array_equal(V2, eV) and same_bits(c2, ec) and same_bits(n2, en) and same_bits(v2, ev)


@pytest.mark.parametrize("name", ["tiny", "kitti"])
def test_one_frame_is_the_single_cloud(name):
    pts, P = synth.make(name)
    r, v, K, M = P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels
    st, sv, sc, sn, sV = oracle.voxelize(pts, r, v, K, M)
    bst, bv, bc, bn, bV = oracle.voxelize_batch(pts, [0, pts.shape[0]], r, v, K, M)
    assert st == bst == 0 and bV[0] == sV
    assert same_bits(bv[0], sv) and same_bits(bn[0], sn) and same_bits(bc[0, :, 1:], sc)
    assert np.all(bc[0, :, 0] == 0)


@pytest.mark.parametrize("three_d", [False, True])
def test_random_tiny_batches_two_ways(three_d):
    rng = np.random.Generator(np.random.PCG64(91 + three_d))
    done = 0
    for _ in range(120):
        pts, off, r, v, K, M = random_tiny_batch(rng, gz_max=4 if three_d else 1)
        st, a, c, n, V = oracle.voxelize_batch(pts, off, r, v, K, M, three_d=three_d)
        assert st == 0
        a2, c2, n2, V2 = oracle.voxelize_batch_numpy(pts, off, r, v, K, M, three_d=three_d)
        assert np.array_equal(V, V2)
        assert same_bits(c, c2), first_difference(c, c2)
        assert same_bits(n, n2) and same_bits(a, a2)
        done += int(V.sum() > 0)
    assert done > 60
