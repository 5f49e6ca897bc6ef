"""Pins of the order-insensitive checker used for the unordered mode.

The checker (oracle.check_unordered) restates the page's own comparison
("Results": sort by the (z, y, x) key, then compare the pillar sets and the
per-pillar counts) and adds validity checks for what a cap leaves open.  It
must accept every valid unordered result -- the canonical oracle output, any
permutation of its rows and of the points inside a row, and any other choice
of points or pillars where a cap binds -- and reject each planted mistake.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle
from lidar_point_cloud_gb300 import synth


def _case(name, K=None, M=None):
    pts, P = synth.make(name)
    K = K or P.max_points
    M = M or P.max_voxels
    st, v, c, n, V = oracle.voxelize(pts, P.point_cloud_range, P.voxel_size, K, M)
    assert st == 0
    return pts, P, K, M, v, c, n, V


def _check(pts, P, K, M, v, c, n, V):
    return oracle.check_unordered(pts, P.point_cloud_range, P.voxel_size, K, M, v, c, n, V)


def _shuffled(v, c, n, V, seed):
    rng = np.random.default_rng(seed)
    perm = rng.permutation(V)
    v2, c2, n2 = v.copy(), c.copy(), n.copy()
    v2[:V], c2[:V], n2[:V] = v[perm], c[perm], n[perm]
    for r in range(V):
        k = int(n2[r])
        v2[r, :k] = v2[r, :k][rng.permutation(k)]
    return v2, c2, n2


@pytest.mark.parametrize("name,K,M", [("tiny", None, None), ("kitti", None, None), ("kitti", 5, 500),
                                      ("uniform_25000", None, None)])
def test_accepts_canonical_and_permuted_results(name, K, M):
    pts, P, K, M, v, c, n, V = _case(name, K, M)
    assert _check(pts, P, K, M, v, c, n, V) == []
    assert _check(pts, P, K, M, *_shuffled(v, c, n, V, 1), V) == []


def test_accepts_another_choice_where_the_caps_bind():
    pts, P, K, M, v, c, n, V = _case("kitti", 4, 300)
    ok, cx, cy, cz, g = oracle.cells_numpy(pts, P.point_cloud_range, P.voxel_size)
    key = cy * g[0] + cx
    # Another point of a full pillar in place of one of its kept points.
    rkey = c[:V, 1].astype(np.int64) * g[0] + c[:V, 2]
    for r in range(V):
        members = np.flatnonzero(ok & (key == rkey[r]))
        if members.size > K:
            v2 = v.copy()
            v2[r, 0] = pts[members[K]]  # the first point past the cap
            assert _check(pts, P, K, M, v2, c, n, V) == []
            break
    else:
        pytest.fail("no full pillar")
    # A dropped pillar in place of a kept one (budget binds), with its own points.
    uniq = np.unique(key[ok])
    dropped = np.setdiff1d(uniq, rkey)
    d = int(dropped[0])
    members = np.flatnonzero(ok & (key == d))[:K]
    v2, c2, n2 = v.copy(), c.copy(), n.copy()
    v2[0] = 0
    v2[0, :members.size] = pts[members]
    c2[0] = (0, d // g[0], d % g[0])
    n2[0] = members.size
    assert _check(pts, P, K, M, v2, c2, n2, V) == []


def test_rejects_planted_mistakes():
    pts, P, K, M, v, c, n, V = _case("kitti")
    full = int(np.flatnonzero(n[:V] >= 3)[0])  # a pillar with at least three points
    small = int(np.flatnonzero((n[:V] >= 2) & (n[:V] < K))[0])
    mistakes = {}
    v2 = v.copy(); v2[0, 0], v2[1, 0] = v[1, 0].copy(), v[0, 0].copy()
    mistakes["points swapped between pillars"] = (v2, c, n, V)
    v2 = v.copy(); v2[small, 1] = v[small, 0]
    mistakes["a point stored twice"] = (v2, c, n, V)
    n2 = n.copy(); n2[full] -= 1
    v2 = v.copy(); v2[full, n2[full]] = 0
    mistakes["a point missing"] = (v2, c, n2, V)
    c2 = c.copy(); c2[0] = c[1]
    mistakes["two rows, one pillar"] = (v, c2, n, V)
    c2 = c.copy(); c2[0, 0] = 1
    mistakes["coordinates outside the grid"] = (v, c2, n, V)
    v2 = v.copy(); v2[V - 1, K - 1, 3] = 1.0
    mistakes["nonzero padding"] = (v2, c, n, V)
    mistakes["V off by one"] = (v, c, n, V - 1)
    v2 = v.copy(); v2[small, 0, 0] = np.nextafter(v[small, 0, 0], np.float32(1e9))
    mistakes["one bit changed"] = (v2, c, n, V)
    for what, (vv, cc, nn, VV) in mistakes.items():
        assert _check(pts, P, K, M, vv, cc, nn, VV), what
