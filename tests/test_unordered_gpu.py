"""GPU checks of the unordered mode (the page's own contract).

Each result is checked with oracle.check_unordered: V, the pillar set, the
counts and, for pillars under the cap, the exact point sets must match the
oracle; where a cap binds, any valid choice passes.  Also: 3-D grids, both
table modes, calls alternating with the canonical mode on one workspace
(the shared table must come back clean), and the device error paths.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle
from _helpers import random_tiny_case, same_bits

torch = pytest.importorskip("torch")
pv = pytest.importorskip("lidar_point_cloud_gb300")
from lidar_point_cloud_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
KR, KV = synth.KITTI_RANGE, synth.KITTI_VOXEL


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pv.load()
    yield
    pv.release_workspace()


def run(pts, r, v, K, M, **opts):
    t = torch.from_numpy(np.ascontiguousarray(pts, dtype=np.float32).reshape(-1, 4)).to(DEV)
    out = pv.alloc_outputs(K, M, DEV)
    for o in out:
        o.view(torch.int32).fill_(0x7FBADBAD)
    pv.voxelize_into(t, r, v, K, M, out, **opts)
    torch.cuda.synchronize()
    vox, coords, counts, num = (o.cpu().numpy() for o in out)
    return vox, coords, counts, int(num[0])


def assert_valid(pts, r, v, K, M, three_d=False, **opts):
    vox, coords, counts, V = run(pts, r, v, K, M, unordered=True, **opts)
    fails = oracle.check_unordered(pts, r, v, K, M, vox, coords, counts, V, three_d=three_d)
    assert fails == [], fails[:3]
    return V


ALL = ["tiny", "kitti", *[f"uniform_{n}" for n in synth.UNIFORM_SIZES], "dense", "adversarial"]


@pytest.mark.parametrize("name", ALL)
def test_unordered_workloads(name):
    pts, P = synth.make(name)
    assert assert_valid(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels) > 0


@pytest.mark.parametrize("name", synth.VOXEL3D_WORKLOADS)
def test_unordered_voxel3d(name):
    pts, P = synth.make(name)
    assert_valid(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels, three_d=True)


@pytest.mark.parametrize("K,M", [(1, 1), (1, 16000), (32, 1), (5, 500), (33, 2000), (64, 3000)])
def test_unordered_caps(K, M):
    pts, P = synth.make("kitti")
    assert_valid(pts, P.point_cloud_range, P.voxel_size, K, M)


def test_unordered_random_tiny_clouds():
    rng = np.random.Generator(np.random.PCG64(404))
    for _ in range(40):
        pts, r, v, K, M = random_tiny_case(rng, gz_max=3)
        assert_valid(pts, r, v, K, M, three_d=True)


def test_unordered_hashed_table():
    pts, P = synth.make("dense")
    assert_valid(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels, table_mode=2)


def test_unordered_under_the_caps_equals_the_canonical_sets():
    # No cap binds: the result is the canonical one up to the order of rows and points.
    pts = synth.uniform(20_000, 41)
    st, ov, oc, on, oV = oracle.voxelize(pts, KR, KV, 1024, 60_000)
    assert st == 0 and on.max() < 1024 and oV < 60_000
    gv, gc, gn, gV = run(pts, KR, KV, 1024, 60_000, unordered=True)
    assert gV == oV
    okey = oc[:oV, 1].astype(np.int64) * 432 + oc[:oV, 2]
    gkey = gc[:gV, 1].astype(np.int64) * 432 + gc[:gV, 2]
    oo, go = np.argsort(okey), np.argsort(gkey)
    assert np.array_equal(okey[oo], gkey[go]) and np.array_equal(on[:oV][oo], gn[:gV][go])
    for a, b in zip(oo[:500], go[:500]):
        n = int(on[a])
        ra = np.sort(ov[a, :n].view(np.uint32).view([("x", "<u4"), ("y", "<u4"), ("z", "<u4"), ("w", "<u4")]), axis=0)
        rb = np.sort(gv[b, :n].view(np.uint32).view([("x", "<u4"), ("y", "<u4"), ("z", "<u4"), ("w", "<u4")]), axis=0)
        assert ra.tobytes() == rb.tobytes()


def test_alternating_with_the_canonical_mode():
    # Both modes share one workspace: each must leave the table clean for the other.
    for name in ["kitti", "dense", "kitti", "adversarial", "kitti"]:
        pts, P = synth.make(name)
        r, v, K, M = P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels
        assert_valid(pts, r, v, K, M)
        st, ov, oc, on, oV = oracle.voxelize(pts, r, v, K, M)
        gv, gc, gn, gV = run(pts, r, v, K, M)
        assert gV == oV and same_bits(gv, ov) and same_bits(gc, oc) and same_bits(gn, on)


def test_unordered_capacity_error_then_recovery():
    pts = synth.uniform(20_000, 12)
    assert run(pts, KR, KV, 32, 16_000, unordered=True, table_mode=2, table_log2=4)[3] == -5
    assert_valid(pts, KR, KV, 32, 16_000, table_mode=2)
    st, ov, oc, on, oV = oracle.voxelize(pts, KR, KV, 32, 16_000)
    gv, gc, gn, gV = run(pts, KR, KV, 32, 16_000)
    assert gV == oV and same_bits(gv, ov)


def test_unordered_wait_timeout_is_reported_and_recovered():
    pts, P = synth.make("kitti")
    r, v, K, M = P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels
    assert run(pts, r, v, K, M, unordered=True, test_stall_barrier=1)[3] == -6  # PV_ERR_TIMEOUT
    assert_valid(pts, r, v, K, M)
