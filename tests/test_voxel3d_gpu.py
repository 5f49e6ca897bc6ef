"""GPU parity for true 3-D voxels (grid_z > 1), bit for bit against the oracle.

The z cell joins the voxel id and the coordinates (z, y, x); everything else
(binning rule, canonical order, caps, zero padding) is the pillar contract.
Covers the three 3-D workloads (hashed and direct tables), random tiny clouds
with up to five layers, forced table modes and the caps.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle
from _helpers import first_difference, random_tiny_case, same_bits

torch = pytest.importorskip("torch")
pv = pytest.importorskip("lidar_point_cloud_gb300")
from lidar_point_cloud_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pv.load()
    yield
    pv.release_workspace()


def assert_parity3d(pts, r, v, K, M, **opts):
    st, ov, oc, on, oV = oracle.voxelize3d(pts, r, v, K, M)
    assert st == 0
    t = torch.from_numpy(np.ascontiguousarray(pts, dtype=np.float32).reshape(-1, 4)).to(DEV)
    out = pv.alloc_outputs(K, M, DEV)
    for o in out:
        o.view(torch.int32).fill_(0x7FBADBAD)
    pv.voxelize_into(t, r, v, K, M, out, **opts)
    torch.cuda.synchronize()
    gv, gc, gn, num = (o.cpu().numpy() for o in out)
    assert int(num[0]) == oV, (int(num[0]), oV)
    assert same_bits(gc, oc), "coords: " + first_difference(gc, oc)
    assert same_bits(gn, on), "counts: " + first_difference(gn, on)
    assert same_bits(gv, ov), "voxels: " + first_difference(gv, ov)
    return oV


@pytest.mark.parametrize("name", synth.VOXEL3D_WORKLOADS)
def test_voxel3d_workload_parity(name):
    pts, P = synth.make(name)
    V = assert_parity3d(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)
    assert V > 1000


def test_voxel3d_table_modes():
    _, P = synth.make("kitti3d")
    assert pv.query_plan(122_880, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)["table_mode"] == "hashed"
    _, P = synth.make("dense3d")
    assert pv.query_plan(1_048_576, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)["table_mode"] == "direct"
    pts, P = synth.make("dense3d")
    assert_parity3d(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels, table_mode=2)


def test_voxel3d_random_tiny_clouds():
    rng = np.random.Generator(np.random.PCG64(303))
    for _ in range(40):
        pts, r, v, K, M = random_tiny_case(rng, gz_max=5)
        assert_parity3d(pts, r, v, K, M)


@pytest.mark.parametrize("K,M", [(1, 1), (1, 40000), (5, 700), (64, 3000)])
def test_voxel3d_caps(K, M):
    pts, P = synth.make("kitti3d")
    assert_parity3d(pts, P.point_cloud_range, P.voxel_size, K, M)


def test_voxel3d_one_layer_is_the_pillar_result():
    pts, P = synth.make("kitti")
    assert_parity3d(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)
