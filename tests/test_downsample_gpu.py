"""GPU checks of voxel-grid centroid downsampling against the oracle.

Exact: V, the voxel order, coordinates, counts and the zero padding.  Centroid
values: within one float32 unit in the last place of the oracle's (both sum
in double; the GPU adds in another order, which can only move a mean that
sits next to a float32 rounding boundary, by one ulp), and bit-equal for
nearly all of them.
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


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pv.load()
    yield
    pv.release_workspace()


def check(pts, r, v, M):
    st, oc, oco, on, oV = oracle.downsample(pts, r, v, M)
    assert st == 0
    t = torch.from_numpy(np.ascontiguousarray(pts, dtype=np.float32).reshape(-1, 4)).to(DEV)
    out = pv.alloc_downsample_outputs(M, DEV)
    for o in out:
        o.view(torch.int32).fill_(0x7FBADBAD)
    pv.downsample_into(t, r, v, M, out)
    torch.cuda.synchronize()
    gc, gco, gn, num = (o.cpu().numpy() for o in out)
    assert int(num[0]) == oV
    assert same_bits(gco, oco) and same_bits(gn, on)
    assert np.all(gc[oV:].view(np.uint32) == 0)
    d = oracle.ulp_distance32(gc[:oV], oc[:oV])
    assert d.max(initial=0) <= 1, d.max()
    return oV, float((d == 0).mean()) if oV else 1.0


@pytest.mark.parametrize("name", ["tiny", "kitti", "kitti3d", "second", "dense3d", "adversarial"])
def test_downsample_workloads(name):
    pts, P = synth.make(name)
    V, exact = check(pts, P.point_cloud_range, P.voxel_size, 1 << 20)
    assert V > 0 and exact > 0.99


@pytest.mark.parametrize("hot", [64, 200])
def test_downsample_hot_voxels(hot):
    # Blocks with several tiles (here 14) learn hot voxels, those in 4 or more
    # warp groups of their first tile, into a shared table of 256 positions:
    # 64 voxels (16 points each a tile) all qualify; 200 (about 5 each) fill
    # the table to a high load.  2 M points in random order over `hot`
    # voxels of a pillar grid.
    rng = np.random.Generator(np.random.PCG64(1000 + hot))
    n = 2 * 1024 * 1024
    r, v = (-20.0, -20.0, -3.0, 20.0, 20.0, 1.0), (0.5, 0.5, 4.0)
    cells = rng.choice(80 * 80, size=hot, replace=False)
    c = cells[rng.integers(0, hot, size=n)]
    pts = np.empty((n, 4), np.float32)
    pts[:, 0] = (r[0] + ((c % 80) + 0.05 + 0.9 * rng.random(n)) * v[0]).astype(np.float32)
    pts[:, 1] = (r[1] + ((c // 80) + 0.05 + 0.9 * rng.random(n)) * v[1]).astype(np.float32)
    pts[:, 2] = (r[2] + 4.0 * rng.random(n)).astype(np.float32)
    pts[:, 3] = rng.random(n).astype(np.float32)
    V, exact = check(pts, r, v, 1000)
    assert V == hot and exact > 0.99


@pytest.mark.parametrize("M", [1, 100, 5000])
def test_downsample_budget(M):
    pts, P = synth.make("kitti3d")
    assert check(pts, P.point_cloud_range, P.voxel_size, M)[0] == M


def test_downsample_random_tiny():
    rng = np.random.Generator(np.random.PCG64(707))
    for _ in range(40):
        pts, r, v, K, M = random_tiny_case(rng, gz_max=4)
        check(pts, r, v, 3 * M)


def test_downsample_empty_and_single():
    _, P = synth.make("kitti3d")
    assert check(np.zeros((0, 4), np.float32), P.point_cloud_range, P.voxel_size, 10)[0] == 0
    one = np.array([[10.0, 0.0, -1.0, 0.5]], np.float32)
    assert check(one, P.point_cloud_range, P.voxel_size, 10)[0] == 1


def test_downsample_alternating_with_voxelize():
    pts, P = synth.make("kitti3d")
    r, v = P.point_cloud_range, P.voxel_size
    for _ in range(2):
        check(pts, r, v, 40_000)
        st, ov, oc, on, oV = oracle.voxelize3d(pts, r, v, 32, 40_000)
        g = pv.voxelize(torch.from_numpy(pts).to(DEV), r, v, 32, 40_000)
        assert g[0].shape[0] == oV and same_bits(g[0].cpu().numpy(), ov[:oV])


def test_downsample_python_api():
    pts, P = synth.make("dense3d")
    cen, coords, counts = pv.downsample(torch.from_numpy(pts).to(DEV), P.point_cloud_range, P.voxel_size)
    ok, *_ = oracle.cells_numpy(pts, P.point_cloud_range, P.voxel_size)
    assert int(counts.sum()) == int(ok.sum()) and cen.shape[0] == coords.shape[0] == counts.shape[0]
