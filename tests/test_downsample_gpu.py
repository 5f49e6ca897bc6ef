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


def test_downsample_voxels_straddling_a_plane():
    """Voxels that contain the planes x = 0, y = 0 and z = 0, their points
    in cancelling pairs, so a mean can be far smaller than the values summed.

    The 1-ulp bound of the other tests rests on the values of a voxel sharing
    one sign: summation errors are relative to the sum of the magnitudes, and
    for one sign that sum is the sum itself.  Here they are not, so this test
    takes the bound that holds whatever the signs: the kernel's float-float
    warp sums and double accumulation err by a few units of 2^-46 of the
    voxel's mean magnitude sum(|x|) / n, plus the final rounding (half an
    ulp of the mean).  It checks every centroid against the exact mean within
    2^-40 sum(|x|) / n plus one ulp, the integers exactly, and the one-ulp
    bound on the voxels whose values do share a sign (the intensities here).
    """
    rng = np.random.Generator(np.random.PCG64(4242))
    r, v = (-2.5, -2.5, -2.5, 2.5, 2.5, 2.5), (1.0, 1.0, 1.0)  # the middle cell [-0.5, 0.5)^3 holds 0
    chunks = []
    for vox in range(27):  # the 3 x 3 x 3 cells around the origin; the centre one straddles all three planes
        c = np.array([vox % 3, (vox // 3) % 3, vox // 9], np.float64) - 1.0
        n = 2 * int(rng.integers(4, 400))
        a = rng.uniform(0.0, 0.49, size=(n // 2, 3))
        tiny = rng.uniform(-1e-6, 1e-6, size=(n // 2, 3)) * (vox % 2)  # half the voxels exactly symmetric
        xyz = np.concatenate([c + a, c - a + tiny]).astype(np.float32)
        w = rng.random(n).astype(np.float32)
        chunks.append(np.concatenate([xyz, w[:, None]], axis=1))
    pts = np.concatenate(chunks).astype(np.float32)
    pts = pts[rng.permutation(pts.shape[0])]
    M = 64
    ex_cen, ex_coords, ex_counts, eV = oracle.downsample_exact(pts, r, v, M)
    t = torch.from_numpy(np.ascontiguousarray(pts)).to(DEV)
    out = pv.alloc_downsample_outputs(M, DEV)
    pv.downsample_into(t, r, v, M, out)
    torch.cuda.synchronize()
    gc, gco, gn, num = (o.cpu().numpy() for o in out)
    assert int(num[0]) == eV == 27
    assert same_bits(gco, ex_coords) and same_bits(gn, ex_counts)
    ok, cx, cy, cz, g = oracle.cells_numpy(pts, r, v)
    key = (cz * g[1] + cy) * g[0] + cx
    for row in range(eV):
        z, y, x = (int(q) for q in ex_coords[row])
        sel = ok & (key == (z * g[1] + y) * g[0] + x)
        mag = np.abs(pts[sel].astype(np.float64)).sum(axis=0) / sel.sum()
        ulp = np.spacing(np.abs(ex_cen[row]).astype(np.float32)).astype(np.float64)
        err = np.abs(gc[row].astype(np.float64) - ex_cen[row].astype(np.float64))
        assert np.all(err <= 2.0 ** -40 * mag + ulp), (row, err, mag, ulp)
    # The intensities (all of one sign) keep the one-ulp bound.
    assert oracle.ulp_distance32(gc[:eV, 3], ex_cen[:eV, 3]).max() <= 1
