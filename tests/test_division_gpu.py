"""Parity at the cell boundaries, where the kernel's binning decides by the
correctly rounded division.

The reading of "Voxelize" > "Binning a point" fixed here is one IEEE binary32
round-to-nearest subtraction and division per axis, then floorf (the page
builds with --use_fast_math and notes in "Results" that boundary points can
fall either way; the reading makes the result unique).  The kernel estimates
the quotient as RN(d * RN(1/v)) and takes the division itself only when the
estimate lies within q * 2^-22 of an integer, so every point near a cell
boundary runs through that filter and its fallback.

The sweep puts points at 0 and +-1 .. +-8 ulps around every cell boundary
lo + k * v (the decimal product rounded to binary32) of the KITTI-shaped,
dense and adversarial pillar grids, on x and on y, 120,326 points in all
(5,103 of them floor to another cell under a reciprocal multiply),
plus the points of tests/golden/division_points.txt.  They go through
pv_voxelize and pv_voxelize_batch and are compared with the oracle bit for
bit.  A CPU test checks that the sweep reaches the cases it is meant for:
points whose reciprocal-multiply floor differs from the division's.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle
from _helpers import first_difference, read_division_points, same_bits

torch = pytest.importorskip("torch")
pv = pytest.importorskip("lidar_point_cloud_gb300")
from lidar_point_cloud_gb300 import synth  # noqa: E402

DEV = "cuda:0"
ULPS = 8  # points at 0, +-1 .. +-ULPS ulps around each boundary

GRIDS = {
    "kitti": (synth.KITTI_RANGE, synth.KITTI_VOXEL),
    "dense": (synth.DENSE_RANGE, synth.DENSE_VOXEL),
    "adversarial": (synth.DENSE_RANGE, synth.ADV_VOXEL),
}


def boundary_values(lo: float, v: float, cells: int) -> np.ndarray:
    """binary32 values at and around lo + k * v for k = 0 .. cells."""
    k = np.arange(cells + 1, dtype=np.float64)
    b = (np.float64(np.float32(lo)) + k * np.float64(np.float32(v))).astype(np.float32)
    out = [b]
    up, down = b.copy(), b.copy()
    for _ in range(ULPS):
        up = np.nextafter(up, np.float32(np.inf))
        down = np.nextafter(down, np.float32(-np.inf))
        out += [up, down]
    return np.concatenate(out)


def sweep(name: str, seed: int) -> np.ndarray:
    """Points around every x boundary and every y boundary of one grid, the
    other coordinates at random cell centres, intensity the point's index;
    shuffled so that neighbours share no order."""
    (r, v) = GRIDS[name]
    g = oracle.grid_py(r, v)
    rng = np.random.default_rng(seed)
    bx = boundary_values(r[0], v[0], g[0])
    by = boundary_values(r[1], v[1], g[1])

    def centres(axis, n):
        c = rng.integers(0, g[axis], n)
        return (np.float64(r[axis]) + (c + 0.5) * np.float64(v[axis])).astype(np.float32)

    zc = np.float32(0.5 * (r[2] + r[5]))
    px = np.stack([bx, centres(1, bx.size), np.full(bx.size, zc, np.float32), np.zeros(bx.size, np.float32)], 1)
    py = np.stack([centres(0, by.size), by, np.full(by.size, zc, np.float32), np.zeros(by.size, np.float32)], 1)
    pts = np.concatenate([px, py]).astype(np.float32)
    pts = pts[rng.permutation(pts.shape[0])]
    pts[:, 3] = np.arange(pts.shape[0], dtype=np.float32)
    return np.ascontiguousarray(pts)


def golden_points() -> np.ndarray:
    pts = []
    for b, _ in read_division_points():
        x = np.array([b], dtype=np.uint32).view(np.float32)[0]
        pts.append([x, 0.0, -1.0, 0.5])
    return np.array(pts, dtype=np.float32)


def test_sweep_reaches_the_division_cases():
    """The sweep holds points where a reciprocal multiply floors to another
    cell than the correctly rounded division (numpy float32 arithmetic is
    IEEE binary32, round to nearest), on every grid."""
    total = 0
    for seed, name in enumerate(GRIDS):
        (r, v) = GRIDS[name]
        pts = sweep(name, seed)
        total += pts.shape[0]
        for axis in (0, 1):
            d = pts[:, axis] - np.float32(r[axis])
            q_div = d / np.float32(v[axis])
            q_rcp = d * (np.float32(1.0) / np.float32(v[axis]))
            assert np.count_nonzero(np.floor(q_div) != np.floor(q_rcp)) > 0, (name, axis)
    assert total >= 100_000


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(GRIDS))
def test_boundary_sweep_single_frame(name):
    (r, v) = GRIDS[name]
    pts = sweep(name, list(GRIDS).index(name))
    if name == "kitti":
        pts = np.concatenate([pts, golden_points()])
    K, M = 32, pts.shape[0]
    st, ov, oc, on, oV = oracle.voxelize(pts, r, v, K, M)
    assert st == 0
    t = torch.from_numpy(pts).to(DEV)
    out = pv.alloc_outputs(K, M, DEV)
    for o in out:
        o.view(torch.int32).fill_(0x7FBADBAD)
    pv.voxelize_into(t, r, v, K, M, out)
    torch.cuda.synchronize()
    gv, gc, gn, gV = (o.cpu().numpy() for o in out)
    assert int(gV[0]) == oV, (int(gV[0]), oV)
    assert same_bits(gc, oc), "coords: " + first_difference(gc, oc)
    assert same_bits(gn, on), "counts: " + first_difference(gn, on)
    assert same_bits(gv, ov), "voxels: " + first_difference(gv, ov)


@pytest.mark.gpu
def test_golden_division_points_cells():
    """The golden points land in the cells the table gives (the cell a
    reciprocal multiply would miss by one)."""
    pts = golden_points()
    r, v = GRIDS["kitti"]
    vox, coords, counts = pv.voxelize(torch.from_numpy(pts).to(DEV), r, v, 32, 16)
    got = sorted(int(x) for x in coords[:, 2].cpu().numpy())
    assert got == sorted(cx for _, cx in read_division_points())


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(GRIDS))
def test_boundary_sweep_batch(name):
    (r, v) = GRIDS[name]
    pts = sweep(name, 10 + list(GRIDS).index(name))
    n = pts.shape[0]
    off = np.array([0, n // 3, n // 3 + 1, (2 * n) // 3, n], dtype=np.int64)  # a one-point frame among them
    K, M = 32, n // 3 + 2
    st, ov, oc, on, oV = oracle.voxelize_batch(pts, off, r, v, K, M)
    assert st == 0
    t = torch.from_numpy(pts).to(DEV)
    B = len(off) - 1
    out = pv.alloc_batch_outputs(B, K, M, DEV)
    for o in out:
        o.view(torch.int32).fill_(0x7FBADBAD)
    pv.voxelize_batch_into(t, off, r, v, K, M, out)
    torch.cuda.synchronize()
    gv, gc, gn, gV = (o.cpu().numpy() for o in out)
    assert np.array_equal(gV, oV), (gV, oV)
    assert same_bits(gc, oc), "coords: " + first_difference(gc, oc)
    assert same_bits(gn, on), "counts: " + first_difference(gn, on)
    assert same_bits(gv, ov), "voxels: " + first_difference(gv, ov)
