"""Seeded synthetic LiDAR clouds for the benchmark and the test suite.

This module only makes inputs.  It holds none of the voxelizer's arithmetic
(no binning, no grouping): it draws points and hands back ``[N, 4]`` float32
arrays (x, y, z, intensity) together with the voxelizer parameters each
workload is run with.  Both the CUDA library and the CPU oracle consume
exactly these arrays.

Workloads (shapes follow the page "Voxelize", ethan-howes.github.io/projects/
voxelize/: a 432 x 496 grid of 0.16 m pillars over [0, 69.12] x
[-39.68, 39.68] x [-3, 1], 32 points per pillar, a 16,000-pillar budget, and
uniform synthetic clouds of 25k-130k points, "Tab. 1" and "Fig. 3"):

* ``tiny``        4,096 uniform points plus 16 boundary points appended last.
* ``kitti``       122,880 returns of a synthetic 64-beam spinning sensor,
                  in sensor order (azimuth-major), 0.1 % NaN/Inf coordinates.
                  Stands in for the page's KITTI frames, which are not here.
* ``uniform_<n>`` n i.i.d. uniform points over the range, random order.
* ``dense``       1,048,576 returns of a 128-beam sensor over
                  [-51.2, 51.2]^2 x [-5, 3] with 0.1 m pillars.
* ``adversarial`` 4,194,304 points in random order: 70 % packed into 64
                  pillars, the rest spread over pillar ids that collide modulo
                  1,600,000 (8 x the pillar budget, the page's table size) and
                  modulo 2^21; 0.05 m pillars on a 2048 x 2048 grid.

Every random draw comes from NumPy's PCG64 with a fixed seed.  Geometry uses
only +, -, *, /, sqrt (correctly rounded everywhere) and ``math`` sin/cos on
short per-beam and per-column tables, so the arrays are the same on x86-64
and AArch64.
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, Tuple

import numpy as np

KITTI_RANGE = (0.0, -39.68, -3.0, 69.12, 39.68, 1.0)
KITTI_VOXEL = (0.16, 0.16, 4.0)
DENSE_RANGE = (-51.2, -51.2, -5.0, 51.2, 51.2, 3.0)
DENSE_VOXEL = (0.1, 0.1, 8.0)
ADV_VOXEL = (0.05, 0.05, 8.0)

UNIFORM_SIZES = (25_000, 50_000, 75_000, 100_000, 130_000)


@dataclass(frozen=True)
class Params:
    """Voxelizer arguments of one workload."""

    point_cloud_range: Tuple[float, float, float, float, float, float]
    voxel_size: Tuple[float, float, float]
    max_points: int
    max_voxels: int


KITTI_PARAMS = Params(KITTI_RANGE, KITTI_VOXEL, 32, 16_000)
DENSE_PARAMS = Params(DENSE_RANGE, DENSE_VOXEL, 32, 60_000)
ADV_PARAMS = Params(DENSE_RANGE, ADV_VOXEL, 32, 200_000)
# True 3-D voxels on the same frames: 0.25 m layers over the KITTI slab
# (432 x 496 x 16), a SECOND-style fine grid (0.05 x 0.05 x 0.1 m over
# [0, 70.4] x [-40, 40] x [-3, 1]: 1408 x 1600 x 40, hashed table), and the
# dense grid in 2 m layers (1024 x 1024 x 4, direct table).
KITTI3D_PARAMS = Params(KITTI_RANGE, (0.16, 0.16, 0.25), 32, 40_000)
SECOND_PARAMS = Params((0.0, -40.0, -3.0, 70.4, 40.0, 1.0), (0.05, 0.05, 0.1), 5, 40_000)
DENSE3D_PARAMS = Params(DENSE_RANGE, (0.1, 0.1, 2.0), 32, 60_000)
VOXEL3D_WORKLOADS = ("kitti3d", "second", "dense3d")


def _f32(bits: int) -> np.float32:
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


# Sixteen boundary points appended to the ``tiny`` cloud.  Each row is
# (x, y, z, intensity) as exact float32 bit patterns; the coordinates not
# under test sit well inside the KITTI-shaped range.  What each one should
# do is stated (and derived) in tests/golden/edge_points.txt.
_MID_X, _MID_Y, _MID_Z, _W = 0x41200000, 0x00000000, 0xBF800000, 0x3F000000  # 10, 0, -1, 0.5
EDGE_POINT_BITS = np.array(
    [
        [0x428A3D71, _MID_Y, _MID_Z, _W],      # x = 69.12 (x_max)
        [0x428A3D70, _MID_Y, _MID_Z, _W],      # x = 69.119995 (one ulp below)
        [0xBA83126F, _MID_Y, _MID_Z, _W],      # x = -0.001
        [0x80000001, _MID_Y, _MID_Z, _W],      # x = -1e-45 (negative subnormal)
        [0x80000000, _MID_Y, _MID_Z, _W],      # x = -0.0
        [_MID_X, 0xC21EB852, _MID_Z, _W],      # y = -39.68 (y_min)
        [_MID_X, 0x421EB851, _MID_Z, _W],      # y = 39.679996 (one ulp below y_max)
        [_MID_X, _MID_Y, 0xC0400000, _W],      # z = -3 (z_min)
        [_MID_X, _MID_Y, 0x3F7FFFFF, _W],      # z = 0.99999994
        [0x3E23D70A, _MID_Y, _MID_Z, _W],      # x = 0.16
        [0x3EA3D70A, _MID_Y, _MID_Z, _W],      # x = 0.32
        [0x3EF5C28F, _MID_Y, _MID_Z, _W],      # x = 0.48
        [0x7FC00000, _MID_Y, _MID_Z, _W],      # x = NaN
        [_MID_X, 0x7F800000, _MID_Z, _W],      # y = +Inf
        [_MID_X, _MID_Y, 0xFF800000, _W],      # z = -Inf
        [0x41A00000, 0x41200000, _MID_Z, 0x7FC00000],  # x = 20, y = 10, intensity = NaN
    ],
    dtype=np.uint32,
)


def edge_points() -> np.ndarray:
    """The sixteen boundary points as a [16, 4] float32 array (exact bits)."""
    return EDGE_POINT_BITS.copy().view(np.float32)


def uniform(n: int, seed: int, pc_range=KITTI_RANGE) -> np.ndarray:
    """``n`` i.i.d. points uniform over the range box, intensity U[0, 1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lo = np.array(pc_range[:3], dtype=np.float64)
    hi = np.array(pc_range[3:], dtype=np.float64)
    u = rng.random((n, 4))
    pts = np.empty((n, 4), dtype=np.float32)
    pts[:, :3] = (lo + (hi - lo) * u[:, :3]).astype(np.float32)
    pts[:, 3] = u[:, 3].astype(np.float32)
    return pts


def tiny(seed: int = 0) -> np.ndarray:
    """4,096 uniform points over the KITTI-shaped range + 16 boundary points."""
    return np.concatenate([uniform(4096, seed), edge_points()], axis=0)


def _sensor_frame(
    seed: int,
    n_points: int,
    n_beams: int,
    elev_deg: Tuple[float, float],
    height: float,
    n_clusters: int = 20,
    cluster_range: Tuple[float, float] = (5.0, 60.0),
    cluster_sigma: Tuple[float, float] = (0.3, 1.5),
    wall_range: Tuple[float, float] = (30.0, 80.0),
    bad_fraction: float = 0.001,
) -> np.ndarray:
    """Returns of a synthetic spinning multi-beam sensor, in sensor order.

    The sensor sits at the origin, the ground plane is z = -height.  Each
    ray returns from the nearest of: a spherical object cluster (20 of them,
    centres at ranges 5-60 m, radius 2 sigma with sigma in 0.3-1.5 m, plus
    2 cm Gaussian jitter), the ground, or a far vertical "wall" whose range
    is drawn per azimuth column in 30-80 m.  A return is kept with a
    probability that falls with range, which makes far rings sparser than the
    geometry alone would; the frame is then trimmed or topped up at random to
    exactly ``n_points`` returns, keeping sensor order and the full 360
    degrees.  Intensity is U[0, 1).  A fraction ``bad_fraction`` of points
    gets NaN, +Inf or -Inf in one of x, y, z.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    n_cols_nominal = n_points // n_beams
    n_cols = (n_cols_nominal * 5) // 4  # extra columns, thinned by the keep draw
    # Per-column azimuth (sorted: the head spins), per-beam elevation.
    az = np.sort(rng.random(n_cols)) * (2.0 * math.pi)
    cos_az = np.array([math.cos(a) for a in az])
    sin_az = np.array([math.sin(a) for a in az])
    el = np.linspace(math.radians(elev_deg[0]), math.radians(elev_deg[1]), n_beams)
    cos_el = np.array([math.cos(e) for e in el])
    sin_el = np.array([math.sin(e) for e in el])
    # Ray directions [n_cols, n_beams, 3], azimuth-major.
    dx = cos_az[:, None] * cos_el[None, :]
    dy = sin_az[:, None] * cos_el[None, :]
    dz = np.broadcast_to(sin_el[None, :], dx.shape)

    far = 1.0e9
    # Far wall: a vertical cylinder at a per-column horizontal range.
    wall = wall_range[0] + (wall_range[1] - wall_range[0]) * rng.random(n_cols)
    t_wall = wall[:, None] / cos_el[None, :]
    # Ground plane z = -height, hit by downward rays only.
    with np.errstate(divide="ignore"):
        t_ground = np.where(dz < 0.0, height / np.maximum(-dz, 1e-300), far)
    t = np.minimum(t_wall, t_ground)
    # Spherical object clusters.
    c_rng = rng.random((n_clusters, 4))
    c_range = cluster_range[0] + (cluster_range[1] - cluster_range[0]) * c_rng[:, 0]
    c_az = c_rng[:, 1] * (2.0 * math.pi)
    c_sigma = cluster_sigma[0] + (cluster_sigma[1] - cluster_sigma[0]) * c_rng[:, 2]
    c_z = -height + c_sigma * 2.0 * c_rng[:, 3]
    for k in range(n_clusters):
        cx = c_range[k] * math.cos(c_az[k])
        cy = c_range[k] * math.sin(c_az[k])
        rad = 2.0 * c_sigma[k]
        # |o + t d - c|^2 = rad^2 with o = 0 and |d| = 1.
        b = dx * cx + dy * cy + dz * c_z[k]
        cc = cx * cx + cy * cy + c_z[k] * c_z[k] - rad * rad
        disc = b * b - cc
        hit = disc > 0.0
        t_hit = np.where(hit, b - np.sqrt(np.where(hit, disc, 0.0)), far)
        t_hit = np.where(t_hit > 0.0, t_hit, far)
        t = np.minimum(t, t_hit)
    jitter = 0.02 * rng.standard_normal((n_cols, n_beams, 3))
    xyz = np.stack([dx * t, dy * t, dz * t], axis=-1) + jitter
    xyz = xyz.reshape(-1, 3)
    rng_h = np.sqrt(xyz[:, 0] * xyz[:, 0] + xyz[:, 1] * xyz[:, 1])
    # Range-dependent keep probability.
    p_keep = np.clip(1.05 - rng_h / 90.0, 0.25, 1.0)
    keep = rng.random(p_keep.shape[0]) < p_keep
    n_kept = int(keep.sum())
    if n_kept > n_points:
        kept_idx = np.flatnonzero(keep)
        drop = rng.choice(kept_idx, size=n_kept - n_points, replace=False)
        keep[drop] = False
    elif n_kept < n_points:
        spare = np.flatnonzero(~keep)
        add = rng.choice(spare, size=n_points - n_kept, replace=False)
        keep[add] = True
    xyz = xyz[keep]
    assert xyz.shape[0] == n_points
    pts = np.empty((n_points, 4), dtype=np.float32)
    pts[:, :3] = xyz.astype(np.float32)
    pts[:, 3] = rng.random(n_points).astype(np.float32)
    n_bad = int(round(bad_fraction * n_points))
    if n_bad:
        bad = rng.choice(n_points, size=n_bad, replace=False)
        field = rng.integers(0, 3, size=n_bad)
        kind = rng.integers(0, 3, size=n_bad)
        vals = np.array([np.nan, np.inf, -np.inf], dtype=np.float32)
        pts[bad, field] = vals[kind]
    return pts


def kitti(seed: int = 1) -> np.ndarray:
    """122,880 returns of a 64-beam sensor (elevation -24.8..+2 deg, 1.73 m)."""
    return _sensor_frame(seed, 122_880, 64, (-24.8, 2.0), 1.73)


def dense(seed: int = 7) -> np.ndarray:
    """1,048,576 returns of a 128-beam sensor (elevation -25..+15 deg, 1.8 m)."""
    return _sensor_frame(seed, 1_048_576, 128, (-25.0, 15.0), 1.8)


ADV_TABLE = 1_600_000  # 8 x the 200,000-pillar budget: the page's table size
ADV_POW2 = 1 << 21


def adversarial_ids(seed: int, grid_cells: int = 2048 * 2048, n_ids: int = 500_000) -> np.ndarray:
    """Distinct pillar ids built to collide modulo ADV_TABLE and modulo 2^21.

    Runs of 64 consecutive residues are drawn; half the runs contribute the
    ids r, r + T, r + 2T (T = 1,600,000), the other half r and r + 2^21.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    ids = []
    total = 0
    turn = 0
    seen = set()
    while total < n_ids:
        if turn % 2 == 0:
            start = int(rng.integers(0, grid_cells - 2 * ADV_TABLE - 64))
            fam = [start + j + m * ADV_TABLE for j in range(64) for m in range(3)]
        else:
            start = int(rng.integers(0, grid_cells - ADV_POW2 - 64))
            fam = [start + j + m * ADV_POW2 for j in range(64) for m in range(2)]
        turn += 1
        new = [f for f in fam if f not in seen]
        seen.update(new)
        ids.extend(new)
        total += len(new)
    return np.array(ids[:n_ids], dtype=np.int64)


def adversarial(seed: int = 8) -> np.ndarray:
    """4,194,304 points: 70 % in 64 hot pillars, 30 % on colliding ids."""
    n = 4_194_304
    n_hot = 2_936_013
    n_spread = n - n_hot
    gx = gy = 2048
    vx = 0.05
    lo_x, lo_y, lo_z, hi_x, hi_y, hi_z = DENSE_RANGE
    rng = np.random.Generator(np.random.PCG64(seed))
    hot = rng.choice(gx * gy, size=64, replace=False)
    spread_ids = adversarial_ids(seed + 1000)
    hot_of_point = hot[rng.integers(0, 64, size=n_hot)]
    spread_of_point = spread_ids[rng.integers(0, spread_ids.shape[0], size=n_spread)]
    ids = np.concatenate([hot_of_point, spread_of_point])
    u = rng.random((n, 4))
    # A position inside the chosen pillar (pillar id = row * 2048 + column).
    col = (ids % gx).astype(np.float64)
    row = (ids // gx).astype(np.float64)
    pts = np.empty((n, 4), dtype=np.float32)
    pts[:, 0] = (lo_x + (col + 0.02 + 0.96 * u[:, 0]) * vx).astype(np.float32)
    pts[:, 1] = (lo_y + (row + 0.02 + 0.96 * u[:, 1]) * vx).astype(np.float32)
    pts[:, 2] = (lo_z + (hi_z - lo_z) * u[:, 2]).astype(np.float32)
    pts[:, 3] = u[:, 3].astype(np.float32)
    perm = rng.permutation(n)
    return np.ascontiguousarray(pts[perm])


def make(name: str) -> Tuple[np.ndarray, Params]:
    """(points, params) of a named workload."""
    if name == "tiny":
        return tiny(0), KITTI_PARAMS
    if name == "kitti":
        return kitti(1), KITTI_PARAMS
    if name.startswith("uniform_"):
        n = int(name.split("_", 1)[1])
        seed = 2 + UNIFORM_SIZES.index(n) if n in UNIFORM_SIZES else 100 + n % 997
        return uniform(n, seed), KITTI_PARAMS
    if name == "dense":
        return dense(7), DENSE_PARAMS
    if name == "adversarial":
        return adversarial(8), ADV_PARAMS
    if name == "kitti3d":
        return kitti(1), KITTI3D_PARAMS
    if name == "second":
        return kitti(1), SECOND_PARAMS
    if name == "dense3d":
        return dense(7), DENSE3D_PARAMS
    raise KeyError(name)


def make_batch(name: str, frames: int) -> Tuple[np.ndarray, np.ndarray, Params]:
    """(points, frame offsets [frames + 1], params): `frames` different frames of
    a named workload (the generator run with consecutive seeds), concatenated."""
    gens = {"kitti": (kitti, 1), "kitti3d": (kitti, 1), "second": (kitti, 1), "dense": (dense, 7),
            "dense3d": (dense, 7), "adversarial": (adversarial, 8), "tiny": (tiny, 0)}
    _, P = make(name)
    if name.startswith("uniform_"):
        n = int(name.split("_", 1)[1])
        parts = [uniform(n, 300 + 7 * b + n % 997) for b in range(frames)]
    else:
        gen, seed0 = gens[name]
        parts = [gen(seed0 + 1000 * b) if b else gen(seed0) for b in range(frames)]
    off = np.concatenate([[0], np.cumsum([p.shape[0] for p in parts])]).astype(np.int64)
    return np.concatenate(parts), off, P


FPS_POINTS = 65_536   # the RadiusFPS page's benchmark: N = 65,536 points,
FPS_SAMPLES = 4_096   # M = 4,096 samples


def fps_cloud(seed: int = 1, n: int = FPS_POINTS) -> np.ndarray:
    """A LiDAR-shaped cloud for farthest point sampling: the first n returns
    of the KITTI-shaped frame of this seed whose x, y, z are finite."""
    pts = kitti(seed)
    ok = np.all(np.isfinite(pts[:, :3]), axis=1)
    return np.ascontiguousarray(pts[ok][:n])


WORKLOADS: Dict[str, str] = {
    "tiny": "4,096 uniform + 16 boundary points, 432x496 grid, 16,000 pillars",
    "kitti": "122,880-return 64-beam frame, 432x496 grid, 16,000 pillars",
    **{f"uniform_{n}": f"{n:,} uniform points, 432x496 grid, 16,000 pillars" for n in UNIFORM_SIZES},
    "dense": "1,048,576-return 128-beam frame, 1024x1024 grid, 60,000 pillars",
    "adversarial": "4,194,304 points, 64 hot pillars + colliding ids, 2048x2048 grid, 200,000 pillars",
    "kitti3d": "122,880-return 64-beam frame, 432x496x16 voxels (0.25 m layers), 40,000 voxels",
    "second": "122,880-return 64-beam frame, 1408x1600x40 voxels (0.05x0.05x0.1 m), 5 points, 40,000 voxels",
    "dense3d": "1,048,576-return 128-beam frame, 1024x1024x4 voxels (2 m layers), 60,000 voxels",
    "lidar65k": "farthest point sampling: 65,536 returns of the 64-beam frame, 4,096 samples",
}
