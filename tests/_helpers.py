"""Shared test helpers: golden-file readers, exact arithmetic, invariants.

None of this is on the product path.  The exact-rational binary32 rounding
below is an independent derivation tool for the golden tables (it does not
call the oracle or the CUDA library).
"""

from __future__ import annotations

import math
import os
import struct
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _strip(line: str) -> str:
    return line.split("#", 1)[0].strip()


def read_edge_points():
    """[(bits[4], expected)], expected = None (dropped) or (cx, cy, cz)."""
    out = []
    with open(os.path.join(GOLDEN, "edge_points.txt")) as f:
        for line in f:
            s = _strip(line)
            if not s:
                continue
            tok = s.split()
            bits = [int(t, 16) for t in tok[:4]]
            exp = None if tok[4] == "drop" else tuple(int(t) for t in tok[4:7])
            out.append((bits, exp))
    return out


def read_division_points():
    out = []
    with open(os.path.join(GOLDEN, "division_points.txt")) as f:
        for line in f:
            s = _strip(line)
            if s:
                b, cx = s.split()
                out.append((int(b, 16), int(cx)))
    return out


def read_worked_example(name: str = "worked_example.txt"):
    """(range, voxel, points[N,4] float32, cases) from a worked-example file."""
    rng = vox = None
    pts = []
    cases = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            s = _strip(line)
            if not s:
                continue
            tok = s.split()
            if tok[0] == "range":
                rng = tuple(float(t) for t in tok[1:7])
            elif tok[0] == "voxel":
                vox = tuple(float(t) for t in tok[1:4])
            elif tok[0] == "point":
                assert int(tok[1]) == len(pts)
                pts.append([float(t) for t in tok[2:6]])
            elif tok[0] == "case":
                kv = dict(t.split("=") for t in tok[1:])
                cases.append({"max_points": int(kv["max_points"]), "max_voxels": int(kv["max_voxels"]),
                              "V": int(kv["V"]), "pillars": []})
            elif tok[0] == "pillar":
                r = int(tok[1])
                coords = tuple(int(t) for t in tok[3:6])
                count = int(tok[7])
                points = [int(t) for t in tok[9:]]
                assert len(points) == count
                cases[-1]["pillars"].append((r, coords, count, points))
    return rng, vox, np.array(pts, dtype=np.float32), cases


def worked_expected(points, case):
    """Expected padded outputs of one worked-example case."""
    K, M = case["max_points"], case["max_voxels"]
    vox = np.zeros((M, K, 4), dtype=np.float32)
    coords = np.zeros((M, 3), dtype=np.int32)
    counts = np.zeros((M,), dtype=np.int32)
    for r, c, n, pidx in case["pillars"]:
        coords[r] = c
        counts[r] = n
        for p, i in enumerate(pidx):
            vox.view(np.uint32)[r, p] = points.view(np.uint32)[i]
    return vox, coords, counts, case["V"]


# --------------------------------------------------------------------------
# Exact binary32 arithmetic on rationals (derivation of the golden tables).
# --------------------------------------------------------------------------

def f32_of_bits(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b & 0xFFFFFFFF))[0]


def bits_of_f32(x) -> int:
    return struct.unpack("<I", struct.pack("<f", float(np.float32(x))))[0]


def rn32(q: Fraction) -> Fraction:
    """Round a rational to the nearest binary32 value, ties to even."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)  # subnormals share the 2^-149 spacing
    ulp = Fraction(2) ** (e - 23)
    m = a / ulp
    fl = math.floor(m)
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * ulp


def exact_cell(coord_bits: int, lo: float, v: float, cells: int):
    """floor(rn(rn(c - lo) / v)) if inside [0, cells), else None."""
    if (coord_bits & 0x7F800000) == 0x7F800000:
        return None
    c = Fraction(f32_of_bits(coord_bits))
    d = rn32(c - Fraction(float(np.float32(lo))))
    q = rn32(d / Fraction(float(np.float32(v))))
    f = math.floor(q)
    return f if 0 <= f < cells else None


# --------------------------------------------------------------------------
# Random tiny clouds for the brute-force comparison.
# --------------------------------------------------------------------------

def _tiny_params(rng: np.random.Generator, gz_max: int):
    g = [int(rng.integers(1, 7)), int(rng.integers(1, 7)), int(rng.integers(1, gz_max + 1))]
    v = [float(np.float32(rng.choice([0.25, 0.5, 1.0, 0.16, 0.1, 0.3]))) for _ in range(2)]
    v.append(float(np.float32(rng.choice([1.0, 2.0, 4.0] if gz_max == 1 else [0.25, 0.5, 0.3, 1.0]))))
    lo = [float(np.float32(rng.uniform(-5, 5))), float(np.float32(rng.uniform(-5, 5))),
          float(np.float32(rng.uniform(-3, 0)))]
    hi = [float(np.float32(lo[a] + g[a] * v[a])) for a in range(3)]
    return g, v, lo, hi


def _tiny_points(rng: np.random.Generator, n: int, g, v, lo, hi) -> np.ndarray:
    pts = np.zeros((n, 4), dtype=np.float32)
    hot = [[lo[a] + (rng.integers(0, g[a]) + 0.5) * v[a] for a in range(3)] for _ in range(2)]
    for i in range(n):
        kind = rng.random()
        p = [0.0, 0.0, 0.0, float(rng.random())]
        if kind < 0.45:
            for a in range(3):
                p[a] = rng.uniform(lo[a] - 0.6 * v[a], hi[a] + 0.6 * v[a])
        elif kind < 0.62:  # on a cell boundary (computed in float32)
            for a in range(3):
                k = int(rng.integers(-1, g[a] + 2))
                p[a] = float(np.float32(np.float32(lo[a]) + np.float32(k) * np.float32(v[a])))
        elif kind < 0.72 and i > 0:  # duplicate of an earlier point
            p = [float(x) for x in pts[int(rng.integers(0, i))]]
        elif kind < 0.77:  # non-finite coordinate
            for a in range(3):
                p[a] = rng.uniform(lo[a], hi[a])
            p[int(rng.integers(0, 3))] = float(rng.choice([np.nan, np.inf, -np.inf]))
        elif kind < 0.82:  # exactly on the origin, one ulp either side, -0.0
            for a in range(3):
                p[a] = rng.uniform(lo[a], hi[a])
            a = int(rng.integers(0, 2))
            l32 = np.float32(lo[a])
            p[a] = float(rng.choice([l32, np.nextafter(l32, np.float32(-1e30)),
                                     np.nextafter(l32, np.float32(1e30))]))
            if lo[a] == 0.0 and rng.random() < 0.5:
                p[a] = -0.0
        else:  # a hot pillar, so the point cap binds
            h = hot[int(rng.integers(0, 2))]
            for a in range(3):
                p[a] = h[a] + rng.uniform(-0.3, 0.3) * v[a]
        pts[i] = np.array(p, dtype=np.float32)
    return pts


def random_tiny_case(rng: np.random.Generator, gz_max: int = 1):
    """A tiny cloud with both caps likely to bind; gz_max > 1 draws a z extent
    of up to gz_max cells (true 3-D voxels)."""
    g, v, lo, hi = _tiny_params(rng, gz_max)
    n = int(rng.integers(0, 260))
    pts = _tiny_points(rng, n, g, v, lo, hi)
    return pts, tuple(lo + hi), tuple(v), int(rng.integers(1, 5)), int(rng.integers(1, 10))


def random_tiny_batch(rng: np.random.Generator, gz_max: int = 1, max_frames: int = 6):
    """A batch of tiny frames on one grid: (points, frame offsets, range, voxel, K, M).
    Frames may be empty."""
    g, v, lo, hi = _tiny_params(rng, gz_max)
    B = int(rng.integers(1, max_frames + 1))
    frames = [_tiny_points(rng, int(rng.integers(0, 120)), g, v, lo, hi) for _ in range(B)]
    off = np.concatenate([[0], np.cumsum([f.shape[0] for f in frames])]).astype(np.int64)
    pts = np.concatenate(frames) if off[-1] else np.zeros((0, 4), dtype=np.float32)
    return pts, off, tuple(lo + hi), tuple(v), int(rng.integers(1, 5)), int(rng.integers(1, 10))


# --------------------------------------------------------------------------
# Output comparison and invariants.
# --------------------------------------------------------------------------

def same_bits(a: np.ndarray, b: np.ndarray) -> bool:
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    return a.shape == b.shape and a.tobytes() == b.tobytes()


def first_difference(a: np.ndarray, b: np.ndarray) -> str:
    av = np.ascontiguousarray(a).view(np.uint32 if a.dtype == np.float32 else a.dtype)
    bv = np.ascontiguousarray(b).view(np.uint32 if b.dtype == np.float32 else b.dtype)
    if av.shape != bv.shape:
        return f"shape {av.shape} vs {bv.shape}"
    d = np.argwhere(av != bv)
    if d.size == 0:
        return "equal"
    idx = tuple(d[0])
    return f"{d.shape[0]} differing elements, first at {idx}: {av[idx]} vs {bv[idx]}"


def check_invariants(points, pc_range, voxel_size, max_points, max_voxels, vox, coords, counts, V,
                     valid_mask, keys, grid_xy):
    """Properties every correct result has, at any size.

    ``valid_mask``/``keys`` come from an independent binning (NumPy float32).
    """
    gx, gy = grid_xy
    K, M = max_points, max_voxels
    distinct, first_idx, n_per = np.unique(keys[valid_mask], return_index=True, return_counts=True)[0:3]
    assert V == min(distinct.size, M), (V, distinct.size, M)
    assert vox.shape == (M, K, 4) and coords.shape == (M, 3) and counts.shape == (M,)
    # Kept pillars: coordinates unique, inside the grid, z = 0.
    c = coords[:V]
    assert np.all(c[:, 0] == 0)
    assert np.all((c[:, 1] >= 0) & (c[:, 1] < gy) & (c[:, 2] >= 0) & (c[:, 2] < gx))
    kk = c[:, 1].astype(np.int64) * gx + c[:, 2]
    assert np.unique(kk).size == V
    # Counts: min(points in pillar, K), at least 1.
    lookup = dict(zip(distinct.tolist(), n_per.tolist()))
    exp = np.array([min(lookup[int(k)], K) for k in kk], dtype=np.int64)
    assert np.array_equal(counts[:V].astype(np.int64), exp)
    # Padding is zero bits.
    vb = vox.view(np.uint32)
    assert not vb[V:].any() and not coords[V:].any() and not counts[V:].any()
    filled = np.arange(K)[None, :] < counts[:V, None]
    assert not vb[:V][~filled].any()
    # Every filled row is bitwise a row of the input whose pillar is that pillar.
    pb = np.ascontiguousarray(points).view(np.uint32).reshape(-1, 4)
    rows = vb[:V][filled]
    rows_key = np.repeat(kk, counts[:V])
    in_rows = {tuple(r): None for r in pb[valid_mask]}
    for r in rows[:: max(1, rows.shape[0] // 2000)]:
        assert tuple(r) in in_rows
    return rows_key


def check_order_with_index_intensity(points_idx, vox, counts, V, valid_mask, keys):
    """With intensity = float(point index), check the canonical order.

    Points inside a pillar ascend; each pillar's first point is its lowest
    valid index; pillars ascend by first point; no kept point has a larger
    index than a dropped point of the same pillar.
    """
    idx = vox[:V, :, 3]
    first = idx[:, 0]
    assert np.all(np.diff(first) > 0)
    for r in range(0, V, max(1, V // 500)):
        n = counts[r]
        row = idx[r, :n]
        assert np.all(np.diff(row) > 0)
    # Lowest valid index of each pillar.
    vi = np.flatnonzero(valid_mask)
    distinct, fpos = np.unique(keys[vi], return_index=True)
    firsts = np.sort(vi[fpos])[:V]
    assert np.array_equal(first.astype(np.int64), firsts)
