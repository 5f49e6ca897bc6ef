"""CPU oracles for pillar voxelization.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this package; the product path must
never route through it.  It shares no code with the CUDA library.

Three independent restatements of one definition (the page "Voxelize",
ethan-howes.github.io/projects/voxelize/, sections "Implementation > Binning
a point", "Claiming a pillar and packing points", "Compaction", "The PyTorch
side" and "Results"):

* :func:`voxelize`            the sequential std::map pass in C++
                              (``pv_oracle.cpp``), the primary oracle;
* :func:`voxelize_numpy`      a vectorised NumPy restatement built on a stable
                              sort (``np.unique`` + ``argsort(kind="stable")``);
* :func:`voxelize_bruteforce` the O(N^2) definition in plain Python, for tiny
                              clouds: rank(i) = number of distinct pillars whose
                              first point precedes pillar(i)'s first point,
                              pos(i) = number of earlier points in pillar(i).

Canonical order (the page's hash-slot order is nondeterministic, "Results";
the deterministic reading used here): pillars in ascending order of their
lowest-index valid point, points inside a pillar in index order, the first
``max_points`` points and the first ``max_voxels`` pillars kept, everything
else zero.
"""

from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from typing import Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pv_oracle.cpp")
_LIB = os.path.join(_HERE, "libpv_oracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
ERR_INVALID = -1
ERR_UNSUPPORTED = -2

GXX_FLAGS = ["-O2", "-std=c++17", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared"]


def build(src: str = _SRC, out: str = _LIB, extra: Sequence[str] = ()) -> str:
    """Compile the C++ oracle into a shared library (plain g++)."""
    cmd = ["g++", *GXX_FLAGS, *extra, src, "-o", out]
    subprocess.run(cmd, check=True)
    return out


def _bind(lib):
    f = ctypes.POINTER(ctypes.c_float)
    i64 = ctypes.POINTER(ctypes.c_int64)
    i32 = ctypes.POINTER(ctypes.c_int32)
    lib.pv_oracle_grid.argtypes = [f, f, i64]
    lib.pv_oracle_grid.restype = ctypes.c_int
    lib.pv_oracle_bin_point.argtypes = [f, f, f, i64, i64]
    lib.pv_oracle_bin_point.restype = ctypes.c_int
    lib.pv_oracle_voxelize.argtypes = [
        f, ctypes.c_int64, f, f, ctypes.c_int, ctypes.c_int, f, i32, i32, i32,
    ]
    lib.pv_oracle_voxelize.restype = ctypes.c_int
    if hasattr(lib, "pv_oracle_voxelize3d"):  # absent from some planted-mistake builds
        lib.pv_oracle_grid3d.argtypes = [f, f, i64]
        lib.pv_oracle_grid3d.restype = ctypes.c_int
        lib.pv_oracle_voxelize3d.argtypes = lib.pv_oracle_voxelize.argtypes
        lib.pv_oracle_voxelize3d.restype = ctypes.c_int
    return lib


def load_path(path: str):
    """Load an already compiled oracle library (e.g. a test's mutant)."""
    return _bind(ctypes.CDLL(path))


def load():
    """Load the oracle library, compiling it first if it is missing or stale."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
                build()
            _lib = load_path(_LIB)
        return _lib


def _fptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _f32(seq) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(seq, dtype=np.float32))


def grid(pc_range, voxel_size, lib=None) -> Tuple[int, Tuple[int, int, int]]:
    """(status, (gx, gy, gz)) from the C++ oracle."""
    lib = lib or load()
    r, v = _f32(pc_range), _f32(voxel_size)
    g = np.zeros(3, dtype=np.int64)
    st = lib.pv_oracle_grid(_fptr(r), _fptr(v), g.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)))
    return st, tuple(int(x) for x in g)


def bin_point(p, pc_range, voxel_size, lib=None):
    """(cx, cy, cz) of one point, or None if it is dropped."""
    lib = lib or load()
    st, g = grid(pc_range, voxel_size, lib)
    assert st == OK, st
    pp, r, v = _f32(p), _f32(pc_range), _f32(voxel_size)
    gg = np.array(g, dtype=np.int64)
    cell = np.zeros(3, dtype=np.int64)
    ok = lib.pv_oracle_bin_point(
        _fptr(pp), _fptr(r), _fptr(v),
        gg.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        cell.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
    )
    return tuple(int(c) for c in cell) if ok else None


def grid3d(pc_range, voxel_size, lib=None) -> Tuple[int, Tuple[int, int, int]]:
    """(status, (gx, gy, gz)) for true 3-D voxels (any z extent)."""
    lib = lib or load()
    r, v = _f32(pc_range), _f32(voxel_size)
    g = np.zeros(3, dtype=np.int64)
    st = lib.pv_oracle_grid3d(_fptr(r), _fptr(v), g.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)))
    return st, tuple(int(x) for x in g)


def voxelize3d(points: np.ndarray, pc_range, voxel_size, max_points: int, max_voxels: int, lib=None):
    """The C++ oracle for true 3-D voxels: coordinates (z, y, x) of the voxel.
    Same return values as :func:`voxelize`."""
    return voxelize(points, pc_range, voxel_size, max_points, max_voxels, lib, three_d=True)


def voxelize(points: np.ndarray, pc_range, voxel_size, max_points: int, max_voxels: int, lib=None,
             three_d: bool = False):
    """The C++ oracle.  Returns (status, voxels, coords, counts, V).

    ``voxels`` is [max_voxels, max_points, 4] float32, ``coords`` [max_voxels, 3]
    int32, ``counts`` [max_voxels] int32; all padded with zeros past V.
    """
    lib = lib or load()
    pts = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 4)
    r, v = _f32(pc_range), _f32(voxel_size)
    vox = np.empty((max(max_voxels, 0), max(max_points, 0), 4), dtype=np.float32)
    coords = np.empty((max(max_voxels, 0), 3), dtype=np.int32)
    counts = np.empty((max(max_voxels, 0),), dtype=np.int32)
    num = np.zeros(1, dtype=np.int32)
    i32 = ctypes.POINTER(ctypes.c_int32)
    fn = lib.pv_oracle_voxelize3d if three_d else lib.pv_oracle_voxelize
    st = fn(
        _fptr(pts) if pts.size else None, pts.shape[0], _fptr(r), _fptr(v),
        int(max_points), int(max_voxels), _fptr(vox),
        coords.ctypes.data_as(i32), counts.ctypes.data_as(i32), num.ctypes.data_as(i32),
    )
    return st, vox, coords, counts, int(num[0])


# --------------------------------------------------------------------------
# NumPy restatement (stable sort), independent of the C++ pass.
# --------------------------------------------------------------------------

def grid_py(pc_range, voxel_size) -> Tuple[int, int, int]:
    """Grid extents: (max - min) / size in double, rounded half away from zero."""
    out = []
    for a in range(3):
        lo = float(np.float32(pc_range[a]))
        hi = float(np.float32(pc_range[a + 3]))
        v = float(np.float32(voxel_size[a]))
        q = (hi - lo) / v
        fl = math.floor(q)
        out.append(int(fl + (1 if q - fl >= 0.5 else 0)))
    return tuple(out)


def bin_numpy(points: np.ndarray, pc_range, voxel_size):
    """Per-point (valid mask, cx, cy) with float32 NumPy arithmetic."""
    ok, cx, cy, _, g = cells_numpy(points, pc_range, voxel_size)
    return ok, cx, cy, g


def cells_numpy(points: np.ndarray, pc_range, voxel_size):
    """Per-point (valid mask, cx, cy, cz, grid) with float32 NumPy arithmetic."""
    pts = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 4)
    g = grid_py(pc_range, voxel_size)
    lo = np.asarray(pc_range[:3], dtype=np.float32)
    v = np.asarray(voxel_size, dtype=np.float32)
    bits = pts.view(np.uint32)[:, :3]
    finite = np.all((bits & np.uint32(0x7F800000)) != np.uint32(0x7F800000), axis=1)
    with np.errstate(all="ignore"):
        q = np.floor((pts[:, :3] - lo) / v)  # float32 subtract, divide, floor
    gf = np.asarray(g, dtype=np.float32)
    ok = finite & np.all(q >= np.float32(0), axis=1) & np.all(q < gf, axis=1)
    cx = np.where(ok, q[:, 0], 0).astype(np.int64)
    cy = np.where(ok, q[:, 1], 0).astype(np.int64)
    cz = np.where(ok, q[:, 2], 0).astype(np.int64)
    return ok, cx, cy, cz, g


def voxelize_numpy(points: np.ndarray, pc_range, voxel_size, max_points: int, max_voxels: int,
                   three_d: bool = False):
    """Vectorised restatement.  Returns (voxels, coords, counts, V).  With
    ``three_d`` the z cell is part of the key and of the coordinates."""
    pts = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 4)
    ok, cx, cy, cz, g = cells_numpy(pts, pc_range, voxel_size)
    vox = np.zeros((max_voxels, max_points, 4), dtype=np.float32)
    coords = np.zeros((max_voxels, 3), dtype=np.int32)
    counts = np.zeros((max_voxels,), dtype=np.int32)
    idx = np.flatnonzero(ok)
    if idx.size == 0:
        return vox, coords, counts, 0
    key = cy[idx] * g[0] + cx[idx]
    if three_d:
        key = key + cz[idx] * (g[0] * g[1])
    uniq, first_pos, inverse = np.unique(key, return_index=True, return_inverse=True)
    first_idx = idx[first_pos]
    order = np.argsort(first_idx, kind="stable")       # pillars by first point
    rank_of_uniq = np.empty_like(order)
    rank_of_uniq[order] = np.arange(order.size)
    rank = rank_of_uniq[inverse.reshape(-1)]            # per valid point
    s = np.argsort(rank, kind="stable")                 # index order inside a pillar
    r_sorted = rank[s]
    start = np.searchsorted(r_sorted, r_sorted, side="left")
    pos = np.empty_like(s)
    pos[s] = np.arange(s.size) - start
    keep = (rank < max_voxels) & (pos < max_points)
    vox.view(np.uint32)[rank[keep], pos[keep]] = pts.view(np.uint32)[idx[keep]]
    V = int(min(uniq.size, max_voxels))
    counts[:V] = np.minimum(np.bincount(rank, minlength=uniq.size)[:V], max_points)
    kept_keys = uniq[order[:V]]
    coords[:V, 0] = kept_keys // (g[0] * g[1])
    coords[:V, 1] = (kept_keys // g[0]) % g[1]
    coords[:V, 2] = kept_keys % g[0]
    return vox, coords, counts, V


# --------------------------------------------------------------------------
# O(N^2) brute force from the definition, plain Python loops (tiny N only).
# --------------------------------------------------------------------------

def voxelize_bruteforce(points: np.ndarray, pc_range, voxel_size, max_points: int, max_voxels: int,
                        three_d: bool = False):
    """Definition written out point by point.  Returns (voxels, coords, counts, V).
    A key is the tuple of the cells that identify the pillar (cy, cx) or, with
    ``three_d``, the voxel (cz, cy, cx)."""
    pts = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 4)
    g = grid_py(pc_range, voxel_size)
    lo = [np.float32(pc_range[a]) for a in range(3)]
    vs = [np.float32(voxel_size[a]) for a in range(3)]
    n = pts.shape[0]
    keys = []
    with np.errstate(all="ignore"):
        for i in range(n):
            p = pts[i]
            key = None
            if all(math.isfinite(float(p[a])) for a in range(3)):
                cells = []
                for a in range(3):
                    q = np.floor(np.float32(p[a] - lo[a]) / vs[a])
                    if q >= np.float32(0) and q < np.float32(g[a]):
                        cells.append(int(q))
                    else:
                        break
                if len(cells) == 3:
                    key = (cells[2], cells[1], cells[0]) if three_d else (0, cells[1], cells[0])
            keys.append(key)
    first = {}
    for i, k in enumerate(keys):
        if k is not None and k not in first:
            first[k] = i
    vox = np.zeros((max_voxels, max_points, 4), dtype=np.float32)
    coords = np.zeros((max_voxels, 3), dtype=np.int32)
    counts = np.zeros((max_voxels,), dtype=np.int32)
    firsts = list(first.values())
    for i, k in enumerate(keys):
        if k is None:
            continue
        rank = sum(1 for f in firsts if f < first[k])
        pos = sum(1 for j in range(i) if keys[j] == k)
        if rank < max_voxels and pos < max_points:
            vox.view(np.uint32)[rank, pos] = pts.view(np.uint32)[i]
            counts[rank] += 1
            coords[rank] = k
    V = min(len(first), max_voxels)
    return vox, coords, counts, V


# --------------------------------------------------------------------------
# Order-insensitive check of an unordered result (the page's own contract).
# --------------------------------------------------------------------------

def check_unordered(points: np.ndarray, pc_range, voxel_size, max_points: int, max_voxels: int,
                    voxels: np.ndarray, coords: np.ndarray, counts: np.ndarray, V: int,
                    three_d: bool = False):
    """Failures (a list of strings, empty if valid) of a result produced under
    the page's unordered contract ("Claiming a pillar and packing points":
    pillars in slot order, points in atomicAdd arrival order, "keep the
    first K"; "Results": compared after sorting by the (z, y, x) key).

    What is unique is compared exactly: V = min(#pillars, max_voxels); every
    row's coordinates name a distinct occupied pillar (all of them when the
    budget does not bind); every count is min(points of the pillar,
    max_points).  The rest is checked for validity: the rows of a pillar are,
    as a multiset of bit patterns, contained in that pillar's points (so a
    pillar under the cap holds exactly its points), and every other byte is
    zero.
    """
    fails = []
    pts = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 4)
    ok, cx, cy, cz, g = cells_numpy(pts, pc_range, voxel_size)
    if not three_d:
        cz = np.zeros_like(cz)
    key = (cz * g[1] + cy) * g[0] + cx
    idx = np.flatnonzero(ok)
    pk = key[idx]
    uniq, n_of = np.unique(pk, return_counts=True)
    exp_V = int(min(uniq.size, max_voxels))
    if V != exp_V:
        return [f"V {V} != {exp_V}"]
    K, M = max_points, max_voxels
    c = np.asarray(coords, dtype=np.int64)[:V]
    rkey = (c[:, 0] * g[1] + c[:, 1]) * g[0] + c[:, 2]
    if V and (np.any(c < 0) or np.any(c[:, 2] >= g[0]) or np.any(c[:, 1] >= g[1]) or np.any(c[:, 0] >= g[2])):
        fails.append("coordinates out of the grid")
        return fails
    if np.unique(rkey).size != V:
        fails.append("two rows name the same pillar")
    pos = np.searchsorted(uniq, rkey)
    pos = np.minimum(pos, max(uniq.size - 1, 0))
    if V and not np.all(uniq[pos] == rkey):
        fails.append("a row names an empty pillar")
        return fails
    if uniq.size <= M and V and not np.array_equal(np.sort(rkey), uniq):
        fails.append("pillar set differs")
    exp_cnt = np.minimum(n_of[pos], K) if V else np.zeros(0, dtype=np.int64)
    got_cnt = np.asarray(counts)[:V].astype(np.int64)
    if not np.array_equal(got_cnt, exp_cnt):
        bad = int(np.flatnonzero(got_cnt != exp_cnt)[0])
        fails.append(f"row {bad}: count {got_cnt[bad]} != {exp_cnt[bad]}")
        return fails
    # Padding: positions >= count of live rows, and every row >= V, all zero bits.
    vb = np.ascontiguousarray(voxels).view(np.uint32).reshape(M, K, 4)
    live = np.zeros((M, K), dtype=bool)
    if V:
        live[:V] = np.arange(K)[None, :] < got_cnt[:, None]
    if np.any(vb[~live] != 0):
        fails.append("nonzero padding in voxels")
    if np.any(np.asarray(coords)[V:] != 0) or np.any(np.asarray(counts)[V:] != 0):
        fails.append("nonzero padding in coords or counts")
    # Multiset containment of the stored rows in their pillar's points.
    rec = np.dtype([("k", "<i8"), ("a", "<u4"), ("b", "<u4"), ("c", "<u4"), ("d", "<u4")])
    pb = pts.view(np.uint32)[idx]
    have = np.empty(idx.size, dtype=rec)
    have["k"], have["a"], have["b"], have["c"], have["d"] = pk, pb[:, 0], pb[:, 1], pb[:, 2], pb[:, 3]
    rr, ee = np.nonzero(live[:V]) if V else (np.zeros(0, int), np.zeros(0, int))
    got = np.empty(rr.size, dtype=rec)
    gb = vb[rr, ee]
    got["k"], got["a"], got["b"], got["c"], got["d"] = rkey[rr] if V else 0, gb[:, 0], gb[:, 1], gb[:, 2], gb[:, 3]
    hu, hc = np.unique(have, return_counts=True)
    gu, gc = np.unique(got, return_counts=True)
    at = np.searchsorted(hu, gu)
    at = np.minimum(at, max(hu.size - 1, 0))
    found = (hu[at] == gu) if hu.size else np.zeros(gu.size, dtype=bool)
    if not np.all(found):
        fails.append("a stored row is not a point of its pillar")
    elif np.any(gc > hc[at]):
        fails.append("a point is stored more often than it occurs")
    return fails


# --------------------------------------------------------------------------
# Batches of frames: each frame voxelized on its own.
# --------------------------------------------------------------------------

def voxelize_batch(points: np.ndarray, frame_offsets, pc_range, voxel_size, max_points: int,
                   max_voxels: int, three_d: bool = False, lib=None):
    """B frames, frame b = points[frame_offsets[b]:frame_offsets[b + 1]], each
    voxelized exactly as one cloud (same grid, caps per frame).  Returns
    (status, voxels [B, M, K, 4], coords [B, M, 4] = (b, z, y, x), counts
    [B, M], V [B]); coordinate rows past V_b are zero, batch index included.
    The batch index in the coordinates follows the batched PointPillars
    layout (one (batch, z, y, x) row per voxel)."""
    off = [int(o) for o in frame_offsets]
    B = len(off) - 1
    vox = np.zeros((B, max_voxels, max_points, 4), dtype=np.float32)
    coords = np.zeros((B, max_voxels, 4), dtype=np.int32)
    counts = np.zeros((B, max_voxels), dtype=np.int32)
    Vs = np.zeros(B, dtype=np.int32)
    pts = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 4)
    for b in range(B):
        st, v, c, n, V = voxelize(pts[off[b]:off[b + 1]], pc_range, voxel_size, max_points, max_voxels, lib,
                                  three_d=three_d)
        if st != OK:
            return st, vox, coords, counts, Vs
        vox[b], counts[b], Vs[b] = v, n, V
        coords[b, :V, 0] = b
        coords[b, :, 1:] = c
    return OK, vox, coords, counts, Vs


def voxelize_batch_numpy(points: np.ndarray, frame_offsets, pc_range, voxel_size, max_points: int,
                         max_voxels: int, three_d: bool = False):
    """Restatement over the whole concatenated cloud: the grouping key is
    (frame, voxel id), voxels are ordered by their first point inside each
    frame and the budget applies per frame.  Same return values as
    :func:`voxelize_batch` without the status."""
    pts = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 4)
    off = np.asarray(frame_offsets, dtype=np.int64)
    B = off.size - 1
    K, M = max_points, max_voxels
    ok, cx, cy, cz, g = cells_numpy(pts, pc_range, voxel_size)
    if not three_d:
        cz = np.zeros_like(cz)
    frame = np.searchsorted(off, np.arange(pts.shape[0]), side="right") - 1
    cells = g[0] * g[1] * g[2]
    key = frame * cells + (cz * g[1] + cy) * g[0] + cx
    vox = np.zeros((B, M, K, 4), dtype=np.float32)
    coords = np.zeros((B, M, 4), dtype=np.int32)
    counts = np.zeros((B, M), dtype=np.int32)
    Vs = np.zeros(B, dtype=np.int32)
    idx = np.flatnonzero(ok)
    if idx.size == 0:
        return vox, coords, counts, Vs
    uniq, first_pos, inverse = np.unique(key[idx], return_index=True, return_inverse=True)
    first_idx = idx[first_pos]
    order = np.argsort(first_idx, kind="stable")        # voxels by first point (frames in order)
    ufr = uniq[order] // cells                           # frame of each voxel, ascending
    start_of_frame = np.searchsorted(ufr, np.arange(B), side="left")
    rank_global = np.empty_like(order)
    rank_global[order] = np.arange(order.size)
    ufr_by_uniq = uniq // cells
    local = rank_global - start_of_frame[ufr_by_uniq]    # rank inside its frame
    p_local = local[inverse.reshape(-1)]
    p_frame = ufr_by_uniq[inverse.reshape(-1)]
    p_rank = rank_global[inverse.reshape(-1)]
    s = np.argsort(p_rank, kind="stable")
    rs = p_rank[s]
    st = np.searchsorted(rs, rs, side="left")
    pos = np.empty_like(s)
    pos[s] = np.arange(s.size) - st
    keep = (p_local < M) & (pos < K)
    vox.view(np.uint32)[p_frame[keep], p_local[keep], pos[keep]] = pts.view(np.uint32)[idx[keep]]
    n_of = np.bincount(inverse.reshape(-1), minlength=uniq.size)
    live = local < M
    counts[ufr_by_uniq[live], local[live]] = np.minimum(n_of[live], K)
    per_frame = np.bincount(ufr_by_uniq, minlength=B)
    Vs[:] = np.minimum(per_frame, M)
    vid = uniq[live] % cells
    coords[ufr_by_uniq[live], local[live], 0] = ufr_by_uniq[live]
    coords[ufr_by_uniq[live], local[live], 1] = vid // (g[0] * g[1])
    coords[ufr_by_uniq[live], local[live], 2] = (vid // g[0]) % g[1]
    coords[ufr_by_uniq[live], local[live], 3] = vid % g[0]
    return vox, coords, counts, Vs


# --------------------------------------------------------------------------
# Voxel-grid centroid downsampling.
# --------------------------------------------------------------------------

def _bind_downsample(lib):
    if not hasattr(lib, "pv_oracle_downsample"):
        return None
    f = ctypes.POINTER(ctypes.c_float)
    i32 = ctypes.POINTER(ctypes.c_int32)
    fn = lib.pv_oracle_downsample
    fn.argtypes = [f, ctypes.c_int64, f, f, ctypes.c_int, f, i32, i32, i32]
    fn.restype = ctypes.c_int
    return fn


def downsample(points: np.ndarray, pc_range, voxel_size, max_voxels: int, lib=None):
    """The C++ oracle of centroid downsampling.  Returns (status, centroids
    [M, 4] float32, coords [M, 3] int32 (z, y, x), counts [M] int32, V)."""
    lib = lib or load()
    fn = _bind_downsample(lib)
    pts = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 4)
    r, v = _f32(pc_range), _f32(voxel_size)
    cen = np.empty((max_voxels, 4), dtype=np.float32)
    coords = np.empty((max_voxels, 3), dtype=np.int32)
    counts = np.empty((max_voxels,), dtype=np.int32)
    num = np.zeros(1, dtype=np.int32)
    i32 = ctypes.POINTER(ctypes.c_int32)
    st = fn(_fptr(pts) if pts.size else None, pts.shape[0], _fptr(r), _fptr(v), int(max_voxels), _fptr(cen),
            coords.ctypes.data_as(i32), counts.ctypes.data_as(i32), num.ctypes.data_as(i32))
    return st, cen, coords, counts, int(num[0])


def time_passes(op: str, points: np.ndarray, pc_range, voxel_size, max_points: int, max_voxels: int, reps: int,
                lib=None) -> np.ndarray:
    """Durations (ns, steady_clock, measured inside the C++ library) of
    `reps` runs of one oracle pass on the same cloud: op "voxelize",
    "voxelize3d" or "downsample".  For the benchmark's CPU baseline only."""
    lib = lib or load()
    fn = lib.pv_oracle_time
    f = ctypes.POINTER(ctypes.c_float)
    i32 = ctypes.POINTER(ctypes.c_int32)
    fn.argtypes = [ctypes.c_int, f, ctypes.c_int64, f, f, ctypes.c_int, ctypes.c_int, f, i32, i32, i32, ctypes.c_int,
                   ctypes.POINTER(ctypes.c_int64)]
    fn.restype = ctypes.c_int
    code = {"voxelize": 0, "voxelize3d": 1, "downsample": 2}[op]
    pts = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 4)
    r, v = _f32(pc_range), _f32(voxel_size)
    width = 1 if code == 2 else max_points
    rows = np.empty((max_voxels, width, 4), dtype=np.float32)
    coords = np.empty((max_voxels, 3), dtype=np.int32)
    counts = np.empty((max_voxels,), dtype=np.int32)
    num = np.zeros(1, dtype=np.int32)
    times = np.zeros(reps, dtype=np.int64)
    st = fn(code, _fptr(pts) if pts.size else None, pts.shape[0], _fptr(r), _fptr(v), int(max_points),
            int(max_voxels), _fptr(rows), coords.ctypes.data_as(i32), counts.ctypes.data_as(i32),
            num.ctypes.data_as(i32), int(reps), times.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)))
    if st != OK:
        raise RuntimeError(f"oracle status {st}")
    return times


def downsample_exact(points: np.ndarray, pc_range, voxel_size, max_voxels: int):
    """Restatement with exact sums: each voxel's mean is the exact rational sum
    of its points' fields over the count (math.fsum is exact for these sums
    of float32 values), then rounded to float32.  Returns (centroids, coords,
    counts, V)."""
    pts = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 4)
    ok, cx, cy, cz, g = cells_numpy(pts, pc_range, voxel_size)
    key = (cz * g[1] + cy) * g[0] + cx
    M = max_voxels
    cen = np.zeros((M, 4), dtype=np.float32)
    coords = np.zeros((M, 3), dtype=np.int32)
    counts = np.zeros((M,), dtype=np.int32)
    idx = np.flatnonzero(ok)
    if idx.size == 0:
        return cen, coords, counts, 0
    uniq, first_pos, inverse = np.unique(key[idx], return_index=True, return_inverse=True)
    order = np.argsort(idx[first_pos], kind="stable")
    V = int(min(uniq.size, M))
    inverse = inverse.reshape(-1)
    for r in range(V):
        u = order[r]
        members = idx[inverse == u]
        n = members.size
        counts[r] = n
        k = int(uniq[u])
        coords[r] = (k // (g[0] * g[1]), (k // g[0]) % g[1], k % g[0])
        for c in range(4):
            vals = pts[members, c].astype(np.float64)
            if not np.all(np.isfinite(vals)):
                cen[r, c] = np.float32(np.nan if np.any(np.isnan(vals)) or np.ptp(vals[np.isinf(vals)]) > 0
                                       else vals[np.isinf(vals)][0])
            else:
                cen[r, c] = np.float32(math.fsum(vals) / n)
    return cen, coords, counts, V


def ulp_distance32(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Units in the last place between float32 arrays (NaN == NaN counts 0)."""
    ai = np.ascontiguousarray(a, dtype=np.float32).view(np.int32).astype(np.int64)
    bi = np.ascontiguousarray(b, dtype=np.float32).view(np.int32).astype(np.int64)
    ai = np.where(ai < 0, -(ai & 0x7FFFFFFF), ai)  # a monotone integer line through +-0
    bi = np.where(bi < 0, -(bi & 0x7FFFFFFF), bi)
    d = np.abs(ai - bi)
    both_nan = np.isnan(a) & np.isnan(b)
    return np.where(both_nan, 0, d)


# --------------------------------------------------------------------------
# Farthest point sampling.
# --------------------------------------------------------------------------

def fps(points: np.ndarray, num_samples: int, start: int = 0, lib=None):
    """The C++ oracle of farthest point sampling.  Returns (status, indices [M] int32)."""
    lib = lib or load()
    fn = lib.pv_oracle_fps
    fn.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                   ctypes.POINTER(ctypes.c_int32)]
    fn.restype = ctypes.c_int
    pts = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 4)
    out = np.zeros(max(int(num_samples), 0), dtype=np.int32)
    st = fn(_fptr(pts) if pts.size else None, pts.shape[0], int(num_samples), int(start),
            out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    return st, out


def fps_numpy(points: np.ndarray, num_samples: int, start: int = 0):
    """Vectorised restatement: one NumPy float32 pass per sample (the same
    operation order, elementwise, so every distance has the same bits), and
    np.argmax, which returns the first maximum."""
    pts = np.ascontiguousarray(points, dtype=np.float32).reshape(-1, 4)
    x, y, z = pts[:, 0], pts[:, 1], pts[:, 2]
    dist = np.full(pts.shape[0], np.inf, dtype=np.float32)
    out = np.zeros(num_samples, dtype=np.int32)
    sel = int(start)
    for k in range(num_samples):
        out[k] = sel
        dx, dy, dz = x - x[sel], y - y[sel], z - z[sel]
        d = (dx * dx + dy * dy) + dz * dz
        np.minimum(dist, d, out=dist)
        sel = int(np.argmax(dist))
    return out
