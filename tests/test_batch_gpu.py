"""GPU parity of the batched entry point (several frames per launch), bit for
bit against the batched oracle (each frame voxelized as one cloud).

Covers eight KITTI-shaped frames, ragged frame sizes (empty frames, one-point
frames, frames that start inside a 1024-point tile), the one-frame case, the
maximum frame count, 3-D voxels, a hashed table, binding caps, random tiny
batches, and calls alternating with single-frame calls on one workspace.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle
from _helpers import first_difference, random_tiny_batch, same_bits

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


def assert_batch_parity(pts, off, r, v, K, M, three_d=False):
    st, ov, oc, on, oV = oracle.voxelize_batch(pts, off, r, v, K, M, three_d=three_d)
    assert st == 0
    B = len(off) - 1
    t = torch.from_numpy(np.ascontiguousarray(pts, dtype=np.float32).reshape(-1, 4)).to(DEV)
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
    return oV


def kitti_frames(seeds):
    frames = [synth.kitti(s) for s in seeds]
    off = np.concatenate([[0], np.cumsum([f.shape[0] for f in frames])]).astype(np.int64)
    return np.concatenate(frames), off


def test_eight_kitti_frames():
    pts, off = kitti_frames(range(1, 9))
    V = assert_batch_parity(pts, off, KR, KV, 32, 16_000)
    assert V.min() > 5000


def test_ragged_frames():
    sizes = [0, 1, 5000, 0, 12_345, 777, 30_000, 1023, 1025, 0]
    frames = [synth.uniform(n, 50 + i) for i, n in enumerate(sizes)]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    assert_batch_parity(np.concatenate(frames), off, KR, KV, 32, 16_000)


def test_one_frame_equals_the_single_call():
    pts, P = synth.make("kitti")
    V = assert_batch_parity(pts, [0, pts.shape[0]], KR, KV, 32, 16_000)
    st, ov, oc, on, oV = oracle.voxelize(pts, KR, KV, 32, 16_000)
    assert V[0] == oV


def test_maximum_frame_count():
    rng = np.random.default_rng(7)
    sizes = rng.integers(0, 600, size=pv.MAX_FRAMES)
    frames = [synth.uniform(int(n), 1000 + i) for i, n in enumerate(sizes)]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    assert_batch_parity(np.concatenate(frames), off, KR, KV, 8, 700)


def test_voxel3d_batch():
    pts, off = kitti_frames([3, 4, 5])
    _, P = synth.make("kitti3d")
    assert_batch_parity(pts, off, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels, three_d=True)


def test_hashed_table_batch():
    pts, off = kitti_frames([6, 7])
    _, P = synth.make("second")
    plan = pv.query_plan(int(off[-1]), P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)
    assert plan["table_mode"] == "hashed"
    assert_batch_parity(pts, off, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels, three_d=True)


@pytest.mark.parametrize("K,M", [(1, 1), (5, 500), (64, 3000)])
def test_batch_caps(K, M):
    pts, off = kitti_frames([1, 2, 3])
    assert_batch_parity(pts, off, KR, KV, K, M)


def test_random_tiny_batches():
    rng = np.random.Generator(np.random.PCG64(505))
    for _ in range(30):
        pts, off, r, v, K, M = random_tiny_batch(rng, gz_max=3)
        assert_batch_parity(pts, off, r, v, K, M, three_d=True)


def test_alternating_with_single_frames():
    pts, off = kitti_frames([1, 2])
    single, P = synth.make("dense")
    for _ in range(2):
        assert_batch_parity(pts, off, KR, KV, 32, 16_000)
        st, ov, oc, on, oV = oracle.voxelize(single, P.point_cloud_range, P.voxel_size, 32, 60_000)
        t = torch.from_numpy(single).to(DEV)
        g = pv.voxelize(t, P.point_cloud_range, P.voxel_size, 32, 60_000)
        assert g[0].shape[0] == oV and same_bits(g[0].cpu().numpy(), ov[:oV])


def test_python_batch_api_concatenates_frames():
    pts, off = kitti_frames([1, 2])
    st, ov, oc, on, oV = oracle.voxelize_batch(pts, off, KR, KV, 32, 16_000)
    vox, coords, counts = pv.voxelize_batch(torch.from_numpy(pts).to(DEV), off, KR, KV, 32, 16_000)
    assert vox.shape[0] == coords.shape[0] == counts.shape[0] == int(oV.sum())
    assert same_bits(coords.cpu().numpy(), np.concatenate([oc[b, :oV[b]] for b in range(2)]))


def test_batch_argument_errors():
    lib = pv.load()
    t = torch.zeros((10, 4), dtype=torch.float32, device=DEV)
    out = pv.alloc_batch_outputs(2, 32, 16, DEV)
    args = lambda offs, B: (ctypes.c_void_p(t.data_ptr()), (ctypes.c_int64 * len(offs))(*offs), B,
                            (ctypes.c_float * 6)(*KR), (ctypes.c_float * 3)(*KV), 32, 16,
                            *[ctypes.c_void_p(o.data_ptr()) for o in out], None)
    assert lib.pv_voxelize_batch(*args([1, 5, 10], 2)) == -1   # first offset not 0
    assert lib.pv_voxelize_batch(*args([0, 6, 5], 2)) == -1    # decreasing
    assert lib.pv_voxelize_batch(*args([0, 10], 0)) == -1      # no frames
    assert lib.pv_voxelize_batch(*args([0] * 258, 257)) == -1  # more than PV_MAX_FRAMES
