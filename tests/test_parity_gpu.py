"""GPU parity: the CUDA library against the CPU oracle, bit for bit.

Every output buffer (the full padded [max_voxels, ...] tensors) and V are
compared byte for byte: the operation is integer/bit-copy work once the
binning is fixed to IEEE round-to-nearest binary32, so the bar is exact
equality.  Covers the five workloads at full size, random tiny clouds where
both caps bind, edge cases (empty, one point, all invalid, one pillar with
many points, caps of 1, caps not a multiple of 4 or 32), both table modes,
several launch shapes, repeated runs (determinism), two streams at once,
the host-buffer entry point (whose result is the first V rows: those are
compared, and the rows past V must still hold what the caller put there)
and the device error paths (undersized table, recovery afterwards).
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


def gpu_run(pts, r, v, K, M, stream=None, **opts):
    t = torch.from_numpy(np.ascontiguousarray(pts, dtype=np.float32).reshape(-1, 4)).to(DEV)
    out = pv.alloc_outputs(K, M, DEV)
    for o in out:  # poison: the kernel must overwrite every byte
        o.view(torch.int32).fill_(0x7FBADBAD)
    pv.voxelize_into(t, r, v, K, M, out, stream=stream, **opts)
    torch.cuda.synchronize()
    vox, coords, counts, num = (o.cpu().numpy() for o in out)
    return vox, coords, counts, int(num[0])


def assert_parity(pts, r, v, K, M, **opts):
    st, ov, oc, on, oV = oracle.voxelize(pts, r, v, K, M)
    assert st == 0
    gv, gc, gn, gV = gpu_run(pts, r, v, K, M, **opts)
    assert gV == oV, (gV, oV)
    assert same_bits(gc, oc), "coords: " + first_difference(gc, oc)
    assert same_bits(gn, on), "counts: " + first_difference(gn, on)
    assert same_bits(gv, ov), "voxels: " + first_difference(gv, ov)
    return oV


WORKLOADS = ["tiny", "kitti", *[f"uniform_{n}" for n in synth.UNIFORM_SIZES], "dense", "adversarial"]


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pv.load()
    yield
    pv.release_workspace()


@pytest.mark.parametrize("name", WORKLOADS)
def test_workload_parity(name):
    pts, P = synth.make(name)
    assert_parity(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)


@pytest.mark.parametrize("name", ["kitti", "dense"])
def test_hashed_table_parity(name):
    pts, P = synth.make(name)
    assert_parity(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels, table_mode=2)


@pytest.mark.parametrize("ctas_per_sm", [1, 2, 3])
def test_launch_shape_does_not_change_result(ctas_per_sm):
    pts, P = synth.make("kitti")
    assert_parity(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels, ctas_per_sm=ctas_per_sm)


@pytest.mark.parametrize("ctas_per_sm", [1, 2])
def test_launch_shape_512_thread_build(ctas_per_sm):
    # The dense frame on the 512-thread build at one block an SM (6,912-point
    # chunks; 25 kept rows a warp, so interleaved gather shares) and at two
    # (3,456-point chunks; block-first contiguous shares).
    pts, P = synth.make("dense")
    args = (P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)
    plan = pv.query_plan(len(pts), *args, ctas_per_sm=ctas_per_sm)
    assert plan["threads"] == 512 and plan["ctas"] % ctas_per_sm == 0, plan
    assert_parity(pts, *args, ctas_per_sm=ctas_per_sm)


def test_random_tiny_clouds():
    rng = np.random.Generator(np.random.PCG64(4242))
    for t in range(150):
        pts, r, v, K, M = random_tiny_case(rng)
        assert_parity(pts, r, v, K, M, table_mode=(2 if t % 3 == 0 else 0))


def test_chunk_sizes_around_tile_boundaries():
    # Each block owns ceil(N / blocks) points rounded up to a warp and sweeps
    # them in tiles from its own start: while a chunk fits one tile of as
    # many points as the block has threads, one such tile; past that (on
    # 512-thread blocks, two an SM, where the planner has that build) a
    # first tile of one point a thread and then tiles of up to two.  So
    # tiles start anywhere and a chunk may end with a short tile, or one
    # whose second half is empty.  For each launch shape, chunks of one warp
    # or exactly one tile, and around the first narrow and the wide tiles;
    # the points are KITTI-shaped returns repeated in sensor order, so
    # pillars span tile and chunk boundaries.
    P = synth.KITTI_PARAMS
    base, _ = synth.make("kitti")
    args = (P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)
    small = pv.query_plan(len(base), *args)
    c1, t1 = small["ctas"], small["threads"]
    big = pv.query_plan(t1 * c1 + 1, *args)
    c2, t2 = big["ctas"], big["threads"]
    cases = [(32, 32 * c1 - 7), (t1, t1 * c1 - 3)]
    cases += [(t2 + 32, t2 * c2 + 1), (2 * t2, 2 * t2 * c2 - 5), (2 * t2 + 32, 2 * t2 * c2 + 40),
              (3 * t2, 3 * t2 * c2 - 3), (5 * t2 + 32, 5 * t2 * c2 + 40)]
    for want_chunk, n in cases:
        plan = pv.query_plan(n, *args)
        assert plan["points_per_cta"] == want_chunk, (n, plan["points_per_cta"])
        pts = np.tile(base, (n // len(base) + 1, 1))[:n]
        assert_parity(pts, *args)


def test_sparse_chunks_of_several_tiles():
    # About six 1024-point tiles a chunk, uniform over a 2048 x 2048 grid of
    # 0.05 m pillars: nearly every point of a tile has its own pillar, so
    # the chunks keep 1024-point tiles (their maps half full), and the
    # pillar budget binds.  Direct and hashed tables.
    r, v = synth.DENSE_RANGE, synth.ADV_VOXEL
    ctas = pv.query_plan(1 << 20, r, v, 32, 200_000)["ctas"]
    n = 3 * 2048 * ctas + 77
    pts = synth.uniform(n, 41, pc_range=r)
    for mode in (0, 2):
        assert_parity(pts, r, v, 32, 200_000, table_mode=mode)


@pytest.mark.parametrize("run", [700, 3000])
def test_tile_width_switches(run):
    # Runs of `run` sensor-ordered returns of the dense frame (few pillars a
    # tile: tiles widen to 2048 points) alternating with runs of uniform
    # points over the same grid (a pillar a point: tiles narrow to 1024), so
    # chunks change tile width both ways, with tiles straddling the runs.
    P = synth.DENSE_PARAMS
    dense, _ = synth.make("dense")
    uni = synth.uniform(dense.shape[0], 43, pc_range=P.point_cloud_range)
    k = np.arange(dense.shape[0]) // run
    pts = np.where((k % 2 == 0)[:, None], dense, uni).astype(np.float32)
    assert_parity(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)


def test_determinism_repeats():
    pts, P = synth.make("kitti")
    ref = gpu_run(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)
    t = torch.from_numpy(pts).to(DEV)
    out = pv.alloc_outputs(P.max_points, P.max_voxels, DEV)
    for _ in range(50):
        pv.voxelize_into(t, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels, out)
        torch.cuda.synchronize()
        got = [o.cpu().numpy() for o in out]
        assert int(got[3][0]) == ref[3]
        for a, b in zip(got[:3], ref[:3]):
            assert same_bits(a, b)


KR, KV = synth.KITTI_RANGE, synth.KITTI_VOXEL


def test_empty_cloud():
    assert assert_parity(np.zeros((0, 4), np.float32), KR, KV, 32, 1000) == 0


def test_single_point():
    assert assert_parity(np.array([[10.0, 0.0, -1.0, 0.5]], np.float32), KR, KV, 32, 100) == 1


def test_all_points_invalid():
    pts = synth.uniform(5000, 11)
    pts[:, 0] = -5.0  # every x below x_min
    assert assert_parity(pts, KR, KV, 32, 100) == 0


def test_one_pillar_many_points():
    rng = np.random.Generator(np.random.PCG64(5))
    pts = np.zeros((200_000, 4), np.float32)
    pts[:, 0] = 10.0 + 0.05 * rng.random(200_000)  # cell 62 only
    pts[:, 1] = 0.01 * rng.random(200_000)
    pts[:, 2] = -1.0
    pts[:, 3] = rng.random(200_000)
    assert assert_parity(pts, KR, KV, 32, 10) == 1


def hot_cloud(n, hot_pillars, hot_frac, seed):
    """A cloud over the KITTI-shaped range with hot_frac of its points inside
    hot_pillars cells, in random order (the hot pillars overflow every cap)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    pts = synth.uniform(n, seed)
    n_hot = int(n * hot_frac)
    cells = rng.choice(432 * 496, size=hot_pillars, replace=False)
    pick = cells[rng.integers(0, hot_pillars, size=n_hot)]
    u = rng.random((n_hot, 2))
    pts[:n_hot, 0] = (0.0 + ((pick % 432) + 0.05 + 0.9 * u[:, 0]) * 0.16).astype(np.float32)
    pts[:n_hot, 1] = (-39.68 + ((pick // 432) + 0.05 + 0.9 * u[:, 1]) * 0.16).astype(np.float32)
    return pts[rng.permutation(n)]


@pytest.mark.parametrize("K", [8, 20, 32, 64, 200, 1024])
def test_hot_pillars_large_caps_twice(K):
    # Most groups of the hot pillars have max_points points before them and are
    # dropped; a second call checks that the first left no list entry behind.
    # With 8..32 points a pillar the hot pillars overflow their append slots.
    pts = hot_cloud(600_000, 8, 0.6, 31)
    for _ in range(2):
        assert_parity(pts, KR, KV, K, 2000)


@pytest.mark.parametrize("K", [32, 1024])
def test_chunk_point_counter_wraps(K):
    # About 70,000 points of one pillar per block chunk: the 16-bit point count
    # of the chunk map wraps; the groups it then lets through are never needed.
    pts = hot_cloud(11_010_048, 1, 0.95, 32)
    for _ in range(2):
        assert_parity(pts, KR, KV, K, 500)


@pytest.mark.parametrize("K,M", [(1, 1), (1, 16000), (32, 1), (5, 500), (8, 300), (20, 4000), (33, 2000),
                                 (64, 3000), (100, 700)])
def test_caps(K, M):
    pts, P = synth.make("kitti")
    assert_parity(pts, P.point_cloud_range, P.voxel_size, K, M)


def test_index_intensity_order():
    pts, P = synth.make("uniform_130000")
    pts = pts.copy()
    pts[:, 3] = np.arange(pts.shape[0], dtype=np.float32)
    assert_parity(pts, P.point_cloud_range, P.voxel_size, P.max_points, 200_000)


def test_large_grid_uses_hashed_table():
    # 1 cm pillars over the KITTI-shaped range: 6912 x 7936 cells, hashed table.
    r, v = KR, (0.01, 0.01, 4.0)
    plan = pv.query_plan(122_880, r, v, 32, 60_000)
    assert plan["table_mode"] == "hashed"
    pts, _ = synth.make("kitti")
    assert_parity(pts, r, v, 32, 60_000)


def test_capacity_error_then_recovery():
    pts = synth.uniform(20_000, 12)
    got = gpu_run(pts, KR, KV, 32, 16_000, table_mode=2, table_log2=4)  # 16 slots
    assert got[3] == -5  # PV_ERR_CAPACITY
    assert_parity(pts, KR, KV, 32, 16_000, table_mode=2)
    assert_parity(pts, KR, KV, 32, 16_000)


def test_wait_timeout_is_reported_and_recovered():
    """A grid barrier that can never complete gives up after its time limit
    (about one second), the call reports PV_ERR_TIMEOUT through V, the
    context stays usable, and the next call on the stream is exact again
    (the kernel resets the table it could not clean)."""
    pts, P = synth.make("kitti")
    got = gpu_run(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels, test_stall_barrier=1)
    assert got[3] == -6  # PV_ERR_TIMEOUT
    assert_parity(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)
    assert_parity(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels, table_mode=2)


def test_two_streams():
    a, Pa = synth.make("kitti")
    b, Pb = synth.make("uniform_100000")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ta, tb = torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV)
    oa, ob = pv.alloc_outputs(32, 16000, DEV), pv.alloc_outputs(32, 16000, DEV)
    torch.cuda.synchronize()
    for _ in range(5):
        pv.voxelize_into(ta, KR, KV, 32, 16000, oa, stream=s1)
        pv.voxelize_into(tb, KR, KV, 32, 16000, ob, stream=s2)
    torch.cuda.synchronize()
    for pts, out in ((a, oa), (b, ob)):
        st, ov, oc, on, oV = oracle.voxelize(pts, KR, KV, 32, 16000)
        assert int(out[3].item()) == oV
        assert same_bits(out[0].cpu().numpy(), ov)


def check_host_result(res, out, oracle_out, fill):
    # The host entry point's result is the first V rows; rows past V keep
    # what the caller had in them.
    vox, coords, counts, V = res
    st, ov, oc, on, oV = oracle_out
    assert V == oV
    if out is None:  # arrays of the wrapper's own, sliced to V
        assert vox.shape[0] == coords.shape[0] == counts.shape[0] == oV
    else:  # the caller's buffers themselves
        assert all(r is o for r, o in zip(res[:3], out[:3]))
    vox, coords, counts = (np.asarray(a)[:oV] for a in (vox, coords, counts))
    assert same_bits(vox, ov[:oV]) and same_bits(coords, oc[:oV]) and same_bits(counts, on[:oV])
    if out is not None:
        for a in out[:3]:
            tail = np.asarray(a)[oV:]
            assert (tail == fill).all()


def test_host_entry_point():
    pts, P = synth.make("kitti")
    res = pv.voxelize_host(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)
    check_host_result(res, None, oracle.voxelize(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels), 0)


@pytest.mark.parametrize("name", ["kitti", "dense", "tiny"])
def test_host_entry_point_pinned_buffers_in_place(name):
    # Pinned input and outputs: the kernel reads and writes them across the
    # host link; pinned input with pageable outputs, and the reverse, mix
    # in-place use with staging copies.
    pts, P = synth.make(name)
    K, M = P.max_points, P.max_voxels
    ref = oracle.voxelize(pts, P.point_cloud_range, P.voxel_size, K, M)
    pin_pts = torch.from_numpy(pts).pin_memory().numpy()
    shapes = (((M, K, 4), torch.float32), ((M, 3), torch.int32), ((M,), torch.int32), ((1,), torch.int32))
    pinned = tuple(torch.full(sh, 7, dtype=dt).pin_memory().numpy() for sh, dt in shapes)
    pageable = tuple(np.full(sh, 7, dtype=np.float32 if dt == torch.float32 else np.int32) for sh, dt in shapes)
    tensors = tuple(torch.from_numpy(a) for a in pinned)  # CPU tensors (pinned) as the buffers
    for src, out in ((pin_pts, pinned), (pin_pts, pageable), (pts, pinned), (torch.from_numpy(pin_pts), tensors)):
        for a in out:
            a.fill(7) if isinstance(a, np.ndarray) else a.fill_(7)
        res = pv.voxelize_host(src, P.point_cloud_range, P.voxel_size, K, M, out=out)
        check_host_result(res, out, ref, 7)


def test_host_entry_point_misaligned_pinned_input():
    # A pinned cloud that starts 4 bytes into its allocation cannot be read in
    # place (16-byte loads): it goes through the staging copy.
    pts, P = synth.make("tiny")
    buf = torch.zeros(pts.size + 1, dtype=torch.float32).pin_memory().numpy()
    view = buf[1:].reshape(-1, 4)
    view[:] = pts
    assert view.ctypes.data % 16 != 0
    res = pv.voxelize_host(view, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)
    check_host_result(res, None, oracle.voxelize(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels), 0)


def test_sliced_python_entry_point():
    pts, P = synth.make("tiny")
    vox, coords, counts = pv.voxelize(torch.from_numpy(pts).to(DEV), P.point_cloud_range, P.voxel_size)
    st, ov, oc, on, oV = oracle.voxelize(pts, P.point_cloud_range, P.voxel_size, 32, 16000)
    assert vox.shape == (oV, 32, 4) and coords.shape == (oV, 3) and counts.shape == (oV,)
    assert same_bits(vox.cpu().numpy(), ov[:oV])


def test_large_cloud_64m_points():
    # 64 M points (1 GiB of input): chunks of about 440,000 points a block, so
    # the chunk map overflows and the per-block loops run hundreds of tiles.
    rng = np.random.Generator(np.random.PCG64(64))
    n = 64 * 1024 * 1024
    pts = np.empty((n, 4), np.float32)
    pts[:, 0] = rng.random(n, dtype=np.float32) * np.float32(69.12)
    pts[:, 1] = rng.random(n, dtype=np.float32) * np.float32(79.36) - np.float32(39.68)
    pts[:, 2] = rng.random(n, dtype=np.float32) * np.float32(4.0) - np.float32(3.0)
    pts[:, 3] = rng.random(n, dtype=np.float32)
    assert_parity(pts, KR, KV, 32, 16_000)
