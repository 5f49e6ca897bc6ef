"""The allocation-free entry point gives exactly what pv_voxelize gives.

Some callers cannot allocate device memory while they run: code recorded
into a CUDA graph under global capture mode, plug-ins whose host owns all
device memory, real-time loops that forbid allocation after start-up.
pv_voxelize_static serves them from one fixed scratch array inside the
library.  These tests call it through the C ABI and compare every output
byte with the workspace entry point and with the CPU oracle, on calls made
back to back, so the second call starts from whatever state the first left
in the shared array.  This file is collected last on purpose.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pv = pytest.importorskip("lidar_point_cloud_gb300")
from lidar_point_cloud_gb300 import _binding, synth  # noqa: E402

pytestmark = pytest.mark.gpu

PV_ERR_TOO_LARGE = -8


def _call(entry, pts, P, K=None, M=None):
    """Run one entry point through the C ABI; returns its status and host copies."""
    K = P.max_points if K is None else K
    M = P.max_voxels if M is None else M
    lib = pv.load()
    t = torch.from_numpy(np.ascontiguousarray(pts, dtype=np.float32)).cuda()
    out = pv.alloc_outputs(K, M, t.device)
    for o in out:  # poison: every byte must be written by the call
        o.view(torch.int32).fill_(0x7FBADBAD)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = getattr(lib, entry)(
        ctypes.c_void_p(t.data_ptr() if t.shape[0] else 0), int(t.shape[0]),
        _binding._f6(P.point_cloud_range, 6), _binding._f6(P.voxel_size, 3), int(K), int(M),
        *[ctypes.c_void_p(o.data_ptr()) for o in out], stream)
    torch.cuda.synchronize()
    return st, [o.cpu().numpy() for o in out]


def _same(a, b):
    return all(x.tobytes() == y.tobytes() for x, y in zip(a, b))


def test_static_entry_point_matches_twice_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tiny, p_tiny = synth.make("tiny")
    cloud = synth.uniform(30_000, 21)
    runs = [(tiny, p_tiny), (cloud, synth.KITTI_PARAMS), (cloud, synth.KITTI_PARAMS)]
    static_out = []
    for pts, P in runs:  # back-to-back calls sharing the one scratch array
        st, out = _call("pv_voxelize_static", pts, P)
        assert st == 0
        static_out.append(out)
    for (pts, P), got in zip(runs, static_out):
        st, ref = _call("pv_voxelize", pts, P)
        assert st == 0
        assert int(got[3][0]) == int(ref[3][0]) > 0
        assert _same(got, ref)
        ost, ov, oc, on, oV = oracle.voxelize(pts, P.point_cloud_range, P.voxel_size, P.max_points, P.max_voxels)
        assert ost == 0 and int(got[3][0]) == oV
        assert _same(got[:3], [ov, oc, on])


def test_static_entry_point_rejects_sizes_beyond_its_limits():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pts = synth.uniform(32_769, 22)
    st, _ = _call("pv_voxelize_static", pts, synth.KITTI_PARAMS)
    assert st == PV_ERR_TOO_LARGE
    st, _ = _call("pv_voxelize_static", pts[:1000], synth.KITTI_PARAMS, K=33)
    assert st == PV_ERR_TOO_LARGE
