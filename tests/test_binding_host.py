"""The Python binding of the host-buffer entry point, without a GPU.

`voxelize_host` only marshals arguments: these tests put a stand-in for the
library's `pv_voxelize_host` in place (it records what it was passed and
writes V the way the library does) and check what the wrapper hands over
and returns: the caller's buffers themselves when it passes them (the
result is their first V rows), arrays of its own sliced to V when it does
not, and an exception for a negative status.  The library's own behaviour
on the device is covered by the GPU parity tests.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest

import lidar_point_cloud_gb300 as pv
from lidar_point_cloud_gb300 import _binding

RNG = (0.0, -39.68, -3.0, 69.12, 39.68, 1.0)
VOX = (0.16, 0.16, 4.0)
K, M = 32, 64


class FakeLib:
    """Stands in for libpv.so's pv_voxelize_host: writes `status` (or V) to the count."""

    def __init__(self, V: int, status: int = 0):
        self.V, self.status, self.calls = V, status, []

    def pv_voxelize_host(self, pts, n, rng, vox, k, m, ov, oc, on, onum, stream):
        self.calls.append(dict(pts=pts, n=n, rng=list(rng), vox=list(vox), k=k, m=m, ov=ov, oc=oc, on=on,
                               onum=onum, stream=stream))
        ctypes.c_int32.from_address(onum).value = self.status if self.status < 0 else self.V
        return self.status


@pytest.fixture
def fake(monkeypatch):
    def make(V, status=0):
        lib = FakeLib(V, status)
        monkeypatch.setattr(_binding, "load", lambda path=None: lib)
        return lib
    return make


def cloud(n=10):
    return np.arange(4 * n, dtype=np.float32).reshape(n, 4)


def test_own_arrays_are_sliced_to_v(fake):
    lib = fake(V=5)
    vox, coords, counts, V = pv.voxelize_host(cloud(), RNG, VOX, K, M)
    assert V == 5
    assert vox.shape == (5, K, 4) and coords.shape == (5, 3) and counts.shape == (5,)
    assert vox.dtype == np.float32 and coords.dtype == np.int32 and counts.dtype == np.int32
    call = lib.calls[0]
    assert call["n"] == 10 and call["k"] == K and call["m"] == M and call["stream"] == 0
    assert call["rng"] == pytest.approx(RNG) and call["vox"] == pytest.approx(VOX)


def test_caller_buffers_come_back_as_given(fake):
    lib = fake(V=7)
    out = (np.full((M, K, 4), 7, np.float32), np.full((M, 3), 7, np.int32), np.full((M,), 7, np.int32),
           np.zeros((1,), np.int32))
    res = pv.voxelize_host(cloud(), RNG, VOX, K, M, out=out)
    assert res[3] == 7 and all(r is o for r, o in zip(res[:3], out[:3]))
    call = lib.calls[0]
    assert (call["ov"], call["oc"], call["on"], call["onum"]) == tuple(a.ctypes.data for a in out)
    # The wrapper writes nothing itself: rows past V keep the caller's values.
    assert (out[0] == 7).all() and (out[1] == 7).all() and (out[2] == 7).all()


def test_torch_cpu_buffers(fake):
    torch = pytest.importorskip("torch")
    fake(V=3)
    out = (torch.zeros((M, K, 4)), torch.zeros((M, 3), dtype=torch.int32), torch.zeros((M,), dtype=torch.int32),
           torch.zeros((1,), dtype=torch.int32))
    res = pv.voxelize_host(torch.from_numpy(cloud()), RNG, VOX, K, M, out=out)
    assert res[3] == 3 and all(r is o for r, o in zip(res[:3], out[:3]))


def test_empty_cloud_passes_no_pointer(fake):
    lib = fake(V=0)
    vox, coords, counts, V = pv.voxelize_host(np.zeros((0, 4), np.float32), RNG, VOX, K, M)
    assert V == 0 and vox.shape == (0, K, 4)
    assert lib.calls[0]["pts"] == 0 and lib.calls[0]["n"] == 0


def test_negative_status_raises(fake):
    fake(V=0, status=-5)
    with pytest.raises(_binding.PVError) as e:
        pv.voxelize_host(cloud(), RNG, VOX, K, M)
    assert e.value.status == -5 and "PV_ERR_CAPACITY" in str(e.value)


def test_rejects_device_or_non_contiguous_buffers(fake):
    fake(V=1)
    out = (np.zeros((M, K, 4), np.float32)[:, ::2], np.zeros((M, 3), np.int32), np.zeros((M,), np.int32),
           np.zeros((1,), np.int32))
    with pytest.raises(ValueError):
        pv.voxelize_host(cloud(), RNG, VOX, K, M, out=out)
