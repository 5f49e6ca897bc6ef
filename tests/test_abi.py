"""The C ABI without a GPU: the library builds, loads, exports every symbol
include/*.h declares, and its host-side logic (grid extents, argument checks,
status strings) behaves as documented.  No kernel is launched here.
"""

from __future__ import annotations

import ctypes
import glob
import os
import re

import numpy as np
import pytest

import lidar_point_cloud_gb300 as pv
from lidar_point_cloud_gb300 import _binding, _build, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if _build.is_stale():
        _build.build()
    return pv.load()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(pv_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert {"pv_voxelize", "pv_voxelize_host", "pv_grid_size", "pv_status_string"} <= names
    assert names == set(_binding.EXPORTS), names ^ set(_binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {_build.LIB}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}\b", out), name


def test_library_built_for_sm103a(lib):
    assert "arch=compute_103a,code=sm_103a" in " ".join(_build.NVCC_FLAGS)
    for flag in ("-ftz=false", "-prec-div=true", "-fmad=false"):
        assert flag in _build.NVCC_FLAGS
    assert "--use_fast_math" not in _build.NVCC_FLAGS


def test_version_and_status_strings(lib):
    assert lib.pv_version() == b"0.1.0"
    for code, name in _binding.STATUS.items():
        assert lib.pv_status_string(code).decode().startswith(name)


@pytest.mark.parametrize("rng_vox", [
    (synth.KITTI_RANGE, synth.KITTI_VOXEL),
    (synth.DENSE_RANGE, synth.DENSE_VOXEL),
    (synth.DENSE_RANGE, synth.ADV_VOXEL),
    ((0, 0, 0, 4, 2, 1), (1, 1, 1)),
    ((-3.3, 1.7, -2, 5.1, 9.9, 2), (0.3, 0.25, 4.0)),
])
def test_grid_size_matches_oracle(lib, rng_vox):
    import oracle

    r, v = rng_vox
    st, g = oracle.grid(r, v)
    assert st == 0
    assert pv.grid_size(r, v) == g


def test_grid_size_errors(lib):
    assert pv.grid_size(synth.KITTI_RANGE, (0.16, 0.16, 1.0)) == (432, 496, 4)  # true 3-D voxels
    with pytest.raises(pv.PVError) as e:  # 2^31 voxels or more: ids would not fit int32
        pv.grid_size((0, 0, 0, 2048, 2048, 512), (1, 1, 1))
    assert e.value.status == -1
    for bad in [(0.0, 0.16, 4.0), (-0.16, 0.16, 4.0), (float("nan"), 0.16, 4.0), (float("inf"), 0.16, 4.0)]:
        with pytest.raises(pv.PVError) as e:
            pv.grid_size(synth.KITTI_RANGE, bad)
        assert e.value.status == -1
    with pytest.raises(pv.PVError):
        pv.grid_size((1, 0, 0, 0, 1, 1), (0.1, 0.1, 1))  # max <= min
    with pytest.raises(pv.PVError):
        pv.grid_size((0, 0, 0, 1e9, 1, 1), (1e-3, 1, 1))  # > 2^24 cells on x


def _call(lib, points, n, out, max_points=32, max_voxels=16):
    r = (ctypes.c_float * 6)(*synth.KITTI_RANGE)
    v = (ctypes.c_float * 3)(*synth.KITTI_VOXEL)
    vox, coords, counts, num = out
    return lib.pv_voxelize(points, n, r, v, max_points, max_voxels, vox, coords, counts, num, None)


def test_host_side_argument_checks(lib):
    # Rejected before any device work: null, host or misaligned pointers, bad sizes.
    host = np.zeros(1024, dtype=np.float32)
    hp = ctypes.c_void_p(host.ctypes.data)
    assert _call(lib, hp, 4, (None, hp, hp, hp)) == -1
    assert _call(lib, None, 4, (hp, hp, hp, hp)) == -1           # N > 0 with no points
    assert _call(lib, hp, 4, (hp, hp, hp, hp)) == -1             # host pointers
    assert _call(lib, hp, 4, (ctypes.c_void_p(host.ctypes.data + 4), hp, hp, hp)) == -1  # misaligned
    assert _call(lib, hp, -1, (hp, hp, hp, hp)) == -1
    assert _call(lib, hp, 4, (hp, hp, hp, hp), max_points=0) == -1


def test_binding_checks_without_gpu(lib):
    import torch

    pts = torch.zeros((4, 4), dtype=torch.float32)
    out = tuple(torch.zeros(s, dtype=d) for s, d in (((16, 32, 4), torch.float32), ((16, 3), torch.int32),
                                                      ((16,), torch.int32), ((1,), torch.int32)))
    with pytest.raises(ValueError):
        pv.voxelize_into(pts, synth.KITTI_RANGE, synth.KITTI_VOXEL, 32, 16, out)  # CPU tensor
    with pytest.raises(TypeError):
        pv.voxelize_into(pts.double(), synth.KITTI_RANGE, synth.KITTI_VOXEL, 32, 16, out)
    with pytest.raises(ValueError):
        pv.voxelize_into(pts[:, :3], synth.KITTI_RANGE, synth.KITTI_VOXEL, 32, 16, out)


def test_no_cpu_fallback_when_library_missing(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        _binding.load(str(tmp_path / "missing.so"))
