"""ctypes binding of libpv.so: argument marshalling only.

Every step of the voxelization runs in the library's CUDA kernel; this file
checks dtypes, devices and shapes the way the page "Voxelize" describes its
C++ wrapper ("The PyTorch side": TORCH_CHECK of dtype, contiguity and device,
then raw pointers), pre-allocates the outputs, and slices them to the real
pillar count V.  There is no CPU fallback: without the compiled library, or
without a GPU, the calls raise.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence, Tuple

from . import _build

STATUS = {
    0: "PV_OK",
    -1: "PV_ERR_INVALID",
    -2: "PV_ERR_UNSUPPORTED",
    -3: "PV_ERR_ALLOC",
    -4: "PV_ERR_CUDA",
    -5: "PV_ERR_CAPACITY",
    -6: "PV_ERR_TIMEOUT",
    -7: "PV_ERR_INTERNAL",
    -8: "PV_ERR_TOO_LARGE",
}

EXPORTS = (
    "pv_voxelize", "pv_voxelize_ex", "pv_voxelize_host", "pv_voxelize_static", "pv_voxelize_batch",
    "pv_voxel_downsample", "pv_fps", "pv_grid_size", "pv_query_plan", "pv_release_workspace", "pv_status_string",
    "pv_version",
)

FPS_MAX_POINTS = 212992  # PV_FPS_MAX_POINTS

MAX_FRAMES = 256  # PV_MAX_FRAMES


class PVError(RuntimeError):
    """A negative status returned by the library."""

    def __init__(self, status: int, where: str = ""):
        self.status = int(status)
        name = STATUS.get(self.status, f"status {self.status}")
        super().__init__(f"{where}: {name}" if where else name)


class Options(ctypes.Structure):
    _fields_ = [("table_mode", ctypes.c_int), ("table_log2", ctypes.c_int),
                ("ctas_per_sm", ctypes.c_int), ("test_stall_barrier", ctypes.c_int),
                ("order", ctypes.c_int), ("reserved", ctypes.c_int * 3)]


class Plan(ctypes.Structure):
    _fields_ = [("grid", ctypes.c_int64 * 3), ("table_mode", ctypes.c_int),
                ("table_slots", ctypes.c_int64), ("list_stride", ctypes.c_int),
                ("ctas", ctypes.c_int), ("threads", ctypes.c_int),
                ("points_per_cta", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB


def load(path: Optional[str] = None):
    """Load libpv.so.  Raises if it has not been built (no fallback)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB
        if not os.path.exists(p):
            raise RuntimeError(
                f"CUDA library {p} is not built; run `python -c \"import __graft_entry__ as g; g.build()\"`")
        lib = ctypes.CDLL(p)
        f = ctypes.POINTER(ctypes.c_float)
        vp = ctypes.c_void_p
        i64 = ctypes.c_int64
        ci = ctypes.c_int
        dev_args = [vp, i64, f, f, ci, ci, vp, vp, vp, vp]
        lib.pv_voxelize.argtypes = dev_args + [vp]
        lib.pv_voxelize.restype = ci
        lib.pv_voxelize_ex.argtypes = dev_args + [ctypes.POINTER(Options), vp]
        lib.pv_voxelize_ex.restype = ci
        lib.pv_voxelize_host.argtypes = dev_args + [vp]
        lib.pv_voxelize_host.restype = ci
        lib.pv_voxelize_static.argtypes = dev_args + [vp]
        lib.pv_voxelize_static.restype = ci
        lib.pv_voxelize_batch.argtypes = [vp, ctypes.POINTER(ctypes.c_int64), ci, f, f, ci, ci, vp, vp, vp, vp, vp]
        lib.pv_voxelize_batch.restype = ci
        lib.pv_voxel_downsample.argtypes = [vp, i64, f, f, ci, vp, vp, vp, vp, vp]
        lib.pv_voxel_downsample.restype = ci
        lib.pv_fps.argtypes = [vp, ci, i64, i64, i64, vp, vp, vp, vp]
        lib.pv_fps.restype = ci
        lib.pv_grid_size.argtypes = [f, f, ctypes.POINTER(ctypes.c_int64)]
        lib.pv_grid_size.restype = ci
        lib.pv_query_plan.argtypes = [i64, f, f, ci, ci, ctypes.POINTER(Options), ctypes.POINTER(Plan)]
        lib.pv_query_plan.restype = ci
        lib.pv_release_workspace.argtypes = []
        lib.pv_release_workspace.restype = ci
        lib.pv_status_string.argtypes = [ci]
        lib.pv_status_string.restype = ctypes.c_char_p
        lib.pv_version.argtypes = []
        lib.pv_version.restype = ctypes.c_char_p
        if path is None:
            _lib = lib
        return lib


def _f6(seq: Sequence[float], n: int):
    vals = [float(x) for x in seq]
    if len(vals) != n:
        raise ValueError(f"expected {n} values, got {len(vals)}")
    return (ctypes.c_float * n)(*vals)


def _options(table_mode=0, table_log2=0, ctas_per_sm=0, test_stall_barrier=0, unordered=False) -> Options:
    o = Options()
    o.table_mode, o.table_log2, o.ctas_per_sm = int(table_mode), int(table_log2), int(ctas_per_sm)
    o.test_stall_barrier = int(test_stall_barrier)
    o.order = 1 if unordered else 0
    return o


def grid_size(point_cloud_range, voxel_size) -> Tuple[int, int, int]:
    g = (ctypes.c_int64 * 3)()
    st = load().pv_grid_size(_f6(point_cloud_range, 6), _f6(voxel_size, 3), g)
    if st != 0:
        raise PVError(st, "pv_grid_size")
    return tuple(int(x) for x in g)


def query_plan(num_points, point_cloud_range, voxel_size, max_points=32, max_voxels=16000, **opts) -> dict:
    p = Plan()
    o = _options(**opts)
    st = load().pv_query_plan(int(num_points), _f6(point_cloud_range, 6), _f6(voxel_size, 3),
                              int(max_points), int(max_voxels), ctypes.byref(o), ctypes.byref(p))
    if st != 0:
        raise PVError(st, "pv_query_plan")
    return {"grid": tuple(p.grid), "table_mode": {1: "direct", 2: "hashed"}[p.table_mode],
            "table_slots": p.table_slots, "list_stride": p.list_stride, "ctas": p.ctas,
            "threads": p.threads, "points_per_cta": p.points_per_cta,
            "workspace_bytes": p.workspace_bytes}


def release_workspace() -> None:
    st = load().pv_release_workspace()
    if st != 0:
        raise PVError(st, "pv_release_workspace")


def _torch():
    import torch

    return torch


def alloc_outputs(max_points: int, max_voxels: int, device):
    torch = _torch()
    vox = torch.empty((max_voxels, max_points, 4), dtype=torch.float32, device=device)
    coords = torch.empty((max_voxels, 3), dtype=torch.int32, device=device)
    counts = torch.empty((max_voxels,), dtype=torch.int32, device=device)
    num = torch.empty((1,), dtype=torch.int32, device=device)
    return vox, coords, counts, num


def voxelize_into(points, point_cloud_range, voxel_size, max_points: int, max_voxels: int,
                  out, stream=None, table_mode: int = 0, table_log2: int = 0, ctas_per_sm: int = 0,
                  test_stall_barrier: int = 0, unordered: bool = False) -> None:
    """Enqueue one voxelization into pre-allocated outputs (no synchronization).

    ``out`` = (voxels [M, K, 4] f32, coords [M, 3] i32, counts [M] i32, num [1] i32),
    all CUDA tensors on the points' device.  ``num`` receives V or a negative
    status once the stream reaches the kernel.  ``unordered`` selects the
    page's own contract (pillars in creation order, points in arrival order).
    """
    torch = _torch()
    vox, coords, counts, num = out
    if not isinstance(points, torch.Tensor) or points.dtype != torch.float32:
        raise TypeError("points must be a float32 torch.Tensor")
    if points.dim() != 2 or points.shape[1] != 4:
        raise ValueError("points must have shape [N, 4]")
    if not points.is_cuda:
        raise ValueError("points must be a CUDA tensor (use voxelize_host for host arrays)")
    if not points.is_contiguous():
        raise ValueError("points must be contiguous")
    for t, dt, shape in ((vox, torch.float32, (max_voxels, max_points, 4)),
                         (coords, torch.int32, (max_voxels, 3)),
                         (counts, torch.int32, (max_voxels,)), (num, torch.int32, (1,))):
        if t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous() or t.device != points.device:
            raise ValueError("output tensor has the wrong dtype, shape, layout or device")
    if stream is None:
        stream = torch.cuda.current_stream(points.device)
    handle = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    lib = load()
    args = (ctypes.c_void_p(points.data_ptr() if points.shape[0] else 0), int(points.shape[0]),
            _f6(point_cloud_range, 6), _f6(voxel_size, 3), int(max_points), int(max_voxels),
            ctypes.c_void_p(vox.data_ptr()), ctypes.c_void_p(coords.data_ptr()),
            ctypes.c_void_p(counts.data_ptr()), ctypes.c_void_p(num.data_ptr()))
    if table_mode or table_log2 or ctas_per_sm or test_stall_barrier or unordered:
        o = _options(table_mode, table_log2, ctas_per_sm, test_stall_barrier, unordered)
        st = lib.pv_voxelize_ex(*args, ctypes.byref(o), handle)
    else:
        st = lib.pv_voxelize(*args, handle)
    if st != 0:
        raise PVError(st, "pv_voxelize")


def voxelize(points, point_cloud_range, voxel_size, max_points: int = 32, max_voxels: int = 16000,
             stream=None, **opts):
    """Voxelize one cloud on its GPU.  Returns (voxels [V,K,4], coords [V,3], counts [V]).

    Mirrors the page's Python entry point: outputs are pre-allocated at
    max_voxels rows, the call runs without autograd, and the results are
    sliced to the real pillar count (which costs one 4-byte device read).
    """
    torch = _torch()
    with torch.no_grad():
        out = alloc_outputs(max_points, max_voxels, points.device)
        voxelize_into(points, point_cloud_range, voxel_size, max_points, max_voxels, out, stream, **opts)
        V = int(out[3].item())
        if V < 0:
            raise PVError(V, "pv_voxelize (device)")
        return out[0][:V], out[1][:V], out[2][:V]


_vec_cache = {}


def _vec(seq, n: int):
    """ctypes float[n] of a range or voxel size, cached by value (read-only on the C side)."""
    key = (seq if type(seq) is tuple else tuple(float(x) for x in seq), n)
    arr = _vec_cache.get(key)
    if arr is None:
        arr = _f6(key[0], n)
        if len(_vec_cache) < 256:
            _vec_cache[key] = arr
    return arr


def _host_ptr(a) -> int:
    """Address of a contiguous host array: a NumPy array or a CPU torch tensor."""
    if hasattr(a, "data_ptr"):
        if a.is_cuda or not a.is_contiguous():
            raise ValueError("host buffers must be contiguous CPU tensors or NumPy arrays")
        return a.data_ptr()
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("output arrays must be C-contiguous")
    return a.ctypes.data


def voxelize_host(points, point_cloud_range, voxel_size, max_points: int = 32, max_voxels: int = 16000,
                  out=None, stream=None):
    """Voxelize a host cloud (NumPy or CPU torch, [N, 4] float32) through pv_voxelize_host.

    Runs on the current CUDA device and writes the first V rows of ``out``
    (NumPy arrays or CPU torch tensors of max_voxels rows); rows past V are
    left as they were.  Returns (voxels, coords, counts, V): with ``out``
    given, its buffers themselves (the result is their first V rows: no
    slicing here, which would cost a few microseconds a call on torch
    tensors); with ``out`` None, NumPy arrays allocated here, sliced to
    [V,K,4], [V,3] and [V].  Pinned buffers (for example ``torch.empty(..).pin_memory()``) are read
    and written in place by the kernel; other host memory is staged on the
    device.
    """
    import numpy as np

    if hasattr(points, "data_ptr"):
        if points.dtype.itemsize != 4 or not points.is_floating_point() or points.is_cuda:
            raise TypeError("points must be a float32 CPU tensor")
        n = int(points.numel()) // 4
        pts_ptr = _host_ptr(points) if n else 0
    else:
        pts = np.ascontiguousarray(np.asarray(points, dtype=np.float32)).reshape(-1, 4)
        n = int(pts.shape[0])
        pts_ptr = pts.ctypes.data if n else 0
    own = out is None
    if own:
        out = (np.empty((max_voxels, max_points, 4), np.float32), np.empty((max_voxels, 3), np.int32),
               np.empty((max_voxels,), np.int32), np.empty((1,), np.int32))
    vox, coords, counts, num = out
    handle = 0 if stream is None else (stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    num_ptr = _host_ptr(num)
    st = load().pv_voxelize_host(pts_ptr, n, _vec(point_cloud_range, 6), _vec(voxel_size, 3), int(max_points),
                                 int(max_voxels), _host_ptr(vox), _host_ptr(coords), _host_ptr(counts), num_ptr,
                                 handle)
    if st != 0:
        raise PVError(st, "pv_voxelize_host")
    V = ctypes.c_int32.from_address(num_ptr).value
    if own:
        return vox[:V], coords[:V], counts[:V], V
    return vox, coords, counts, V


def alloc_batch_outputs(num_frames: int, max_points: int, max_voxels: int, device):
    """Outputs of a batched call: voxels [B, M, K, 4], coords [B, M, 4] (batch, z, y, x),
    counts [B, M], num [B]."""
    torch = _torch()
    return (torch.empty((num_frames, max_voxels, max_points, 4), dtype=torch.float32, device=device),
            torch.empty((num_frames, max_voxels, 4), dtype=torch.int32, device=device),
            torch.empty((num_frames, max_voxels), dtype=torch.int32, device=device),
            torch.empty((num_frames,), dtype=torch.int32, device=device))


def voxelize_batch_into(points, frame_offsets, point_cloud_range, voxel_size, max_points: int, max_voxels: int,
                        out, stream=None) -> None:
    """Enqueue one batched voxelization (frame b = points[off[b]:off[b+1]]) into
    pre-allocated outputs (see :func:`alloc_batch_outputs`); no synchronization."""
    torch = _torch()
    off = [int(o) for o in frame_offsets]
    B = len(off) - 1
    vox, coords, counts, num = out
    if not isinstance(points, torch.Tensor) or points.dtype != torch.float32 or not points.is_cuda:
        raise TypeError("points must be a float32 CUDA tensor")
    if points.dim() != 2 or points.shape[1] != 4 or not points.is_contiguous():
        raise ValueError("points must be a contiguous [N, 4] tensor")
    if B < 1 or off[-1] != points.shape[0]:
        raise ValueError("frame_offsets must hold num_frames + 1 offsets ending at N")
    for t, dt, shape in ((vox, torch.float32, (B, max_voxels, max_points, 4)),
                         (coords, torch.int32, (B, max_voxels, 4)),
                         (counts, torch.int32, (B, max_voxels)), (num, torch.int32, (B,))):
        if t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous() or t.device != points.device:
            raise ValueError("output tensor has the wrong dtype, shape, layout or device")
    if stream is None:
        stream = torch.cuda.current_stream(points.device)
    handle = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    offs = (ctypes.c_int64 * (B + 1))(*off)
    st = load().pv_voxelize_batch(
        ctypes.c_void_p(points.data_ptr() if points.shape[0] else 0), offs, B,
        _f6(point_cloud_range, 6), _f6(voxel_size, 3), int(max_points), int(max_voxels),
        ctypes.c_void_p(vox.data_ptr()), ctypes.c_void_p(coords.data_ptr()),
        ctypes.c_void_p(counts.data_ptr()), ctypes.c_void_p(num.data_ptr()), handle)
    if st != 0:
        raise PVError(st, "pv_voxelize_batch")


def voxelize_batch(points, frame_offsets, point_cloud_range, voxel_size, max_points: int = 32,
                   max_voxels: int = 16000, stream=None):
    """Voxelize a batch of frames in one launch.  Returns the batched
    PointPillars tensors, frames concatenated: voxels [sum V, K, 4], coords
    [sum V, 4] (batch, z, y, x), counts [sum V]."""
    torch = _torch()
    B = len(frame_offsets) - 1
    with torch.no_grad():
        out = alloc_batch_outputs(B, max_points, max_voxels, points.device)
        voxelize_batch_into(points, frame_offsets, point_cloud_range, voxel_size, max_points, max_voxels, out, stream)
        Vs = out[3].tolist()
        if any(v < 0 for v in Vs):
            raise PVError(min(Vs), "pv_voxelize_batch (device)")
        return (torch.cat([out[0][b, :v] for b, v in enumerate(Vs)]),
                torch.cat([out[1][b, :v] for b, v in enumerate(Vs)]),
                torch.cat([out[2][b, :v] for b, v in enumerate(Vs)]))


def alloc_downsample_outputs(max_voxels: int, device):
    """Outputs of a downsampling call: centroids [M, 4] f32, coords [M, 3] i32, counts [M] i32, num [1] i32."""
    torch = _torch()
    return (torch.empty((max_voxels, 4), dtype=torch.float32, device=device),
            torch.empty((max_voxels, 3), dtype=torch.int32, device=device),
            torch.empty((max_voxels,), dtype=torch.int32, device=device),
            torch.empty((1,), dtype=torch.int32, device=device))


def downsample_into(points, point_cloud_range, voxel_size, max_voxels: int, out, stream=None) -> None:
    """Enqueue one voxel-grid centroid downsampling into pre-allocated outputs."""
    torch = _torch()
    cen, coords, counts, num = out
    if not isinstance(points, torch.Tensor) or points.dtype != torch.float32 or not points.is_cuda:
        raise TypeError("points must be a float32 CUDA tensor")
    if points.dim() != 2 or points.shape[1] != 4 or not points.is_contiguous():
        raise ValueError("points must be a contiguous [N, 4] tensor")
    for t, dt, shape in ((cen, torch.float32, (max_voxels, 4)), (coords, torch.int32, (max_voxels, 3)),
                         (counts, torch.int32, (max_voxels,)), (num, torch.int32, (1,))):
        if t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous() or t.device != points.device:
            raise ValueError("output tensor has the wrong dtype, shape, layout or device")
    if stream is None:
        stream = torch.cuda.current_stream(points.device)
    handle = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    st = load().pv_voxel_downsample(
        ctypes.c_void_p(points.data_ptr() if points.shape[0] else 0), int(points.shape[0]),
        _f6(point_cloud_range, 6), _f6(voxel_size, 3), int(max_voxels), ctypes.c_void_p(cen.data_ptr()),
        ctypes.c_void_p(coords.data_ptr()), ctypes.c_void_p(counts.data_ptr()), ctypes.c_void_p(num.data_ptr()),
        handle)
    if st != 0:
        raise PVError(st, "pv_voxel_downsample")


def downsample(points, point_cloud_range, voxel_size, max_voxels: int = 1 << 20, stream=None):
    """Voxel-grid centroid downsampling on the points' GPU.  Returns
    (centroids [V, 4], coords [V, 3], counts [V])."""
    torch = _torch()
    with torch.no_grad():
        out = alloc_downsample_outputs(max_voxels, points.device)
        downsample_into(points, point_cloud_range, voxel_size, max_voxels, out, stream)
        V = int(out[3].item())
        if V < 0:
            raise PVError(V, "pv_voxel_downsample (device)")
        return out[0][:V], out[1][:V], out[2][:V]


def fps_into(points, num_samples: int, out_indices, out_samples=None, out_status=None, start: int = 0,
             stream=None) -> None:
    """Enqueue farthest point sampling of one cloud [N, 4] or a batch [B, N, 4]
    into out_indices ([M] or [B, M] int32) and optionally out_samples
    ([.., M, 4] float32).  out_status (one int32, device) receives 0 or a
    negative status; it is allocated and checked by :func:`fps` when not given."""
    torch = _torch()
    if not isinstance(points, torch.Tensor) or points.dtype != torch.float32 or not points.is_cuda:
        raise TypeError("points must be a float32 CUDA tensor")
    if points.dim() not in (2, 3) or points.shape[-1] != 4 or not points.is_contiguous():
        raise ValueError("points must be a contiguous [N, 4] or [B, N, 4] tensor")
    B = 1 if points.dim() == 2 else int(points.shape[0])
    N = int(points.shape[-2])
    M = int(num_samples)
    want = (M,) if points.dim() == 2 else (B, M)
    if out_indices.dtype != torch.int32 or tuple(out_indices.shape) != want or not out_indices.is_contiguous():
        raise ValueError("out_indices has the wrong dtype, shape or layout")
    if out_samples is not None and (out_samples.dtype != torch.float32 or tuple(out_samples.shape) != want + (4,)
                                    or not out_samples.is_contiguous()):
        raise ValueError("out_samples has the wrong dtype, shape or layout")
    if out_status is None or out_status.dtype != torch.int32 or out_status.numel() != 1:
        raise ValueError("out_status must be one int32 on the device")
    if stream is None:
        stream = torch.cuda.current_stream(points.device)
    handle = ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    st = load().pv_fps(ctypes.c_void_p(points.data_ptr()), B, N, M, int(start),
                       ctypes.c_void_p(out_indices.data_ptr()),
                       ctypes.c_void_p(out_samples.data_ptr() if out_samples is not None else 0),
                       ctypes.c_void_p(out_status.data_ptr()), handle)
    if st != 0:
        raise PVError(st, "pv_fps")


def fps(points, num_samples: int, start: int = 0, return_samples: bool = False, stream=None):
    """Farthest point sampling (exact; ties to the lowest index).  Returns the
    sample indices ([M] or [B, M] int32) and, if asked, the sampled points."""
    torch = _torch()
    with torch.no_grad():
        lead = () if points.dim() == 2 else (int(points.shape[0]),)
        idx = torch.empty(lead + (int(num_samples),), dtype=torch.int32, device=points.device)
        smp = (torch.empty(lead + (int(num_samples), 4), dtype=torch.float32, device=points.device)
               if return_samples else None)
        status = torch.empty((1,), dtype=torch.int32, device=points.device)
        fps_into(points, num_samples, idx, smp, status, start, stream)
        st = int(status.item())
        if st != 0:
            raise PVError(st, "pv_fps (device)")
        return (idx, smp) if return_samples else idx
