"""GB300-native pillar voxelization (PointPillars preprocessing).

The CUDA library ``libpv.so`` (C ABI in ``include/pv.h``) does the work; this
package is its thin Python binding plus seeded synthetic inputs
(:mod:`lidar_point_cloud_gb300.synth`).
"""

from ._binding import (  # noqa: F401
    EXPORTS,
    FPS_MAX_POINTS,
    MAX_FRAMES,
    PVError,
    alloc_batch_outputs,
    alloc_downsample_outputs,
    alloc_outputs,
    downsample,
    downsample_into,
    fps,
    fps_into,
    grid_size,
    lib_path,
    load,
    query_plan,
    release_workspace,
    voxelize,
    voxelize_batch,
    voxelize_batch_into,
    voxelize_host,
    voxelize_into,
)

__version__ = "0.1.0"
