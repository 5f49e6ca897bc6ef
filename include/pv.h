/*
 * pv.h - C ABI of the GB300 pillar voxelizer (libpv.so).
 *
 * The operation is the one described on the page "Voxelize"
 * (ethan-howes.github.io/projects/voxelize/): an unordered [N, 4] float32
 * LiDAR cloud (x, y, z, intensity) becomes the three PointPillars tensors,
 * a [V, max_points, 4] stack of per-pillar points, [V, 3] int32 pillar
 * coordinates (z = 0, y, x) and [V] int32 per-pillar point counts.
 *
 * Semantics, section by section of that page:
 *   "Implementation > Binning a point": a point is dropped if x, y or z is
 *     NaN or +-Inf; its cell on each axis is floorf((c - c_min) / v_c), with
 *     the subtraction and the division each one IEEE binary32 operation
 *     rounded to nearest (no fast-math, no flush of subnormals); a point is
 *     dropped unless 0 <= cell < grid on every axis (a strict < on the upper
 *     bound, so a point exactly on x_max is excluded; z outside the slab is
 *     dropped the same way).  The pillar id is cy * grid_x + cx.
 *   True 3-D voxels (grid_z > 1): the same rule on z gives cz, the voxel id
 *     is (cz * grid_y + cy) * grid_x + cx and the coordinates are
 *     (cz, cy, cx), as the voxel-grid downsampling kernel of the cuda-kdtree
 *     ICP page ("4.4", voxel_downsample) bins all three axes.  Everything
 *     else below holds per voxel; with grid_z == 1 it is the pillar case.
 *   "Claiming a pillar and packing points": one pillar per distinct id, with
 *     coordinates (0, id / grid_x, id % grid_x); at most max_points points
 *     per pillar ("keep the first K"); the intensity is copied bit for bit.
 *   "Compaction" and "The PyTorch side": pillars are compacted into dense
 *     outputs pre-allocated at max_voxels rows; V is the real pillar count.
 *   Order (the page's hash-slot order varies from run to run, "Results";
 *     this library fixes it): pillars in ascending order of their
 *     lowest-index valid point, points inside a pillar in index order, the
 *     first max_points points of each pillar and the first max_voxels pillars
 *     kept.  Every output byte is written: rows past a pillar's count and
 *     pillars past V are zero.  The result is therefore unique and
 *     bit-reproducible.
 *
 * Grid extents: grid_c = round((max_c - min_c) / v_c), computed in double
 * and rounded half away from zero (432 x 496 for the page's 0.16 m cells over
 * [0, 69.12] x [-39.68, 39.68], "Fig. 2").  Each of grid_x, grid_y, grid_z
 * must be <= 2^24 and grid_x * grid_y * grid_z < 2^31.
 *
 * Errors: a status found on the host is returned and nothing is enqueued;
 * *out_num_voxels is then left untouched.  A status found on the device is
 * written, negative, into *out_num_voxels in place of V; the other outputs
 * are then unspecified.
 */
#ifndef PV_H_
#define PV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* pv_stream_t;

typedef enum pv_status {
  PV_OK = 0,
  PV_ERR_INVALID = -1,     /* bad argument: null/misaligned pointer, host pointer where a
                              device pointer is needed, non-finite or non-positive cell
                              size, max <= min, size out of range */
  PV_ERR_UNSUPPORTED = -2, /* a request this build does not support (a device index past
                              the allocation-free entry point's table) */
  PV_ERR_ALLOC = -3,       /* the library's device workspace could not be allocated */
  PV_ERR_CUDA = -4,        /* a CUDA runtime call failed (launch, copy, ...) */
  PV_ERR_CAPACITY = -5,    /* device: the pillar table ran out of slots (only with a
                              forced undersized table, see pv_options) */
  PV_ERR_TIMEOUT = -6,     /* device: a bounded wait inside the kernel gave up (about
                              one second); the workspace is then fully reset by the
                              next call on the same stream */
  PV_ERR_INTERNAL = -7,    /* device: a consistency check failed (a point index read
                              from the pillar table was out of range); the workspace is
                              fully reset by the next call on the same stream */
  PV_ERR_TOO_LARGE = -8    /* pv_voxelize_static only: more points or a larger
                              max_points than its fixed scratch holds */
} pv_status;

/* Largest max_points accepted. */
#define PV_MAX_POINTS_LIMIT 1024

/*
 * pv_voxelize - voxelize one cloud, asynchronously on `stream`.
 *
 *   points          device, [num_points, 4] float32 row-major (x, y, z, intensity),
 *                   16-byte aligned; may be NULL when num_points == 0.  Read only.
 *   num_points      0 <= num_points < 2^29.
 *   point_cloud_range  host, {x_min, y_min, z_min, x_max, y_max, z_max}.
 *   voxel_size      host, {v_x, v_y, v_z}, finite and > 0.
 *   max_points      points kept per pillar, 1..PV_MAX_POINTS_LIMIT (PointPillars: 32).
 *   max_voxels      pillars kept, >= 1, max_voxels * max_points < 2^31.
 *   out_voxels      device, [max_voxels, max_points, 4] float32, 16-byte aligned.
 *   out_coords      device, [max_voxels, 3] int32, (z, y, x); z = 0 on a pillar grid.
 *   out_counts      device, [max_voxels] int32.
 *   out_num_voxels  device, one int32: V (>= 0) or a negative pv_status.
 *   stream          CUDA stream the work is enqueued on.
 *
 * All pointers belong to the caller and must be device memory of one device;
 * the call runs on that device.  Outputs are fully overwritten.  The call
 * does not synchronize: V is read back by the caller when it needs it.
 * The library keeps a grow-only workspace per (device, stream); calls on one
 * stream run one after another, calls on different streams do not share
 * state.  A call that grows the workspace synchronizes the stream once.
 * Returns PV_OK or a negative pv_status found on the host.
 */
int pv_voxelize(const float* points, int64_t num_points, const float point_cloud_range[6],
                const float voxel_size[3], int max_points, int max_voxels, float* out_voxels,
                int32_t* out_coords, int32_t* out_counts, int32_t* out_num_voxels,
                pv_stream_t stream);

/*
 * Options of pv_voxelize_ex.  Zero in any field means "use the library's
 * choice".  Apart from `order`, the result never depends on these settings.
 *   order        0 the canonical order (the contract above); 1 the page's own
 *                unordered contract ("The hash slot is the output index",
 *                "Claiming a pillar and packing points", "Compaction"): the
 *                same pillar set and counts, but pillars in whatever order
 *                they were created, the points of a pillar in arrival order,
 *                and, where a cap binds, whichever max_points points and
 *                max_voxels pillars arrived first.  Zero padding as above.
 *                The result may differ from run to run; the page checks its
 *                own kernel the same way ("Results": sort by (z, y, x), then
 *                compare the pillar sets and counts).
 *   table_mode   0 auto, 1 direct (one slot per grid cell), 2 hashed (open
 *                addressing, linear probing).
 *   table_log2   hashed mode only: force 2^table_log2 slots.  A table smaller
 *                than the number of distinct pillars makes the call fail with
 *                PV_ERR_CAPACITY (used by the tests of that error path).
 *   ctas_per_sm  resident blocks per SM of the single cooperative launch
 *                (capped at what fits).
 *   test_stall_barrier  for tests of the timeout path only (see the field).
 */
typedef struct pv_options {
  int table_mode;
  int table_log2;
  int ctas_per_sm;
  int test_stall_barrier;  /* test hook: nonzero makes the first grid barrier wait for
                              one arrival that never comes, so the bounded wait runs out
                              (about 1 s) and the call reports PV_ERR_TIMEOUT */
  int order;
  int reserved[3];
} pv_options;

/*
 * A batch of frames in one launch.  Frame b is points[frame_offsets[b] ..
 * frame_offsets[b + 1]) and is voxelized exactly as pv_voxelize voxelizes it
 * alone (same grid, max_points and max_voxels per frame; canonical order
 * inside the frame).  Batching spreads one launch and its grid barriers over
 * many small frames; the page measures that a frame's cost is dominated by
 * that fixed overhead ("voxelize latency vs point count", Tab. 2).
 *   points          device, [frame_offsets[num_frames], 4] float32, 16-byte aligned.
 *   frame_offsets   HOST, [num_frames + 1] int64: 0, then never decreasing (empty
 *                   frames allowed); read before the call returns.
 *   num_frames      1 .. PV_MAX_FRAMES.
 *   out_voxels      device, [num_frames, max_voxels, max_points, 4] float32.
 *   out_coords      device, [num_frames, max_voxels, 4] int32, (batch, z, y, x):
 *                   the batched PointPillars layout; rows past a frame's V are zero.
 *   out_counts      device, [num_frames, max_voxels] int32.
 *   out_num_voxels  device, [num_frames] int32: V of each frame, or the (same)
 *                   negative status in every entry.
 * num_frames * (grid voxels) must stay below 2^31, and num_frames *
 * max_voxels * max_points below 2^31.  Errors, ownership and streams as for
 * pv_voxelize.
 */
#define PV_MAX_FRAMES 256
int pv_voxelize_batch(const float* points, const int64_t* frame_offsets, int num_frames,
                      const float point_cloud_range[6], const float voxel_size[3], int max_points, int max_voxels,
                      float* out_voxels, int32_t* out_coords, int32_t* out_counts, int32_t* out_num_voxels,
                      pv_stream_t stream);

/*
 * Voxel-grid centroid downsampling.  The cuda-kdtree ICP page ("4.4",
 * voxel_downsample) replaces the voxel-grid filter: every occupied voxel
 * becomes one point, the centroid of the points in it.  Cells follow the
 * binning rule above on all three axes (any grid_z); voxels are in the
 * canonical order (first point), the first max_voxels kept.  Every point of a
 * kept voxel counts (no per-voxel cap).  A centroid is (mean x, mean y,
 * mean z, mean intensity): the defining computation is a double sum in index
 * order divided by the count in double and rounded to float.  The library
 * accumulates in parallel with at least that precision (float-float sums of
 * each warp's points, then double sums) and divides in float-float, so a mean
 * may differ from the definition by one float32 unit in the last place (for
 * the points of a voxel of one sign, as LiDAR cells are unless they straddle
 * a coordinate plane through the origin); counts, coordinates, V and the
 * order are exact.
 *   out_centroids   device, [max_voxels, 4] float32, 16-byte aligned.
 *   out_coords      device, [max_voxels, 3] int32, (z, y, x).
 *   out_counts      device, [max_voxels] int32, points per voxel.
 *   out_num_voxels  device, one int32: V or a negative status.
 * Rows past V are zero.  Errors, ownership and streams as for pv_voxelize.
 */
int pv_voxel_downsample(const float* points, int64_t num_points, const float point_cloud_range[6],
                        const float voxel_size[3], int max_voxels, float* out_centroids, int32_t* out_coords,
                        int32_t* out_counts, int32_t* out_num_voxels, pv_stream_t stream);

/*
 * Farthest point sampling, the operation the RadiusFPS page accelerates
 * ("Baseline: classic GPU FPS"; its spherical-voxel pruning skips only
 * updates that cannot change a distance, so the samples are those of plain
 * FPS).  From point `start`, every point keeps its smallest squared distance
 * to the samples so far, ((dx*dx) + (dy*dy)) + (dz*dz) in float rounded to
 * nearest (intensity ignored); the next sample is the point with the largest
 * one, ties to the lowest index.  The result is unique and bit-reproducible.
 *   points        device, [num_clouds, num_points, 4] float32, 16-byte aligned;
 *                 x, y, z finite (else *out_status = PV_ERR_INVALID).
 *   num_points    points per cloud, 1 .. PV_FPS_MAX_POINTS.
 *   num_samples   samples per cloud, >= 1 (past the distinct points the
 *                 remaining distances are 0 and the lowest index repeats).
 *   start         first sample, 0 .. num_points - 1 (PointNet++ takes 0).
 *   out_indices   device, [num_clouds, num_samples] int32, indices inside each cloud.
 *   out_samples   device, [num_clouds, num_samples, 4] float32 copies of the
 *                 sampled points, or NULL.
 *   out_status    device, one int32: 0, or a negative status found on the device.
 * Returns PV_OK or a negative status found on the host (nothing enqueued).
 * Each cloud runs in one thread-block cluster holding it on chip (16 CTAs
 * while the launch's clouds fit on the GPU at once in such clusters, else 8;
 * clouds of more than 106,496 points always take 16, and on a device
 * without 16-CTA clusters return PV_ERR_UNSUPPORTED); clouds run side by side.
 */
#define PV_FPS_MAX_POINTS 212992
int pv_fps(const float* points, int num_clouds, int64_t num_points, int64_t num_samples, int64_t start,
           int32_t* out_indices, float* out_samples, int32_t* out_status, pv_stream_t stream);

int pv_voxelize_ex(const float* points, int64_t num_points, const float point_cloud_range[6],
                   const float voxel_size[3], int max_points, int max_voxels, float* out_voxels,
                   int32_t* out_coords, int32_t* out_counts, int32_t* out_num_voxels,
                   const pv_options* options, pv_stream_t stream);

/*
 * pv_voxelize_host - the same operation on HOST buffers, synchronous.
 *
 * Runs pv_voxelize on `stream` for a cloud in host memory, writes the first
 * V rows of the three row outputs (each voxel row zero-padded past its
 * count, as pv_voxelize writes it) and V itself, and waits for the stream.
 * Rows V .. max_voxels-1 of the host buffers are left as they were: the
 * result is the outputs sliced to the pillar count, as the page's Python
 * entry point returns them ("Voxelize" > "The PyTorch side"), and no zero row
 * crosses the host link.  Pinned buffers (page-locked and mapped: cudaHostAlloc,
 * cudaHostRegister) aligned as pv_voxelize requires (16 bytes for points and
 * voxels, 4 for the rest) are used in place: the kernel reads the points and
 * writes the outputs across the host link.  Any other host buffer (pageable,
 * or less aligned) goes through a device copy in the library's per-(device,
 * stream) workspace, copied in before or out after the kernel.
 * Returns PV_OK, a host-side error, or the negative status the device wrote
 * (then *out_num_voxels_host holds it too).
 */
int pv_voxelize_host(const float* points_host, int64_t num_points, const float point_cloud_range[6],
                     const float voxel_size[3], int max_points, int max_voxels,
                     float* out_voxels_host, int32_t* out_coords_host, int32_t* out_counts_host,
                     int32_t* out_num_voxels_host, pv_stream_t stream);

/*
 * pv_voxelize_static - pv_voxelize without any device allocation.
 *
 * The page has no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory while they run: code being recorded
 * into a CUDA graph under global capture mode (where cudaMalloc is not
 * allowed), inference plug-ins whose host owns all device memory, and
 * real-time pipelines that forbid allocation after start-up.  It takes the
 * same arguments and gives the same result as pv_voxelize, but its scratch
 * (table, per-point arrays, control block) lives in one fixed array of
 * 18,419,968 bytes (about 17.6 MiB) of device memory, declared in the library at file scope:
 * every GPU that loads the library holds it until the process exits.  The
 * caller still owns and passes the input and the outputs.
 *
 * Limits: num_points <= 32768 and max_points <= 32; beyond either the call
 * returns PV_ERR_TOO_LARGE and enqueues nothing.  The table is always the
 * hashed kind, with at most 2^16 slots.
 *
 * The first call on a device sets that device up: it looks up the array's
 * device address, sets the kernel's shared-memory attribute and enqueues
 * one memset of the array on `stream`.  Make that first call before any
 * stream capture.  Every call on every stream of a device shares the one
 * array, which keeps the state the last call left (the kernel empties its
 * table and rearms its control block before it ends), so calls must not
 * overlap on the GPU: calls on one stream are safe, calls on different
 * streams race unless the caller orders them.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 */
int pv_voxelize_static(const float* points, int64_t num_points, const float point_cloud_range[6],
                       const float voxel_size[3], int max_points, int max_voxels, float* out_voxels,
                       int32_t* out_coords, int32_t* out_counts, int32_t* out_num_voxels,
                       pv_stream_t stream);

/* Grid extents for a range and a cell size: PV_OK, PV_ERR_INVALID or
 * PV_ERR_UNSUPPORTED, with grid_out = {grid_x, grid_y, grid_z}. */
int pv_grid_size(const float point_cloud_range[6], const float voxel_size[3], int64_t grid_out[3]);

/* What pv_voxelize would launch for these sizes on the current device. */
typedef struct pv_plan {
  int64_t grid[3];          /* pillar grid extents */
  int table_mode;           /* 1 direct, 2 hashed */
  int64_t table_slots;      /* pillar slots in the table */
  int list_stride;          /* 64-bit list entries per slot: a head row of 4, plus a tail
                               row of max_points rounded up to 4, less 4 */
  int ctas;                 /* blocks of the cooperative launch */
  int threads;              /* threads per block */
  int64_t points_per_cta;   /* contiguous points each block owns */
  int64_t workspace_bytes;  /* device workspace the call needs */
} pv_plan;

int pv_query_plan(int64_t num_points, const float point_cloud_range[6], const float voxel_size[3],
                  int max_points, int max_voxels, const pv_options* options, pv_plan* plan_out);

/* Frees every cached workspace of every device and stream (waits for them
 * to be idle first).  Returns PV_OK or PV_ERR_CUDA. */
int pv_release_workspace(void);

/* Static, human-readable name of a status. */
const char* pv_status_string(int status);

/* Library version, "major.minor.patch". */
const char* pv_version(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* PV_H_ */
