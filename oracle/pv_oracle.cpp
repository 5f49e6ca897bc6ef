// Pillar-voxelization oracle: plain, sequential, single-threaded C++.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link or
// call this file: only the test suite, the smoke check and the benchmark's
// CPU-baseline leg use it. It shares no code, header, table or constant with
// the CUDA library; the status codes below are restated from the public
// contract, not included from it.
//
// What it computes follows the page "Voxelize" (ethan-howes.github.io/
// projects/voxelize/):
//   * "Implementation > Binning a point": NaN/Inf points are dropped, the
//     cell is floorf((c - c_min) / v_c) per axis, a cell outside [0, grid)
//     (strict < on the upper bound) drops the point, the pillar id is
//     cy * grid_x + cx.
//   * "Claiming a pillar and packing points": one pillar per distinct id,
//     coordinates (0, id / grid_x, id % grid_x), points past max_points are
//     dropped ("keep the first K").
//   * "Results": the CPU reference assigns pillars with a dictionary in one
//     sequential pass.  That sequential pass is written out here with a
//     std::map, which fixes the canonical order: pillars in order of their
//     first (lowest-index) valid point, points inside a pillar in index
//     order, the first max_voxels pillars kept, zero padding everywhere else.
//   * "The PyTorch side": outputs are pre-allocated at [max_voxels, ...] and
//     the caller slices them to the real pillar count V.
//
// Floating point: IEEE-754 binary32, round-to-nearest-even, no flush of
// subnormals, no contraction.  The build uses -O2 -fno-fast-math
// -ffp-contract=off; on x86-64 (SSE) and AArch64 `float` arithmetic is plain
// binary32, so each subtraction and division below is one correctly rounded
// operation.
//
// Parity is pinned (see tests/test_oracle_pins.py) by the grid size the page
// prints, a hand-derived table of boundary points, a hand-worked example,
// an O(N^2) brute force, a NumPy stable-sort restatement and invariants.

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <vector>

namespace {

// Status values of the public contract, restated (not shared) here.
constexpr int kOk = 0;
constexpr int kErrInvalid = -1;
constexpr int kErrUnsupported = -2;

// Largest grid extent per axis.  Keeps every grid size exactly representable
// as a float, so the "cell < grid" test is exact.
constexpr int64_t kMaxAxisCells = int64_t(1) << 24;

bool is_finite_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  return (u & 0x7f800000u) != 0x7f800000u;  // exponent all ones = NaN or Inf
}

// Grid extent along one axis: the range length divided by the cell size,
// rounded to the nearest integer in double precision.  With the page's
// 0.16 m cells over [0, 69.12] x [-39.68, 39.68] this gives 432 x 496, i.e.
// the 214,272 pillars the page prints ("Fig. 2").  The float quotient
// 69.12f / 0.16f is 432.00003, so a ceiling would give 433; rounding is the
// reading that reproduces the page.
int64_t axis_cells(float lo, float hi, float v) {
  double len = static_cast<double>(hi) - static_cast<double>(lo);
  return static_cast<int64_t>(std::llround(len / static_cast<double>(v)));
}

// Cell index of one coordinate ("Binning a point"): floorf of the IEEE
// quotient, with the bounds tested on the float cell before any integer
// conversion (a huge or infinite quotient can never reach the cast).
bool bin_axis(float c, float lo, float v, int64_t cells, int64_t* out) {
  float d = c - lo;      // one binary32 subtraction, rounded to nearest
  float q = d / v;       // one binary32 division, rounded to nearest
  float f = std::floor(q);
  if (!(f >= 0.0f)) return false;                        // below the origin
  if (!(f < static_cast<float>(cells))) return false;    // strict upper bound
  *out = static_cast<int64_t>(f);
  return true;
}

}  // namespace

extern "C" {

// Grid extents (x, y, z) for a range and a cell size, with the argument
// checks of the public contract.  Returns kOk, kErrInvalid or
// kErrUnsupported (a z extent other than one pillar).
int pv_oracle_grid(const float range[6], const float voxel_size[3],
                   int64_t grid_out[3]) {
  for (int a = 0; a < 3; ++a) {
    float lo = range[a], hi = range[a + 3], v = voxel_size[a];
    if (!std::isfinite(lo) || !std::isfinite(hi) || !std::isfinite(v))
      return kErrInvalid;
    if (!(v > 0.0f) || !(hi > lo)) return kErrInvalid;
    int64_t g = axis_cells(lo, hi, v);
    if (g < 1 || g > kMaxAxisCells) return kErrInvalid;
    grid_out[a] = g;
  }
  if (grid_out[0] * grid_out[1] >= (int64_t(1) << 31)) return kErrInvalid;
  if (grid_out[2] != 1) return kErrUnsupported;
  return kOk;
}

// Cell of one point: writes (cx, cy, cz) and returns 1 if the point lands
// inside the grid, 0 if it is dropped.  Exposed so the tests can check the
// binning rule point by point against the hand-derived boundary table.
int pv_oracle_bin_point(const float p[4], const float range[6],
                        const float voxel_size[3], const int64_t grid[3],
                        int64_t cell_out[3]) {
  // "checks for NaN/Inf": x, y and z only; the intensity is payload.
  if (!is_finite_bits(p[0]) || !is_finite_bits(p[1]) || !is_finite_bits(p[2]))
    return 0;
  for (int a = 0; a < 3; ++a)
    if (!bin_axis(p[a], range[a], voxel_size[a], grid[a], &cell_out[a]))
      return 0;
  return 1;
}

// The whole operation, one sequential pass in point-index order.
//   points       [N, 4] float32 row-major (x, y, z, intensity)
//   out_voxels   [max_voxels, max_points, 4] float32
//   out_coords   [max_voxels, 3] int32, (z = 0, y, x)
//   out_counts   [max_voxels] int32
//   out_num      number of pillars V written
// Every output element is written: zero wherever no point lands.
// With three_d the z cell is kept: voxel id (cz * grid_y + cy) * grid_x + cx
// and coordinates (cz, cy, cx); see pv_oracle_voxelize3d.
static int voxelize_pass(const float* points, int64_t N, const float range[6],
                         const float voxel_size[3], const int64_t grid[3],
                         int max_points, int max_voxels, float* out_voxels,
                         int32_t* out_coords, int32_t* out_counts,
                         int32_t* out_num, bool three_d) {
  const size_t row_floats = static_cast<size_t>(max_points) * 4;
  std::memset(out_voxels, 0,
              sizeof(float) * row_floats * static_cast<size_t>(max_voxels));
  std::memset(out_coords, 0, sizeof(int32_t) * 3 * static_cast<size_t>(max_voxels));
  std::memset(out_counts, 0, sizeof(int32_t) * static_cast<size_t>(max_voxels));

  std::map<int64_t, int32_t> pillar;  // pillar (or voxel) id -> output row
  int32_t V = 0;
  for (int64_t i = 0; i < N; ++i) {
    const float* p = points + 4 * i;
    int64_t cell[3];
    if (!pv_oracle_bin_point(p, range, voxel_size, grid, cell)) continue;
    const int64_t id = three_d ? (cell[2] * grid[1] + cell[1]) * grid[0] + cell[0]
                               : cell[1] * grid[0] + cell[0];  // flattened pillar id
    auto it = pillar.find(id);
    int32_t r;
    if (it == pillar.end()) {
      // A new pillar is only opened while the budget lasts; once max_voxels
      // pillars exist, later pillars (and all of their points) are dropped.
      if (V >= max_voxels) continue;
      r = V++;
      pillar.emplace(id, r);
      if (three_d) {
        out_coords[3 * r + 0] = static_cast<int32_t>(cell[2]);
        out_coords[3 * r + 1] = static_cast<int32_t>(cell[1]);
        out_coords[3 * r + 2] = static_cast<int32_t>(cell[0]);
      } else {
        out_coords[3 * r + 0] = 0;  // pillars have no z extent
        out_coords[3 * r + 1] = static_cast<int32_t>(id / grid[0]);
        out_coords[3 * r + 2] = static_cast<int32_t>(id % grid[0]);
      }
    } else {
      r = it->second;
    }
    const int32_t k = out_counts[r];
    if (k >= max_points) continue;  // pillar full: keep the first K points
    std::memcpy(out_voxels + static_cast<size_t>(r) * row_floats +
                    static_cast<size_t>(k) * 4,
                p, 4 * sizeof(float));  // bitwise copy of the whole row
    out_counts[r] = k + 1;
  }
  *out_num = V;
  return kOk;
}

static int check_args(const float* points, int64_t N, int max_points, int max_voxels,
                      const float* out_voxels, const int32_t* out_coords,
                      const int32_t* out_counts, const int32_t* out_num) {
  if (N < 0 || N >= (int64_t(1) << 31) || max_points < 1 || max_voxels < 1)
    return kErrInvalid;
  if (N > 0 && points == nullptr) return kErrInvalid;
  if (!out_voxels || !out_coords || !out_counts || !out_num) return kErrInvalid;
  return kOk;
}

int pv_oracle_voxelize(const float* points, int64_t N, const float range[6],
                       const float voxel_size[3], int max_points,
                       int max_voxels, float* out_voxels, int32_t* out_coords,
                       int32_t* out_counts, int32_t* out_num) {
  int st = check_args(points, N, max_points, max_voxels, out_voxels, out_coords, out_counts, out_num);
  if (st != kOk) return st;
  int64_t grid[3];
  st = pv_oracle_grid(range, voxel_size, grid);
  if (st != kOk) return st;
  return voxelize_pass(points, N, range, voxel_size, grid, max_points, max_voxels,
                       out_voxels, out_coords, out_counts, out_num, false);
}

// Grid extents for true 3-D voxels: the checks of pv_oracle_grid without the
// pillar restriction on the z extent; the voxel count must stay below 2^31.
int pv_oracle_grid3d(const float range[6], const float voxel_size[3],
                     int64_t grid_out[3]) {
  for (int a = 0; a < 3; ++a) {
    float lo = range[a], hi = range[a + 3], v = voxel_size[a];
    if (!std::isfinite(lo) || !std::isfinite(hi) || !std::isfinite(v))
      return kErrInvalid;
    if (!(v > 0.0f) || !(hi > lo)) return kErrInvalid;
    int64_t g = axis_cells(lo, hi, v);
    if (g < 1 || g > kMaxAxisCells) return kErrInvalid;
    grid_out[a] = g;
  }
  if (grid_out[0] * grid_out[1] * grid_out[2] >= (int64_t(1) << 31))
    return kErrInvalid;
  return kOk;
}

// True 3-D voxels.  The page "Voxelize" hard-codes z = 0 because a pillar
// spans the whole z slab ("Claiming a pillar and packing points"); the
// voxel-grid downsampling kernel of the cuda-kdtree ICP page ("4.4",
// "voxel_downsample") bins all three axes.  This is the same sequential
// pass with the z cell kept: voxel id (cz * grid_y + cy) * grid_x + cx,
// coordinates (cz, cy, cx), the same binning rule on every axis (floorf,
// strict upper bound), the same canonical order, caps and zero padding.
// With grid_z == 1 it equals pv_oracle_voxelize.
int pv_oracle_voxelize3d(const float* points, int64_t N, const float range[6],
                         const float voxel_size[3], int max_points,
                         int max_voxels, float* out_voxels,
                         int32_t* out_coords, int32_t* out_counts,
                         int32_t* out_num) {
  int st = check_args(points, N, max_points, max_voxels, out_voxels, out_coords, out_counts, out_num);
  if (st != kOk) return st;
  int64_t grid[3];
  st = pv_oracle_grid3d(range, voxel_size, grid);
  if (st != kOk) return st;
  return voxelize_pass(points, N, range, voxel_size, grid, max_points, max_voxels,
                       out_voxels, out_coords, out_counts, out_num, true);
}

// Voxel-grid centroid downsampling: the cuda-kdtree ICP page ("4.4",
// voxel_downsample) replaces PCL's voxel-grid filter: every occupied voxel
// becomes one point, the centroid of the points that fall in it
// ("accumulate into the voxel centre", then a reduce by key).  Read here
// with the Voxelize binning rule on all three axes (floorf, strict upper
// bound, NaN/Inf dropped; the page's integer truncation would put points
// just below the origin in cell 0, which "Binning a point" on the Voxelize
// page rules out) and the canonical order (voxels by their first point, the
// first max_voxels kept).  Every point of a kept voxel counts (no per-voxel
// cap).  Per voxel: the four fields (x, y, z, intensity) summed in double
// precision in point-index order, each sum divided by the count in double,
// the quotient rounded to float.
//   out_centroids [max_voxels, 4] float32, out_coords [max_voxels, 3] int32
//   (z, y, x), out_counts [max_voxels] int32, out_num the voxel count V;
//   zeros past V.
int pv_oracle_downsample(const float* points, int64_t N, const float range[6],
                         const float voxel_size[3], int max_voxels,
                         float* out_centroids, int32_t* out_coords,
                         int32_t* out_counts, int32_t* out_num) {
  int st = check_args(points, N, 1, max_voxels, out_centroids, out_coords, out_counts, out_num);
  if (st != kOk) return st;
  int64_t grid[3];
  st = pv_oracle_grid3d(range, voxel_size, grid);
  if (st != kOk) return st;
  std::memset(out_centroids, 0, sizeof(float) * 4 * static_cast<size_t>(max_voxels));
  std::memset(out_coords, 0, sizeof(int32_t) * 3 * static_cast<size_t>(max_voxels));
  std::memset(out_counts, 0, sizeof(int32_t) * static_cast<size_t>(max_voxels));
  std::map<int64_t, int32_t> voxel;  // voxel id -> output row
  std::vector<double> sum(4 * static_cast<size_t>(max_voxels), 0.0);
  int32_t V = 0;
  for (int64_t i = 0; i < N; ++i) {
    const float* p = points + 4 * i;
    int64_t cell[3];
    if (!pv_oracle_bin_point(p, range, voxel_size, grid, cell)) continue;
    const int64_t id = cell[0] + grid[0] * (cell[1] + grid[1] * cell[2]);  // (cz * gy + cy) * gx + cx
    auto it = voxel.find(id);
    int32_t r;
    if (it == voxel.end()) {
      if (V >= max_voxels) continue;  // budget spent: this voxel is dropped
      r = V++;
      voxel.emplace(id, r);
      for (int a = 0; a < 3; ++a) out_coords[3 * r + a] = static_cast<int32_t>(cell[2 - a]);  // (z, y, x)
    } else {
      r = it->second;
    }
    for (int c = 0; c < 4; ++c) sum[4 * static_cast<size_t>(r) + c] += static_cast<double>(p[c]);
    out_counts[r] += 1;
  }
  for (int32_t r = 0; r < V; ++r)
    for (int c = 0; c < 4; ++c)
      out_centroids[4 * static_cast<size_t>(r) + c] =
          static_cast<float>(sum[4 * static_cast<size_t>(r) + c] / static_cast<double>(out_counts[r]));
  *out_num = V;
  return kOk;
}

// Farthest point sampling, the operation RadiusFPS accelerates (the RadiusFPS
// page: "Baseline: classic GPU FPS"; its spherical-voxel pruning skips only
// work that cannot change the result, so the samples are those of plain
// FPS).  Start at point `start`; every point keeps its smallest squared
// distance to the samples so far (the page's min_dist, starting above every
// distance); the next sample is the point with the largest such distance.
// Ties go to the lowest index (the page leaves tie-breaking open and notes
// it; fixing it makes the result unique).  The squared distance of the page's
// baseline kernel, (px-qx)^2 + (py-qy)^2 + (pz-qz)^2, is evaluated in float
// as ((dx * dx) + (dy * dy)) + (dz * dz), every operation rounded to nearest.
// Intensity is ignored.  Points must be finite (status kErrInvalid if not).
//   points [N, 4] float32; out_idx [M] int32.
int pv_oracle_fps(const float* points, int64_t N, int64_t M, int64_t start,
                  int32_t* out_idx) {
  if (N < 1 || N >= (int64_t(1) << 31) || M < 1 || start < 0 || start >= N)
    return kErrInvalid;
  if (!points || !out_idx) return kErrInvalid;
  for (int64_t i = 0; i < N; ++i)
    for (int c = 0; c < 3; ++c)
      if (!is_finite_bits(points[4 * i + c])) return kErrInvalid;
  std::vector<float> min_dist(static_cast<size_t>(N), INFINITY);
  int64_t sel = start;
  for (int64_t k = 0; k < M; ++k) {
    out_idx[k] = static_cast<int32_t>(sel);
    const float qx = points[4 * sel], qy = points[4 * sel + 1], qz = points[4 * sel + 2];
    int64_t best = 0;
    float best_d = -1.0f;  // below every distance: index 0 wins if all are zero
    for (int64_t i = 0; i < N; ++i) {
      const float dx = points[4 * i] - qx;
      const float dy = points[4 * i + 1] - qy;
      const float dz = points[4 * i + 2] - qz;
      const float d = (dx * dx + dy * dy) + dz * dz;
      min_dist[i] = std::min(min_dist[i], d);  // each point's distance to its nearest sample so far
      if (min_dist[i] > best_d) {  // strict: the first (lowest-index) maximum stays
        best_d = min_dist[i];
        best = i;
      }
    }
    sel = best;
  }
  return kOk;
}

// Benchmark helper, not part of any definition above: runs one of the
// passes `reps` times on the same cloud and writes each run's duration on
// std::chrono::steady_clock, in nanoseconds, to times_ns.  op 0 is
// pv_oracle_voxelize, 1 pv_oracle_voxelize3d, 2 pv_oracle_downsample (which
// takes no max_points and writes [max_voxels, 4] centroids).  Returns the
// first non-zero status of a pass, else 0.
int pv_oracle_time(int op, const float* points, int64_t N, const float range[6], const float voxel_size[3],
                   int max_points, int max_voxels, float* out_rows, int32_t* out_coords, int32_t* out_counts,
                   int32_t* out_num, int reps, int64_t* times_ns) {
  if (reps < 1 || times_ns == nullptr || op < 0 || op > 2) return kErrInvalid;
  for (int r = 0; r < reps; ++r) {
    const auto t0 = std::chrono::steady_clock::now();
    int st;
    if (op == 0)
      st = pv_oracle_voxelize(points, N, range, voxel_size, max_points, max_voxels, out_rows, out_coords, out_counts,
                              out_num);
    else if (op == 1)
      st = pv_oracle_voxelize3d(points, N, range, voxel_size, max_points, max_voxels, out_rows, out_coords,
                                out_counts, out_num);
    else
      st = pv_oracle_downsample(points, N, range, voxel_size, max_voxels, out_rows, out_coords, out_counts, out_num);
    const auto t1 = std::chrono::steady_clock::now();
    if (st != kOk) return st;
    times_ns[r] = std::chrono::duration_cast<std::chrono::nanoseconds>(t1 - t0).count();
  }
  return kOk;
}

}  // extern "C"
