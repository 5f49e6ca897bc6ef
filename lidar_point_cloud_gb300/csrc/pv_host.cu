// Host side of libpv.so: argument checks, the planner (table kind and size,
// launch shape), the per-(device, stream) workspace, the launches, the
// allocation-free entry point's fixed scratch, and the C ABI declared in
// pv.h.  The kernels are in pv_ordered.cu, pv_unordered.cu and
// pv_downsample.cu (shared device code in pv_device.cuh), farthest point
// sampling with its own entry in pv_fps.cu.

#include "pv_device.cuh"

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>

namespace {

using namespace pvk;

// ------------------------------------------------------------ host side

struct DeviceInfo {
  int sms = 0;
  int blocks_per_sm = 0;       // 1024-thread kernels
  int blocks_per_sm_half = 0;  // the block-tile kernel's 512-thread build (0: not used)
  int blocks_per_sm_ds_half = 0;  // the downsampling kernel's 512-thread build (0: not used)
  bool cooperative = false;
};

// Block size of the block-tile kernel's second build (pv_ordered_half.cu).
constexpr int kHalfThreads = 512;
// Kept rows per warp of the grid from which the gather interleaves its shares.
constexpr int64_t kInterleaveMinRowsPerWarp = 16;

struct Workspace {
  std::mutex mu;
  int device = 0;
  Control* ctl = nullptr;
  unsigned int* counts = nullptr;  // [kMaxCtas]
  int32_t* slot_of_point = nullptr;
  int32_t* firsts = nullptr;
  float4* tile_rows = nullptr;
  unsigned long long* recs = nullptr;
  size_t points_cap = 0;
  unsigned long long* lists = nullptr;  // 64-bit entries
  size_t list_words_cap = 0;
  int32_t* keys = nullptr;
  size_t key_words_cap = 0;
  unsigned int* row_cnt = nullptr;  // unordered mode, [max_voxels]
  size_t row_cnt_cap = 0;
  VoxAcc* acc = nullptr;            // downsampling, [T]
  size_t acc_cap = 0;
  // Device copies used by pv_voxelize_host.
  unsigned char* staging = nullptr;
  size_t staging_cap = 0;
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;
std::map<std::pair<int, pv_stream_t>, Workspace*> g_ws;

struct Plan {
  unsigned int stall = 0;  // test hook (pv_options.test_stall_barrier)
  bool keep_tail = false;  // rows past V left unwritten (pv_voxelize_host)
  int frames = 1;
  bool batched = false;    // pv_voxelize_batch (any frame count): batched layout of the outputs
  bool downsample = false; // pv_voxel_downsample: per-voxel accumulators instead of lists
  int64_t cells = 0;       // voxels of one frame's grid
  bool unordered = false;  // pv_options.order == 1
  int64_t g[3];
  int mode;
  int64_t T;
  int KT;             // tail entries per slot
  int append = 0;     // append lists (ordered voxelization, kAppendMinK <= max_points <= 32)
  int64_t pool_n = 0; // append lists: overflow lists in the pool
  int threads = kThreads;  // block size of the launch
  bool half = false;       // block-tile kernel, 512-thread build
  int ctas;
  int64_t chunk;
  unsigned int mask;
  size_t list_words;
  size_t key_words;
  size_t row_words;   // unordered mode: per-row point counters (max_voxels)
  size_t acc_slots = 0;  // downsampling: accumulators (T)
  size_t bytes;
};

int64_t next_pow2(int64_t v) {
  int64_t p = 1;
  while (p < v) p <<= 1;
  return p;
}

int grid_extents(const float r[6], const float v[3], int64_t g[3]) {
  if (!r || !v) return PV_ERR_INVALID;
  for (int a = 0; a < 3; ++a) {
    const float lo = r[a], hi = r[a + 3], s = v[a];
    if (!std::isfinite(lo) || !std::isfinite(hi) || !std::isfinite(s)) return PV_ERR_INVALID;
    if (!(s > 0.0f) || !(hi > lo)) return PV_ERR_INVALID;
    const double q = (static_cast<double>(hi) - static_cast<double>(lo)) / static_cast<double>(s);
    if (!(q < 2.0 * static_cast<double>(kMaxAxisCells))) return PV_ERR_INVALID;
    const int64_t cells = static_cast<int64_t>(std::llround(q));  // half away from zero
    if (cells < 1 || cells > kMaxAxisCells) return PV_ERR_INVALID;
    g[a] = cells;
  }
  if (g[0] * g[1] * g[2] >= (int64_t(1) << 31)) return PV_ERR_INVALID;  // ids stay int32
  return PV_OK;
}

// Shared-memory opt-in of every kernel; the resident blocks per SM of the
// kernel that fits fewest (0 on failure).
int prepare_kernels() {
  const int ordered = prepare_ordered_1024();
  const int down = prepare_downsample_1024();
  return std::min(ordered, down);
}

int device_info(int dev, DeviceInfo* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_devices.find(dev);
  if (it != g_devices.end()) {
    *out = it->second;
    return PV_OK;
  }
  DeviceInfo d;
  int coop = 0;
  if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PV_ERR_CUDA;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) return PV_ERR_CUDA;
  d.blocks_per_sm = prepare_kernels();
  d.blocks_per_sm_half = prepare_ordered_512();
  d.blocks_per_sm_ds_half = prepare_downsample_512();
  d.cooperative = coop != 0;
  if (d.blocks_per_sm < 1 || !d.cooperative) return PV_ERR_CUDA;
  g_devices[dev] = d;
  *out = d;
  return PV_OK;
}

int make_plan(int64_t N, const float range[6], const float vsize[3], int K, int M, const pv_options* opt,
              const DeviceInfo& dev, Plan* pl, int frames = 1) {
  if (N < 0 || N >= (int64_t(1) << 29)) return PV_ERR_INVALID;
  if (K < 1 || K > PV_MAX_POINTS_LIMIT || M < 1) return PV_ERR_INVALID;
  if (static_cast<int64_t>(K) * M >= (int64_t(1) << 31)) return PV_ERR_INVALID;
  int st = grid_extents(range, vsize, pl->g);
  if (st != PV_OK) return st;
  pv_options o{};
  if (opt) o = *opt;
  if (o.table_mode < 0 || o.table_mode > 2 || o.table_log2 < 0 || o.table_log2 > 31 || o.ctas_per_sm < 0)
    return PV_ERR_INVALID;
  pl->stall = o.test_stall_barrier ? 1u : 0u;
  if (o.order < 0 || o.order > 1) return PV_ERR_INVALID;
  pl->unordered = o.order == 1;
  pl->cells = pl->g[0] * pl->g[1] * pl->g[2];
  pl->frames = frames;
  if (frames < 1 || frames > kMaxFrames) return PV_ERR_INVALID;
  if (pl->cells * frames >= (int64_t(1) << 31)) return PV_ERR_INVALID;  // batched ids stay int32
  const int64_t cells = pl->cells * frames;  // one key space per frame
  const int64_t distinct_bound = std::max<int64_t>(1, std::min(N, cells));
  // Hashed tables at most a quarter full: a warp waits for its longest probe
  // chain, each probe a dependent L2 round trip.
  const int64_t hashed_T = next_pow2(std::max<int64_t>(4 * distinct_bound, 1024));
  pl->KT = std::max(0, ((K + 3) & ~3) - kHead);
  const int64_t direct_bytes = cells * (kHead + pl->KT) * 8;
  // Direct (one slot per cell, no probing) whenever it is not much larger
  // than the hashed table would be, or costs at most 256 MB whatever the
  // cloud (a small cloud on the KITTI pillar grid: 55 MB), up to 2 GB.
  int mode = o.table_mode;
  if (mode == 0)
    mode = ((cells <= 2 * hashed_T || direct_bytes <= (int64_t(256) << 20)) && direct_bytes <= (int64_t(1) << 31))
               ? 1
               : 2;
  pl->mode = mode;
  if (mode == 1) {
    pl->T = cells;
    pl->mask = 0;
  } else {
    pl->T = o.table_log2 ? (int64_t(1) << std::max(2, o.table_log2)) : hashed_T;
    if (pl->T > (int64_t(1) << 30)) return PV_ERR_INVALID;  // slots stay below the leader bit
    pl->mask = static_cast<unsigned int>(pl->T - 1);
  }
  // Append lists need an overflow pool: a slot overflows only with more
  // than S - 2 entries, each at least one point, so N / (S - 1) + 1 lists
  // always suffice.
  const int S = kHead + pl->KT;
  pl->append = (!pl->unordered && !pl->downsample && K >= kAppendMinK && K <= 32) ? 1 : 0;
  pl->pool_n = pl->append ? N / (S - 1) + 1 : 0;
  pl->list_words = static_cast<size_t>(pl->T) * S + static_cast<size_t>(pl->pool_n) * S;
  pl->key_words = mode == 2 ? static_cast<size_t>(pl->T) : 0;
  const int per_sm = o.ctas_per_sm ? std::min(o.ctas_per_sm, dev.blocks_per_sm) : dev.blocks_per_sm;
  // The count scan after the second barrier takes one count per thread.
  pl->threads = kThreads;
  pl->half = false;
  pl->ctas = std::min(std::min(kMaxCtas, kThreads), std::max(1, dev.sms * per_sm));
  // Block-tile voxelization whose chunks would span several 1024-point
  // tiles: the 512-thread build, two blocks an SM (measured on GB300: the
  // dense frame 50.8 -> 46.6 us, 8 KITTI-shaped frames 66.0 -> 60.3 us; the
  // KITTI-shaped frame itself, one tile a chunk, is faster on 1024 threads,
  // whose longer chunks split fewer pillars into more than three groups).
  // The same for centroid downsampling (dense3d frame 49.5 -> 45.5 us).
  const int half_blocks = pl->downsample ? dev.blocks_per_sm_ds_half : dev.blocks_per_sm_half;
  if (!pl->unordered && half_blocks >= 1 && N > static_cast<int64_t>(pl->ctas) * kThreads) {
    const int per_half = o.ctas_per_sm ? std::min(o.ctas_per_sm, half_blocks) : half_blocks;
    pl->half = true;
    pl->threads = kHalfThreads;
    pl->ctas = std::min(std::min(kMaxCtas, kHalfThreads), std::max(1, dev.sms * per_half));
  }
  // Contiguous chunks, as even as whole warps allow: phase 1 and phase 2
  // share them, and a block's tiles start at its chunk's start.
  const int64_t per = (N + pl->ctas - 1) / pl->ctas;
  pl->chunk = std::max<int64_t>(32, (per + 31) / 32 * 32);
  pl->row_words = pl->unordered ? static_cast<size_t>(M) : 0;
  pl->bytes = sizeof(Control) + 4 * static_cast<size_t>(kMaxCtas) + 32 * static_cast<size_t>(N) +
              8 * pl->list_words + 4 * pl->key_words + 4 * pl->row_words;
  return PV_OK;
}

// Grows one workspace region.  New memory is set to `fill` on `stream`.
template <typename T>
int grow(T** ptr, size_t* cap, size_t need, int fill, pv_stream_t stream, bool* synced) {
  if (*cap >= need) return PV_OK;
  if (!*synced) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PV_ERR_CUDA;
    *synced = true;
  }
  if (*ptr) cudaFree(*ptr);
  *ptr = nullptr;
  *cap = 0;
  void* mem = nullptr;
  if (cudaMalloc(&mem, need * sizeof(T)) != cudaSuccess) {
    cudaGetLastError();
    return PV_ERR_ALLOC;
  }
  if (cudaMemsetAsync(mem, fill, need * sizeof(T), stream) != cudaSuccess) {
    cudaFree(mem);
    return PV_ERR_CUDA;
  }
  *ptr = static_cast<T*>(mem);
  *cap = need;
  return PV_OK;
}

int get_workspace(int dev, pv_stream_t stream, Workspace** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_pair(dev, stream);
  auto it = g_ws.find(key);
  if (it != g_ws.end()) {
    *out = it->second;
    return PV_OK;
  }
  Workspace* ws = new (std::nothrow) Workspace();
  if (!ws) return PV_ERR_ALLOC;
  ws->device = dev;
  void* ctl = nullptr;
  if (cudaMalloc(&ctl, sizeof(Control)) != cudaSuccess) {
    cudaGetLastError();
    delete ws;
    return PV_ERR_ALLOC;
  }
  Control init{};
  init.epoch = 1;
  if (cudaMemcpy(ctl, &init, sizeof init, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(ctl);
    delete ws;
    return PV_ERR_CUDA;
  }
  ws->ctl = static_cast<Control*>(ctl);
  void* cnt = nullptr;
  if (cudaMalloc(&cnt, sizeof(unsigned int) * (kMaxCtas + kMaxFrames + 1)) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(ctl);
    delete ws;
    return PV_ERR_ALLOC;
  }
  ws->counts = static_cast<unsigned int*>(cnt);
  g_ws[key] = ws;
  *out = ws;
  return PV_OK;
}

size_t round_up(size_t v, size_t m) { return (v + m - 1) / m * m; }

// The device address of a pinned host buffer (page-locked and mapped into
// the device's address space: cudaHostAlloc, cudaHostRegister) when it is
// aligned to `align` bytes, or null for any other pointer.
void* mapped_host(const void* ptr, size_t align) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
  return reinterpret_cast<uintptr_t>(a.devicePointer) % align == 0 ? a.devicePointer : nullptr;
}

// Makes every region big enough for `pl` (caller holds ws->mu).
int reserve(Workspace* ws, const Plan& pl, int64_t N, pv_stream_t stream) {
  bool synced = false;
  int st;
  const size_t np = round_up(static_cast<size_t>(std::max<int64_t>(N, 1)), 65536);
  if (ws->points_cap < np) {
    const size_t want = std::max(np, ws->points_cap + ws->points_cap / 2);
    size_t cap_a = ws->points_cap, cap_b = ws->points_cap, cap_c = ws->points_cap, cap_d = ws->points_cap;
    if ((st = grow(&ws->slot_of_point, &cap_a, want, 0, stream, &synced)) != PV_OK) return st;
    if ((st = grow(&ws->firsts, &cap_b, want, 0, stream, &synced)) != PV_OK) return st;
    if ((st = grow(&ws->tile_rows, &cap_c, want, 0, stream, &synced)) != PV_OK) return st;
    if ((st = grow(&ws->recs, &cap_d, want, 0, stream, &synced)) != PV_OK) return st;
    ws->points_cap = want;
  }
  if (pl.list_words &&
      (st = grow(&ws->lists, &ws->list_words_cap, round_up(pl.list_words, 2), 0xFF, stream, &synced)) != PV_OK)
    return st;
  if (pl.acc_slots && (st = grow(&ws->acc, &ws->acc_cap, pl.acc_slots, 0, stream, &synced)) != PV_OK) return st;
  if (pl.key_words &&
      (st = grow(&ws->keys, &ws->key_words_cap, pl.key_words, 0xFF, stream, &synced)) != PV_OK)
    return st;
  if (pl.row_words &&
      (st = grow(&ws->row_cnt, &ws->row_cnt_cap, pl.row_words, 0, stream, &synced)) != PV_OK)
    return st;
  return PV_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device that owns a pointer, or -1 if it is not device (or managed) memory.
int device_of(const void* ptr) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return -1;
  return at.device;
}

class DeviceGuard {
 public:
  explicit DeviceGuard(int dev) {
    cudaGetDevice(&prev_);
    if (prev_ != dev) {
      ok_ = cudaSetDevice(dev) == cudaSuccess;
      changed_ = true;
    }
  }
  ~DeviceGuard() {
    if (changed_) cudaSetDevice(prev_);
  }
  bool ok() const { return ok_; }

 private:
  int prev_ = 0;
  bool changed_ = false;
  bool ok_ = true;
};

int launch(Workspace* ws, const Plan& pl, const float* points, int64_t N, const float range[6],
           const float vsize[3], int K, int M, float* out_voxels, int32_t* out_coords, int32_t* out_counts,
           int32_t* out_num, pv_stream_t stream, const int64_t* frame_offsets = nullptr) {
  KParams kp;
  kp.points = reinterpret_cast<const float4*>(points);
  kp.n = N;
  kp.chunk = pl.chunk;
  kp.lo_x = range[0];
  kp.lo_y = range[1];
  kp.lo_z = range[2];
  kp.v_x = vsize[0];
  kp.v_y = vsize[1];
  kp.v_z = vsize[2];
  // Reciprocal estimates for the binning filter; only normal, finite values are used.
  const float rx = 1.0f / vsize[0], ry = 1.0f / vsize[1], rz = 1.0f / vsize[2];
  kp.r_x = std::isnormal(rx) ? rx : 0.0f;
  kp.r_y = std::isnormal(ry) ? ry : 0.0f;
  kp.r_z = std::isnormal(rz) ? rz : 0.0f;
  kp.g_xf = static_cast<float>(pl.g[0]);
  kp.g_yf = static_cast<float>(pl.g[1]);
  kp.g_zf = static_cast<float>(pl.g[2]);
  kp.g_x = static_cast<int>(pl.g[0]);
  kp.g_y = static_cast<int>(pl.g[1]);
  kp.div_x = make_fast_div(static_cast<unsigned int>(pl.g[0]));
  kp.div_y = make_fast_div(static_cast<unsigned int>(pl.g[1]));
  kp.K = K;
  kp.KT = pl.KT;
  kp.append = pl.append;
  kp.pool = ws->lists + static_cast<size_t>(pl.T) * (kHead + pl.KT);
  kp.pool_n = static_cast<unsigned int>(pl.pool_n);
  kp.max_voxels = M;
  kp.hash_mode = pl.mode == 2 ? 1 : 0;
  kp.bar_extra = pl.stall;
  kp.zero_tail = pl.keep_tail ? 0 : 1;
  kp.table_mask = pl.mask;
  kp.lists = ws->lists;
  kp.tails = ws->lists + static_cast<size_t>(pl.T) * kHead;
  kp.keys = ws->keys;
  kp.slot_of_point = ws->slot_of_point;
  kp.firsts = ws->firsts;
  kp.tile_rows = ws->tile_rows;
  kp.recs = ws->recs;
  kp.counts = ws->counts;
  kp.ctl = ws->ctl;
  kp.list_words_cap = ws->list_words_cap;
  kp.key_words_cap = ws->key_words_cap;
  kp.out_voxels = reinterpret_cast<float4*>(out_voxels);
  kp.out_coords = out_coords;
  kp.out_counts = out_counts;
  kp.out_num = out_num;
  kp.row_cnt = ws->row_cnt;
  kp.row_cnt_cap = ws->row_cnt_cap;
  kp.frames = pl.frames;
  kp.cells = static_cast<int>(pl.cells);
  kp.div_cells = make_fast_div(static_cast<unsigned int>(std::max<int64_t>(1, pl.cells)));
  kp.frame_cnt = ws->counts + kMaxCtas;
  kp.acc = ws->acc;
  kp.acc_cap = ws->acc_cap;
  // The gather's share per warp grows with the rows; long lists bunch up in
  // some warps' contiguous shares once a share holds more than a few rows,
  // and queuing them per block is then worth its block barrier (a kernel
  // of its own: the queue's code alone slows the small frames' gather).
  const bool queue = static_cast<int64_t>(M) >= kQueueMinRowsPerWarp * pl.ctas * (pl.threads / 32);
  // Interleaved gather shares once warps have many rows (all frames' rows in
  // a batch): measured on GB300, the adversarial cloud (41 rows a warp)
  // 281 -> 264 us and 8 KITTI-shaped frames (26) 60.8 -> 55.2 us, against the
  // dense frame (12) 46.5 -> 47.0 us and a 130K uniform cloud (3) 24.8 -> 25.7 us.
  kp.interleave = static_cast<int64_t>(M) * pl.frames >= kInterleaveMinRowsPerWarp * pl.ctas * (pl.threads / 32) ? 1 : 0;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned int>(pl.ctas));
  cfg.blockDim = dim3(static_cast<unsigned int>(pl.threads));
  cfg.dynamicSmemBytes = pl.unordered ? 0 : (pl.half ? ordered_smem_512() : ordered_smem_1024());
  // One-tile chunks need only the first tile map (the long-list queue, if
  // any, then holds what fits in it); the rest of the SM's 256 KB stays L1
  // (measured: KITTI-shaped 16.14 -> 15.78 us, 130K uniform 24.84 -> 21.78
  // us, kitti3d with its queue 23.28 -> 20.15 us).  The kernel checks what
  // it got.
  if (!pl.unordered && !pl.downsample && !pl.half && pl.chunk <= kThreads)
    cfg.dynamicSmemBytes = kMapBytes;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  // Cooperative (every block resident: the grid barriers) and programmatic
  // stream serialization (the kernels wait for the previous grid first, so
  // the launch's set-up may overlap that grid's end; measured: KITTI-shaped
  // 15.65 -> 15.44 us, tiny 14.41 -> 13.76 us, dense 46.61 -> 45.78 us a launch
  // back to back).
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e;
  if (pl.downsample) {
    cfg.dynamicSmemBytes = pl.half ? downsample_smem_512() : downsample_smem_1024();
    e = pl.half ? launch_downsample_512(cfg, kp) : launch_downsample_1024(cfg, kp);
  } else if (pl.unordered) {
    e = launch_unordered(cfg, kp);
  } else {
    const int64_t* fo = pl.batched ? frame_offsets : nullptr;
    e = pl.half ? launch_ordered_512(cfg, kp, queue, fo, pl.frames, N) : launch_ordered_1024(cfg, kp, queue, fo, pl.frames, N);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PV_ERR_CUDA;
  }
  return PV_OK;
}

int voxelize_impl(const float* points, int64_t N, const float range[6], const float vsize[3], int K, int M,
                  float* out_voxels, int32_t* out_coords, int32_t* out_counts, int32_t* out_num,
                  const pv_options* opt, pv_stream_t stream, const int64_t* frame_offsets = nullptr,
                  int frames = 1) {
  if (!range || !vsize) return PV_ERR_INVALID;
  if (!out_voxels || !out_coords || !out_counts || !out_num) return PV_ERR_INVALID;
  if (N > 0 && !points) return PV_ERR_INVALID;
  if (!aligned(out_voxels, 16) || !aligned(out_coords, 4) || !aligned(out_counts, 4) || !aligned(out_num, 4))
    return PV_ERR_INVALID;
  if (N > 0 && !aligned(points, 16)) return PV_ERR_INVALID;
  const int dev = device_of(out_voxels);
  if (dev < 0) return PV_ERR_INVALID;
  if (device_of(out_coords) != dev || device_of(out_counts) != dev || device_of(out_num) != dev)
    return PV_ERR_INVALID;
  if (N > 0 && device_of(points) != dev) return PV_ERR_INVALID;
  DeviceGuard guard(dev);
  if (!guard.ok()) return PV_ERR_CUDA;
  DeviceInfo di;
  int st = device_info(dev, &di);
  if (st != PV_OK) return st;
  Plan pl;
  if ((st = make_plan(N, range, vsize, K, M, opt, di, &pl, frames)) != PV_OK) return st;
  pl.batched = frame_offsets != nullptr;
  Workspace* ws = nullptr;
  if ((st = get_workspace(dev, stream, &ws)) != PV_OK) return st;
  std::lock_guard<std::mutex> lk(ws->mu);
  if ((st = reserve(ws, pl, N, stream)) != PV_OK) return st;
  return launch(ws, pl, points, N, range, vsize, K, M, out_voxels, out_coords, out_counts, out_num, stream,
                frame_offsets);
}

// Centroid downsampling: the same checks and workspace, accumulators in
// place of lists.
int downsample_impl(const float* points, int64_t N, const float range[6], const float vsize[3], int M,
                    float* out_centroids, int32_t* out_coords, int32_t* out_counts, int32_t* out_num,
                    pv_stream_t stream) {
  if (!range || !vsize) return PV_ERR_INVALID;
  if (!out_centroids || !out_coords || !out_counts || !out_num) return PV_ERR_INVALID;
  if (N > 0 && !points) return PV_ERR_INVALID;
  if (!aligned(out_centroids, 16) || !aligned(out_coords, 4) || !aligned(out_counts, 4) || !aligned(out_num, 4))
    return PV_ERR_INVALID;
  if (N > 0 && !aligned(points, 16)) return PV_ERR_INVALID;
  const int dev = device_of(out_centroids);
  if (dev < 0) return PV_ERR_INVALID;
  if (device_of(out_coords) != dev || device_of(out_counts) != dev || device_of(out_num) != dev)
    return PV_ERR_INVALID;
  if (N > 0 && device_of(points) != dev) return PV_ERR_INVALID;
  DeviceGuard guard(dev);
  if (!guard.ok()) return PV_ERR_CUDA;
  DeviceInfo di;
  int st = device_info(dev, &di);
  if (st != PV_OK) return st;
  Plan pl;
  pl.downsample = true;  // (read by make_plan)
  if ((st = make_plan(N, range, vsize, 1, M, nullptr, di, &pl)) != PV_OK) return st;
  pl.list_words = 0;
  pl.acc_slots = static_cast<size_t>(pl.T);
  Workspace* ws = nullptr;
  if ((st = get_workspace(dev, stream, &ws)) != PV_OK) return st;
  std::lock_guard<std::mutex> lk(ws->mu);
  if ((st = reserve(ws, pl, N, stream)) != PV_OK) return st;
  return launch(ws, pl, points, N, range, vsize, 1, M, out_centroids, out_coords, out_counts, out_num, stream);
}

// A batch of frames: offsets on the host, checked here (first 0, never
// decreasing); the total is the last offset.
int voxelize_batch_impl(const float* points, const int64_t* frame_offsets, int frames, const float range[6],
                        const float vsize[3], int K, int M, float* out_voxels, int32_t* out_coords,
                        int32_t* out_counts, int32_t* out_num, pv_stream_t stream) {
  if (!frame_offsets || frames < 1 || frames > kMaxFrames) return PV_ERR_INVALID;
  if (frame_offsets[0] != 0) return PV_ERR_INVALID;
  for (int b = 0; b < frames; ++b)
    if (frame_offsets[b + 1] < frame_offsets[b]) return PV_ERR_INVALID;
  if (static_cast<int64_t>(frames) * M * K >= (int64_t(1) << 31)) return PV_ERR_INVALID;  // output rows
  return voxelize_impl(points, frame_offsets[frames], range, vsize, K, M, out_voxels, out_coords, out_counts,
                       out_num, nullptr, stream, frame_offsets, frames);
}

// ------------------------------------------------------------ allocation-free variant

// pv_voxelize_static keeps all of its scratch in one file-scope device array
// instead of the per-stream workspace, for callers that must not allocate
// device memory.  Limits: num_points <= kStaticMaxPoints and max_points <=
// kStaticMaxK; the table is always hashed, with at most 2^kStaticTableLog2
// slots.  Layout (256-byte aligned regions): control block, per-block
// counts, hashed keys, slot lists, then four per-point arrays.
constexpr int64_t kStaticMaxPoints = 32768;
constexpr int kStaticMaxK = 32;
constexpr int kStaticTableLog2 = 16;
constexpr size_t kStaticSlots = size_t(1) << kStaticTableLog2;
constexpr size_t kStaticOffCounts = 256;
constexpr size_t kStaticOffKeys = kStaticOffCounts + 4 * kMaxCtas;
constexpr size_t kStaticOffLists = kStaticOffKeys + 4 * kStaticSlots;
constexpr size_t kStaticPoolWords = 40960;  // append lists' overflow pool: (32768 / 7 + 1) x 8 words at most
constexpr size_t kStaticListWords = kStaticSlots * kStaticMaxK + kStaticPoolWords;  // 64-bit entries
// The pool must hold an overflow list for every slot that can overflow: with
// the shortest append rows (kAppendMinK words) a slot overflows only past
// kAppendMinK - 2 entries of at least one point each.
static_assert((kStaticMaxPoints / (kAppendMinK - 1) + 1) * kAppendMinK <= static_cast<int64_t>(kStaticPoolWords),
              "the static overflow pool holds every list an append plan can take");
constexpr size_t kStaticOffRows = kStaticOffLists + 8 * kStaticListWords;
constexpr size_t kStaticOffRecs = kStaticOffRows + 16 * static_cast<size_t>(kStaticMaxPoints);
constexpr size_t kStaticOffPoints = kStaticOffRecs + 8 * static_cast<size_t>(kStaticMaxPoints);
constexpr size_t kStaticBytes = kStaticOffPoints + 2 * 4 * static_cast<size_t>(kStaticMaxPoints);
static_assert(sizeof(Control) <= kStaticOffCounts, "control block fits its region");
static_assert(kStaticOffKeys % 256 == 0 && kStaticOffLists % 256 == 0 && kStaticOffRows % 256 == 0 &&
                  kStaticOffPoints % 256 == 0,
              "regions stay 256-byte aligned");

static __device__ __align__(256) unsigned char g_static_scratch[kStaticBytes];

// Per-device set-up state; fixed size, so no call allocates host memory either.
constexpr int kStaticMaxDevices = 64;
struct StaticDevice {
  bool ready = false;
  unsigned char* base = nullptr;  // device address of g_static_scratch on this device
  DeviceInfo info;
};
std::mutex g_static_mu;
StaticDevice g_static_dev[kStaticMaxDevices];

// Once per device, with that device current: look up the array's device
// address (the host-side symbol is only a stand-in), prepare the kernel's
// attributes, and put the array in its initial state on `stream` (control
// block and counts zero, table empty).
int static_setup(int dev, pv_stream_t stream, StaticDevice** out) {
  if (dev < 0 || dev >= kStaticMaxDevices) return PV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_static_mu);
  StaticDevice& sd = g_static_dev[dev];
  if (!sd.ready) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return PV_ERR_CUDA;
    }
    DeviceInfo d;
    int coop = 0;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) {
      cudaGetLastError();
      return PV_ERR_CUDA;
    }
    d.blocks_per_sm = prepare_kernels();
    d.cooperative = coop != 0;
    if (d.blocks_per_sm < 1 || !d.cooperative) return PV_ERR_CUDA;
    unsigned char* base = static_cast<unsigned char*>(ptr);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(base, 0, kStaticOffKeys, s) != cudaSuccess ||
        cudaMemsetAsync(base + kStaticOffKeys, 0xFF, kStaticOffRows - kStaticOffKeys, s) != cudaSuccess) {
      cudaGetLastError();
      return PV_ERR_CUDA;
    }
    sd.base = base;
    sd.info = d;
    sd.ready = true;
  }
  *out = &sd;
  return PV_OK;
}

int voxelize_static_impl(const float* points, int64_t N, const float range[6], const float vsize[3], int K, int M,
                         float* out_voxels, int32_t* out_coords, int32_t* out_counts, int32_t* out_num,
                         pv_stream_t stream) {
  if (!range || !vsize) return PV_ERR_INVALID;
  if (!out_voxels || !out_coords || !out_counts || !out_num) return PV_ERR_INVALID;
  if (N > 0 && !points) return PV_ERR_INVALID;
  if (N > kStaticMaxPoints || K > kStaticMaxK) return PV_ERR_TOO_LARGE;
  if (!aligned(out_voxels, 16) || !aligned(out_coords, 4) || !aligned(out_counts, 4) || !aligned(out_num, 4))
    return PV_ERR_INVALID;
  if (N > 0 && !aligned(points, 16)) return PV_ERR_INVALID;
  const int dev = device_of(out_voxels);
  if (dev < 0) return PV_ERR_INVALID;
  if (device_of(out_coords) != dev || device_of(out_counts) != dev || device_of(out_num) != dev)
    return PV_ERR_INVALID;
  if (N > 0 && device_of(points) != dev) return PV_ERR_INVALID;
  DeviceGuard guard(dev);
  if (!guard.ok()) return PV_ERR_CUDA;
  StaticDevice* sd = nullptr;
  int st = static_setup(dev, stream, &sd);
  if (st != PV_OK) return st;
  pv_options opt{};
  opt.table_mode = 2;  // hashed: the static table has a fixed number of slots
  opt.table_log2 = kStaticTableLog2;
  Plan pl;
  if ((st = make_plan(N, range, vsize, K, M, &opt, sd->info, &pl)) != PV_OK) return st;
  if (pl.T > static_cast<int64_t>(kStaticSlots) || pl.list_words > kStaticListWords) return PV_ERR_TOO_LARGE;
  // A stack view of the array in the workspace's shape; nothing is allocated.
  Workspace view;
  view.device = dev;
  view.ctl = reinterpret_cast<Control*>(sd->base);
  view.counts = reinterpret_cast<unsigned int*>(sd->base + kStaticOffCounts);
  view.keys = reinterpret_cast<int32_t*>(sd->base + kStaticOffKeys);
  view.key_words_cap = kStaticSlots;
  view.lists = reinterpret_cast<unsigned long long*>(sd->base + kStaticOffLists);
  view.list_words_cap = kStaticListWords;
  view.tile_rows = reinterpret_cast<float4*>(sd->base + kStaticOffRows);
  view.recs = reinterpret_cast<unsigned long long*>(sd->base + kStaticOffRecs);
  int32_t* pts = reinterpret_cast<int32_t*>(sd->base + kStaticOffPoints);
  view.slot_of_point = pts;
  view.firsts = pts + kStaticMaxPoints;
  view.points_cap = kStaticMaxPoints;
  return launch(&view, pl, points, N, range, vsize, K, M, out_voxels, out_coords, out_counts, out_num, stream);
}

}  // namespace

// ------------------------------------------------------------ C ABI

extern "C" {

int pv_voxelize(const float* points, int64_t num_points, const float point_cloud_range[6],
                const float voxel_size[3], int max_points, int max_voxels, float* out_voxels,
                int32_t* out_coords, int32_t* out_counts, int32_t* out_num_voxels, pv_stream_t stream) {
  return voxelize_impl(points, num_points, point_cloud_range, voxel_size, max_points, max_voxels, out_voxels,
                       out_coords, out_counts, out_num_voxels, nullptr, stream);
}

int pv_voxelize_ex(const float* points, int64_t num_points, const float point_cloud_range[6],
                   const float voxel_size[3], int max_points, int max_voxels, float* out_voxels,
                   int32_t* out_coords, int32_t* out_counts, int32_t* out_num_voxels, const pv_options* options,
                   pv_stream_t stream) {
  return voxelize_impl(points, num_points, point_cloud_range, voxel_size, max_points, max_voxels, out_voxels,
                       out_coords, out_counts, out_num_voxels, options, stream);
}

int pv_voxelize_batch(const float* points, const int64_t* frame_offsets, int num_frames,
                      const float point_cloud_range[6], const float voxel_size[3], int max_points, int max_voxels,
                      float* out_voxels, int32_t* out_coords, int32_t* out_counts, int32_t* out_num_voxels,
                      pv_stream_t stream) {
  return voxelize_batch_impl(points, frame_offsets, num_frames, point_cloud_range, voxel_size, max_points,
                             max_voxels, out_voxels, out_coords, out_counts, out_num_voxels, stream);
}

int pv_voxel_downsample(const float* points, int64_t num_points, const float point_cloud_range[6],
                        const float voxel_size[3], int max_voxels, float* out_centroids, int32_t* out_coords,
                        int32_t* out_counts, int32_t* out_num_voxels, pv_stream_t stream) {
  return downsample_impl(points, num_points, point_cloud_range, voxel_size, max_voxels, out_centroids, out_coords,
                         out_counts, out_num_voxels, stream);
}

int pv_voxelize_host(const float* points_host, int64_t num_points, const float point_cloud_range[6],
                     const float voxel_size[3], int max_points, int max_voxels, float* out_voxels_host,
                     int32_t* out_coords_host, int32_t* out_counts_host, int32_t* out_num_voxels_host,
                     pv_stream_t stream) {
  if (!point_cloud_range || !voxel_size) return PV_ERR_INVALID;
  if (!out_voxels_host || !out_coords_host || !out_counts_host || !out_num_voxels_host) return PV_ERR_INVALID;
  if (num_points > 0 && !points_host) return PV_ERR_INVALID;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PV_ERR_CUDA;
  DeviceInfo di;
  int st = device_info(dev, &di);
  if (st != PV_OK) return st;
  Plan pl;
  if ((st = make_plan(num_points, point_cloud_range, voxel_size, max_points, max_voxels, nullptr, di, &pl)) !=
      PV_OK)
    return st;
  Workspace* ws = nullptr;
  if ((st = get_workspace(dev, stream, &ws)) != PV_OK) return st;
  std::lock_guard<std::mutex> lk(ws->mu);
  if ((st = reserve(ws, pl, num_points, stream)) != PV_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The result is the first V rows (the page's Python entry point slices
  // its padded outputs to the pillar count): rows past V are not written,
  // so no zero row crosses the host link.
  pl.keep_tail = true;
  // Pinned buffers (page-locked and mapped) are used in place: the kernel
  // reads the points and writes the outputs across the host link itself, so
  // each byte crosses it once, as with copies, without a copy's set-up or
  // its wait for the kernel.  Other host memory goes through device staging.
  const float* in_pts = static_cast<const float*>(num_points > 0 ? mapped_host(points_host, 16) : nullptr);
  float* mv = static_cast<float*>(mapped_host(out_voxels_host, 16));
  int32_t* mc = static_cast<int32_t*>(mapped_host(out_coords_host, 4));
  int32_t* mn = static_cast<int32_t*>(mapped_host(out_counts_host, 4));
  int32_t* mu = static_cast<int32_t*>(mapped_host(out_num_voxels_host, 4));
  const bool in_place = mv && mc && mn && mu;
  // Staging layout: points | voxels | coords | counts | num, each 256-byte aligned (only what is needed).
  const size_t b_pts = in_pts ? 0 : round_up(16 * static_cast<size_t>(num_points), 256);
  const size_t b_vox = in_place ? 0 : round_up(16 * static_cast<size_t>(max_voxels) * max_points, 256);
  const size_t b_crd = in_place ? 0 : round_up(12 * static_cast<size_t>(max_voxels), 256);
  const size_t b_cnt = in_place ? 0 : round_up(4 * static_cast<size_t>(max_voxels), 256);
  const size_t need = b_pts + b_vox + b_crd + b_cnt + 256;
  bool synced = false;
  if ((st = grow(&ws->staging, &ws->staging_cap, need, 0, stream, &synced)) != PV_OK) return st;
  unsigned char* base = ws->staging;
  if (!in_pts) {
    float* d_pts = reinterpret_cast<float*>(base);
    if (num_points > 0 &&
        cudaMemcpyAsync(d_pts, points_host, 16 * static_cast<size_t>(num_points), cudaMemcpyHostToDevice, s) !=
            cudaSuccess)
      return PV_ERR_CUDA;
    in_pts = d_pts;
  }
  if (in_place) {
    if ((st = launch(ws, pl, in_pts, num_points, point_cloud_range, voxel_size, max_points, max_voxels, mv, mc, mn,
                     mu, stream)) != PV_OK)
      return st;
  } else {
    float* d_vox = reinterpret_cast<float*>(base + b_pts);
    int32_t* d_crd = reinterpret_cast<int32_t*>(base + b_pts + b_vox);
    int32_t* d_cnt = reinterpret_cast<int32_t*>(base + b_pts + b_vox + b_crd);
    int32_t* d_num = reinterpret_cast<int32_t*>(base + b_pts + b_vox + b_crd + b_cnt);
    if ((st = launch(ws, pl, in_pts, num_points, point_cloud_range, voxel_size, max_points, max_voxels, d_vox,
                     d_crd, d_cnt, d_num, stream)) != PV_OK)
      return st;
    // V first, then its rows only.
    if (cudaMemcpyAsync(out_num_voxels_host, d_num, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return PV_ERR_CUDA;
    const int32_t V = *out_num_voxels_host;
    if (V < 0) return V;
    const size_t rows = static_cast<size_t>(std::min(V, max_voxels));
    if (rows > 0 &&
        (cudaMemcpyAsync(out_voxels_host, d_vox, 16 * rows * max_points, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
         cudaMemcpyAsync(out_coords_host, d_crd, 12 * rows, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
         cudaMemcpyAsync(out_counts_host, d_cnt, 4 * rows, cudaMemcpyDeviceToHost, s) != cudaSuccess))
      return PV_ERR_CUDA;
  }
  if (cudaStreamSynchronize(s) != cudaSuccess) return PV_ERR_CUDA;
  return *out_num_voxels_host < 0 ? *out_num_voxels_host : PV_OK;
}

int pv_grid_size(const float point_cloud_range[6], const float voxel_size[3], int64_t grid_out[3]) {
  if (!grid_out) return PV_ERR_INVALID;
  return grid_extents(point_cloud_range, voxel_size, grid_out);
}

int pv_query_plan(int64_t num_points, const float point_cloud_range[6], const float voxel_size[3],
                  int max_points, int max_voxels, const pv_options* options, pv_plan* plan_out) {
  if (!plan_out) return PV_ERR_INVALID;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return PV_ERR_CUDA;
  }
  DeviceInfo di;
  int st = device_info(dev, &di);
  if (st != PV_OK) return st;
  Plan pl;
  if ((st = make_plan(num_points, point_cloud_range, voxel_size, max_points, max_voxels, options, di, &pl)) !=
      PV_OK)
    return st;
  for (int a = 0; a < 3; ++a) plan_out->grid[a] = pl.g[a];
  plan_out->table_mode = pl.mode;
  plan_out->table_slots = pl.T;
  plan_out->list_stride = kHead + pl.KT;
  plan_out->ctas = pl.ctas;
  plan_out->threads = pl.threads;
  plan_out->points_per_cta = pl.chunk;
  plan_out->workspace_bytes = static_cast<int64_t>(pl.bytes);
  return PV_OK;
}

int pv_release_workspace(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int st = PV_OK;
  for (auto& kv : g_ws) {
    Workspace* ws = kv.second;
    DeviceGuard guard(ws->device);
    if (cudaDeviceSynchronize() != cudaSuccess) st = PV_ERR_CUDA;
    cudaFree(ws->ctl);
    cudaFree(ws->counts);
    cudaFree(ws->slot_of_point);
    cudaFree(ws->firsts);
    cudaFree(ws->tile_rows);
    cudaFree(ws->recs);
    cudaFree(ws->lists);
    cudaFree(ws->keys);
    cudaFree(ws->row_cnt);
    cudaFree(ws->acc);
    cudaFree(ws->staging);
    delete ws;
  }
  g_ws.clear();
  return st;
}

const char* pv_status_string(int status) {
  switch (status) {
    case PV_OK: return "PV_OK";
    case PV_ERR_INVALID: return "PV_ERR_INVALID: invalid argument";
    case PV_ERR_UNSUPPORTED: return "PV_ERR_UNSUPPORTED: a request this build does not support";
    case PV_ERR_ALLOC: return "PV_ERR_ALLOC: device workspace allocation failed";
    case PV_ERR_CUDA: return "PV_ERR_CUDA: CUDA runtime error";
    case PV_ERR_CAPACITY: return "PV_ERR_CAPACITY: pillar table full";
    case PV_ERR_TIMEOUT: return "PV_ERR_TIMEOUT: a bounded device wait gave up";
    case PV_ERR_INTERNAL: return "PV_ERR_INTERNAL: device consistency check failed";
    case PV_ERR_TOO_LARGE: return "PV_ERR_TOO_LARGE: beyond the limits of the allocation-free entry point";
    default: return status >= 0 ? "pillar count" : "unknown status";
  }
}

int pv_voxelize_static(const float* points, int64_t num_points, const float point_cloud_range[6],
                       const float voxel_size[3], int max_points, int max_voxels, float* out_voxels,
                       int32_t* out_coords, int32_t* out_counts, int32_t* out_num_voxels, pv_stream_t stream) {
  return voxelize_static_impl(points, num_points, point_cloud_range, voxel_size, max_points, max_voxels,
                              out_voxels, out_coords, out_counts, out_num_voxels, stream);
}

const char* pv_version(void) { return "0.1.0"; }

}  // extern "C"
