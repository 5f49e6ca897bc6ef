// Device code shared by the kernels of libpv.so (the block-tile voxelizer,
// the unordered voxelizer, centroid downsampling) and the types and
// constants the host code passes to them: kernel parameters, the control
// block, limits, PTX helpers, binning, the pillar table and its lists, the
// gather helpers.  Each kernel file includes it and compiles its own copy of
// the device functions; the launch entry points declared at the end are
// defined in the kernel files.

#pragma once

#include "pv.h"

#include <cuda_runtime.h>

#include <cstdint>

namespace pvk {


constexpr uint32_t kEmpty = 0xFFFFFFFFu;   // empty 32-bit marker
constexpr unsigned long long kEmpty64 = ~0ull;  // empty list entry (also an all-0xFF memset)
constexpr int32_t kLeaderBit = 1 << 30;    // slot_of_point: the point leads its tile group
constexpr int32_t kNoKey = -1;             // empty hashed slot
#ifndef PV_BLOCK_THREADS
#define PV_BLOCK_THREADS 1024
#endif
constexpr int kThreads = PV_BLOCK_THREADS;  // also the tile: points grouped together in shared memory
#define PV_CAT_(a, b) a##b
#define PV_CAT(a, b) PV_CAT_(a, b)
// A build's own name for an entry point: name##<block threads>.
#define PV_BLOCK_NAME(name) PV_CAT(name, PV_BLOCK_THREADS)
constexpr int kWarps = kThreads / 32;
static_assert(kWarps <= 32 && kWarps % 16 == 0, "warp 0 scans one value per warp; 16-byte counter rows");
constexpr int kMinBlocksPerSM = 1024 / kThreads;
constexpr int kMaxCtas = 1024;             // blocks per launch (prefix lives in shared memory)
static_assert(kMaxCtas < 0x10000, "finished blocks are counted in 16 bits");
constexpr int kFlagUnroll = 4;             // block-wide tiles in flight when flagging
constexpr int kFlagUnrollWide = 8;         // the same, in launches whose chunks span up to 8 block tiles
static_assert(kWarps == 32 || kWarps == 16, "the flag prefix gives each lane consecutive (tile, warp) counts");
#ifndef PV_HEAD_ENTRIES
#define PV_HEAD_ENTRIES 4
#endif
// List positions 0 .. kHead-1 of every slot sit together in one dense head
// array (kHead * 8 bytes per slot), positions kHead .. max_points-1 in a
// separate tail array: most pillars hold a few groups, so the random
// accesses of a launch stay inside a table a fraction of the size.
constexpr int kHead = PV_HEAD_ENTRIES;
static_assert(kHead == 4 || kHead == 8, "head rows are 32 or 64 bytes");
#ifndef PV_EMIT_LANES
#define PV_EMIT_LANES 8
#endif
constexpr int kEmitLanes = PV_EMIT_LANES;    // lanes per pillar when copying short lists
constexpr int kEmitPer = 32 / kEmitLanes;    // pillars in flight per warp
static_assert(kEmitLanes >= 2 && kEmitLanes <= 32 && 32 % kEmitLanes == 0, "emit batches tile a warp");
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // bounded spins: 1 s
constexpr int64_t kMaxAxisCells = int64_t(1) << 24;

// Control block of one workspace (device memory, zero at creation, epoch 1).
struct Control {
  unsigned int bar;     // grid-barrier arrivals in the running launch
  unsigned int done;    // blocks finished in the running launch
  int err;              // most negative status recorded in the running launch
  unsigned int dirty;   // 1: the table may hold stale entries
  unsigned int epoch;   // launch number
  unsigned int created; // unordered mode: pillars created in the running launch
  unsigned int pool;    // append lists: overflow lists handed out in the running launch
  unsigned int pad;
};

// Division of n < 2^31 by a divisor 1 <= d < 2^31 fixed per call, as one
// 64-bit multiply and a shift: with l = ceil(log2 d), s = 31 + l and
// m = ceil(2^s / d), the error e = m d - 2^s is below d <= 2^l, so n e < 2^s
// and floor(n m / 2^s) = floor(n / d); m <= 2^32, so n m fits 64 bits.
struct FastDiv {
  unsigned long long m;
  unsigned int s;
  unsigned int d;
};

__host__ __device__ __forceinline__ unsigned int fast_div(unsigned int n, const FastDiv& f) {
  return static_cast<unsigned int>((static_cast<unsigned long long>(n) * f.m) >> f.s);
}

inline FastDiv make_fast_div(unsigned int d) {
  unsigned int l = 0;
  while ((1ull << l) < d) ++l;
  FastDiv f;
  f.s = 31 + l;
  f.m = ((1ull << f.s) + d - 1) / d;
  f.d = d;
  return f;
}

struct KParams {
  const float4* points;
  long long n;
  long long chunk;   // points owned by each block in phase 2
  float lo_x, lo_y, lo_z;
  float v_x, v_y, v_z;
  float r_x, r_y, r_z;   // RN(1 / v) per axis, or 0 to always divide
  float g_xf, g_yf, g_zf;
  int g_x;
  int g_y;
  FastDiv div_x;     // by g_x
  FastDiv div_y;     // by g_y
  FastDiv div_cells; // by cells (a batched id's frame)
  int K;             // max_points
  int KT;            // tail entries per slot (max_points rounded up to 4, less kHead; >= 0)
  int append;        // 1: append lists (kAppendMinK <= max_points <= 32), 0: sorted lists
  int interleave;    // gather: 1: warp w takes ranks w, w + warps, ...; 0: a contiguous share
  int zero_tail;     // 1: rows V .. max_voxels-1 are zero-filled; 0: left as they were
  unsigned long long* pool;  // append lists: overflow lists, kHead + KT words each
  unsigned int pool_n;       // overflow lists available
  int max_voxels;
  int hash_mode;
  unsigned int bar_extra;  // test hook: extra arrivals the first barrier waits for
  unsigned int table_mask;
  unsigned long long* lists;  // heads [T][kHead], then tails [T][KT]; entries (leader << 32) | info
  unsigned long long* tails;  // lists + T * kHead
  int32_t* keys;
  int32_t* slot_of_point;
  int32_t* firsts;
  float4* tile_rows;     // [N] each tile's point rows, grouped by pillar
  unsigned long long* recs;  // [N] phase 1a records of a block's groups (the block's chunk region)
  unsigned int* counts;  // [kMaxCtas] first points per block
  Control* ctl;
  size_t list_words_cap;  // whole allocation (64-bit entries), for the dirty reset
  size_t key_words_cap;
  float4* out_voxels;
  int32_t* out_coords;
  int32_t* out_counts;
  int32_t* out_num;
  unsigned int* row_cnt;  // unordered mode: [max_voxels] points that reached each row (zero between calls)
  size_t row_cnt_cap;
  int frames;             // frames in the call (1 but for pv_voxelize_batch)
  int cells;              // voxels of one frame's grid; a batched id is frame * cells + id
  unsigned int* frame_cnt;  // batched: [frames + 1] first points of a frame start's block before it
  struct VoxAcc* acc;     // downsampling: [T] per-voxel sums (zero between calls)
  size_t acc_cap;
};

// Downsampling accumulator of one voxel (48 bytes, one L2 line half): the
// four fields summed in double, the point count, and the complement of the
// lowest point index (all-zero bytes = empty, so atomicMax finds the minimum).
struct VoxAcc {
  double s[4];
  unsigned int count;
  unsigned int first_c;
  unsigned int pad[2];
};
static_assert(sizeof(VoxAcc) == 48, "three 16-byte words");

// Frame start offsets of a batched call, passed by value with the launch
// (frame b is points [off[b], off[b + 1])).
constexpr int kMaxFrames = PV_MAX_FRAMES;
template <int NF>
struct Frames {
  long long off[NF + 1];
};

// Frame holding point i: the largest b < B with off[b] <= i (empty frames skipped).
__device__ __forceinline__ int frame_of(const long long* off, int B, long long i) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= i) lo = mid; else hi = mid;
  }
  return lo;
}

// Largest b < B with cum[b] <= k, for a non-decreasing cum.
__device__ __forceinline__ int slot_in_cum(const unsigned int* cum, int B, unsigned int k) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cum[mid] <= k) lo = mid; else hi = mid;
  }
  return lo;
}

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned int ld_relaxed(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ long long lmin(long long a, long long b) { return a < b ? a : b; }

__device__ __forceinline__ unsigned int atom_add_acq_rel(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Programmatic dependent launch: every launch of these kernels carries the
// programmatic stream serialization attribute, so the next launch's set-up
// may overlap this grid's end.  A kernel waits for the stream's previous
// grid to complete, its memory operations visible, before it touches
// memory, and lets the next grid launch once its own work is done.
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ unsigned int lanemask_lt() {
  unsigned int m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// ------------------------------------------------------------ instrumentation

// A PV_INSTRUMENT build stamps the global timer per block at each phase
// boundary (read back with pv_debug_phase_times); the normal build has none.
#ifdef PV_INSTRUMENT
constexpr int kStampCtas = 4096;
constexpr int kStamps = 8;
static __device__ unsigned long long g_phase_ns[kStampCtas][kStamps];
static __device__ unsigned long long g_p1_ns[kStampCtas][kStamps];
static __device__ unsigned long long g_insert_stats[4];  // inserts, atomics, rejected up front, max atomics
#define PV_SUB(k)                                                            \
  do {                                                                       \
    if (first_tile) {                                                        \
      __syncthreads();                                                       \
      if (threadIdx.x == 0 && blockIdx.x < kStampCtas)                       \
        g_p1_ns[blockIdx.x][k] = global_timer_ns();                          \
    }                                                                        \
  } while (0)
#define PV_STAMP(k)                                                          \
  do {                                                                       \
    __syncthreads();                                                         \
    if (threadIdx.x == 0 && blockIdx.x < kStampCtas)                         \
      g_phase_ns[blockIdx.x][k] = global_timer_ns();                         \
  } while (0)
#else
#define PV_STAMP(k) \
  do {              \
  } while (0)
#define PV_SUB(k) \
  do {            \
  } while (0)
#endif

// ------------------------------------------------------------ block-wide helpers

// All blocks of the cooperative launch arrive; returns false if the wait ran
// past the time limit (PV_ERR_TIMEOUT is then recorded).  `target` counts
// arrivals since the launch began (P for the first barrier, 2P for the next).
// Thread 0 arrives with a release reduction (the block's earlier writes are
// ordered before it by the CTA barrier), polls with relaxed loads, acquires
// the count once it is reached, and the closing CTA barrier passes the
// acquired view to the rest of the block.
static __device__ bool grid_sync(Control* ctl, unsigned int target, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    // No separate fences: the release reduction covers the block's earlier
    // writes (ordered before it by the CTA barrier above) and the acquire
    // load, with the CTA barrier below, passes the other blocks' writes on.
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&ctl->bar) : "memory");
    unsigned int v = ld_acquire(&ctl->bar);
    if (v < target) {
      const unsigned long long t0 = global_timer_ns();
      do {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          atomicMin(&ctl->err, PV_ERR_TIMEOUT);
          ok = 0;
          break;
        }
        v = ld_relaxed(&ctl->bar);  // relaxed polls; the count is acquired once it is reached
      } while (v < target);
      if (ok) v = ld_acquire(&ctl->bar);
    }
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}

// Exclusive prefix sum over the block; *total receives the block sum.
// Warp shuffle scan, then warp 0 scans the kWarps warp totals; s_tmp holds
// kWarps + 1 words.
static __device__ unsigned int block_exclusive_scan(unsigned int x, unsigned int* s_tmp, unsigned int* total) {
  const unsigned int lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  unsigned int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= static_cast<unsigned int>(o)) incl += y;
  }
  if (lane == 31) s_tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned int w = lane < static_cast<unsigned int>(kWarps) ? s_tmp[lane] : 0u;
    unsigned int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= static_cast<unsigned int>(o)) wi += y;
    }
    if (lane < static_cast<unsigned int>(kWarps)) s_tmp[lane] = wi - w;
    if (lane == 31) s_tmp[kWarps] = wi;
  }
  __syncthreads();
  const unsigned int before = s_tmp[warp];
  *total = s_tmp[kWarps];
  __syncthreads();  // s_tmp may be reused right after
  return before + incl - x;
}

// Exclusive prefix, in place, of the U x kWarps first-point counts
// (position u * kWarps + w: block tile u, warp w, in index order), run by
// warp 0; *total receives the sum.  Lane l sums the U consecutive positions
// from l * U, one warp scan orders the lanes' sums.
template <int U>
static __device__ __forceinline__ void flag_prefix(unsigned int* flat, unsigned int* total, unsigned int lane) {
  constexpr int E = U * kWarps / 32;  // consecutive (tile, warp) counts per lane
  static_assert(E >= 1 && U * kWarps % 32 == 0, "whole counts per lane");
  unsigned int c[E];
  unsigned int sum = 0;
#pragma unroll
  for (int k = 0; k < E; ++k) {
    c[k] = flat[lane * E + k];
    sum += c[k];
  }
  unsigned int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= static_cast<unsigned int>(o)) incl += y;
  }
  unsigned int run = incl - sum;
#pragma unroll
  for (int k = 0; k < E; ++k) {
    flat[lane * E + k] = run;
    run += c[k];
  }
  if (lane == 31) *total = incl;
}

// ------------------------------------------------------------ binning

__device__ __forceinline__ bool finite_bits(float f) {
  return (__float_as_uint(f) & 0x7f800000u) != 0x7f800000u;
}

// Cell of one coordinate: floorf of the IEEE round-to-nearest quotient
// RN((c - lo) / v), bounds tested on the float cell so a huge or infinite
// quotient never reaches the integer cast.
//
// The quotient is first estimated as qa = RN(d * RN(1 / v)).  Each of the two
// roundings is within a relative 2^-24, and RN(d / v) is within a relative
// 2^-24 of d / v, so |qa - RN(d / v)| < 1.5 * 2^-23 * qa (1 + 2^-22) < qa * 2^-22.
// When qa is farther than qa * 2^-22 from both neighbouring integers, no
// integer lies between qa and RN(d / v), so floorf(qa) is the exact cell;
// otherwise the cell is taken from the correctly rounded division itself.
// (qa - floor(qa) and floor(qa) + 1 - qa are exact for 0 <= qa < 2^24, and
// quotients in (0, 1) floor to 0 however they round, so the filter is safe for
// subnormal quotients too.)  A negative difference (not -0.0) has a negative
// quotient and is outside the grid.  rcp <= 0 turns the estimate off.
__device__ __forceinline__ bool bin_axis(float c, float lo, float v, float rcp, float g, int* cell) {
  const float d = __fsub_rn(c, lo);
  if (d < 0.0f) return false;
  float f;
  const float qa = __fmul_rn(d, rcp);
  const float fa = floorf(qa);
  const float tol = qa * 0x1p-22f;
  if (rcp > 0.0f && (qa - fa) > tol && (fa + 1.0f - qa) > tol) {
    f = fa;
  } else {
    f = floorf(__fdiv_rn(d, v));
  }
  const bool ok = (f >= 0.0f) && (f < g);
  *cell = ok ? static_cast<int>(f) : 0;
  return ok;
}

__device__ __forceinline__ bool bin_point(const float4& q, const KParams& p, int* key) {
  if (!(finite_bits(q.x) && finite_bits(q.y) && finite_bits(q.z))) return false;
  int cx, cy, cz;
  if (!bin_axis(q.x, p.lo_x, p.v_x, p.r_x, p.g_xf, &cx)) return false;
  if (!bin_axis(q.y, p.lo_y, p.v_y, p.r_y, p.g_yf, &cy)) return false;
  if (!bin_axis(q.z, p.lo_z, p.v_z, p.r_z, p.g_zf, &cz)) return false;
  *key = (cz * p.g_y + cy) * p.g_x + cx;  // cz = 0 on a pillar grid
  return true;
}

// ------------------------------------------------------------ pillar table

__device__ __forceinline__ unsigned int mix32(unsigned int h) {
  // Murmur3 finaliser: spreads ids that differ by large strides.
  h ^= h >> 16;
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  h *= 0xc2b2ae35u;
  h ^= h >> 16;
  return h;
}

// Find or claim the hashed slot of `key`.  At most table-size probes; -1 if
// the table is full.
#ifdef PV_INSTRUMENT
static __device__ unsigned long long g_probe_hist[34];  // lookups by positions probed: 1 .. 32, more, table full
#define PV_PROBES(n) atomicAdd(&g_probe_hist[(n) < 33u ? (n) : 33u], 1ull)
#else
#define PV_PROBES(n) \
  do {               \
  } while (0)
#endif

__device__ __forceinline__ int claim_slot(int32_t* keys, unsigned int mask, int key) {
  unsigned int h = mix32(static_cast<unsigned int>(key)) & mask;
  for (unsigned int probe = 0; probe <= mask; ++probe) {
    const int cur = __ldcg(keys + h);
    if (cur == key) {
      PV_PROBES(probe < 32u ? probe + 1u : 32u);
      return static_cast<int>(h);
    }
    if (cur == kNoKey) {
      const int old = atomicCAS(keys + h, kNoKey, key);
      if (old == kNoKey || old == key) {
        PV_PROBES(probe < 32u ? probe + 1u : 32u);
        return static_cast<int>(h);
      }
    }
    h = (h + 1) & mask;
  }
  PV_PROBES(33u);
  return -1;
}

// Insert entry x into list L, which keeps the K smallest entries of a pillar
// in ascending order.  An entry is (leader index << 32) | group info, and
// leader indices are distinct, so entries order like their leaders.  The
// atomicMin cascade: each position keeps the minimum of what reaches it and
// passes the larger value on, so position k ends as the (k+1)-th smallest
// whatever order inserts arrive in.  An entry may enter the cascade at any
// position that does not exceed its final rank: the positions it skips would
// have kept a smaller entry and passed it on unchanged.  The bound used is
// crank (the number of this chunk's groups of the pillar before x, exact)
// plus the length of the strictly increasing run of entries read below x
// that come from other chunks (leaders outside [cbase, cbase + cspan)):
// distinct smaller leaders, none counted twice.  Values in a list only ever
// decrease, so an entry read below x stays below x.  Only the head row is
// read up front; the tail only while the run goes on.
//
// A group whose pillar has K points before it never contributes a point.
// The groups of that run lie in other tiles than x's and have smaller
// leaders, so all their points come before x's: when their sizes add up to K
// the entry is dropped.  Dropping such entries changes nothing for the
// others: every entry compares below a dropped one, so the needed entries
// (those with fewer than K points before them) cascade exactly as if it had
// never existed and end in positions 0, 1, ... in order, which is all the
// emit reads before it has K points.
__device__ __forceinline__ unsigned long long ull_of(uint32_t lo, uint32_t hi) {
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}

// Append lists (8 <= max_points <= 32).  A slot's S = kHead + KT words:
// word 0 is (lowest leader << 32) | ~count, words 1 .. S-2 hold the first
// S-2 entries in arrival order, word S-1 the index of the slot's overflow
// list.  All-ones is the empty slot (count 0, no leader, no overflow list).
// An insert is one atomicAdd on the count (its arrival index) and one
// atomicMin on the lowest leader, then a plain store of the entry: no
// cascade.  Entries past S-2 go, sorted by the cascade of list_insert, into
// an overflow list taken from a pool by the slot's first overflowing entry;
// the later ones wait (bounded) for its index.  The gather sorts the stored
// entries in a warp and merges the overflow list in.
constexpr int kAppendMinK = 8;

__device__ __forceinline__ unsigned long long* slot_word(unsigned long long* head, unsigned long long* tail, int w) {
  return w < kHead ? head + w : tail + (w - kHead);
}

// List entry: (leader index << 32) | (chunk rank << 22) | (d << 10) | (size - 1),
// where the group's rows start in tile_rows at leader index + d (d signed,
// 12 bits: a group lies inside its block tile of at most 2048 points), the
// chunk rank is below max_points <= 1024, and size is the group's point
// count capped at max_points (1 .. 1024): no group contributes more, and a
// capped size still tells that max_points points lie before later groups.
__device__ __forceinline__ unsigned long long make_entry(long long leader, unsigned int crank, long long row,
                                                         unsigned int size) {
  const unsigned int d = static_cast<unsigned int>(row - leader) & 4095u;
  return (static_cast<unsigned long long>(leader) << 32) | (crank << 22) | (d << 10) | (size - 1u);
}
__device__ __forceinline__ long long entry_row(unsigned long long ent) {
  const int d = static_cast<int>(static_cast<unsigned int>(ent) << 10) >> 20;  // bits 10..21, sign-extended
  return static_cast<long long>(ent >> 32) + d;
}
__device__ __forceinline__ unsigned int entry_size(unsigned long long ent) {
  return (static_cast<unsigned int>(ent) & 1023u) + 1u;
}
__device__ __forceinline__ int entry_crank(unsigned long long ent) {
  return static_cast<int>((static_cast<unsigned int>(ent) >> 22) & 1023u);
}

// A slot's list: positions 0 .. kHead-1 in its head row, the rest in its tail row.
struct ListRef {
  unsigned long long* head;
  unsigned long long* tail;
  __device__ __forceinline__ unsigned long long* at(int k) const { return k < kHead ? head + k : tail + (k - kHead); }
};

__device__ __forceinline__ ListRef list_of(const KParams& p, int slot) {
  return ListRef{p.lists + static_cast<size_t>(slot) * kHead, p.tails + static_cast<size_t>(slot) * p.KT};
}

// h: the list's head row, read by the caller (any time earlier: a stale
// copy only shortens the run).
__device__ __forceinline__ void list_insert(const ListRef& L, const uint4 (&h)[kHead / 2], int K, int KT,
                                            unsigned long long x, int crank, uint32_t cbase, uint32_t cspan) {
  const uint4 e4 = make_uint4(kEmpty, kEmpty, kEmpty, kEmpty);
  int a = 0;
  unsigned int before = 0;  // points in the run's groups
  unsigned long long prev = 0;
  bool run = true;
  auto step = [&](unsigned long long y) {
    if (!run || static_cast<uint32_t>(y >> 32) - cbase < cspan) return;  // own chunk: counted by crank
    if (y < x && (a == 0 || y > prev)) {
      prev = y;
      ++a;
      before += entry_size(y);
    } else {
      run = false;
    }
  };
#pragma unroll
  for (int t = 0; t < kHead / 2; ++t) {
    step(ull_of(h[t].x, h[t].y));
    step(ull_of(h[t].z, h[t].w));
  }
  for (int e = 0; run && kHead + e < K && before < static_cast<unsigned int>(K); e += 8) {  // tail: 8 per trip
    uint4 q[4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
      q[t] = (e + 2 * t < KT) ? __ldcg(reinterpret_cast<const uint4*>(L.tail + e + 2 * t)) : e4;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      step(ull_of(q[t].x, q[t].y));
      step(ull_of(q[t].z, q[t].w));
    }
  }
  if (before >= static_cast<unsigned int>(K)) {
#ifdef PV_INSTRUMENT_INSERTS
    atomicAdd(&g_insert_stats[2], 1ull);
#endif
    return;
  }
  // Stride padding past K reads empty, so a >= K only if K entries are below x.
#ifdef PV_INSTRUMENT_INSERTS
  unsigned long long n_atomics = 0;
#endif
  for (int k = a + crank; k < K; ++k) {
    const unsigned long long old = atomicMin(L.at(k), x);
#ifdef PV_INSTRUMENT_INSERTS
    ++n_atomics;
#endif
    if (old == kEmpty64) break;
    x = old > x ? old : x;
  }
#ifdef PV_INSTRUMENT_INSERTS
  atomicAdd(&g_insert_stats[0], 1ull);
  atomicAdd(&g_insert_stats[1], n_atomics);
  atomicMax(&g_insert_stats[3], n_atomics);
#endif
}

// Append-list insert of entry x into slot L (see kAppendMinK).  cbase/cspan:
// this block's chunk (for the overflow list's cascade).
static __device__ void append_insert(const KParams& p, const ListRef& L, unsigned long long x, uint32_t cbase,
                              uint32_t cspan) {
  const int S = kHead + p.KT;
  unsigned int* w0 = reinterpret_cast<unsigned int*>(L.head);
  const unsigned int j = ~atomicAdd(w0, 0xFFFFFFFFu);  // the count is kept complemented
  // Only a chunk's first group of the pillar (chunk rank 0, also what a
  // full chunk map reports) can hold the lowest leader: the chunk's other
  // groups come after it.
  if (entry_crank(x) == 0) atomicMin(w0 + 1, static_cast<unsigned int>(x >> 32));
  if (j < static_cast<unsigned int>(S - 2)) {
    *slot_word(L.head, L.tail, 1 + static_cast<int>(j)) = x;
    return;
  }
  // Overflow: the first overflowing entry takes a list from the pool and
  // publishes its index in word S-1; the others wait for it (bounded).
  unsigned long long* ow = slot_word(L.head, L.tail, S - 1);
  unsigned long long idx = kEmpty64;
  if (j == static_cast<unsigned int>(S - 2)) {
    const unsigned int got = atomicAdd(&p.ctl->pool, 1u);
    idx = got;
    // Published even when it is out of range (the pool is exhausted), so
    // that the waiters leave at once through their range check.
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(ow), "l"(idx) : "memory");
    if (got >= p.pool_n) {
      atomicMin(&p.ctl->err, PV_ERR_CAPACITY);
      return;
    }
  } else {
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(idx) : "l"(ow) : "memory");
    if (idx == kEmpty64) {
      const unsigned long long t0 = global_timer_ns();
      do {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          atomicMin(&p.ctl->err, PV_ERR_TIMEOUT);
          return;
        }
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(idx) : "l"(ow) : "memory");
      } while (idx == kEmpty64);
    }
    if (idx >= p.pool_n) return;  // the taker ran out of pool and recorded it
  }
  unsigned long long* base = p.pool + idx * static_cast<unsigned long long>(S);
  const ListRef O{base, base + kHead};
  uint4 h[kHead / 2];
#pragma unroll
  for (int t = 0; t < kHead / 2; ++t) h[t] = __ldcg(reinterpret_cast<const uint4*>(base) + t);
  list_insert(O, h, p.K, p.KT, x, 0, cbase, cspan);
}

// ------------------------------------------------------------ block tiles

// Shared-memory grouping of one block tile (kThreads or 2 kThreads
// consecutive points, each warp holding a run of 32 or 64 of them): an
// open-addressing map slot -> map position, per (position, warp) the number
// of the warp's points in that slot, and per position the group's offset in
// the tile's grouped layout.  A point's rank among the tile's points of its
// pillar is the sum over earlier warps plus its rank in its own warp's run.
// The map has a position per point of the largest tile, so it never fills.
constexpr int kTileHash = 2 * kThreads;

constexpr int kChunkHash = 4096;   // chunk map positions (see chunk_rank)
#ifndef PV_CHUNK_PROBES
#define PV_CHUNK_PROBES 8
#endif
constexpr int kChunkProbes = PV_CHUNK_PROBES;  // a full chunk map costs this many probes per lookup

// Dynamic shared memory of the kernel: two tile maps, used by alternate
// tiles so one can be emptied while the other is filled.
constexpr int kMapBytes = kTileHash * kWarps + kTileHash * 4 + kTileHash * 4;
constexpr int kDynSmem = 2 * kMapBytes + 2 * 4 * kChunkHash;
static_assert(kMapBytes % 16 == 0, "maps stay 16-byte aligned");
static_assert(kWarps * 32 * 8 <= kMapBytes, "the gather's merge buffers fit one tile map");
// After phase 1 the same shared memory holds the gather's per-warp merge
// buffers (32 entries each) and the block's queue of long lists (at most
// kQueueCap entries; fewer when the launch has less dynamic shared memory).
constexpr unsigned int kQueueCap = kDynSmem / 8 - kWarps * 32;
constexpr unsigned int kQueueDrop = 0xFFFFFFFFu;  // queue row of a list past the budget (emptied only)
constexpr int64_t kQueueMinRowsPerWarp = 8;        // rows per warp from which the gather queues long lists

struct TileMap {
  unsigned int* cnt;         // [kTileHash][kWarps / 4] packed byte counters
  int* key;                  // [kTileHash], -1 = free
  unsigned int* off;         // [kTileHash] (rows to write << 16) | group offset in the tile layout
  unsigned int* layout;      // rows handed out in the tile layout
};

static __device__ __forceinline__ TileMap tile_map(unsigned char* base, unsigned int* layout) {
  TileMap m;
  m.cnt = reinterpret_cast<unsigned int*>(base);
  m.key = reinterpret_cast<int*>(base + kTileHash * kWarps);
  m.off = reinterpret_cast<unsigned int*>(base + kTileHash * kWarps + kTileHash * 4);
  m.layout = layout;
  return m;
}

// Empty the map positions h = tid, tid + kThreads, ... (keys and counters).
static __device__ __forceinline__ void tile_clear(const TileMap& m, unsigned int tid) {
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int h = static_cast<int>(tid); h < kTileHash; h += kThreads) {
    if (m.key[h] != -1) {
      m.key[h] = -1;
      uint4* row = reinterpret_cast<uint4*>(m.cnt + h * (kWarps / 4));
#pragma unroll
      for (int r = 0; r < kWarps / 16; ++r) row[r] = z;
    }
  }
}

// The warp-group leader claims (or finds) the map position of `slot`.
static __device__ __forceinline__ int tile_claim(const TileMap& m, int slot) {
  unsigned int h = mix32(static_cast<unsigned int>(slot)) & (kTileHash - 1);
  for (int probe = 0; probe < kTileHash; ++probe) {  // at most kThreads keys: never full
    const int cur = atomicCAS(m.key + h, -1, slot);
    if (cur == -1 || cur == slot) return static_cast<int>(h);
    h = (h + 1) & (kTileHash - 1);
  }
  return -1;
}

// Chunk map: pillar -> (tile groups << 16) | points of this block's chunk
// seen so far.  Tiles of a chunk are grouped one after the other, so what a
// tile group reads is its rank among the chunk's groups of the pillar and the
// number of the pillar's points in earlier tiles of the chunk.  Both are
// exact while they matter: a group is kept only with fewer than max_points
// (<= 1024) points before it, so neither field has wrapped by then; after
// that the values only decide to drop the group.  When the map is full both
// fall back to 0, which is still a valid lower bound.

static __device__ __forceinline__ unsigned int chunk_rank(int* ckey, unsigned int* ccnt, int slot, unsigned int size) {
  unsigned int h = mix32(static_cast<unsigned int>(slot) ^ 0x9e3779b9u) & (kChunkHash - 1);
  for (int probe = 0; probe < kChunkProbes; ++probe) {
    int cur = *reinterpret_cast<volatile int*>(ckey + h);  // a plain read first: most probes find a key
    if (cur == -1) cur = atomicCAS(ckey + h, -1, slot);
    if (cur == -1 || cur == slot) return atomicAdd(ccnt + h, (1u << 16) | size);
    h = (h + 1) & (kChunkHash - 1);
  }
  return 0u;
}

// Byte counters at map position h: *before = warps 0 .. warp-1, *total = all.
// Each word holds four warps' counts (at most 64 each), summed with dp4a
// against ones; the words before this warp's count whole, its own word only
// in the bytes of lower warps.
static __device__ __forceinline__ void tile_counts(const TileMap& m, int h, unsigned int warp, unsigned int* before,
                                            unsigned int* total) {
  const uint4* row = reinterpret_cast<const uint4*>(m.cnt + static_cast<size_t>(h) * (kWarps / 4));
  const unsigned int pc = warp >> 2;                       // word holding this warp's byte
  const unsigned int pm = (1u << (8u * (warp & 3u))) - 1u;  // bytes of lower warps in that word
  unsigned int b = 0, t = 0;
#pragma unroll
  for (int r = 0; r < kWarps / 16; ++r) {
    const uint4 q = row[r];
    const unsigned int w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const unsigned int idx = static_cast<unsigned int>(4 * r + c);
      t = __dp4a(w[c], 0x01010101u, t);
      const unsigned int msk = idx < pc ? 0xFFFFFFFFu : (idx == pc ? pm : 0u);
      b = __dp4a(w[c] & msk, 0x01010101u, b);
    }
  }
  *before = b;
  *total = t;
}

// Slot of the pillar with rank r: binary search of the owner block in the
// exclusive prefix (s_prefix[0..P], s_prefix[P] = total), then its
// compacted first-point list.
__device__ __forceinline__ int slot_of_rank(const KParams& p, const unsigned int* s_prefix, unsigned int P,
                                            unsigned int r) {
  unsigned int lo = 0, hi = P;  // invariant: s_prefix[lo] <= r < s_prefix[hi]
  while (hi - lo > 1) {
    const unsigned int mid = (lo + hi) >> 1;
    if (s_prefix[mid] <= r) lo = mid; else hi = mid;
  }
  return __ldcg(p.firsts + static_cast<long long>(lo) * p.chunk + (r - s_prefix[lo]));
}

// The head row of a pillar's slot, as one lane reads it: a sorted list's
// first four entries, or an append list's first three entries sorted here.
// few: the pillar's points all come from groups among them: either the list
// ends there (a sorted list: a group is missing after ng present ones and
// the groups hold fewer than max_points points, and a needed group is never
// missing before another, so nothing follows; an append list: it holds at
// most three entries, all present) or the first ng groups already hold
// max_points points (filled; unused entries may then follow anywhere).
struct Head {
  unsigned long long e[4];
  unsigned int n;   // points taken: min(points of the first ng groups, max_points)
  int ng;           // groups the points come from (0: none present)
  bool few;
  bool filled;
};

__device__ __forceinline__ Head read_head(const KParams& p, const unsigned long long* L, bool valid) {
  Head h;
  uint4 a = make_uint4(kEmpty, kEmpty, kEmpty, kEmpty), b = a;
  if (valid) {  // positions 0..3 (head row; positions past max_points are never written and read empty)
    a = __ldcg(reinterpret_cast<const uint4*>(L));
    b = __ldcg(reinterpret_cast<const uint4*>(L) + 1);
  }
  if (p.append) {
    // Word 0: the count (complemented); words 1..3: the first three entries
    // in arrival order, sorted here.  Served from the head only when the
    // slot holds at most three entries.
    const unsigned int cnt = ~a.x;
    unsigned long long e0 = ull_of(a.z, a.w), e1 = ull_of(b.x, b.y), e2 = ull_of(b.z, b.w);
    if (cnt < 3u) e2 = kEmpty64;
    if (cnt < 2u) e1 = kEmpty64;
    if (cnt < 1u) e0 = kEmpty64;
    const unsigned long long m01 = e0 < e1 ? e0 : e1, x01 = e0 < e1 ? e1 : e0;
    const unsigned long long m12 = x01 < e2 ? x01 : e2, x12 = x01 < e2 ? e2 : x01;
    h.e[0] = m01 < m12 ? m01 : m12;
    h.e[1] = m01 < m12 ? m12 : m01;
    h.e[2] = x12;
    h.e[3] = kEmpty64;
    unsigned int cum = 0;
    int g = 0;
    bool filled = false;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const bool good = h.e[j] != kEmpty64 && (h.e[j] >> 32) < static_cast<unsigned long long>(p.n);
      if (!filled && g == j && good) {
        cum += entry_size(h.e[j]);
        g = j + 1;
        if (cum >= static_cast<unsigned int>(p.K)) filled = true;
      }
    }
    h.ng = g;
    h.filled = filled;
    h.few = g > 0 && cnt <= 3u && (filled || static_cast<unsigned int>(g) == cnt);
    h.n = filled ? static_cast<unsigned int>(p.K) : cum;
    return h;
  }
  h.e[0] = ull_of(a.x, a.y);
  h.e[1] = ull_of(a.z, a.w);
  h.e[2] = ull_of(b.x, b.y);
  h.e[3] = ull_of(b.z, b.w);
  unsigned int cum = 0;
  int g = 0;
  bool filled = false, gap_clean = true;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const bool good = h.e[j] != kEmpty64 && (h.e[j] >> 32) < static_cast<unsigned long long>(p.n);
    if (!filled && g == j && good) {
      cum += entry_size(h.e[j]);
      g = j + 1;
      if (cum >= static_cast<unsigned int>(p.K)) filled = true;
    } else if (!filled && h.e[j] != kEmpty64) {
      gap_clean = false;  // something after a missing or bad position
    }
  }
  h.ng = g;
  h.filled = filled;
  h.few = g > 0 && (filled || (g < 4 && gap_clean));
  h.n = filled ? static_cast<unsigned int>(p.K) : cum;
  return h;
}

// Copy descriptor of a pillar served by its first groups, computed by the
// lane that read its head: the points taken n, the starts of groups 1..3 in
// the output row (clamped to n; a missing group starts at n), and per group
// j its first point's row in tile_rows minus its start, so that position e
// of group j comes from row o[j] + e.
struct CopyDesc {
  unsigned int w0;  // n | s1 << 16
  unsigned int w1;  // s2 | s3 << 16
  int o[4];
};

__device__ __forceinline__ CopyDesc copy_desc(const Head& h) {
  CopyDesc d;
  unsigned int st[4];
  unsigned int run = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const unsigned long long ej = h.e[j];
    d.o[j] = static_cast<int>(entry_row(ej) - static_cast<long long>(run));
    st[j] = j < h.ng ? (run < h.n ? run : h.n) : h.n;
    run += entry_size(ej);  // (unused past the groups present)
  }
  d.w0 = h.n | (st[1] << 16);
  d.w1 = st[2] | (st[3] << 16);
  return d;
}

// Writes the output row of a pillar from its whole list: groups in list
// order, each group's points in index order, max_points at most, zeros
// after them; empties every list position.  Returns the points written.
// All 32 lanes call it with the same arguments.  With max_points <= 32 and
// the groups in positions 0 .. G-1, lane e takes position e from the last
// group whose running start is <= e; otherwise the groups are walked 32
// list positions at a time.  An entry whose leader is out of range (never
// in a clean table) is skipped and reported through *stale.
static __device__ unsigned int emit_groups(const KParams& p, const ListRef& L, float4* orow, int K, unsigned int lane,
                                    bool* stale) {
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  const unsigned long long raw = static_cast<int>(lane) < K ? __ldcg(L.at(lane)) : kEmpty64;
  unsigned long long ent = raw;
  if (ent != kEmpty64 && (ent >> 32) >= static_cast<unsigned long long>(p.n)) {
    ent = kEmpty64;
    *stale = true;
  }
  const unsigned int present = __ballot_sync(0xffffffffu, ent != kEmpty64);
  unsigned int written = 0;
  if (K <= 32 && (present & (present + 1u)) == 0u) {
    const int G = __popc(present);
    const unsigned int size = ent != kEmpty64 ? entry_size(ent) : 0u;
    unsigned int incl = size;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= static_cast<unsigned int>(o)) incl += y;
    }
    const int gstart = static_cast<int>(incl - size);
    const unsigned int all = __shfl_sync(0xffffffffu, incl, 31);
    written = all < static_cast<unsigned int>(K) ? all : static_cast<unsigned int>(K);
    const int e = static_cast<int>(lane);
    int g = 0;
#pragma unroll
    for (int step = 16; step >= 1; step >>= 1) {
      const int j = g + step;
      const int st = __shfl_sync(0xffffffffu, gstart, j < 32 ? j : 31);
      if (j < G && st <= e) g = j;
    }
    const unsigned long long ge = __shfl_sync(0xffffffffu, ent, g);
    const int gs = __shfl_sync(0xffffffffu, gstart, g);
    if (e < K) {
      float4 row = z4;
      if (static_cast<unsigned int>(e) < written) {
        row = __ldcg(p.tile_rows + entry_row(ge) + (e - gs));
      }
      orow[e] = row;
    }
    if (raw != kEmpty64) *L.at(lane) = kEmpty64;
    return written;
  }
  unsigned long long chunk = ent, chunk_raw = raw;
  for (int g0 = 0; g0 < K; g0 += 32) {
    if (g0 > 0) {
      chunk_raw = (g0 + static_cast<int>(lane) < K) ? __ldcg(L.at(g0 + lane)) : kEmpty64;
      chunk = chunk_raw;
      if (chunk != kEmpty64 && (chunk >> 32) >= static_cast<unsigned long long>(p.n)) {
        chunk = kEmpty64;
        *stale = true;
      }
    }
    const unsigned int here = __ballot_sync(0xffffffffu, chunk != kEmpty64);
    for (unsigned int m = here; m != 0u && written < static_cast<unsigned int>(K); m &= m - 1u) {
      const unsigned long long ge = __shfl_sync(0xffffffffu, chunk, __ffs(m) - 1);
      const unsigned int gsz = entry_size(ge);
      const unsigned int room = static_cast<unsigned int>(K) - written;
      const unsigned int n = gsz < room ? gsz : room;
      const long long base = entry_row(ge);
      for (unsigned int j = lane; j < n; j += 32) orow[written + j] = __ldcg(p.tile_rows + base + j);
      written += n;
    }
    if (chunk_raw != kEmpty64) *L.at(g0 + lane) = kEmpty64;
  }
  for (unsigned int e = written + lane; e < static_cast<unsigned int>(K); e += 32) orow[e] = z4;
  return written;
}

// Empties an append slot, and its overflow list if it has one.  All 32
// lanes call it with the same slot.
static __device__ void app_clear_with(const KParams& p, const ListRef& L, unsigned int lane, unsigned long long ow) {
  const int S = kHead + p.KT;
  if (ow < p.pool_n) {
    unsigned long long* base = p.pool + ow * static_cast<unsigned long long>(S);
    for (int w = static_cast<int>(lane); w < S; w += 32) base[w] = kEmpty64;
  }
  __syncwarp();
  for (int w = static_cast<int>(lane); w < S; w += 32) *slot_word(L.head, L.tail, w) = kEmpty64;
}

static __device__ void app_clear(const KParams& p, const ListRef& L, unsigned int lane) {
  app_clear_with(p, L, lane, __ldcg(slot_word(L.head, L.tail, kHead + p.KT - 1)));
}

// Writes the output row of an append-list pillar that is not served from
// its head: lane l reads stored entry l, the warp sorts them by leader
// (bitonic), merges in the slot's sorted overflow list if it has one (the
// first 32 of the union, through a per-warp shared buffer), and copies the
// first max_points points as emit_groups does; empties the slot.  All 32
// lanes call it with the same arguments (max_points <= 32).
static __device__ unsigned int emit_app(const KParams& p, const ListRef& L, float4* orow, int K, unsigned int lane,
                                 unsigned long long* wbuf, bool* stale) {
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  const int S = kHead + p.KT;
  // Lane w reads word w of the slot (one round trip for the count, the
  // stored entries and the overflow index); entry j moves to lane j.
  const unsigned long long word = static_cast<int>(lane) < S ? __ldcg(slot_word(L.head, L.tail, lane)) : kEmpty64;
  const unsigned int cnt = ~static_cast<unsigned int>(__shfl_sync(0xffffffffu, static_cast<unsigned int>(word), 0));
  const int nent = cnt < static_cast<unsigned int>(S - 2) ? static_cast<int>(cnt) : S - 2;
  const unsigned long long next = (static_cast<unsigned long long>(__shfl_down_sync(0xffffffffu, static_cast<unsigned int>(word >> 32), 1)) << 32) |
                                  __shfl_down_sync(0xffffffffu, static_cast<unsigned int>(word), 1);
  unsigned long long ent = static_cast<int>(lane) < nent ? next : kEmpty64;
  const unsigned long long owl = (static_cast<unsigned long long>(__shfl_sync(0xffffffffu, static_cast<unsigned int>(word >> 32), S - 1)) << 32) |
                                 __shfl_sync(0xffffffffu, static_cast<unsigned int>(word), S - 1);
  const unsigned long long ow = cnt > static_cast<unsigned int>(S - 2) ? owl : kEmpty64;
  if (ent != kEmpty64 && (ent >> 32) >= static_cast<unsigned long long>(p.n)) {
    ent = kEmpty64;
    *stale = true;
  }
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, ent, j);
      const bool up = (lane & static_cast<unsigned int>(k)) == 0u;
      const bool lower = (lane & static_cast<unsigned int>(j)) == 0u;
      const unsigned long long mn = ent < o ? ent : o, mx = ent < o ? o : ent;
      ent = (lower == up) ? mn : mx;
    }
  }
  if (cnt > static_cast<unsigned int>(S - 2)) {
    // The overflow list holds the smallest of the entries that did not fit,
    // ascending in positions 0 .. max_points-1.
    unsigned long long ov = kEmpty64;
    if (ow < p.pool_n) {
      const unsigned long long* base = p.pool + ow * static_cast<unsigned long long>(S);
      ov = static_cast<int>(lane) < K ? __ldcg(slot_word(const_cast<unsigned long long*>(base),
                                                         const_cast<unsigned long long*>(base) + kHead, lane))
                                      : kEmpty64;
      if (ov != kEmpty64 && (ov >> 32) >= static_cast<unsigned long long>(p.n)) {
        ov = kEmpty64;
        *stale = true;
      }
    } else {
      *stale = true;  // a count past the stored entries without an overflow list
    }
    // Rank of each element in the union (leaders are distinct): its own
    // index plus the number of the other list's elements below it.
    int ra = 0, rb = 0;  // elements of the other list below ent / below ov
#pragma unroll
    for (int step = 16; step >= 1; step >>= 1) {
      const unsigned long long ob = __shfl_sync(0xffffffffu, ov, ra + step - 1);
      if (ob < ent) ra += step;
      const unsigned long long oa = __shfl_sync(0xffffffffu, ent, rb + step - 1);
      if (oa < ov) rb += step;
    }
    {
      const unsigned long long ob = __shfl_sync(0xffffffffu, ov, ra < 32 ? ra : 31);
      if (ra < 32 && ob < ent) ++ra;
      const unsigned long long oa = __shfl_sync(0xffffffffu, ent, rb < 32 ? rb : 31);
      if (rb < 32 && oa < ov) ++rb;
    }
    const int pa = static_cast<int>(lane) + ra, pb = static_cast<int>(lane) + rb;
    if (ent != kEmpty64 && pa < 32) wbuf[pa] = ent;
    if (ov != kEmpty64 && pb < 32) wbuf[pb] = ov;
    const unsigned int na = __popc(__ballot_sync(0xffffffffu, ent != kEmpty64));
    const unsigned int nb = __popc(__ballot_sync(0xffffffffu, ov != kEmpty64));
    __syncwarp();
    ent = lane < na + nb ? wbuf[lane] : kEmpty64;
    __syncwarp();
  }
  const unsigned int present = __ballot_sync(0xffffffffu, ent != kEmpty64);
  const int G = __popc(present);
  const unsigned int size = ent != kEmpty64 ? entry_size(ent) : 0u;
  unsigned int incl = size;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= static_cast<unsigned int>(o)) incl += y;
  }
  const int gstart = static_cast<int>(incl - size);
  const unsigned int all = __shfl_sync(0xffffffffu, incl, 31);
  const unsigned int written = all < static_cast<unsigned int>(K) ? all : static_cast<unsigned int>(K);
  const int e = static_cast<int>(lane);
  int g = 0;
#pragma unroll
  for (int step = 16; step >= 1; step >>= 1) {
    const int jj = g + step;
    const int st = __shfl_sync(0xffffffffu, gstart, jj < 32 ? jj : 31);
    if (jj < G && st <= e) g = jj;
  }
  const unsigned long long ge = __shfl_sync(0xffffffffu, ent, g);
  const int gs = __shfl_sync(0xffffffffu, gstart, g);
  if (e < K) {
    float4 row = z4;
    if (static_cast<unsigned int>(e) < written) row = __ldcg(p.tile_rows + entry_row(ge) + (e - gs));
    orow[e] = row;
  }
  app_clear_with(p, L, lane, owl);
  return written;
}

// Up to four queued append-list pillars at once, eight lanes each (group g =
// lanes 8g .. 8g+7, with the queue entry `qe` valid where `mine`).  A kept
// pillar whose slot holds at most min(7, S - 2) entries (so no overflow list)
// is served here: its group reads slot words 0..7 (one request a group), lane
// s takes entry s (word s + 1), the group sorts its entries by leader (a
// bitonic network over 8 lanes), sums the group sizes, and copies positions
// s, s + 8, s + 16, s + 24 of the row, zeros past the points taken, then
// writes the count and empties the words it read.  Returns true on the lanes
// of a group whose pillar needs the whole-warp way (more entries, an overflow
// list, or a list past the budget).  All 32 lanes call it.
static __device__ bool emit_app_quad(const KParams& p, unsigned long long qe, bool mine, unsigned int lane, int K,
                              bool* stale) {
  const unsigned int sl = lane & 7u, base = lane & ~7u;
  const int S = kHead + p.KT;
  const unsigned int qrow = static_cast<unsigned int>(qe >> 32);
  const bool kept = mine && qrow != kQueueDrop;
  const ListRef L = list_of(p, kept ? static_cast<int>(static_cast<unsigned int>(qe)) : 0);
  const unsigned long long w = kept ? __ldcg(slot_word(L.head, L.tail, static_cast<int>(sl))) : kEmpty64;
  const unsigned int cnt = ~__shfl_sync(0xffffffffu, static_cast<unsigned int>(w), static_cast<int>(base));
  const unsigned int cap = S - 2 < 7 ? static_cast<unsigned int>(S - 2) : 7u;
  const bool fast = kept && cnt >= 1u && cnt <= cap;
  const int src = lane < 31u ? static_cast<int>(lane) + 1 : 31;  // entry s is word s + 1 (s < cnt <= 7)
  unsigned long long ent = (static_cast<unsigned long long>(__shfl_sync(0xffffffffu, static_cast<unsigned int>(w >> 32), src)) << 32) |
                           __shfl_sync(0xffffffffu, static_cast<unsigned int>(w), src);
  if (!(fast && sl < cnt)) ent = kEmpty64;
  if (ent != kEmpty64 && (ent >> 32) >= static_cast<unsigned long long>(p.n)) {
    ent = kEmpty64;
    *stale = true;
  }
#pragma unroll
  for (int size = 2; size <= 8; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int o_src = static_cast<int>(lane ^ static_cast<unsigned int>(stride));
      const unsigned long long o = (static_cast<unsigned long long>(__shfl_sync(0xffffffffu, static_cast<unsigned int>(ent >> 32), o_src)) << 32) |
                                   __shfl_sync(0xffffffffu, static_cast<unsigned int>(ent), o_src);
      const bool up = (sl & static_cast<unsigned int>(size)) == 0u;
      const bool lower = (sl & static_cast<unsigned int>(stride)) == 0u;
      const unsigned long long mn = ent < o ? ent : o, mx = ent < o ? o : ent;
      ent = (lower == up) ? mn : mx;
    }
  }
  const unsigned int sz = ent != kEmpty64 ? entry_size(ent) : 0u;
  unsigned int incl = sz;
#pragma unroll
  for (int d = 1; d < 8; d <<= 1) {
    const unsigned int y = __shfl_up_sync(0xffffffffu, incl, d, 8);
    if (sl >= static_cast<unsigned int>(d)) incl += y;
  }
  const unsigned int st = incl - sz;  // the group's first position in the row
  const unsigned int all = __shfl_sync(0xffffffffu, incl, static_cast<int>(base) + 7);
  const unsigned int tk = all < static_cast<unsigned int>(K) ? all : static_cast<unsigned int>(K);
  const unsigned int G = (__ballot_sync(0xffffffffu, ent != kEmpty64) >> base) & 0xFFu;
  const int ng = __popc(G);
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 v[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const unsigned int e = sl + 8u * static_cast<unsigned int>(k);
    int gi = 0;
#pragma unroll
    for (int step = 4; step >= 1; step >>= 1) {
      const int c = gi + step;
      const unsigned int sc = __shfl_sync(0xffffffffu, st, static_cast<int>(base) + (c < 8 ? c : 7));
      if (c < ng && sc <= e) gi = c;
    }
    const int gl = static_cast<int>(base) + gi;
    const unsigned long long ge = (static_cast<unsigned long long>(__shfl_sync(0xffffffffu, static_cast<unsigned int>(ent >> 32), gl)) << 32) |
                                  __shfl_sync(0xffffffffu, static_cast<unsigned int>(ent), gl);
    const unsigned int gs = __shfl_sync(0xffffffffu, st, gl);
    v[k] = (fast && e < tk) ? __ldcg(p.tile_rows + entry_row(ge) + (e - gs)) : z4;
  }
  if (fast) {
    float4* orow = p.out_voxels + static_cast<size_t>(qrow) * K;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const unsigned int e = sl + 8u * static_cast<unsigned int>(k);
      if (e < static_cast<unsigned int>(K)) orow[e] = v[k];
    }
    if (sl == 0u) p.out_counts[qrow] = static_cast<int32_t>(tk);
  }
  __syncwarp();
  if (fast) *slot_word(L.head, L.tail, static_cast<int>(sl)) = kEmpty64;  // words 0..7: the count and every entry
  return mine && !fast;
}

// Recovery after a failed launch (the control block's dirty flag): every
// table a launch of any kind fills is emptied whole, since the next launch
// may be of another kind: lists, hashed keys, unordered-mode row counters,
// downsampling accumulators.  A grid barrier must follow.
static __device__ void reset_tables(const KParams& p, size_t gtid, size_t gthreads) {
  const uint4 e4 = make_uint4(kEmpty, kEmpty, kEmpty, kEmpty);
  const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
  uint4* l4 = reinterpret_cast<uint4*>(p.lists);
  for (size_t q = gtid; q < p.list_words_cap / 2; q += gthreads) l4[q] = e4;
  for (size_t q = gtid; q < p.key_words_cap; q += gthreads) p.keys[q] = kNoKey;
  for (size_t q = gtid; q < p.row_cnt_cap; q += gthreads) p.row_cnt[q] = 0u;
  uint4* a4 = reinterpret_cast<uint4*>(p.acc);
  for (size_t q = gtid; q < 3 * p.acc_cap; q += gthreads) a4[q] = z4;
}


constexpr int kDsHash = 2 * kThreads;  // count map positions (a tile's warp groups)
constexpr int kDsHot = 256;            // hot table positions (at most half used)
constexpr unsigned int kDsHotGroups = 4;  // warp groups of one voxel in the first tile that make it hot
constexpr int kDsSmem = kDsHash * (4 + 4) + kDsHot * (4 + 16 + 16 + 4 + 4);

// ------------------------------------------------------------ host side: launch entry points of the kernel files

// The block-tile kernel is built twice: with 1024-thread blocks, one an SM
// (pv_ordered.cu), and with 512-thread blocks, two an SM (pv_ordered_half.cu,
// the same source), the second for clouds whose 1024-thread chunks would
// span several tiles.  Each build names its entry points after its block
// size.
//
// Shared-memory opt-in of the block-tile kernel's instantiations; the
// resident blocks per SM of the one that fits fewest (0 on failure).
int prepare_ordered_1024();
int prepare_ordered_512();
// Dynamic shared memory of a launch of the block-tile kernel.
int ordered_smem_1024();
int ordered_smem_512();
// Shared-memory opt-in of the downsampling kernel (built with 1024- and with
// 512-thread blocks, like the block-tile kernel); its resident blocks per SM.
int prepare_downsample_1024();
int prepare_downsample_512();
// Dynamic shared memory of a launch of the downsampling kernel.
int downsample_smem_1024();
int downsample_smem_512();
// One cooperative launch of the block-tile kernel: one frame (frame_offsets
// null; queue picks the instantiation that shares long lists out per
// block) or a batch of `frames` frames (host offsets, frames + 1 of them).
cudaError_t launch_ordered_1024(const cudaLaunchConfig_t& cfg, const KParams& kp, bool queue,
                                const int64_t* frame_offsets, int frames, long long n);
cudaError_t launch_ordered_512(const cudaLaunchConfig_t& cfg, const KParams& kp, bool queue,
                               const int64_t* frame_offsets, int frames, long long n);
cudaError_t launch_unordered(const cudaLaunchConfig_t& cfg, const KParams& kp);
cudaError_t launch_downsample_1024(const cudaLaunchConfig_t& cfg, const KParams& kp);
cudaError_t launch_downsample_512(const cudaLaunchConfig_t& cfg, const KParams& kp);

}  // namespace pvk
