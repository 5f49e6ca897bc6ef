// GB300 (sm_103a) pillar voxelizer: kernels and the C ABI declared in pv.h.
//
// What is computed is the page "Voxelize" (ethan-howes.github.io/projects/
// voxelize/): bin every point into a pillar ("Implementation > Binning a
// point"), group points that share a pillar ("Claiming a pillar and packing
// points"), compact the pillars into dense outputs ("Compaction"), with the
// canonical order stated in pv.h.  How it is computed differs from the
// page's one-thread-per-point kernel + Thrust copy_if + gather:
//
//   * one cooperative launch, one 1024-thread block per SM, all resident,
//     and two grid-wide barriers;
//   * phase 1 (before the first barrier): blocks sweep the cloud in tiles of
//     1024 consecutive points, in index order across the grid.  Each point is
//     read with one 16-byte load and binned with IEEE round-to-nearest
//     subtract/divide and floorf.  In shared memory the tile is grouped by
//     pillar (warp match + a small open-addressing map), which gives every
//     point its rank among the tile's points of its pillar and lays the tile
//     out group by group in a per-tile buffer.  Only each group's first point
//     (its leader) touches the pillar's slot in an L2-resident table.  For
//     8..32 points a pillar the slot is an append list: a count taken with
//     atomicAdd gives the group its position, an atomicMin keeps the lowest
//     leader (the pillar's first point: the page's atomicCAS claim plus an
//     atomicMin of the first index), and the gather sorts the entries; a
//     pillar with more groups than the slot holds spills into an overflow
//     list of the other kind.  Otherwise the slot keeps the max_points
//     smallest leader indices sorted with atomicMin (entry k keeps the
//     minimum of what reaches it and passes the larger value on, so it ends
//     as the (k+1)-th smallest whatever order the inserts came in), entry 0
//     being the first point.  The pillar's points in index order are its
//     groups concatenated in leader order.  The table is
//     direct-mapped (one slot per grid cell) when the grid is small enough,
//     else open addressing with linear probing (the page's hash table, "A
//     hash table instead of a sort"), probes bounded by the table size;
//   * phase 2: each block owns a contiguous range of point indices.  A point
//     is the first of its pillar iff its index is its slot's lowest leader.
//     Blocks compact their first points in index order and publish the
//     count; after the second barrier every block scans all counts into
//     shared memory, so every pillar's rank (its order of first appearance)
//     is known everywhere.  All warps share the output rows: rank r finds
//     its owner block by binary search in the prefix, reads its groups,
//     gathers the first max_points points (16-byte rows) and writes the row
//     stack, coordinates and count; the slots of pillars past the budget are
//     emptied; rows past V are zero-filled.
//
// The table cleans itself: every slot a call fills is emptied by the same
// call, so no memset runs per call.  A launch that fails on the device marks
// the table dirty and the next launch resets it whole first.  Every wait is
// bounded by the global timer (about 1 s), after which the kernel records
// PV_ERR_TIMEOUT and returns.

#include "pv.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>

namespace {

constexpr uint32_t kEmpty = 0xFFFFFFFFu;   // empty 32-bit marker
constexpr unsigned long long kEmpty64 = ~0ull;  // empty list entry (also an all-0xFF memset)
constexpr int32_t kLeaderBit = 1 << 30;    // slot_of_point: the point leads its tile group
constexpr int32_t kNoKey = -1;             // empty hashed slot
#ifndef PV_BLOCK_THREADS
#define PV_BLOCK_THREADS 1024
#endif
constexpr int kThreads = PV_BLOCK_THREADS;  // also the tile: points grouped together in shared memory
constexpr int kWarps = kThreads / 32;
static_assert(kWarps <= 32 && kWarps % 16 == 0, "warp 0 scans one value per warp; 16-byte counter rows");
constexpr int kMinBlocksPerSM = 1024 / kThreads;
constexpr int kMaxCtas = 1024;             // blocks per launch (prefix lives in shared memory)
static_assert(kMaxCtas < 0x10000, "finished blocks are counted in 16 bits");
constexpr int kFlagUnroll = 4;             // block-wide tiles in flight when flagging
constexpr int kFlagUnrollWide = 8;         // the same, in launches whose chunks span up to 8 block tiles
static_assert(kWarps == 32, "the flag prefix gives each lane U consecutive (tile, warp) counts");
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
__device__ unsigned long long g_phase_ns[kStampCtas][kStamps];
__device__ unsigned long long g_p1_ns[kStampCtas][kStamps];
__device__ unsigned long long g_insert_stats[4];  // inserts, atomics, rejected up front, max atomics
__device__ __forceinline__ void pv_wait_reg(unsigned int v) {
  unsigned int d;
  asm volatile("mov.b32 %0, %1;" : "=r"(d) : "r"(v));
}
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
__device__ bool grid_sync(Control* ctl, unsigned int target, int* s_flag) {
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
__device__ unsigned int block_exclusive_scan(unsigned int x, unsigned int* s_tmp, unsigned int* total) {
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
__device__ __forceinline__ void flag_prefix(unsigned int* flat, unsigned int* total, unsigned int lane) {
  unsigned int c[U];
  unsigned int sum = 0;
#pragma unroll
  for (int k = 0; k < U; ++k) {
    c[k] = flat[lane * U + k];
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
  for (int k = 0; k < U; ++k) {
    flat[lane * U + k] = run;
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
__device__ unsigned long long g_probe_hist[34];  // lookups by positions probed: 1 .. 32, more, table full
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

// List entry: (leader index << 32) | (chunk rank << 22) | (d << 11) | size,
// where the group's rows start in tile_rows at leader index + d (d signed,
// 11 bits: a group lies inside its 1024-point tile) and the chunk rank is
// below max_points <= 1024.
__device__ __forceinline__ unsigned long long make_entry(long long leader, unsigned int crank, long long row,
                                                         unsigned int size) {
  const unsigned int d = static_cast<unsigned int>(row - leader) & 2047u;
  return (static_cast<unsigned long long>(leader) << 32) | (crank << 22) | (d << 11) | size;
}
__device__ __forceinline__ long long entry_row(unsigned long long ent) {
  const int d = static_cast<int>(static_cast<unsigned int>(ent) << 10) >> 21;  // bits 11..21, sign-extended
  return static_cast<long long>(ent >> 32) + d;
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
      before += static_cast<unsigned int>(y) & 2047u;
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
__device__ void append_insert(const KParams& p, const ListRef& L, unsigned long long x, uint32_t cbase,
                              uint32_t cspan) {
  const int S = kHead + p.KT;
  unsigned int* w0 = reinterpret_cast<unsigned int*>(L.head);
  const unsigned int j = ~atomicAdd(w0, 0xFFFFFFFFu);  // the count is kept complemented
  atomicMin(w0 + 1, static_cast<unsigned int>(x >> 32));
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

// Shared-memory grouping of one block tile (kThreads consecutive points):
// an open-addressing map slot -> map position, per (position, warp) the
// number of the warp's points in that slot, and per position the group's
// offset in the tile's grouped layout.  A point's rank among the tile's
// points of its pillar is the sum over earlier warps plus its rank in its
// own warp (lanes hold consecutive indices).
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
// After phase 1 the same shared memory holds the gather's per-warp merge
// buffers (32 entries each) and the block's queue of long lists.
constexpr unsigned int kQueueCap = kDynSmem / 8 - kWarps * 32;
constexpr unsigned int kQueueDrop = 0xFFFFFFFFu;  // queue row of a list past the budget (emptied only)
constexpr int64_t kQueueMinRowsPerWarp = 8;        // rows per warp from which the gather queues long lists

struct TileMap {
  unsigned int* cnt;         // [kTileHash][kWarps / 4] packed byte counters
  int* key;                  // [kTileHash], -1 = free
  unsigned int* off;         // [kTileHash] (rows to write << 16) | group offset in the tile layout
  unsigned int* layout;      // rows handed out in the tile layout
};

__device__ __forceinline__ TileMap tile_map(unsigned char* base, unsigned int* layout) {
  TileMap m;
  m.cnt = reinterpret_cast<unsigned int*>(base);
  m.key = reinterpret_cast<int*>(base + kTileHash * kWarps);
  m.off = reinterpret_cast<unsigned int*>(base + kTileHash * kWarps + kTileHash * 4);
  m.layout = layout;
  return m;
}

// Empty the map positions h = tid, tid + kThreads, ... (keys and counters).
__device__ __forceinline__ void tile_clear(const TileMap& m, unsigned int tid) {
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
__device__ __forceinline__ int tile_claim(const TileMap& m, int slot) {
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

__device__ __forceinline__ unsigned int chunk_rank(int* ckey, unsigned int* ccnt, int slot, unsigned int size) {
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
// Each word holds four warps' counts (at most 32 each), summed with dp4a
// against ones; the words before this warp's count whole, its own word only
// in the bytes of lower warps.
__device__ __forceinline__ void tile_counts(const TileMap& m, int h, unsigned int warp, unsigned int* before,
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
        cum += static_cast<unsigned int>(h.e[j]) & 2047u;
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
      cum += static_cast<unsigned int>(h.e[j]) & 2047u;
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
    run += static_cast<unsigned int>(ej) & 2047u;
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
__device__ unsigned int emit_groups(const KParams& p, const ListRef& L, float4* orow, int K, unsigned int lane,
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
    const unsigned int size = ent != kEmpty64 ? (static_cast<unsigned int>(ent) & 2047u) : 0u;
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
      const unsigned int info = static_cast<unsigned int>(ge);
      const unsigned int room = static_cast<unsigned int>(K) - written;
      const unsigned int n = (info & 2047u) < room ? (info & 2047u) : room;
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
__device__ void app_clear_with(const KParams& p, const ListRef& L, unsigned int lane, unsigned long long ow) {
  const int S = kHead + p.KT;
  if (ow < p.pool_n) {
    unsigned long long* base = p.pool + ow * static_cast<unsigned long long>(S);
    for (int w = static_cast<int>(lane); w < S; w += 32) base[w] = kEmpty64;
  }
  __syncwarp();
  for (int w = static_cast<int>(lane); w < S; w += 32) *slot_word(L.head, L.tail, w) = kEmpty64;
}

__device__ void app_clear(const KParams& p, const ListRef& L, unsigned int lane) {
  app_clear_with(p, L, lane, __ldcg(slot_word(L.head, L.tail, kHead + p.KT - 1)));
}

// Writes the output row of an append-list pillar that is not served from
// its head: lane l reads stored entry l, the warp sorts them by leader
// (bitonic), merges in the slot's sorted overflow list if it has one (the
// first 32 of the union, through a per-warp shared buffer), and copies the
// first max_points points as emit_groups does; empties the slot.  All 32
// lanes call it with the same arguments (max_points <= 32).
__device__ unsigned int emit_app(const KParams& p, const ListRef& L, float4* orow, int K, unsigned int lane,
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
  const unsigned int size = ent != kEmpty64 ? (static_cast<unsigned int>(ent) & 2047u) : 0u;
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
__device__ bool emit_app_quad(const KParams& p, unsigned long long qe, bool mine, unsigned int lane, int K,
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
  const unsigned int sz = ent != kEmpty64 ? (static_cast<unsigned int>(ent) & 2047u) : 0u;
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
__device__ void reset_tables(const KParams& p, size_t gtid, size_t gthreads) {
  const uint4 e4 = make_uint4(kEmpty, kEmpty, kEmpty, kEmpty);
  const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
  uint4* l4 = reinterpret_cast<uint4*>(p.lists);
  for (size_t q = gtid; q < p.list_words_cap / 2; q += gthreads) l4[q] = e4;
  for (size_t q = gtid; q < p.key_words_cap; q += gthreads) p.keys[q] = kNoKey;
  for (size_t q = gtid; q < p.row_cnt_cap; q += gthreads) p.row_cnt[q] = 0u;
  uint4* a4 = reinterpret_cast<uint4*>(p.acc);
  for (size_t q = gtid; q < 3 * p.acc_cap; q += gthreads) a4[q] = z4;
}

// ------------------------------------------------------------ the kernel

// NF = 1: one cloud (pv_voxelize); NF = kMaxFrames: a batch of up to NF
// frames (pv_voxelize_batch), where a voxel's id carries its frame, each
// frame keeps its own first max_voxels voxels and writes its own rows.
template <int NF, bool kQueue>
__global__ void __launch_bounds__(kThreads, kMinBlocksPerSM) pv_voxelize_kernel(const KParams p, const Frames<NF> fr) {
  constexpr bool kBatched = NF > 1;
  // Block tiles in flight in the first-point pass: 8 where chunks are long
  // (the launches that queue long lists), else 4 (fewer empty tiles to scan).
  constexpr int FU = kQueue ? kFlagUnrollWide : kFlagUnroll;
  extern __shared__ __align__(16) unsigned char s_dyn[];
  __shared__ unsigned int s_prefix[kMaxCtas + 1];
  __shared__ long long s_off[NF + 1];
  __shared__ unsigned int s_fpre[NF + 1];  // batched: first points before each frame start (global)
  __shared__ unsigned int s_vcum[NF + 1];  // batched: rows emitted by earlier frames
  __shared__ unsigned int s_dcum[NF + 1];  // batched: voxels past the budget in earlier frames
  __shared__ unsigned int s_tile[FU][kWarps];
  __shared__ unsigned int s_tmp[kWarps + 1];
  __shared__ int s_flag;
  __shared__ unsigned int s_dirty;
  __shared__ unsigned int s_layout[2];
  __shared__ unsigned int s_nrec;
  __shared__ unsigned int s_qn, s_qh;  // gather: long lists queued by the block, and taken

  const unsigned int P = gridDim.x;
  const unsigned int cta = blockIdx.x;
  const unsigned int tid = threadIdx.x;
  const unsigned int lane = tid & 31u;
  const unsigned int warp = tid >> 5;
  const size_t gtid = static_cast<size_t>(cta) * kThreads + tid;
  const size_t gthreads = static_cast<size_t>(P) * kThreads;
  const long long gwarp = static_cast<long long>(cta) * kWarps + warp;
  const long long nwarps = static_cast<long long>(P) * kWarps;
  const int K = p.K;
  const long long begin = lmin(p.n, static_cast<long long>(cta) * p.chunk);
  const long long end = lmin(p.n, begin + p.chunk);

  // The first tile's points are loaded and the shared maps emptied while the
  // control block's words are in flight.
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  long long tb = begin;  // this block's contiguous chunk, in tiles from its start
  float4 q = (tb + tid < end) ? __ldg(p.points + tb + tid) : z4;
  // Thread 0 alone reads the control block (the same word read by every
  // thread would queue thousands of requests on one L2 line); the dirty flag
  // reaches the block through shared memory, the epoch only thread 0 needs.
  unsigned int epoch = 0, dirty_word = 0;
  if (tid == 0) {
    epoch = ld_relaxed(&p.ctl->epoch);
    dirty_word = ld_relaxed(&p.ctl->dirty);
  }
  unsigned int bar_target = P;
  bool alive = true;
  const int B = kBatched ? p.frames : 1;
  if (kBatched)
    for (int b = static_cast<int>(tid); b <= B; b += kThreads) s_off[b] = fr.off[b];  // read after a block barrier
  PV_STAMP(0);
  const bool multi = end - begin > kThreads;  // more than one tile: second map and chunk map in use
  int* ckey = reinterpret_cast<int*>(s_dyn + 2 * kMapBytes);
  unsigned int* ccnt = reinterpret_cast<unsigned int*>(ckey + kChunkHash);
  {  // tile map 0 empty (counters zero, keys -1); map 1 and the chunk map only if used
    uint4* d4 = reinterpret_cast<uint4*>(s_dyn);
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const uint4 m1 = make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
    const int maps = multi ? 2 : 1;
    for (int m = 0; m < maps; ++m) {
      uint4* base = d4 + m * (kMapBytes / 16);
      for (int j = static_cast<int>(tid); j < kTileHash * kWarps / 16; j += kThreads) base[j] = z;
      for (int j = static_cast<int>(tid); j < kTileHash * 4 / 16; j += kThreads)
        base[kTileHash * kWarps / 16 + j] = m1;
    }
    if (multi) {
      uint4* c4 = reinterpret_cast<uint4*>(ckey);
      for (int j = static_cast<int>(tid); j < kChunkHash / 4; j += kThreads) {
        c4[j] = m1;
        c4[kChunkHash / 4 + j] = z;
      }
    }
  }
  if (tid == 0) {
    s_layout[0] = s_layout[1] = 0;
    s_nrec = 0;
    s_qn = s_qh = 0;
    s_dirty = dirty_word;
  }
  __syncthreads();  // maps empty, dirty flag shared
  const bool dirty = s_dirty != 0u;

  // Recovery after a failed launch: empty the whole table first.
  if (dirty) {
    reset_tables(p, gtid, gthreads);
    alive = grid_sync(p.ctl, bar_target, &s_flag);
    bar_target += P;
  }

  // ---- phase 1a: bin every point; lay each block tile out grouped by pillar
  // (groups in any order inside the tile, points of a group in index order)
  // and record one entry per (pillar, tile) group, with the group's rank among
  // this chunk's groups of the pillar.  Two barriers per tile: after the warp
  // groups register in the tile map, and after the group offsets are handed
  // out.  No global atomics in this loop.
  // ---- phase 1b: insert the recorded groups into the pillars' lists, all at
  // once (their chunk ranks keep them apart).
  if (alive) {
#ifdef PV_INSTRUMENT
    if (tid == 0 && cta < kStampCtas) g_p1_ns[cta][6] = global_timer_ns();
#endif
    int buf = 0;
    int own_rs = -1;                  // one-tile chunk: the record this thread leads, if any
    unsigned long long own_entry = 0;
    for (; tb < end; tb += kThreads, buf ^= 1) {
#ifdef PV_INSTRUMENT
      const bool first_tile = tb == begin;
#endif
      PV_SUB(0);
      const TileMap tm = tile_map(s_dyn + buf * kMapBytes, &s_layout[buf]);
      const TileMap prev = tile_map(s_dyn + (buf ^ 1) * kMapBytes, &s_layout[buf ^ 1]);
      const long long i = tb + tid;
      const long long inext = i + kThreads;
      const float4 qn = inext < end ? __ldg(p.points + inext) : z4;  // next tile, in flight early
      int slot = -1;
      if (i < end) {
        int key;
        if (bin_point(q, p, &key)) {
          if (kBatched) key += frame_of(s_off, B, i) * p.cells;
          slot = p.hash_mode ? claim_slot(p.keys, p.table_mask, key) : key;
          if (slot < 0) atomicMin(&p.ctl->err, PV_ERR_CAPACITY);
        }
      }
      PV_SUB(1);
      const unsigned int peers = __match_any_sync(0xffffffffu, slot);
      const int leader = __ffs(peers) - 1;
      int h = -1;
      if (slot >= 0 && static_cast<int>(lane) == leader) {
        h = tile_claim(tm, slot);
        if (h >= 0) {
          reinterpret_cast<unsigned char*>(tm.cnt + h * (kWarps / 4))[warp] =
              static_cast<unsigned char>(__popc(peers));
        } else {  // cannot happen: at most kThreads keys in 2 * kThreads positions
          atomicMin(&p.ctl->err, PV_ERR_INTERNAL);
        }
      }
      h = __shfl_sync(0xffffffffu, h, leader);
      if (h < 0) slot = -1;
      __syncthreads();  // (A) every warp group registered; the previous tile's map is read
      PV_SUB(2);
      // Empty the previous tile's map (used again by the next tile, after barrier B).
      if (multi) {
        if (tid == 0) *prev.layout = 0;
        tile_clear(prev, tid);
      }
      // The group's counts before this warp and in all: read by the leader,
      // shared with the group (one warp) by shuffles.
      unsigned int trank = 0, tot = 0;
      if (slot >= 0 && static_cast<int>(lane) == leader) tile_counts(tm, h, warp, &trank, &tot);
      trank = __shfl_sync(0xffffffffu, trank, leader);
      tot = __shfl_sync(0xffffffffu, tot, leader);
      if (slot >= 0) trank += __popc(peers & lanemask_lt());
      const bool lead = slot >= 0 && trank == 0;
      const unsigned int cseen = (lead && multi) ? chunk_rank(ckey, ccnt, slot, tot) : 0u;
      const int crank = static_cast<int>(cseen >> 16);
      {  // group offsets and record slots: one shared-memory atomic per warp each
        const unsigned int need = lead ? tot : 0u;
        // A group with max_points of its pillar's points before it in this
        // chunk (or max_points groups) can never be kept: not recorded.
        const unsigned int wants =
            (lead && crank < K && (cseen & 0xFFFFu) < static_cast<unsigned int>(K)) ? 1u : 0u;
        // One scan for both: a warp's groups hold at most kThreads points
        // (low half) and it has at most 32 records (high half).
        unsigned int pk = need | (wants << 16);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned int y = __shfl_up_sync(0xffffffffu, pk, o);
          if (lane >= static_cast<unsigned int>(o)) pk += y;
        }
        const unsigned int psum = __shfl_sync(0xffffffffu, pk, 31);
        const unsigned int incl = pk & 0xFFFFu, rincl = pk >> 16;
        const unsigned int wsum = psum & 0xFFFFu, rsum = psum >> 16;
        unsigned int base = 0, rbase = 0;
        if (lane == 31) {
          if (wsum) base = atomicAdd(tm.layout, wsum);
          if (rsum) rbase = atomicAdd(&s_nrec, rsum);
        }
        base = __shfl_sync(0xffffffffu, base, 31);
        rbase = __shfl_sync(0xffffffffu, rbase, 31);
        if (lead) {
          const unsigned int off = base + incl - need;
          // Rows of the group that can ever be emitted: those with fewer than
          // max_points of the pillar's points before them in the chunk.
          const unsigned int cpts = cseen & 0xFFFFu;
          const unsigned int room = cpts < static_cast<unsigned int>(K) ? static_cast<unsigned int>(K) - cpts : 0u;
          tm.off[h] = ((tot < room ? tot : room) << 16) | off;
          if (wants) {
            const unsigned long long ent = make_entry(i, static_cast<unsigned int>(crank), tb + off, tot);
            if (multi) {
              const long long rj = begin + rbase + rincl - wants;
              p.firsts[rj] = slot;  // the record's slot (firsts is rewritten after the barrier)
              p.recs[rj] = ent;
            } else {  // one tile: the leader inserts its own record
              own_rs = slot;
              own_entry = ent;
            }
          }
        }
      }
      if (i < end) p.slot_of_point[i] = slot < 0 ? -1 : (lead ? (slot | kLeaderBit) : slot);
      __syncthreads();  // (B) group offsets handed out; the previous map is empty
      PV_SUB(3);
      if (slot >= 0) {
        const unsigned int ow = tm.off[h];
        if (trank < (ow >> 16)) p.tile_rows[tb + (ow & 0xFFFFu) + trank] = q;
      }
      PV_SUB(4);
      q = qn;
    }
    __syncthreads();  // every record written
#ifdef PV_INSTRUMENT
    if (tid == 0 && cta < kStampCtas) g_p1_ns[cta][5] = global_timer_ns();
#endif
    const unsigned int nrec = s_nrec;
    // One record per thread at a time; the thread's next record is read
    // while the current one's cascade runs.  A one-tile chunk's leaders
    // insert their own records, held in registers.
    if (!multi) {
      if (own_rs >= 0) {
        if (p.append) {
          append_insert(p, list_of(p, own_rs), own_entry, static_cast<uint32_t>(begin),
                        static_cast<uint32_t>(end - begin));
        } else {
          uint4 h[kHead / 2];
#pragma unroll
          for (int t = 0; t < kHead / 2; ++t)
            h[t] = __ldcg(reinterpret_cast<const uint4*>(p.lists + static_cast<size_t>(own_rs) * kHead) + t);
          list_insert(list_of(p, own_rs), h, K, p.KT, own_entry, 0, static_cast<uint32_t>(begin),
                      static_cast<uint32_t>(end - begin));
        }
      }
    } else {
      unsigned int j0 = tid;
      int rs = j0 < nrec ? __ldcg(p.firsts + begin + j0) : -1;
      unsigned long long entry = j0 < nrec ? __ldcg(p.recs + begin + j0) : 0ull;
      for (; j0 < nrec; j0 += kThreads) {
        const unsigned int j1 = j0 + kThreads;
        const int rs1 = j1 < nrec ? __ldcg(p.firsts + begin + j1) : -1;
        const unsigned long long entry1 = j1 < nrec ? __ldcg(p.recs + begin + j1) : 0ull;
        if (p.append) {
          append_insert(p, list_of(p, rs), entry, static_cast<uint32_t>(begin), static_cast<uint32_t>(end - begin));
        } else {
          uint4 h[kHead / 2];
#pragma unroll
          for (int t = 0; t < kHead / 2; ++t)
            h[t] = __ldcg(reinterpret_cast<const uint4*>(p.lists + static_cast<size_t>(rs) * kHead) + t);
          list_insert(list_of(p, rs), h, K, p.KT, entry, entry_crank(entry),
                      static_cast<uint32_t>(begin), static_cast<uint32_t>(end - begin));
        }
        rs = rs1;
        entry = entry1;
      }
    }
    PV_STAMP(1);
    alive = grid_sync(p.ctl, bar_target + p.bar_extra, &s_flag);
  }
  PV_STAMP(2);

  const unsigned int M = static_cast<unsigned int>(p.max_voxels);
  unsigned int V = 0;

  if (alive) {
    // ---- phase 2a: first points of this block's range, compacted in index order.
    unsigned int local = 0;
    for (long long base = begin; base < end; base += static_cast<long long>(FU) * kThreads) {
      int s[FU];
      uint32_t head[FU];
#pragma unroll
      for (int u = 0; u < FU; ++u) {
        const long long i = base + u * kThreads + tid;
        s[u] = i < end ? __ldcg(p.slot_of_point + i) : -1;
      }
#pragma unroll
      for (int u = 0; u < FU; ++u) {
        // Only a tile-group leader can be its pillar's first point.
        head[u] = (s[u] >= 0 && (s[u] & kLeaderBit))
                      ? static_cast<uint32_t>(__ldcg(p.lists + static_cast<size_t>(s[u] & ~kLeaderBit) * kHead) >> 32)
                      : kEmpty;
        s[u] = s[u] >= 0 ? (s[u] & ~kLeaderBit) : -1;
      }
      unsigned int ball[FU];
#pragma unroll
      for (int u = 0; u < FU; ++u) {
        const long long i = base + u * kThreads + tid;
        ball[u] = __ballot_sync(0xffffffffu, s[u] >= 0 && head[u] == static_cast<uint32_t>(i));
        if (lane == 0) s_tile[u][warp] = __popc(ball[u]);
      }
      __syncthreads();
      if (warp == 0) flag_prefix<FU>(&s_tile[0][0], &s_tmp[kWarps], lane);
      __syncthreads();
      unsigned int run = local;
#pragma unroll
      for (int u = 0; u < FU; ++u) {
        const unsigned int before = run + s_tile[u][warp] + __popc(ball[u] & lanemask_lt());
        if ((ball[u] >> lane) & 1u) p.firsts[begin + before] = s[u];
        if (kBatched) {  // a frame start at i records this block's first points before it
          const long long i = base + u * kThreads + tid;
          if (i < end)
            for (int b = frame_of(s_off, B, i); b >= 1 && s_off[b] == i; --b) p.frame_cnt[b] = before;
        }
      }
      run += s_tmp[kWarps];
      local = run;
      __syncthreads();
    }
    PV_STAMP(3);

    // ---- phase 2b: publish the count; after a second barrier every block
    // scans all counts itself (one count per thread) into shared memory.
    if (tid == 0) p.counts[cta] = local;
    alive = grid_sync(p.ctl, bar_target + P, &s_flag);
  }

  unsigned int total = 0;
  int seen_err = 0;   // thread 0: the error word once the second barrier is passed
  bool bad = false;   // a ranked pillar without its first group (never in a clean table)
  if (alive) {
    if (tid == 0) seen_err = static_cast<int>(ld_relaxed(reinterpret_cast<const unsigned int*>(&p.ctl->err)));
    const unsigned int c = tid < P ? __ldcg(p.counts + tid) : 0u;
    const unsigned int excl = block_exclusive_scan(c, s_tmp, &total);
    if (tid < P) s_prefix[tid] = excl;
    if (tid == 0) s_prefix[P] = total;
    __syncthreads();
    if (kBatched) {
      // Per frame: voxels (first points between its start and the next), rows
      // kept (at most max_voxels) and voxels past its budget, as exclusive sums.
      for (int b = static_cast<int>(tid); b <= B; b += kThreads) {
        const long long o = s_off[b];
        unsigned int pre = 0;
        if (b > 0) pre = o >= p.n ? total : s_prefix[o / p.chunk] + __ldcg(p.frame_cnt + b);
        s_fpre[b] = pre;
      }
      __syncthreads();
      const unsigned int cnt_b = static_cast<int>(tid) < B ? s_fpre[tid + 1] - s_fpre[tid] : 0u;
      const unsigned int keep = cnt_b < M ? cnt_b : M;
      unsigned int vt = 0, dt = 0;
      const unsigned int ve = block_exclusive_scan(keep, s_tmp, &vt);
      const unsigned int de = block_exclusive_scan(cnt_b - keep, s_tmp, &dt);
      if (static_cast<int>(tid) < B) {
        s_vcum[tid] = ve;
        s_dcum[tid] = de;
      }
      if (tid == 0) {
        s_vcum[B] = vt;
        s_dcum[B] = dt;
      }
      __syncthreads();
      V = vt;  // rows written over all frames
    } else {
      V = total < M ? total : M;
    }
    PV_STAMP(4);

    // ---- phase 2e, issued first: zero rows V .. max_voxels-1 (of every
    // frame; all blocks share it).  These stores depend on nothing else, so
    // they overlap the gather's load latencies instead of trailing it.
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    const size_t Kz = static_cast<size_t>(K);
    constexpr size_t cw = kBatched ? 4 : 3;
    for (int b = 0; b < B; ++b) {
      const unsigned int Vb = kBatched ? s_vcum[b + 1] - s_vcum[b] : V;
      const size_t lo = static_cast<size_t>(b) * M + Vb, hi = static_cast<size_t>(b + 1) * M;
      for (size_t q = lo * Kz + gtid; q < hi * Kz; q += gthreads) p.out_voxels[q] = z4;
      for (size_t q = cw * lo + gtid; q < cw * hi; q += gthreads) p.out_coords[q] = 0;
      for (size_t q = lo + gtid; q < hi; q += gthreads) p.out_counts[q] = 0;
    }

    PV_STAMP(5);

    // ---- phase 2c+2d: every ranked pillar, kept or past the budget.  Every
    // warp of the grid takes an equal contiguous share of the kept rows (so
    // its output rows are contiguous) and an equal contiguous share of the
    // pillars past the budget (which only have their lists emptied), and
    // works through both together, 32 at a time.  Lane l finds the slot of
    // its pillar and reads list positions 0..3 (one round trip each for 32
    // pillars).  Past the budget (its frame's, in a batch): a list known to
    // end inside positions 0..3 loses those, any other list every position.
    // Kept: a pillar whose points all come from those groups (its list ends
    // inside them, or they already hold max_points points) is copied by the
    // warp kEmitPer pillars at a time; the others are emitted one by one
    // from their whole list.
    bool stale = false;
    unsigned long long* wbuf = reinterpret_cast<unsigned long long*>(s_dyn) + warp * 32;  // append lists' merge buffer
    unsigned long long* s_queue = reinterpret_cast<unsigned long long*>(s_dyn) + kWarps * 32;  // (row << 32) | slot
    // (Counts of pillars and warps fit 32 bits: N < 2^29, at most 1024 x 32 warps.)
    const unsigned int dropped = kBatched ? s_dcum[B] : total - V;
    const unsigned int nw = static_cast<unsigned int>(nwarps), gw = static_cast<unsigned int>(gwarp);
    const unsigned int pk = (V + nw - 1) / nw;
    const unsigned int kw0 = gw * pk < V ? gw * pk : V;
    const unsigned int nk = (kw0 + pk < V ? kw0 + pk : V) - kw0;
    const unsigned int pd = (dropped + nw - 1) / nw;
    const unsigned int dw0 = gw * pd < dropped ? gw * pd : dropped;
    const unsigned int nd = (dw0 + pd < dropped ? dw0 + pd : dropped) - dw0;
    for (unsigned int t0 = 0; t0 < nk + nd; t0 += 32) {
      const unsigned int t = t0 + lane;
      const bool valid = t < nk;                  // kept: an output row
      const bool drop = !valid && t < nk + nd;    // past the budget
      const bool in_range = valid || drop;
      long long row = 0;
      unsigned int rank = 0;
      int fb = 0;
      if (valid) {
        const unsigned int k = kw0 + t;  // the k-th row written (frames one after the other)
        rank = k;
        row = k;
        if (kBatched) {
          fb = slot_in_cum(s_vcum, B, k);
          const unsigned int loc = k - s_vcum[fb];
          rank = s_fpre[fb] + loc;
          row = static_cast<long long>(fb) * M + loc;
        }
      } else if (drop) {
        const unsigned int j = dw0 + (t - nk);  // the j-th pillar past a budget
        rank = M + j;
        if (kBatched) {
          const int b = slot_in_cum(s_dcum, B, j);
          rank = s_fpre[b] + M + (j - s_dcum[b]);
        }
      }
      int slot = 0;
      if (in_range) slot = slot_of_rank(p, s_prefix, P, rank);
      unsigned long long* L = p.lists + static_cast<size_t>(slot) * kHead;  // head row
      Head hd = read_head(p, L, in_range);
      // Long lists (kept ones not served by their first groups, and those
      // past the budget that need more than their head emptied) go to the
      // block's queue and are shared out over its warps after this pass,
      // since a warp's contiguous share of ranks can hold many of them; a
      // full queue leaves them to this warp.
      const bool short_drop = drop && hd.few && !hd.filled;
      const bool longv = (valid && !hd.few) || (drop && !short_drop);
      bool inl = longv;  // long, processed here: always without the queue, else when it is full
      if constexpr (kQueue) {
        const unsigned int lm = __ballot_sync(0xffffffffu, longv);
        unsigned int qb = 0;
        if (lane == 0 && lm) qb = atomicAdd(&s_qn, static_cast<unsigned int>(__popc(lm)));
        qb = __shfl_sync(0xffffffffu, qb, 0) + __popc(lm & lanemask_lt());
        if (longv && qb < kQueueCap) {
          const unsigned int qrow = valid ? static_cast<unsigned int>(row) : kQueueDrop;
          s_queue[qb] = (static_cast<unsigned long long>(qrow) << 32) | static_cast<unsigned int>(slot);
          inl = false;
        }
      }
      {  // past the budget: empty the list
        if (short_drop) {
          const uint4 e4 = make_uint4(kEmpty, kEmpty, kEmpty, kEmpty);
          reinterpret_cast<uint4*>(L)[0] = e4;
          reinterpret_cast<uint4*>(L)[1] = e4;
        }
        if (drop && p.hash_mode) p.keys[slot] = kNoKey;
        for (unsigned int m = __ballot_sync(0xffffffffu, drop && inl); m != 0u; m &= m - 1u) {
          const ListRef Lu = list_of(p, __shfl_sync(0xffffffffu, slot, __ffs(m) - 1));
          if (p.append)
            app_clear(p, Lu, lane);
          else
            for (int e = static_cast<int>(lane); e < K; e += 32) *Lu.at(e) = kEmpty64;
        }
      }

      int key = slot;
      if (valid && p.hash_mode) key = __ldcg(p.keys + slot);
      const bool few = valid && hd.few;
      const unsigned int cnt0 = few ? hd.n : 0u;
      unsigned int cnt = cnt0;
      const unsigned int fmask = __ballot_sync(0xffffffffu, few);
      // Pillars served by their first groups, kEmitPer at a time: kEmitLanes
      // lanes per pillar, each copying positions sub, sub + kEmitLanes, ...
      // from the descriptor its pillar's lane computed.
      {
        const CopyDesc cd = copy_desc(hd);
        const unsigned int sub = lane % kEmitLanes;
        const unsigned int pu = lane / kEmitLanes;
        for (int u0 = 0; u0 < 32; u0 += kEmitPer) {
          if (((fmask >> u0) & ((1u << kEmitPer) - 1u)) == 0u) continue;
          const int u = u0 + static_cast<int>(pu);
          const unsigned int w0 = __shfl_sync(0xffffffffu, cd.w0, u);
          const unsigned int w1 = __shfl_sync(0xffffffffu, cd.w1, u);
          int o[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) o[j] = __shfl_sync(0xffffffffu, cd.o[j], u);
          const long long row_u = __shfl_sync(0xffffffffu, row, u);
          const unsigned int n = w0 & 0xFFFFu, s1 = w0 >> 16, s2 = w1 & 0xFFFFu, s3 = w1 >> 16;
          float4* orow = p.out_voxels + static_cast<size_t>(row_u) * K;
          const unsigned int kend = ((fmask >> u) & 1u) ? static_cast<unsigned int>(K) : 0u;  // lanes of a pillar not served here copy nothing
          for (unsigned int e0 = sub; e0 < kend; e0 += 4 * kEmitLanes) {
            float4 v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const unsigned int e = e0 + k * kEmitLanes;
              const int oe = e >= s3 ? o[3] : e >= s2 ? o[2] : e >= s1 ? o[1] : o[0];
              v[k] = e < n ? __ldcg(p.tile_rows + (static_cast<long long>(oe) + e)) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const unsigned int e = e0 + k * kEmitLanes;
              if (e < static_cast<unsigned int>(K)) orow[e] = v[k];
            }
          }
        }
      }
      // A list whose first groups fill the pillar may hold unused entries
      // anywhere after them: empty every position.
      for (unsigned int m = __ballot_sync(0xffffffffu, few && hd.filled); m != 0u; m &= m - 1u) {
        const ListRef Lu = list_of(p, __shfl_sync(0xffffffffu, slot, __ffs(m) - 1));
        for (int e = static_cast<int>(lane); e < K; e += 32) *Lu.at(e) = kEmpty64;
      }
      // Long lists the queue had no room for, one pillar at a time from its whole list.
      for (unsigned int m = __ballot_sync(0xffffffffu, valid && inl); m != 0u; m &= m - 1u) {
        const int u = __ffs(m) - 1;
        const ListRef Lu = list_of(p, __shfl_sync(0xffffffffu, slot, u));
        const long long row_u = __shfl_sync(0xffffffffu, row, u);
        float4* orow_u = p.out_voxels + static_cast<size_t>(row_u) * K;
        const unsigned int w = p.append ? emit_app(p, Lu, orow_u, K, lane, wbuf, &stale)
                                        : emit_groups(p, Lu, orow_u, K, lane, &stale);
        if (static_cast<int>(lane) == u) cnt = w;
      }
      if (valid) {
        if (hd.ng == 0) stale = true;  // a ranked pillar always has its first group
        if (few && !hd.filled) {  // the list held only these entries
          const uint4 e4 = make_uint4(kEmpty, kEmpty, kEmpty, kEmpty);
          reinterpret_cast<uint4*>(L)[0] = e4;
          reinterpret_cast<uint4*>(L)[1] = e4;
        }
        const unsigned int ukey = static_cast<unsigned int>(key);
        const int id = kBatched ? static_cast<int>(ukey - fast_div(ukey, p.div_cells) * static_cast<unsigned int>(p.cells))
                                : key;  // the frame is the row's, not the id's
        const int kxy = static_cast<int>(fast_div(static_cast<unsigned int>(id), p.div_x));
        const int kz = static_cast<int>(fast_div(static_cast<unsigned int>(kxy), p.div_y));
        constexpr int cw = kBatched ? 4 : 3;  // (batch,) z, y, x
        int32_t* co = p.out_coords + cw * static_cast<size_t>(row);
        if (kBatched) co[0] = fb;
        co[cw - 3] = kz;  // 0 on a pillar grid
        co[cw - 2] = kxy - kz * p.g_y;
        co[cw - 1] = id - kxy * p.g_x;
        if (few || inl) p.out_counts[static_cast<size_t>(row)] = static_cast<int32_t>(cnt);
        if (p.hash_mode) p.keys[slot] = kNoKey;
      }
    }
    // The block's queued long lists, taken one at a time by whichever warp is free.
    if constexpr (kQueue) {
      __syncthreads();
      const unsigned int qn = s_qn < kQueueCap ? s_qn : kQueueCap;
      // Four queued lists at a time: append lists of up to seven entries are
      // served eight lanes a pillar; the rest one at a time by the whole warp.
      for (;;) {
        unsigned int j = 0;
        if (lane == 0) j = atomicAdd(&s_qh, 4u);
        j = __shfl_sync(0xffffffffu, j, 0);
        if (j >= qn) break;
        const bool mine = j + (lane >> 3) < qn;
        const unsigned long long qe4 = mine ? s_queue[j + (lane >> 3)] : 0ull;
        const bool slow = p.append ? emit_app_quad(p, qe4, mine, lane, K, &stale) : mine;
        for (unsigned int m = __ballot_sync(0xffffffffu, slow && (lane & 7u) == 0u); m != 0u; m &= m - 1u) {
          const int u = __ffs(m) - 1;
          const unsigned long long qe = (static_cast<unsigned long long>(__shfl_sync(0xffffffffu, static_cast<unsigned int>(qe4 >> 32), u)) << 32) |
                                        __shfl_sync(0xffffffffu, static_cast<unsigned int>(qe4), u);
          const ListRef Lq = list_of(p, static_cast<int>(static_cast<unsigned int>(qe)));
          const unsigned int qrow = static_cast<unsigned int>(qe >> 32);
          if (qrow == kQueueDrop) {
            if (p.append)
              app_clear(p, Lq, lane);
            else
              for (int e = static_cast<int>(lane); e < K; e += 32) *Lq.at(e) = kEmpty64;
          } else {
            float4* orow_q = p.out_voxels + static_cast<size_t>(qrow) * K;
            const unsigned int w = p.append ? emit_app(p, Lq, orow_q, K, lane, wbuf, &stale)
                                            : emit_groups(p, Lq, orow_q, K, lane, &stale);
            if (lane == 0) p.out_counts[qrow] = static_cast<int32_t>(w);
          }
        }
      }
    }
    if (stale) atomicMin(&p.ctl->err, PV_ERR_INTERNAL);
    bad = stale;
    PV_STAMP(6);

  }

  // ---- the last block to finish publishes the status and rearms the control block.
  PV_STAMP(7);
  // A block counts itself finished, in the low half of the word, and, in the
  // high half, whether it knows of an error: one recorded before the second
  // barrier (read after it), a failed wait of its own, or one of its
  // gathers finding a list inconsistent.  Only then does the last block read
  // the error word; the acquire-release count makes every block's writes
  // (their errors included) visible to it.
  const int any_bad = __syncthreads_or(bad || !alive);
  if (tid == 0) {
    const unsigned int mine = (any_bad || seen_err != 0) ? 0x10001u : 1u;
    const unsigned int prev = atom_add_acq_rel(&p.ctl->done, mine);
    if ((prev & 0xFFFFu) == P - 1) {
      const int err = ((prev + mine) >> 16) != 0 ? *reinterpret_cast<volatile int*>(&p.ctl->err) : 0;
      if (kBatched) {
        for (int b = 0; b < B; ++b)
          p.out_num[b] = err != 0 ? err : static_cast<int32_t>(s_vcum[b + 1] - s_vcum[b]);
      } else {
        *p.out_num = err != 0 ? err : static_cast<int32_t>(V);
      }
      p.ctl->dirty = err != 0 ? 1u : 0u;
      p.ctl->err = 0;
      p.ctl->bar = 0;
      p.ctl->done = 0;
      p.ctl->pool = 0;
      const unsigned int next = epoch + 1;
      p.ctl->epoch = next == 0 ? 1u : next;
    }
  }
}

// ------------------------------------------------------------ unordered mode

// The page's own contract, without the canonical order ("The hash slot is
// the output index", "Claiming a pillar and packing points", "Compaction"):
// a pillar's row is handed out when the pillar is created, its points take
// positions in the order their counter increments arrive ("Claiming a
// pillar and packing points"), points past max_points are dropped, and
// pillars created after max_voxels rows are taken are dropped whole.  Which
// points and pillars survive a cap, and in what order, varies from run to
// run, as the page says of its own kernel ("Results"); the pillar set, the
// counts and, for pillars under the cap, the point sets do not.
//
// One cooperative launch and one grid barrier.  Phase U1, every point: bin,
// find the slot (direct or hashed, as in the ordered kernel), group the
// warp's points by slot (match), and let one leader per group claim the
// slot's head word: free -> pending with atomicCAS; the creators of the
// warp take consecutive row numbers with one atomicAdd and publish them;
// other leaders wait (bounded) while the word is pending.  The leader then
// reserves the group's positions in the row with one atomicAdd and every
// point stores its row at its position.  A warp finishes all of its own
// claims before any lane waits, so a wait only ever waits for a warp that
// is past its claim.  Phase U2, after the barrier: counts (capped),
// coordinates, zero padding, and the clean-up of every slot created
// (recorded by creation number).
constexpr unsigned long long kRowPending = ~1ull;  // head word 0 while its creator takes a row
constexpr unsigned long long kRowDropped = ~2ull;  // pillar created past max_voxels

__device__ __forceinline__ unsigned long long ld_volatile_u64(const unsigned long long* p) {
  return *reinterpret_cast<const volatile unsigned long long*>(p);
}

__global__ void __launch_bounds__(kThreads, kMinBlocksPerSM) pv_unordered_kernel(const KParams p) {
  __shared__ int s_flag;
  __shared__ unsigned int s_dirty;
  __shared__ unsigned int s_total;
  const unsigned int P = gridDim.x;
  const unsigned int tid = threadIdx.x;
  const unsigned int lane = tid & 31u;
  const size_t gtid = static_cast<size_t>(blockIdx.x) * kThreads + tid;
  const size_t gthreads = static_cast<size_t>(P) * kThreads;
  const long long gwarp = static_cast<long long>(blockIdx.x) * kWarps + (tid >> 5);
  const long long nwarps = static_cast<long long>(P) * kWarps;
  const int K = p.K;
  const unsigned int M = static_cast<unsigned int>(p.max_voxels);
  unsigned int epoch = 0;  // thread 0 alone reads the control block (one L2 line)
  if (tid == 0) {
    epoch = ld_relaxed(&p.ctl->epoch);
    s_dirty = ld_relaxed(&p.ctl->dirty);
  }
  __syncthreads();
  const bool dirty = s_dirty != 0u;
  unsigned int bar_target = P;
  bool alive = true;

  if (dirty) {  // recovery after a failed launch: empty every table first
    reset_tables(p, gtid, gthreads);
    if (gtid == 0) p.ctl->created = 0u;
    alive = grid_sync(p.ctl, bar_target, &s_flag);
    bar_target += P;
  }

  // ---- phase U1.  Every lane of a warp runs the same trips (the grid stride
  // is a multiple of 32), so the match and the shuffles see the whole warp.
  if (alive) {
    for (long long base = 0; base < p.n; base += static_cast<long long>(gthreads)) {
      const long long i = base + static_cast<long long>(gtid);
      const float4 q = i < p.n ? __ldg(p.points + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      int slot = -1, key = 0;
      if (i < p.n) {
        if (bin_point(q, p, &key)) {
          slot = p.hash_mode ? claim_slot(p.keys, p.table_mask, key) : key;
          if (slot < 0) atomicMin(&p.ctl->err, PV_ERR_CAPACITY);
        }
      }
      const unsigned int peers = __match_any_sync(0xffffffffu, slot);
      const int leader = __ffs(peers) - 1;
      const bool lead = slot >= 0 && static_cast<int>(lane) == leader;
      unsigned long long* const head = p.lists + static_cast<size_t>(slot < 0 ? 0 : slot) * kHead;
      unsigned long long word = 0;
      if (lead) word = atomicCAS(head, kEmpty64, kRowPending);
      const bool creator = lead && word == kEmpty64;
      const unsigned int cm = __ballot_sync(0xffffffffu, creator);
      unsigned int cbase = 0;
      if (cm != 0u) {
        const int first = __ffs(cm) - 1;
        if (static_cast<int>(lane) == first) cbase = atomicAdd(&p.ctl->created, static_cast<unsigned int>(__popc(cm)));
        cbase = __shfl_sync(0xffffffffu, cbase, first);
      }
      long long row = -1;
      if (creator) {
        const unsigned int a = cbase + __popc(cm & lanemask_lt());
        p.firsts[a] = slot;  // creation records (at most one per distinct slot): slot for the clean-up,
        p.slot_of_point[a] = key;  // id for the coordinates
        row = a < M ? static_cast<long long>(a) : -1;
        atomicExch(head, a < M ? static_cast<unsigned long long>(a) : kRowDropped);
      }
      __syncwarp();
      if (lead && !creator) {
        if (word == kRowPending) {  // bounded wait for the creator's row
          const unsigned long long t0 = global_timer_ns();
          do {
            word = ld_volatile_u64(head);
            if (word != kRowPending) break;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
              atomicMin(&p.ctl->err, PV_ERR_TIMEOUT);
              break;
            }
          } while (true);
        }
        row = word < static_cast<unsigned long long>(M) ? static_cast<long long>(word) : -1;
      }
      row = __shfl_sync(0xffffffffu, row, leader);
      unsigned int pbase = 0;
      if (lead && row >= 0) pbase = atomicAdd(p.row_cnt + row, static_cast<unsigned int>(__popc(peers)));
      pbase = __shfl_sync(0xffffffffu, pbase, leader);
      const unsigned int pos = pbase + __popc(peers & lanemask_lt());
      if (slot >= 0 && row >= 0 && pos < static_cast<unsigned int>(K))
        p.out_voxels[static_cast<size_t>(row) * K + pos] = q;
    }
    alive = grid_sync(p.ctl, bar_target + p.bar_extra, &s_flag);
  }

  unsigned int V = 0;
  if (alive) {
    if (tid == 0) s_total = ld_relaxed(&p.ctl->created);  // thread 0 alone: one L2 line
    __syncthreads();
    const unsigned int total = s_total;
    V = total < M ? total : M;
    // ---- phase U2: one warp per row: count, coordinates, zeros past the count.
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long r = gwarp; r < static_cast<long long>(M); r += nwarps) {
      unsigned int c = 0;
      int key = 0;
      if (r < static_cast<long long>(V)) {
        c = __ldcg(p.row_cnt + r);
        c = c < static_cast<unsigned int>(K) ? c : static_cast<unsigned int>(K);
        key = __ldcg(p.slot_of_point + r);
      }
      __syncwarp();
      for (unsigned int e = c + lane; e < static_cast<unsigned int>(K); e += 32)
        p.out_voxels[static_cast<size_t>(r) * K + e] = z4;
      if (lane == 0) {
        const bool live = r < static_cast<long long>(V);
        const int kxy = static_cast<int>(fast_div(static_cast<unsigned int>(key), p.div_x));
        const int kz = static_cast<int>(fast_div(static_cast<unsigned int>(kxy), p.div_y));
        p.out_counts[r] = static_cast<int32_t>(c);
        p.out_coords[3 * r] = live ? kz : 0;
        p.out_coords[3 * r + 1] = live ? kxy - kz * p.g_y : 0;
        p.out_coords[3 * r + 2] = live ? key - kxy * p.g_x : 0;
        if (live) p.row_cnt[r] = 0u;
      }
    }
    // Clean-up of every created slot (rows and dropped pillars alike).
    for (size_t a = gtid; a < total; a += gthreads) {
      const int slot = __ldcg(p.firsts + a);
      p.lists[static_cast<size_t>(slot) * kHead] = kEmpty64;
      if (p.hash_mode) p.keys[slot] = kNoKey;
    }
  }

  __syncthreads();
  if (tid == 0) {
    // Acquire-release count of finished blocks: the last one sees every
    // block's writes (their error words included) before it reads them.
    const unsigned int prev = atom_add_acq_rel(&p.ctl->done, 1u);
    if (prev == P - 1) {
      const int err = *reinterpret_cast<volatile int*>(&p.ctl->err);
      *p.out_num = err != 0 ? err : static_cast<int32_t>(V);
      p.ctl->dirty = err != 0 ? 1u : 0u;
      p.ctl->err = 0;
      p.ctl->bar = 0;
      p.ctl->done = 0;
      p.ctl->created = 0;
      const unsigned int next = epoch + 1;
      p.ctl->epoch = next == 0 ? 1u : next;
    }
  }
}

// ------------------------------------------------------------ centroid downsampling

// Voxel-grid downsampling (the cuda-kdtree ICP page, "4.4": voxel_downsample
// replaces the voxel-grid filter, accumulating every point into its voxel,
// then a reduce by key): every occupied voxel becomes the mean of its points
// (x, y, z, intensity), in the canonical voxel order (first point), the first
// max_voxels voxels kept; cells by the Voxelize binning rule.  Sums are
// double; the order of the additions differs from the sequential oracle,
// which can move a mean by one float32 unit in the last place at most (see
// the tests).  Counts, coordinates and the order are exact.
//
// One cooperative launch, two grid barriers, the ordered kernel's skeleton:
// phase D1 per 1024-point tile of the block's chunk: bin, find the slot,
// sum each warp's points of one voxel by pointer jumping along the group
// (five shuffle rounds at most, none for single points), add the warp sums
// into a shared-memory map of the tile's voxels, then flush the map with one
// set of global atomics per voxel (4 double adds, the count, the first
// index).  Phase D2: a point is its voxel's first iff it is a warp-group
// leader whose index the accumulator holds; blocks compact their first
// points in index order; counts, barrier, scan.  Phase D3: rank r reads its
// voxel's accumulator, writes the centroid (double quotient rounded to
// float), coordinates and count, and empties the accumulator.
// (*ah, *al) += (bh, bl) in float-float: the high parts' exact two-sum, the
// low parts folded into its error, and an exact two-sum to renormalise.  The
// result is within a few units of 2^-46 of the operands' magnitudes.
__device__ __forceinline__ void two_sum(float a, float b, float* s, float* e) {
  *s = __fadd_rn(a, b);
  const float bb = __fsub_rn(*s, a);
  *e = __fadd_rn(__fsub_rn(a, __fsub_rn(*s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ void ff_add(float* ah, float* al, float bh, float bl) {
  float s, e;
  two_sum(*ah, bh, &s, &e);
  e = __fadd_rn(e, __fadd_rn(*al, bl));
  two_sum(s, e, ah, al);
}

// A double sum divided by a count, rounded to float, within one float ulp
// of float(s / n) and without a double division (slow on GB300): s split
// into two floats, the quotient of the high part by n from a correctly
// rounded 1/n, then one correction with the exact remainder and the low
// part.  Counts from 2^24 (not exact as floats) take the double division.
__device__ __forceinline__ float mean_of(double s, unsigned int count) {
  if (count >= (1u << 24)) return static_cast<float>(s / static_cast<double>(count));
  const float sh = __double2float_rn(s);
  const float sl = __double2float_rn(s - static_cast<double>(sh));
  const float nf = static_cast<float>(count);
  const float rcp = __frcp_rn(nf);
  const float q = __fmul_rn(sh, rcp);
  const float rem = __fmaf_rn(-q, nf, sh);  // sh - q * n, rounded once
  return __fmaf_rn(__fadd_rn(rem, sl), rcp, q);
}

constexpr int kDsHash = 2 * kThreads;  // count map positions (a tile's warp groups)
constexpr int kDsHot = 256;            // hot table positions (at most half used)
constexpr unsigned int kDsHotGroups = 4;  // warp groups of one voxel in the first tile that make it hot
constexpr int kDsSmem = kDsHash * (4 + 4) + kDsHot * (4 + 16 + 16 + 4 + 4);

__global__ void __launch_bounds__(kThreads, kMinBlocksPerSM) pv_downsample_kernel(const KParams p) {
  extern __shared__ __align__(16) unsigned char s_dyn[];
  __shared__ unsigned int s_prefix[kMaxCtas + 1];
  __shared__ unsigned int s_tile[kFlagUnroll][kWarps];
  __shared__ unsigned int s_tmp[kWarps + 1];
  __shared__ int s_flag;
  __shared__ unsigned int s_dirty;
  __shared__ int s_hot;  // the hot table holds a voxel

  const unsigned int P = gridDim.x;
  const unsigned int cta = blockIdx.x;
  const unsigned int tid = threadIdx.x;
  const unsigned int lane = tid & 31u;
  const unsigned int warp = tid >> 5;
  const size_t gtid = static_cast<size_t>(cta) * kThreads + tid;
  const size_t gthreads = static_cast<size_t>(P) * kThreads;
  const long long gwarp = static_cast<long long>(cta) * kWarps + warp;
  const long long nwarps = static_cast<long long>(P) * kWarps;
  const long long begin = lmin(p.n, static_cast<long long>(cta) * p.chunk);
  const long long end = lmin(p.n, begin + p.chunk);
  const unsigned int M = static_cast<unsigned int>(p.max_voxels);
  unsigned int epoch = 0;  // thread 0 alone reads the control block (one L2 line)
  if (tid == 0) {
    epoch = ld_relaxed(&p.ctl->epoch);
    s_dirty = ld_relaxed(&p.ctl->dirty);
  }
  __syncthreads();
  const bool dirty = s_dirty != 0u;
  unsigned int bar_target = P;
  bool alive = true;

  if (dirty) {
    reset_tables(p, gtid, gthreads);
    alive = grid_sync(p.ctl, bar_target, &s_flag);
    bar_target += P;
  }

  if (alive) {
    // ---- phase D1, every tile: bin and find the slot; each warp sums its
    // points of one voxel by pointer jumping along the group (at most five
    // shuffle rounds; none for lone points) in float-float (exact two-sums in
    // fp32: GB300's fp64 rate is a small fraction of its fp32 rate), and the
    // group's leader adds the sums' high and low parts to the voxel's double
    // accumulator with global reductions, with the count and the first index.
    //
    // Hot voxels (one voxel in many warps of a tile) would pile those
    // reductions onto one address.  A block with several tiles learns them
    // from its first tile (warp groups registered per voxel in a shared
    // count map) and sums them for the rest of its chunk in a shared table
    // instead: fp32 atomics whose exact rounding error (a two-sum with the
    // returned old value) goes into a second fp32 accumulator, flushed once
    // at the end.
    int* c_key = reinterpret_cast<int*>(s_dyn);                                 // [kDsHash] count map
    unsigned int* c_n = reinterpret_cast<unsigned int*>(c_key + kDsHash);       // [kDsHash]
    int* h_key = reinterpret_cast<int*>(c_n + kDsHash);                         // [kDsHot] hot table
    float* h_hi = reinterpret_cast<float*>(h_key + kDsHot);                     // [4][kDsHot]
    float* h_lo = h_hi + 4 * kDsHot;                                            // [4][kDsHot]
    unsigned int* h_n = reinterpret_cast<unsigned int*>(h_lo + 4 * kDsHot);     // [kDsHot]
    unsigned int* h_first = h_n + kDsHot;                                       // [kDsHot]
    const bool learn = end - begin > kThreads;  // several tiles: learn from the first
    if (learn) {
      for (int h = static_cast<int>(tid); h < kDsHash; h += kThreads) {
        c_key[h] = -1;
        c_n[h] = 0u;
      }
      for (int h = static_cast<int>(tid); h < kDsHot; h += kThreads) {
        h_key[h] = -1;
        for (int c = 0; c < 4; ++c) h_hi[c * kDsHot + h] = h_lo[c * kDsHot + h] = 0.f;
        h_n[h] = 0u;
        h_first[h] = 0xFFFFFFFFu;
      }
      if (tid == 0) s_hot = 0;
      __syncthreads();
    }
    for (long long tb = begin; tb < end; tb += kThreads) {
      const long long i = tb + tid;
      const float4 q = i < end ? __ldg(p.points + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      int slot = -1;
      if (i < end) {
        int key;
        if (bin_point(q, p, &key)) {
          slot = p.hash_mode ? claim_slot(p.keys, p.table_mask, key) : key;
          if (slot < 0) atomicMin(&p.ctl->err, PV_ERR_CAPACITY);
        }
      }
      const unsigned int peers = __match_any_sync(0xffffffffu, slot);
      const int leader = __ffs(peers) - 1;
      float hi[4] = {q.x, q.y, q.z, q.w}, lo[4] = {0.f, 0.f, 0.f, 0.f};
      int nxt = __ffs(peers & ~((2u << lane) - 1u)) - 1;  // the next member above this lane, or -1
      if (lane == 31u) nxt = -1;                           // (2 << 31 wraps to 0: no member above)
      while (__any_sync(0xffffffffu, nxt >= 0)) {
        const int src = nxt >= 0 ? nxt : static_cast<int>(lane);
        float oh[4], ol[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          oh[c] = __shfl_sync(0xffffffffu, hi[c], src);
          ol[c] = __shfl_sync(0xffffffffu, lo[c], src);
        }
        const int onext = __shfl_sync(0xffffffffu, nxt, src);
        if (nxt >= 0) {
#pragma unroll
          for (int c = 0; c < 4; ++c) ff_add(&hi[c], &lo[c], oh[c], ol[c]);
          nxt = onext;
        }
      }
      const bool lead = slot >= 0 && static_cast<int>(lane) == leader;
      if (i < end) p.slot_of_point[i] = slot < 0 ? -1 : (lead ? (slot | kLeaderBit) : slot);
      const bool first_tile = tb == begin;
      int hp = -1;  // hot table position of this group's voxel
      if (lead && learn && !first_tile && s_hot) {
        unsigned int h = mix32(static_cast<unsigned int>(slot)) & (kDsHot - 1);
        for (int probe = 0; probe < kDsHot; ++probe) {  // the table is fixed: read-only probes
          const int cur = h_key[h];
          if (cur == slot) {
            hp = static_cast<int>(h);
            break;
          }
          if (cur == -1) break;
          h = (h + 1) & (kDsHot - 1);
        }
      }
      if (hp >= 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float old = atomicAdd(h_hi + c * kDsHot + hp, hi[c]);
          float sum, err;
          two_sum(old, hi[c], &sum, &err);  // sum is what the atomic stored; err its exact rounding error
          atomicAdd(h_lo + c * kDsHot + hp, __fadd_rn(err, lo[c]));
        }
        atomicAdd(h_n + hp, static_cast<unsigned int>(__popc(peers)));
        atomicMin(h_first + hp, static_cast<unsigned int>(i));
      } else if (lead) {
        VoxAcc* A = p.acc + slot;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          atomicAdd(&A->s[c], static_cast<double>(hi[c]));
          if (lo[c] != 0.f) atomicAdd(&A->s[c], static_cast<double>(lo[c]));
        }
        atomicAdd(&A->count, static_cast<unsigned int>(__popc(peers)));
        atomicMax(&A->first_c, ~static_cast<unsigned int>(i));  // the leader holds the group's lowest index
      }
      if (learn && first_tile) {  // register the tile's warp groups, then keep the voxels with many
        if (lead) {
          unsigned int h = mix32(static_cast<unsigned int>(slot)) & (kDsHash - 1);
          for (int probe = 0; probe < kDsHash; ++probe) {  // at most kThreads keys: never full
            const int cur = atomicCAS(c_key + h, -1, slot);
            if (cur == -1 || cur == slot) break;
            h = (h + 1) & (kDsHash - 1);
          }
          atomicAdd(c_n + h, 1u);
        }
        __syncthreads();
        for (int h = static_cast<int>(tid); h < kDsHash; h += kThreads) {
          if (c_key[h] < 0 || c_n[h] < kDsHotGroups) continue;
          const int key = c_key[h];
          unsigned int t = mix32(static_cast<unsigned int>(key)) & (kDsHot - 1);
          for (int probe = 0; probe < kDsHot / 2; ++probe) {  // at most half full: later ones stay direct
            const int cur = atomicCAS(h_key + t, -1, key);
            if (cur == -1) {
              s_hot = 1;
              break;
            }
            t = (t + 1) & (kDsHot - 1);
          }
        }
        __syncthreads();  // the hot table is fixed from here on
      }
    }
    if (learn) {  // flush the hot table
      __syncthreads();
      for (int h = static_cast<int>(tid); h < kDsHot; h += kThreads) {
        const int key = h_key[h];
        if (key < 0 || h_n[h] == 0u) continue;
        VoxAcc* A = p.acc + key;
        for (int c = 0; c < 4; ++c) {
          atomicAdd(&A->s[c], static_cast<double>(h_hi[c * kDsHot + h]));
          atomicAdd(&A->s[c], static_cast<double>(h_lo[c * kDsHot + h]));
        }
        atomicAdd(&A->count, h_n[h]);
        atomicMax(&A->first_c, ~h_first[h]);
      }
    }
    alive = grid_sync(p.ctl, bar_target + p.bar_extra, &s_flag);
  }

  unsigned int V = 0;
  if (alive) {
    // ---- phase D2: first points of this block's range, compacted in index order.
    unsigned int local = 0;
    for (long long base = begin; base < end; base += static_cast<long long>(kFlagUnroll) * kThreads) {
      int s[kFlagUnroll];
      unsigned int fc[kFlagUnroll];
#pragma unroll
      for (int u = 0; u < kFlagUnroll; ++u) {
        const long long i = base + u * kThreads + tid;
        s[u] = i < end ? __ldcg(p.slot_of_point + i) : -1;
      }
#pragma unroll
      for (int u = 0; u < kFlagUnroll; ++u) {
        fc[u] = (s[u] >= 0 && (s[u] & kLeaderBit)) ? __ldcg(&p.acc[s[u] & ~kLeaderBit].first_c) : 0u;
        s[u] = s[u] >= 0 ? (s[u] & ~kLeaderBit) : -1;
      }
      unsigned int ball[kFlagUnroll];
#pragma unroll
      for (int u = 0; u < kFlagUnroll; ++u) {
        const long long i = base + u * kThreads + tid;
        ball[u] = __ballot_sync(0xffffffffu, s[u] >= 0 && fc[u] == ~static_cast<unsigned int>(i));
        if (lane == 0) s_tile[u][warp] = __popc(ball[u]);
      }
      __syncthreads();
      if (warp == 0) flag_prefix<kFlagUnroll>(&s_tile[0][0], &s_tmp[kWarps], lane);
      __syncthreads();
#pragma unroll
      for (int u = 0; u < kFlagUnroll; ++u)
        if ((ball[u] >> lane) & 1u)
          p.firsts[begin + local + s_tile[u][warp] + __popc(ball[u] & lanemask_lt())] = s[u];
      local += s_tmp[kWarps];
      __syncthreads();
    }
    if (tid == 0) p.counts[cta] = local;
    alive = grid_sync(p.ctl, bar_target + P, &s_flag);
  }

  if (alive) {
    unsigned int total = 0;
    const unsigned int c = tid < P ? __ldcg(p.counts + tid) : 0u;
    const unsigned int excl = block_exclusive_scan(c, s_tmp, &total);
    if (tid < P) s_prefix[tid] = excl;
    if (tid == 0) s_prefix[P] = total;
    __syncthreads();
    V = total < M ? total : M;
    // ---- phase D3: one voxel per thread; voxels past the budget only have
    // their accumulators emptied.  Runs of 32 ranks go to the warps of all
    // blocks in turn (block-major order would leave the first blocks alone
    // with every kept voxel's double divisions, which GB300 runs slowly).
    const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
    const size_t r0 = (static_cast<size_t>(warp) * P + cta) * 32 + lane;
    for (size_t r = r0; r < total; r += gthreads) {
      const int slot = slot_of_rank(p, s_prefix, P, static_cast<unsigned int>(r));
      uint4* a4 = reinterpret_cast<uint4*>(p.acc + slot);
      if (r < V) {
        VoxAcc A;  // written by other blocks' atomics: read from L2
        reinterpret_cast<uint4*>(&A)[0] = __ldcg(a4);
        reinterpret_cast<uint4*>(&A)[1] = __ldcg(a4 + 1);
        reinterpret_cast<uint4*>(&A)[2] = __ldcg(a4 + 2);
        p.out_voxels[r] = make_float4(mean_of(A.s[0], A.count), mean_of(A.s[1], A.count),
                                      mean_of(A.s[2], A.count), mean_of(A.s[3], A.count));
        const int key = p.hash_mode ? __ldcg(p.keys + slot) : slot;
        const int kxy = static_cast<int>(fast_div(static_cast<unsigned int>(key), p.div_x));
        const int kz = static_cast<int>(fast_div(static_cast<unsigned int>(kxy), p.div_y));
        p.out_coords[3 * r] = kz;
        p.out_coords[3 * r + 1] = kxy - kz * p.g_y;
        p.out_coords[3 * r + 2] = key - kxy * p.g_x;
        p.out_counts[r] = static_cast<int32_t>(A.count);
      }
      a4[0] = z4;
      a4[1] = z4;
      a4[2] = z4;
      if (p.hash_mode) p.keys[slot] = kNoKey;
    }
    // Rows V .. max_voxels-1 are zero.
    for (size_t r = static_cast<size_t>(V) + gtid; r < M; r += gthreads) {
      p.out_voxels[r] = make_float4(0.f, 0.f, 0.f, 0.f);
      p.out_coords[3 * r] = 0;
      p.out_coords[3 * r + 1] = 0;
      p.out_coords[3 * r + 2] = 0;
      p.out_counts[r] = 0;
    }
  }

  __syncthreads();
  if (tid == 0) {
    // Acquire-release count of finished blocks: the last one sees every
    // block's writes (their error words included) before it reads them.
    const unsigned int prev = atom_add_acq_rel(&p.ctl->done, 1u);
    if (prev == P - 1) {
      const int err = *reinterpret_cast<volatile int*>(&p.ctl->err);
      *p.out_num = err != 0 ? err : static_cast<int32_t>(V);
      p.ctl->dirty = err != 0 ? 1u : 0u;
      p.ctl->err = 0;
      p.ctl->bar = 0;
      p.ctl->done = 0;
      const unsigned int next = epoch + 1;
      p.ctl->epoch = next == 0 ? 1u : next;
    }
  }
  (void)gwarp;
  (void)nwarps;
}

// ------------------------------------------------------------ host side

struct DeviceInfo {
  int sms = 0;
  int blocks_per_sm = 0;
  bool cooperative = false;
};

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

// Dynamic shared memory opt-in for both instantiations of the ordered kernel;
// returns the resident blocks per SM of the smaller one (0 on failure).
int prepare_kernels() {
  int single = 0, queued = 0, batched = 0;
  if (cudaFuncSetAttribute(pv_voxelize_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(pv_voxelize_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(pv_voxelize_kernel<kMaxFrames, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kDynSmem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&single, pv_voxelize_kernel<1, false>, kThreads, kDynSmem) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&queued, pv_voxelize_kernel<1, true>, kThreads, kDynSmem) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&batched, pv_voxelize_kernel<kMaxFrames, false>, kThreads,
                                                    kDynSmem) != cudaSuccess ||
      cudaFuncSetAttribute(pv_downsample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDsSmem) !=
          cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return std::min(std::min(single, queued), batched);
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
  pl->ctas = std::min(std::min(kMaxCtas, kThreads), std::max(1, dev.sms * per_sm));
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
  const bool queue = static_cast<int64_t>(M) >= kQueueMinRowsPerWarp * pl.ctas * kWarps;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned int>(pl.ctas));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.unordered ? 0 : kDynSmem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (pl.downsample) {
    cfg.dynamicSmemBytes = kDsSmem;
    e = cudaLaunchKernelEx(&cfg, pv_downsample_kernel, kp);
  } else if (pl.unordered) {
    e = cudaLaunchKernelEx(&cfg, pv_unordered_kernel, kp);
  } else if (!pl.batched) {
    Frames<1> fr;
    fr.off[0] = 0;
    fr.off[1] = N;
    e = queue ? cudaLaunchKernelEx(&cfg, pv_voxelize_kernel<1, true>, kp, fr)
              : cudaLaunchKernelEx(&cfg, pv_voxelize_kernel<1, false>, kp, fr);
  } else {
    Frames<kMaxFrames> fr;  // copied into the launch: the caller's array may go at once
    for (int b = 0; b <= kMaxFrames; ++b) fr.off[b] = b <= pl.frames ? frame_offsets[b] : N;
    e = cudaLaunchKernelEx(&cfg, pv_voxelize_kernel<kMaxFrames, false>, kp, fr);
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
  if ((st = make_plan(N, range, vsize, 1, M, nullptr, di, &pl)) != PV_OK) return st;
  pl.downsample = true;
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
    if (cudaMemcpyAsync(out_voxels_host, d_vox, 16 * static_cast<size_t>(max_voxels) * max_points,
                        cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(out_coords_host, d_crd, 12 * static_cast<size_t>(max_voxels), cudaMemcpyDeviceToHost,
                        s) != cudaSuccess ||
        cudaMemcpyAsync(out_counts_host, d_cnt, 4 * static_cast<size_t>(max_voxels), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(out_num_voxels_host, d_num, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
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
  plan_out->threads = kThreads;
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

#ifdef PV_INSTRUMENT
// Instrumented builds only: copies and clears the list-insert statistics.
int pv_debug_insert_stats(unsigned long long* out) {
  if (cudaMemcpyFromSymbol(out, g_insert_stats, sizeof(unsigned long long) * 4) != cudaSuccess) return PV_ERR_CUDA;
  static const unsigned long long zeros[4] = {};
  if (cudaMemcpyToSymbol(g_insert_stats, zeros, sizeof zeros) != cudaSuccess) return PV_ERR_CUDA;
  return PV_OK;
}

// Instrumented builds only: copies [max_ctas][8] phase-1 first-tile stamps (ns) to host.
int pv_debug_p1_times(unsigned long long* out, int max_ctas) {
  const int n = max_ctas < kStampCtas ? max_ctas : kStampCtas;
  if (cudaMemcpyFromSymbol(out, g_p1_ns, sizeof(unsigned long long) * kStamps * n) != cudaSuccess)
    return PV_ERR_CUDA;
  return PV_OK;
}

// Instrumented builds only: copies [max_ctas][8] phase stamps (ns) to host.
// Instrumented builds only: lookups in the hashed table by positions probed
// (index 0 unused, 1 .. 32, 32 = 32 or more, 33 = table full); reset after the read.
int pv_debug_probe_hist(unsigned long long* out) {
  if (cudaMemcpyFromSymbol(out, g_probe_hist, sizeof(g_probe_hist)) != cudaSuccess) return PV_ERR_CUDA;
  const unsigned long long zero[34] = {};
  if (cudaMemcpyToSymbol(g_probe_hist, zero, sizeof(zero)) != cudaSuccess) return PV_ERR_CUDA;
  return PV_OK;
}

int pv_debug_phase_times(unsigned long long* out, int max_ctas) {
  const int n = max_ctas < kStampCtas ? max_ctas : kStampCtas;
  if (cudaMemcpyFromSymbol(out, g_phase_ns, sizeof(unsigned long long) * kStamps * n) != cudaSuccess)
    return PV_ERR_CUDA;
  return PV_OK;
}
#endif

}  // extern "C"
