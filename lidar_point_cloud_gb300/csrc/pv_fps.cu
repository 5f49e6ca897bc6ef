// GB300 (sm_103a) farthest point sampling: the pv_fps entry of pv.h.
//
// What is computed is plain farthest point sampling, the operation the
// RadiusFPS page accelerates ("Baseline: classic GPU FPS"): from a start
// point, every point keeps its smallest squared distance to the samples so
// far and the next sample is the point whose distance is largest (ties to
// the lowest index).  The page's spherical-voxel pruning (its pruning
// theorem) skips only updates that cannot change a distance, so it never
// changes the samples.
//
// How: one thread-block cluster of 8 CTAs per cloud keeps the whole cloud in
// registers (8 points a thread: clouds up to 65,536 points) or in shared
// memory (16 bytes a point, up to 13,312 points a CTA), so an iteration never
// touches global memory.  Iteration k: every thread updates its running
// minima against the last sample and keeps its farthest point as one 64-bit
// key (distance bits high, complement of the index low: a larger key is a
// larger distance, then a lower index); warps, then warp 0, reduce the keys,
// and warp 0 pushes the CTA's best (key and coordinates) into every CTA of
// the cluster through distributed shared memory, into slots kept by
// iteration parity; one cluster barrier; then every warp picks the winner
// among the 8 CTA bests from its own shared memory: the next query.  One
// block barrier and one cluster barrier per sample; nothing waits on
// another cluster.
//
// Distances: ((dx * dx) + (dy * dy)) + (dz * dz) in float, each operation
// rounded to nearest and none contracted, as in the oracle, so the keys and
// therefore the samples are bit-identical.

#include "pv.h"

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace cg = cooperative_groups;

namespace {

constexpr int kCluster = 8;
constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kCapPerCta = PV_FPS_MAX_POINTS / kCluster;  // points held by one CTA
constexpr int kSmemBytes = kCapPerCta * 16;
static_assert(kSmemBytes + 2048 <= 227 * 1024, "a CTA's share of the cloud and the exchange slots fit");

struct FpsParams {
  const float4* points;  // [B][n]
  long long n;
  long long m;
  long long start;
  int32_t* out_idx;      // [B][m]
  float4* out_samples;   // [B][m] or null
  int32_t* status;       // one int32: 0 or a negative status
};

// A best point of an iteration: distance bits (a non-negative float orders
// like its bits), index, coordinates.  Larger distance wins, then the lower
// index.
struct Best {
  unsigned int dbits;
  unsigned int idx;
  float x, y, z;
  unsigned int pad[3];
};
static_assert(sizeof(Best) == 32, "two 16-byte stores");

__device__ __forceinline__ bool finite3(const float4& v) {
  return ((__float_as_uint(v.x) & 0x7f800000u) != 0x7f800000u) &&
         ((__float_as_uint(v.y) & 0x7f800000u) != 0x7f800000u) &&
         ((__float_as_uint(v.z) & 0x7f800000u) != 0x7f800000u);
}

// Squared distance exactly as the oracle evaluates it.
__device__ __forceinline__ float dist2(float px, float py, float pz, float qx, float qy, float qz) {
  const float dx = __fsub_rn(px, qx);
  const float dy = __fsub_rn(py, qy);
  const float dz = __fsub_rn(pz, qz);
  return __fadd_rn(__fadd_rn(__fmul_rn(dx, dx), __fmul_rn(dy, dy)), __fmul_rn(dz, dz));
}

// The same for two points at once with the paired fp32 instructions (each
// half rounded to nearest on its own, as the scalar operations).
__device__ __forceinline__ unsigned long long f32x2(float lo, float hi) {
  return (static_cast<unsigned long long>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}

__device__ __forceinline__ void dist2_x2(unsigned long long px, unsigned long long py, unsigned long long pz,
                                         unsigned long long qx, unsigned long long qy, unsigned long long qz,
                                         float* d0, float* d1) {
  unsigned long long dx, dy, dz, sx, sy, sz, s;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(dx) : "l"(px), "l"(qx));
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(dy) : "l"(py), "l"(qy));
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(dz) : "l"(pz), "l"(qz));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(sx) : "l"(dx), "l"(dx));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(sy) : "l"(dy), "l"(dy));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(sz) : "l"(dz), "l"(dz));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(s) : "l"(sx), "l"(sy));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(s) : "l"(s), "l"(sz));
  *d0 = __uint_as_float(static_cast<unsigned int>(s));
  *d1 = __uint_as_float(static_cast<unsigned int>(s >> 32));
}

// Warp argmax of (dbits, idx): the largest distance, then the lowest index.
// Returns both to every lane.
__device__ __forceinline__ void warp_best(unsigned int dbits, unsigned int idx, unsigned int* bd, unsigned int* bi) {
  const unsigned int d = __reduce_max_sync(0xffffffffu, dbits);
  *bi = __reduce_min_sync(0xffffffffu, dbits == d ? idx : 0xFFFFFFFFu);
  *bd = d;
}

// kRegs: the thread's kPerThread points live in registers (clouds of up to
// kCluster * kThreads * kPerThread points), with a copy of the coordinates in
// shared memory to look the winner up; otherwise the points live in shared
// memory.
constexpr int kPerThread = 8;

template <bool kRegs>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1) pv_fps_kernel(const FpsParams p) {
  extern __shared__ __align__(16) float4 s_pts[];  // (x, y, z, running minimum; unused in the register variant)
  __shared__ __align__(16) Best s_warp[kWarps];     // this CTA's warp bests
  __shared__ __align__(16) Best s_in[2][kCluster];  // every CTA's best, pushed by iteration parity
  __shared__ int s_bad;

  cg::cluster_group cluster = cg::this_cluster();
  const unsigned int rank = cluster.block_rank();
  const unsigned int tid = threadIdx.x;
  const unsigned int lane = tid & 31u;
  const unsigned int warp = tid >> 5;
  const long long cloud = blockIdx.x / kCluster;
  const float4* pts = p.points + cloud * p.n;
  const long long per = (p.n + kCluster - 1) / kCluster;
  const long long lo = static_cast<long long>(rank) * per;
  const long long cnt = lo < p.n ? (p.n - lo < per ? p.n - lo : per) : 0;
  const float inf = __int_as_float(0x7f800000);

  if (tid == 0) s_bad = 0;
  __syncthreads();
  bool bad = false;
  constexpr int R = kRegs ? kPerThread : 2;
  unsigned long long px2[R / 2], py2[R / 2], pz2[R / 2];
  float pd[R];
  for (long long j = tid; j < cnt; j += kThreads) {
    float4 v = __ldg(pts + lo + j);
    bad |= !finite3(v);
    v.w = inf;  // above every distance
    s_pts[j] = v;
  }
  if (kRegs) {
#pragma unroll
    for (int t = 0; t < kPerThread; t += 2) {
      const long long j0 = tid + static_cast<long long>(t) * kThreads, j1 = j0 + kThreads;
      const float4 a = j0 < cnt ? __ldg(pts + lo + j0) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 b = j1 < cnt ? __ldg(pts + lo + j1) : make_float4(0.f, 0.f, 0.f, 0.f);
      px2[t / 2] = f32x2(a.x, b.x);
      py2[t / 2] = f32x2(a.y, b.y);
      pz2[t / 2] = f32x2(a.z, b.z);
      pd[t] = j0 < cnt ? inf : -inf;  // -inf: no point, never the farthest
      pd[t + 1] = j1 < cnt ? inf : -inf;
    }
  }
  if (bad) s_bad = 1;
  const float4 q0 = __ldg(pts + p.start);
  float qx = q0.x, qy = q0.y, qz = q0.z;
  if (rank == 0 && tid == 0) p.out_idx[cloud * p.m] = static_cast<int32_t>(p.start);
  __syncthreads();

  for (long long k = 1; k < p.m; ++k) {
    const int par = static_cast<int>(k & 1);
    // Update the running minima against the last sample; this thread's farthest point.
    float m = -1.0f;
    long long bj = -1;  // point index inside this CTA
    if (kRegs) {
      const unsigned long long qx2 = f32x2(qx, qx), qy2 = f32x2(qy, qy), qz2 = f32x2(qz, qz);
#pragma unroll
      for (int t = 0; t < kPerThread; t += 2) {
        float d0, d1;
        dist2_x2(px2[t / 2], py2[t / 2], pz2[t / 2], qx2, qy2, qz2, &d0, &d1);
        pd[t] = fminf(pd[t], d0);
        pd[t + 1] = fminf(pd[t + 1], d1);
      }
#pragma unroll
      for (int t = 0; t < kPerThread; ++t) m = fmaxf(m, pd[t]);
#pragma unroll
      for (int t = kPerThread - 1; t >= 0; --t)  // the lowest slot (lowest index) holding the maximum
        if (pd[t] == m) bj = tid + static_cast<long long>(t) * kThreads;
    } else {
      for (long long j = tid; j < cnt; j += kThreads) {
        float4 v = s_pts[j];
        const float d = dist2(v.x, v.y, v.z, qx, qy, qz);
        if (d < v.w) {
          v.w = d;
          s_pts[j].w = d;
        }
        if (v.w > m) {  // strict: the lowest index among equal distances stays
          m = v.w;
          bj = j;
        }
      }
    }
    const bool has = m >= 0.0f;  // a thread without points (or only -inf) offers nothing
    const unsigned int dbits = has ? __float_as_uint(m) : 0u;
    const unsigned int gidx = has ? static_cast<unsigned int>(lo + bj) : 0xFFFFFFFFu;
    unsigned int wd, wi;
    warp_best(dbits, gidx, &wd, &wi);
    if (has && dbits == wd && gidx == wi) {  // the warp's winner records itself
      const float4 v = s_pts[bj];
      Best b;
      b.dbits = wd;
      b.idx = wi;
      b.x = v.x;
      b.y = v.y;
      b.z = v.z;
      s_warp[warp] = b;
    } else if (lane == 0 && wi == 0xFFFFFFFFu) {  // a warp without points
      Best b;
      b.dbits = 0u;
      b.idx = 0xFFFFFFFFu;
      b.x = b.y = b.z = 0.f;
      s_warp[warp] = b;
    }
    __syncthreads();
    if (warp == 0) {  // the CTA's best, pushed into every CTA of the cluster (lane c writes CTA c)
      const Best mine = s_warp[lane];
      unsigned int cd, ci;
      warp_best(mine.dbits, mine.idx, &cd, &ci);
      const int c = __ffs(__ballot_sync(0xffffffffu, mine.dbits == cd && mine.idx == ci)) - 1;
      if (lane < static_cast<unsigned int>(kCluster)) *cluster.map_shared_rank(&s_in[par][rank], lane) = s_warp[c];
    }
    cluster.sync();  // every CTA's best of iteration k is in every CTA
    // Every warp picks the winner among the 8 CTA bests, from its own shared memory.
    const bool in = lane < static_cast<unsigned int>(kCluster);
    const unsigned int td = in ? s_in[par][lane].dbits : 0u;
    const unsigned int ti = in ? s_in[par][lane].idx : 0xFFFFFFFFu;
    unsigned int gd, gi;
    warp_best(td, ti, &gd, &gi);
    const int src = __ffs(__ballot_sync(0xffffffffu, in && td == gd && ti == gi)) - 1;
    qx = s_in[par][src].x;
    qy = s_in[par][src].y;
    qz = s_in[par][src].z;
    if (rank == 0 && tid == 0) p.out_idx[cloud * p.m + k] = static_cast<int32_t>(gi);
  }
  cluster.sync();  // no CTA leaves while a peer may still write into it

  if (rank == 0 && p.out_samples) {
    __syncthreads();  // thread 0's index writes are visible to the block
    for (long long k = tid; k < p.m; k += kThreads)
      p.out_samples[cloud * p.m + k] = __ldg(pts + p.out_idx[cloud * p.m + k]);
  }
  if (tid == 0 && s_bad) atomicMin(p.status, PV_ERR_INVALID);
}

int device_of(const void* ptr) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged ? a.device : -1;
}

std::mutex g_fps_mu;
bool g_fps_ready[64];

}  // namespace

extern "C" int pv_fps(const float* points, int num_clouds, int64_t num_points, int64_t num_samples, int64_t start,
                      int32_t* out_indices, float* out_samples, int32_t* out_status, pv_stream_t stream) {
  if (!points || !out_indices || !out_status) return PV_ERR_INVALID;
  if (num_clouds < 1 || num_points < 1 || num_samples < 1 || start < 0 || start >= num_points) return PV_ERR_INVALID;
  if (num_samples >= (int64_t(1) << 31) || static_cast<int64_t>(num_clouds) * num_samples >= (int64_t(1) << 31))
    return PV_ERR_INVALID;
  if (num_points > PV_FPS_MAX_POINTS) return PV_ERR_TOO_LARGE;
  if (reinterpret_cast<uintptr_t>(points) % 16 || (out_samples && reinterpret_cast<uintptr_t>(out_samples) % 16) ||
      reinterpret_cast<uintptr_t>(out_indices) % 4 || reinterpret_cast<uintptr_t>(out_status) % 4)
    return PV_ERR_INVALID;
  const int dev = device_of(points);
  if (dev < 0 || device_of(out_indices) != dev || device_of(out_status) != dev ||
      (out_samples && device_of(out_samples) != dev))
    return PV_ERR_INVALID;
  if (dev >= 64) return PV_ERR_UNSUPPORTED;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return PV_ERR_CUDA;
  if (prev != dev && cudaSetDevice(dev) != cudaSuccess) return PV_ERR_CUDA;
  int st = PV_OK;
  {
    std::lock_guard<std::mutex> lk(g_fps_mu);
    if (!g_fps_ready[dev]) {
      if (cudaFuncSetAttribute(pv_fps_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
              cudaSuccess ||
          cudaFuncSetAttribute(pv_fps_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kThreads * kPerThread * 16) != cudaSuccess) {
        cudaGetLastError();
        st = PV_ERR_CUDA;
      } else {
        g_fps_ready[dev] = true;
      }
    }
  }
  if (st == PV_OK) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    FpsParams fp;
    fp.points = reinterpret_cast<const float4*>(points);
    fp.n = num_points;
    fp.m = num_samples;
    fp.start = start;
    fp.out_idx = out_indices;
    fp.out_samples = reinterpret_cast<float4*>(out_samples);
    fp.status = out_status;
    const long long per = (num_points + kCluster - 1) / kCluster;
    if (cudaMemsetAsync(out_status, 0, sizeof(int32_t), s) != cudaSuccess) {
      st = PV_ERR_CUDA;
    } else {
      const size_t smem = static_cast<size_t>(per) * 16;
      if (per <= static_cast<long long>(kThreads) * kPerThread)
        pv_fps_kernel<true><<<num_clouds * kCluster, kThreads, smem, s>>>(fp);
      else
        pv_fps_kernel<false><<<num_clouds * kCluster, kThreads, smem, s>>>(fp);
      if (cudaGetLastError() != cudaSuccess) st = PV_ERR_CUDA;
    }
  }
  if (prev != dev) cudaSetDevice(prev);
  return st;
}
