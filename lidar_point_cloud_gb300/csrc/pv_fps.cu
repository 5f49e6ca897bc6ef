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
// How: one thread-block cluster per cloud keeps the whole cloud on chip, so
// an iteration never touches global memory: 16 CTAs of 256 threads with 16
// points a thread in registers, or 8 CTAs of 256 threads with 32 points a
// thread when a launch has more clouds than the GPU holds 16-CTA clusters
// (clouds up to 65,536 points); beyond, 16 or 8 CTAs of 1024 threads with the
// points in shared memory (16 bytes a point, up to 13,312 points a CTA).
// Iteration k: every thread updates its running minima against the last
// sample and takes its farthest point (largest distance, then lowest index);
// each warp reduces (distance bits, index) with two redux instructions, one
// block barrier, and warp 0 reduces the warps' bests, reads the winner's
// coordinates from the CTA's shared copy and stores (distance bits, index,
// coordinates) into this CTA's slot in every CTA of the cluster (st.async
// into distributed shared memory, slots and barriers kept by iteration
// parity), each store counting its bytes on the receiving CTA's mbarrier.
// When a CTA's barrier has seen every CTA's entry, each of its warps picks
// the winner from its own shared memory: the next query.  No cluster barrier
// inside the loop; nothing waits on another cluster.
//
// Distances: ((dx * dx) + (dy * dy)) + (dz * dz) in float, each operation
// rounded to nearest and none contracted, as in the oracle, so the samples
// are bit-identical.  The scalar intrinsics are used on purpose: the paired
// fp32 instructions (sub/mul/add.rn.f32x2) were fused by the code generator
// into a multiply-add in this kernel's context despite the explicit rounding
// mode, which changed about one distance in five by an ulp and with it, on
// LiDAR-shaped clouds full of near-ties, the samples.

#include "pv.h"

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace cg = cooperative_groups;

namespace {

// Clouds up to 65,536 points live in registers: in clusters of 16 CTAs (the
// non-portable cluster size) while a launch's clouds all fit on the GPU at
// once in such clusters, else in clusters of 8 CTAs; up to 131,072 points,
// 16 CTAs with 32 points a thread while the clouds fit at once.  Otherwise
// (up to PV_FPS_MAX_POINTS) the points live in shared memory, in clusters of
// 16 CTAs of 1024 threads on the same rule (always past 106,496 points, which
// 8 CTAs cannot hold), else 8.  Measured on the 65,536-point LiDAR-shaped
// cloud with 4,096 samples: 16 CTAs x 256 threads 2.51 ms (x 512: 2.77,
// x 128: 2.52); 8 CTAs x 256 threads 3.9 ms, and 3.6 ms for 15 clouds at once.
constexpr int kRegsPoints = 65536;
constexpr int kWideCluster = 16;
constexpr int kWideThreads = 256;
constexpr int kWidePer = kRegsPoints / (kWideCluster * kWideThreads);
constexpr int kBigRegsPoints = 131072;  // 16 CTAs x 256 threads x 32 points
constexpr int kBigPer = kBigRegsPoints / (kWideCluster * kWideThreads);
constexpr int kNarrowCluster = 8;
constexpr int kNarrowThreads = 256;
constexpr int kNarrowPer = kRegsPoints / (kNarrowCluster * kNarrowThreads);
constexpr int kClusterSmem = 8;
constexpr int kWideSmemCluster = 16;
constexpr int kThreadsSmem = 1024;
constexpr int kCapPerCta = 13312;  // points one CTA holds in shared memory
constexpr int kSmemBytes = kCapPerCta * 16;
static_assert(kCapPerCta * kWideSmemCluster == PV_FPS_MAX_POINTS, "16 CTAs hold the largest cloud");
// One CTA a SM: a cluster spread over as many SMs as it has CTAs.
constexpr int kSmemFloor = 120 * 1024;
static_assert(kWidePer * kWideCluster * kWideThreads == kRegsPoints && kNarrowPer * kNarrowCluster * kNarrowThreads == kRegsPoints,
              "65,536 points fill the registers");
static_assert(kSmemBytes + 2 * kClusterSmem * (kThreadsSmem / 32) * 24 + 256 <= 227 * 1024,
              "a CTA's share of the cloud and the exchange slots fit");

struct FpsParams {
  const float4* points;  // [B][n]
  long long n;
  long long m;
  long long start;
  int32_t* out_idx;      // [B][m]
  float4* out_samples;   // [B][m] or null
  int32_t* status;       // one int32: 0 or a negative status
};

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

// Warp argmax of (dbits, idx): the largest distance, then the lowest index.
// Returns both to every lane.
__device__ __forceinline__ void warp_best(unsigned int dbits, unsigned int idx, unsigned int* bd, unsigned int* bi) {
  const unsigned int d = __reduce_max_sync(0xffffffffu, dbits);
  *bi = __reduce_min_sync(0xffffffffu, dbits == d ? idx : 0xFFFFFFFFu);
  *bd = d;
}

__device__ __forceinline__ unsigned int smem_addr(const void* ptr) {
  return static_cast<unsigned int>(__cvta_generic_to_shared(ptr));
}

// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ unsigned int peer_addr(unsigned int addr, unsigned int rank) {
  unsigned int r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_init(unsigned int bar, unsigned int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// The local arrival of a phase, announcing the bytes the peers will store.
__device__ __forceinline__ void mbar_expect(unsigned int bar, unsigned int bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_test(unsigned int bar, unsigned int parity) {
  unsigned int ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `parity` to complete, for about a second at most.
__device__ __forceinline__ bool mbar_wait(unsigned int bar, unsigned int parity) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_test(bar, parity))
    if (global_ns() - t0 > 1000000000ull) return false;
  return true;
}

// Stores into a peer CTA's shared memory that count their bytes on the
// peer's barrier (`bar` is the peer's barrier address).
__device__ __forceinline__ void push_key(unsigned int addr, unsigned int d, unsigned int i, unsigned int bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(addr),
               "r"(d), "r"(i), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void push_xyz(unsigned int addr, float x, float y, float z, unsigned int bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "f"(x), "f"(y), "f"(z), "f"(0.0f), "r"(bar)
               : "memory");
}

// One cluster of kC CTAs of kT threads per cloud.  kP > 0: each thread holds
// kP points in registers (point tid + t * kT of the CTA's share in slot t),
// with a copy of the coordinates in shared memory to look a winner up;
// kP == 0: the points live in shared memory with their running minima.
//
// Per sample, every warp pushes its best (distance bits, index, coordinates)
// into every CTA of the cluster, into the slot of (CTA, warp) of the buffer
// of the sample's parity; each CTA's barrier of that parity completes when
// all kC * kT / 32 entries have landed, and every warp then takes the winner
// among them from its own shared memory.  A buffer is written again two
// samples later, only by a warp that has seen the next sample's entries of
// every warp of the cluster, each pushed after its warp had read this buffer.
template <int kC, int kT, int kP>
__global__ void __launch_bounds__(kT, 1) pv_fps_kernel(const FpsParams p) {
  constexpr int kW = kT / 32;
  constexpr int kE = kC;  // entries a CTA receives per sample: one from each CTA
  constexpr unsigned int kTx = kE * (8 + 16);
  extern __shared__ __align__(16) float4 s_pts[];  // (x, y, z, running minimum; unused with kP > 0)
  __shared__ __align__(8) uint2 s_wk[kW];          // each warp's best (distance bits, index)
  __shared__ __align__(16) float4 s_q[2][kE];      // coordinates of each entry
  __shared__ __align__(8) uint2 s_k[2][kE];        // (distance bits, index) of each entry
  __shared__ __align__(8) unsigned long long s_bar[2];
  __shared__ int s_bad, s_late;

  cg::cluster_group cluster = cg::this_cluster();
  const unsigned int rank = cluster.block_rank();
  const unsigned int tid = threadIdx.x;
  const unsigned int lane = tid & 31u;
  const unsigned int warp = tid >> 5;
  const long long cloud = blockIdx.x / kC;
  const float4* pts = p.points + cloud * p.n;
  const long long per = (p.n + kC - 1) / kC;
  const long long lo = static_cast<long long>(rank) * per;
  const long long cnt = lo < p.n ? (p.n - lo < per ? p.n - lo : per) : 0;
  const float inf = __int_as_float(0x7f800000);

  if (tid == 0) {
    s_bad = 0;
    s_late = 0;
    mbar_init(smem_addr(&s_bar[0]), 1);
    mbar_init(smem_addr(&s_bar[1]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  bool bad = false;
  constexpr int R = kP > 0 ? kP : 1;
  float px[R], py[R], pz[R], pd[R];
  for (long long j = tid; j < cnt; j += kT) {
    float4 v = __ldg(pts + lo + j);
    bad |= !finite3(v);
    v.w = inf;  // above every distance
    s_pts[j] = v;
  }
  if (kP > 0) {
#pragma unroll
    for (int t = 0; t < kP; ++t) {
      const long long j = tid + static_cast<long long>(t) * kT;
      const float4 v = j < cnt ? __ldg(pts + lo + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      px[t] = v.x;
      py[t] = v.y;
      pz[t] = v.z;
      pd[t] = j < cnt ? inf : -inf;  // -inf: no point, never the farthest
    }
  }
  // Lane c < kC of warp 0 stores this CTA's entry into its slot (rank) in CTA c.
  const unsigned int slot = rank;
  const unsigned int tgt = lane < static_cast<unsigned int>(kC) ? lane : 0u;
  const unsigned int rk0 = peer_addr(smem_addr(&s_k[0][slot]), tgt), rk1 = peer_addr(smem_addr(&s_k[1][slot]), tgt);
  const unsigned int rq0 = peer_addr(smem_addr(&s_q[0][slot]), tgt), rq1 = peer_addr(smem_addr(&s_q[1][slot]), tgt);
  const unsigned int rb0 = peer_addr(smem_addr(&s_bar[0]), tgt), rb1 = peer_addr(smem_addr(&s_bar[1]), tgt);
  const unsigned int lb0 = smem_addr(&s_bar[0]), lb1 = smem_addr(&s_bar[1]);
  const float4 q0 = __ldg(pts + p.start);
  float qx = q0.x, qy = q0.y, qz = q0.z;
  // Rank 0's last warp, which does not push, writes the sample indices.
  const bool writer = rank == 0 && warp == static_cast<unsigned int>(kW - 1);
  int32_t* const out_idx = p.out_idx + cloud * p.m;
  if (writer && lane == 0) out_idx[0] = static_cast<int32_t>(p.start);
  __syncthreads();   // the shared copy of the points is complete
  cluster.sync();    // every CTA's barriers are initialised before any entry is pushed
  if (bad) s_bad = 1;

  for (long long k = 1; k < p.m; ++k) {
    const int par = static_cast<int>(k & 1);
    const unsigned int parity = static_cast<unsigned int>((k - 1) >> 1) & 1u;
    const unsigned int lb = par ? lb1 : lb0;
    if (tid == 0) mbar_expect(lb, kTx);
    // Update the running minima against the last sample; this thread's farthest point.
    float m = -1.0f;
    long long bj = -1;  // point index inside this CTA
    if (kP > 0) {
#pragma unroll
      for (int t = 0; t < kP; ++t) pd[t] = fminf(pd[t], dist2(px[t], py[t], pz[t], qx, qy, qz));
#pragma unroll
      for (int t = 0; t < kP; ++t) m = fmaxf(m, pd[t]);
      int bt = 0;
#pragma unroll
      for (int t = kP - 1; t >= 0; --t)  // the lowest slot (lowest index) holding the maximum
        if (pd[t] == m) bt = t;
      bj = tid + static_cast<long long>(bt) * kT;
    } else {
      for (long long j = tid; j < cnt; j += kT) {
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
    if (lane == 0) s_wk[warp] = make_uint2(wd, wi);  // (0, none) from a warp without points
    __syncthreads();
    if (warp == 0) {  // the CTA's best, into every CTA of the cluster (lane c stores into CTA c)
      const bool in = lane < static_cast<unsigned int>(kW);
      const uint2 e = in ? s_wk[lane] : make_uint2(0u, 0xFFFFFFFFu);
      unsigned int cd, ci;
      warp_best(e.x, e.y, &cd, &ci);
      // The CTA's best is one of its own points: its coordinates from the shared copy.
      const float4 v = ci != 0xFFFFFFFFu ? s_pts[static_cast<long long>(ci) - lo] : make_float4(0.f, 0.f, 0.f, 0.f);
      if (lane < static_cast<unsigned int>(kC)) {
        const unsigned int rb = par ? rb1 : rb0;
        push_key(par ? rk1 : rk0, cd, ci, rb);
        push_xyz(par ? rq1 : rq0, v.x, v.y, v.z, rb);
      }
    }
    if (!__all_sync(0xffffffffu, mbar_wait(lb, parity))) {  // a peer stopped: give up
      if (lane == 0) s_late = 1;
      break;
    }
    // The winner among the cluster's entries, from this CTA's shared memory.
    const bool inq = lane < static_cast<unsigned int>(kC);
    const uint2 bk = inq ? s_k[par][lane] : make_uint2(0u, 0xFFFFFFFFu);
    const float4 bq = inq ? s_q[par][lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    unsigned int gd, gi;
    warp_best(bk.x, bk.y, &gd, &gi);
    const int sl = __ffs(__ballot_sync(0xffffffffu, inq && bk.x == gd && bk.y == gi)) - 1;
    qx = __shfl_sync(0xffffffffu, bq.x, sl);
    qy = __shfl_sync(0xffffffffu, bq.y, sl);
    qz = __shfl_sync(0xffffffffu, bq.z, sl);
    if (writer && lane == 0) out_idx[k] = static_cast<int32_t>(gi);
  }
  cluster.sync();  // no CTA leaves while a peer may still store into it

  if (rank == 0 && p.out_samples && !s_late) {
    __syncthreads();  // the index writes are visible to the block
    for (long long k = tid; k < p.m; k += kT) p.out_samples[cloud * p.m + k] = __ldg(pts + out_idx[k]);
  }
  if (tid == 0 && s_bad) atomicMin(p.status, PV_ERR_INVALID);
  if (tid == 0 && s_late) atomicMin(p.status, PV_ERR_TIMEOUT);
}

// ------------------------------------------------------------ host side

template <int kC, int kT, int kP>
cudaError_t launch_fps(const FpsParams& fp, int clouds, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned int>(clouds) * kC, 1, 1);
  cfg.blockDim = dim3(kT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kC;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pv_fps_kernel<kC, kT, kP>, fp);
}

// Dynamic shared memory of a register-variant CTA: the coordinates of its
// points, and at least kSmemFloor so that one CTA takes a whole SM.
inline size_t regs_smem(long long points) {
  const size_t b = static_cast<size_t>(points) * 16;
  return b < static_cast<size_t>(kSmemFloor) ? static_cast<size_t>(kSmemFloor) : b;
}

// How many clusters of this kernel the GPU runs at once (0 if the query fails).
template <int kC, int kT, int kP>
int max_clusters(size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kC, 1, 1);
  cfg.blockDim = dim3(kT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kC;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, pv_fps_kernel<kC, kT, kP>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int kC, int kT, int kP>
bool prepare_fps(size_t smem) {
  if (cudaFuncSetAttribute(pv_fps_kernel<kC, kT, kP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return false;
  if (kC > 8 && cudaFuncSetAttribute(pv_fps_kernel<kC, kT, kP>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                    cudaSuccess)
    return false;
  return true;
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
int g_wide_clusters[64];       // 16-CTA clusters the GPU holds at once (0: never take them)
int g_wide_smem_clusters[64];  // the same for the shared-memory variant
int g_big_clusters[64];        // the same for 32 points a thread in registers

}  // namespace

extern "C" int pv_fps(const float* points, int num_clouds, int64_t num_points, int64_t num_samples, int64_t start,
                      int32_t* out_indices, float* out_samples, int32_t* out_status, pv_stream_t stream) {
  if (!points || !out_indices || !out_status) return PV_ERR_INVALID;
  if (num_clouds < 1 || num_clouds > (1 << 26) || num_points < 1 || num_samples < 1 || start < 0 ||
      start >= num_points)
    return PV_ERR_INVALID;
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
      if (!prepare_fps<kClusterSmem, kThreadsSmem, 0>(kSmemBytes) ||
          !prepare_fps<kNarrowCluster, kNarrowThreads, kNarrowPer>(regs_smem(kNarrowThreads * kNarrowPer))) {
        cudaGetLastError();
        st = PV_ERR_CUDA;
      } else {
        // 16-CTA clusters are optional: without them every cloud takes 8 (and
        // clouds past 8 CTAs' shared memory are refused).
        const size_t wide = regs_smem(kWideThreads * kWidePer);
        g_wide_clusters[dev] = prepare_fps<kWideCluster, kWideThreads, kWidePer>(wide)
                                   ? max_clusters<kWideCluster, kWideThreads, kWidePer>(wide)
                                   : 0;
        cudaGetLastError();
        g_wide_smem_clusters[dev] = prepare_fps<kWideSmemCluster, kThreadsSmem, 0>(kSmemBytes)
                                        ? max_clusters<kWideSmemCluster, kThreadsSmem, 0>(kSmemBytes)
                                        : 0;
        cudaGetLastError();
        const size_t big = regs_smem(kWideThreads * kBigPer);
        g_big_clusters[dev] = prepare_fps<kWideCluster, kWideThreads, kBigPer>(big)
                                  ? max_clusters<kWideCluster, kWideThreads, kBigPer>(big)
                                  : 0;
        cudaGetLastError();
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
    if (cudaMemsetAsync(out_status, 0, sizeof(int32_t), s) != cudaSuccess) {
      st = PV_ERR_CUDA;
    } else {
      cudaError_t e;
      if (num_points <= kRegsPoints && num_clouds <= g_wide_clusters[dev]) {
        const long long per = (num_points + kWideCluster - 1) / kWideCluster;
        e = launch_fps<kWideCluster, kWideThreads, kWidePer>(fp, num_clouds, regs_smem(per), s);
      } else if (num_points <= kRegsPoints) {
        const long long per = (num_points + kNarrowCluster - 1) / kNarrowCluster;
        e = launch_fps<kNarrowCluster, kNarrowThreads, kNarrowPer>(fp, num_clouds, regs_smem(per), s);
      } else if (num_points <= kBigRegsPoints && num_clouds <= g_big_clusters[dev]) {
        const long long per = (num_points + kWideCluster - 1) / kWideCluster;
        e = launch_fps<kWideCluster, kWideThreads, kBigPer>(fp, num_clouds, regs_smem(per), s);
      } else {
        // Points in shared memory: 16-CTA clusters while the clouds fit on the
        // GPU at once in them (or when 8 CTAs cannot hold a cloud), else 8.
        const long long per8 = (num_points + kClusterSmem - 1) / kClusterSmem;
        const long long per16 = (num_points + kWideSmemCluster - 1) / kWideSmemCluster;
        const bool wide = g_wide_smem_clusters[dev] > 0 &&
                          (num_clouds <= g_wide_smem_clusters[dev] || per8 > kCapPerCta);
        if (wide) {
          e = launch_fps<kWideSmemCluster, kThreadsSmem, 0>(fp, num_clouds, regs_smem(per16), s);
        } else if (per8 <= kCapPerCta) {
          e = launch_fps<kClusterSmem, kThreadsSmem, 0>(fp, num_clouds, static_cast<size_t>(per8) * 16, s);
        } else {
          st = PV_ERR_UNSUPPORTED;  // no 16-CTA clusters on this device
          e = cudaSuccess;
        }
      }
      if (e != cudaSuccess) {
        cudaGetLastError();
        st = PV_ERR_CUDA;
      }
    }
  }
  if (prev != dev) cudaSetDevice(prev);
  return st;
}
