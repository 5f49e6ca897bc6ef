// Voxel-grid centroid downsampling (pv_voxel_downsample): one cooperative
// launch, two grid barriers; the reading and the design are in the comment
// before the kernel.  Built with 1024-thread blocks here and with 512-thread
// blocks, two an SM, by pv_downsample_half.cu (entry points named after the
// block size).

#include "pv_device.cuh"

namespace pvk {
namespace {

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


// First points of [begin, end) (a point whose index is its voxel's first),
// compacted in index order into firsts[begin ...]; FU block tiles a step.
// s_tile holds FU x kWarps counts, s_tmp kWarps + 1.  Returns the count.
template <int FU>
static __device__ unsigned int flag_firsts(const KParams& p, long long begin, long long end, unsigned int* s_tile,
                                           unsigned int* s_tmp) {
  const unsigned int tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
  unsigned int local = 0;
  for (long long base = begin; base < end; base += static_cast<long long>(FU) * kThreads) {
    int s[FU];
    unsigned int fc[FU];
#pragma unroll
    for (int u = 0; u < FU; ++u) {
      const long long i = base + u * kThreads + tid;
      s[u] = i < end ? __ldcg(p.slot_of_point + i) : -1;
    }
#pragma unroll
    for (int u = 0; u < FU; ++u) {
      fc[u] = (s[u] >= 0 && (s[u] & kLeaderBit)) ? __ldcg(&p.acc[s[u] & ~kLeaderBit].first_c) : 0u;
      s[u] = s[u] >= 0 ? (s[u] & ~kLeaderBit) : -1;
    }
    unsigned int ball[FU];
#pragma unroll
    for (int u = 0; u < FU; ++u) {
      const long long i = base + u * kThreads + tid;
      ball[u] = __ballot_sync(0xffffffffu, s[u] >= 0 && fc[u] == ~static_cast<unsigned int>(i));
      if (lane == 0) s_tile[u * kWarps + warp] = __popc(ball[u]);
    }
    __syncthreads();
    if (warp == 0) flag_prefix<FU>(s_tile, &s_tmp[kWarps], lane);
    __syncthreads();
#pragma unroll
    for (int u = 0; u < FU; ++u)
      if ((ball[u] >> lane) & 1u)
        p.firsts[begin + local + s_tile[u * kWarps + warp] + __popc(ball[u] & lanemask_lt())] = s[u];
    local += s_tmp[kWarps];
    __syncthreads();
  }
  return local;
}

__global__ void __launch_bounds__(kThreads, kMinBlocksPerSM) pv_downsample_kernel(const KParams p) {
  wait_prior_grid();
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
    // A chunk of one block tile (at most kThreads points) takes one step of
    // one tile (two on 512-thread blocks, so that one lane holds one whole
    // count); longer chunks take kFlagUnroll tiles a step.
    const unsigned int local = end - begin <= static_cast<long long>(kThreads)
                                   ? flag_firsts<(kWarps >= 32 ? 1 : 32 / kWarps)>(p, begin, end, &s_tile[0][0], s_tmp)
                                   : flag_firsts<kFlagUnroll>(p, begin, end, &s_tile[0][0], s_tmp);
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

  allow_next_grid();
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

}  // namespace

// ------------------------------------------------------------ host side

int PV_BLOCK_NAME(prepare_downsample_)() {
  int blocks = 0;
  if (cudaFuncSetAttribute(pv_downsample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDsSmem) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, pv_downsample_kernel, kThreads, kDsSmem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return blocks;
}

int PV_BLOCK_NAME(downsample_smem_)() { return kDsSmem; }

cudaError_t PV_BLOCK_NAME(launch_downsample_)(const cudaLaunchConfig_t& cfg, const KParams& kp) {
  return cudaLaunchKernelEx(&cfg, pv_downsample_kernel, kp);
}

}  // namespace pvk
