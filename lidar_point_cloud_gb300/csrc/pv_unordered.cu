// The unordered voxelizer (pv_voxelize_ex with order 1): one cooperative
// launch, one grid barrier; the contract and the design are in the comment
// before the kernel.

#include "pv_device.cuh"

namespace pvk {
namespace {

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
  wait_prior_grid();
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
      p.ctl->created = 0;
      const unsigned int next = epoch + 1;
      p.ctl->epoch = next == 0 ? 1u : next;
    }
  }
}

}  // namespace

// ------------------------------------------------------------ host side

cudaError_t launch_unordered(const cudaLaunchConfig_t& cfg, const KParams& kp) {
  return cudaLaunchKernelEx(&cfg, pv_unordered_kernel, kp);
}

}  // namespace pvk
