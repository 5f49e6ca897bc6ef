// GB300 (sm_103a) pillar voxelizer: kernels and the C ABI declared in pv.h.
//
// What is computed is the page "Voxelize" (ethan-howes.github.io/projects/
// voxelize/): bin every point into a pillar ("Implementation > Binning a
// point"), group points that share a pillar ("Claiming a pillar and packing
// points"), compact the pillars into dense outputs ("Compaction"), with the
// canonical order stated in pv.h.  How it is computed differs from the
// page's one-thread-per-point kernel + Thrust copy_if + gather:
//
//   * one cooperative launch, one 1024-thread block per SM (two 512-thread
//     blocks per SM, this file built again by pv_ordered_half.cu, for clouds
//     whose 1024-thread chunks would span several tiles), all resident, and
//     two grid-wide barriers;
//   * phase 1 (before the first barrier): blocks sweep the cloud in tiles of
//     consecutive points, one a thread (two a thread, tile by tile, where a
//     block's chunk spans several tiles), in index order across the grid.
//     Each point is read with one 16-byte load and binned with IEEE
//     round-to-nearest subtract/divide and floorf.  In shared memory the tile is grouped by
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
//     emptied; rows past V are zero-filled (left as they were for a
//     caller that takes only the first V rows: the host-buffer entry point).
//
// The table cleans itself: every slot a call fills is emptied by the same
// call, so no memset runs per call.  A launch that fails on the device marks
// the table dirty and the next launch resets it whole first.  Every wait is
// bounded by the global timer (about 1 s), after which the kernel records
// PV_ERR_TIMEOUT and returns.

#include "pv_device.cuh"

namespace pvk {
namespace {

// ------------------------------------------------------------ the kernel

// NF = 1: one cloud (pv_voxelize); NF = kMaxFrames: a batch of up to NF
// frames (pv_voxelize_batch), where a voxel's id carries its frame, each
// frame keeps its own first max_voxels voxels and writes its own rows.
// U: points per thread in a block tile at most.  A tile of S sub-tiles
// (S <= U) is S * kThreads consecutive points; warp w holds its points
// 32S.w .. 32S.w + 32S - 1, sub-tile u the 32 of them from 32S.w + 32u.
// With U = 2 a block's chunk starts with a one-sub-tile tile, and each next
// tile takes two sub-tiles while the last one had few tile groups (at most
// kThreads / 2 to widen, 5/8 of 2 kThreads to stay wide), so the maps
// stay at most 5/8 full: wide tiles halve the block barriers per point and
// the tile groups per pillar on clouds whose consecutive points share
// pillars; sparse clouds keep tiles of one point a thread.
template <int NF, bool kQueue, int U>
__global__ void __launch_bounds__(kThreads, kMinBlocksPerSM) pv_voxelize_kernel(const KParams p, const Frames<NF> fr) {
  static_assert(U == 1 || U == 2, "one or two points per thread in a tile");
  static_assert(U * kThreads <= kTileHash, "a tile's keys fit its map");
  wait_prior_grid();
  constexpr bool kBatched = NF > 1;
  // Block tiles in flight in the first-point pass: 8 where chunks are long
  // (the launches that queue long lists), else 4 (fewer empty tiles to scan).
  // With one point a thread a chunk is one tile (at most kThreads points):
  // its pass over points is one block tile (two on 512-thread blocks, so
  // that the counts fill whole lanes).
  constexpr int FU = U == 1 ? (kWarps >= 32 ? 1 : 32 / kWarps) : (kQueue ? kFlagUnrollWide : kFlagUnroll);
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
  __shared__ unsigned int s_groups[2];  // tile groups (distinct pillars) of the tile using each map
  __shared__ unsigned int s_nrec;
  __shared__ unsigned int s_qn, s_qh;  // gather: long lists queued by the block, and taken
  __shared__ unsigned int s_wrec[kWarps];  // single frame: records of each warp in the current tile

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
  int nsub = 1;  // sub-tiles of the current tile (see U)
  float4 q[U];
#pragma unroll
  for (int u = 0; u < U; ++u) q[u] = z4;
  if (tb + 32u * warp + lane < end) q[0] = __ldg(p.points + tb + 32u * warp + lane);
  // Thread 0 alone reads the control block (the same word read by every
  // thread would queue thousands of requests on one L2 line); the dirty flag
  // reaches the block through shared memory, the epoch only thread 0 needs.
  unsigned int epoch = 0, dirty_word = 0;
  if (tid == 0) {
    epoch = ld_relaxed(&p.ctl->epoch);
    dirty_word = ld_relaxed(&p.ctl->dirty);
  }
  unsigned int bar_target = P;
  // The dynamic shared memory this launch has: a launch of one-tile chunks
  // uses the first tile map alone (and, after phase 1, the gather's merge
  // buffers and the long-list queue in the same space, the queue as long as
  // it fits), and the host gives it kMapBytes; a launch of longer chunks
  // needs kDynSmem.  Too little: an error, no work (the same in every
  // block, so no barrier waits for a missing block).
  unsigned int dyn_bytes;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_bytes));
  const bool smem_short = dyn_bytes < static_cast<unsigned int>(kDynSmem) && (U > 1 || p.chunk > kThreads);
  bool alive = !smem_short;
  if (smem_short && cta == 0 && tid == 0) atomicMin(&p.ctl->err, PV_ERR_INTERNAL);
  const int B = kBatched ? p.frames : 1;
  if (kBatched)
    for (int b = static_cast<int>(tid); b <= B; b += kThreads) s_off[b] = fr.off[b];  // read after a block barrier
  PV_STAMP(0);
  // More than one tile (always so with U = 2): second map, chunk map and records in use.
  const bool multi = U > 1 || end - begin > kThreads;
  int* ckey = reinterpret_cast<int*>(s_dyn + 2 * kMapBytes);
  unsigned int* ccnt = reinterpret_cast<unsigned int*>(ckey + kChunkHash);
  {  // tile map 0 empty (counters zero, keys -1); map 1 and the chunk map only if used
    uint4* d4 = reinterpret_cast<uint4*>(s_dyn);
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const uint4 m1 = make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
    const int maps = smem_short ? 0 : (multi ? 2 : 1);
    for (int m = 0; m < maps; ++m) {
      uint4* base = d4 + m * (kMapBytes / 16);
      for (int j = static_cast<int>(tid); j < kTileHash * kWarps / 16; j += kThreads) base[j] = z;
      for (int j = static_cast<int>(tid); j < kTileHash * 4 / 16; j += kThreads)
        base[kTileHash * kWarps / 16 + j] = m1;
    }
    if (multi && !smem_short) {
      uint4* c4 = reinterpret_cast<uint4*>(ckey);
      for (int j = static_cast<int>(tid); j < kChunkHash / 4; j += kThreads) {
        c4[j] = m1;
        c4[kChunkHash / 4 + j] = z;
      }
    }
  }
  if (tid == 0) {
    s_layout[0] = s_layout[1] = 0;
    s_groups[0] = s_groups[1] = 0;
    s_nrec = 0;
    s_qn = s_qh = 0;
    s_dirty = dirty_word;
  }
  __syncthreads();  // maps empty, dirty flag shared
  const bool dirty = s_dirty != 0u;

  // Recovery after a failed launch: empty the whole table first.
  if (dirty && alive) {
    reset_tables(p, gtid, gthreads);
    alive = grid_sync(p.ctl, bar_target, &s_flag);
    bar_target += P;
  }

  // A single frame's chunk of several tiles lays its records out in index
  // order (tile by tile; in a tile by warp, sub-tile, lane), with their slots
  // in slot_of_point: the first-point pass then walks the records instead of
  // the points.  A batch records in arrival order, with the slots in firsts,
  // and tags every point in slot_of_point, as does a chunk of one tile.
  int32_t* const rec_slot = kBatched ? p.firsts : p.slot_of_point;

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
    unsigned int rec_run = 0;  // single frame: records of the chunk's earlier tiles
    for (; tb < end; buf ^= 1) {
#ifdef PV_INSTRUMENT
      const bool first_tile = tb == begin;
#endif
      PV_SUB(0);
      const TileMap tm = tile_map(s_dyn + buf * kMapBytes, &s_layout[buf]);
      const TileMap prev = tile_map(s_dyn + (buf ^ 1) * kMapBytes, &s_layout[buf ^ 1]);
      const unsigned int wofs = 32u * nsub * warp + lane;  // this thread's first point in the tile
      const long long tl = static_cast<long long>(nsub) * kThreads;
      long long i[U];
      float4 qn[U];
      int slot[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        i[u] = u < nsub ? tb + wofs + 32 * u : end;
        const long long inext = i[u] + tl;  // the next tile's point if it has as many sub-tiles
        qn[u] = (u < nsub && inext < end) ? __ldg(p.points + inext) : z4;  // in flight early
        slot[u] = -1;
        if (i[u] < end) {
          int key;
          if (bin_point(q[u], p, &key)) {
            if (kBatched) key += frame_of(s_off, B, i[u]) * p.cells;
            slot[u] = p.hash_mode ? claim_slot(p.keys, p.table_mask, key) : key;
            if (slot[u] < 0) atomicMin(&p.ctl->err, PV_ERR_CAPACITY);
          }
        }
      }
      PV_SUB(1);
      // Warp groups register in the tile map: per (position, warp) a byte
      // counts the warp's points of the pillar.  With U = 2 the counter is
      // added to atomically and sub-tile 1 reads how many of the warp's
      // sub-tile 0 points share its pillar (they come first).
      unsigned int peers[U], wb[U];
      int h[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (u >= nsub) {  // (block-uniform)
          peers[u] = 0u;
          wb[u] = 0u;
          h[u] = -1;
          continue;
        }
        peers[u] = __match_any_sync(0xffffffffu, slot[u]);
        const int leader = __ffs(peers[u]) - 1;
        int hh = -1;
        unsigned int old = 0;
        if (slot[u] >= 0 && static_cast<int>(lane) == leader) {
          hh = tile_claim(tm, slot[u]);
          if (hh >= 0) {
            if constexpr (U == 1) {
              reinterpret_cast<unsigned char*>(tm.cnt + hh * (kWarps / 4))[warp] =
                  static_cast<unsigned char>(__popc(peers[u]));
            } else {
              const unsigned int sh = 8u * (warp & 3u);
              old = atomicAdd(tm.cnt + hh * (kWarps / 4) + (warp >> 2), static_cast<unsigned int>(__popc(peers[u])) << sh);
              old = (old >> sh) & 0xFFu;
            }
          } else {  // cannot happen: at most U * kThreads keys in kTileHash >= U * kThreads positions
            atomicMin(&p.ctl->err, PV_ERR_INTERNAL);
          }
        }
        h[u] = __shfl_sync(0xffffffffu, hh, leader);
        wb[u] = U == 1 ? 0u : __shfl_sync(0xffffffffu, old, leader);
        if (h[u] < 0) slot[u] = -1;
        if (U > 1) __syncwarp();  // sub-tile u's counts land before sub-tile u + 1 reads them
      }
      __syncthreads();  // (A) every warp group registered; the previous tile's map is read
      PV_SUB(2);
      // Empty the previous tile's map (used again by the next tile, after barrier B).
      if (multi) {
        if (tid == 0) {
          *prev.layout = 0;
          s_groups[buf ^ 1] = 0;
        }
        tile_clear(prev, tid);
      }
      // Per point: its rank among the tile's points of its pillar; the
      // group's counts before this warp and in all are read by the leader
      // and shared by shuffles.  A group's first point (rank 0) leads it.
      unsigned int trank[U], tot[U], cseen[U];
      bool lead[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (u >= nsub) {  // (block-uniform)
          trank[u] = tot[u] = cseen[u] = 0u;
          lead[u] = false;
          continue;
        }
        const int leader = __ffs(peers[u]) - 1;
        unsigned int tr = 0, tt = 0;
        if (slot[u] >= 0 && static_cast<int>(lane) == leader) tile_counts(tm, h[u], warp, &tr, &tt);
        tr = __shfl_sync(0xffffffffu, tr, leader);
        tt = __shfl_sync(0xffffffffu, tt, leader);
        if (slot[u] >= 0) tr += wb[u] + __popc(peers[u] & lanemask_lt());
        trank[u] = tr;
        tot[u] = tt;
        lead[u] = slot[u] >= 0 && tr == 0;
        cseen[u] = (lead[u] && multi) ? chunk_rank(ckey, ccnt, slot[u], tt) : 0u;
      }
      unsigned int rpos[U];         // single frame: each record's place among its warp's records
      unsigned long long rent[U];  // single frame: the records, written after barrier B
      {  // group offsets and record slots: one shared-memory atomic per warp each
        // A group with max_points of its pillar's points before it in this
        // chunk (or max_points groups) can never be kept: not recorded.
        unsigned int need = 0, nrec_l = 0;
        bool wants[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          wants[u] = lead[u] && (cseen[u] >> 16) < static_cast<unsigned int>(K) &&
                     (cseen[u] & 0xFFFFu) < static_cast<unsigned int>(K);
          need += lead[u] ? tot[u] : 0u;
          nrec_l += (kBatched && multi && wants[u]) ? 1u : 0u;
        }
        // One scan for both: a warp's groups hold at most U * kThreads points (low
        // half) and it has at most 32U records (high half).
        unsigned int pk = need | (nrec_l << 16);
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
        if constexpr (U > 1) {  // the tile's groups, which set the next tile's width
          unsigned int ng = __popc(__ballot_sync(0xffffffffu, lead[0]));
          if (nsub > 1) ng += __popc(__ballot_sync(0xffffffffu, lead[1]));
          if (lane == 0 && ng) atomicAdd(&s_groups[buf], ng);
        }
        unsigned int off = base + incl - need;
        long long rj = begin + rbase + rincl - nrec_l;
        if (!kBatched && multi) {  // this warp's records: their places in it, its count to the block
          unsigned int wr = 0;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const unsigned int bw = u < nsub ? __ballot_sync(0xffffffffu, wants[u]) : 0u;
            rpos[u] = wr + __popc(bw & lanemask_lt());
            wr += __popc(bw);
          }
          if (lane == 0) s_wrec[warp] = wr;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          rent[u] = kEmpty64;
          if (lead[u]) {
            // Rows of the group that can ever be emitted: those with fewer than
            // max_points of the pillar's points before them in the chunk.
            const unsigned int cpts = cseen[u] & 0xFFFFu;
            const unsigned int room = cpts < static_cast<unsigned int>(K) ? static_cast<unsigned int>(K) - cpts : 0u;
            tm.off[h[u]] = ((tot[u] < room ? tot[u] : room) << 16) | off;
            if (wants[u]) {
              const unsigned int size = tot[u] < static_cast<unsigned int>(K) ? tot[u] : static_cast<unsigned int>(K);
              const unsigned long long ent = make_entry(i[u], cseen[u] >> 16, tb + off, size);
              if (!multi) {  // one tile (U = 1): the leader inserts its own record
                own_rs = slot[u];
                own_entry = ent;
              } else if (!kBatched) {
                rent[u] = ent;  // written once the block's warp counts are known (barrier B)
              } else {
                p.firsts[rj] = slot[u];  // the record's slot (firsts is rewritten after the barrier)
                p.recs[rj] = ent;
                ++rj;
              }
            }
            off += tot[u];
          }
        }
      }
      if (kBatched || !multi) {  // slot tags for the first-point pass over points
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (i[u] < end) p.slot_of_point[i[u]] = slot[u] < 0 ? -1 : (lead[u] ? (slot[u] | kLeaderBit) : slot[u]);
      }
      __syncthreads();  // (B) group offsets handed out; the previous map is empty
      PV_SUB(3);
      if (!kBatched && multi) {  // this tile's records, after the chunk's earlier ones, in index order
        const unsigned int cw = lane < static_cast<unsigned int>(kWarps) ? s_wrec[lane] : 0u;
        const unsigned int wbase = __reduce_add_sync(0xffffffffu, lane < warp ? cw : 0u);
        const unsigned int ttot = __reduce_add_sync(0xffffffffu, cw);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (rent[u] != kEmpty64) {
            const long long r = begin + rec_run + wbase + rpos[u];
            rec_slot[r] = slot[u];
            p.recs[r] = rent[u];
          }
        }
        rec_run += ttot;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (slot[u] >= 0) {
          const unsigned int ow = tm.off[h[u]];
          if (trank[u] < (ow >> 16)) p.tile_rows[tb + (ow & 0xFFFFu) + trank[u]] = q[u];
        }
      }
      PV_SUB(4);
      tb += tl;
      int next = 1;
      if constexpr (U > 1) {  // this tile's groups are all counted (barrier B)
        const unsigned int g = s_groups[buf];
        next = (nsub == 1 ? g <= kThreads / 2u : g <= kThreads * 5u / 4u) ? 2 : 1;
      }
      if (next == nsub) {
#pragma unroll
        for (int u = 0; u < U; ++u) q[u] = qn[u];
      } else {  // another width: the prefetched points are not the next tile's
        nsub = next;
        const unsigned int w2 = 32u * nsub * warp + lane;
#pragma unroll
        for (int u = 0; u < U; ++u)
          q[u] = (u < nsub && tb + w2 + 32 * u < end) ? __ldg(p.points + tb + w2 + 32 * u) : z4;
      }
    }
    if (!kBatched && multi && tid == 0) s_nrec = rec_run;
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
      int rs = j0 < nrec ? __ldcg(rec_slot + begin + j0) : -1;
      unsigned long long entry = j0 < nrec ? __ldcg(p.recs + begin + j0) : 0ull;
      for (; j0 < nrec; j0 += kThreads) {
        const unsigned int j1 = j0 + kThreads;
        const int rs1 = j1 < nrec ? __ldcg(rec_slot + begin + j1) : -1;
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
    if (!kBatched && multi) {
      // Over the chunk's records, in index order: a pillar's first point
      // leads the first group of the pillar in its chunk (chunk rank 0), so
      // only those records are tested against the slot's lowest leader.
      constexpr int FR = FU;
      const unsigned int nrec = s_nrec;
      for (unsigned int r0 = 0; r0 < nrec; r0 += FR * kThreads) {
        int s[FR];
        unsigned long long e[FR];
#pragma unroll
        for (int u = 0; u < FR; ++u) {
          const unsigned int r = r0 + u * kThreads + tid;
          s[u] = r < nrec ? __ldcg(rec_slot + begin + r) : -1;
          e[u] = r < nrec ? __ldcg(p.recs + begin + r) : kEmpty64;
        }
        uint32_t head[FR];
#pragma unroll
        for (int u = 0; u < FR; ++u)
          head[u] = (s[u] >= 0 && entry_crank(e[u]) == 0)
                        ? static_cast<uint32_t>(__ldcg(p.lists + static_cast<size_t>(s[u]) * kHead) >> 32)
                        : kEmpty;
        unsigned int ball[FR];
#pragma unroll
        for (int u = 0; u < FR; ++u) {
          ball[u] = __ballot_sync(0xffffffffu, s[u] >= 0 && head[u] == static_cast<uint32_t>(e[u] >> 32));
          if (lane == 0) s_tile[u][warp] = __popc(ball[u]);
        }
        __syncthreads();
        if (warp == 0) flag_prefix<FR>(&s_tile[0][0], &s_tmp[kWarps], lane);
        __syncthreads();
        unsigned int run = local;
#pragma unroll
        for (int u = 0; u < FR; ++u) {
          const unsigned int before = run + s_tile[u][warp] + __popc(ball[u] & lanemask_lt());
          if ((ball[u] >> lane) & 1u) p.firsts[begin + before] = s[u];
        }
        run += s_tmp[kWarps];
        local = run;
        __syncthreads();
      }
    } else {
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
    // Skipped where the caller takes only the first V rows (outputs in host
    // memory, where every byte crosses the host link).
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    const size_t Kz = static_cast<size_t>(K);
    constexpr size_t cw = kBatched ? 4 : 3;
    for (int b = 0; b < (p.zero_tail ? B : 0); ++b) {
      const unsigned int Vb = kBatched ? s_vcum[b + 1] - s_vcum[b] : V;
      const size_t lo = static_cast<size_t>(b) * M + Vb, hi = static_cast<size_t>(b + 1) * M;
      for (size_t q = lo * Kz + gtid; q < hi * Kz; q += gthreads) p.out_voxels[q] = z4;
      for (size_t q = cw * lo + gtid; q < cw * hi; q += gthreads) p.out_coords[q] = 0;
      for (size_t q = lo + gtid; q < hi; q += gthreads) p.out_counts[q] = 0;
    }

    PV_STAMP(5);

    // ---- phase 2c+2d: every ranked pillar, kept or past the budget.  Every
    // warp of the grid takes an equal share of the kept rows and an equal
    // share of the pillars past the budget (which only have their lists
    // emptied), and works through both together, 32 at a time.  Lane l finds the slot of
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
    const unsigned int qcap = dyn_bytes / 8u - static_cast<unsigned int>(kWarps) * 32u;  // queue entries that fit
    // (Counts of pillars and warps fit 32 bits: N < 2^29, at most 1024 x 32 warps.)
    const unsigned int dropped = kBatched ? s_dcum[B] : total - V;
    const unsigned int nw = static_cast<unsigned int>(nwarps), gw = static_cast<unsigned int>(gwarp);
    // A contiguous share of ranks per warp, or, where warps have many rows
    // (p.interleave), ranks gw, gw + nw, ...: pillars ranked near one another
    // lie near one another, and their long lists would bunch up in a few
    // blocks' shares.
    unsigned int kw0, nk, dw0, nd, stride;
    if (p.interleave) {
      kw0 = dw0 = gw;
      stride = nw;
      nk = V > gw ? (V - gw - 1) / nw + 1 : 0u;
      nd = dropped > gw ? (dropped - gw - 1) / nw + 1 : 0u;
    } else {
      // Share s = warp * blocks + block: a block's shares lie spread over the
      // rank range, so its queue meets its fair part of the long lists, and
      // with fewer shares than warps every block keeps warps busy.
      const unsigned int gs = warp * P + cta;
      const unsigned int pk = (V + nw - 1) / nw;
      kw0 = gs * pk < V ? gs * pk : V;
      nk = (kw0 + pk < V ? kw0 + pk : V) - kw0;
      const unsigned int pd = (dropped + nw - 1) / nw;
      dw0 = gs * pd < dropped ? gs * pd : dropped;
      nd = (dw0 + pd < dropped ? dw0 + pd : dropped) - dw0;
      stride = 1;
    }
    for (unsigned int t0 = 0; t0 < nk + nd; t0 += 32) {
      const unsigned int t = t0 + lane;
      const bool valid = t < nk;                  // kept: an output row
      const bool drop = !valid && t < nk + nd;    // past the budget
      const bool in_range = valid || drop;
      long long row = 0;
      unsigned int rank = 0;
      int fb = 0;
      if (valid) {
        const unsigned int k = kw0 + t * stride;  // the k-th row written (frames one after the other)
        rank = k;
        row = k;
        if (kBatched) {
          fb = slot_in_cum(s_vcum, B, k);
          const unsigned int loc = k - s_vcum[fb];
          rank = s_fpre[fb] + loc;
          row = static_cast<long long>(fb) * M + loc;
        }
      } else if (drop) {
        const unsigned int j = dw0 + (t - nk) * stride;  // the j-th pillar past a budget
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
        if (longv && qb < qcap) {
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
      const unsigned int qn = s_qn < qcap ? s_qn : qcap;
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
  allow_next_grid();
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

}  // namespace

// ------------------------------------------------------------ host side

// (static: the 512-thread build of this file has its own, with its own
// shared-memory size)
template <typename F>
static int prepare_one(F kern) {
  int blocks = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, kThreads, kDynSmem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return blocks;
}

int PV_BLOCK_NAME(prepare_ordered_)() {
  const int b[6] = {prepare_one(pv_voxelize_kernel<1, false, 1>), prepare_one(pv_voxelize_kernel<1, true, 1>),
                    prepare_one(pv_voxelize_kernel<1, false, 2>), prepare_one(pv_voxelize_kernel<1, true, 2>),
                    prepare_one(pv_voxelize_kernel<kMaxFrames, false, 1>),
                    prepare_one(pv_voxelize_kernel<kMaxFrames, false, 2>)};
  int m = b[0];
  for (int k = 1; k < 6; ++k) m = b[k] < m ? b[k] : m;
  return m;
}

// Launches whose block chunks span more than one 1024-point tile group
// them in tiles of 1024 or 2048 points (U = 2), chosen tile by tile.
int PV_BLOCK_NAME(ordered_smem_)() { return kDynSmem; }

cudaError_t PV_BLOCK_NAME(launch_ordered_)(const cudaLaunchConfig_t& cfg, const KParams& kp, bool queue,
                                           const int64_t* frame_offsets, int frames, long long n) {
  if (!frame_offsets) {
    Frames<1> fr;
    fr.off[0] = 0;
    fr.off[1] = n;
    if (kp.chunk > kThreads)
      return queue ? cudaLaunchKernelEx(&cfg, pv_voxelize_kernel<1, true, 2>, kp, fr)
                   : cudaLaunchKernelEx(&cfg, pv_voxelize_kernel<1, false, 2>, kp, fr);
    return queue ? cudaLaunchKernelEx(&cfg, pv_voxelize_kernel<1, true, 1>, kp, fr)
                 : cudaLaunchKernelEx(&cfg, pv_voxelize_kernel<1, false, 1>, kp, fr);
  }
  Frames<kMaxFrames> fr;  // copied into the launch: the caller's array may go at once
  for (int b = 0; b <= kMaxFrames; ++b) fr.off[b] = b <= frames ? frame_offsets[b] : n;
  if (kp.chunk > kThreads) return cudaLaunchKernelEx(&cfg, pv_voxelize_kernel<kMaxFrames, false, 2>, kp, fr);
  return cudaLaunchKernelEx(&cfg, pv_voxelize_kernel<kMaxFrames, false, 1>, kp, fr);
}

}  // namespace pvk

#if defined(PV_INSTRUMENT) && PV_BLOCK_THREADS == 1024
// Instrumented builds only: the stamps and counters of this file's kernels
// (the 1024-thread build's).
extern "C" {

using namespace pvk;

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

}  // extern "C"
#endif
