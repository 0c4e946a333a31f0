// Persistent warp-specialised tcgen05 engine for thread-block clusters whose
// CTAs share an operand through TMA multicast.
//
// A work item is one cluster-wide unit (for example the d/128 row tiles of one
// output column block); CTA `rank` of the cluster computes tile (item, rank).
// Every stage of the shared-memory ring is filled by this CTA's own loads plus
// one slice of the shared operand from each CTA of the cluster, multicast to
// all of them, so the shared operand is read from L2 once per cluster instead
// of once per CTA. A stage is refilled only after every CTA of the cluster has
// consumed it: each MMA warp commits to the `empty` barrier of every CTA
// (arrival count = cluster size). Two TMEM accumulators alternate between
// tiles, so the epilogue of one tile overlaps the MMAs of the next.
//
//   warp 0 (one lane)  TMA producer;  warp 1 (one lane)  MMA issuer (and TMEM
//   allocation);  warps 2..(1 + kEpiWarps)  epilogue (warp w reads TMEM lanes
//   32*(w%4)..+31; with eight epilogue warps, two per lane quarter, each takes
//   one half of the tile's columns).
//
// Every wait is bounded by the caller's timeout; after an abort each role
// stops, the producer waits (bounded) for its own copies, the MMA warp for its
// own MMAs, the cluster meets at a final barrier, TMEM is freed and the CTA
// returns. Nothing traps.
//
// An operation `Op` provides:
//   Params (with a `TcCommon cm` member), Tile;
//   static constexpr int kStages, kStageBytes, kAccCols (<= 256), kEpiWarps (4 or 8);
//   static __device__ int  num_work(const Params&);
//   static __device__ void tile_of(const Params&, int item, int rank, Tile&);
//   static __device__ int  num_kblocks(const Params&, const Tile&)   (same for every rank of an item)
//   static __device__ uint32_t stage_tx(const Params&, const Tile&, int kb)  bytes landing in THIS CTA
//   static __device__ void produce(const Params&, const Tile&, int kb, uint8_t* stage, uint64_t* bar,
//                                  int rank, int cs, uint16_t mask)
//        issues this CTA's own loads and its multicast slice (mask = every CTA)
//   static __device__ void consume(const Params&, const Tile&, int kb, uint32_t stage_addr, uint32_t tmem)
//   static constexpr uint32_t kEpiBytes   shared memory for the epilogue (a multiple of 4 KB
//                                         per epilogue warp, or 0)
//   struct Pre; static __device__ Pre pre(const Params&, const Tile&, int row)
//        values the epilogue needs from global memory, loaded before the
//        accumulator wait (so their latency hides under the tile's MMAs)
//   static __device__ void epilogue(const Params&, const Tile&, uint32_t tmem_lane_base, int row,
//                                   uint8_t* epi, uint32_t& es, const Pre&, int half)
//        warp-uniform control flow around tcgen05.ld is required; half = which half
//        of the columns this warp takes (always 0 with four epilogue warps); epi =
//        this warp's kEpiBytes / kEpiWarps of staging, es = a per-warp counter the epilogue may use for
//        its buffers; TMA stores it issues (lane 0, bulk groups) complete before
//        the CTA exits
#pragma once

#include "tc_kernel.cuh"

namespace ttt {

template <class Op>
__host__ __device__ constexpr size_t tc_mc_smem_bytes() {
  return (size_t)Op::kStages * Op::kStageBytes + Op::kEpiBytes + 1024 + 256;
}

template <class Op>
__host__ __device__ constexpr int tc_mc_threads() {
  return 64 + 32 * Op::kEpiWarps;
}

template <class Op>
__global__ void __launch_bounds__(tc_mc_threads<Op>(), 1) tc_mc_kernel(const __grid_constant__ typename Op::Params p) {
  static_assert(Op::kEpiWarps == 4 || Op::kEpiWarps == 8, "four or eight epilogue warps");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* epi = smem + (size_t)Op::kStages * Op::kStageBytes;  // epilogue staging (kEpiBytes)
  uint64_t* full = reinterpret_cast<uint64_t*>(epi + Op::kEpiBytes);
  uint64_t* empty = full + Op::kStages;
  uint64_t* accf = empty + Op::kStages;
  uint64_t* acce = accf + 2;
  uint64_t* drainb = acce + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drainb + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cs = (int)ptx::cluster_nctarank();
  const int rank = (int)ptx::cluster_ctarank();
  const int cluster = (int)(blockIdx.x / (unsigned)cs);
  const int n_clusters = (int)(gridDim.x / (unsigned)cs);
  const uint16_t mask = (uint16_t)((1u << cs) - 1u);
  const int n_work = Op::num_work(p);
#if !TTT_HAS_MULTICAST
  // this build shares nothing across CTAs: only clusters of one CTA are valid
  if (cs != 1) {
    if (threadIdx.x == 0) set_status(p.cm.status, TTT_ERR_DEVICE);
    return;
  }
#endif

  if (threadIdx.x == 0) {
    for (int s = 0; s < Op::kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], (uint32_t)cs);  // one MMA commit per CTA of the cluster
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&accf[s], 1);
      ptx::mbar_init(&acce[s], Op::kEpiWarps);  // one arrival per epilogue warp
    }
    ptx::mbar_init(drainb, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tslot, 2 * Op::kAccCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // peers multicast into this CTA's ring and arrive on its barriers: every CTA
  // of the cluster must have initialised them first
  ptx::cluster_sync();
  const uint32_t tmem = *tslot;

  uint32_t pc = 0;  // producer: stages filled
  if (warp == 0) {
    if (lane == 0 && !p.cm.stall) {
      for (int w = cluster; w < n_work && !*abort_flag; w += n_clusters) {
        typename Op::Tile t;
        Op::tile_of(p, w, rank, t);
        const int nkb = Op::num_kblocks(p, t);
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = pc % Op::kStages;
          if (!tc_wait(&empty[s], ((pc / Op::kStages) & 1u) ^ 1u, p.cm, abort_flag)) break;
          uint8_t* st = smem + (size_t)s * Op::kStageBytes;
          ptx::mbar_expect_tx(&full[s], Op::stage_tx(p, t, kb));
          Op::produce(p, t, kb, st, &full[s], rank, cs, mask);
          ++pc;
        }
      }
      if (*abort_flag)
        for (uint32_t k = pc > (uint32_t)Op::kStages ? pc - Op::kStages : 0; k < pc; ++k)
          tc_drain(&full[k % Op::kStages], (k / Op::kStages) & 1u, p.cm);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t mc = 0, at = 0;
      for (int w = cluster; w < n_work && !*abort_flag; w += n_clusters) {
        typename Op::Tile t;
        Op::tile_of(p, w, rank, t);
        const int nkb = Op::num_kblocks(p, t);
        const uint32_t acc = at & 1u;
        if (!tc_wait(&acce[acc], ((at >> 1) & 1u) ^ 1u, p.cm, abort_flag)) break;
        ptx::tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = mc % Op::kStages;
          if (!tc_wait(&full[s], (mc / Op::kStages) & 1u, p.cm, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          Op::consume(p, t, kb, ptx::smem_u32(smem + (size_t)s * Op::kStageBytes), tmem + acc * Op::kAccCols);
          ptx::mma_commit_shared(&empty[s], mask);
          ++mc;
        }
        if (!ok) break;
        ptx::mma_commit(&accf[acc]);
        ++at;
      }
      if (*abort_flag) {
        ptx::mma_commit(drainb);
        tc_drain(drainb, 0, p.cm);
      }
    }
  } else {
    const int g = warp & 3;
    const int half = (warp - 2) >> 2;
    uint32_t et = 0, es = 0;
    uint8_t* epi_w = epi + (size_t)(warp - 2) * (Op::kEpiBytes / Op::kEpiWarps);
    for (int w = cluster; w < n_work; w += n_clusters) {
      if (*abort_flag) break;
      typename Op::Tile t;
      Op::tile_of(p, w, rank, t);
      const uint32_t acc = et & 1u;
      // global loads the epilogue needs, issued while the tile's MMAs run
      const typename Op::Pre pre = Op::pre(p, t, 32 * g + lane);
      int ok = 0;
      if (lane == 0) ok = tc_wait(&accf[acc], (et >> 1) & 1u, p.cm, abort_flag) && !*abort_flag;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ptx::tc_fence_after();
      Op::epilogue(p, t, tmem + acc * Op::kAccCols + ((uint32_t)(32 * g) << 16), 32 * g + lane, epi_w, es, pre,
                   half);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&acce[acc]);
      ++et;
    }
    if (Op::kEpiBytes && lane == 0) ptx::bulk_wait_all();  // the epilogue's TMA stores are done
    __syncwarp();
  }
  ptx::tc_fence_before();
  __syncwarp();
  __syncthreads();
  // no CTA may leave while a peer can still multicast into it or arrive on it
  ptx::cluster_sync();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, 2 * Op::kAccCols);
}

}  // namespace ttt
