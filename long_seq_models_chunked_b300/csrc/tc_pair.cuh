// Persistent warp-specialised tcgen05 engine on CTA pairs (cta_group::2).
//
// A work item is one 256-row tile computed by the two CTAs of a two-CTA
// cluster. CTA `prank` (0 or 1) of the pair loads its own 128 rows of A and
// its half of B's columns into its own shared memory, at the same stage
// offsets as its peer. The even CTA (the lead) counts both CTAs' bytes on its
// `full` barrier (TMA loads of the .cta_group::2 form signal the lead's
// barrier), issues the M = 256 MMAs over both CTAs' shared memory and commits
// to both CTAs' `empty` and accumulator barriers. Each CTA's epilogue reads its
// own 128 TMEM lanes (all N columns) and returns the accumulator with a
// cluster-scope arrival on the lead's `acce` barrier. Two accumulators
// alternate, so the epilogue of one tile overlaps the MMAs of the next.
//
// Per CTA, B takes half the shared memory and half the operand ingress of a
// one-CTA tile of the same N, and each MMA instruction carries twice the work:
// an N = 256 pair MMA keeps each SM's tensor pipe busy for 128 cycles, enough
// for the one issuing thread to also wait on the next stage without leaving
// the pipe idle.
//
//   warp 0 (one lane)  TMA producer;  warp 1 (one lane of the lead)  MMA issuer
//   (warp 1 of both CTAs allocates TMEM);  warps 2..5  epilogue.
//
// Every wait is bounded by the caller's timeout; after an abort each role
// stops, the lead's producer waits (bounded) for the copies counted on its
// barriers, the peer's gives its own copies a bounded time to land, the lead's
// MMA warp waits for its MMAs, the pair meets at a final cluster barrier, TMEM
// is freed and both CTAs return. Nothing traps.
//
// The pair MMA's commits arrive on both CTAs' barriers through the multicast
// form of tcgen05.commit, so the engine exists only in the single-GPU build.
//
// An operation `Op` provides:
//   Params (with a `TcCommon cm` member), Tile;
//   static constexpr int kStages, kStageBytes, kAccCols (<= 256);
//   static constexpr uint32_t kEpiBytes   (a multiple of 4 KB per epilogue warp, or 0)
//   static __device__ int  num_work(const Params&);
//   static __device__ void tile_of(const Params&, int item, int prank, Tile&);
//   static __device__ int  num_kblocks(const Params&, const Tile&)   (the same for both CTAs)
//   static __device__ uint32_t stage_tx(const Params&, const Tile&, int kb)  bytes ONE CTA loads
//                                                                            (the same for both)
//   static __device__ void produce(const Params&, const Tile&, int kb, uint8_t* stage,
//                                  uint32_t full_lead, int prank)
//        issues this CTA's loads of k-block kb, completing on the lead's barrier
//        at cluster address `full_lead`
//   static __device__ void consume(const Params&, const Tile&, int kb, uint32_t stage_addr, uint32_t tmem)
//        pair MMAs of k-block kb (lead only)
//   struct Pre; static __device__ Pre pre(const Params&, const Tile&, int row)
//   static __device__ void epilogue(const Params&, const Tile&, uint32_t tmem_lane_base, int row,
//                                   uint8_t* epi, uint32_t& es, const Pre&)
//        warp-uniform control flow around tcgen05.ld is required
#pragma once

#include "tc_kernel.cuh"

#if TTT_HAS_MULTICAST

namespace ttt {

template <class Op>
__host__ __device__ constexpr size_t tc_pair_smem_bytes() {
  return (size_t)Op::kStages * Op::kStageBytes + Op::kEpiBytes + 1024 + 256;
}

// Bounded wait with cluster-scope acquire, for barriers that the other CTA of
// the pair arrives on.
__device__ __forceinline__ bool tc_wait_cluster(uint64_t* bar, uint32_t parity, const TcCommon& cm,
                                                volatile int* abort_flag) {
  if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (true) {
    if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    if ((++it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > cm.timeout_ns) {
        *abort_flag = 1;
        set_status(cm.status, TTT_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

template <class Op>
__global__ void __launch_bounds__(kTcThreads, 1) tc_pair_kernel(const __grid_constant__ typename Op::Params p) {
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
  const uint32_t crank = ptx::cluster_ctarank();
  const int prank = (int)(crank & 1u);
  const uint32_t lead = crank & ~1u;
  const uint16_t pair_mask = (uint16_t)(3u << lead);
  const int pair = (int)(blockIdx.x >> 1), n_pairs = (int)(gridDim.x >> 1);
  const int n_work = Op::num_work(p);

  if (threadIdx.x == 0) {
    for (int s = 0; s < Op::kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&accf[s], 1);
      ptx::mbar_init(&acce[s], 8);  // four epilogue warps in each CTA of the pair
    }
    ptx::mbar_init(drainb, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc2(tslot, 2 * Op::kAccCols);
    ptx::tmem_relinquish2();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  ptx::cluster_sync();  // both CTAs' barriers exist before either signals the other
  const uint32_t tmem = *tslot;
  const uint32_t full_lead = ptx::mapa(ptx::smem_u32(full), lead);
  const uint32_t acce_lead = ptx::mapa(ptx::smem_u32(acce), lead);

  if (warp == 0) {
    if (lane == 0 && !p.cm.stall) {
      uint32_t pc = 0;
      for (int w = pair; w < n_work && !*abort_flag; w += n_pairs) {
        typename Op::Tile t;
        Op::tile_of(p, w, prank, t);
        const int nkb = Op::num_kblocks(p, t);
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = pc % Op::kStages;
          if (!tc_wait(&empty[s], ((pc / Op::kStages) & 1u) ^ 1u, p.cm, abort_flag)) break;
          if (prank == 0) ptx::mbar_expect_tx(&full[s], 2u * Op::stage_tx(p, t, kb));
          Op::produce(p, t, kb, smem + (size_t)s * Op::kStageBytes, full_lead + 8u * (uint32_t)s, prank);
          ++pc;
        }
      }
      if (*abort_flag) {
        if (prank == 0) {
          for (uint32_t k = pc > (uint32_t)Op::kStages ? pc - Op::kStages : 0; k < pc; ++k)
            tc_drain(&full[k % Op::kStages], (k / Op::kStages) & 1u, p.cm);
        } else {
          // the peer cannot wait on the lead's barriers: give its own copies a
          // bounded time to land before the CTA can leave
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 200000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && prank == 0) {
      uint32_t mc = 0, at = 0;
      for (int w = pair; w < n_work && !*abort_flag; w += n_pairs) {
        typename Op::Tile t;
        Op::tile_of(p, w, 0, t);
        const int nkb = Op::num_kblocks(p, t);
        const uint32_t acc = at & 1u;
        if (!tc_wait_cluster(&acce[acc], ((at >> 1) & 1u) ^ 1u, p.cm, abort_flag)) break;
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
          ptx::mma2_commit_mc(&empty[s], pair_mask);
          ++mc;
        }
        if (!ok) break;
        ptx::mma2_commit_mc(&accf[acc], pair_mask);
        ++at;
      }
      if (*abort_flag) {
        ptx::mma2_commit_mc(drainb, (uint16_t)(1u << lead));
        tc_drain(drainb, 0, p.cm);
      }
    }
  } else {
    const int g = warp & 3;
    uint32_t et = 0, es = 0;
    uint8_t* epi_w = epi + (size_t)g * (Op::kEpiBytes / 4);
    for (int w = pair; w < n_work; w += n_pairs) {
      if (*abort_flag) break;
      typename Op::Tile t;
      Op::tile_of(p, w, prank, t);
      const uint32_t acc = et & 1u;
      const typename Op::Pre pre = Op::pre(p, t, 32 * g + lane);
      int ok = 0;
      if (lane == 0) ok = tc_wait(&accf[acc], (et >> 1) & 1u, p.cm, abort_flag) && !*abort_flag;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ptx::tc_fence_after();
      Op::epilogue(p, t, tmem + acc * Op::kAccCols + ((uint32_t)(32 * g) << 16), 32 * g + lane, epi_w, es, pre);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(acce_lead + 8u * acc);
      ++et;
    }
    if (Op::kEpiBytes && lane == 0) ptx::bulk_wait_all();  // the epilogue's TMA stores are done
    __syncwarp();
  }
  ptx::tc_fence_before();
  __syncwarp();
  __syncthreads();
  // no CTA leaves while its peer can still signal it or read its shared memory
  ptx::cluster_sync();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc2(tmem, 2 * Op::kAccCols);
}

}  // namespace ttt

#endif  // TTT_HAS_MULTICAST
