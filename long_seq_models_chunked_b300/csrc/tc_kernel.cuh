// Generic warp-specialised tcgen05 tile kernel.
//
// One CTA computes one 128-row output tile into TMEM and hands it to an
// operation-specific epilogue:
//   warp 0 (one lane)  TMA producer: fills a ring of shared-memory stages;
//   warp 1 (one lane)  MMA issuer:   tcgen05.mma per 16-deep K step, then
//                                    tcgen05.commit frees the stage;
//                      (warp 1 also allocates and frees the TMEM columns)
//   warps 2..5         epilogue:     tcgen05.ld of the accumulator rows
//                                    (warp w reads TMEM lanes 32*(w%4)..+31).
// Every wait is bounded by the caller's timeout (%globaltimer); on expiry the
// CTA records TTT_ERR_TIMEOUT in the status word, the other roles stop, TMEM is
// freed and the CTA returns. Nothing traps.
//
// An operation `Op` provides:
//   Params (with a `TcCommon cm` member), Tile,
//   static constexpr int kStages, kStageBytes, kTmemCols;
//   static __device__ bool tile_of(const Params&, Tile&)            (false: no work)
//   static __device__ int  num_kblocks(const Params&, const Tile&)  (>= 1)
//   static __device__ uint32_t stage_tx(const Params&, const Tile&, int kb)  bytes k-block kb loads
//   static __device__ void produce(const Params&, const Tile&, int kb, uint8_t* stage, uint64_t* bar)
//        issues the TMA loads of k-block kb (exactly stage_tx bytes)
//   static __device__ void consume(const Params&, const Tile&, int kb, uint32_t stage_addr, uint32_t tmem)
//   static __device__ void epilogue(const Params&, const Tile&, uint32_t tmem_lane_base, int row,
//                                   float* ep_smem, bool ok)
//        called on every epilogue thread; when !ok (the accumulator never completed)
//        it must skip TMEM and global memory but still pass its named barriers;
//        row = the accumulator row (TMEM lane) this thread owns; warp-uniform control
//        flow is required around tcgen05.ld; ep_smem = 64 floats of scratch shared by
//        the 128 epilogue threads (named barrier 1 synchronises them)
#pragma once

#include "tc_ptx.cuh"
#include "ttt_common.cuh"

namespace ttt {

struct TcCommon {
  int* status;
  unsigned long long timeout_ns;
  int stall;  // failure-detection test: the producer issues no load, so the first wait runs out
};

constexpr int kTcThreads = 192;

// Bounded mbarrier wait. Returns false when it gave up (timeout or another
// role's abort); the first timeout is recorded in the status word.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, const TcCommon& cm,
                                        volatile int* abort_flag) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
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

// Waits, bounded by the timeout alone, for the copy tracked by `bar` to land.
// Used after an abort: a CTA must not exit while a TMA copy into its shared
// memory is still in flight, whatever the abort flag says.
__device__ __forceinline__ void tc_drain(uint64_t* bar, uint32_t parity, const TcCommon& cm) {
  const uint64_t t0 = globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity) && globaltimer_ns() - t0 <= cm.timeout_ns) {
  }
}

template <class Op>
__host__ __device__ constexpr size_t tc_smem_bytes() {
  return (size_t)Op::kStages * Op::kStageBytes + 1024 + 512;
}

template <class Op>
__global__ void __launch_bounds__(kTcThreads, 1) tc_kernel(const __grid_constant__ typename Op::Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)Op::kStages * Op::kStageBytes);
  uint64_t* empty = full + Op::kStages;
  uint64_t* accb = empty + Op::kStages;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(accb + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  float* ep_smem = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 256);  // 64 floats

  typename Op::Tile tile;
  if (!Op::tile_of(p, tile)) return;  // uniform over the CTA

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Op::kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(accb, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tslot, Op::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tslot;
  const int nkb = Op::num_kblocks(p, tile);

  if (warp == 0) {
    if (lane == 0 && !p.cm.stall) {
      int issued = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % Op::kStages;
        const uint32_t round = (uint32_t)(kb / Op::kStages);
        if (!tc_wait(&empty[s], (round & 1u) ^ 1u, p.cm, abort_flag)) break;
        uint8_t* st = smem + (size_t)s * Op::kStageBytes;
        // expect-tx is armed with the byte count the op will issue for this k-block
        ptx::mbar_expect_tx(&full[s], Op::stage_tx(p, tile, kb));
        Op::produce(p, tile, kb, st, &full[s]);
        issued = kb + 1;
      }
      if (*abort_flag) {
        // drain the copies this thread started before the CTA returns
        for (int kb = issued - Op::kStages > 0 ? issued - Op::kStages : 0; kb < issued; ++kb)
          tc_drain(&full[kb % Op::kStages], (uint32_t)(kb / Op::kStages) & 1u, p.cm);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % Op::kStages;
        const uint32_t round = (uint32_t)(kb / Op::kStages);
        if (!tc_wait(&full[s], round & 1u, p.cm, abort_flag)) break;
        ptx::tc_fence_after();
        Op::consume(p, tile, kb, ptx::smem_u32(smem + (size_t)s * Op::kStageBytes), tmem);
        ptx::mma_commit(&empty[s]);
      }
      ptx::mma_commit(accb);
      // after an abort nobody waits for the accumulator: the MMAs already issued
      // must finish before TMEM is freed
      if (*abort_flag) tc_drain(accb, 0, p.cm);
    }
  } else {
    const int g = warp & 3;  // TMEM lane group this warp may access
    int ok = 0;
    if (lane == 0) ok = tc_wait(accb, 0, p.cm, abort_flag) && !*abort_flag;
    ok = __shfl_sync(0xffffffffu, ok, 0);  // warp-uniform: tcgen05.ld is .sync.aligned
    ptx::tc_fence_after();
    // always called (so named barriers inside stay matched); `ok` is warp-uniform
    Op::epilogue(p, tile, tmem + ((uint32_t)(32 * g) << 16), 32 * g + lane, ep_smem, ok != 0);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, Op::kTmemCols);
}

}  // namespace ttt
