// Cluster-multicast forms of the operand- and signal-sharing primitives
// (sm_103a). Compiled only into the single-GPU build of the library: the
// multicast loads read this GPU's own memory into every CTA of a cluster.
#pragma once

#include <stdint.h>

#define TTT_HAS_MULTICAST 1

namespace ttt {
namespace ptx {

// TMA tile load delivered to the same shared-memory offset of every CTA in
// `cta_mask` (this cluster); each destination's mbarrier at `bar`'s offset
// receives the bytes that land in that CTA.
__device__ __forceinline__ void tma_load_3d_shared(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1,
                                               int c2, uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "h"(cta_mask)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d_shared(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1,
                                               int c2, int c3, uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)), "h"(cta_mask)
      : "memory");
}

// Arrives on the mbarrier at `bar`'s offset in every CTA of `cta_mask` once
// every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void mma_commit_shared(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Arrives on the mbarrier at `bar`'s offset in every CTA of `cta_mask` once the
// pair MMAs issued so far by this thread are done.
__device__ __forceinline__ void mma2_commit_mc(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

}  // namespace ptx
}  // namespace ttt
