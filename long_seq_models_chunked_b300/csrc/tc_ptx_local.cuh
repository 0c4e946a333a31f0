// CTA-local forms of the operand- and signal-sharing primitives, for the build
// of the library that processes running on several GPUs load: no cluster
// multicast anywhere. Each form is exact for a cluster of one CTA (cta_mask ==
// 1, the CTA itself), which is the only cluster size the engines use in this
// build; CTA pairs (cta_group::2) are not built.
#pragma once

#include <stdint.h>

#define TTT_HAS_MULTICAST 0

namespace ttt {
namespace ptx {

// The tile, loaded into this CTA only.
__device__ __forceinline__ void tma_load_3d_shared(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1,
                                                   int c2, uint16_t /*cta_mask == 1*/) {
  tma_load_3d(dst, m, bar, c0, c1, c2);
}

__device__ __forceinline__ void tma_load_4d_shared(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1,
                                                   int c2, int c3, uint16_t /*cta_mask == 1*/) {
  tma_load_4d(dst, m, bar, c0, c1, c2, c3);
}

// Arrival on this CTA's barrier once this thread's tcgen05 operations are done.
__device__ __forceinline__ void mma_commit_shared(uint64_t* bar, uint16_t /*cta_mask == 1*/) { mma_commit(bar); }

}  // namespace ptx
}  // namespace ttt
