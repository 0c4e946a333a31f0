// Shared device/host helpers of the TTT-layer kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/ttt.h"

namespace ttt {

constexpr size_t kStatusBytes = 256;   // header of every workspace
constexpr int kMaxMaskChunks = 4096;   // update mask passed by value as a bitset

struct MaskBits {
  uint32_t w[kMaxMaskChunks / 32];
};

__host__ __device__ inline bool mask_bit(const MaskBits& m, int c) {
  return (m.w[c >> 5] >> (c & 31)) & 1u;
}

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Records the first device-side error in the status word (later ones are dropped).
__device__ inline void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Storage-type loads and stores (bf16 <-> fp32 conversions are exact / RNE).
__device__ inline float ld_val(const void* p, size_t i, int dtype) {
  if (dtype == TTT_DTYPE_F32) return static_cast<const float*>(p)[i];
  return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

__device__ inline void st_val(void* p, size_t i, int dtype, float v) {
  if (dtype == TTT_DTYPE_F32)
    static_cast<float*>(p)[i] = v;
  else
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
}

__device__ inline float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

// The same through the fast intrinsics (a few ulp of fp32; for the bf16
// tensor-core epilogues, whose operands round to 2^-9). For x < -88 the
// exponential overflows to +inf and the quotient is 0, the limit.
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// Nanosecond clock shared by all SMs (for bounded waits).
__device__ inline uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

}  // namespace ttt
