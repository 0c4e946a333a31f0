// Helpers shared by the tensor-core kernels: operand packing and stores,
// shared-memory descriptors of the 128-byte-swizzled tiles, and the host-side
// TMA tensor-map construction.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_ptx.cuh"

namespace ttt {
namespace tcu {

using bf16 = __nv_bfloat16;
using f16 = __half;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr uint32_t kABytes = BM * BK * 2;   // K-major A tile, or two MN-major boxes
constexpr uint32_t kBox = 64 * BK * 2;      // one 64 x 64 bf16 box (MN-major)

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void st_bf16x32(bf16* dst, const float* v) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
    d[q] = w;
  }
}

__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Two values as a bf16 pair (hi = bf16(x), rounded to nearest) and the pair of
// their remainders (lo = bf16(x - hi)); hi is read back from its packed bits.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& h, uint32_t& l) {
  h = pack_bf16(a, b);
  l = pack_bf16(a - __uint_as_float(h << 16), b - __uint_as_float(h & 0xffff0000u));
}

__device__ __forceinline__ void st_bf16pair32(bf16* hi, bf16* lo, const float* v) {
  uint4* dh = reinterpret_cast<uint4*>(hi);
  uint4* dl = reinterpret_cast<uint4*>(lo);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 h, l;
    split_bf16x2(v[8 * q + 0], v[8 * q + 1], h.x, l.x);
    split_bf16x2(v[8 * q + 2], v[8 * q + 3], h.y, l.y);
    split_bf16x2(v[8 * q + 4], v[8 * q + 5], h.z, l.z);
    split_bf16x2(v[8 * q + 6], v[8 * q + 7], h.w, l.w);
    dh[q] = h;
    dl[q] = l;
  }
}

__device__ __forceinline__ void st_f32x32(float* dst, const float* v) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < 8; ++q) d[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// Row `lane` of a 32 x 32 block of 2-byte elements staged for a TMA store in
// the 64-byte swizzle: 16-byte chunk q of row r at 64 r + 16 (q ^ ((r >> 1) & 3)),
// so a warp's 16-byte writes are bank-conflict free. 2 KB per block.
__device__ __forceinline__ uint32_t stage_off64(int lane, int q) { return 64u * lane + 16u * (q ^ ((lane >> 1) & 3)); }

__device__ __forceinline__ float bf_rest(float x) { return x - __bfloat162float(__float2bfloat16_rn(x)); }

// bf16 (hi) at buf; with `lo`, bf16(x - hi) at buf + 2048
template <bool LO>
__device__ __forceinline__ void stage_bf16x32(uint8_t* buf, int lane, const float* v) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 h, l;
    if (LO) {
      split_bf16x2(v[8 * q + 0], v[8 * q + 1], h.x, l.x);
      split_bf16x2(v[8 * q + 2], v[8 * q + 3], h.y, l.y);
      split_bf16x2(v[8 * q + 4], v[8 * q + 5], h.z, l.z);
      split_bf16x2(v[8 * q + 6], v[8 * q + 7], h.w, l.w);
      *reinterpret_cast<uint4*>(buf + 2048 + stage_off64(lane, q)) = l;
    } else {
      h.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
      h.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
      h.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
      h.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
    }
    *reinterpret_cast<uint4*>(buf + stage_off64(lane, q)) = h;
  }
}

// One operand: a bf16 (hi, lo) pair (SPLIT) or fp16.
template <bool SPLIT>
__device__ __forceinline__ void stage_op32(uint8_t* buf, int lane, const float* v) {
  if (SPLIT) {
    stage_bf16x32<true>(buf, lane, v);
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 h;
      h.x = pack_f16(v[8 * q + 0], v[8 * q + 1]);
      h.y = pack_f16(v[8 * q + 2], v[8 * q + 3]);
      h.z = pack_f16(v[8 * q + 4], v[8 * q + 5]);
      h.w = pack_f16(v[8 * q + 6], v[8 * q + 7]);
      *reinterpret_cast<uint4*>(buf + stage_off64(lane, q)) = h;
    }
  }
}

// K-major operand descriptor for K step kk of a 64-deep stage.
__device__ __forceinline__ uint64_t kdesc(uint32_t base, int kk) { return ptx::sdesc(base + kk * 32, 16, 1024); }
// MN-major operand descriptor (64-wide groups kBox apart) for K step kk.
__device__ __forceinline__ uint64_t mdesc(uint32_t base, int kk) { return ptx::sdesc(base + kk * 2048, kBox, 1024); }

__device__ __forceinline__ void st_shadow(bf16* hi, bf16* lo, size_t o, float v) {
  const bf16 h = __float2bfloat16_rn(v);
  hi[o] = h;
  if (lo) lo[o] = __float2bfloat16_rn(v - __bfloat162float(h));
}

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Tensor map over a row-major array with dims (innermost first) and box; the
// elements are 4 bytes for FLOAT32, else 2.
inline bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint32_t* box,
              CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn || !base) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  uint64_t stride = dt == CU_TENSOR_MAP_DATA_TYPE_FLOAT32 ? 4 : 2;
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i > 0) gs[i - 1] = stride;
    stride *= dims[i];
  }
  const CUresult r = fn(m, dt, rank, const_cast<void*>(base), gd, gs, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

inline bool map3(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1,
          CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
          CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint32_t box[3] = {b0, b1, 1};
  return make_map(m, base, 3, dims, box, dt, swz);
}

}  // namespace tcu
}  // namespace ttt
