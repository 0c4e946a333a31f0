// bf16 tensor-core path of the chunked TTT layer (SwiGLU fast net, inner-product
// loss): every dense contraction runs on tcgen05 MMAs with TMEM accumulators fed
// by TMA; fp32 master weights, fp32 accumulation, bf16 operands.
//
// Per chunk (LaCT page §2.1; shifted order of §3.2, update-then-apply of §3.1,
// update mask of §3.3), batched over every (batch, head):
//   fwd     [A|B] = X [W1;W3]^T for X = Q_c and K_c rows, Dm = V_c W2 (K rows);
//           epilogue: H_q = silu(A)*B for queries; for keys the SwiGLU backward
//           DA = Dm'*B*silu'(A), DB = Dm'*silu(A), He = -lr*H with Dm' = -lr*Dm
//   apply   O_c = H_q W2^T
//   grad    G1^T = K^T DA, G2 = V^T He, G3^T = K^T DB   (sums over the chunk's tokens)
//   muon    X0 = G/||G||_F; 5 x { S = X X^T; P = bS + cS^2; X = aX + P X }
//           (LaCT page §2.2.1, eq. 9-10, on the wide orientation d x dh)
//   update  W <- W - step*U, then every row of W1, W2, W3 rescaled to its W0 norm
//           (LaCT page §2.2.1, eq. 8)
// The fast weights are kept transposed where that makes every update elementwise:
// M1 = W1^T, M2 = W2, M3 = W3^T, all [d, dh] fp32 plus a bf16 shadow that the
// GEMMs read (K-major or MN-major as each product needs).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

#include "../../include/ttt_debug.h"
#include "tc_kernel.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

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

__device__ __forceinline__ void st_f16x32(f16* dst, const float* v) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_f16(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_f16(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_f16(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_f16(v[8 * q + 6], v[8 * q + 7]);
    d[q] = w;
  }
}

// Stores 32 values as one fp16 operand (SINGLE) or as a bf16 hi/lo pair (SPLIT):
// hi = bf16(v), lo = bf16(v - hi), so hi + lo carries ~16 significant bits.
template <bool SPLIT>
__device__ __forceinline__ void st_op32(void* hi, void* lo, size_t o, const float* v) {
  if (SPLIT) {
    float l[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) l[i] = v[i] - __bfloat162float(__float2bfloat16_rn(v[i]));
    st_bf16x32(static_cast<bf16*>(hi) + o, v);
    st_bf16x32(static_cast<bf16*>(lo) + o, l);
  } else {
    st_f16x32(static_cast<f16*>(hi) + o, v);
  }
}

__device__ __forceinline__ void st_bf16pair32(bf16* hi, bf16* lo, const float* v) {
  float l[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) l[i] = v[i] - __bfloat162float(__float2bfloat16_rn(v[i]));
  st_bf16x32(hi, v);
  st_bf16x32(lo, l);
}

__device__ __forceinline__ void st_f32x32(float* dst, const float* v) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < 8; ++q) d[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

__device__ __forceinline__ void ld_f32x32(const float* src, float* v) {
  const float4* s = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 x = s[q];
    v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
  }
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// K-major operand descriptor for K step kk of a 64-deep stage.
__device__ __forceinline__ uint64_t kdesc(uint32_t base, int kk) { return ptx::sdesc(base + kk * 32, 16, 1024); }
// MN-major operand descriptor (64-wide groups kBox apart) for K step kk.
__device__ __forceinline__ uint64_t mdesc(uint32_t base, int kk) { return ptx::sdesc(base + kk * 2048, kBox, 1024); }

// ============================================================ fwd (apply-1 + update forward)
struct FwdOp {
  struct Params {
    CUtensorMap mQ, mK, mV;  // 3D {d, T, BH}, box {64, 128, 1}
    CUtensorMap mW;          // bf16 shadows [3BH][d][dh] as 3D {dh, d, 3BH}, box {64, 64, 1}
    CUtensorMap mWl;         // low halves of the shadows (split precision)
    const float* lr;
    bf16* Hq;                // [BH][Cp][dh]
    bf16* E;                 // [BH][3][Cp][dh]: DA, He, DB
    bf16* El;                // low halves of E (split precision)
    int d, dh, T, Cp, chunk_start, valid, q_tiles, k_tiles, n_tiles, split;
    TcCommon cm;
  };
  struct Tile {
    int bh, row0, j0;
    bool is_k;
  };
  static constexpr int kStages = 4;
  static constexpr int kStageBytes = kABytes + 4 * kBox;
  static constexpr int kTmemCols = 512;

  static __device__ bool tile_of(const Params& p, Tile& t) {
    const int nt = blockIdx.x % p.n_tiles, rt = blockIdx.x / p.n_tiles;
    if (rt >= p.q_tiles + p.k_tiles) return false;
    t.is_k = rt >= p.q_tiles;
    t.row0 = (t.is_k ? rt - p.q_tiles : rt) * BM;
    t.j0 = nt * 128;
    t.bh = blockIdx.y;
    return true;
  }
  // k-blocks: segment 0 ([A|B], the weights' hi then, when split, lo halves),
  // then for key tiles segment 1 (Dm, same order). The keys/values are exact bf16,
  // so W = hi + lo needs two products, not three.
  static __device__ int seg0_blocks(const Params& p, const Tile& t) {
    return (t.is_k && p.split ? 2 : 1) * (p.d / BK);
  }
  static __device__ int num_kblocks(const Params& p, const Tile& t) {
    return t.is_k ? 2 * seg0_blocks(p, t) : seg0_blocks(p, t);
  }
  static __device__ uint32_t stage_tx(const Params& p, const Tile& t, int kb) {
    return kb < seg0_blocks(p, t) ? kABytes + 4 * kBox : kABytes + 2 * kBox;
  }
  static __device__ void produce(const Params& p, const Tile& t, int kb, uint8_t* st, uint64_t* bar) {
    const int nk = p.d / BK;
    const int n0 = seg0_blocks(p, t);
    const int z = t.bh * 3;
    if (kb < n0) {
      const int k = kb % nk;
      const CUtensorMap* w = kb >= nk ? &p.mWl : &p.mW;
      ptx::tma_load_3d(st, t.is_k ? &p.mK : &p.mQ, bar, k * BK, p.chunk_start + t.row0, t.bh);
      for (int g = 0; g < 2; ++g) {
        ptx::tma_load_3d(st + kABytes + g * kBox, w, bar, t.j0 + g * 64, k * BK, z + 0);
        ptx::tma_load_3d(st + kABytes + (2 + g) * kBox, w, bar, t.j0 + g * 64, k * BK, z + 2);
      }
    } else {
      const int k2 = kb - n0, k = k2 % nk;
      const CUtensorMap* w = k2 >= nk ? &p.mWl : &p.mW;
      ptx::tma_load_3d(st, &p.mV, bar, k * BK, p.chunk_start + t.row0, t.bh);
      for (int g = 0; g < 2; ++g)
        ptx::tma_load_3d(st + kABytes + g * kBox, w, bar, t.j0 + g * 64, k * BK, z + 1);
    }
  }
  static __device__ void consume(const Params& p, const Tile& t, int kb, uint32_t st, uint32_t tmem) {
    const int n0 = seg0_blocks(p, t);
    const uint32_t a = st, b = st + kABytes;
    if (kb < n0) {
      constexpr uint32_t id = ptx::idesc_bf16(128, 256, false, true);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) ptx::mma_bf16(tmem, kdesc(a, kk), mdesc(b, kk), id, (kb | kk) != 0);
    } else {
      const int k2 = kb - n0;
      constexpr uint32_t id = ptx::idesc_bf16(128, 128, false, true);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) ptx::mma_bf16(tmem + 256, kdesc(a, kk), mdesc(b, kk), id, (k2 | kk) != 0);
    }
  }
  static __device__ void epilogue(const Params& p, const Tile& t, uint32_t tm, int r, float*, bool ok) {
    if (!ok) return;
    const int tl = t.row0 + r;  // token index inside the chunk
    const bool valid = tl < p.valid;
    float va[32], vb[32];
    if (!t.is_k) {
      bf16* dst = p.Hq + ((size_t)t.bh * p.Cp + tl) * p.dh + t.j0;
      for (int c = 0; c < 128; c += 32) {
        ptx::tmem_ld32(tm + c, va);
        ptx::tmem_ld32(tm + 128 + c, vb);
#pragma unroll
        for (int i = 0; i < 32; ++i) va[i] = va[i] * sigmoidf_(va[i]) * vb[i];
        if (valid) st_bf16x32(dst + c, va);
      }
    } else {
      const float eta = valid ? p.lr[(size_t)t.bh * p.T + p.chunk_start + tl] : 0.f;
      const size_t plane = (size_t)p.Cp * p.dh;
      const size_t oA = ((size_t)t.bh * 3 * p.Cp + tl) * p.dh + t.j0;
      bf16* dA = p.E + oA;
      bf16* dH = dA + plane;
      bf16* dB = dA + 2 * plane;
      float vd[32];
      for (int c = 0; c < 128; c += 32) {
        ptx::tmem_ld32(tm + c, va);
        ptx::tmem_ld32(tm + 128 + c, vb);
        ptx::tmem_ld32(tm + 256 + c, vd);
        float oh[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float a = va[i], b = vb[i];
          const float g = -eta * vd[i];         // dl/dh = W2^T (-lr v)
          const float sg = sigmoidf_(a);
          const float s = a * sg;
          oh[i] = -eta * s * b;                 // -lr * h  (G2 = V^T He)
          va[i] = g * b * sg * (1.f + a * (1.f - sg));
          vb[i] = g * s;
        }
        if (p.split) {
          st_bf16pair32(dA + c, p.El + oA + c, va);
          st_bf16pair32(dH + c, p.El + oA + plane + c, oh);
          st_bf16pair32(dB + c, p.El + oA + 2 * plane + c, vb);
        } else {
          st_bf16x32(dA + c, va);
          st_bf16x32(dH + c, oh);
          st_bf16x32(dB + c, vb);
        }
      }
    }
  }
};

// ============================================================ apply-2: O = H_q W2^T
template <int BN>
struct OOp {
  struct Params {
    CUtensorMap mH;   // Hq 3D {dh, Cp, BH}, box {64, 128, 1}
    CUtensorMap mW2;  // shadows 3D {dh, d, 3BH}, box {64, BN, 1}
    bf16* O;
    int d, dh, T, chunk_start, valid, m_tiles, n_tiles;
    TcCommon cm;
  };
  struct Tile {
    int bh, row0, n0;
  };
  static constexpr int kStages = 4;
  static constexpr int kStageBytes = kABytes + BN * BK * 2;
  static constexpr int kTmemCols = BN <= 128 ? 128 : 256;

  static __device__ bool tile_of(const Params& p, Tile& t) {
    const int nt = blockIdx.x % p.n_tiles, mt = blockIdx.x / p.n_tiles;
    if (mt >= p.m_tiles) return false;
    t.row0 = mt * BM;
    t.n0 = nt * BN;
    t.bh = blockIdx.y;
    return true;
  }
  static __device__ int num_kblocks(const Params& p, const Tile&) { return p.dh / BK; }
  static __device__ uint32_t stage_tx(const Params&, const Tile&, int) { return kStageBytes; }
  static __device__ void produce(const Params& p, const Tile& t, int kb, uint8_t* st, uint64_t* bar) {
    ptx::tma_load_3d(st, &p.mH, bar, kb * BK, t.row0, t.bh);
    ptx::tma_load_3d(st + kABytes, &p.mW2, bar, kb * BK, t.n0, t.bh * 3 + 1);
  }
  static __device__ void consume(const Params&, const Tile&, int kb, uint32_t st, uint32_t tmem) {
    constexpr uint32_t id = ptx::idesc_bf16(128, BN, false, false);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) ptx::mma_bf16(tmem, kdesc(st, kk), kdesc(st + kABytes, kk), id, (kb | kk) != 0);
  }
  static __device__ void epilogue(const Params& p, const Tile& t, uint32_t tm, int r, float*, bool ok) {
    if (!ok) return;
    const int tl = t.row0 + r;
    const bool valid = tl < p.valid;
    bf16* dst = p.O + ((size_t)t.bh * p.T + p.chunk_start + tl) * p.d + t.n0;
    float v[32];
    for (int c = 0; c < BN; c += 32) {
      ptx::tmem_ld32(tm + c, v);
      if (valid && t.n0 + c < p.d) st_bf16x32(dst + c, v);
    }
  }
};

// ============================================================ chunk gradients
// z = bh*3 + j:  j=0  G1^T = K^T DA;  j=1  G2 = V^T He;  j=2  G3^T = K^T DB  (all [d, dh])
template <int BN>
struct GOp {
  struct Params {
    CUtensorMap mK4, mV4;  // 4D {d, C, n_full, BH}, box {64, 64, 1, 1}  (full chunks)
    CUtensorMap mK3, mV3;  // 3D {d, T, BH}, box {64, 64, 1}            (ragged last chunk)
    CUtensorMap mE;        // 3D {dh, Cp, 3BH}, box {64, 64, 1}
    CUtensorMap mEl;       // low halves of E (split precision)
    float* G;              // [Z][d][dh] fp32   (splits == 1)
    float* part;           // [Z][part_stride] sums of squares per tile (splits == 1)
    float* split_out;      // [splits][Z][d][dh] fp32 (splits > 1)
    int d, dh, Z, chunk_idx, chunk_start, valid, use4d, m_tiles, n_tiles, splits, kb_per_split, part_stride;
    int prec_split;        // E carried as hi + lo: two k passes over the tokens
    TcCommon cm;
  };
  struct Tile {
    int z, bh, j, m0, n0, kb0, nkb, split, tile_id;
  };
  static constexpr int kStages = 4;
  static constexpr int kStageBytes = kABytes + BN * BK * 2;
  static constexpr int kTmemCols = BN <= 128 ? 128 : 256;

  static __device__ bool tile_of(const Params& p, Tile& t) {
    const int nt = blockIdx.x % p.n_tiles, mt = blockIdx.x / p.n_tiles;
    if (mt >= p.m_tiles) return false;
    t.tile_id = blockIdx.x;
    t.m0 = mt * BM;
    t.n0 = nt * BN;
    t.z = blockIdx.y;
    t.bh = t.z / 3;
    t.j = t.z % 3;
    t.split = blockIdx.z;
    const int total = (p.valid + BK - 1) / BK;
    t.kb0 = t.split * p.kb_per_split;
    t.nkb = min(total, t.kb0 + p.kb_per_split) - t.kb0;
    return t.nkb > 0;
  }
  static __device__ int num_kblocks(const Params& p, const Tile& t) { return t.nkb * (p.prec_split ? 2 : 1); }
  static __device__ uint32_t stage_tx(const Params&, const Tile&, int) { return kStageBytes; }
  static __device__ void produce(const Params& p, const Tile& t, int kb, uint8_t* st, uint64_t* bar) {
    const CUtensorMap* e = kb >= t.nkb ? &p.mEl : &p.mE;
    const int tok = (t.kb0 + kb % t.nkb) * BK;
    for (int g = 0; g < 2; ++g) {
      if (p.use4d)
        ptx::tma_load_4d(st + g * kBox, t.j == 1 ? &p.mV4 : &p.mK4, bar, t.m0 + g * 64, tok, p.chunk_idx, t.bh);
      else
        ptx::tma_load_3d(st + g * kBox, t.j == 1 ? &p.mV3 : &p.mK3, bar, t.m0 + g * 64, p.chunk_start + tok, t.bh);
    }
#pragma unroll
    for (int g = 0; g < BN / 64; ++g) ptx::tma_load_3d(st + kABytes + g * kBox, e, bar, t.n0 + g * 64, tok, t.z);
  }
  static __device__ void consume(const Params&, const Tile&, int kb, uint32_t st, uint32_t tmem) {
    constexpr uint32_t id = ptx::idesc_bf16(128, BN, true, true);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) ptx::mma_bf16(tmem, mdesc(st, kk), mdesc(st + kABytes, kk), id, (kb | kk) != 0);
  }
  static __device__ void epilogue(const Params& p, const Tile& t, uint32_t tm, int r, float* red, bool ok) {
    const int m = t.m0 + r;
    const bool valid = ok && m < p.d;
    float ss = 0.f;
    float v[32];
    if (ok) {
      for (int c = 0; c < BN; c += 32) {
        ptx::tmem_ld32(tm + c, v);
        if (!valid || t.n0 + c >= p.dh) continue;
        if (p.splits == 1) {
          const size_t o = ((size_t)t.z * p.d + m) * p.dh + t.n0 + c;
          st_f32x32(p.G + o, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) ss = fmaf(v[i], v[i], ss);
        } else {
          st_f32x32(p.split_out + (((size_t)t.split * p.Z + t.z) * p.d + m) * p.dh + t.n0 + c, v);
        }
      }
    }
    if (p.splits == 1) {
      // deterministic per-tile sum of squares: warp butterfly, then 4 warps in lane-group order
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if ((r & 31) == 0) red[r >> 5] = ss;
      epi_bar();
      if (r == 0) p.part[(size_t)t.z * p.part_stride + t.tile_id] = ((red[0] + red[1]) + red[2]) + red[3];
      epi_bar();
    }
  }
};

// ============================================================ Newton-Schulz GEMMs
// Operands of the iteration: SINGLE precision uses one fp16 operand per matrix
// (11-bit significand at the bf16 tensor rate; X is normalised first, so X, S
// and P stay within fp16's range); SPLIT precision carries every operand as a
// bf16 pair (hi, lo) and forms each product from three MMAs
// (hi*hi + hi*lo + lo*hi, the lo*lo term is below the pair's resolution).
// X itself (the aX term) and S (the bS term) are also kept in fp32.
//
// k-block order of a SPLIT product: [hi*hi | hi*lo | lo*hi], each over the full K.
template <bool SPLIT>
__device__ __forceinline__ int ns_part(int kb, int nk) { return SPLIT ? kb / nk : 0; }

// Gram: S = X X^T (d x d, K = dh)
template <int BN, bool SPLIT>
struct GramOp {
  struct Params {
    CUtensorMap mXa, mXal;  // X hi / lo 3D {dh, d, Z}, box {64, 128, 1}
    CUtensorMap mXn, mXnl;  // same buffers, box {64, BN, 1}
    float* S;
    void* Sh;
    void* Sl;
    int d, dh, m_tiles, n_tiles;
    TcCommon cm;
  };
  struct Tile {
    int z, m0, n0;
  };
  static constexpr int kStages = 4;
  static constexpr int kStageBytes = kABytes + BN * BK * 2;
  static constexpr int kTmemCols = BN <= 128 ? 128 : 256;
  static __device__ bool tile_of(const Params& p, Tile& t) {
    const int nt = blockIdx.x % p.n_tiles, mt = blockIdx.x / p.n_tiles;
    if (mt >= p.m_tiles) return false;
    t.m0 = mt * BM;
    t.n0 = nt * BN;
    t.z = blockIdx.y;
    return true;
  }
  static __device__ int num_kblocks(const Params& p, const Tile&) { return (SPLIT ? 3 : 1) * (p.dh / BK); }
  static __device__ uint32_t stage_tx(const Params&, const Tile&, int) { return kStageBytes; }
  static __device__ void produce(const Params& p, const Tile& t, int kb, uint8_t* st, uint64_t* bar) {
    const int nk = p.dh / BK, part = ns_part<SPLIT>(kb, nk), k = kb % nk;
    ptx::tma_load_3d(st, part == 2 ? &p.mXal : &p.mXa, bar, k * BK, t.m0, t.z);
    ptx::tma_load_3d(st + kABytes, part == 1 ? &p.mXnl : &p.mXn, bar, k * BK, t.n0, t.z);
  }
  static __device__ void consume(const Params&, const Tile&, int kb, uint32_t st, uint32_t tmem) {
    constexpr uint32_t id = ptx::idesc_bf16(128, BN, false, false, !SPLIT);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) ptx::mma_bf16(tmem, kdesc(st, kk), kdesc(st + kABytes, kk), id, (kb | kk) != 0);
  }
  static __device__ void epilogue(const Params& p, const Tile& t, uint32_t tm, int r, float*, bool ok) {
    if (!ok) return;
    const int m = t.m0 + r;
    float v[32];
    for (int c = 0; c < BN; c += 32) {
      ptx::tmem_ld32(tm + c, v);
      if (m >= p.d || t.n0 + c >= p.d) continue;
      const size_t o = ((size_t)t.z * p.d + m) * p.d + t.n0 + c;
      st_f32x32(p.S + o, v);
      st_op32<SPLIT>(p.Sh, p.Sl, o, v);
    }
  }
};

// Poly: P = b S + c S S  (d x d, K = d; S is symmetric, so S^T serves as the B operand)
template <int BN, bool SPLIT>
struct PolyOp {
  struct Params {
    CUtensorMap mSa, mSal;  // S hi / lo 3D {d, d, Z}, box {64, 128, 1}
    CUtensorMap mSn, mSnl;  // box {64, BN, 1}
    const float* S;
    void* Ph;
    void* Pl;
    float b, c;
    int d, m_tiles, n_tiles;
    TcCommon cm;
  };
  struct Tile {
    int z, m0, n0;
  };
  static constexpr int kStages = 4;
  static constexpr int kStageBytes = kABytes + BN * BK * 2;
  static constexpr int kTmemCols = BN <= 128 ? 128 : 256;
  static __device__ bool tile_of(const Params& p, Tile& t) {
    const int nt = blockIdx.x % p.n_tiles, mt = blockIdx.x / p.n_tiles;
    if (mt >= p.m_tiles) return false;
    t.m0 = mt * BM;
    t.n0 = nt * BN;
    t.z = blockIdx.y;
    return true;
  }
  static __device__ int num_kblocks(const Params& p, const Tile&) { return (SPLIT ? 3 : 1) * (p.d / BK); }
  static __device__ uint32_t stage_tx(const Params&, const Tile&, int) { return kStageBytes; }
  static __device__ void produce(const Params& p, const Tile& t, int kb, uint8_t* st, uint64_t* bar) {
    const int nk = p.d / BK, part = ns_part<SPLIT>(kb, nk), k = kb % nk;
    ptx::tma_load_3d(st, part == 2 ? &p.mSal : &p.mSa, bar, k * BK, t.m0, t.z);
    ptx::tma_load_3d(st + kABytes, part == 1 ? &p.mSnl : &p.mSn, bar, k * BK, t.n0, t.z);
  }
  static __device__ void consume(const Params&, const Tile&, int kb, uint32_t st, uint32_t tmem) {
    constexpr uint32_t id = ptx::idesc_bf16(128, BN, false, false, !SPLIT);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) ptx::mma_bf16(tmem, kdesc(st, kk), kdesc(st + kABytes, kk), id, (kb | kk) != 0);
  }
  static __device__ void epilogue(const Params& p, const Tile& t, uint32_t tm, int r, float*, bool ok) {
    if (!ok) return;
    const int m = t.m0 + r;
    float v[32], s[32];
    for (int c = 0; c < BN; c += 32) {
      ptx::tmem_ld32(tm + c, v);
      if (m >= p.d || t.n0 + c >= p.d) continue;
      const size_t o = ((size_t)t.z * p.d + m) * p.d + t.n0 + c;
      ld_f32x32(p.S + o, s);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = p.b * s[i] + p.c * v[i];
      st_op32<SPLIT>(p.Ph, p.Pl, o, v);
    }
  }
};

// Xupd: X <- a X + P X  (d x dh, K = d); P K-major, X as the MN-major B operand.
template <int BN, bool SPLIT>
struct XupdOp {
  struct Params {
    CUtensorMap mPa, mPal;  // P hi / lo 3D {d, d, Z}, box {64, 128, 1}
    CUtensorMap mXm, mXml;  // current X hi / lo 3D {dh, d, Z}, box {64, 64, 1}
    float* X;               // fp32 [Z][d][dh], updated in place
    void* Xh_next;          // operand copy of the new X (hi)
    void* Xl_next;          // (lo, SPLIT only)
    float a;
    int d, dh, m_tiles, n_tiles;
    TcCommon cm;
  };
  struct Tile {
    int z, m0, n0;
  };
  static constexpr int kStages = 4;
  static constexpr int kStageBytes = kABytes + BN * BK * 2;
  static constexpr int kTmemCols = BN <= 128 ? 128 : 256;
  static __device__ bool tile_of(const Params& p, Tile& t) {
    const int nt = blockIdx.x % p.n_tiles, mt = blockIdx.x / p.n_tiles;
    if (mt >= p.m_tiles) return false;
    t.m0 = mt * BM;
    t.n0 = nt * BN;
    t.z = blockIdx.y;
    return true;
  }
  static __device__ int num_kblocks(const Params& p, const Tile&) { return (SPLIT ? 3 : 1) * (p.d / BK); }
  static __device__ uint32_t stage_tx(const Params&, const Tile&, int) { return kStageBytes; }
  static __device__ void produce(const Params& p, const Tile& t, int kb, uint8_t* st, uint64_t* bar) {
    const int nk = p.d / BK, part = ns_part<SPLIT>(kb, nk), k = kb % nk;
    ptx::tma_load_3d(st, part == 2 ? &p.mPal : &p.mPa, bar, k * BK, t.m0, t.z);
    const CUtensorMap* xb = part == 1 ? &p.mXml : &p.mXm;
#pragma unroll
    for (int g = 0; g < BN / 64; ++g) ptx::tma_load_3d(st + kABytes + g * kBox, xb, bar, t.n0 + g * 64, k * BK, t.z);
  }
  static __device__ void consume(const Params&, const Tile&, int kb, uint32_t st, uint32_t tmem) {
    constexpr uint32_t id = ptx::idesc_bf16(128, BN, false, true, !SPLIT);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) ptx::mma_bf16(tmem, kdesc(st, kk), mdesc(st + kABytes, kk), id, (kb | kk) != 0);
  }
  static __device__ void epilogue(const Params& p, const Tile& t, uint32_t tm, int r, float*, bool ok) {
    if (!ok) return;
    const int m = t.m0 + r;
    float v[32], x[32];
    for (int c = 0; c < BN; c += 32) {
      ptx::tmem_ld32(tm + c, v);
      if (m >= p.d || t.n0 + c >= p.dh) continue;
      const size_t o = ((size_t)t.z * p.d + m) * p.dh + t.n0 + c;
      ld_f32x32(p.X + o, x);
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = p.a * x[i] + v[i];
      st_f32x32(p.X + o, x);
      st_op32<SPLIT>(p.Xh_next, p.Xl_next, o, x);
    }
  }
};

// ============================================================ plain GEMM (test hook)
template <bool AMN, bool BMN>
struct PlainOp {
  struct Params {
    CUtensorMap mA, mB;
    float* D;
    int M, N, K, m_tiles, n_tiles;
    TcCommon cm;
  };
  struct Tile {
    int z, m0, n0;
  };
  static constexpr int BN = 128;
  static constexpr int kStages = 4;
  static constexpr int kStageBytes = kABytes + BN * BK * 2;
  static constexpr int kTmemCols = 128;
  static __device__ bool tile_of(const Params& p, Tile& t) {
    const int nt = blockIdx.x % p.n_tiles, mt = blockIdx.x / p.n_tiles;
    if (mt >= p.m_tiles) return false;
    t.m0 = mt * BM;
    t.n0 = nt * BN;
    t.z = blockIdx.y;
    return true;
  }
  static __device__ int num_kblocks(const Params& p, const Tile&) { return p.K / BK; }
  static __device__ uint32_t stage_tx(const Params&, const Tile&, int) { return kStageBytes; }
  static __device__ void produce(const Params& p, const Tile& t, int kb, uint8_t* st, uint64_t* bar) {
    if (AMN) {
      for (int g = 0; g < 2; ++g) ptx::tma_load_3d(st + g * kBox, &p.mA, bar, t.m0 + g * 64, kb * BK, t.z);
    } else {
      ptx::tma_load_3d(st, &p.mA, bar, kb * BK, t.m0, t.z);
    }
    if (BMN) {
      for (int g = 0; g < BN / 64; ++g)
        ptx::tma_load_3d(st + kABytes + g * kBox, &p.mB, bar, t.n0 + g * 64, kb * BK, t.z);
    } else {
      ptx::tma_load_3d(st + kABytes, &p.mB, bar, kb * BK, t.n0, t.z);
    }
  }
  static __device__ void consume(const Params&, const Tile&, int kb, uint32_t st, uint32_t tmem) {
    constexpr uint32_t id = ptx::idesc_bf16(128, BN, AMN, BMN);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t a = AMN ? mdesc(st, kk) : kdesc(st, kk);
      const uint64_t b = BMN ? mdesc(st + kABytes, kk) : kdesc(st + kABytes, kk);
      ptx::mma_bf16(tmem, a, b, id, (kb | kk) != 0);
    }
  }
  static __device__ void epilogue(const Params& p, const Tile& t, uint32_t tm, int r, float*, bool ok) {
    if (!ok) return;
    const int m = t.m0 + r;
    float v[32];
    for (int c = 0; c < BN; c += 32) {
      ptx::tmem_ld32(tm + c, v);
      if (m < p.M && t.n0 + c < p.N) st_f32x32(p.D + ((size_t)t.z * p.M + m) * p.N + t.n0 + c, v);
    }
  }
};

// ============================================================ SIMT helper kernels
__device__ __forceinline__ void st_shadow(bf16* hi, bf16* lo, size_t o, float v) {
  const bf16 h = __float2bfloat16_rn(v);
  hi[o] = h;
  if (lo) lo[o] = __float2bfloat16_rn(v - __bfloat162float(h));
}

// W0 (out x in, per head) -> M = [W1^T, W2, W3^T] fp32 + bf16 shadow (hi, and lo
// when the weights are carried split), per (b, h).
__global__ void import_kernel(const float* W1, const float* W2, const float* W3, float* M, bf16* Ms, bf16* Msl,
                              int H, int d, int dh, int w0_per_batch) {
  __shared__ float tile[32][33];
  const int z = blockIdx.z, bh = z / 3, j = z % 3;
  const int src_head = w0_per_batch ? bh : bh % H;
  const size_t n = (size_t)d * dh;
  float* dst = M + (size_t)z * n;
  bf16* dh_ = Ms + (size_t)z * n;
  bf16* dl_ = Msl ? Msl + (size_t)z * n : nullptr;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  if (j == 1) {
    const float* src = W2 + (size_t)src_head * n;  // [d][dh]
    const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    for (int rr = ty; rr < 32; rr += 8) {
      const int r = r0 + rr, c = c0 + tx;
      if (r < d && c < dh) {
        const float v = src[(size_t)r * dh + c];
        dst[(size_t)r * dh + c] = v;
        st_shadow(dh_, dl_, (size_t)r * dh + c, v);
      }
    }
    return;
  }
  const float* src = (j == 0 ? W1 : W3) + (size_t)src_head * n;  // [dh][d]
  // output block: rows i in [r0, r0+32) of d, cols jj in [c0, c0+32) of dh
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  for (int rr = ty; rr < 32; rr += 8) {  // read src rows jj = c0 + rr, cols i = r0 + tx
    const int jj = c0 + rr, i = r0 + tx;
    tile[rr][tx] = (jj < dh && i < d) ? src[(size_t)jj * d + i] : 0.f;
  }
  __syncthreads();
  for (int rr = ty; rr < 32; rr += 8) {
    const int i = r0 + rr, jj = c0 + tx;
    if (i < d && jj < dh) {
      const float v = tile[tx][rr];
      dst[(size_t)i * dh + jj] = v;
      st_shadow(dh_, dl_, (size_t)i * dh + jj, v);
    }
  }
}

// M -> Wf (out x in): Wf1 = M1^T, Wf2 = M2, Wf3 = M3^T
__global__ void export_kernel(const float* M, float* Wf1, float* Wf2, float* Wf3, int d, int dh) {
  __shared__ float tile[32][33];
  const int z = blockIdx.z, bh = z / 3, j = z % 3;
  const size_t n = (size_t)d * dh;
  const float* src = M + (size_t)z * n;  // [d][dh]
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;  // src rows i, cols jj
  if (j == 1) {
    float* dst = Wf2 + (size_t)bh * n;
    for (int rr = ty; rr < 32; rr += 8) {
      const int r = r0 + rr, c = c0 + tx;
      if (r < d && c < dh) dst[(size_t)r * dh + c] = src[(size_t)r * dh + c];
    }
    return;
  }
  float* dst = (j == 0 ? Wf1 : Wf3) + (size_t)bh * n;  // [dh][d]
  for (int rr = ty; rr < 32; rr += 8) {
    const int i = r0 + rr, jj = c0 + tx;
    tile[rr][tx] = (i < d && jj < dh) ? src[(size_t)i * dh + jj] : 0.f;
  }
  __syncthreads();
  for (int rr = ty; rr < 32; rr += 8) {
    const int jj = c0 + rr, i = r0 + tx;
    if (jj < dh && i < d) dst[(size_t)jj * d + i] = tile[tx][rr];
  }
}

// Row norms of W0 in the internal layout: columns of M1/M3 (over d), rows of M2 (over dh).
// One block of 256 threads per (z, 32-column slab) for j = 0, 2 and per (z, 8 rows) for j = 1.
__global__ void norms_kernel(const float* M, float* n0, int d, int dh) {
  __shared__ float red[8][33];
  const int z = blockIdx.y, j = z % 3;
  const float* src = M + (size_t)z * d * dh;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (j == 1) {
    const int r = blockIdx.x * 8 + w;
    if (blockIdx.x * 8 >= d) return;
    float s = 0.f;
    if (r < d)
      for (int c = lane; c < dh; c += 32) s = fmaf(src[(size_t)r * dh + c], src[(size_t)r * dh + c], s);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0 && r < d) n0[(size_t)z * dh + r] = sqrtf(s);
  } else {
    const int c = blockIdx.x * 32 + lane;
    if (blockIdx.x * 32 >= dh) return;
    float s = 0.f;
    if (c < dh)
      for (int r = w; r < d; r += 8) s = fmaf(src[(size_t)r * dh + c], src[(size_t)r * dh + c], s);
    red[w][lane] = s;
    __syncthreads();
    if (w == 0 && c < dh) {
      float t = 0.f;
      for (int k = 0; k < 8; ++k) t += red[k][lane];
      n0[(size_t)z * dh + c] = sqrtf(t);
    }
  }
}

// M <- M - step*U; optional weight norm back to n0 (LaCT page §2.2.1, eq. 8; the
// rows of W1/W3 are the columns of M1/M3); refresh the bf16 shadow(s).
__global__ void update_kernel(float* M, bf16* Ms, bf16* Msl, const float* U, const float* n0, float step,
                              int wnorm, float floor_, int d, int dh) {
  __shared__ float red[8][33];
  const int z = blockIdx.y, j = z % 3;
  const size_t base = (size_t)z * d * dh;
  float* m = M + base;
  bf16* ms = Ms + base;
  bf16* ml = Msl ? Msl + base : nullptr;
  const float* u = U + base;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (j == 1) {
    if (blockIdx.x * 8 >= d) return;
    const int r = blockIdx.x * 8 + w;
    if (r >= d) return;  // warp-uniform
    float s = 0.f;
    for (int c = lane; c < dh; c += 32) {
      const float x = m[(size_t)r * dh + c] - step * u[(size_t)r * dh + c];
      s = fmaf(x, x, s);
    }
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float sc = wnorm ? n0[(size_t)z * dh + r] / fmaxf(sqrtf(s), floor_) : 1.f;
    for (int c = lane; c < dh; c += 32) {
      const float x = (m[(size_t)r * dh + c] - step * u[(size_t)r * dh + c]) * sc;
      m[(size_t)r * dh + c] = x;
      st_shadow(ms, ml, (size_t)r * dh + c, x);
    }
  } else {
    if (blockIdx.x * 32 >= dh) return;
    const int c = blockIdx.x * 32 + lane;
    float s = 0.f;
    if (c < dh)
      for (int r = w; r < d; r += 8) {
        const float x = m[(size_t)r * dh + c] - step * u[(size_t)r * dh + c];
        s = fmaf(x, x, s);
      }
    red[w][lane] = s;
    __syncthreads();
    float t = 0.f;
    for (int k = 0; k < 8; ++k) t += red[k][lane];
    const float sc = (wnorm && c < dh) ? n0[(size_t)z * dh + c] / fmaxf(sqrtf(t), floor_) : 1.f;
    if (c < dh)
      for (int r = w; r < d; r += 8) {
        const float x = (m[(size_t)r * dh + c] - step * u[(size_t)r * dh + c]) * sc;
        m[(size_t)r * dh + c] = x;
        st_shadow(ms, ml, (size_t)r * dh + c, x);
      }
  }
}

// Split-K reduction of the gradient: fixed split order; sums of squares per block.
__global__ void gsplit_reduce_kernel(const float* parts, float* G, float* part, int splits, int Z,
                                     size_t per_z, int part_stride) {
  __shared__ float red[256];
  const int z = blockIdx.y;
  float ss = 0.f;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < per_z; e += (size_t)gridDim.x * blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) acc += parts[((size_t)s * Z + z) * per_z + e];
    G[(size_t)z * per_z + e] = acc;
    ss = fmaf(acc, acc, ss);
  }
  red[threadIdx.x] = ss;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) part[(size_t)z * part_stride + blockIdx.x] = red[0];
}

// X0 = G / (||G||_F + eps) in place (fp32) plus its operand copy (fp16, or a
// bf16 hi/lo pair). Every block sums the per-tile squares of its matrix in the
// same order, so all of them use the same norm.
template <bool SPLIT>
__global__ void ns_normalize_kernel(float* G, void* Xh, void* Xl, const float* part, int n_part,
                                    int part_stride, float eps, size_t per_z) {
  const int z = blockIdx.y;
  float s = 0.f;
  for (int i = 0; i < n_part; ++i) s += part[(size_t)z * part_stride + i];
  const float inv = 1.f / (sqrtf(s) + eps);
  float* g = G + (size_t)z * per_z;
  for (size_t e = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; e < per_z;
       e += (size_t)gridDim.x * blockDim.x * 4) {
    float4 v = *reinterpret_cast<float4*>(g + e);
    v.x *= inv; v.y *= inv; v.z *= inv; v.w *= inv;
    *reinterpret_cast<float4*>(g + e) = v;
    const size_t o = (size_t)z * per_z + e;
    if (SPLIT) {
      uint2 h, l;
      h.x = pack_bf16(v.x, v.y);
      h.y = pack_bf16(v.z, v.w);
      const __nv_bfloat162 h0 = *reinterpret_cast<__nv_bfloat162*>(&h.x);
      const __nv_bfloat162 h1 = *reinterpret_cast<__nv_bfloat162*>(&h.y);
      l.x = pack_bf16(v.x - __low2float(h0), v.y - __high2float(h0));
      l.y = pack_bf16(v.z - __low2float(h1), v.w - __high2float(h1));
      *reinterpret_cast<uint2*>(static_cast<bf16*>(Xh) + o) = h;
      *reinterpret_cast<uint2*>(static_cast<bf16*>(Xl) + o) = l;
    } else {
      uint2 h;
      h.x = pack_f16(v.x, v.y);
      h.y = pack_f16(v.z, v.w);
      *reinterpret_cast<uint2*>(static_cast<f16*>(Xh) + o) = h;
    }
  }
}

// ============================================================ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 16-bit tensor map over a row-major array with dims (innermost first) and box.
bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint32_t* box,
              CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn();
  if (!fn || !base) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  uint64_t stride = 2;
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i > 0) gs[i - 1] = stride;
    stride *= dims[i];
  }
  const CUresult r = fn(m, dt, rank, const_cast<void*>(base), gd, gs, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool map3(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1,
          CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint32_t box[3] = {b0, b1, 1};
  return make_map(m, base, 3, dims, box, dt);
}

template <class Op>
int launch_op(int kind, const typename Op::Params& p, dim3 grid, cudaStream_t st) {
  const size_t smem = tc_smem_bytes<Op>();
  if (cudaFuncSetAttribute(tc_kernel<Op>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return TTT_ERR_CUDA;
  prof_before(kind, st);
  tc_kernel<Op><<<grid, kTcThreads, smem, st>>>(p);
  prof_after(kind, st);
  return cudaGetLastError() == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

// Plain kernel launch with accounting.
#define TTT_LAUNCH(kind, st, ...)      \
  do {                                 \
    prof_before(kind, st);             \
    __VA_ARGS__;                       \
    prof_after(kind, st);              \
    if (cudaGetLastError() != cudaSuccess) return TTT_ERR_CUDA; \
  } while (0)

struct Plan {
  int BH, Z, d, dh, C, Cp, T, split;
  int bn_o, bn_dd;        // N tile of the apply GEMM (over d) and of the d x d NS GEMMs
  int g_mt, g_nt, splits, kb_per_split, part_stride, reduce_blocks;
  size_t off_M, off_Ms, off_Msl, off_n0, off_Hq, off_E, off_El, off_G, off_Xh[2], off_Xl[2], off_S, off_Sh,
      off_Sl, off_Ph, off_Pl, off_part, off_split, total;
};

int pick_bn_d(int d) {
  if (d % 256 == 0) return 256;
  if (d % 192 == 0 && d <= 192) return 192;
  return 128;
}

Plan make_plan(const ttt_cfg& g) {
  Plan P{};
  P.BH = g.B * g.H;
  P.Z = 3 * P.BH;
  P.d = g.d;
  P.dh = g.dh;
  P.T = g.T;
  P.split = g.precision == TTT_PREC_SPLIT ? 1 : 0;
  P.C = std::min(g.chunk, g.T);
  P.Cp = (P.C + BM - 1) / BM * BM;
  P.bn_o = pick_bn_d(g.d);
  P.bn_dd = pick_bn_d(g.d);
  const int gbn = (g.dh % 256 == 0) ? 256 : 128;
  P.g_mt = (g.d + BM - 1) / BM;
  P.g_nt = g.dh / gbn;
  const int tiles = P.g_mt * P.g_nt * P.Z;
  const int kbs = (P.C + BK - 1) / BK;
  int splits = 1;
  if (tiles < 2 * 148) splits = std::min(std::max(1, kbs / 16), (2 * 148 + tiles - 1) / tiles);
  P.kb_per_split = (kbs + splits - 1) / splits;
  P.splits = (kbs + P.kb_per_split - 1) / P.kb_per_split;
  P.reduce_blocks = 32;
  P.part_stride = std::max(P.g_mt * P.g_nt, P.reduce_blocks);
  const size_t wz = (size_t)P.Z * g.d * g.dh;
  const size_t dd = (size_t)P.Z * g.d * g.d;
  const size_t lo = P.split ? 1 : 0;  // the low halves exist only in split precision
  size_t off = kStatusBytes;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  P.off_M = take(wz * 4);
  P.off_Ms = take(wz * 2);
  P.off_Msl = take(lo * wz * 2);
  P.off_n0 = take((size_t)P.Z * g.dh * 4);
  P.off_Hq = take((size_t)P.BH * P.Cp * g.dh * 2);
  P.off_E = take((size_t)P.BH * 3 * P.Cp * g.dh * 2);
  P.off_El = take(lo * P.BH * 3 * P.Cp * g.dh * 2);
  P.off_G = take(wz * 4);
  for (int i = 0; i < 2; ++i) {
    P.off_Xh[i] = take(wz * 2);
    P.off_Xl[i] = take(lo * wz * 2);
  }
  P.off_S = take(dd * 4);
  P.off_Sh = take(dd * 2);
  P.off_Sl = take(lo * dd * 2);
  P.off_Ph = take(dd * 2);
  P.off_Pl = take(lo * dd * 2);
  P.off_part = take((size_t)P.Z * P.part_stride * 4);
  P.off_split = take(P.splits > 1 ? (size_t)P.splits * wz * 4 : 0);
  P.total = off;
  return P;
}

// Launches one Newton-Schulz iteration's three GEMMs for a fixed N tile choice.
template <int BND, int BNX, bool SPLIT>
int ns_iteration(const CUtensorMap* mXa, const CUtensorMap* mXn, const CUtensorMap* mXm, const CUtensorMap* mSa,
                 const CUtensorMap* mSn, const CUtensorMap* mPa, float* X, void* xh_next, void* xl_next, float* S,
                 void* Sh, void* Sl, void* Ph, void* Pl, const ttt_cfg& g, int Z, const TcCommon& cm,
                 cudaStream_t st) {
  const int d = g.d, dh = g.dh;
  const int mt = (d + BM - 1) / BM, ntd = (d + BND - 1) / BND, ntx = dh / BNX;
  {
    typename GramOp<BND, SPLIT>::Params p{};
    p.mXa = mXa[0]; p.mXal = mXa[1]; p.mXn = mXn[0]; p.mXnl = mXn[1];
    p.S = S; p.Sh = Sh; p.Sl = Sl; p.d = d; p.dh = dh; p.m_tiles = mt; p.n_tiles = ntd; p.cm = cm;
    const int r = launch_op<GramOp<BND, SPLIT>>(TTT_KERNEL_GRAM, p, dim3(mt * ntd, Z), st);
    if (r != TTT_OK) return r;
  }
  {
    typename PolyOp<BND, SPLIT>::Params p{};
    p.mSa = mSa[0]; p.mSal = mSa[1]; p.mSn = mSn[0]; p.mSnl = mSn[1];
    p.S = S; p.Ph = Ph; p.Pl = Pl; p.b = g.ns_b; p.c = g.ns_c; p.d = d; p.m_tiles = mt; p.n_tiles = ntd;
    p.cm = cm;
    const int r = launch_op<PolyOp<BND, SPLIT>>(TTT_KERNEL_POLY, p, dim3(mt * ntd, Z), st);
    if (r != TTT_OK) return r;
  }
  typename XupdOp<BNX, SPLIT>::Params p{};
  p.mPa = mPa[0]; p.mPal = mPa[1]; p.mXm = mXm[0]; p.mXml = mXm[1];
  p.X = X; p.Xh_next = xh_next; p.Xl_next = xl_next; p.a = g.ns_a; p.d = d; p.dh = dh; p.m_tiles = mt;
  p.n_tiles = ntx; p.cm = cm;
  return launch_op<XupdOp<BNX, SPLIT>>(TTT_KERNEL_XUPD, p, dim3(mt * ntx, Z), st);
}

template <bool SPLIT>
int ns_iteration_any(int bnd, int bnx, const CUtensorMap* mXa, const CUtensorMap* mXn, const CUtensorMap* mXm,
                     const CUtensorMap* mSa, const CUtensorMap* mSn, const CUtensorMap* mPa, float* X,
                     void* xh_next, void* xl_next, float* S, void* Sh, void* Sl, void* Ph, void* Pl,
                     const ttt_cfg& g, int Z, const TcCommon& cm, cudaStream_t st) {
#define TTT_NS_CASE(BD, BX)                                                                                  \
  if (bnd == BD && bnx == BX)                                                                                 \
    return ns_iteration<BD, BX, SPLIT>(mXa, mXn, mXm, mSa, mSn, mPa, X, xh_next, xl_next, S, Sh, Sl, Ph, Pl, \
                                       g, Z, cm, st);
  TTT_NS_CASE(256, 256)
  TTT_NS_CASE(256, 128)
  TTT_NS_CASE(192, 256)
  TTT_NS_CASE(192, 128)
  TTT_NS_CASE(128, 256)
  TTT_NS_CASE(128, 128)
#undef TTT_NS_CASE
  return TTT_ERR_UNSUPPORTED;
}

}  // namespace

bool tc_supported(const ttt_cfg& g) {
  return g.dtype == TTT_DTYPE_BF16 && g.fast_net == TTT_NET_SWIGLU && g.loss == TTT_LOSS_IP && g.d % 64 == 0 &&
         g.dh % 128 == 0 && g.d <= g.dh && g.d <= 4096 && g.dh <= 16384;
}

size_t tc_workspace_bytes(const ttt_cfg& g) { return make_plan(g).total; }

int tc_run(const Call& c) {
  const ttt_cfg& g = c.cfg;
  const Plan P = make_plan(g);
  const bool split = P.split != 0;
  const cudaStream_t st = c.stream;
  char* ws = c.ws;
  auto at = [&](size_t off, size_t n) -> void* { return n ? static_cast<void*>(ws + off) : nullptr; };
  float* M = reinterpret_cast<float*>(ws + P.off_M);
  bf16* Ms = reinterpret_cast<bf16*>(ws + P.off_Ms);
  bf16* Msl = split ? reinterpret_cast<bf16*>(ws + P.off_Msl) : nullptr;
  float* n0 = reinterpret_cast<float*>(ws + P.off_n0);
  bf16* Hq = reinterpret_cast<bf16*>(ws + P.off_Hq);
  bf16* E = reinterpret_cast<bf16*>(ws + P.off_E);
  bf16* El = split ? reinterpret_cast<bf16*>(ws + P.off_El) : nullptr;
  float* G = reinterpret_cast<float*>(ws + P.off_G);
  void* Xh[2] = {ws + P.off_Xh[0], ws + P.off_Xh[1]};
  void* Xl[2] = {at(P.off_Xl[0], split), at(P.off_Xl[1], split)};
  float* S = reinterpret_cast<float*>(ws + P.off_S);
  void* Sh = ws + P.off_Sh;
  void* Sl = at(P.off_Sl, split);
  void* Ph = ws + P.off_Ph;
  void* Pl = at(P.off_Pl, split);
  float* part = reinterpret_cast<float*>(ws + P.off_part);
  float* splitbuf = reinterpret_cast<float*>(ws + P.off_split);
  int* status = reinterpret_cast<int*>(ws);
  const TcCommon cm{status, (unsigned long long)c.cfg.timeout_us * 1000ull};
  const int d = g.d, dh = g.dh, BH = P.BH, Z = P.Z, T = g.T;
  const int n_full = T / P.C;
  const CUtensorMapDataType ns_dt = split ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;

  // ---- tensor maps ([0] = hi or single operand, [1] = lo; lo maps alias hi in SINGLE precision)
  CUtensorMap mQ, mK, mV, mK3, mV3, mK4, mV4, mW[2], mHq, mW2o, mE[2];
  CUtensorMap mXa[2][2], mXn[2][2], mXm[2][2], mSa[2], mSn[2], mPa[2];
  bool ok = true;
  ok &= map3(&mQ, c.Q, d, T, BH, 64, 128);
  ok &= map3(&mK, c.K, d, T, BH, 64, 128);
  ok &= map3(&mV, c.V, d, T, BH, 64, 128);
  ok &= map3(&mK3, c.K, d, T, BH, 64, 64);
  ok &= map3(&mV3, c.V, d, T, BH, 64, 64);
  if (n_full > 0) {
    // 4D view {d, C, n_full, BH}: a chunk's token range ends at the chunk boundary
    auto fn = encode_fn();
    if (!fn) return TTT_ERR_CUDA;
    CUtensorMap* outs[2] = {&mK4, &mV4};
    const void* bases[2] = {c.K, c.V};
    for (int i = 0; i < 2; ++i) {
      cuuint64_t gd[4] = {(cuuint64_t)d, (cuuint64_t)P.C, (cuuint64_t)n_full, (cuuint64_t)BH};
      cuuint64_t gs[3] = {(cuuint64_t)d * 2, (cuuint64_t)P.C * d * 2, (cuuint64_t)T * d * 2};
      cuuint32_t bx[4] = {64, 64, 1, 1};
      cuuint32_t es[4] = {1, 1, 1, 1};
      ok &= fn(outs[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(bases[i]), gd, gs, bx, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
  } else {
    mK4 = mK3;
    mV4 = mV3;
  }
  ok &= map3(&mW[0], Ms, dh, d, Z, 64, 64);
  ok &= map3(&mW[1], split ? Msl : Ms, dh, d, Z, 64, 64);
  ok &= map3(&mHq, Hq, dh, P.Cp, BH, 64, 128);
  ok &= map3(&mW2o, Ms, dh, d, Z, 64, P.bn_o);
  ok &= map3(&mE[0], E, dh, P.Cp, Z, 64, 64);
  ok &= map3(&mE[1], split ? El : E, dh, P.Cp, Z, 64, 64);
  for (int i = 0; i < 2; ++i)      // ping-pong buffer
    for (int h = 0; h < 2; ++h) {  // hi / lo
      const void* b = (h && split) ? Xl[i] : Xh[i];
      ok &= map3(&mXa[i][h], b, dh, d, Z, 64, 128, ns_dt);
      ok &= map3(&mXn[i][h], b, dh, d, Z, 64, P.bn_dd, ns_dt);
      ok &= map3(&mXm[i][h], b, dh, d, Z, 64, 64, ns_dt);
    }
  for (int h = 0; h < 2; ++h) {
    const void* sb = (h && split) ? Sl : Sh;
    const void* pb = (h && split) ? Pl : Ph;
    ok &= map3(&mSa[h], sb, d, d, Z, 64, 128, ns_dt);
    ok &= map3(&mSn[h], sb, d, d, Z, 64, P.bn_dd, ns_dt);
    ok &= map3(&mPa[h], pb, d, d, Z, 64, 128, ns_dt);
  }
  if (!ok) return TTT_ERR_CUDA;

  int rc;
  // ---- import W0, reference row norms
  {
    const dim3 grid((dh + 31) / 32, (d + 31) / 32, Z);
    TTT_LAUNCH(TTT_KERNEL_AUX, st,
               import_kernel<<<grid, 256, 0, st>>>(c.W0[0], c.W0[1], c.W0[2], M, Ms, Msl, g.H, d, dh,
                                                   g.w0_per_batch));
    const dim3 gn(std::max((dh + 31) / 32, (d + 7) / 8), Z);
    TTT_LAUNCH(TTT_KERNEL_AUX, st, norms_kernel<<<gn, 256, 0, st>>>(M, n0, d, dh));
  }

  auto run_fwd = [&](int s, int valid, bool q, bool k) -> int {
    FwdOp::Params p{};
    p.mQ = mQ; p.mK = mK; p.mV = mV; p.mW = mW[0]; p.mWl = mW[1];
    p.lr = c.lr; p.Hq = Hq; p.E = E; p.El = El;
    p.d = d; p.dh = dh; p.T = T; p.Cp = P.Cp; p.chunk_start = s; p.valid = valid;
    const int tiles = (valid + BM - 1) / BM;
    p.q_tiles = q ? tiles : 0;
    p.k_tiles = k ? tiles : 0;
    p.n_tiles = dh / 128;
    p.split = split ? 1 : 0;
    p.cm = cm;
    return launch_op<FwdOp>(TTT_KERNEL_FWD, p, dim3((p.q_tiles + p.k_tiles) * p.n_tiles, BH), st);
  };
  auto run_o = [&](int s, int valid) -> int {
    const int mt = (valid + BM - 1) / BM, nt = (d + P.bn_o - 1) / P.bn_o;
    auto fill = [&](auto& p) {
      p.mH = mHq; p.mW2 = mW2o; p.O = static_cast<bf16*>(c.O);
      p.d = d; p.dh = dh; p.T = T; p.chunk_start = s; p.valid = valid; p.m_tiles = mt; p.n_tiles = nt; p.cm = cm;
    };
    const dim3 grid(mt * nt, BH);
    if (P.bn_o == 256) { typename OOp<256>::Params p{}; fill(p); return launch_op<OOp<256>>(TTT_KERNEL_APPLY, p, grid, st); }
    if (P.bn_o == 192) { typename OOp<192>::Params p{}; fill(p); return launch_op<OOp<192>>(TTT_KERNEL_APPLY, p, grid, st); }
    typename OOp<128>::Params p{}; fill(p); return launch_op<OOp<128>>(TTT_KERNEL_APPLY, p, grid, st);
  };
  auto run_grad = [&](int ci, int s, int valid, int& n_part) -> int {
    const bool full = (s + P.C <= T) && ci < n_full;
    const int kbs = (valid + BK - 1) / BK;
    const int splits = (kbs + P.kb_per_split - 1) / P.kb_per_split;
    auto fill = [&](auto& p) {
      p.mK4 = mK4; p.mV4 = mV4; p.mK3 = mK3; p.mV3 = mV3; p.mE = mE[0]; p.mEl = mE[1];
      p.G = G; p.part = part; p.split_out = splitbuf;
      p.d = d; p.dh = dh; p.Z = Z; p.chunk_idx = ci; p.chunk_start = s; p.valid = valid; p.use4d = full ? 1 : 0;
      p.m_tiles = P.g_mt; p.n_tiles = P.g_nt; p.splits = splits; p.kb_per_split = P.kb_per_split;
      p.part_stride = P.part_stride; p.prec_split = split ? 1 : 0; p.cm = cm;
    };
    const dim3 grid(P.g_mt * P.g_nt, Z, splits);
    int r;
    if (dh % 256 == 0) { typename GOp<256>::Params p{}; fill(p); r = launch_op<GOp<256>>(TTT_KERNEL_GRAD, p, grid, st); }
    else { typename GOp<128>::Params p{}; fill(p); r = launch_op<GOp<128>>(TTT_KERNEL_GRAD, p, grid, st); }
    if (r != TTT_OK) return r;
    if (splits > 1)
      TTT_LAUNCH(TTT_KERNEL_GRAD, st,
                 gsplit_reduce_kernel<<<dim3(P.reduce_blocks, Z), 256, 0, st>>>(splitbuf, G, part, splits, Z,
                                                                                 (size_t)d * dh, P.part_stride));
    n_part = splits > 1 ? P.reduce_blocks : P.g_mt * P.g_nt;
    return TTT_OK;
  };
  auto run_ns = [&](int n_part) -> int {
    if (split)
      TTT_LAUNCH(TTT_KERNEL_AUX, st,
                 ns_normalize_kernel<true><<<dim3(16, Z), 256, 0, st>>>(G, Xh[0], Xl[0], part, n_part,
                                                                        P.part_stride, g.ns_eps, (size_t)d * dh));
    else
      TTT_LAUNCH(TTT_KERNEL_AUX, st,
                 ns_normalize_kernel<false><<<dim3(16, Z), 256, 0, st>>>(G, Xh[0], Xl[0], part, n_part,
                                                                         P.part_stride, g.ns_eps, (size_t)d * dh));
    const int bnx = (dh % 256 == 0) ? 256 : 128;
    for (int it = 0; it < g.ns_iters; ++it) {
      const int cur = it & 1, nxt = cur ^ 1;
      const int r = split ? ns_iteration_any<true>(P.bn_dd, bnx, mXa[cur], mXn[cur], mXm[cur], mSa, mSn, mPa, G,
                                                   Xh[nxt], Xl[nxt], S, Sh, Sl, Ph, Pl, g, Z, cm, st)
                          : ns_iteration_any<false>(P.bn_dd, bnx, mXa[cur], mXn[cur], mXm[cur], mSa, mSn, mPa,
                                                    G, Xh[nxt], Xl[nxt], S, Sh, Sl, Ph, Pl, g, Z, cm, st);
      if (r != TTT_OK) return r;
    }
    return TTT_OK;
  };
  auto run_update = [&]() -> int {
    const dim3 grid(std::max((dh + 31) / 32, (d + 7) / 8), Z);
    TTT_LAUNCH(TTT_KERNEL_UPDATE, st,
               update_kernel<<<grid, 256, 0, st>>>(M, Ms, Msl, G, n0, g.step, g.wnorm, g.wnorm_eps, d, dh));
    return TTT_OK;
  };
  auto do_update = [&](int ci, int s, int valid) -> int {
    int n_part = 0;
    int r = run_grad(ci, s, valid, n_part);
    if (r != TTT_OK) return r;
    if (g.muon) {
      r = run_ns(n_part);
      if (r != TTT_OK) return r;
    }
    return run_update();
  };

  for (int ci = 0; ci < c.n_chunks; ++ci) {
    const int s = ci * g.chunk;
    const int valid = std::min(g.chunk, T - s);
    const bool upd = call_updates(c, ci);
    if (g.mode == TTT_MODE_SHIFTED) {
      rc = run_fwd(s, valid, true, upd);
      if (rc == TTT_OK) rc = run_o(s, valid);
      if (rc == TTT_OK && upd) rc = do_update(ci, s, valid);
    } else {
      rc = TTT_OK;
      if (upd) {
        rc = run_fwd(s, valid, false, true);
        if (rc == TTT_OK) rc = do_update(ci, s, valid);
      }
      if (rc == TTT_OK) rc = run_fwd(s, valid, true, false);
      if (rc == TTT_OK) rc = run_o(s, valid);
    }
    if (rc != TTT_OK) return rc;
  }
  {
    const dim3 grid((dh + 31) / 32, (d + 31) / 32, Z);
    TTT_LAUNCH(TTT_KERNEL_AUX, st, export_kernel<<<grid, 256, 0, st>>>(M, c.Wf[0], c.Wf[1], c.Wf[2], d, dh));
  }
  return TTT_OK;
}

}  // namespace ttt

// ============================================================ test hook
extern "C" int ttt_dbg_gemm_bf16(const void* A, int a_mn_major, const void* B, int b_mn_major, float* D, int Z,
                                 int M, int N, int K, void* stream) {
  using namespace ttt;
  if (!A || !B || !D || Z < 1 || M < 64 || N < 64 || K < 64 || M % 64 || N % 64 || K % 64) return TTT_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(D)) & 15u)
    return TTT_ERR_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUtensorMap mA, mB;
  bool ok = a_mn_major ? map3(&mA, A, M, K, Z, 64, 64) : map3(&mA, A, K, M, Z, 64, 128);
  ok &= b_mn_major ? map3(&mB, B, N, K, Z, 64, 64) : map3(&mB, B, K, N, Z, 64, 128);
  if (!ok) return TTT_ERR_CUDA;
  const int mt = (M + 127) / 128, nt = (N + 127) / 128;
  const dim3 grid(mt * nt, Z);
  const TcCommon cm{nullptr, 2000000000ull};
  auto go = [&](auto op) -> int {
    using Op = decltype(op);
    typename Op::Params p{};
    p.mA = mA; p.mB = mB; p.D = D; p.M = M; p.N = N; p.K = K; p.m_tiles = mt; p.n_tiles = nt; p.cm = cm;
    return launch_op<Op>(TTT_KERNEL_AUX, p, grid, st);
  };
  if (a_mn_major && b_mn_major) return go(PlainOp<true, true>{});
  if (a_mn_major) return go(PlainOp<true, false>{});
  if (b_mn_major) return go(PlainOp<false, true>{});
  return go(PlainOp<false, false>{});
}
