// Fused Muon step of the tensor-core path: Newton-Schulz orthogonalisation of
// every fast-weight gradient (the LaCT page, "Large Chunk Test-Time Training",
// §2.2.1, eq. 9-10: the gradient turned into an approximately orthogonal
// matrix), then the update W <- W - step*U and the L2 row weight norm (§2.2.1,
// eq. 8), for every matrix of every (batch, head), in ONE cooperative launch.
//
// Matrices are stored in the wide orientation d x dh (d <= dh), z = 3*bh + j.
// Phases, separated by grid-wide barriers (global memory carries the data):
//   normalise  X0 = G / (||G||_F + eps)                 (SIMT; rows of each matrix
//                                                         split over a group of CTAs)
//   5 x { gram  R = X X^T + beta I         d x d,  K = dh   (tcgen05)
//         poly  P = c R R + alpha I        d x d,  K = d    (tcgen05; R is symmetric)
//         xupd  X <- P X                   d x dh, K = d    (tcgen05) }
// The quintic step X <- (a I + b S + c S^2) X with S = X X^T is written with its
// square completed, a + b s + c s^2 = c (s + beta)^2 + alpha, beta = b / (2c),
// alpha = a - b^2 / (4c): one symmetric operand R feeds both sides of the
// second product, and no epilogue reads an fp32 matrix back from memory.
//   update     M <- M - step*U; rows of W1, W2, W3 back to their W0 norms   (SIMT)
// The tiles of all matrices are spread over every SM. Inside the GEMM phases
// each CTA is a persistent warp-specialised engine:
//   warp 0 (one lane)  TMA producer over a shared-memory ring;
//   warp 1 (one lane)  tcgen05.mma issuer into one of two TMEM accumulators;
//   warps 2..5         epilogue (TMEM -> registers -> fused math -> global),
// so the epilogue of one tile overlaps the MMAs of the next. Operand precision:
// SPLIT carries X, S, T and P as bf16 (hi, lo) pairs, loads both halves of both
// operands once per stage and forms each product from three MMAs
// (hi*hi + hi*lo + lo*hi); SINGLE uses one fp16 operand.
// Every wait (mbarriers, grid barriers) is bounded (timeout -> status word, no
// trap); after an abort every thread still passes every barrier and skips the work.
#include <algorithm>
#include <cstring>

#include "tc_kernel.cuh"
#include "tc_util.cuh"
#include "ttt_internal.h"
#include "ttt_ns.h"

namespace ttt {
namespace {

using namespace tcu;

constexpr int kNsThreads = 192;
constexpr int kAccCols = 256;  // columns of one TMEM accumulator buffer
constexpr int kMaxGroup = 16;  // CTAs sharing one matrix in the element-wise phases

enum { PH_GRAM = 0, PH_POLY = 1, PH_XUPD = 2 };

struct NsParams {
  CUtensorMap mXa[2][2];  // X operand [ping-pong][hi, lo]: {dh, d, Z}, box {32, 128}, 64-byte swizzle
  CUtensorMap mXb[2][2];  //   box {32, BNS}, 64-byte swizzle  (Gram B operand, K-major)
  CUtensorMap mXm[2][2];  //   box {64, 32}, 128-byte swizzle  (X update B operand, MN-major)
  CUtensorMap mRa[2];          // R operand [hi, lo]: {d, d, Z}, box {32, 128}, 64-byte swizzle
  CUtensorMap mRb[2];          //   box {32, BNS}
  CUtensorMap mPa[2];          // P operand [hi, lo]: {d, d, Z}, box {32, 128}
  float* X;         // [Z][d][dh] fp32: the gradient on entry, the result U on exit
  void* Xop[2][2];  // operand copies of X [ping-pong][hi, lo]
  void* Rop[2];
  void* Pop[2];
  float* M;         // [Z][d][dh] fp32 master weights (M1 = W1^T, M2 = W2, M3 = W3^T)
  bf16* Ms;         // bf16 shadow (hi)
  bf16* Msl;        // bf16 shadow (lo) or nullptr
  const float* n0;  // [Z][dh] reference row norms
  float* nsq;       // [Z][gs] partial sums of squares
  float* colpart;   // [Z][gs][dh] partial column sums of squares
  unsigned* bar;    // grid-barrier counter (zeroed before the launch)
  float alpha, beta, c, eps, step, wnorm_eps;
  int Z, d, dh, iters, gs, wnorm;
  TcCommon cm;
};

// Shared-memory ring. SPLIT stages hold both halves of both operands
// [A hi | A lo | B hi | B lo], so one load serves all three products; SINGLE
// stages hold [A | B].
// Stages hold 32 elements of K: K-major operands in the 64-byte swizzle (rows
// of 64 B, 8-row atoms of 512 B), the MN-major X operand of the update in
// 128-byte-swizzled boxes of 64 x 32. Small stages keep more of the ring in
// flight: four stages of 48 KB (SPLIT) or eight of 24 KB.
constexpr int kNsBK = 32;
constexpr uint32_t kNsABytes = BM * kNsBK * 2;       // 8 KB: 128 rows x 64 B
constexpr uint32_t kNsMNBox = 64 * kNsBK * 2;        // 4 KB: one 64 x 32 MN-major box

template <int BNS, int BNX, bool SPLIT>
struct NsGeom {
  static constexpr int kOps = SPLIT ? 2 : 1;
  static constexpr int kBmax = BNS > BNX ? BNS : BNX;
  static constexpr uint32_t kBBytes = (uint32_t)kBmax * kNsBK * 2;
  static constexpr uint32_t kStageBytes = kOps * (kNsABytes + kBBytes);
  static constexpr int kStages = SPLIT ? 4 : 8;
  static constexpr size_t kSmem = (size_t)kStages * kStageBytes + 1024 + 512;
};

// K-major operand in the 64-byte swizzle; K step kk of 16 elements
__device__ __forceinline__ uint64_t kdesc64(uint32_t base, int kk) { return ptx::sdesc_l(base + kk * 32, 16, 512, 4); }
// MN-major operand: 64-wide groups kNsMNBox apart, 128-byte swizzle; K step kk
__device__ __forceinline__ uint64_t mdesc32(uint32_t base, int kk) {
  return ptx::sdesc_l(base + kk * 2048, kNsMNBox, 1024, 2);
}

struct PhaseDesc {
  int mt, nt, nk1, bn;
};

template <int BNS, int BNX>
__device__ __forceinline__ PhaseDesc phase_desc(const NsParams& p, int kind) {
  PhaseDesc q;
  q.mt = (p.d + BM - 1) / BM;
  if (kind == PH_XUPD) {
    q.nt = p.dh / BNX;
    q.nk1 = p.d / kNsBK;
    q.bn = BNX;
  } else {
    q.nt = (p.d + BNS - 1) / BNS;
    q.nk1 = (kind == PH_GRAM ? p.dh : p.d) / kNsBK;
    q.bn = BNS;
  }
  return q;
}

__device__ __forceinline__ float ldcg(const float* p) { return __ldcg(p); }

__device__ __forceinline__ float bf_rest(float x) { return x - __bfloat162float(__float2bfloat16_rn(x)); }

// Four consecutive values as operands: bf16 (hi, lo) pairs (SPLIT) or fp16.
template <bool SPLIT>
__device__ __forceinline__ void st_op4(void* hi, void* lo, size_t o, float4 v) {
  if (SPLIT) {
    uint2 h, l;
    h.x = pack_bf16(v.x, v.y);
    h.y = pack_bf16(v.z, v.w);
    l.x = pack_bf16(bf_rest(v.x), bf_rest(v.y));
    l.y = pack_bf16(bf_rest(v.z), bf_rest(v.w));
    *reinterpret_cast<uint2*>(static_cast<bf16*>(hi) + o) = h;
    *reinterpret_cast<uint2*>(static_cast<bf16*>(lo) + o) = l;
  } else {
    uint2 h;
    h.x = pack_f16(v.x, v.y);
    h.y = pack_f16(v.z, v.w);
    *reinterpret_cast<uint2*>(static_cast<f16*>(hi) + o) = h;
  }
}

__device__ __forceinline__ float4 ldcg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

__device__ __forceinline__ float4 axpy4(float4 m, float s, float4 u) {
  return make_float4(m.x - s * u.x, m.y - s * u.y, m.z - s * u.z, m.w - s * u.w);
}

__device__ __forceinline__ float4 scale4(float4 v, float s) { return make_float4(v.x * s, v.y * s, v.z * s, v.w * s); }

__device__ __forceinline__ float sumsq4(float4 v, float acc) {
  return fmaf(v.w, v.w, fmaf(v.z, v.z, fmaf(v.y, v.y, fmaf(v.x, v.x, acc))));
}

constexpr int kUnroll = 4;  // independent 16-byte loads in flight per thread in the SIMT phases

// Deterministic block-wide sum (192 threads): warp butterflies, then the six
// warp totals in warp order. Every thread gets the result.
__device__ __forceinline__ float block_sum(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kNsThreads / 32; ++w) t += red[w];
  return t;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of a cooperative launch (every thread calls it). Thread 0
// publishes the CTA's writes and waits, bounded, for every CTA's arrival;
// afterwards every thread sees an error recorded anywhere in the grid.
__device__ __forceinline__ void grid_barrier(const NsParams& p, unsigned& n_bar, volatile int* abort_flag) {
  __syncwarp();
  __syncthreads();
  ++n_bar;
  if (threadIdx.x == 0) {
    const unsigned target = n_bar * gridDim.x;
    __threadfence();
    atomicAdd(p.bar, 1u);
    if (!*abort_flag) {
      const uint64_t t0 = globaltimer_ns();
      uint32_t it = 0;
      while (ld_acquire_gpu(p.bar) < target) {
        if ((++it & 63u) == 0) {
          if (*reinterpret_cast<volatile int*>(p.cm.status) != 0) break;
          if (globaltimer_ns() - t0 > p.cm.timeout_ns) {
            set_status(p.cm.status, TTT_ERR_TIMEOUT);
            break;
          }
        }
      }
    }
    __threadfence();
    if (*reinterpret_cast<volatile int*>(p.cm.status) != 0) *abort_flag = 1;
  }
  __syncthreads();
  ptx::fence_proxy_async_global();  // later TMA reads see the data the barrier published
}

template <int BNS, int BNX, bool SPLIT>
__global__ void __launch_bounds__(kNsThreads, 1) ns_fused_kernel(const __grid_constant__ NsParams p) {
  using Geo = NsGeom<BNS, BNX, SPLIT>;
  constexpr int kNsStages = Geo::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kNsStages * Geo::kStageBytes);
  uint64_t* empty = full + kNsStages;
  uint64_t* accf = empty + kNsStages;
  uint64_t* acce = accf + 2;
  uint64_t* drainb = acce + 2;  // MMAs in flight at an abort
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drainb + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  float* red = reinterpret_cast<float*>(tslot + 4);  // 8 floats

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = p.d, dh = p.dh, Z = p.Z;
  const int G = (int)gridDim.x;
  unsigned n_bar = 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNsStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&accf[s], 1);
      ptx::mbar_init(&acce[s], 4);  // one arrival per epilogue warp
    }
    ptx::mbar_init(drainb, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tslot, 2 * kAccCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tslot;

  // SIMT phases: matrix z is split by rows over `gs` members (z, k); work item
  // i = k * Z + z belongs to CTA i % G (several items per CTA when Z > G)
  const int gs = p.gs;
  const int rows_per = (d + gs - 1) / gs;
  const int n_items = Z * gs;

  // ---------------------------------------------------------------- normalise
  for (int i = blockIdx.x; i < n_items; i += G) {
    const int z = i % Z, k = i / Z;
    const int r0 = min(d, k * rows_per), r1 = min(d, r0 + rows_per);
    const float* g = p.X + (size_t)z * d * dh + (size_t)r0 * dh;
    const int n4 = (r1 - r0) * dh / 4;
    float ss = 0.f;
    if (!*abort_flag)
      for (int b = threadIdx.x; b < n4; b += kNsThreads * kUnroll) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (b + u * kNsThreads < n4) v[u] = ldcg4(g + 4 * (b + u * kNsThreads));
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (b + u * kNsThreads < n4) ss = sumsq4(v[u], ss);
      }
    ss = block_sum(ss, red);
    if (threadIdx.x == 0) p.nsq[(size_t)z * gs + k] = ss;
  }
  grid_barrier(p, n_bar, abort_flag);
  for (int i = blockIdx.x; i < n_items; i += G) {
    const int z = i % Z, k = i / Z;
    const int r0 = min(d, k * rows_per), r1 = min(d, r0 + rows_per);
    const size_t base = (size_t)z * d * dh + (size_t)r0 * dh;
    const int n4 = (r1 - r0) * dh / 4;
    float tot = 0.f;
    for (int q = 0; q < gs; ++q) tot += ldcg(p.nsq + (size_t)z * gs + q);
    const float inv = 1.f / (sqrtf(tot) + p.eps);
    if (!*abort_flag)
      for (int b = threadIdx.x; b < n4; b += kNsThreads * kUnroll) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (b + u * kNsThreads < n4) v[u] = ldcg4(p.X + base + 4 * (b + u * kNsThreads));
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (b + u * kNsThreads < n4) {
            const size_t o = base + 4 * (size_t)(b + u * kNsThreads);
            const float4 x = scale4(v[u], inv);
            *reinterpret_cast<float4*>(p.X + o) = x;
            st_op4<SPLIT>(p.Xop[0][0], p.Xop[0][1], o, x);
          }
      }
  }
  ptx::fence_proxy_async_global();
  grid_barrier(p, n_bar, abort_flag);

  // ---------------------------------------------------------------- GEMM phases
  // tiles of every matrix are spread over the whole grid: tile t -> CTA t % G
  uint32_t pc = 0;   // producer: k-blocks issued
  uint32_t mc = 0;   // MMA: k-blocks consumed
  uint32_t at = 0;   // MMA: tiles accumulated
  uint32_t et = 0;   // epilogue: tiles drained
  for (int it = 0; it < p.iters; ++it) {
    const int cur = it & 1;
    for (int kind = 0; kind < 3; ++kind) {
      const PhaseDesc q = phase_desc<BNS, BNX>(p, kind);
      const int per_z = q.mt * q.nt;
      const int n_tiles = Z * per_z;
      const int nkb = q.nk1;
      if (warp == 0) {
        if (lane == 0 && !*abort_flag) {
          const uint32_t tx = Geo::kOps * (kNsABytes + (uint32_t)q.bn * kNsBK * 2);
          for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += G) {
            const int z = t / per_z, tl = t % per_z;
            const int m0 = (tl / q.nt) * BM, n0 = (tl % q.nt) * q.bn;
            for (int kb = 0; kb < nkb; ++kb) {
              const int s = pc % kNsStages;
              if (!tc_wait(&empty[s], ((pc / kNsStages) & 1u) ^ 1u, p.cm, abort_flag)) break;
              uint8_t* st = smem + (size_t)s * Geo::kStageBytes;
              ptx::mbar_expect_tx(&full[s], tx);
              const int k = kb * kNsBK;
              for (int h = 0; h < Geo::kOps; ++h) {
                uint8_t* sa = st + h * kNsABytes;
                uint8_t* sb = st + Geo::kOps * kNsABytes + h * Geo::kBBytes;
                if (kind == PH_GRAM) {
                  ptx::tma_load_3d(sa, &p.mXa[cur][h], &full[s], k, m0, z);
                  ptx::tma_load_3d(sb, &p.mXb[cur][h], &full[s], k, n0, z);
                } else if (kind == PH_POLY) {
                  ptx::tma_load_3d(sa, &p.mRa[h], &full[s], k, m0, z);
                  ptx::tma_load_3d(sb, &p.mRb[h], &full[s], k, n0, z);
                } else {
                  ptx::tma_load_3d(sa, &p.mPa[h], &full[s], k, m0, z);
                  for (int g = 0; g < BNX / 64; ++g)
                    ptx::tma_load_3d(sb + g * kNsMNBox, &p.mXm[cur][h], &full[s], n0 + g * 64, k, z);
                }
              }
              ++pc;
            }
          }
        }
      } else if (warp == 1) {
        if (lane == 0 && !*abort_flag) {
          for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += G) {
            const uint32_t acc = at & 1u;
            if (!tc_wait(&acce[acc], ((at >> 1) & 1u) ^ 1u, p.cm, abort_flag)) break;
            ptx::tc_fence_after();
            const uint32_t dt = tmem + acc * kAccCols;
            bool ok = true;
            for (int kb = 0; kb < nkb; ++kb) {
              const int s = mc % kNsStages;
              if (!tc_wait(&full[s], (mc / kNsStages) & 1u, p.cm, abort_flag)) { ok = false; break; }
              ptx::tc_fence_after();
              // [A hi, A lo] at sa0, sa0 + kABytes; [B hi, B lo] at sb0, sb0 + kBBytes
              const uint32_t sa0 = ptx::smem_u32(smem + (size_t)s * Geo::kStageBytes);
              const uint32_t sb0 = sa0 + Geo::kOps * kNsABytes;
              // products: hi*hi, then (SPLIT) hi*lo and lo*hi
              constexpr int kProd = SPLIT ? 3 : 1;
#pragma unroll
              for (int pr = 0; pr < kProd; ++pr) {
                const uint32_t sa = sa0 + (pr == 2 ? kNsABytes : 0u);
                const uint32_t sb = sb0 + (pr == 1 ? Geo::kBBytes : 0u);
                if (kind == PH_XUPD) {
                  constexpr uint32_t id = ptx::idesc_bf16(128, BNX, false, true, !SPLIT);
#pragma unroll
                  for (int kk = 0; kk < kNsBK / 16; ++kk)
                    ptx::mma_bf16(dt, kdesc64(sa, kk), mdesc32(sb, kk), id, (kb | kk | pr) != 0);
                } else {
                  constexpr uint32_t id = ptx::idesc_bf16(128, BNS, false, false, !SPLIT);
#pragma unroll
                  for (int kk = 0; kk < kNsBK / 16; ++kk)
                    ptx::mma_bf16(dt, kdesc64(sa, kk), kdesc64(sb, kk), id, (kb | kk | pr) != 0);
                }
              }
              ptx::mma_commit(&empty[s]);
              ++mc;
            }
            if (!ok) break;
            ptx::mma_commit(&accf[acc]);
            ++at;
          }
        }
      } else {
        const int g = warp & 3;  // TMEM lane group of this warp
        const int r = 32 * g + lane;
        const bool last = it + 1 == p.iters;
        for (int t = blockIdx.x; t < n_tiles; t += G) {
          if (*abort_flag) break;  // uniform within the warp (read after a barrier or a wait)
          const uint32_t acc = et & 1u;
          int ok = 0;
          if (lane == 0) ok = tc_wait(&accf[acc], (et >> 1) & 1u, p.cm, abort_flag) && !*abort_flag;
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          ptx::tc_fence_after();
          const int z = t / per_z, tl = t % per_z;
          const uint32_t ta = tmem + acc * kAccCols + ((uint32_t)(32 * g) << 16);
          const int m = (tl / q.nt) * BM + r, n0 = (tl % q.nt) * q.bn;
          const bool row_ok = m < d;
          float v[32];
          for (int c = 0; c < q.bn; c += 32) {
            ptx::tmem_ld32(ta + c, v);
            const int n = n0 + c;
            // warp-uniform: n, and whether this is the last iteration
            if (kind == PH_GRAM) {
              if (n < d) {
                const size_t o = ((size_t)z * d + m) * d + n;
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] += (m == n + i ? p.beta : 0.f);
                if (row_ok) st_op32<SPLIT>(p.Rop[0], p.Rop[1], o, v);
              }
            } else if (kind == PH_POLY) {
              if (n < d) {
                const size_t o = ((size_t)z * d + m) * d + n;
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = p.c * v[i] + (m == n + i ? p.alpha : 0.f);
                if (row_ok) st_op32<SPLIT>(p.Pop[0], p.Pop[1], o, v);
              }
            } else {
              const size_t o = (size_t)z * d * dh + (size_t)m * dh + n;
              if (last) {
                if (row_ok) st_f32x32(p.X + o, v);
              } else {
                if (row_ok) st_op32<SPLIT>(p.Xop[cur ^ 1][0], p.Xop[cur ^ 1][1], o, v);
              }
            }
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&acce[acc]);
          ++et;
        }
        ptx::fence_proxy_async_global();
      }
      grid_barrier(p, n_bar, abort_flag);
    }
  }

  // ---------------------------------------------------------------- update + weight norm
  // pass 1: M <- M - step*U (rows of W2 renormalised at once; partial column
  // sums of W1 / W3 published); pass 2 (after a grid barrier): column scales.
  // Every loop keeps kUnroll independent 16-byte loads in flight per thread.
  for (int pass = 0; pass < 2; ++pass) {
    for (int i = blockIdx.x; i < n_items; i += G) {
      const int z = i % Z, k = i / Z, j = z % 3;
      const int r0 = min(d, k * rows_per), r1 = min(d, r0 + rows_per);
      const size_t zoff = (size_t)z * d * dh;
      const float* u = p.X + zoff;
      float* mm = p.M + zoff;
      const float* n0 = p.n0 + (size_t)z * dh;
      // M and its bf16 shadow(s) at element offset e (4 consecutive values)
      auto put4 = [&](size_t e, float4 x) {
        *reinterpret_cast<float4*>(mm + e) = x;
        uint2 h;
        h.x = pack_bf16(x.x, x.y);
        h.y = pack_bf16(x.z, x.w);
        *reinterpret_cast<uint2*>(p.Ms + zoff + e) = h;
        if (p.Msl) {
          uint2 l;
          l.x = pack_bf16(bf_rest(x.x), bf_rest(x.y));
          l.y = pack_bf16(bf_rest(x.z), bf_rest(x.w));
          *reinterpret_cast<uint2*>(p.Msl + zoff + e) = l;
        }
      };
      if (*abort_flag) continue;
      if (!p.wnorm) {
        if (pass == 0) {
          const int n4 = (r1 - r0) * dh / 4;
          const size_t e0 = (size_t)r0 * dh;
          for (int b = threadIdx.x; b < n4; b += kNsThreads * kUnroll) {
            float4 mv[kUnroll], uv[kUnroll];
#pragma unroll
            for (int q = 0; q < kUnroll; ++q)
              if (b + q * kNsThreads < n4) {
                const size_t e = e0 + 4 * (size_t)(b + q * kNsThreads);
                mv[q] = ldcg4(mm + e);
                uv[q] = ldcg4(u + e);
              }
#pragma unroll
            for (int q = 0; q < kUnroll; ++q)
              if (b + q * kNsThreads < n4) put4(e0 + 4 * (size_t)(b + q * kNsThreads), axpy4(mv[q], p.step, uv[q]));
          }
        }
      } else if (j == 1) {
        // rows of W2 are rows of M2: one warp per row, lanes over 16-byte groups
        if (pass == 0)
          for (int row = r0 + warp; row < r1; row += kNsThreads / 32) {
            const size_t base = (size_t)row * dh;
            const int n4 = dh / 4;
            float ss = 0.f;
            for (int b = lane; b < n4; b += 32 * kUnroll) {
              float4 mv[kUnroll], uv[kUnroll];
#pragma unroll
              for (int q = 0; q < kUnroll; ++q)
                if (b + 32 * q < n4) {
                  mv[q] = ldcg4(mm + base + 4 * (b + 32 * q));
                  uv[q] = ldcg4(u + base + 4 * (b + 32 * q));
                }
#pragma unroll
              for (int q = 0; q < kUnroll; ++q)
                if (b + 32 * q < n4) ss = sumsq4(axpy4(mv[q], p.step, uv[q]), ss);
            }
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float sc = n0[row] / fmaxf(sqrtf(ss), p.wnorm_eps);
            for (int b = lane; b < n4; b += 32 * kUnroll) {
              float4 mv[kUnroll], uv[kUnroll];
#pragma unroll
              for (int q = 0; q < kUnroll; ++q)
                if (b + 32 * q < n4) {
                  mv[q] = ldcg4(mm + base + 4 * (b + 32 * q));
                  uv[q] = ldcg4(u + base + 4 * (b + 32 * q));
                }
#pragma unroll
              for (int q = 0; q < kUnroll; ++q)
                if (b + 32 * q < n4) put4(base + 4 * (b + 32 * q), scale4(axpy4(mv[q], p.step, uv[q]), sc));
            }
          }
      } else {
        // rows of W1 / W3 are columns of M1 / M3: a thread owns 4 consecutive
        // columns and walks this item's rows
        float* cp = p.colpart + ((size_t)z * gs + k) * dh;
        for (int c4 = threadIdx.x; c4 < dh / 4; c4 += kNsThreads) {
          const int col = 4 * c4;
          if (pass == 0) {
            float4 ss = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int row = r0; row < r1; row += kUnroll) {
              float4 mv[kUnroll], uv[kUnroll];
#pragma unroll
              for (int q = 0; q < kUnroll; ++q)
                if (row + q < r1) {
                  mv[q] = ldcg4(mm + (size_t)(row + q) * dh + col);
                  uv[q] = ldcg4(u + (size_t)(row + q) * dh + col);
                }
#pragma unroll
              for (int q = 0; q < kUnroll; ++q)
                if (row + q < r1) {
                  const float4 x = axpy4(mv[q], p.step, uv[q]);
                  *reinterpret_cast<float4*>(mm + (size_t)(row + q) * dh + col) = x;
                  ss.x = fmaf(x.x, x.x, ss.x); ss.y = fmaf(x.y, x.y, ss.y);
                  ss.z = fmaf(x.z, x.z, ss.z); ss.w = fmaf(x.w, x.w, ss.w);
                }
            }
            *reinterpret_cast<float4*>(cp + col) = ss;
          } else {
            float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int q = 0; q < gs; ++q) {
              const float4 v = ldcg4(p.colpart + ((size_t)z * gs + q) * dh + col);
              tot.x += v.x; tot.y += v.y; tot.z += v.z; tot.w += v.w;
            }
            const float4 nn = *reinterpret_cast<const float4*>(n0 + col);
            const float4 sc = make_float4(nn.x / fmaxf(sqrtf(tot.x), p.wnorm_eps), nn.y / fmaxf(sqrtf(tot.y), p.wnorm_eps),
                                          nn.z / fmaxf(sqrtf(tot.z), p.wnorm_eps), nn.w / fmaxf(sqrtf(tot.w), p.wnorm_eps));
            for (int row = r0; row < r1; row += kUnroll) {
              float4 mv[kUnroll];
#pragma unroll
              for (int q = 0; q < kUnroll; ++q)
                if (row + q < r1) mv[q] = ldcg4(mm + (size_t)(row + q) * dh + col);
#pragma unroll
              for (int q = 0; q < kUnroll; ++q)
                if (row + q < r1)
                  put4((size_t)(row + q) * dh + col,
                       make_float4(mv[q].x * sc.x, mv[q].y * sc.y, mv[q].z * sc.z, mv[q].w * sc.w));
            }
          }
        }
      }
    }
    if (pass == 0) grid_barrier(p, n_bar, abort_flag);
  }

  // ---------------------------------------------------------------- teardown
  if (warp == 0 && lane == 0 && *abort_flag) {
    // the copies this thread started must land before the CTA exits
    for (uint32_t k = pc > (uint32_t)kNsStages ? pc - kNsStages : 0; k < pc; ++k)
      tc_drain(&full[k % kNsStages], (k / kNsStages) & 1u, p.cm);
  }
  if (warp == 1 && lane == 0 && *abort_flag) {
    // and the MMAs this thread issued must finish before TMEM is freed
    ptx::mma_commit(drainb);
    tc_drain(drainb, 0, p.cm);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, 2 * kAccCols);
}

// Grid of the cooperative launch: every CTA resident at once (one per SM at
// this shared-memory size), capped by the work there is.
template <int BNS, int BNX, bool SPLIT>
int grid_size(int* resident) {
  auto kern = ns_fused_kernel<BNS, BNX, SPLIT>;
  const size_t smem = NsGeom<BNS, BNX, SPLIT>::kSmem;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return -1;
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kNsThreads, smem) != cudaSuccess)
    return -1;
  if (resident) *resident = sms * per_sm;
  return sms * per_sm;
}

int g_forced_grid = 0;  // test hook: 0 = every SM, else this many CTAs

template <int BNS, int BNX, bool SPLIT>
int launch_ns(NsParams& p, cudaStream_t st) {
  auto kern = ns_fused_kernel<BNS, BNX, SPLIT>;
  const size_t smem = NsGeom<BNS, BNX, SPLIT>::kSmem;
  int G = grid_size<BNS, BNX, SPLIT>(nullptr);
  if (G <= 0) return TTT_ERR_CUDA;
  if (g_forced_grid > 0 && g_forced_grid < G) G = g_forced_grid;
  p.gs = std::max(1, std::min(kMaxGroup, G / p.Z));
  if (cudaMemsetAsync(p.bar, 0, sizeof(unsigned), st) != cudaSuccess) return TTT_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kNsThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  prof_before(TTT_KERNEL_NS, st);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  prof_after(TTT_KERNEL_NS, st);
  return e == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

}  // namespace

bool ns_fused_supported(const ttt_cfg& g) { return g.d % 64 == 0 && g.dh % 128 == 0 && g.d <= g.dh; }

void ns_force_grid(int ctas) { g_forced_grid = ctas; }

int ns_build_params(const NsFusedArgs& a, NsParams& p);

namespace {

// Everything the launch parameters are built from: the 18 tensor maps are
// encoded once and reused while a call's chunks (and later calls on the same
// buffers) launch with the same arguments.
struct NsKey {
  const void* ptrs[16];
  float coef[6];
  int ints[6];
};

NsKey ns_key(const NsFusedArgs& a) {
  NsKey k;
  std::memset(&k, 0, sizeof(k));
  const void* ps[16] = {a.X, a.Xh[0], a.Xh[1], a.Xl[0], a.Xl[1], a.Rh, a.Rl, a.Ph, a.Pl, a.M, a.Ms, a.Msl,
                        a.n0, a.scratch, a.cm.status, nullptr};
  for (int i = 0; i < 16; ++i) k.ptrs[i] = ps[i];
  const ttt_cfg& g = *a.cfg;
  const float cf[6] = {g.ns_a, g.ns_b, g.ns_c, g.ns_eps, g.step, g.wnorm_eps};
  for (int i = 0; i < 6; ++i) k.coef[i] = cf[i];
  const int in[6] = {a.Z, g.d, g.dh, g.ns_iters, g.wnorm, a.split ? 1 : 0};
  for (int i = 0; i < 6; ++i) k.ints[i] = in[i];
  return k;
}

thread_local NsKey t_key;
thread_local NsParams t_params;
thread_local bool t_have = false;

}  // namespace

int ns_fused_run(const NsFusedArgs& a, cudaStream_t st) {
  const ttt_cfg& g = *a.cfg;
  const int d = g.d, dh = g.dh, Z = a.Z;
  const bool split = a.split;
  const int bns = (d % 256 == 0) ? 256 : 128;
  const int bnx = (dh % 256 == 0) ? 256 : 128;
  const NsKey key = ns_key(a);
  if (!t_have || std::memcmp(&key, &t_key, sizeof(key)) != 0) {
    t_have = false;
    if (ns_build_params(a, t_params) != TTT_OK) return TTT_ERR_CUDA;
    t_key = key;
    t_have = true;
  }
  NsParams p = t_params;
  p.cm = a.cm;
#define TTT_NS_LAUNCH(BS, BX)                                                        \
  if (bns == BS && bnx == BX)                                                        \
    return split ? launch_ns<BS, BX, true>(p, st) : launch_ns<BS, BX, false>(p, st);
  TTT_NS_LAUNCH(256, 256)
  TTT_NS_LAUNCH(128, 256)
  TTT_NS_LAUNCH(128, 128)
  TTT_NS_LAUNCH(256, 128)
#undef TTT_NS_LAUNCH
  return TTT_ERR_UNSUPPORTED;
}

int ns_build_params(const NsFusedArgs& a, NsParams& p) {
  const ttt_cfg& g = *a.cfg;
  const int d = g.d, dh = g.dh, Z = a.Z;
  const bool split = a.split;
  const CUtensorMapDataType dt = split ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int bns = (d % 256 == 0) ? 256 : 128;
  p = NsParams{};
  bool ok = true;
  for (int i = 0; i < 2; ++i)
    for (int h = 0; h < 2; ++h) {
      const void* b = (h && split) ? a.Xl[i] : a.Xh[i];
      ok &= map3(&p.mXa[i][h], b, dh, d, Z, kNsBK, 128, dt, CU_TENSOR_MAP_SWIZZLE_64B);
      ok &= map3(&p.mXb[i][h], b, dh, d, Z, kNsBK, bns, dt, CU_TENSOR_MAP_SWIZZLE_64B);
      ok &= map3(&p.mXm[i][h], b, dh, d, Z, 64, kNsBK, dt);
      p.Xop[i][h] = const_cast<void*>(b);
    }
  for (int h = 0; h < 2; ++h) {
    const void* rb = (h && split) ? a.Rl : a.Rh;
    const void* pb = (h && split) ? a.Pl : a.Ph;
    ok &= map3(&p.mRa[h], rb, d, d, Z, kNsBK, 128, dt, CU_TENSOR_MAP_SWIZZLE_64B);
    ok &= map3(&p.mRb[h], rb, d, d, Z, kNsBK, bns, dt, CU_TENSOR_MAP_SWIZZLE_64B);
    ok &= map3(&p.mPa[h], pb, d, d, Z, kNsBK, 128, dt, CU_TENSOR_MAP_SWIZZLE_64B);
    p.Rop[h] = const_cast<void*>(rb);
    p.Pop[h] = const_cast<void*>(pb);
  }
  if (!ok) return TTT_ERR_CUDA;
  p.X = a.X;
  p.M = a.M;
  p.Ms = static_cast<bf16*>(a.Ms);
  p.Msl = static_cast<bf16*>(a.Msl);
  p.n0 = a.n0;
  p.nsq = a.scratch;
  p.colpart = a.scratch + (size_t)Z * kMaxGroup;
  p.bar = reinterpret_cast<unsigned*>(p.colpart + (size_t)Z * kMaxGroup * dh);
  // a + b s + c s^2 = c (s + beta)^2 + alpha
  p.c = g.ns_c;
  p.beta = g.ns_b / (2.f * g.ns_c);
  p.alpha = g.ns_a - g.ns_b * g.ns_b / (4.f * g.ns_c);
  p.eps = g.ns_eps;
  p.step = g.step; p.wnorm_eps = g.wnorm_eps; p.wnorm = g.wnorm;
  p.Z = Z; p.d = d; p.dh = dh; p.iters = g.ns_iters;
  p.cm = a.cm;
  return TTT_OK;
}

int ns_fused_plan(const ttt_cfg& g, int* resident) {
  const bool split = g.precision == TTT_PREC_SPLIT;
  const int bns = (g.d % 256 == 0) ? 256 : 128;
  const int bnx = (g.dh % 256 == 0) ? 256 : 128;
#define TTT_NS_PLAN(BS, BX)                                                                       \
  if (bns == BS && bnx == BX)                                                                     \
    return split ? grid_size<BS, BX, true>(resident) : grid_size<BS, BX, false>(resident);
  TTT_NS_PLAN(256, 256)
  TTT_NS_PLAN(128, 256)
  TTT_NS_PLAN(128, 128)
  TTT_NS_PLAN(256, 128)
#undef TTT_NS_PLAN
  return -1;
}

size_t ns_fused_scratch_floats(const ttt_cfg& g, int Z) {
  // per-member partial sums (norm and column norms), then the barrier counter
  return (size_t)Z * kMaxGroup * (1 + (size_t)g.dh) + 64;
}

}  // namespace ttt
