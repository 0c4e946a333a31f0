// Fused Muon step of the tensor-core path: Newton-Schulz orthogonalisation of
// every fast-weight gradient (the LaCT page, "Large Chunk Test-Time Training",
// §2.2.1, eq. 9-10: the gradient turned into an approximately orthogonal
// matrix), then the update W <- W - step*U and the L2 row weight norm (§2.2.1,
// eq. 8), for every matrix of every (batch, head): one launch for Newton-Schulz
// and the update, one for the weight norm.
//
// Matrices are stored in the wide orientation d x dh (d <= dh), z = 3*bh + j.
// Phases of one matrix (global memory carries the data between them):
//   norm1   sum of squares of G (or of the momentum buffer B <- mu B + G)    SIMT
//   norm2   X0 = G / (||G||_F + eps) as MMA operands                            SIMT
//   5 x { gram  R = X X^T + beta I         d x d,  K = dh                       tcgen05
//         poly  P = c R R + alpha I        d x d,  K = d   (R is symmetric)     tcgen05
//         xupd  X <- P X                   d x dh, K = d                        tcgen05 }
// then, in a second launch (ns_wnorm_kernel), the rows of W1, W2, W3 back to
// their W0 norms and the bf16 shadows.
// The quintic step X <- (a I + b S + c S^2) X with S = X X^T is written with its
// square completed, a + b s + c s^2 = c (s + beta)^2 + alpha, beta = b / (2c),
// alpha = a - b^2 / (4c): one symmetric operand R feeds both sides of the
// second product, and no epilogue reads an fp32 matrix back from memory. The
// update M <- M - step*U is fused into the last X update's epilogue, with
// partial sums of squares of the new weight rows for the weight norm.
//
// Scheduling (dataflow, no grid-wide barrier): a matrix's items of one phase
// need every item of that matrix's earlier phases, and nothing else. Each
// finished item adds one arrival per epilogue warp to its matrix's completion
// counter, and an item starts once the counter has reached the arrivals of the
// phases before it. The items form one list in (phase, matrix, tile) order,
// dealt round-robin to the CTAs (item g to CTA g % grid), so one matrix's
// phase spreads over as many CTAs as it has tiles. (Measured on the language
// model workload: matrices pinned to their own CTA groups, and items claimed
// dynamically from a global counter, were both slower.) Every CTA is resident
// (cooperative launch), walks its items in list order and only waits on
// earlier items, so the earliest unfinished item can always run: no deadlock.
//
// Inside a CTA the roles are warp-specialised:
//   warp 0 (one lane)  TMA producer over a shared-memory ring (waits on the
//                      completion counters before an item's loads);
//   warp 1 (one lane)  tcgen05.mma issuer into one of two TMEM accumulators;
//   warps 2..9         epilogue (TMEM -> registers -> fused math -> TMA stores),
//                      two warps per TMEM lane quarter, each half of the columns
// Operand precision: SPLIT carries X, R and P as bf16 (hi, lo) pairs and forms
// each product from three MMAs (hi*hi + hi*lo + lo*hi); SINGLE uses one fp16
// operand. Every wait is bounded (timeout -> status word, no trap); after an
// abort every role stops, in-flight copies and MMAs are drained, TMEM is freed.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "tc_kernel.cuh"
#include "tc_util.cuh"
#include "ttt_internal.h"
#include "ttt_ns.h"

namespace ttt {
namespace {

using namespace tcu;

// Eight epilogue warps, two per TMEM lane quarter: the first four take the
// left half of a tile's columns, the other four the right half.
constexpr int kEpiWarps = 8;
constexpr int kColHalves = kEpiWarps / 4;
constexpr int kNsThreads = 64 + 32 * kEpiWarps;
constexpr int kAccCols = 256;     // columns of one TMEM accumulator buffer
constexpr unsigned kArrivals = kEpiWarps;  // completion-counter arrivals per finished item
#ifndef TTT_NS_EPI_BUFS
#define TTT_NS_EPI_BUFS 1
#endif
#ifndef TTT_NS_SPLIT_STAGES
#define TTT_NS_SPLIT_STAGES 4
#endif
constexpr int kEpiBufs = TTT_NS_EPI_BUFS;  // 4 KB staging buffers per epilogue warp

enum { K_GRAM = 0, K_POLY = 1, K_XUPD = 2 };

struct NsParams {
  CUtensorMap mXa[2][2];  // X operand [ping-pong][hi, lo]: {dh, d, Z}, box {32, 128}, 64-byte swizzle
  CUtensorMap mXb[2][2];  //   box {32, BNS}, 64-byte swizzle  (Gram B operand, K-major)
  CUtensorMap mXm[2][2];  //   box {64, 32}, 128-byte swizzle  (X update B operand, MN-major)
  CUtensorMap mRa[2];     // R operand [hi, lo]: {d, d, Z}, box {32, 128}, 64-byte swizzle
  CUtensorMap mRb[2];     //   box {32, BNS}
  CUtensorMap mPa[2];     // P operand [hi, lo]: {d, d, Z}, box {32, 128}
  // epilogue stores of 32 x 32 blocks from shared memory
  CUtensorMap sR[2];      // R [hi, lo]: {d, d, Z}, box {32, 32}, 64-byte swizzle
  CUtensorMap sP[2];      // P [hi, lo]
  CUtensorMap sX[2][2];   // X operand [ping-pong][hi, lo]: {dh, d, Z}
  CUtensorMap sM;         // fp32 M: {dh, d, Z}, box {32, 32}, 128-byte swizzle
  void* Xop[2][2];  // operand copies of X [ping-pong][hi, lo]
  float* M;         // [Z][d][dh] fp32 master weights (M1 = W1^T, M2 = W2, M3 = W3^T)
  bf16* Ms;         // bf16 shadow (hi)
  bf16* Msl;        // bf16 shadow (lo) or nullptr
  const float* n0;  // [Z][dh] reference row norms (W2: the first d entries)
  float* rowpart;   // [Z][dh / (BNX / 2)][d] partial sums of squares of the rows of M2, one per half column tile
  float* colpart;   // [Z][d / 32][dh] partial sums of squares of the columns of M1 / M3, one per 32 rows
  unsigned* cnt;    // [Z] completion counters (zeroed before the launch)
  // X0's operands are written before the launch. fused: UNSCALED (G, or the
  // momentum buffer), with per-z partial sums of squares nsqg[z][nsq_n]; the
  // first Gram and X update scale their results by 1 / (||G||_F + eps)^2 and
  // 1 / (||G||_F + eps). Otherwise X0 = G / (||G||_F + eps) already.
  int fused;
  const float* nsqg;
  int nsq_n;
  int trace;        // test hook: record per-phase timestamps in g_ns_trace
  int stall;        // test hook: CTA 0 withholds the completion of its first item
  float alpha, beta, c, eps, step, wnorm_eps;
  int Z, d, dh, iters, wnorm;
  int mt, ntS, ntX;  // tiles: 128-row blocks; column tiles of the d x d and d x dh products
  int sym;           // 1: the d x d products compute only tiles that meet the upper triangle
  int nS;            // tiles of one d x d product per matrix
  TcCommon cm;
};
static_assert(sizeof(NsParams) <= 4096, "the launch parameters fit the classic 4 KB limit");

// Shared-memory ring. SPLIT stages hold both halves of both operands
// [A hi | A lo | B hi | B lo], so one load serves all three products; SINGLE
// stages hold [A | B]. Stages hold 32 elements of K: K-major operands in the
// 64-byte swizzle (rows of 64 B, 8-row atoms of 512 B), the MN-major X operand
// of the update in 128-byte-swizzled boxes of 64 x 32. Four stages of 48 KB
// (SPLIT) or eight of 24 KB.
constexpr int kNsBK = 32;
constexpr uint32_t kNsABytes = BM * kNsBK * 2;  // 8 KB: 128 rows x 64 B
constexpr uint32_t kNsMNBox = 64 * kNsBK * 2;   // 4 KB: one 64 x 32 MN-major box

template <int BNS, int BNX, bool SPLIT>
struct NsGeom {
  static constexpr int kOps = SPLIT ? 2 : 1;
  static constexpr int kBmax = BNS > BNX ? BNS : BNX;
  static constexpr uint32_t kBBytes = (uint32_t)kBmax * kNsBK * 2;
  static constexpr uint32_t kStageBytes = kOps * (kNsABytes + kBBytes);
  static constexpr int kStages = SPLIT ? TTT_NS_SPLIT_STAGES : 8;
  // epilogue staging: kEpiBufs 4 KB buffers per epilogue warp (a 32 x 32 block
  // as a bf16 pair, one fp16 operand, or fp32)
  static constexpr uint32_t kEpiBytes = kEpiWarps * kEpiBufs * 4096;
  static constexpr size_t kSmem = (size_t)kStages * kStageBytes + kEpiBytes + 1024 + 512;
};

// K-major operand in the 64-byte swizzle; K step kk of 16 elements
__device__ __forceinline__ uint64_t kdesc64(uint32_t base, int kk) { return ptx::sdesc_l(base + kk * 32, 16, 512, 4); }
// MN-major operand: 64-wide groups kNsMNBox apart, 128-byte swizzle; K step kk
__device__ __forceinline__ uint64_t mdesc32(uint32_t base, int kk) {
  return ptx::sdesc_l(base + kk * 2048, kNsMNBox, 1024, 2);
}

__device__ __forceinline__ float ldcg(const float* p) { return __ldcg(p); }
__device__ __forceinline__ float4 ldcg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 scale4(float4 v, float s) { return make_float4(v.x * s, v.y * s, v.z * s, v.w * s); }
__device__ __forceinline__ float sumsq4(float4 v, float acc) {
  return fmaf(v.w, v.w, fmaf(v.z, v.z, fmaf(v.y, v.y, fmaf(v.x, v.x, acc))));
}

// The transpose of a warp's 32 x 32 block as operands, staged for a TMA store
// in the 64-byte swizzle: lane l holds row l (v[i] = element (l, i)), which is
// column l of the transpose, so it writes element (i, l) of the staged block
// for every i (two bytes per store; the lanes of one store fill one 64-byte
// row, without bank conflicts). SPLIT: bf16 hi at buf, lo at buf + 2048;
// else fp16.
template <bool SPLIT>
__device__ __forceinline__ void stage_op32_t(uint8_t* buf, int lane, const float* v) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const uint32_t off = stage_off64(i, lane >> 3) + 2u * (lane & 7);
    if (SPLIT) {
      const bf16 h = __float2bfloat16_rn(v[i]);
      *reinterpret_cast<bf16*>(buf + off) = h;
      *reinterpret_cast<bf16*>(buf + 2048 + off) = __float2bfloat16_rn(v[i] - __bfloat162float(h));
    } else {
      *reinterpret_cast<f16*>(buf + off) = __float2half_rn(v[i]);
    }
  }
}

__device__ __forceinline__ void stage_f32x32(uint8_t* buf, int lane, const float* v) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    *reinterpret_cast<float4*>(buf + 128u * lane + 16u * (q ^ (lane & 7))) =
        make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// Column sums over a warp: each lane holds 32 values (columns n..n+31 of its
// row); afterwards a[0] of lane l is the sum over the 32 lanes of column l.
// 31 shuffles, a fixed order (deterministic).
__device__ __forceinline__ void warp_column_sums(float* a, int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? a[i] : a[i + w];
      const float keep = upper ? a[i + w] : a[i];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
}

// Per-phase timeline of the last traced launch (test hook): for phase i (in
// list order) slot 3i holds the earliest start of one of its items and slot
// 3i+1 the latest finish (%globaltimer, ns); slot 2 the kernel's start.
constexpr int kTraceSlots = 96;
__device__ unsigned long long g_ns_trace[kTraceSlots];

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---- the item list ----------------------------------------------------------
struct Item {
  int kind, it, z, t, phase;
  unsigned need;  // arrivals on cnt[z] before the item may start
};

__device__ __forceinline__ int n_phases(const NsParams& p) { return 3 * p.iters; }

// Items of one matrix in phase P (3 it + k: Gram, polynomial, X update of iteration it).
__device__ __forceinline__ int phase_items(const NsParams& p, int P) {
  return (P % 3 == 2) ? p.mt * p.ntX : p.nS;
}

// Item t of matrix z in phase P; `need` = the arrivals of every item of z in
// the phases before P.
__device__ __forceinline__ Item make_item(const NsParams& p, int P, int z, int t) {
  Item x{};
  x.phase = P;
  x.z = z;
  x.t = t;
  const int nS = p.nS, nX = p.mt * p.ntX;
  x.it = P / 3;
  const int k = P % 3;
  x.kind = K_GRAM + k;
  x.need = (unsigned)(x.it * (2 * nS + nX) + (k >= 1 ? nS : 0) + (k == 2 ? nS : 0)) * kArrivals;
  return x;
}

// Item g of the whole list, in (phase, matrix, tile) order.
__device__ __forceinline__ Item decode(const NsParams& p, int g) {
  const int NP = n_phases(p);
  for (int P = 0; P < NP; ++P) {
    const int n = p.Z * phase_items(p, P);
    if (g < n) return make_item(p, P, g / phase_items(p, P), g % phase_items(p, P));
    g -= n;
  }
  Item x{};
  x.kind = -1;  // past the end
  return x;
}

__device__ __forceinline__ int total_items(const NsParams& p) {
  int n = 0;
  for (int P = 0; P < n_phases(p); ++P) n += p.Z * phase_items(p, P);
  return n;
}

// Whether the 128 x bn tile (mi, nj) of a symmetric d x d product meets the
// upper triangle (some element with column >= row).
__host__ __device__ __forceinline__ bool sym_tile_needed(int mi, int nj, int bn) { return bn * nj + bn - 1 >= BM * mi; }

// Origin (m0, n0) of tile t of an item's product. The symmetric products
// (sym) enumerate only the tiles that meet the upper triangle, row by row.
__device__ __forceinline__ void tile_origin(const NsParams& p, int t, bool xu, int bn, int& m0, int& n0) {
  const int nt = xu ? p.ntX : p.ntS;
  if (xu || !p.sym) {
    m0 = (t / nt) * BM;
    n0 = (t % nt) * bn;
    return;
  }
  int k = 0;
  for (int mi = 0; mi < p.mt; ++mi)
    for (int nj = 0; nj < nt; ++nj)
      if (sym_tile_needed(mi, nj, bn)) {
        if (k == t) {
          m0 = mi * BM;
          n0 = nj * bn;
          return;
        }
        ++k;
      }
  m0 = n0 = 0;  // not reached for t < nS
}

// Waits, bounded, until matrix z's counter has `need` arrivals. Returns false
// on a timeout (recorded in the status word) or once another CTA has recorded
// an error.
__device__ __forceinline__ bool wait_count(const NsParams& p, int z, unsigned need) {
  const unsigned* c = p.cnt + z;
  if (ld_acquire_gpu(c) >= need) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (ld_acquire_gpu(c) < need) {
    if ((++it & 63u) == 0) {
      if (*reinterpret_cast<volatile int*>(p.cm.status) != 0) return false;
      if (globaltimer_ns() - t0 > p.cm.timeout_ns) {
        set_status(p.cm.status, TTT_ERR_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

// One epilogue warp's arrival on matrix z's counter, after its writes (TMA
// stores and plain stores) are complete and visible to later TMA loads.
__device__ __forceinline__ void arrive_count(const NsParams& p, int z, bool tma_stores) {
  if (tma_stores) ptx::bulk_wait_all();
  ptx::fence_proxy_async_global();
  __threadfence();
  atomicAdd(p.cnt + z, 1u);
}

__device__ __forceinline__ void trace_min(const NsParams& p, int slot) {
  if (p.trace && slot < kTraceSlots) atomicMin(&g_ns_trace[slot], globaltimer_ns());
}
__device__ __forceinline__ void trace_max(const NsParams& p, int slot) {
  if (p.trace && slot < kTraceSlots) atomicMax(&g_ns_trace[slot], globaltimer_ns());
}

template <int BNS, int BNX, bool SPLIT>
__global__ void __launch_bounds__(kNsThreads, 1) ns_fused_kernel(const __grid_constant__ NsParams p) {
  using Geo = NsGeom<BNS, BNX, SPLIT>;
  constexpr int kSt = Geo::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* epi = smem + (size_t)kSt * Geo::kStageBytes;  // epilogue staging
  uint64_t* full = reinterpret_cast<uint64_t*>(epi + Geo::kEpiBytes);
  uint64_t* empty = full + kSt;
  uint64_t* accf = empty + kSt;
  uint64_t* acce = accf + 2;
  uint64_t* drainb = acce + 2;  // MMAs in flight at an abort
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drainb + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = p.d, dh = p.dh;
  const int G = (int)gridDim.x;
  const int total = total_items(p);
  if (p.trace && blockIdx.x == 0 && threadIdx.x == 0) g_ns_trace[0] = globaltimer_ns();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSt; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&accf[s], 1);
      ptx::mbar_init(&acce[s], kEpiWarps);  // one arrival per epilogue warp
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

  uint32_t pc = 0;  // producer: k-blocks issued
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int g = blockIdx.x; g < total && !*abort_flag; g += G) {
        const Item x = decode(p, g);
        if (x.kind != K_GRAM && x.kind != K_POLY && x.kind != K_XUPD) continue;
        // the item's operands are complete once its matrix's earlier phases are
        if (!wait_count(p, x.z, x.need)) {
          *abort_flag = 1;
          break;
        }
        ptx::fence_proxy_async_global();  // the TMA loads below see what the counter published
        const int cur = x.it & 1;
        const bool xu = x.kind == K_XUPD;
        const int bn = xu ? BNX : BNS;
        int m0, n0;
        tile_origin(p, x.t, xu, bn, m0, n0);
        const int nkb = (x.kind == K_GRAM ? dh : d) / kNsBK;
        const uint32_t tx = Geo::kOps * (kNsABytes + (uint32_t)bn * kNsBK * 2);
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = pc % kSt;
          if (!tc_wait(&empty[s], ((pc / kSt) & 1u) ^ 1u, p.cm, abort_flag)) break;
          uint8_t* st = smem + (size_t)s * Geo::kStageBytes;
          ptx::mbar_expect_tx(&full[s], tx);
          const int k = kb * kNsBK;
          for (int h = 0; h < Geo::kOps; ++h) {
            uint8_t* sa = st + h * kNsABytes;
            uint8_t* sb = st + Geo::kOps * kNsABytes + h * Geo::kBBytes;
            if (x.kind == K_GRAM) {
              ptx::tma_load_3d(sa, &p.mXa[cur][h], &full[s], k, m0, x.z);
              ptx::tma_load_3d(sb, &p.mXb[cur][h], &full[s], k, n0, x.z);
            } else if (x.kind == K_POLY) {
              ptx::tma_load_3d(sa, &p.mRa[h], &full[s], k, m0, x.z);
              ptx::tma_load_3d(sb, &p.mRb[h], &full[s], k, n0, x.z);
            } else {
              ptx::tma_load_3d(sa, &p.mPa[h], &full[s], k, m0, x.z);
              for (int gg = 0; gg < bn / 64; ++gg)
                ptx::tma_load_3d(sb + gg * kNsMNBox, &p.mXm[cur][h], &full[s], n0 + gg * 64, k, x.z);
            }
          }
          ++pc;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t mc = 0, at = 0;
      for (int g = blockIdx.x; g < total && !*abort_flag; g += G) {
        const Item x = decode(p, g);
        if (x.kind != K_GRAM && x.kind != K_POLY && x.kind != K_XUPD) continue;
        const uint32_t acc = at & 1u;
        if (!tc_wait(&acce[acc], ((at >> 1) & 1u) ^ 1u, p.cm, abort_flag)) break;
        ptx::tc_fence_after();
        const uint32_t dt = tmem + acc * kAccCols;
        const int nkb = (x.kind == K_GRAM ? dh : d) / kNsBK;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = mc % kSt;
          if (!tc_wait(&full[s], (mc / kSt) & 1u, p.cm, abort_flag)) {
            ok = false;
            break;
          }
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
            if (x.kind == K_XUPD) {
              constexpr uint32_t id = ptx::idesc_bf16(BM, BNX, false, true, !SPLIT);
#pragma unroll
              for (int kk = 0; kk < kNsBK / 16; ++kk)
                ptx::mma_bf16(dt, kdesc64(sa, kk), mdesc32(sb, kk), id, (kb | kk | pr) != 0);
            } else {
              constexpr uint32_t id = ptx::idesc_bf16(BM, BNS, false, false, !SPLIT);
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
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;          // epilogue warp 0..7
    const int gq = warp & 3;          // TMEM lane group this warp may access
    const int r = 32 * gq + lane;     // accumulator row of this thread
    const int eh = ew >> 2;           // which half of a tile's columns it takes
    uint8_t* const ebuf = epi + (size_t)ew * kEpiBufs * 4096;
    uint32_t et_n = 0;                // GEMM tiles drained
    uint32_t es = 0;                  // staging buffers used (this warp)
    bool first = true;
    for (int g = blockIdx.x; g < total; g += G) {
      if (*abort_flag) break;  // uniform within the warp (read after a wait)
      const Item x = decode(p, g);
      const bool withhold = p.stall && first && blockIdx.x == 0;  // test hook
      first = false;
      const bool xu = x.kind == K_XUPD;
      const bool last = xu && x.it + 1 == p.iters;
      const int bn = xu ? BNX : BNS;
      const int z = x.z, j = z % 3;
      int m0, n0;
      tile_origin(p, x.t, xu, bn, m0, n0);
      const int m = m0 + r;
      const int m_warp = m - lane;  // first row of this warp (warp-uniform)
      const bool row_ok = m < d;
      const uint32_t acc = et_n & 1u;
      if (last && row_ok) {
        // while this tile's MMAs run, pull this thread's row of M into L2
        ptx::prefetch_l2_bulk(p.M + ((size_t)z * d + m) * dh + n0, (uint32_t)bn * 4u);
      }
      // fused normalisation: 1 / (||G||_F + eps) of matrix z from the gradient
      // kernel's partial sums (a fixed order, the same in every warp)
      float gscale = 1.f;
      if (p.fused && x.it == 0 && x.kind != K_POLY) {
        const float* part = p.nsqg + (size_t)z * p.nsq_n;
        float ssum = 0.f;
        for (int k = lane; k < p.nsq_n; k += 32) ssum += ldcg(part + k);
        for (int o = 16; o > 0; o >>= 1) ssum += __shfl_down_sync(0xffffffffu, ssum, o);
        const float inv = 1.f / (sqrtf(__shfl_sync(0xffffffffu, ssum, 0)) + p.eps);
        gscale = x.kind == K_GRAM ? inv * inv : inv;
      }
      int ok = 0;
      if (lane == 0) ok = tc_wait(&accf[acc], (et_n >> 1) & 1u, p.cm, abort_flag) && !*abort_flag;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      ++et_n;
      if (ok) {
        ptx::tc_fence_after();
        if (lane == 0) trace_min(p, 2 + 2 * x.phase);
        const uint32_t ta = tmem + acc * kAccCols + ((uint32_t)(32 * gq) << 16);
        const int cur = x.it & 1;
        float rs = 0.f;  // last X update, weight norm on, W2: this row's sum of squares over the tile
        float v[32];
        float4 mA[8], mB[8];  // last X update: M of an even block and of the next one, loaded together
        // each 32 x 32 block of the warp goes through its staging buffer and
        // one TMA store per operand half; warp-uniform control flow
        const int hw = bn / kColHalves;  // columns per half (a multiple of 64)
        for (int c = eh * hw; c < (eh + 1) * hw; c += 32) {
          const int n = n0 + c;
          if (m_warp >= d || (!xu && n >= d)) continue;  // block outside the matrix
          ptx::tmem_ld32(ta + c, v);
          if (gscale != 1.f) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= gscale;
          }
          uint8_t* buf = ebuf + (size_t)(es % kEpiBufs) * 4096;
          if (lane == 0) ptx::bulk_wait_read<kEpiBufs - 1>();  // the store that used this buffer has read it
          __syncwarp();
          const CUtensorMap* mh;
          const CUtensorMap* ml = nullptr;
          if (x.kind == K_GRAM) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] += (m == n + i ? p.beta : 0.f);
            stage_op32<SPLIT>(buf, lane, v);
            mh = &p.sR[0];
            ml = &p.sR[1];
          } else if (x.kind == K_POLY) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = p.c * v[i] + (m == n + i ? p.alpha : 0.f);
            stage_op32<SPLIT>(buf, lane, v);
            mh = &p.sP[0];
            ml = &p.sP[1];
          } else if (!last) {
            stage_op32<SPLIT>(buf, lane, v);
            mh = &p.sX[cur ^ 1][0];
            ml = &p.sX[cur ^ 1][1];
          } else {
            // the update, fused: M <- M - step*U
            if (row_ok) {
              const bool odd = ((c >> 5) & 1) != 0;  // warp-uniform
              if (!odd) {
                const float* mrow = p.M + (size_t)z * d * dh + (size_t)m * dh + n;
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) mA[q4] = ldcg4(mrow + 4 * q4);
                if (c + 32 < (eh + 1) * hw) {
#pragma unroll
                  for (int q4 = 0; q4 < 8; ++q4) mB[q4] = ldcg4(mrow + 32 + 4 * q4);
                }
              }
              auto upd = [&](const float4(&mq)[8]) {
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                  v[4 * q4 + 0] = mq[q4].x - p.step * v[4 * q4 + 0];
                  v[4 * q4 + 1] = mq[q4].y - p.step * v[4 * q4 + 1];
                  v[4 * q4 + 2] = mq[q4].z - p.step * v[4 * q4 + 2];
                  v[4 * q4 + 3] = mq[q4].w - p.step * v[4 * q4 + 3];
                }
              };
              if (odd)
                upd(mB);
              else
                upd(mA);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = 0.f;
            }
            stage_f32x32(buf, lane, v);
            mh = &p.sM;
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_3d(mh, buf, n, m_warp, z);
            if (SPLIT && ml) ptx::tma_store_3d(ml, buf + 2048, n, m_warp, z);
            ptx::bulk_commit();
          }
          ++es;
          // symmetric products: a strictly upper 32 x 32 block whose mirror lies in
          // no computed tile is also written transposed, at (n, m_warp)
          if (!xu && p.sym && n > m_warp &&
              !sym_tile_needed(n / BM, m_warp / BNS, BNS)) {
            uint8_t* tb = ebuf + (size_t)(es % kEpiBufs) * 4096;
            if (lane == 0) ptx::bulk_wait_read<kEpiBufs - 1>();
            __syncwarp();
            stage_op32_t<SPLIT>(tb, lane, v);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_3d(mh, tb, m_warp, n, z);
              if (SPLIT && ml) ptx::tma_store_3d(ml, tb + 2048, m_warp, n, z);
              ptx::bulk_commit();
            }
            ++es;
          }
          if (last) {
            if (!p.wnorm) {
              // final: the bf16 shadow(s) too
              const size_t o = (size_t)z * d * dh + (size_t)m * dh + n;
              if (row_ok) {
                if (p.Msl)
                  st_bf16pair32(p.Ms + o, p.Msl + o, v);
                else
                  st_bf16x32(p.Ms + o, v);
              }
            } else if (j == 1) {
#pragma unroll
              for (int i = 0; i < 32; ++i) rs = fmaf(v[i], v[i], rs);
            } else {
              // columns of M1 / M3 are rows of W1 / W3: sums over this warp's 32 rows
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] *= v[i];
              warp_column_sums(v, lane);
              p.colpart[((size_t)z * (d / 32) + m_warp / 32) * dh + n + lane] = v[0];
            }
          }
        }
        if (last && p.wnorm && j == 1 && row_ok)
          p.rowpart[((size_t)z * (dh / hw) + n0 / hw + eh) * d + m] = rs;
        ptx::tc_fence_before();
        ptx::fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&acce[acc]);
        // this warp's stores of the tile are complete before the counter says so
        if (lane == 0 && !withhold) arrive_count(p, z, true);
        if (lane == 0) trace_max(p, 3 + 2 * x.phase);
      }
      __syncwarp();
    }
    if (lane == 0) ptx::bulk_wait_all();  // stores still in flight after an abort
    __syncwarp();
  }

  // ---------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {
    // the copies started into this CTA must land before it exits: the `full`
    // barriers count them
    for (uint32_t k = pc > (uint32_t)kSt ? pc - kSt : 0; k < pc; ++k)
      tc_drain(&full[k % kSt], (k / kSt) & 1u, p.cm);
  }
  if (warp == 1 && lane == 0 && *abort_flag) {
    // and the MMAs this CTA issued must finish before TMEM is freed
    ptx::mma_commit(drainb);
    tc_drain(drainb, 0, p.cm);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, 2 * kAccCols);
  if (p.trace && threadIdx.x == 0) atomicMax(&g_ns_trace[1], globaltimer_ns());
}

// ---------------------------------------------------------------- weight norm
// After the fused Muon kernel: M holds M - step*U and the last X update wrote
// partial sums of squares of the new weight rows (rowpart for the rows of M2,
// one per column tile; colpart for the columns of M1 / M3, one per 32 rows).
// One CTA per (matrix z, 32 rows of M): the scales of its rows (M2) or of every
// column (M1, M3) are summed from the partials in a fixed order into shared
// memory, then its elements are scaled (every row of W1, W2, W3 back to its W0
// norm: the LaCT page's §2.2.1, eq. 8) and written with their bf16 shadow(s).
struct WnormParams {
  float* M;
  bf16* Ms;
  bf16* Msl;
  const float* n0;
  const float* rowpart;  // [Z][dh / bnx][d]
  const float* colpart;  // [Z][d / 32][dh]
  int d, dh, bnx;
  float eps;
};

constexpr int kWnThreads = 256;

__global__ void __launch_bounds__(kWnThreads) ns_wnorm_kernel(const __grid_constant__ WnormParams p) {
  extern __shared__ float sc[];  // 32 row scales, or dh column scales
  const int z = blockIdx.y, j = z % 3;
  const int d = p.d, dh = p.dh;
  const int r0 = blockIdx.x * 32, r1 = min(d, r0 + 32);
  const float* n0 = p.n0 + (size_t)z * dh;
  if (j == 1) {
    const int ntc = dh / p.bnx;
    for (int row = r0 + (int)threadIdx.x; row < r1; row += kWnThreads) {
      float t = 0.f;
      for (int q = 0; q < ntc; ++q) t += p.rowpart[((size_t)z * ntc + q) * d + row];
      sc[row - r0] = n0[row] / fmaxf(sqrtf(t), p.eps);
    }
  } else {
    const int nb = d / 32;
    for (int col = threadIdx.x; col < dh; col += kWnThreads) {
      float t = 0.f;
      for (int b = 0; b < nb; ++b) t += p.colpart[((size_t)z * nb + b) * dh + col];
      sc[col] = n0[col] / fmaxf(sqrtf(t), p.eps);
    }
  }
  __syncthreads();
  const size_t e0 = ((size_t)z * d + r0) * dh;
  const int n4 = (r1 - r0) * dh / 4;
  constexpr int kU = 8;  // independent 16-byte loads in flight per thread
  for (int b = threadIdx.x; b < n4; b += kWnThreads * kU) {
    float4 mv[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (b + u * kWnThreads < n4) mv[u] = __ldcg(reinterpret_cast<const float4*>(p.M + e0) + b + u * kWnThreads);
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (b + u * kWnThreads < n4) {
        const int w = 4 * (b + u * kWnThreads);
        const int row = w / dh, col = w % dh;
        const float4 f = j == 1 ? make_float4(sc[row], sc[row], sc[row], sc[row])
                                : *reinterpret_cast<const float4*>(sc + col);
        const float4 x = make_float4(mv[u].x * f.x, mv[u].y * f.y, mv[u].z * f.z, mv[u].w * f.w);
        const size_t e = e0 + (size_t)w;
        *reinterpret_cast<float4*>(p.M + e) = x;
        uint2 h;
        h.x = pack_bf16(x.x, x.y);
        h.y = pack_bf16(x.z, x.w);
        *reinterpret_cast<uint2*>(p.Ms + e) = h;
        if (p.Msl) {
          uint2 l;
          l.x = pack_bf16(bf_rest(x.x), bf_rest(x.y));
          l.y = pack_bf16(bf_rest(x.z), bf_rest(x.w));
          *reinterpret_cast<uint2*>(p.Msl + e) = l;
        }
      }
  }
}

// ---------------------------------------------------------------- input
// Newton-Schulz's input from fp32 gradients: one warp per (matrix z, row m,
// column tile of bn) sums `splits` partials in split order, advances the
// momentum buffer (B <- mu B + G), writes bf16 (hi, lo) operands (unless Xh is
// NULL) and the tile row's sum of squares nsq[(z d + m) nt + tile].
__global__ void ns_input_kernel(const float* parts, int splits, int Z, int d, int dh, int bn, float* mom, float mu,
                                bf16* Xh, bf16* Xl, float* nsq) {
  const int lane = threadIdx.x & 31;
  const int nt = dh / bn;
  const long long n_rows = (long long)Z * d * nt;
  const size_t n = (size_t)Z * d * dh;
  for (long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < n_rows;
       w += ((long long)gridDim.x * blockDim.x) >> 5) {
    const int tile = (int)(w % nt);
    const long long zm = w / nt;  // z * d + m
    const size_t row0 = (size_t)zm * dh + (size_t)tile * bn;
    float ss = 0.f;
    for (int c = 4 * lane; c < bn; c += 128) {
      const size_t e = row0 + c;
      float4 acc = *reinterpret_cast<const float4*>(parts + e);
      for (int sp = 1; sp < splits; ++sp) {
        const float4 v = *reinterpret_cast<const float4*>(parts + (size_t)sp * n + e);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      if (mom) {
        float4* mb = reinterpret_cast<float4*>(mom + e);
        const float4 b = *mb;
        acc = make_float4(fmaf(mu, b.x, acc.x), fmaf(mu, b.y, acc.y), fmaf(mu, b.z, acc.z), fmaf(mu, b.w, acc.w));
        *mb = acc;
      }
      if (Xh) {
        uint2 h, l;
        h.x = pack_bf16(acc.x, acc.y);
        h.y = pack_bf16(acc.z, acc.w);
        l.x = pack_bf16(bf_rest(acc.x), bf_rest(acc.y));
        l.y = pack_bf16(bf_rest(acc.z), bf_rest(acc.w));
        *reinterpret_cast<uint2*>(Xh + e) = h;
        *reinterpret_cast<uint2*>(Xl + e) = l;
      }
      ss = fmaf(acc.w, acc.w, fmaf(acc.z, acc.z, fmaf(acc.y, acc.y, fmaf(acc.x, acc.x, ss))));
    }
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) nsq[(size_t)zm * nt + tile] = ss;
  }
}

// X0 = B / (||B||_F + eps) as fp16 operands (single precision), one CTA per
// (matrix z, 32 rows); ||B||^2 from the partial sums, in order.
__global__ void ns_scale_f16_kernel(const float* src, const float* nsq, int nsq_n, float eps, f16* X0, int d,
                                    int dh) {
  __shared__ float inv;
  const int z = blockIdx.y;
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int k = 0; k < nsq_n; ++k) t += nsq[(size_t)z * nsq_n + k];
    inv = 1.f / (sqrtf(t) + eps);
  }
  __syncthreads();
  const int r0 = blockIdx.x * 32, r1 = min(d, r0 + 32);
  const size_t e0 = ((size_t)z * d + r0) * dh;
  const int n4 = (r1 - r0) * dh / 4;
  for (int b = threadIdx.x; b < n4; b += blockDim.x) {
    const float4 v = reinterpret_cast<const float4*>(src + e0)[b];
    uint2 h;
    h.x = pack_f16(v.x * inv, v.y * inv);
    h.y = pack_f16(v.z * inv, v.w * inv);
    reinterpret_cast<uint2*>(X0 + e0)[b] = h;
  }
}

// Grid of the launch: every CTA resident at once (one per SM at this
// shared-memory size), so that no dependency waits on a CTA that is not
// running (the cooperative-launch occupancy).
template <int BNS, int BNX, bool SPLIT>
int grid_size(int* resident) {
  auto kern = ns_fused_kernel<BNS, BNX, SPLIT>;
  const size_t smem = NsGeom<BNS, BNX, SPLIT>::kSmem;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return -1;
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kNsThreads, smem) != cudaSuccess)
    return -1;
  if (resident) *resident = sms * per_sm;
  return sms * per_sm;
}

int g_forced_grid = 0;  // test hook: 0 = every SM, else this many CTAs
// test hook: symmetric d x d products on (1), off (0), or chosen by the shape
// (-1, default): on when an iteration has more than four tiles per SM, where
// the products' throughput bounds the step; with fewer, each matrix's chain of
// phases bounds it, and the mirrored stores would only lengthen its epilogues
int g_sym = -1;
bool g_trace = false;   // test hook: record the phase timeline of every launch
std::atomic<int> g_stall_next{0};  // test hook: the next launch loses one item's completion

template <int BNS, int BNX, bool SPLIT>
int launch_ns(NsParams& p, cudaStream_t st) {
  auto kern = ns_fused_kernel<BNS, BNX, SPLIT>;
  const size_t smem = NsGeom<BNS, BNX, SPLIT>::kSmem;
  int G = grid_size<BNS, BNX, SPLIT>(nullptr);
  if (G <= 0) return TTT_ERR_CUDA;
  if (g_forced_grid > 0 && g_forced_grid < G) G = g_forced_grid;
  if (cudaMemsetAsync(p.cnt, 0, sizeof(unsigned) * (size_t)p.Z, st) != cudaSuccess) return TTT_ERR_CUDA;
  p.trace = g_trace ? 1 : 0;
  p.stall = g_stall_next.exchange(0);
  if (g_trace) {
    unsigned long long init[kTraceSlots];
    for (int i = 0; i < kTraceSlots; ++i) init[i] = (i >= 2 && i % 2 == 0) ? ~0ull : 0ull;
    if (cudaMemcpyToSymbolAsync(g_ns_trace, init, sizeof(init), 0, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return TTT_ERR_CUDA;
  }
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
  if (e != cudaSuccess) return TTT_ERR_CUDA;
  if (!p.wnorm) return TTT_OK;
  WnormParams w{};
  w.M = p.M; w.Ms = p.Ms; w.Msl = p.Msl; w.n0 = p.n0; w.rowpart = p.rowpart; w.colpart = p.colpart;
  w.d = p.d; w.dh = p.dh; w.bnx = BNX / kColHalves; w.eps = p.wnorm_eps;
  const size_t wsm = (size_t)std::max(32, p.dh) * sizeof(float);
  if (wsm > 48 * 1024 &&
      cudaFuncSetAttribute(ns_wnorm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wsm) != cudaSuccess)
    return TTT_ERR_CUDA;
  prof_before(TTT_KERNEL_UPDATE, st);
  ns_wnorm_kernel<<<dim3((p.d + 31) / 32, p.Z), kWnThreads, wsm, st>>>(w);
  prof_after(TTT_KERNEL_UPDATE, st);
  return cudaGetLastError() == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

int g_tile_s = 0, g_tile_x = 0;  // test hook: forced column-tile widths (0 = by shape)
// 256-wide tiles of the d x d products from d = 512 on, even when d is not a
// multiple (the padding rows load as zeros): M = 128, N = 128 MMAs run well
// below the rate of N = 256 ones (measured: video d = 640, 724 against
// 784 us per launch); below 512, 128-wide tiles waste less on padding
int pick_bns(int d) { return g_tile_s ? g_tile_s : (d % 256 == 0 || d >= 512) ? 256 : 128; }
int pick_bnx(int dh) { return (g_tile_x && dh % g_tile_x == 0) ? g_tile_x : (dh % 256 == 0) ? 256 : 128; }

}  // namespace

bool ns_fused_supported(const ttt_cfg& g) { return g.d % 64 == 0 && g.dh % 128 == 0 && g.d <= g.dh; }

void ns_force_grid(int ctas) { g_forced_grid = ctas; }

int ns_input_launch(const float* parts, int splits, int Z, int d, int dh, int bn, float* mom, float mu, void* Xh,
                    void* Xl, float* nsq, cudaStream_t st) {
  prof_before(TTT_KERNEL_AUX, st);
  ns_input_kernel<<<4 * 148, 256, 0, st>>>(parts, splits, Z, d, dh, bn, mom, mu, static_cast<bf16*>(Xh),
                                           static_cast<bf16*>(Xl), nsq);
  prof_after(TTT_KERNEL_AUX, st);
  return cudaGetLastError() == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

int ns_build_params(const NsFusedArgs& a, NsParams& p);

namespace {

// Everything the launch parameters are built from: the tensor maps are encoded
// once and reused while a call's chunks (and later calls on the same buffers)
// launch with the same arguments.
struct NsKey {
  const void* ptrs[17];
  float coef[7];
  int ints[10];
};

NsKey ns_key(const NsFusedArgs& a) {
  NsKey k;
  std::memset(&k, 0, sizeof(k));
  const void* ps[17] = {a.X, a.Xh[0], a.Xh[1], a.Xl[0], a.Xl[1], a.Rh, a.Rl, a.Ph, a.Pl, a.M, a.Ms, a.Msl,
                        a.n0, a.scratch, a.cm.status, a.mom, a.nsqg};
  for (int i = 0; i < 17; ++i) k.ptrs[i] = ps[i];
  const ttt_cfg& g = *a.cfg;
  const float cf[7] = {g.ns_a, g.ns_b, g.ns_c, g.ns_eps, g.step, g.wnorm_eps, a.mu};
  for (int i = 0; i < 7; ++i) k.coef[i] = cf[i];
  const int in[10] = {a.Z, g.d, g.dh, g.ns_iters, g.wnorm, a.split ? 1 : 0, g_sym, a.fused ? 1 : 0,
                      g_tile_s, g_tile_x};
  for (int i = 0; i < 10; ++i) k.ints[i] = in[i];
  return k;
}

thread_local NsKey t_key;
thread_local NsParams t_params;
thread_local bool t_have = false;

}  // namespace

int ns_fused_run(const NsFusedArgs& in, cudaStream_t st) {
  NsFusedArgs a = in;
  const ttt_cfg& g = *a.cfg;
  if (!a.fused) {
    // X0 from the fp32 gradient: split precision writes the unscaled operands
    // and partial norms (the kernel scales); single precision normalises first
    const int nsq_bn = 128;
    const int rc = ns_input_launch(a.X, 1, a.Z, g.d, g.dh, nsq_bn, a.mom, a.mu, a.split ? a.Xh[0] : nullptr,
                                   a.split ? a.Xl[0] : nullptr, const_cast<float*>(a.nsqg), st);
    if (rc != TTT_OK) return rc;
    a.nsq_n = g.d * (g.dh / nsq_bn);
    if (a.split) {
      a.fused = true;
    } else {
      prof_before(TTT_KERNEL_AUX, st);
      ns_scale_f16_kernel<<<dim3((g.d + 31) / 32, a.Z), 256, 0, st>>>(a.mom ? a.mom : a.X, a.nsqg, a.nsq_n, g.ns_eps,
                                                                      static_cast<f16*>(a.Xh[0]), g.d, g.dh);
      prof_after(TTT_KERNEL_AUX, st);
      if (cudaGetLastError() != cudaSuccess) return TTT_ERR_CUDA;
    }
  }
  const int bns = pick_bns(g.d), bnx = pick_bnx(g.dh);
  const bool split = a.split;
  const NsKey key = ns_key(a);
  if (!t_have || std::memcmp(&key, &t_key, sizeof(key)) != 0) {
    t_have = false;
    if (ns_build_params(a, t_params) != TTT_OK) return TTT_ERR_CUDA;
    t_key = key;
    t_have = true;
  }
  NsParams p = t_params;
  p.cm = a.cm;
#define TTT_NS_LAUNCH(BS, BX)                                                                 \
  if (bns == BS && bnx == BX)                                                                 \
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
  const int bns = pick_bns(d), bnx = pick_bnx(dh);
  p = NsParams{};
  bool ok = true;
  for (int i = 0; i < 2; ++i)
    for (int h = 0; h < 2; ++h) {
      const void* b = (h && split) ? a.Xl[i] : a.Xh[i];
      ok &= map3(&p.mXa[i][h], b, dh, d, Z, kNsBK, 128, dt, CU_TENSOR_MAP_SWIZZLE_64B);
      ok &= map3(&p.mXb[i][h], b, dh, d, Z, kNsBK, bns, dt, CU_TENSOR_MAP_SWIZZLE_64B);
      ok &= map3(&p.mXm[i][h], b, dh, d, Z, 64, kNsBK, dt);
      ok &= map3(&p.sX[i][h], b, dh, d, Z, 32, 32, dt, CU_TENSOR_MAP_SWIZZLE_64B);
      p.Xop[i][h] = const_cast<void*>(b);
    }
  for (int h = 0; h < 2; ++h) {
    const void* rb = (h && split) ? a.Rl : a.Rh;
    const void* pb = (h && split) ? a.Pl : a.Ph;
    ok &= map3(&p.mRa[h], rb, d, d, Z, kNsBK, 128, dt, CU_TENSOR_MAP_SWIZZLE_64B);
    ok &= map3(&p.mRb[h], rb, d, d, Z, kNsBK, bns, dt, CU_TENSOR_MAP_SWIZZLE_64B);
    ok &= map3(&p.mPa[h], pb, d, d, Z, kNsBK, 128, dt, CU_TENSOR_MAP_SWIZZLE_64B);
    ok &= map3(&p.sR[h], rb, d, d, Z, 32, 32, dt, CU_TENSOR_MAP_SWIZZLE_64B);
    ok &= map3(&p.sP[h], pb, d, d, Z, 32, 32, dt, CU_TENSOR_MAP_SWIZZLE_64B);
  }
  ok &= map3(&p.sM, a.M, dh, d, Z, 32, 32, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return TTT_ERR_CUDA;
  p.M = a.M;
  p.Ms = static_cast<bf16*>(a.Ms);
  p.Msl = static_cast<bf16*>(a.Msl);
  p.n0 = a.n0;
  p.rowpart = a.scratch;
  p.colpart = p.rowpart + (size_t)Z * (dh / 64) * d;
  p.cnt = reinterpret_cast<unsigned*>(p.colpart + (size_t)Z * (d / 32) * dh);
  // a + b s + c s^2 = c (s + beta)^2 + alpha
  p.c = g.ns_c;
  p.beta = g.ns_b / (2.f * g.ns_c);
  p.alpha = g.ns_a - g.ns_b * g.ns_b / (4.f * g.ns_c);
  p.eps = g.ns_eps;
  p.step = g.step;
  p.wnorm_eps = g.wnorm_eps;
  p.wnorm = g.wnorm;
  p.Z = Z;
  p.d = d;
  p.dh = dh;
  p.iters = g.ns_iters;
  p.mt = (d + BM - 1) / BM;
  p.ntS = (d + bns - 1) / bns;
  p.ntX = dh / bnx;
  if (g_sym >= 0) {
    p.sym = g_sym;
  } else {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return TTT_ERR_CUDA;
    const long long tiles = (long long)Z * (2 * p.mt * p.ntS + p.mt * p.ntX);
    p.sym = tiles > 4LL * sms ? 1 : 0;
  }
  p.fused = a.fused ? 1 : 0;
  p.nsqg = a.nsqg;
  p.nsq_n = a.nsq_n;
  p.nS = 0;
  for (int mi = 0; mi < p.mt; ++mi)
    for (int nj = 0; nj < p.ntS; ++nj) p.nS += (!p.sym || sym_tile_needed(mi, nj, bns)) ? 1 : 0;
  p.cm = a.cm;
  return TTT_OK;
}

int ns_fused_plan(const ttt_cfg& g, int* resident) {
  const bool split = g.precision == TTT_PREC_SPLIT;
  const int bns = pick_bns(g.d), bnx = pick_bnx(g.dh);
#define TTT_NS_PLAN(BS, BX)                                                                         \
  if (bns == BS && bnx == BX) return split ? grid_size<BS, BX, true>(resident) : grid_size<BS, BX, false>(resident);
  TTT_NS_PLAN(256, 256)
  TTT_NS_PLAN(128, 256)
  TTT_NS_PLAN(128, 128)
  TTT_NS_PLAN(256, 128)
#undef TTT_NS_PLAN
  return -1;
}

size_t ns_fused_scratch_floats(const ttt_cfg& g, int Z) {
  // partial sums: of the rows of M2 per
  // half column tile (at most dh / 64 of them), of the columns of M1 / M3 per
  // 32 rows; then the per-matrix completion counters
  return (size_t)Z * ((size_t)(g.dh / 64) * g.d + (size_t)(g.d / 32) * g.dh) + (size_t)Z + 64;
}

}  // namespace ttt

extern "C" int ttt_dbg_ns_trace(int on) {
  ttt::g_trace = on != 0;
  return TTT_OK;
}

extern "C" int ttt_dbg_ns_trace_read(unsigned long long* out, int n) {
  if (!out || n < 1 || n > ttt::kTraceSlots) return TTT_ERR_ARG;
  return cudaMemcpyFromSymbol(out, ttt::g_ns_trace, sizeof(unsigned long long) * (size_t)n) == cudaSuccess
             ? TTT_OK
             : TTT_ERR_CUDA;
}

extern "C" void ttt_dbg_stall_next_ns(void) { ttt::g_stall_next.store(1); }

extern "C" int ttt_dbg_ns_symmetric(int on) {
  ttt::g_sym = on < 0 ? -1 : (on ? 1 : 0);
  return TTT_OK;
}

extern "C" int ttt_dbg_ns_tiles(int bns, int bnx) {
  if ((bns != 0 && bns != 128 && bns != 256) || (bnx != 0 && bnx != 128 && bnx != 256)) return TTT_ERR_ARG;
  ttt::g_tile_s = bns;
  ttt::g_tile_x = bnx;
  return TTT_OK;
}
