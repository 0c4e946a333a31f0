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
//   update     fused into the last X update's epilogue: M <- M - step*U, with
//              partial sums of squares of the weight rows
//   weight norm rows of W1, W2, W3 back to their W0 norms, bf16 shadows   (SIMT)
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
#include <atomic>
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
  // epilogue stores of 32 x 32 blocks from shared memory
  CUtensorMap sR[2];           // R [hi, lo]: {d, d, Z}, box {32, 32}, 64-byte swizzle
  CUtensorMap sP[2];           // P [hi, lo]
  CUtensorMap sX[2][2];        // X operand [ping-pong][hi, lo]: {dh, d, Z}
  CUtensorMap sM;              // fp32 M: {dh, d, Z}, box {32, 32}, 128-byte swizzle
  float* X;         // [Z][d][dh] fp32: the gradient (read only)
  float* mom;       // [Z][d][dh] momentum buffers, or nullptr: B <- mu B + G replaces G
  float mu;
  void* Xop[2][2];  // operand copies of X [ping-pong][hi, lo]
  void* Rop[2];
  void* Pop[2];
  float* M;         // [Z][d][dh] fp32 master weights (M1 = W1^T, M2 = W2, M3 = W3^T)
  bf16* Ms;         // bf16 shadow (hi)
  bf16* Msl;        // bf16 shadow (lo) or nullptr
  const float* n0;  // [Z][dh] reference row norms (W2: the first d entries)
  float* nsq;       // [Z][gs] partial sums of squares of the gradient
  float* rowpart;   // [Z][dh / BNX][d] partial sums of squares of the rows of M2, one per column tile
  float* colpart;   // [Z][d / 32][dh] partial sums of squares of the columns of M1 / M3, one per 32 rows
  unsigned* bar;    // grid-barrier counter (zeroed before the launch)
  int trace;        // test hook: record phase timestamps in g_ns_trace
  int stall_barrier;  // test hook: the last CTA never arrives at the first grid barrier
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
static_assert(sizeof(NsParams) <= 4096, "the launch parameters fit the classic 4 KB limit");

constexpr int kNsBK = 32;
constexpr uint32_t kNsABytes = BM * kNsBK * 2;       // 8 KB: 128 rows x 64 B
constexpr uint32_t kNsMNBox = 64 * kNsBK * 2;        // 4 KB: one 64 x 32 MN-major box

// PAIR: tiles of 256 rows computed by a CTA pair (cta_group::2); each CTA
// holds its own 128 rows of A and half of B, so a stage is a third smaller and
// the ring one third deeper.
template <int BNS, int BNX, bool SPLIT, bool PAIR>
struct NsGeom {
  static constexpr int kOps = SPLIT ? 2 : 1;
  static constexpr int kBmax = BNS > BNX ? BNS : BNX;
  static constexpr int kBrows = PAIR ? kBmax / 2 : kBmax;  // B rows (or columns) held by one CTA
  static constexpr uint32_t kBBytes = (uint32_t)kBrows * kNsBK * 2;
  static constexpr uint32_t kStageBytes = kOps * (kNsABytes + kBBytes);
  static constexpr int kStages = (SPLIT ? 4 : 8) * (PAIR ? 3 : 2) / 2;
  // epilogue staging: two 4 KB buffers per epilogue warp (a 32 x 32 block as a
  // bf16 pair, one fp16 operand, or fp32)
  static constexpr uint32_t kEpiBytes = 4 * 2 * 4096;
  static constexpr size_t kSmem = (size_t)kStages * kStageBytes + kEpiBytes + 1024 + 512;
  static constexpr int kRowsPerTile = PAIR ? 2 * BM : BM;
};

// K-major operand in the 64-byte swizzle; K step kk of 16 elements
__device__ __forceinline__ uint64_t kdesc64(uint32_t base, int kk) { return ptx::sdesc_l(base + kk * 32, 16, 512, 4); }
// MN-major operand: 64-wide groups kNsMNBox apart, 128-byte swizzle; K step kk
__device__ __forceinline__ uint64_t mdesc32(uint32_t base, int kk) {
  return ptx::sdesc_l(base + kk * 2048, kNsMNBox, 1024, 2);
}

// Commit of the MMAs issued so far to the barrier at `bar`'s offset in the CTAs
// of `mask`: the CTA's own barrier, or (CTA pairs, single-GPU build only) both
// CTAs' barriers through a multicast commit.
template <bool PAIR>
__device__ __forceinline__ void commit_to(uint64_t* bar, uint16_t mask);
template <>
__device__ __forceinline__ void commit_to<false>(uint64_t* bar, uint16_t) { ptx::mma_commit(bar); }
#if TTT_HAS_MULTICAST
template <>
__device__ __forceinline__ void commit_to<true>(uint64_t* bar, uint16_t mask) { ptx::mma2_commit_mc(bar, mask); }
#endif

struct PhaseDesc {
  int mt, nt, nk1, bn;
};

template <int BNS, int BNX, int ROWS>
__device__ __forceinline__ PhaseDesc phase_desc(const NsParams& p, int kind) {
  PhaseDesc q;
  q.mt = (p.d + ROWS - 1) / ROWS;
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

__device__ __forceinline__ float4 scale4(float4 v, float s) { return make_float4(v.x * s, v.y * s, v.z * s, v.w * s); }

__device__ __forceinline__ float sumsq4(float4 v, float acc) {
  return fmaf(v.w, v.w, fmaf(v.z, v.z, fmaf(v.y, v.y, fmaf(v.x, v.x, acc))));
}

constexpr int kStream = 16;  // independent 16-byte loads in flight per thread in the SIMT phases

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

// Phase timeline of the last traced launch (test hook): slot 0 the start, slot
// 1 the last CTA's exit; for grid barrier i >= 1, slots 3i, 3i+1, 3i+2 hold the
// first and the last CTA's arrival and CTA 0's departure (%globaltimer, ns).
constexpr int kTraceSlots = 96;
__device__ unsigned long long g_ns_trace[kTraceSlots];

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
    if (p.trace && 3 * n_bar + 2 < (unsigned)kTraceSlots) {
      const unsigned long long now = globaltimer_ns();
      atomicMin(&g_ns_trace[3 * n_bar], now);
      atomicMax(&g_ns_trace[3 * n_bar + 1], now);
    }
    __threadfence();
    // (test hook: withholding one arrival makes every CTA's wait run out)
    if (!(p.stall_barrier && n_bar == 1 && blockIdx.x == gridDim.x - 1)) atomicAdd(p.bar, 1u);
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
    if (p.trace && blockIdx.x == 0 && 3 * n_bar + 2 < (unsigned)kTraceSlots) g_ns_trace[3 * n_bar + 2] = globaltimer_ns();
  }
  __syncthreads();
  ptx::fence_proxy_async_global();  // later TMA reads see the data the barrier published
}

template <int BNS, int BNX, bool SPLIT, bool PAIR>
__global__ void __launch_bounds__(kNsThreads, 1) ns_fused_kernel(const __grid_constant__ NsParams p) {
  using Geo = NsGeom<BNS, BNX, SPLIT, PAIR>;
  constexpr int kNsStages = Geo::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* epi = smem + (size_t)kNsStages * Geo::kStageBytes;  // epilogue staging
  uint64_t* full = reinterpret_cast<uint64_t*>(epi + Geo::kEpiBytes);
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
  if (p.trace && blockIdx.x == 0 && threadIdx.x == 0) g_ns_trace[0] = globaltimer_ns();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNsStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&accf[s], 1);
      ptx::mbar_init(&acce[s], PAIR ? 8 : 4);  // one arrival per epilogue warp (of both CTAs of a pair)
    }
    ptx::mbar_init(drainb, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    if (PAIR) {
      ptx::tmem_alloc2(tslot, 2 * kAccCols);
      ptx::tmem_relinquish2();
    } else {
      ptx::tmem_alloc(tslot, 2 * kAccCols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (PAIR) ptx::cluster_sync();  // both CTAs' barriers exist before either signals the other
  const uint32_t tmem = *tslot;
  // pair roles: rank 0 of the pair (the lead) counts both CTAs' loads on its
  // `full` barriers, issues the MMAs and collects both epilogues on `acce`
  const uint32_t crank = PAIR ? ptx::cluster_ctarank() : 0u;
  const uint32_t prank = crank & 1u, lead = crank & ~1u;
  const uint16_t pair_mask = (uint16_t)(3u << lead);
  const uint32_t full_lead = PAIR ? ptx::mapa(ptx::smem_u32(full), lead) : 0u;
  const uint32_t acce_lead = PAIR ? ptx::mapa(ptx::smem_u32(acce), lead) : 0u;
  const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;  // tile-processing unit: a CTA or a pair
  const int n_units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

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
      for (int b = threadIdx.x; b < n4; b += kNsThreads * kStream) {
        float4 v[kStream];
#pragma unroll
        for (int u = 0; u < kStream; ++u)
          if (b + u * kNsThreads < n4) v[u] = ldcg4(g + 4 * (b + u * kNsThreads));
        if (p.mom) {
          // momentum: B <- mu B + G (stored; Newton-Schulz normalises B)
          float* mb = p.mom + (g - p.X);
#pragma unroll
          for (int u = 0; u < kStream; ++u)
            if (b + u * kNsThreads < n4) {
              float4* q = reinterpret_cast<float4*>(mb + 4 * (b + u * kNsThreads));
              const float4 o = __ldcg(q);
              v[u] = make_float4(fmaf(p.mu, o.x, v[u].x), fmaf(p.mu, o.y, v[u].y), fmaf(p.mu, o.z, v[u].z),
                                 fmaf(p.mu, o.w, v[u].w));
              *q = v[u];
            }
        }
#pragma unroll
        for (int u = 0; u < kStream; ++u)
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
      for (int b = threadIdx.x; b < n4; b += kNsThreads * kStream) {
        float4 v[kStream];
#pragma unroll
        for (int u = 0; u < kStream; ++u)
          if (b + u * kNsThreads < n4) v[u] = ldcg4((p.mom ? p.mom : p.X) + base + 4 * (b + u * kNsThreads));
#pragma unroll
        for (int u = 0; u < kStream; ++u)
          if (b + u * kNsThreads < n4) {
            const size_t o = base + 4 * (size_t)(b + u * kNsThreads);
            st_op4<SPLIT>(p.Xop[0][0], p.Xop[0][1], o, scale4(v[u], inv));
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
  uint32_t es = 0;   // epilogue: staging buffers used (this warp)
  for (int it = 0; it < p.iters; ++it) {
    const int cur = it & 1;
    for (int kind = 0; kind < 3; ++kind) {
      const PhaseDesc q = phase_desc<BNS, BNX, Geo::kRowsPerTile>(p, kind);
      const int per_z = q.mt * q.nt;
      const int n_tiles = Z * per_z;
      const int nkb = q.nk1;
      // B rows (Gram, poly) or columns (X update) this CTA loads: all of the
      // tile's, or its half of the pair's
      const int bpart = PAIR ? q.bn / 2 : q.bn;
      if (warp == 0) {
        if (lane == 0 && !*abort_flag) {
          // bytes one CTA loads per stage; the pair's lead expects both CTAs'
          const uint32_t tx = Geo::kOps * (kNsABytes + (uint32_t)bpart * kNsBK * 2);
          for (int t = unit; t < n_tiles && !*abort_flag; t += n_units) {
            const int z = t / per_z, tl = t % per_z;
            const int m0 = (tl / q.nt) * Geo::kRowsPerTile + BM * (int)prank;
            const int n0 = (tl % q.nt) * q.bn + bpart * (int)prank;
            for (int kb = 0; kb < nkb; ++kb) {
              const int s = pc % kNsStages;
              if (!tc_wait(&empty[s], ((pc / kNsStages) & 1u) ^ 1u, p.cm, abort_flag)) break;
              uint8_t* st = smem + (size_t)s * Geo::kStageBytes;
              if (!PAIR || prank == 0) ptx::mbar_expect_tx(&full[s], PAIR ? 2 * tx : tx);
              const uint32_t fb = full_lead + 8u * (uint32_t)s;
              // one TMA load into this CTA, counted on its own `full` barrier or the lead's
              auto load = [&](void* dst, const CUtensorMap* m, int c0, int c1) {
                if (PAIR)
                  ptx::tma_load_3d_pair(dst, m, fb, c0, c1, z);
                else
                  ptx::tma_load_3d(dst, m, &full[s], c0, c1, z);
              };
              const int k = kb * kNsBK;
              for (int h = 0; h < Geo::kOps; ++h) {
                uint8_t* sa = st + h * kNsABytes;
                uint8_t* sb = st + Geo::kOps * kNsABytes + h * Geo::kBBytes;
                if (kind == PH_GRAM) {
                  load(sa, &p.mXa[cur][h], k, m0);
                  load(sb, &p.mXb[cur][h], k, n0);
                } else if (kind == PH_POLY) {
                  load(sa, &p.mRa[h], k, m0);
                  load(sb, &p.mRb[h], k, n0);
                } else {
                  load(sa, &p.mPa[h], k, m0);
                  for (int g = 0; g < bpart / 64; ++g) load(sb + g * kNsMNBox, &p.mXm[cur][h], n0 + g * 64, k);
                }
              }
              ++pc;
            }
          }
        }
      } else if (warp == 1) {
        if (lane == 0 && !*abort_flag && (!PAIR || prank == 0)) {
          for (int t = unit; t < n_tiles && !*abort_flag; t += n_units) {
            const uint32_t acc = at & 1u;
            if (PAIR) {
              // the peer's epilogue arrives here too: cluster-scope acquire, bounded
              const uint32_t par = ((at >> 1) & 1u) ^ 1u;
              const uint64_t t0 = globaltimer_ns();
              bool got;
              while (!(got = ptx::mbar_try_wait_cluster(&acce[acc], par)))
                if (*abort_flag || globaltimer_ns() - t0 > p.cm.timeout_ns) break;
              if (!got) {
                *abort_flag = 1;
                set_status(p.cm.status, TTT_ERR_TIMEOUT);
                break;
              }
            } else if (!tc_wait(&acce[acc], ((at >> 1) & 1u) ^ 1u, p.cm, abort_flag)) {
              break;
            }
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
                  constexpr uint32_t id = ptx::idesc_bf16(Geo::kRowsPerTile, BNX, false, true, !SPLIT);
#pragma unroll
                  for (int kk = 0; kk < kNsBK / 16; ++kk) {
                    if (PAIR)
                      ptx::mma2_bf16(dt, kdesc64(sa, kk), mdesc32(sb, kk), id, (kb | kk | pr) != 0);
                    else
                      ptx::mma_bf16(dt, kdesc64(sa, kk), mdesc32(sb, kk), id, (kb | kk | pr) != 0);
                  }
                } else {
                  constexpr uint32_t id = ptx::idesc_bf16(Geo::kRowsPerTile, BNS, false, false, !SPLIT);
#pragma unroll
                  for (int kk = 0; kk < kNsBK / 16; ++kk) {
                    if (PAIR)
                      ptx::mma2_bf16(dt, kdesc64(sa, kk), kdesc64(sb, kk), id, (kb | kk | pr) != 0);
                    else
                      ptx::mma_bf16(dt, kdesc64(sa, kk), kdesc64(sb, kk), id, (kb | kk | pr) != 0);
                  }
                }
              }
              commit_to<PAIR>(&empty[s], pair_mask);
              ++mc;
            }
            if (!ok) break;
            commit_to<PAIR>(&accf[acc], pair_mask);
            ++at;
          }
        }
      } else {
        const int g = warp & 3;  // TMEM lane group of this warp
        const int r = 32 * g + lane;
        const bool last = it + 1 == p.iters;
        for (int t = unit; t < n_tiles; t += n_units) {
          if (*abort_flag) break;  // uniform within the warp (read after a barrier or a wait)
          const uint32_t acc = et & 1u;
          if (kind == PH_XUPD && last) {
            // while this tile's MMAs run, pull this thread's row of M into L2
            const int zz = t / per_z, tt = t % per_z;
            const int mm = (tt / q.nt) * Geo::kRowsPerTile + BM * (int)prank + r;
            if (mm < d) ptx::prefetch_l2_bulk(p.M + ((size_t)zz * d + mm) * dh + (tt % q.nt) * q.bn, (uint32_t)q.bn * 4u);
          }
          int ok = 0;
          if (lane == 0) ok = tc_wait(&accf[acc], (et >> 1) & 1u, p.cm, abort_flag) && !*abort_flag;
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          ptx::tc_fence_after();
          const int z = t / per_z, tl = t % per_z;
          const uint32_t ta = tmem + acc * kAccCols + ((uint32_t)(32 * g) << 16);
          const int m = (tl / q.nt) * Geo::kRowsPerTile + BM * (int)prank + r, n0 = (tl % q.nt) * q.bn;
          const int m_warp = m - lane;  // first row of this warp (warp-uniform)
          const bool row_ok = m < d;
          const int j = z % 3;
          float rs = 0.f;  // last X update, weight norm on, W2: this row's sum of squares over the tile
          float v[32];
          float4 mA[8], mB[8];  // last X update: M of an even chunk and of the next one, loaded together
          // each 32 x 32 block of the warp goes through its staging buffer and
          // one TMA store per operand half; warp-uniform control flow
          for (int c = 0; c < q.bn; c += 32) {
            const int n = n0 + c;
            if (m_warp >= d || (kind != PH_XUPD && n >= d)) continue;  // block outside the matrix
            ptx::tmem_ld32(ta + c, v);
            uint8_t* buf = epi + (size_t)(2 * g + (es & 1u)) * 4096;
            if (lane == 0) ptx::bulk_wait_read<1>();  // the store that used this buffer has read it
            __syncwarp();
            const CUtensorMap* mh;
            const CUtensorMap* ml = nullptr;
            if (kind == PH_GRAM) {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] += (m == n + i ? p.beta : 0.f);
              stage_op32<SPLIT>(buf, lane, v);
              mh = &p.sR[0];
              ml = &p.sR[1];
            } else if (kind == PH_POLY) {
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
                  if (c + 32 < q.bn) {
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
            if (kind == PH_XUPD && last) {
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
          if (kind == PH_XUPD && last && p.wnorm && j == 1 && row_ok)
            p.rowpart[((size_t)z * (dh / BNX) + n0 / BNX) * d + m] = rs;
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (PAIR)
              ptx::mbar_arrive_cluster(acce_lead + 8u * acc);
            else
              ptx::mbar_arrive(&acce[acc]);
          }
          ++et;
        }
        // this phase's stores are complete before the grid barrier publishes them
        if (lane == 0) ptx::bulk_wait_all();
        __syncwarp();
        ptx::fence_proxy_async_global();
      }
      grid_barrier(p, n_bar, abort_flag);
    }
  }

  // ---------------------------------------------------------------- weight norm
  // The last X update's epilogue wrote M - step*U and its partial sums of
  // squares. One pass per item: the scales of its rows (W2: rows of M2) or of
  // every column (W1, W3: columns of M1 / M3), from the partials in a fixed
  // order, into shared memory (the operand ring is idle now); then the item's
  // elements are scaled and written with their bf16 shadow(s).
  if (p.wnorm) {
    float* sc = reinterpret_cast<float*>(smem);
    for (int i = blockIdx.x; i < n_items; i += G) {
      const int z = i % Z, k = i / Z, j = z % 3;
      const int r0 = min(d, k * rows_per), r1 = min(d, r0 + rows_per);
      const size_t zoff = (size_t)z * d * dh;
      const float* n0 = p.n0 + (size_t)z * dh;
      if (*abort_flag) continue;  // uniform: read after a grid barrier
      __syncthreads();            // the previous item's readers of sc are done
      if (j == 1) {
        const int ntc = dh / BNX;
        for (int row = r0 + threadIdx.x; row < r1; row += kNsThreads) {
          float t = 0.f;
          for (int q2 = 0; q2 < ntc; ++q2) t += ldcg(p.rowpart + ((size_t)z * ntc + q2) * d + row);
          sc[row - r0] = n0[row] / fmaxf(sqrtf(t), p.wnorm_eps);
        }
      } else {
        // four columns per thread, eight partials of each in flight (summed in
        // ascending block order)
        const int nb = d / 32;
        for (int c0 = 0; c0 < dh; c0 += 4 * kNsThreads) {
          float t[4] = {0.f, 0.f, 0.f, 0.f};
          for (int b0 = 0; b0 < nb; b0 += 8) {
            float x[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
              for (int bb = 0; bb < 8; ++bb) {
                const int col = c0 + threadIdx.x + u * kNsThreads;
                x[u][bb] = (col < dh && b0 + bb < nb) ? ldcg(p.colpart + ((size_t)z * nb + b0 + bb) * dh + col) : 0.f;
              }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
              for (int bb = 0; bb < 8; ++bb) t[u] += x[u][bb];
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int col = c0 + threadIdx.x + u * kNsThreads;
            if (col < dh) sc[col] = n0[col] / fmaxf(sqrtf(t[u]), p.wnorm_eps);
          }
        }
      }
      __syncthreads();
      const int n4 = (r1 - r0) * dh / 4;
      const size_t e0 = zoff + (size_t)r0 * dh;
      for (int b = threadIdx.x; b < n4; b += kNsThreads * kStream) {
        float4 mv[kStream];
#pragma unroll
        for (int u = 0; u < kStream; ++u)
          if (b + u * kNsThreads < n4) mv[u] = ldcg4(p.M + e0 + 4 * (size_t)(b + u * kNsThreads));
#pragma unroll
        for (int u = 0; u < kStream; ++u)
          if (b + u * kNsThreads < n4) {
            const int w = 4 * (b + u * kNsThreads);  // element offset inside the item
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
  }

  // ---------------------------------------------------------------- teardown
  if (warp == 0 && lane == 0 && *abort_flag && (!PAIR || prank == 0)) {
    // the copies started into this CTA (and, for a pair, its peer) must land
    // before the CTA exits: the `full` barriers count them
    for (uint32_t k = pc > (uint32_t)kNsStages ? pc - kNsStages : 0; k < pc; ++k)
      tc_drain(&full[k % kNsStages], (k / kNsStages) & 1u, p.cm);
  }
  if (PAIR && warp == 0 && lane == 0 && *abort_flag && prank == 1) {
    // the peer cannot wait on the lead's barriers: give the copies it started
    // (at most one ring ahead of what the lead drains) a bounded time to land
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) {
    }
  }
  if (warp == 1 && lane == 0 && *abort_flag && (!PAIR || prank == 0)) {
    // and the MMAs this thread issued must finish before TMEM is freed
    commit_to<PAIR>(drainb, (uint16_t)(1u << lead));
    tc_drain(drainb, 0, p.cm);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (PAIR) ptx::cluster_sync();  // no CTA leaves while its peer can still signal it or read its memory
  ptx::tc_fence_after();
  if (warp == 1) {
    if (PAIR)
      ptx::tmem_dealloc2(tmem, 2 * kAccCols);
    else
      ptx::tmem_dealloc(tmem, 2 * kAccCols);
  }
  if (p.trace && threadIdx.x == 0) atomicMax(&g_ns_trace[1], globaltimer_ns());
}

#if TTT_HAS_MULTICAST
// ---------------------------------------------------------------- CTA-pair GEMM
// D[z] = A[z] B[z]^T on 256 x 256 tiles computed by CTA pairs (cta_group::2),
// with the operand layouts of the Newton-Schulz phases (32-deep k-blocks,
// 64-byte-swizzled K-major tiles, 128-byte-swizzled 64 x 32 MN-major boxes).
// Each CTA of a pair loads its own 128 rows of A and its half of B (128 rows,
// or 128 columns when B is MN-major); the even CTA counts both halves on its
// `full` barrier and issues the M = 256 MMAs; its commits release the stage
// and hand the accumulator to both CTAs; every epilogue warp of the pair
// returns the accumulator with a cluster-scope arrival on the even CTA's
// `acce` barrier. Test hook for the pair primitives.
struct PairParams {
  CUtensorMap mA;  // {K, M, Z} box {32, 128}, 64-byte swizzle
  CUtensorMap mB;  // K-major {K, N, Z} box {32, 128}; MN-major {N, K, Z} box {64, 32}
  float* D;
  int Z, M, N, K, b_mn;
  TcCommon cm;
};

constexpr int kPairStages = 8;
constexpr uint32_t kPairStage = 2 * kNsABytes;  // A: 128 x 32, B half: 128 x 32
constexpr size_t kPairSmem = (size_t)kPairStages * kPairStage + 1024 + 512;

__global__ void __launch_bounds__(kNsThreads, 1) pair_gemm_kernel(const __grid_constant__ PairParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kPairStages * kPairStage);
  uint64_t* empty = full + kPairStages;
  uint64_t* accf = empty + kPairStages;
  uint64_t* acce = accf + 2;
  uint64_t* drainb = acce + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drainb + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank() & 1u;
  const uint32_t lead = ptx::cluster_ctarank() & ~1u;
  const int pair = (int)(blockIdx.x >> 1), n_pairs = (int)(gridDim.x >> 1);
  const int mt = p.M / 256, nt = p.N / 256, per_z = mt * nt, n_tiles = p.Z * per_z;
  const int nkb = p.K / kNsBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
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
    ptx::tmem_alloc2(tslot, 2 * kAccCols);
    ptx::tmem_relinquish2();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  ptx::cluster_sync();  // both CTAs' barriers exist before either signals the other
  const uint32_t tmem = *tslot;
  const uint32_t full_lead = ptx::mapa(ptx::smem_u32(full), lead);
  const uint32_t acce_lead = ptx::mapa(ptx::smem_u32(acce), lead);

  uint32_t pc = 0;
  if (warp == 0) {
    if (lane == 0) {
      for (int t = pair; t < n_tiles && !*abort_flag; t += n_pairs) {
        const int z = t / per_z, tl = t % per_z;
        const int m0 = (tl / nt) * 256 + 128 * (int)rank, n0 = (tl % nt) * 256 + 128 * (int)rank;
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = pc % kPairStages;
          if (!tc_wait(&empty[s], ((pc / kPairStages) & 1u) ^ 1u, p.cm, abort_flag)) break;
          uint8_t* st = smem + (size_t)s * kPairStage;
          if (rank == 0) ptx::mbar_expect_tx(&full[s], 2 * kPairStage);
          const uint32_t fb = full_lead + 8u * (uint32_t)s;
          const int k = kb * kNsBK;
          ptx::tma_load_3d_pair(st, &p.mA, fb, k, m0, z);
          if (p.b_mn) {
            ptx::tma_load_3d_pair(st + kNsABytes, &p.mB, fb, n0, k, z);
            ptx::tma_load_3d_pair(st + kNsABytes + kNsMNBox, &p.mB, fb, n0 + 64, k, z);
          } else {
            ptx::tma_load_3d_pair(st + kNsABytes, &p.mB, fb, k, n0, z);
          }
          ++pc;
        }
      }
      if (*abort_flag && rank == 0)
        for (uint32_t k = pc > (uint32_t)kPairStages ? pc - kPairStages : 0; k < pc; ++k)
          tc_drain(&full[k % kPairStages], (k / kPairStages) & 1u, p.cm);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      uint32_t mc = 0, at = 0;
      for (int t = pair; t < n_tiles && !*abort_flag; t += n_pairs) {
        const uint32_t acc = at & 1u;
        // bounded wait with cluster-scope acquire: the peer's epilogue arrives here
        {
          const uint32_t par = ((at >> 1) & 1u) ^ 1u;
          const uint64_t t0 = globaltimer_ns();
          bool ok = false;
          while (!(ok = ptx::mbar_try_wait_cluster(&acce[acc], par))) {
            if (*abort_flag || globaltimer_ns() - t0 > p.cm.timeout_ns) break;
          }
          if (!ok) {
            *abort_flag = 1;
            set_status(p.cm.status, TTT_ERR_TIMEOUT);
            break;
          }
        }
        ptx::tc_fence_after();
        const uint32_t dt = tmem + acc * kAccCols;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = mc % kPairStages;
          if (!tc_wait(&full[s], (mc / kPairStages) & 1u, p.cm, abort_flag)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(smem + (size_t)s * kPairStage);
          const uint32_t sb = sa + kNsABytes;
          if (p.b_mn) {
            constexpr uint32_t id = ptx::idesc_bf16(256, 256, false, true);
#pragma unroll
            for (int kk = 0; kk < kNsBK / 16; ++kk) ptx::mma2_bf16(dt, kdesc64(sa, kk), mdesc32(sb, kk), id, (kb | kk) != 0);
          } else {
            constexpr uint32_t id = ptx::idesc_bf16(256, 256, false, false);
#pragma unroll
            for (int kk = 0; kk < kNsBK / 16; ++kk) ptx::mma2_bf16(dt, kdesc64(sa, kk), kdesc64(sb, kk), id, (kb | kk) != 0);
          }
          ptx::mma2_commit_mc(&empty[s], (uint16_t)(3u << lead));
          ++mc;
        }
        if (!ok) break;
        ptx::mma2_commit_mc(&accf[acc], (uint16_t)(3u << lead));
        ++at;
      }
      if (*abort_flag) {
        ptx::mma2_commit_mc(drainb, (uint16_t)(1u << lead));
        tc_drain(drainb, 0, p.cm);
      }
    }
  } else {
    const int g = warp & 3;
    const int r = 32 * g + lane;
    uint32_t et = 0;
    for (int t = pair; t < n_tiles; t += n_pairs) {
      if (*abort_flag) break;
      const uint32_t acc = et & 1u;
      int ok = 0;
      if (lane == 0) ok = tc_wait(&accf[acc], (et >> 1) & 1u, p.cm, abort_flag) && !*abort_flag;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ptx::tc_fence_after();
      const int z = t / per_z, tl = t % per_z;
      const int m = (tl / nt) * 256 + 128 * (int)rank + r, n0 = (tl % nt) * 256;
      const uint32_t ta = tmem + acc * kAccCols + ((uint32_t)(32 * g) << 16);
      float v[32];
      for (int c = 0; c < 256; c += 32) {
        ptx::tmem_ld32(ta + c, v);
        st_f32x32(p.D + ((size_t)z * p.M + m) * p.N + n0 + c, v);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(acce_lead + 8u * acc);
      ++et;
    }
  }
  ptx::tc_fence_before();
  __syncwarp();
  __syncthreads();
  // no CTA leaves while its peer can still signal it or read its shared memory
  ptx::cluster_sync();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc2(tmem, 2 * kAccCols);
}

#endif  // TTT_HAS_MULTICAST

// Grid of the launch: every CTA resident at once (one per SM at this
// shared-memory size), so that the grid barriers cannot wait on a CTA that is
// not running. Single CTAs: the cooperative-launch occupancy; pairs: twice the
// number of two-CTA clusters that fit.
template <int BNS, int BNX, bool SPLIT, bool PAIR>
int grid_size(int* resident) {
  auto kern = ns_fused_kernel<BNS, BNX, SPLIT, PAIR>;
  const size_t smem = NsGeom<BNS, BNX, SPLIT, PAIR>::kSmem;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return -1;
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (PAIR) {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kNsThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int pairs = 0;
    if (cudaOccupancyMaxActiveClusters(&pairs, kern, &cfg) != cudaSuccess || pairs < 1) {
      cudaGetLastError();
      return -1;
    }
    if (resident) *resident = 2 * pairs;
    return 2 * pairs;
  }
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kNsThreads, smem) != cudaSuccess)
    return -1;
  if (resident) *resident = sms * per_sm;
  return sms * per_sm;
}

int g_forced_grid = 0;  // test hook: 0 = every SM, else this many CTAs
std::atomic<int> g_stall_next_barrier{0};  // test hook: the next launch's first grid barrier loses an arrival
bool g_trace = false;   // test hook: record the phase timeline of every launch

template <int BNS, int BNX, bool SPLIT, bool PAIR>
int launch_ns(NsParams& p, cudaStream_t st) {
  auto kern = ns_fused_kernel<BNS, BNX, SPLIT, PAIR>;
  const size_t smem = NsGeom<BNS, BNX, SPLIT, PAIR>::kSmem;
  int G = grid_size<BNS, BNX, SPLIT, PAIR>(nullptr);
  if (G <= 0) return TTT_ERR_CUDA;
  if (g_forced_grid > 0 && g_forced_grid < G) G = PAIR ? std::max(2, g_forced_grid & ~1) : g_forced_grid;
  p.gs = std::max(1, std::min(kMaxGroup, G / p.Z));
  if (cudaMemsetAsync(p.bar, 0, sizeof(unsigned), st) != cudaSuccess) return TTT_ERR_CUDA;
  p.trace = g_trace ? 1 : 0;
  p.stall_barrier = g_stall_next_barrier.exchange(0);
  if (g_trace) {
    unsigned long long init[kTraceSlots];
    for (int i = 0; i < kTraceSlots; ++i) init[i] = (i >= 3 && i % 3 == 0) ? ~0ull : 0ull;
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
  if (PAIR) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  prof_before(TTT_KERNEL_NS, st);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  prof_after(TTT_KERNEL_NS, st);
  return e == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

bool g_pairs = false;  // test hook: CTA pairs allowed (measured slower on the Muon step's phases)

// CTA pairs whenever every tile is whole: d and dh multiples of 256.
bool ns_use_pairs(const ttt_cfg& g) { return TTT_HAS_MULTICAST && g_pairs && g.d % 256 == 0 && g.dh % 256 == 0; }

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
  float coef[7];
  int ints[7];
};

NsKey ns_key(const NsFusedArgs& a) {
  NsKey k;
  std::memset(&k, 0, sizeof(k));
  const void* ps[16] = {a.X, a.Xh[0], a.Xh[1], a.Xl[0], a.Xl[1], a.Rh, a.Rl, a.Ph, a.Pl, a.M, a.Ms, a.Msl,
                        a.n0, a.scratch, a.cm.status, a.mom};
  for (int i = 0; i < 16; ++i) k.ptrs[i] = ps[i];
  const ttt_cfg& g = *a.cfg;
  const float cf[7] = {g.ns_a, g.ns_b, g.ns_c, g.ns_eps, g.step, g.wnorm_eps, a.mu};
  for (int i = 0; i < 7; ++i) k.coef[i] = cf[i];
  const int in[7] = {a.Z, g.d, g.dh, g.ns_iters, g.wnorm, a.split ? 1 : 0, ns_use_pairs(g) ? 1 : 0};
  for (int i = 0; i < 7; ++i) k.ints[i] = in[i];
  return k;
}

thread_local NsKey t_key;
thread_local NsParams t_params;
thread_local bool t_have = false;

}  // namespace

int ns_fused_run(const NsFusedArgs& a, cudaStream_t st) {
  const ttt_cfg& g = *a.cfg;
  const int d = g.d, dh = g.dh;
  const bool split = a.split;
  const int bns = (d % 256 == 0) ? 256 : 128;
  const int bnx = (dh % 256 == 0) ? 256 : 128;
  const bool pair = ns_use_pairs(g);
  const NsKey key = ns_key(a);
  if (!t_have || std::memcmp(&key, &t_key, sizeof(key)) != 0) {
    t_have = false;
    if (ns_build_params(a, t_params) != TTT_OK) return TTT_ERR_CUDA;
    t_key = key;
    t_have = true;
  }
  NsParams p = t_params;
  p.cm = a.cm;
#if TTT_HAS_MULTICAST
  if (pair) return split ? launch_ns<256, 256, true, true>(p, st) : launch_ns<256, 256, false, true>(p, st);
#endif
#define TTT_NS_LAUNCH(BS, BX)                                                                      \
  if (bns == BS && bnx == BX)                                                                      \
    return split ? launch_ns<BS, BX, true, false>(p, st) : launch_ns<BS, BX, false, false>(p, st);
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
  // rows of one B box (Gram and poly): the tile's, or half of it for a pair
  const int brows = ns_use_pairs(g) ? bns / 2 : bns;
  p = NsParams{};
  bool ok = true;
  for (int i = 0; i < 2; ++i)
    for (int h = 0; h < 2; ++h) {
      const void* b = (h && split) ? a.Xl[i] : a.Xh[i];
      ok &= map3(&p.mXa[i][h], b, dh, d, Z, kNsBK, 128, dt, CU_TENSOR_MAP_SWIZZLE_64B);
      ok &= map3(&p.mXb[i][h], b, dh, d, Z, kNsBK, brows, dt, CU_TENSOR_MAP_SWIZZLE_64B);
      ok &= map3(&p.mXm[i][h], b, dh, d, Z, 64, kNsBK, dt);
      ok &= map3(&p.sX[i][h], b, dh, d, Z, 32, 32, dt, CU_TENSOR_MAP_SWIZZLE_64B);
      p.Xop[i][h] = const_cast<void*>(b);
    }
  for (int h = 0; h < 2; ++h) {
    const void* rb = (h && split) ? a.Rl : a.Rh;
    const void* pb = (h && split) ? a.Pl : a.Ph;
    ok &= map3(&p.mRa[h], rb, d, d, Z, kNsBK, 128, dt, CU_TENSOR_MAP_SWIZZLE_64B);
    ok &= map3(&p.mRb[h], rb, d, d, Z, kNsBK, brows, dt, CU_TENSOR_MAP_SWIZZLE_64B);
    ok &= map3(&p.mPa[h], pb, d, d, Z, kNsBK, 128, dt, CU_TENSOR_MAP_SWIZZLE_64B);
    ok &= map3(&p.sR[h], rb, d, d, Z, 32, 32, dt, CU_TENSOR_MAP_SWIZZLE_64B);
    ok &= map3(&p.sP[h], pb, d, d, Z, 32, 32, dt, CU_TENSOR_MAP_SWIZZLE_64B);
    p.Rop[h] = const_cast<void*>(rb);
    p.Pop[h] = const_cast<void*>(pb);
  }
  ok &= map3(&p.sM, a.M, dh, d, Z, 32, 32, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return TTT_ERR_CUDA;
  p.X = a.X;
  p.mom = a.mom;
  p.mu = a.mu;
  p.M = a.M;
  p.Ms = static_cast<bf16*>(a.Ms);
  p.Msl = static_cast<bf16*>(a.Msl);
  p.n0 = a.n0;
  p.nsq = a.scratch;
  p.rowpart = p.nsq + (size_t)Z * kMaxGroup;
  p.colpart = p.rowpart + (size_t)Z * (dh / 128) * d;
  p.bar = reinterpret_cast<unsigned*>(p.colpart + (size_t)Z * (d / 32) * dh);
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
#if TTT_HAS_MULTICAST
  if (ns_use_pairs(g)) return split ? grid_size<256, 256, true, true>(resident) : grid_size<256, 256, false, true>(resident);
#endif
#define TTT_NS_PLAN(BS, BX)                                                                                   \
  if (bns == BS && bnx == BX)                                                                                 \
    return split ? grid_size<BS, BX, true, false>(resident) : grid_size<BS, BX, false, false>(resident);
  TTT_NS_PLAN(256, 256)
  TTT_NS_PLAN(128, 256)
  TTT_NS_PLAN(128, 128)
  TTT_NS_PLAN(256, 128)
#undef TTT_NS_PLAN
  return -1;
}

size_t ns_fused_scratch_floats(const ttt_cfg& g, int Z) {
  // partial sums: of the gradient's squares per member, of the rows of M2 per
  // column tile (at most dh / 128 tiles), of the columns of M1 / M3 per 32 rows;
  // then the barrier counter
  return (size_t)Z * (kMaxGroup + (size_t)(g.dh / 128) * g.d + (size_t)(g.d / 32) * g.dh) + 64;
}

}  // namespace ttt

extern "C" int ttt_dbg_gemm_pair_bf16(const void* A, const void* B, int b_mn_major, float* D, int Z, int M, int N,
                                      int K, void* stream) {
  using namespace ttt;
#if !TTT_HAS_MULTICAST
  (void)A; (void)B; (void)b_mn_major; (void)D; (void)Z; (void)M; (void)N; (void)K; (void)stream;
  return TTT_ERR_UNSUPPORTED;  // CTA pairs are built only into the single-GPU library
#else
  if (!A || !B || !D || Z < 1 || M < 256 || N < 256 || K < 32 || M % 256 || N % 256 || K % 32) return TTT_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(D)) & 15u)
    return TTT_ERR_ARG;
  PairParams p{};
  const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  bool ok = tcu::map3(&p.mA, A, K, M, Z, kNsBK, 128, dt, CU_TENSOR_MAP_SWIZZLE_64B);
  if (b_mn_major)
    ok &= tcu::map3(&p.mB, B, N, K, Z, 64, kNsBK, dt);
  else
    ok &= tcu::map3(&p.mB, B, K, N, Z, kNsBK, 128, dt, CU_TENSOR_MAP_SWIZZLE_64B);
  if (!ok) return TTT_ERR_CUDA;
  p.D = D;
  p.Z = Z; p.M = M; p.N = N; p.K = K; p.b_mn = b_mn_major ? 1 : 0;
  int* status = nullptr;
  if (cudaMalloc(&status, sizeof(int)) != cudaSuccess) return TTT_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = TTT_OK;
  if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) rc = TTT_ERR_CUDA;
  p.cm.status = status;
  p.cm.timeout_ns = 2000000000ull;
  if (rc == TTT_OK && cudaFuncSetAttribute(pair_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kPairSmem) != cudaSuccess)
    rc = TTT_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(kNsThreads);
  cfg.dynamicSmemBytes = kPairSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  int max_pairs = 0;
  if (rc == TTT_OK) {
    cfg.gridDim = dim3(2);
    if (cudaOccupancyMaxActiveClusters(&max_pairs, pair_gemm_kernel, &cfg) != cudaSuccess || max_pairs < 1) {
      cudaGetLastError();
      rc = TTT_ERR_CUDA;
    }
  }
  if (rc == TTT_OK) {
    const int tiles = Z * (M / 256) * (N / 256);
    cfg.gridDim = dim3(2 * std::min(tiles, max_pairs));
    if (cudaLaunchKernelEx(&cfg, pair_gemm_kernel, p) != cudaSuccess) rc = TTT_ERR_CUDA;
  }
  int h = 0;
  if (rc == TTT_OK && (cudaMemcpyAsync(&h, status, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
                       cudaStreamSynchronize(st) != cudaSuccess))
    rc = TTT_ERR_CUDA;
  cudaFree(status);
  if (rc == TTT_OK && h != 0) rc = h;
  return rc;
#endif
}

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

extern "C" void ttt_dbg_stall_next_ns_barrier(void) { ttt::g_stall_next_barrier.store(1); }

extern "C" int ttt_dbg_ns_pairs(int on) {
  ttt::g_pairs = on != 0;
  return TTT_OK;
}
