// Linear small-chunk path: the fast weight is one d x d matrix per head
// (f(x) = W x, the tutorial page "Test-Time Training layers" §3-§4 linear inner
// model) updated every chunk of 64-token tiles with the chunk-summed gradient
// of the MSE (or inner-product) loss and plain SGD (the LaCT page §1.1 regime of
// 16-64-token updates, run in the shifted block-causal order of §3.2):
//
//   per chunk c:  O_c = Q_c W^T ;  R = K_c W^T - V_c (MSE) or -V_c (IP)
//                 G = (eta * R)^T K_c ;  W <- W - step * G   (at the chunk's end)
//
// The work per token is tiny (d = 64) and strictly sequential over chunks, so
// the kernel is bound by HBM bandwidth and per-chunk latency, not by tensor
// throughput. Design:
//   * one CTA per (batch, head), two CTAs per SM (every head resident at once);
//   * eight warps: each takes a 16 x 32 block of the queries' and the keys'
//     products, then of G, so all carry equal work between the two barriers;
//   * W lives in registers in fp32 (each thread owns 32 entries in the layout of
//     the G accumulator), with a bf16 hi/lo copy in shared memory for the MMAs;
//   * Q, K, V tiles (64 x 64 bf16, 128-byte swizzle) and the lr tile stream in
//     through a 3-stage TMA ring, so the next chunks load while one computes;
//   * the 64 x 64 x 64 products run on warp-level bf16 MMAs (m16n8k16) with fp32
//     accumulation; in SPLIT precision (the default) the keys' product and G use
//     hi + lo operands (the inputs are exact bf16), so W accumulates its updates
//     at ~16-bit operand precision; SINGLE precision drops the lo products.
// Waits on the TMA barriers are bounded (timeout -> status word, no trap).
#include "tc_kernel.cuh"
#include "tc_util.cuh"
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

using namespace tcu;

constexpr int kNQ = 2;                    // column groups of 64 / kNQ columns (2 measured fastest)
constexpr int kNT = 8 / kNQ;              // n-tiles (8 columns) per warp
constexpr int kLinThreads = 128 * kNQ;    // 4 row blocks x kNQ column groups
constexpr int kLinD = 64;
constexpr int kTile = 64;               // tokens per tile
constexpr int kLinStages = 3;
constexpr uint32_t kTileBytes = kTile * kLinD * 2;   // 8 KB (bf16)
constexpr uint32_t kLrBytes = kTile * 4;             // 256 B
constexpr uint32_t kLinStageBytes = 3 * kTileBytes + 1024;  // Q, K, V, then lr (1 KB slot)

struct LinParams {
  CUtensorMap mQ, mK, mV;  // bf16 {d, T, BH}, box {64, 64, 1}, 128-byte swizzle
  CUtensorMap mLr;         // fp32 {T, BH}, box {64, 1}
  const float* W0;         // [H or B*H][d][d]
  float* Wf;               // [B*H][d][d]
  __nv_bfloat16* O;        // [B*H][T][d]
  int H, T, chunk, n_tiles, w0_per_batch, mse;
  float step;
  MaskBits mask;
  int has_mask;
  int stall;               // test hook: never start the loads, so the first wait runs out
  int split;               // W and eta*R carried as bf16 hi + lo (TTT_PREC_SPLIT)
  int inclusive;           // inclusive order (chunks of one 64-token tile): O -= step tril(Q K^T) (eta R)
  TcCommon cm;
};

// Byte offset of element (row, col) of a 64 x 64 bf16 tile stored with the
// 128-byte swizzle (16-byte chunk index XOR row % 8).
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return (uint32_t)(row * 128 + ((((col >> 3) ^ (row & 7)) << 4) | ((col & 7) << 1)));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A * B on a 16 x 8 x 16 bf16 tile (fp32 accumulate).
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t bf2(float x, float y) { return pack_bf16(x, y); }

__device__ __forceinline__ float bf_lo(float x) { return x - __bfloat162float(__float2bfloat16_rn(x)); }

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(ptx::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(ptx::smem_u32(bar))
      : "memory");
}

__global__ void __launch_bounds__(kLinThreads, 2) linear_chunk_kernel(const __grid_constant__ LinParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage0 = smem;                                        // kLinStages x kLinStageBytes
  uint8_t* wh = smem + kLinStages * kLinStageBytes;               // W hi, swizzled [i][k]
  uint8_t* wl = wh + kTileBytes;                                  // W lo
  uint8_t* rh = wl + kTileBytes;                                  // eta*R hi, swizzled [t][i]
  uint8_t* rl = rh + kTileBytes;                                  // eta*R lo
  uint64_t* full = reinterpret_cast<uint64_t*>(rl + kTileBytes);  // kLinStages barriers
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + kLinStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c4 = lane & 3;
  const int bh = blockIdx.x;
  const int h = bh % p.H;

  if (tid == 0) {
    for (int s = 0; s < kLinStages; ++s) ptx::mbar_init(&full[s], 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();

  int issued = 0;            // tiles whose loads thread 0 has started
  auto issue = [&](int u) {  // tile u into stage u % kLinStages (thread 0)
    const int s = u % kLinStages;
    uint8_t* st = stage0 + s * kLinStageBytes;
    ptx::mbar_expect_tx(&full[s], 3 * kTileBytes + kLrBytes);
    const int t0 = u * kTile;
    ptx::tma_load_3d(st, &p.mQ, &full[s], 0, t0, bh);
    ptx::tma_load_3d(st + kTileBytes, &p.mK, &full[s], 0, t0, bh);
    ptx::tma_load_3d(st + 2 * kTileBytes, &p.mV, &full[s], 0, t0, bh);
    tma_load_2d(st + 3 * kTileBytes, &p.mLr, &full[s], t0, bh);
    issued = u + 1;
  };
  if (tid == 0)
    for (int u = 0; u < kLinStages && u < p.n_tiles && !p.stall; ++u) issue(u);

  // ---- W in registers: warp w owns rows i in [16 mr, 16 mr + 16) and columns
  // [8 kNT nh, 8 kNT (nh + 1)) (mr = w % 4, nh = w / 4), the layout of a
  // 16 x 8 kNT accumulator (kNT n-tiles x 4 values per thread)
  const int mr = warp & 3, nh = warp >> 2;  // row block, column group
  float W[kNT][4];
  {
    const float* w0 = p.W0 + (size_t)(p.w0_per_batch ? bh : h) * kLinD * kLinD;
#pragma unroll
    for (int ln = 0; ln < kNT; ++ln)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = 16 * mr + g + (q >> 1) * 8, j = (kNT * nh + ln) * 8 + 2 * c4 + (q & 1);
        W[ln][q] = w0[i * kLinD + j];
      }
  }
  auto write_w_operands = [&]() {
#pragma unroll
    for (int ln = 0; ln < kNT; ++ln)
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {
        const int i = 16 * mr + g + hq * 8, j = (kNT * nh + ln) * 8 + 2 * c4;
        const float x = W[ln][2 * hq], y = W[ln][2 * hq + 1];
        *reinterpret_cast<uint32_t*>(wh + swz(i, j)) = bf2(x, y);
        *reinterpret_cast<uint32_t*>(wl + swz(i, j)) = bf2(bf_lo(x), bf_lo(y));
      }
  };
  write_w_operands();
  __syncthreads();

  float Gacc[kNT][4];
#pragma unroll
  for (int ln = 0; ln < kNT; ++ln)
#pragma unroll
    for (int q = 0; q < 4; ++q) Gacc[ln][q] = 0.f;

  const int tiles_per_chunk = p.chunk / kTile;
  const uint32_t wh_a = ptx::smem_u32(wh), wl_a = ptx::smem_u32(wl);
  const uint32_t rh_a = ptx::smem_u32(rh), rl_a = ptx::smem_u32(rl);

  for (int u = 0; u < p.n_tiles; ++u) {
    const int s = u % kLinStages;
    uint8_t* st = stage0 + s * kLinStageBytes;
    // wait for the tile (bounded)
    {
      int ok = 1;
      if (lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        uint32_t it = 0;
        while (!ptx::mbar_try_wait(&full[s], (uint32_t)(u / kLinStages) & 1u)) {
          if ((++it & 63u) == 0 && (*abort_flag || globaltimer_ns() - t0 > p.cm.timeout_ns)) {
            *abort_flag = 1;
            set_status(p.cm.status, TTT_ERR_TIMEOUT);
            ok = 0;
            break;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (__syncthreads_or(!ok)) break;
    }
    const int chunk_idx = u / tiles_per_chunk;
    const bool upd = !p.has_mask || mask_bit(p.mask, chunk_idx);
    const bool chunk_end = (u + 1) % tiles_per_chunk == 0 || u + 1 == p.n_tiles;
    const uint32_t sq = ptx::smem_u32(st), sk = sq + kTileBytes;
    const uint8_t* sv = st + 2 * kTileBytes;
    const float* slr = reinterpret_cast<const float*>(st + 3 * kTileBytes);
    const int t_base = u * kTile;

    // ---- phase 1: warp (mr, nh) computes rows [16 mr, +16) x its column group
    // of O = Q W^T and, for an MSE update, of R = K W^T - V (keys' product with
    // W = hi + lo)
    {
      const int r0 = 16 * mr;
      const bool do_r = upd && p.mse;
      float ao[kNT][4], ar[kNT][4];
#pragma unroll
      for (int ln = 0; ln < kNT; ++ln)
#pragma unroll
        for (int q = 0; q < 4; ++q) ao[ln][q] = ar[ln][q] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const int arow = r0 + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int acol = 16 * ks + 8 * (lane >> 4);
        uint32_t aq[4], ak[4];
        ldsm_x4(sq + swz(arow, acol), aq[0], aq[1], aq[2], aq[3]);
        if (do_r) ldsm_x4(sk + swz(arow, acol), ak[0], ak[1], ak[2], ak[3]);
#pragma unroll
        for (int lp = 0; lp < kNT / 2; ++lp) {  // this warp's pairs of n-tiles
          // matrices: (n 0-7, k 0-7), (n 0-7, k 8-15), (n 8-15, k 0-7), (n 8-15, k 8-15)
          const int nrow = 16 * (kNT / 2 * nh + lp) + (lane & 7) + 8 * (lane >> 4);
          const int kcol = 16 * ks + 8 * ((lane >> 3) & 1);
          uint32_t b[4];
          ldsm_x4(wh_a + swz(nrow, kcol), b[0], b[1], b[2], b[3]);
          mma16816(ao[2 * lp], aq, b[0], b[1]);
          mma16816(ao[2 * lp + 1], aq, b[2], b[3]);
          if (do_r) {
            mma16816(ar[2 * lp], ak, b[0], b[1]);
            mma16816(ar[2 * lp + 1], ak, b[2], b[3]);
            if (p.split) {
              ldsm_x4(wl_a + swz(nrow, kcol), b[0], b[1], b[2], b[3]);
              mma16816(ar[2 * lp], ak, b[0], b[1]);
              mma16816(ar[2 * lp + 1], ak, b[2], b[3]);
            }
          }
        }
      }
      // O rows: token t_base + row, bf16 (inclusive order: after the correction below)
      if (!(p.inclusive && upd)) {
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
          const int row = r0 + g + 8 * hq;
          if (t_base + row < p.T) {
            __nv_bfloat16* dst = p.O + ((size_t)bh * p.T + t_base + row) * kLinD;
#pragma unroll
            for (int ln = 0; ln < kNT; ++ln)
              *reinterpret_cast<uint32_t*>(dst + (kNT * nh + ln) * 8 + 2 * c4) = bf2(ao[ln][2 * hq], ao[ln][2 * hq + 1]);
          }
        }
      }
      if (upd) {
        // eta * dl/df -> hi/lo operands, [t][i]: (K W^T - V) for MSE, -V for the
        // inner product
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
          const int row = r0 + g + 8 * hq;
          const float eta = slr[row];
#pragma unroll
          for (int ln = 0; ln < kNT; ++ln) {
            const int col = (kNT * nh + ln) * 8 + 2 * c4;
            const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(sv + swz(row, col));
            const float x = eta * (ar[ln][2 * hq] - __low2float(v2));
            const float y = eta * (ar[ln][2 * hq + 1] - __high2float(v2));
            *reinterpret_cast<uint32_t*>(rh + swz(row, col)) = bf2(x, y);
            *reinterpret_cast<uint32_t*>(rl + swz(row, col)) = bf2(bf_lo(x), bf_lo(y));
          }
        }
      }
    }
    __syncthreads();

    // ---- inclusive order (tutorial page §3: each query sees its own token's
    // update): with one tile per chunk, o_t = W q_t - step sum_{u <= t} (q_t.k_u) eta_u r_u,
    // i.e. O -= step S (eta R) with S = tril(Q K^T). S goes to the W-lo buffer,
    // idle until the chunk-end refresh of the operands.
    if (p.inclusive && upd) {
      const int r0 = 16 * mr;
      float as[kNT][4];
#pragma unroll
      for (int ln = 0; ln < kNT; ++ln)
#pragma unroll
        for (int q = 0; q < 4; ++q) as[ln][q] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {  // over d
        const int arow = r0 + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int acol = 16 * ks + 8 * (lane >> 4);
        uint32_t aq[4];
        ldsm_x4(sq + swz(arow, acol), aq[0], aq[1], aq[2], aq[3]);
#pragma unroll
        for (int lp = 0; lp < kNT / 2; ++lp) {
          const int nrow = 16 * (kNT / 2 * nh + lp) + (lane & 7) + 8 * (lane >> 4);  // key token u
          const int kcol = 16 * ks + 8 * ((lane >> 3) & 1);
          uint32_t b[4];
          ldsm_x4(sk + swz(nrow, kcol), b[0], b[1], b[2], b[3]);
          mma16816(as[2 * lp], aq, b[0], b[1]);
          mma16816(as[2 * lp + 1], aq, b[2], b[3]);
        }
      }
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {
        const int t = r0 + g + 8 * hq;
#pragma unroll
        for (int ln = 0; ln < kNT; ++ln) {
          const int u = (kNT * nh + ln) * 8 + 2 * c4;
          const float x = u <= t ? as[ln][2 * hq] : 0.f;
          const float y = u + 1 <= t ? as[ln][2 * hq + 1] : 0.f;
          *reinterpret_cast<uint32_t*>(wl + swz(t, u)) = bf2(x, y);
        }
      }
      __syncthreads();
      float ac[kNT][4];
#pragma unroll
      for (int ln = 0; ln < kNT; ++ln)
#pragma unroll
        for (int q = 0; q < 4; ++q) ac[ln][q] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {  // over key tokens u
        const int arow = r0 + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int acol = 16 * ks + 8 * (lane >> 4);
        uint32_t a[4];
        ldsm_x4(wl_a + swz(arow, acol), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int lp = 0; lp < kNT / 2; ++lp) {
          // B = eta R: rows u (k), cols i (n), stored [u][i] -> transposed loads
          const int kt = 16 * ks + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int ic = 16 * (kNT / 2 * nh + lp) + 8 * (lane >> 4);
          uint32_t b[4];
          ldsm_x4_t(rh_a + swz(kt, ic), b[0], b[1], b[2], b[3]);
          mma16816(ac[2 * lp], a, b[0], b[1]);
          mma16816(ac[2 * lp + 1], a, b[2], b[3]);
          if (p.split) {
            ldsm_x4_t(rl_a + swz(kt, ic), b[0], b[1], b[2], b[3]);
            mma16816(ac[2 * lp], a, b[0], b[1]);
            mma16816(ac[2 * lp + 1], a, b[2], b[3]);
          }
        }
      }
      // O = Q W^T - step S (eta R): the first product again (phase 1's values
      // are gone), then the correction, stored as bf16
      float ao[kNT][4];
#pragma unroll
      for (int ln = 0; ln < kNT; ++ln)
#pragma unroll
        for (int q = 0; q < 4; ++q) ao[ln][q] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const int arow = r0 + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int acol = 16 * ks + 8 * (lane >> 4);
        uint32_t aq[4];
        ldsm_x4(sq + swz(arow, acol), aq[0], aq[1], aq[2], aq[3]);
#pragma unroll
        for (int lp = 0; lp < kNT / 2; ++lp) {
          const int nrow = 16 * (kNT / 2 * nh + lp) + (lane & 7) + 8 * (lane >> 4);
          const int kcol = 16 * ks + 8 * ((lane >> 3) & 1);
          uint32_t b[4];
          ldsm_x4(wh_a + swz(nrow, kcol), b[0], b[1], b[2], b[3]);
          mma16816(ao[2 * lp], aq, b[0], b[1]);
          mma16816(ao[2 * lp + 1], aq, b[2], b[3]);
        }
      }
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {
        const int row = r0 + g + 8 * hq;
        if (t_base + row < p.T) {
          __nv_bfloat16* dst = p.O + ((size_t)bh * p.T + t_base + row) * kLinD;
#pragma unroll
          for (int ln = 0; ln < kNT; ++ln)
            *reinterpret_cast<uint32_t*>(dst + (kNT * nh + ln) * 8 + 2 * c4) =
                bf2(ao[ln][2 * hq] - p.step * ac[ln][2 * hq], ao[ln][2 * hq + 1] - p.step * ac[ln][2 * hq + 1]);
        }
      }
      __syncthreads();  // S in the W-lo buffer is read; the chunk end may refresh it
    }

    // ---- phase 2: G += (eta R)^T K, warp (mr, nh): rows i in [16 mr, +16),
    // columns j in its column group
    if (upd) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {  // 16 tokens per step
        // A = (eta R)^T: rows i, cols t; stored [t][i] -> transposed loads
        const int trow = 16 * ks + (lane & 7) + 8 * (lane >> 4);
        const int icol = 16 * mr + 8 * ((lane >> 3) & 1);
        uint32_t ah[4], al[4];
        ldsm_x4_t(rh_a + swz(trow, icol), ah[0], ah[1], ah[2], ah[3]);
        ldsm_x4_t(rl_a + swz(trow, icol), al[0], al[1], al[2], al[3]);
#pragma unroll
        for (int lp = 0; lp < kNT / 2; ++lp) {
          // B = K: rows t (k), cols j (n), stored [t][j] -> transposed loads;
          // matrices: (t 0-7, j 0-7), (t 8-15, j 0-7), (t 0-7, j 8-15), (t 8-15, j 8-15)
          const int kt = 16 * ks + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int jc = 16 * (kNT / 2 * nh + lp) + 8 * (lane >> 4);
          uint32_t b[4];
          ldsm_x4_t(sk + swz(kt, jc), b[0], b[1], b[2], b[3]);
          mma16816(Gacc[2 * lp], ah, b[0], b[1]);
          mma16816(Gacc[2 * lp + 1], ah, b[2], b[3]);
          if (p.split) {
            mma16816(Gacc[2 * lp], al, b[0], b[1]);
            mma16816(Gacc[2 * lp + 1], al, b[2], b[3]);
          }
        }
      }
      if (chunk_end) {
#pragma unroll
        for (int ln = 0; ln < kNT; ++ln)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            W[ln][q] -= p.step * Gacc[ln][q];
            Gacc[ln][q] = 0.f;
          }
        write_w_operands();  // phase 1 of this tile is finished; nobody reads W now
      }
    }
    __syncthreads();  // the stage and the operands may be reused
    if (tid == 0 && u + kLinStages < p.n_tiles) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(u + kLinStages);
    }
  }

  if (!*abort_flag) {
    float* wf = p.Wf + (size_t)bh * kLinD * kLinD;
#pragma unroll
    for (int ln = 0; ln < kNT; ++ln)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = 16 * mr + g + (q >> 1) * 8, j = (kNT * nh + ln) * 8 + 2 * c4 + (q & 1);
        wf[i * kLinD + j] = W[ln][q];
      }
  } else if (tid == 0) {
    // let the copies in flight land before the CTA exits (bounded)
    for (int k = issued > kLinStages ? issued - kLinStages : 0; k < issued; ++k) {
      const uint64_t t0 = globaltimer_ns();
      while (!ptx::mbar_try_wait(&full[k % kLinStages], (uint32_t)(k / kLinStages) & 1u) &&
             globaltimer_ns() - t0 < p.cm.timeout_ns) {
      }
    }
  }
}

constexpr size_t kLinSmem = 1024 + kLinStages * kLinStageBytes + 4 * kTileBytes + 64;

}  // namespace

int g_linear_stall_next = 0;  // test hook: the next launch withholds its loads

bool linear_supported(const ttt_cfg& g) {
  // (no momentum buffer: the kernel keeps W alone in registers; with one
  // matrix, per-matrix rates have the per-token layout)
  // (the inclusive order's dual form is built for chunks of one 64-token tile)
  return g.fast_net == TTT_NET_LINEAR && g.dtype == TTT_DTYPE_BF16 && g.d == kLinD && g.muon == 0 &&
         g.wnorm == 0 && g.momentum == 0.f && g.chunk % kTile == 0 && g.T % 4 == 0 &&
         (g.mode == TTT_MODE_SHIFTED || (g.mode == TTT_MODE_INCLUSIVE && g.chunk == kTile));
}

size_t linear_workspace_bytes(const ttt_cfg&) { return kStatusBytes; }

int linear_run(const Call& c) {
  const ttt_cfg& g = c.cfg;
  if (!c.mask_all && c.n_chunks > kMaxMaskChunks) return TTT_ERR_UNSUPPORTED;
  LinParams p{};
  const int BH = g.B * g.H;
  bool ok = true;
  ok &= map3(&p.mQ, c.Q, kLinD, g.T, BH, 64, 64);
  ok &= map3(&p.mK, c.K, kLinD, g.T, BH, 64, 64);
  ok &= map3(&p.mV, c.V, kLinD, g.T, BH, 64, 64);
  {
    auto fn = encode_fn();
    if (!fn) return TTT_ERR_CUDA;
    cuuint64_t gd[2] = {(cuuint64_t)g.T, (cuuint64_t)BH};
    cuuint64_t gs[1] = {(cuuint64_t)g.T * 4};
    cuuint32_t bx[2] = {64, 1};
    cuuint32_t es[2] = {1, 1};
    ok &= fn(&p.mLr, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(c.lr), gd, gs, bx, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  if (!ok) return TTT_ERR_CUDA;
  p.W0 = c.W0[0];
  p.Wf = c.Wf[0];
  p.O = static_cast<__nv_bfloat16*>(c.O);
  p.H = g.H;
  p.T = g.T;
  p.chunk = g.chunk;
  p.n_tiles = (g.T + kTile - 1) / kTile;
  p.w0_per_batch = g.w0_per_batch;
  p.mse = g.loss == TTT_LOSS_MSE ? 1 : 0;
  p.step = g.step;
  p.has_mask = c.mask_all ? 0 : 1;
  p.stall = g_linear_stall_next ? 1 : 0;
  p.split = g.precision == TTT_PREC_SPLIT ? 1 : 0;
  p.inclusive = g.mode == TTT_MODE_INCLUSIVE ? 1 : 0;
  g_linear_stall_next = 0;
  if (p.has_mask)
    for (int i = 0; i < c.n_chunks; ++i)
      if (c.mask[i]) p.mask.w[i >> 5] |= 1u << (i & 31);
  p.cm = TcCommon{reinterpret_cast<int*>(c.ws), (unsigned long long)g.timeout_us * 1000ull};
  if (cudaFuncSetAttribute(linear_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLinSmem) !=
      cudaSuccess)
    return TTT_ERR_CUDA;
  prof_before(TTT_KERNEL_LINEAR, c.stream);
  linear_chunk_kernel<<<BH, kLinThreads, kLinSmem, c.stream>>>(p);
  prof_after(TTT_KERNEL_LINEAR, c.stream);
  return cudaGetLastError() == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

}  // namespace ttt

// Test hook (declared in ttt_debug.h): the next linear-path launch starts no
// loads, so its first bounded wait expires and it records TTT_ERR_TIMEOUT.
extern "C" void ttt_dbg_stall_next_linear(void) { ttt::g_linear_stall_next = 1; }
