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
#include <atomic>
#include <cstring>
#include <mutex>

#include "../../include/ttt_debug.h"
#include "tc_kernel.cuh"
#include "tc_mc.cuh"
#include "tc_pair.cuh"
#include "tc_util.cuh"
#include "ttt_internal.h"
#include "ttt_ns.h"

namespace ttt {
namespace {

using namespace tcu;

int g_split_mask = 7;  // test hook: stages that carry split operands in SPLIT precision
std::atomic<int> g_stall_next_fwd{0};  // test hook: the next forward launch withholds its loads
bool g_grad_pairs = true;               // test hook: the chunk gradient on CTA pairs (single-GPU build)
// (the apply runs on CTA pairs in the single-GPU build whenever a chunk has two token tiles)


// ============================================================ forward, multicast
// Forward of the fast net on 128-token tiles (LaCT page §2.1): the clusters'
// CTAs take consecutive token tiles of one (b, h, hidden slice) and share that
// slice's weights by TMA multicast (each CTA loads a share of the weight
// boxes); the token rows are each CTA's own.
//   query tile (128 hidden): [A|B] = Q [W1;W3]^T -> H_q = silu(A) * B    (apply-1)
//   key tile (64 hidden):    [A|B] = K [W1;W3]^T, Dm = Y W2 -> DA, He, DB (SwiGLU
//               backward, scaled by each token's rates), the gradient kernel's E
//               operand; Y = dl/df = -V for the inner-product loss, f(k) - V for MSE
//   key-hidden tile (64 hidden, MSE): [A|B] = K [W1;W3]^T -> H_k = silu(A) * B as
//               split operands, from which the next kernel forms Y = H_k W2^T - V
// Every MMA of a query tile is N = 256 and the split weight halves of the Dm
// product share one N = 128 MMA (W2 hi | W2 lo side by side): one thread issues
// the MMAs, and products narrower than that leave the tensor pipe waiting on
// the issuing thread between k-blocks.
// TMEM of one 256-column accumulator: query [A|B] in columns 0-255; key and
// key-hidden [A|B] in 0-127, Dm (hi part, lo part) in 128-191 and 192-255.
struct FwdMcParams {
  CUtensorMap mQ, mK, mV;  // 3D {d, T, BH}, box {64, 128, 1}
  CUtensorMap mW, mWl;     // bf16 shadows (hi, lo) [3BH][d][dh] as 3D {dh, d, 3BH}, box {64, 64, 1}
  CUtensorMap sHq;         // stores: H_q {dh, Cp, BH}, box {32, 32, 1}, 64-byte swizzle
  CUtensorMap sE, sEl;     //         E (hi, lo) {dh, Cp, 3BH}, box {32, 32, 1}
  const float* lr;
  bf16* Hq;                // [BH][Cp][dh]
  bf16* E;                 // [BH][3][Cp][dh]: DA, He, DB
  bf16* El;                // low halves of E (split precision)
  int d, dh, T, Cp, chunk_start, valid;
  int n_tok, groups, n_jq, BH, cs;  // n_jq: 128-wide hidden slices
  int q, k, h;             // which kinds of tiles this launch computes (query, key, key-hidden)
  int w_split, e_split;
  int lr_stride;           // 1: one rate per token; 3: one per token and matrix (W1, W2, W3)
  int mse;                 // key tiles: Dm = Y W2 with Y (hi, lo) from mY / mYl (MSE loss)
  CUtensorMap mY, mYl;     // Y (hi, lo) {d, Cp, BH}, box {64, 128, 1}: tokens relative to the chunk
  CUtensorMap sHk, sHkl;   // stores: H_k (hi, lo) {dh, Cp, BH}, box {32, 32, 1}, 64-byte swizzle
  TcCommon cm;
};

// EW: epilogue warps (4, or 8 = two per TMEM lane quarter, each taking half of
// a tile's hidden columns). Eight pay where the epilogue bounds the tile (a
// short K = d loop: d < 512; imageset_1m's forward 5.71 -> 4.47 ms); where d
// is larger the tile is bound by its operand ingest and the four extra warps
// only compete with the one thread that issues the MMAs (lm_chunk2k 128 -> 134 us).
template <int EW>
struct FwdMcOpT {
  using Params = FwdMcParams;

  struct Tile {
    int bh, hid0, tok, kind;  // kind: 0 query (128 hidden), 1 key, 2 key-hidden (64 hidden)
    bool is_k, real;
  };
  static constexpr int kStages = 4;
  static constexpr int kStageBytes = kABytes + 4 * kBox;
  static constexpr int kAccCols = 256;
  static constexpr int kEpiWarps = EW;
  static constexpr uint32_t kEpiBytes = 8 * 4096;  // 4 x 8 KB or 8 x 4 KB of staging (two or one 4 KB buffers per warp)

  // items per (b, h, 128-wide hidden slice, token group): one query tile, two
  // key-hidden tiles, two key tiles (those the launch computes)
  static __device__ int n_sub(const Params& p) { return p.q + 2 * p.h + 2 * p.k; }
  static __device__ int num_work(const Params& p) { return p.BH * p.n_jq * p.groups * n_sub(p); }
  static __device__ void tile_of(const Params& p, int w, int rank, Tile& t) {
    const int ns = n_sub(p);
    int c = w % ns;
    w /= ns;
    const int g = w % p.groups;
    w /= p.groups;
    const int jq = w % p.n_jq;
    t.bh = w / p.n_jq;
    t.hid0 = jq * 128;
    if (c < p.q) {
      t.kind = 0;
    } else {
      c -= p.q;
      t.kind = (p.h && c < 2) ? 2 : 1;
      t.hid0 += 64 * (c & 1);
    }
    t.is_k = t.kind == 1;
    t.tok = g * p.cs + rank;
    t.real = t.tok < p.n_tok;
  }
  static __device__ int num_kblocks(const Params& p, const Tile& t) { return (t.is_k ? 2 : 1) * (p.d / BK); }
  // weight boxes of k-block kb: queries [W1, W1', W3, W3'] (hi; ' = the next
  // 64 hidden); keys and key hiddens, segment 0 [W1 hi, W3 hi, W1 lo, W3 lo];
  // keys, segment 1 [W2 hi, W2 lo]
  static __device__ int n_boxes(const Params& p, const Tile& t, int kb) {
    if (t.kind == 0) return 4;
    return (kb < p.d / BK ? 2 : 1) * (p.w_split ? 2 : 1);
  }
  static __device__ bool y_seg(const Params& p, const Tile& t, int kb) { return p.mse && t.is_k && kb >= p.d / BK; }
  static __device__ uint32_t stage_tx(const Params& p, const Tile& t, int kb) {
    return kABytes * (y_seg(p, t, kb) ? 2u : 1u) + (uint32_t)n_boxes(p, t, kb) * kBox;
  }
  static __device__ void produce(const Params& p, const Tile& t, int kb, uint8_t* st, uint64_t* bar, int rank,
                                 int cs, uint16_t mask) {
    const int nk = p.d / BK;
    const bool seg1 = t.is_k && kb >= nk;
    const int k = (seg1 ? kb - nk : kb) * BK;
    // the Y segment (MSE) keeps its rows hi at 0 and lo at kABytes, its W2 boxes two slots on
    const int wslot = y_seg(p, t, kb) ? 2 : 0;
    if (y_seg(p, t, kb)) {
      ptx::tma_load_3d(st, &p.mY, bar, k, t.tok * BM, t.bh);
      ptx::tma_load_3d(st + kABytes, &p.mYl, bar, k, t.tok * BM, t.bh);
    } else {
      const CUtensorMap* x = seg1 ? &p.mV : (t.kind == 0 ? &p.mQ : &p.mK);
      ptx::tma_load_3d(st, x, bar, k, p.chunk_start + t.tok * BM, t.bh);
    }
    const int z = t.bh * 3;
    const int nb = n_boxes(p, t, kb);
    for (int b = rank; b < nb; b += cs) {
      const bool q = t.kind == 0;
      const bool lo = q ? false : seg1 ? b == 1 : b >= 2;
      const int zz = q ? z + (b >= 2 ? 2 : 0) : seg1 ? z + 1 : z + ((b & 1) ? 2 : 0);
      const int col = t.hid0 + (q ? 64 * (b & 1) : 0);
      ptx::tma_load_3d_shared(st + kABytes + (b + wslot) * kBox, lo ? &p.mWl : &p.mW, bar, col, k, zz, mask);
    }
  }
  static __device__ void consume(const Params& p, const Tile& t, int kb, uint32_t st, uint32_t tmem) {
    const int nk = p.d / BK;
    const uint32_t a = st, b = st + kABytes;
    if (t.kind == 0) {
      // [A|B] over 128 hidden: one N = 256 MMA per 16 of K
      constexpr uint32_t id = ptx::idesc_bf16(128, 256, false, true);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) ptx::mma_bf16(tmem, kdesc(a, kk), mdesc(b, kk), id, (kb | kk) != 0);
    } else if (kb < nk) {
      constexpr uint32_t id = ptx::idesc_bf16(128, 128, false, true);
      const bool two = t.kind != 0 && p.w_split;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        ptx::mma_bf16(tmem, kdesc(a, kk), mdesc(b, kk), id, (kb | kk) != 0);
        if (two) ptx::mma_bf16(tmem, kdesc(a, kk), mdesc(b + 2 * kBox, kk), id, 1u);
      }
    } else if (p.mse) {
      // Dm = Y W2 with both split: Yh [W2h | W2l] (N = 128: the hi part in
      // columns 128-191, the lo part in 192-255) + Yl W2h (into the hi part)
      const int k2 = kb - nk;
      constexpr uint32_t id2 = ptx::idesc_bf16(128, 128, false, true);
      constexpr uint32_t id1 = ptx::idesc_bf16(128, 64, false, true);
      const uint32_t yl = st + kABytes, wh = st + kABytes + 2 * kBox;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        ptx::mma_bf16(tmem + 128, kdesc(a, kk), mdesc(wh, kk), id2, (k2 | kk) != 0);
        ptx::mma_bf16(tmem + 128, kdesc(yl, kk), mdesc(wh, kk), id1, 1u);
      }
    } else {
      // Dm = V [W2h | W2l] (N = 128, hi and lo parts side by side), or V W2h
      const int k2 = kb - nk;
      if (p.w_split) {
        constexpr uint32_t id = ptx::idesc_bf16(128, 128, false, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) ptx::mma_bf16(tmem + 128, kdesc(a, kk), mdesc(b, kk), id, (k2 | kk) != 0);
      } else {
        constexpr uint32_t id = ptx::idesc_bf16(128, 64, false, true);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) ptx::mma_bf16(tmem + 128, kdesc(a, kk), mdesc(b, kk), id, (k2 | kk) != 0);
      }
    }
  }
  // The SwiGLU (backward) epilogue through shared memory: eight warps, two per
  // TMEM lane quarter, each taking half of the tile's hidden columns; each
  // stages its 32 x 32 blocks (64-byte swizzle) in its buffer and writes them
  // with TMA stores, hi and lo halves alike. Rows past the chunk's tokens get
  // lr 0 (zero E rows) and zero H_q rows.
  // the key rows' rates (W1, W2, W3), loaded before the accumulator wait;
  // rows past the chunk's tokens get rate 0, so their E rows are zero
  struct Pre {
    float e1, e2, e3;
  };
  static __device__ Pre pre(const Params& p, const Tile& t, int r) {
    Pre x{0.f, 0.f, 0.f};
    const int tl = t.tok * BM + r;
    if (t.is_k && t.real && tl < p.valid) {
      const float* lp = p.lr + ((size_t)t.bh * p.T + p.chunk_start + tl) * p.lr_stride;
      x.e1 = lp[0];
      x.e2 = p.lr_stride > 1 ? lp[1] : x.e1;
      x.e3 = p.lr_stride > 1 ? lp[2] : x.e1;
    }
    return x;
  }
  static __device__ void epilogue(const Params& p, const Tile& t, uint32_t tm, int r, uint8_t* epi,
                                  uint32_t& es, const Pre& pr, int half) {
    if (!t.real) return;  // a CTA past the chunk's last token tile stores nothing
    const int lane = r & 31;
    const int tl = t.tok * BM + r;        // token index inside the chunk
    const int row0 = tl - lane;           // this warp's first row (warp-uniform)
    const bool valid = tl < p.valid;
    const int j0 = t.hid0;
    // stage one 32 x 32 block and store it at (column x, this warp's rows, plane z)
    auto put = [&](const float* v, bool lo, const CUtensorMap* mh, const CUtensorMap* ml, int x, int z) {
      uint8_t* buf = epi + (EW == 4 ? (es & 1u) * 4096u : 0u);
      if (lane == 0) {  // the store that used this buffer has read it
        if (EW == 4)
          ptx::bulk_wait_read<1>();
        else
          ptx::bulk_wait_read<0>();
      }
      __syncwarp();
      if (lo)
        stage_bf16x32<true>(buf, lane, v);
      else
        stage_bf16x32<false>(buf, lane, v);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_3d(mh, buf, x, row0, z);
        if (lo) ptx::tma_store_3d(ml, buf + 2048, x, row0, z);
        ptx::bulk_commit();
      }
      ++es;
    };
    float va[32], vb[32];
    if (!t.is_k) {
      const bool hk = t.kind == 2;  // key hiddens: split operands of the MSE's Y = H_k W2^T - V
      const int wa = hk ? 64 : 128;  // hidden columns of the tile: A in [0, wa), B in [wa, 2 wa)
      const int cw = EW == 8 ? wa / 2 : wa;  // this warp's columns
      for (int c = half * cw; c < (half + 1) * cw; c += 32) {
        ptx::tmem_ld32(tm + c, va);
        ptx::tmem_ld32(tm + wa + c, vb);
#pragma unroll
        for (int i = 0; i < 32; ++i) va[i] = valid ? va[i] * sigmoid_fast(va[i]) * vb[i] : 0.f;
        if (hk)
          put(va, true, &p.sHk, &p.sHkl, j0 + c, t.bh);
        else
          put(va, false, &p.sHq, &p.sHq, j0 + c, t.bh);
      }
    } else {
      // the rates of W1, W2, W3 (one shared rate, or one per matrix; 0 past the chunk)
      const float e1 = pr.e1, e2 = pr.e2, e3 = pr.e3;
      const bool lo = p.e_split != 0;
      float vd[32];
      for (int c = 32 * half; c < 64; c += (EW == 8 ? 64 : 32)) {
        ptx::tmem_ld32(tm + c, va);
        ptx::tmem_ld32(tm + 64 + c, vb);
        ptx::tmem_ld32(tm + 128 + c, vd);
        float oh[32];
        if (p.w_split) {  // Dm's lo part
          ptx::tmem_ld32(tm + 192 + c, oh);
#pragma unroll
          for (int i = 0; i < 32; ++i) vd[i] += oh[i];
        }
        // inner product: Dm = V W2 and dl/dh = -Dm, G2 = V^T (-lr2 H);
        // MSE: Dm = Y W2 = dl/dh, G2 = Y^T (lr2 H)
        const float sgn = p.mse ? 1.f : -1.f;
        const float s1 = sgn * e1, s2 = sgn * e2, s3 = sgn * e3;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float a = va[i], b = vb[i];
          const float g1 = s1 * vd[i];          // lr1 * dl/dh
          const float g3 = s3 * vd[i];          // lr3 * dl/dh
          const float sg = sigmoid_fast(a);
          const float s = a * sg;
          oh[i] = s2 * s * b;                   // the G2 operand He
          va[i] = g1 * b * sg * (1.f + a * (1.f - sg));
          vb[i] = g3 * s;
        }
        const int z = t.bh * 3;
        put(va, lo, &p.sE, &p.sEl, j0 + c, z);
        put(oh, lo, &p.sE, &p.sEl, j0 + c, z + 1);
        put(vb, lo, &p.sE, &p.sEl, j0 + c, z + 2);
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

// ============================================================ MSE: Y = H_k W2^T - V
// The keys' output error of the MSE loss (tutorial page §3: l = 1/2 ||f(k) - v||^2,
// dl/df = f(k) - v) for the key rows of a chunk, as bf16 (hi, lo) operands
// [BH][Cp][d] (tokens relative to the chunk; rows past its tokens are zero).
// H_k and W2 are both split: every product is Hh Wh + Hh Wl + Hl Wh.
struct YOp {
  struct Params {
    CUtensorMap mH, mHl;    // H_k (hi, lo) {dh, Cp, BH}, box {64, 128, 1}
    CUtensorMap mW2, mW2l;  // shadows (hi, lo) {dh, d, 3BH}, box {64, 128, 1}
    const bf16* V;          // [BH][T][d]
    bf16* Y;                // [BH][Cp][d]
    bf16* Yl;
    int d, dh, T, Cp, chunk_start, valid, m_tiles, n_tiles;
    TcCommon cm;
  };
  struct Tile {
    int bh, row0, n0;
  };
  static constexpr int BN = 128;
  static constexpr int kStages = 3;
  static constexpr int kStageBytes = 4 * kABytes;  // [H hi | H lo | W2 hi | W2 lo], 128 x 64 each
  static constexpr int kTmemCols = 128;

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
    ptx::tma_load_3d(st + kABytes, &p.mHl, bar, kb * BK, t.row0, t.bh);
    ptx::tma_load_3d(st + 2 * kABytes, &p.mW2, bar, kb * BK, t.n0, t.bh * 3 + 1);
    ptx::tma_load_3d(st + 3 * kABytes, &p.mW2l, bar, kb * BK, t.n0, t.bh * 3 + 1);
  }
  static __device__ void consume(const Params&, const Tile&, int kb, uint32_t st, uint32_t tmem) {
    constexpr uint32_t id = ptx::idesc_bf16(128, BN, false, false);
    const uint32_t hh = st, hl = st + kABytes, wh = st + 2 * kABytes, wl = st + 3 * kABytes;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      ptx::mma_bf16(tmem, kdesc(hh, kk), kdesc(wh, kk), id, (kb | kk) != 0);
      ptx::mma_bf16(tmem, kdesc(hh, kk), kdesc(wl, kk), id, 1u);
      ptx::mma_bf16(tmem, kdesc(hl, kk), kdesc(wh, kk), id, 1u);
    }
  }
  static __device__ void epilogue(const Params& p, const Tile& t, uint32_t tm, int r, float*, bool ok) {
    if (!ok) return;
    const int tl = t.row0 + r;  // token index inside the chunk
    const bool valid = tl < p.valid;
    const bf16* vrow = p.V + ((size_t)t.bh * p.T + p.chunk_start + tl) * p.d;
    const size_t o = ((size_t)t.bh * p.Cp + tl) * p.d;
    float v[32];
    for (int c = 0; c < BN; c += 32) {
      const int n = t.n0 + c;
      if (n >= p.d) break;
      ptx::tmem_ld32(tm + c, v);
      if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(vrow + n);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 w = src[q];
          const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v[8 * q + 2 * e] -= __uint_as_float(u[e] << 16);
            v[8 * q + 2 * e + 1] -= __uint_as_float(u[e] & 0xffff0000u);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
      st_bf16pair32(p.Y + o + n, p.Yl + o + n, v);
    }
  }
};

// ============================================================ chunk gradients, multicast
// Cluster of cs CTAs per work item (z, n-block, token split, row group): CTA
// `rank` computes rows [128 (g cs + rank), +128) of G_z^T (d x dh) over the
// item's tokens; the E operand (the item's dh columns) is the same for every
// rank and is multicast, each CTA loading a share of its 64-column boxes. With
// multicast cs = ceil(d/128) and one row group; without it cs = 1 and
// ceil(d/128) row groups.
//   z = bh*3 + j:  j=0  G1^T = K^T DA;  j=1  G2 = V^T He;  j=2  G3^T = K^T DB
// With split E (hi + lo) both halves sit in one stage and every A tile feeds
// two MMAs.
template <int BN, bool MSE = false>
struct GradMcOp {
  struct Params {
    CUtensorMap mK4, mV4;  // 4D {d, C, n_full, BH}, box {64, 32, 1, 1}  (full chunks)
    CUtensorMap mK3, mV3;  // 3D {d, T, BH}, box {64, 32, 1}            (ragged last chunk)
    CUtensorMap mE, mEl;   // 3D {dh, Cp, 3BH}, box {64, 32, 1}
    CUtensorMap mY, mYl;   // MSE: Y (hi, lo) {d, Cp, BH}, box {64, 32, 1}, G2's operand instead of V
    float* G;              // [Z][d][dh] fp32 (splits == 1)
    float* split_out;      // [splits][Z][d][dh] fp32 (splits > 1)
    int d, dh, Z, chunk_idx, chunk_start, valid, use4d, nt, splits, kb_per_split, e_split;
    int mg, cs;            // row groups per item and CTAs per cluster (mg * cs = ceil(d / 128))
    // Newton-Schulz input (splits == 1, Xh != NULL): instead of fp32 G the
    // epilogue writes the gradient (or the momentum buffer B <- mu B + G, with
    // mom != NULL) as bf16 (hi, lo) operands and, per row and column tile, the
    // sum of squares nsq[(z d + m) nt + n0 / BN] for the Frobenius norm
    bf16* Xh;
    bf16* Xl;
    float* mom;
    float mu;
    float* nsq;
    TcCommon cm;
  };
  struct Tile {
    int z, bh, j, m0, n0, kb0, nkb, split;
  };
  // 32 tokens per stage: five stages (200 KB) keep four in flight
  static constexpr int kTok = 32;
  static constexpr uint32_t kBoxG = 64 * kTok * 2;       // one 64 x 32 box
  static constexpr uint32_t kAB = 2 * kBoxG;              // A: 128 rows of d
  static constexpr uint32_t kEB = (BN / 64) * kBoxG;      // one half of E
  // MSE: the stage also holds the low half of Y (G2's A operand, computed)
  static constexpr int kStages = MSE ? 4 : 5;
  static constexpr int kStageBytes = kAB + 2 * kEB + (MSE ? kAB : 0);
  static constexpr int kAccCols = BN;
  static constexpr int kEpiWarps = 4;
  static constexpr uint32_t kEpiBytes = 0;

  static __device__ int num_work(const Params& p) { return p.Z * p.nt * p.mg * p.splits; }
  static __device__ void tile_of(const Params& p, int w, int rank, Tile& t) {
    const int per_split = p.Z * p.nt * p.mg;
    t.split = w / per_split;
    int r = w % per_split;
    const int g = r % p.mg;
    r /= p.mg;
    t.z = r / p.nt;
    t.n0 = (r % p.nt) * BN;
    t.bh = t.z / 3;
    t.j = t.z % 3;
    t.m0 = (g * p.cs + rank) * BM;
    const int total = (p.valid + kTok - 1) / kTok;
    t.kb0 = t.split * p.kb_per_split;
    t.nkb = max(0, min(total, t.kb0 + p.kb_per_split) - t.kb0);
  }
  static __device__ int num_kblocks(const Params&, const Tile& t) { return t.nkb; }
  static __device__ uint32_t stage_tx(const Params& p, const Tile& t, int) {
    return kAB + (p.e_split ? 2u : 1u) * kEB + ((MSE && t.j == 1) ? kAB : 0u);
  }
  static __device__ void produce(const Params& p, const Tile& t, int kb, uint8_t* st, uint64_t* bar, int rank,
                                 int cs, uint16_t mask) {
    const int tok = (t.kb0 + kb) * kTok;
    if (MSE && t.j == 1) {
      // G2 = Y^T He: Y (hi, lo) of the chunk's tokens, relative to its start
      for (int g = 0; g < 2; ++g) {
        ptx::tma_load_3d(st + g * kBoxG, &p.mY, bar, t.m0 + g * 64, tok, t.bh);
        ptx::tma_load_3d(st + kAB + 2 * kEB + g * kBoxG, &p.mYl, bar, t.m0 + g * 64, tok, t.bh);
      }
    } else
    for (int g = 0; g < 2; ++g) {
      if (p.use4d)
        ptx::tma_load_4d(st + g * kBoxG, t.j == 1 ? &p.mV4 : &p.mK4, bar, t.m0 + g * 64, tok, p.chunk_idx, t.bh);
      else
        ptx::tma_load_3d(st + g * kBoxG, t.j == 1 ? &p.mV3 : &p.mK3, bar, t.m0 + g * 64, p.chunk_start + tok, t.bh);
    }
    constexpr int nb = BN / 64;
    const int boxes = nb * (p.e_split ? 2 : 1);
    for (int b = rank; b < boxes; b += cs) {
      const int half = b / nb, g = b % nb;
      ptx::tma_load_3d_shared(st + kAB + half * kEB + g * kBoxG, half ? &p.mEl : &p.mE, bar, t.n0 + g * 64, tok,
                          t.z, mask);
    }
  }
  static __device__ void consume(const Params& p, const Tile& t, int kb, uint32_t st, uint32_t tmem) {
    constexpr uint32_t id = ptx::idesc_bf16(128, BN, true, true);
    const uint32_t eh = st + kAB, el = eh + kEB;
    const bool ylo = MSE && t.j == 1;  // a computed A operand: three products
    // MN-major operands of 64-wide groups kBoxG apart, 16 tokens per MMA
#pragma unroll
    for (int kk = 0; kk < kTok / 16; ++kk) {
      const uint64_t a = ptx::sdesc(st + kk * 2048, kBoxG, 1024);
      ptx::mma_bf16(tmem, a, ptx::sdesc(eh + kk * 2048, kBoxG, 1024), id, (kb | kk) != 0);
      if (p.e_split) ptx::mma_bf16(tmem, a, ptx::sdesc(el + kk * 2048, kBoxG, 1024), id, 1u);
      if (ylo) {
        const uint64_t al = ptx::sdesc(st + kAB + 2 * kEB + kk * 2048, kBoxG, 1024);
        ptx::mma_bf16(tmem, al, ptx::sdesc(eh + kk * 2048, kBoxG, 1024), id, 1u);
      }
    }
  }
  struct Pre {};
  static __device__ Pre pre(const Params&, const Tile&, int) { return {}; }
  static __device__ void epilogue(const Params& p, const Tile& t, uint32_t tm, int r, uint8_t*, uint32_t&,
                                  const Pre&, int) {
    const int m = t.m0 + r;
    float v[32];
    if (p.Xh && p.splits == 1) {
      float ss = 0.f;
      for (int c = 0; c < BN; c += 32) {
        ptx::tmem_ld32(tm + c, v);
        if (m < p.d) {
          const size_t o = ((size_t)t.z * p.d + m) * p.dh + t.n0 + c;
          if (p.mom) {
            float4* mb = reinterpret_cast<float4*>(p.mom + o);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 b = mb[q];
              v[4 * q + 0] = fmaf(p.mu, b.x, v[4 * q + 0]);
              v[4 * q + 1] = fmaf(p.mu, b.y, v[4 * q + 1]);
              v[4 * q + 2] = fmaf(p.mu, b.z, v[4 * q + 2]);
              v[4 * q + 3] = fmaf(p.mu, b.w, v[4 * q + 3]);
              mb[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
          }
          st_bf16pair32(p.Xh + o, p.Xl + o, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) ss = fmaf(v[i], v[i], ss);
        }
      }
      if (m < p.d) p.nsq[((size_t)t.z * p.d + m) * p.nt + t.n0 / BN] = ss;
      return;
    }
    float* dst = p.splits > 1 ? p.split_out + (size_t)t.split * p.Z * p.d * p.dh : p.G;
    for (int c = 0; c < BN; c += 32) {
      ptx::tmem_ld32(tm + c, v);
      if (m < p.d) st_f32x32(dst + ((size_t)t.z * p.d + m) * p.dh + t.n0 + c, v);
    }
  }
};

#if TTT_HAS_MULTICAST
// ============================================================ chunk gradients on CTA pairs
// The gradient of GradMcOp<256, MSE> on CTA pairs: a pair computes rows
// [256 g, +256) of G_z^T (each CTA its 128, row group g of ceil(d / 256)) and
// 256 columns; each CTA holds its 128 rows of the K / V (or Y) operand and
// half of E's 256 columns, so it takes 24 KB (MSE's G2: 32 KB) per 32 tokens
// instead of the 40 KB of a one-CTA tile, and every pair MMA is 256 x 256 x 16.
// The row groups, token splits and the epilogue are GradMcOp's (with cs = 2).
template <bool MSE = false>
struct GradPairOp {
  using Base = GradMcOp<256, MSE>;
  using Params = typename Base::Params;
  using Tile = typename Base::Tile;
  using Pre = typename Base::Pre;
  static constexpr int kTok = Base::kTok;
  static constexpr uint32_t kBoxG = Base::kBoxG;  // one 64 x 32 box
  static constexpr uint32_t kAB = 2 * kBoxG;      // this CTA's 128 rows of A
  static constexpr uint32_t kEH = 2 * kBoxG;      // this CTA's 128 columns of one half of E
  static constexpr int kStageBytes = kAB + 2 * kEH + (MSE ? kAB : 0);
  static constexpr int kStages = MSE ? 6 : 8;  // 192 KB
  static constexpr int kAccCols = 256;
  static constexpr uint32_t kEpiBytes = 0;

  static __device__ int num_work(const Params& p) { return Base::num_work(p); }
  static __device__ void tile_of(const Params& p, int w, int prank, Tile& t) { Base::tile_of(p, w, prank, t); }
  static __device__ int num_kblocks(const Params& p, const Tile& t) { return t.nkb; }
  static __device__ uint32_t stage_tx(const Params& p, const Tile& t, int) {
    return kAB + (p.e_split ? 2u : 1u) * kEH + ((MSE && t.j == 1) ? kAB : 0u);
  }
  static __device__ void produce(const Params& p, const Tile& t, int kb, uint8_t* st, uint32_t fb, int prank) {
    const int tok = (t.kb0 + kb) * kTok;
    for (int g = 0; g < 2; ++g) {
      if (MSE && t.j == 1) {
        ptx::tma_load_3d_pair(st + g * kBoxG, &p.mY, fb, t.m0 + g * 64, tok, t.bh);
        ptx::tma_load_3d_pair(st + kAB + 2 * kEH + g * kBoxG, &p.mYl, fb, t.m0 + g * 64, tok, t.bh);
      } else if (p.use4d) {
        ptx::tma_load_4d_pair(st + g * kBoxG, t.j == 1 ? &p.mV4 : &p.mK4, fb, t.m0 + g * 64, tok, p.chunk_idx, t.bh);
      } else {
        ptx::tma_load_3d_pair(st + g * kBoxG, t.j == 1 ? &p.mV3 : &p.mK3, fb, t.m0 + g * 64, p.chunk_start + tok,
                              t.bh);
      }
      // this CTA's half of E: columns n0 + 128 prank + [0, 128)
      const int col = t.n0 + 128 * prank + 64 * g;
      ptx::tma_load_3d_pair(st + kAB + g * kBoxG, &p.mE, fb, col, tok, t.z);
      if (p.e_split) ptx::tma_load_3d_pair(st + kAB + kEH + g * kBoxG, &p.mEl, fb, col, tok, t.z);
    }
  }
  static __device__ void consume(const Params& p, const Tile& t, int kb, uint32_t st, uint32_t tmem) {
    constexpr uint32_t id = ptx::idesc_bf16(256, 256, true, true);
    const uint32_t eh = st + kAB, el = eh + kEH;
    const bool ylo = MSE && t.j == 1;
#pragma unroll
    for (int kk = 0; kk < kTok / 16; ++kk) {
      const uint64_t a = ptx::sdesc(st + kk * 2048, kBoxG, 1024);
      const uint64_t bh = ptx::sdesc(eh + kk * 2048, kBoxG, 1024);
      ptx::mma2_bf16(tmem, a, bh, id, (kb | kk) != 0);
      if (p.e_split) ptx::mma2_bf16(tmem, a, ptx::sdesc(el + kk * 2048, kBoxG, 1024), id, 1u);
      if (ylo) ptx::mma2_bf16(tmem, ptx::sdesc(st + kAB + 2 * kEH + kk * 2048, kBoxG, 1024), bh, id, 1u);
    }
  }
  static __device__ Pre pre(const Params& p, const Tile& t, int r) { return Base::pre(p, t, r); }
  static __device__ void epilogue(const Params& p, const Tile& t, uint32_t tm, int r, uint8_t* epi, uint32_t& es,
                                  const Pre& pr) {
    Base::epilogue(p, t, tm, r, epi, es, pr, 0);
  }
};

// ============================================================ apply-2 on CTA pairs
// O = H_q W2^T on CTA pairs: a pair computes 256 token rows (each CTA its 128)
// by a 256-wide column tile of O, each CTA holding its 128 rows of H_q and 128
// of the tile's W2 rows: 32 KB per CTA per 64 of K for 256 x 256 x 16 MMAs,
// where a one-CTA 128 x 256 tile takes 48 KB.
struct OPairOp {
  struct Params {
    CUtensorMap mH;   // Hq 3D {dh, Cp, BH}, box {64, 128, 1}
    CUtensorMap mW2;  // shadows 3D {dh, d, 3BH}, box {64, 128, 1}
    bf16* O;
    int d, dh, T, chunk_start, valid, m_pairs, n_tiles, BH;
    TcCommon cm;
  };
  struct Tile {
    int bh, row0, n0;
  };
  struct Pre {};
  static constexpr int kStages = 6;
  static constexpr int kStageBytes = 2 * kABytes;  // 128 rows of H_q + 128 rows of W2, 64 of K each
  static constexpr int kAccCols = 256;
  static constexpr uint32_t kEpiBytes = 0;

  static __device__ int num_work(const Params& p) { return p.BH * p.m_pairs * p.n_tiles; }
  static __device__ void tile_of(const Params& p, int w, int prank, Tile& t) {
    const int nt = w % p.n_tiles;
    w /= p.n_tiles;
    const int mp = w % p.m_pairs;
    t.bh = w / p.m_pairs;
    t.n0 = nt * 256;
    t.row0 = (2 * mp + prank) * BM;
  }
  static __device__ int num_kblocks(const Params& p, const Tile&) { return p.dh / BK; }
  static __device__ uint32_t stage_tx(const Params&, const Tile&, int) { return 2 * kABytes; }
  static __device__ void produce(const Params& p, const Tile& t, int kb, uint8_t* st, uint32_t fb, int prank) {
    ptx::tma_load_3d_pair(st, &p.mH, fb, kb * BK, t.row0, t.bh);
    ptx::tma_load_3d_pair(st + kABytes, &p.mW2, fb, kb * BK, t.n0 + 128 * prank, t.bh * 3 + 1);
  }
  static __device__ void consume(const Params&, const Tile&, int kb, uint32_t st, uint32_t tmem) {
    constexpr uint32_t id = ptx::idesc_bf16(256, 256, false, false);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) ptx::mma2_bf16(tmem, kdesc(st, kk), kdesc(st + kABytes, kk), id, (kb | kk) != 0);
  }
  static __device__ Pre pre(const Params&, const Tile&, int) { return {}; }
  static __device__ void epilogue(const Params& p, const Tile& t, uint32_t tm, int r, uint8_t*, uint32_t&,
                                  const Pre&) {
    const int tl = t.row0 + r;
    const bool valid = tl < p.valid;
    bf16* dst = p.O + ((size_t)t.bh * p.T + p.chunk_start + tl) * p.d + t.n0;
    float v[32];
    for (int c = 0; c < 256; c += 32) {
      ptx::tmem_ld32(tm + c, v);
      if (valid && t.n0 + c < p.d) st_bf16x32(dst + c, v);
    }
  }
};
#endif  // TTT_HAS_MULTICAST

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
// With a momentum buffer (mom != NULL) the step is B = mu*B + U, and B is
// stored back.
__global__ void update_kernel(float* M, bf16* Ms, bf16* Msl, const float* U, float* mom, float mu,
                              const float* n0, float step, int wnorm, float floor_, int d, int dh) {
  __shared__ float red[8][33];
  const int z = blockIdx.y, j = z % 3;
  const size_t base = (size_t)z * d * dh;
  float* m = M + base;
  bf16* ms = Ms + base;
  bf16* ml = Msl ? Msl + base : nullptr;
  const float* u = U + base;
  float* mb = mom ? mom + base : nullptr;
  // the step of element o: the gradient, or the advanced momentum buffer
  auto stp = [&](size_t o) { return mb ? fmaf(mu, mb[o], u[o]) : u[o]; };
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (j == 1) {
    if (blockIdx.x * 8 >= d) return;
    const int r = blockIdx.x * 8 + w;
    if (r >= d) return;  // warp-uniform
    float s = 0.f;
    for (int c = lane; c < dh; c += 32) {
      const float x = m[(size_t)r * dh + c] - step * stp((size_t)r * dh + c);
      s = fmaf(x, x, s);
    }
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float sc = wnorm ? n0[(size_t)z * dh + r] / fmaxf(sqrtf(s), floor_) : 1.f;
    for (int c = lane; c < dh; c += 32) {
      const size_t o = (size_t)r * dh + c;
      const float b = stp(o);
      const float x = (m[o] - step * b) * sc;
      m[o] = x;
      if (mb) mb[o] = b;
      st_shadow(ms, ml, o, x);
    }
  } else {
    if (blockIdx.x * 32 >= dh) return;
    const int c = blockIdx.x * 32 + lane;
    float s = 0.f;
    if (c < dh)
      for (int r = w; r < d; r += 8) {
        const float x = m[(size_t)r * dh + c] - step * stp((size_t)r * dh + c);
        s = fmaf(x, x, s);
      }
    red[w][lane] = s;
    __syncthreads();
    float t = 0.f;
    for (int k = 0; k < 8; ++k) t += red[k][lane];
    const float sc = (wnorm && c < dh) ? n0[(size_t)z * dh + c] / fmaxf(sqrtf(t), floor_) : 1.f;
    if (c < dh)
      for (int r = w; r < d; r += 8) {
        const size_t o = (size_t)r * dh + c;
        const float b = stp(o);
        const float x = (m[o] - step * b) * sc;
        m[o] = x;
        if (mb) mb[o] = b;
        st_shadow(ms, ml, o, x);
      }
  }
}

// Token-split reduction of the gradient partials in a fixed split order (the
// result does not depend on scheduling), 4 values per thread.
__global__ void gsplit_reduce_kernel(const float* parts, float* G, int splits, size_t n) {
  for (size_t e = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; e < n; e += (size_t)gridDim.x * blockDim.x * 4) {
    float4 acc = *reinterpret_cast<const float4*>(parts + e);
    for (int s = 1; s < splits; ++s) {
      const float4 v = *reinterpret_cast<const float4*>(parts + (size_t)s * n + e);
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    *reinterpret_cast<float4*>(G + e) = acc;
  }
}

// ============================================================ host side

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

// SM count the workspace plan assumes when it sizes the token-split buffers
// (B300: 148); the launches query the device itself.
constexpr int kNumSmsHint = 148;

// Clusters of `cs` CTAs of the multicast engine that fit on the device at once
// (cached per operation and cluster size).
template <class Op>
int mc_max_clusters(int cs) {
  static int cached[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
  static int cached_dev[9] = {-1, -1, -1, -1, -1, -1, -1, -1, -1};
  static std::mutex mu;  // host threads may launch at once
  std::lock_guard<std::mutex> lk(mu);
  if (cs < 1 || cs > 8) return -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cached_dev[cs] == dev) return cached[cs];
  auto kern = tc_mc_kernel<Op>;
  const size_t smem = tc_mc_smem_bytes<Op>();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return -1;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(cs);
  cfg.blockDim = dim3(tc_mc_threads<Op>());
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  cached[cs] = n;
  cached_dev[cs] = dev;
  return n;
}

// Persistent cluster launch: one cluster per work item up to the device's
// capacity, each cluster looping over items.
template <class Op>
int launch_mc(int kind, const typename Op::Params& p, int cs, int n_work, cudaStream_t st) {
  auto kern = tc_mc_kernel<Op>;
  const size_t smem = tc_mc_smem_bytes<Op>();
  const int max_cl = mc_max_clusters<Op>(cs);
  if (max_cl <= 0) return TTT_ERR_CUDA;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return TTT_ERR_CUDA;
  const int n_cl = std::max(1, std::min(n_work, max_cl));
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(n_cl * cs);
  cfg.blockDim = dim3(tc_mc_threads<Op>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  prof_before(kind, st);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  prof_after(kind, st);
  return e == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

#if TTT_HAS_MULTICAST
// CTA pairs of the pair engine that fit on the device at once (cached per operation).
template <class Op>
int pair_max(int* out) {
  static int cached = 0, cached_dev = -1;
  static std::mutex mu;  // host threads may launch at once
  std::lock_guard<std::mutex> lk(mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TTT_ERR_CUDA;
  if (cached_dev != dev) {
    auto kern = tc_pair_kernel<Op>;
    const size_t smem = tc_pair_smem_bytes<Op>();
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return TTT_ERR_CUDA;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return TTT_ERR_CUDA;
    }
    cached = n;
    cached_dev = dev;
  }
  *out = cached;
  return TTT_OK;
}

// Persistent pair launch: one pair per work item up to the device's capacity.
template <class Op>
int launch_pair(int kind, const typename Op::Params& p, int n_work, cudaStream_t st) {
  auto kern = tc_pair_kernel<Op>;
  const size_t smem = tc_pair_smem_bytes<Op>();
  int max_pairs = 0;
  const int rc = pair_max<Op>(&max_pairs);
  if (rc != TTT_OK) return rc;
  const int n_pairs = std::max(1, std::min(n_work, max_pairs));
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(2 * n_pairs);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  prof_before(kind, st);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  prof_after(kind, st);
  return e == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}
#endif  // TTT_HAS_MULTICAST

// A side stream (and two events) per device and host thread, created on first
// use, for the apply that overlaps the gradient. Returns NULL if it cannot be
// created (the caller then runs everything on its own stream).
struct SideStream {
  cudaStream_t stream;
  cudaEvent_t fwd_done, apply_done;
};

constexpr int kMaxSideDev = 64;
struct SideStreams {
  SideStream slot[kMaxSideDev];
  bool made[kMaxSideDev];
};
thread_local SideStreams t_side = {};

SideStream* side_stream() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxSideDev) return nullptr;
  if (!t_side.made[dev]) {
    SideStream& x = t_side.slot[dev];
    if (cudaStreamCreateWithFlags(&x.stream, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&x.fwd_done, cudaEventDisableTiming) != cudaSuccess) {
      cudaStreamDestroy(x.stream);
      cudaGetLastError();
      return nullptr;
    }
    if (cudaEventCreateWithFlags(&x.apply_done, cudaEventDisableTiming) != cudaSuccess) {
      cudaEventDestroy(x.fwd_done);
      cudaStreamDestroy(x.stream);
      cudaGetLastError();
      return nullptr;
    }
    t_side.made[dev] = true;
  }
  return &t_side.slot[dev];
}

// Destroys the calling thread's side streams and events (every device).
int side_streams_release() {
  int rc = TTT_OK;
  for (int dev = 0; dev < kMaxSideDev; ++dev) {
    if (!t_side.made[dev]) continue;
    SideStream& x = t_side.slot[dev];
    if (cudaStreamSynchronize(x.stream) != cudaSuccess) rc = TTT_ERR_CUDA;
    if (cudaEventDestroy(x.fwd_done) != cudaSuccess || cudaEventDestroy(x.apply_done) != cudaSuccess ||
        cudaStreamDestroy(x.stream) != cudaSuccess)
      rc = TTT_ERR_CUDA;
    t_side.made[dev] = false;
  }
  if (rc != TTT_OK) cudaGetLastError();
  return rc;
}

struct Plan {
  int BH, Z, d, dh, C, Cp, T, split;
  int bn_o;               // N tile of the apply GEMM (over d)
  int g_cs, g_mg;         // gradient: cluster size and row groups (g_cs * g_mg = ceil(d / 128) row tiles)
  int g_bn, g_nt;         //           N tile over dh, N tiles
  int g_splits_max;       // token splits the workspace has room for
  size_t off_mom;         // momentum buffers [Z][d][dh] fp32 (momentum != 0 only)
  size_t off_nsqg;        // per-row sums of squares of the gradient [Z][d][dh / g_bn] (Muon)
  size_t off_Hk[2], off_Y[2];  // MSE: key hiddens (hi, lo) [BH][Cp][dh]; Y (hi, lo) [BH][Cp][d]
  size_t off_M, off_Ms, off_Msl, off_n0, off_Hq, off_E, off_El, off_G, off_Xh[2], off_Xl[2], off_Sh,
      off_Sl, off_Ph, off_Pl, off_split, off_nsq, total;
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
  P.g_cs = TTT_HAS_MULTICAST ? (g.d + BM - 1) / BM : 1;
  P.g_mg = (g.d + BM - 1) / BM / P.g_cs;
  P.g_bn = (g.dh % 256 == 0) ? 256 : 128;
  P.g_nt = g.dh / P.g_bn;
  // token splits when the (z, n-block) items alone leave SMs idle (up to 8)
  const int kbs = (P.C + BK - 1) / BK;
  P.g_splits_max = std::max(1, std::min({8, kbs / 8, (kNumSmsHint / P.g_cs) / (P.Z * P.g_nt * P.g_mg)}));
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
  P.off_Sh = take(dd * 2);
  P.off_Sl = take(lo * dd * 2);
  P.off_Ph = take(dd * 2);
  P.off_Pl = take(lo * dd * 2);
  P.off_split = take(P.g_splits_max > 1 ? (size_t)P.g_splits_max * wz * 4 : 0);
  P.off_nsq = take(ns_fused_scratch_floats(g, P.Z) * 4);
  P.off_mom = take(g.momentum != 0.f ? wz * 4 : 0);
  P.off_nsqg = take(g.muon ? (size_t)P.Z * g.d * (g.dh / 128) * 4 : 0);
  const size_t mse = g.loss == TTT_LOSS_MSE ? 1 : 0;
  for (int i = 0; i < 2; ++i) {
    P.off_Hk[i] = take(mse * P.BH * P.Cp * g.dh * 2);
    P.off_Y[i] = take(mse * P.BH * P.Cp * g.d * 2);
  }
  P.total = off;
  return P;
}

}  // namespace

bool tc_supported(const ttt_cfg& g) {
  // d <= 1024: the gradient's clusters hold d / 128 <= 8 CTAs
  // (the fused Muon step completes the square of its quintic, so it needs c != 0,
  // and fuses the update into its last iteration, so it needs at least one)
  // (the MSE loss adds computed operands, H_k and Y, that need split precision)
  return g.dtype == TTT_DTYPE_BF16 && g.fast_net == TTT_NET_SWIGLU &&
         (g.loss == TTT_LOSS_IP || g.precision == TTT_PREC_SPLIT) && g.mode != TTT_MODE_INCLUSIVE && g.d % 64 == 0 &&
         g.dh % 128 == 0 && g.d <= g.dh && g.d <= 1024 && g.dh <= 16384 &&
         (!g.muon || (g.ns_c != 0.f && g.ns_iters >= 1));
}

size_t tc_workspace_bytes(const ttt_cfg& g) { return make_plan(g).total; }

namespace {

// One call's view of the tensor-core path: the workspace plan, the pointers
// into the workspace, the tensor maps and the launch helpers of each step of a
// chunk. ttt_fwd drives it chunk by chunk; the context-parallel entry points
// drive the same steps one at a time.
class TcLayer {
 public:
  int init(const ttt_cfg& g, char* ws, cudaStream_t st) {
    g_ = g;
    P = make_plan(g);
    st_ = st;
    ws_ = ws;
    const bool split = P.split != 0;
    mse = g.loss == TTT_LOSS_MSE;
    // which stages carry split operands (all of them unless a test hook
    // narrowed it; the MSE path keeps its forward and gradient split)
    split_fwd = split && ((g_split_mask & 1) || mse);
    split_grad = split && ((g_split_mask & 2) || mse);
    split_ns = split && (g_split_mask & 4);
    auto at = [&](size_t off, bool on) -> void* { return on ? static_cast<void*>(ws + off) : nullptr; };
    M = reinterpret_cast<float*>(ws + P.off_M);
    Ms = reinterpret_cast<bf16*>(ws + P.off_Ms);
    Msl = split ? reinterpret_cast<bf16*>(ws + P.off_Msl) : nullptr;
    n0 = reinterpret_cast<float*>(ws + P.off_n0);
    Hq = reinterpret_cast<bf16*>(ws + P.off_Hq);
    E = reinterpret_cast<bf16*>(ws + P.off_E);
    El = split ? reinterpret_cast<bf16*>(ws + P.off_El) : nullptr;
    G = reinterpret_cast<float*>(ws + P.off_G);
    splitbuf = reinterpret_cast<float*>(ws + P.off_split);
    mom = g.momentum != 0.f ? reinterpret_cast<float*>(ws + P.off_mom) : nullptr;
    cm = TcCommon{reinterpret_cast<int*>(ws), (unsigned long long)g.timeout_us * 1000ull, 0};
    const int d = g.d, dh = g.dh, BH = P.BH, Z = P.Z;
    bool ok = true;
    ok &= map3(&mW[0], Ms, dh, d, Z, 64, 64);
    ok &= map3(&mW[1], split_fwd ? Msl : Ms, dh, d, Z, 64, 64);
    ok &= map3(&mHq, Hq, dh, P.Cp, BH, 64, 128);
    ok &= map3(&mW2o, Ms, dh, d, Z, 64, P.bn_o);
    ok &= map3(&mW2p, Ms, dh, d, Z, 64, 128);
    ok &= map3(&mE[0], E, dh, P.Cp, Z, 64, 32);
    ok &= map3(&mE[1], split_grad ? El : E, dh, P.Cp, Z, 64, 32);
    ok &= map3(&sHq, Hq, dh, P.Cp, BH, 32, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_64B);
    ok &= map3(&sE[0], E, dh, P.Cp, Z, 32, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_64B);
    ok &= map3(&sE[1], split_grad ? El : E, dh, P.Cp, Z, 32, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
               CU_TENSOR_MAP_SWIZZLE_64B);
    if (mse) {
      for (int i = 0; i < 2; ++i) {
        Hk[i] = reinterpret_cast<bf16*>(ws + P.off_Hk[i]);
        Y[i] = reinterpret_cast<bf16*>(ws + P.off_Y[i]);
        ok &= map3(&mHk[i], Hk[i], dh, P.Cp, BH, 64, 128);
        ok &= map3(&sHk[i], Hk[i], dh, P.Cp, BH, 32, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_64B);
        ok &= map3(&mYf[i], Y[i], d, P.Cp, BH, 64, 128);
        ok &= map3(&mYg[i], Y[i], d, P.Cp, BH, 64, 32);
      }
      ok &= map3(&mW2y[0], Ms, dh, d, Z, 64, 128);
      ok &= map3(&mW2y[1], Msl, dh, d, Z, 64, 128);
    }
    nsa = NsFusedArgs{};
    nsa.cfg = &g_;
    nsa.Z = Z;
    nsa.split = split_ns;
    nsa.X = G;
    for (int i = 0; i < 2; ++i) {
      nsa.Xh[i] = ws + P.off_Xh[i];
      nsa.Xl[i] = at(P.off_Xl[i], split);
    }
    nsa.Rh = ws + P.off_Sh;
    nsa.Rl = at(P.off_Sl, split);
    nsa.Ph = ws + P.off_Ph;
    nsa.Pl = at(P.off_Pl, split);
    nsa.M = M;
    nsa.Ms = Ms;
    nsa.Msl = Msl;
    nsa.n0 = n0;
    nsa.scratch = reinterpret_cast<float*>(ws + P.off_nsq);
    nsa.mom = mom;
    nsa.mu = g.momentum;
    nsa.cm = cm;
    // Newton-Schulz in split precision takes its input straight from the
    // gradient kernel (operands and partial norms), with no normalise pass
    fused_ns = g.muon && split_ns;
    nsqg = reinterpret_cast<float*>(ws + P.off_nsqg);
    nsa.nsqg = nsqg;
    return ok ? TTT_OK : TTT_ERR_CUDA;
  }

  // Token tensors of the following steps: [B, H, T, d] (lr [B, H, T(, 3)]);
  // any of them may be NULL when no step reads it.
  int bind_tokens(const void* Q, const void* K, const void* V, const float* lr, void* O, int T) {
    const int d = g_.d, BH = P.BH;
    T_ = T;
    V_ = static_cast<const bf16*>(V);
    lr_ = lr;
    O_ = O;
    n_full = P.C > 0 ? T / P.C : 0;
    bool ok = true;
    if (Q) ok &= map3(&mQ, Q, d, T, BH, 64, 128);
    if (K) {
      ok &= map3(&mK, K, d, T, BH, 64, 128);
      ok &= map3(&mK3, K, d, T, BH, 64, 32);  // gradient: 32-token boxes
    }
    if (V) {
      ok &= map3(&mV, V, d, T, BH, 64, 128);
      ok &= map3(&mV3, V, d, T, BH, 64, 32);
    }
    mK4 = mK3;
    mV4 = mV3;
    if (K && V && n_full > 0) {
      // 4D view {d, C, n_full, BH}: a chunk's token range ends at the chunk boundary
      auto fn = encode_fn();
      if (!fn) return TTT_ERR_CUDA;
      CUtensorMap* outs[2] = {&mK4, &mV4};
      const void* bases[2] = {K, V};
      for (int i = 0; i < 2; ++i) {
        cuuint64_t gd[4] = {(cuuint64_t)d, (cuuint64_t)P.C, (cuuint64_t)n_full, (cuuint64_t)BH};
        cuuint64_t gs[3] = {(cuuint64_t)d * 2, (cuuint64_t)P.C * d * 2, (cuuint64_t)T * d * 2};
        cuuint32_t bx[4] = {64, 32, 1, 1};
        cuuint32_t es[4] = {1, 1, 1, 1};
        ok &= fn(outs[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(bases[i]), gd, gs, bx, es,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
      }
    }
    return ok ? TTT_OK : TTT_ERR_CUDA;
  }

  // W0 -> master weights, bf16 shadows and reference row norms; momentum buffers start at zero.
  int import_w0(const float* const W0[3]) {
    const int d = g_.d, dh = g_.dh, Z = P.Z;
    cudaStream_t st = st_;
    if (mom && cudaMemsetAsync(mom, 0, (size_t)Z * d * dh * sizeof(float), st) != cudaSuccess) return TTT_ERR_CUDA;
    const dim3 grid((dh + 31) / 32, (d + 31) / 32, Z);
    TTT_LAUNCH(TTT_KERNEL_AUX, st,
               import_kernel<<<grid, 256, 0, st>>>(W0[0], W0[1], W0[2], M, Ms, Msl, g_.H, d, dh, g_.w0_per_batch));
    const dim3 gn(std::max((dh + 31) / 32, (d + 7) / 8), Z);
    TTT_LAUNCH(TTT_KERNEL_AUX, st, norms_kernel<<<gn, 256, 0, st>>>(M, n0, d, dh));
    return TTT_OK;
  }

  int export_w(float* const Wf[3]) {
    const int d = g_.d, dh = g_.dh;
    cudaStream_t st = st_;
    const dim3 grid((dh + 31) / 32, (d + 31) / 32, P.Z);
    TTT_LAUNCH(TTT_KERNEL_AUX, st, export_kernel<<<grid, 256, 0, st>>>(M, Wf[0], Wf[1], Wf[2], d, dh));
    return TTT_OK;
  }

  // Forward of tokens [s, s + valid): query tiles (H_q) and/or key tiles (E).
  // With the MSE loss the key tiles need Y = f(k) - v first: one launch for
  // the queries and the key hiddens H_k, one for Y = H_k W2^T - V, then the key
  // tiles with Dm = Y W2.
  int fwd(int s, int valid, bool q, bool k) {
    if (k && mse) {
      int rc = fwd_launch(s, valid, q, false, true);
      if (rc == TTT_OK) rc = y_launch(s, valid);
      if (rc == TTT_OK) rc = fwd_launch(s, valid, false, true, false);
      return rc;
    }
    return fwd_launch(s, valid, q, k, false);
  }

  int y_launch(int s, int valid) {
    YOp::Params p{};
    p.mH = mHk[0]; p.mHl = mHk[1]; p.mW2 = mW2y[0]; p.mW2l = mW2y[1];
    p.V = V_; p.Y = Y[0]; p.Yl = Y[1];
    p.d = g_.d; p.dh = g_.dh; p.T = T_; p.Cp = P.Cp; p.chunk_start = s; p.valid = valid;
    p.m_tiles = (valid + BM - 1) / BM;
    p.n_tiles = (g_.d + YOp::BN - 1) / YOp::BN;
    p.cm = cm;
    return launch_op<YOp>(TTT_KERNEL_FWD, p, dim3(p.m_tiles * p.n_tiles, P.BH), st_);
  }

  int fwd_launch(int s, int valid, bool q, bool k, bool h) {
    FwdMcParams p{};
    p.mQ = mQ; p.mK = mK; p.mV = mV; p.mW = mW[0]; p.mWl = mW[1];
    p.sHq = sHq; p.sE = sE[0]; p.sEl = sE[1];
    p.lr = lr_; p.Hq = Hq; p.E = E; p.El = El;
    p.lr_stride = g_.lr_per_matrix ? 3 : 1;
    p.d = g_.d; p.dh = g_.dh; p.T = T_; p.Cp = P.Cp; p.chunk_start = s; p.valid = valid;
    p.n_tok = (valid + BM - 1) / BM;
    // pairs of consecutive token tiles share each weight slice by multicast:
    // clusters of two fill all 148 SMs (clusters of four leave 16 idle); the
    // build without multicast runs clusters of one
    p.cs = (TTT_HAS_MULTICAST && p.n_tok >= 2) ? 2 : 1;
    p.groups = (p.n_tok + p.cs - 1) / p.cs;
    p.n_jq = g_.dh / 128;
    p.BH = P.BH;
    p.q = q ? 1 : 0;
    p.k = k ? 1 : 0;
    p.h = h ? 1 : 0;
    p.mse = mse ? 1 : 0;
    if (mse) {
      p.mY = mYf[0]; p.mYl = mYf[1]; p.sHk = sHk[0]; p.sHkl = sHk[1];
    }
    p.w_split = split_fwd ? 1 : 0;
    p.e_split = split_grad ? 1 : 0;
    p.cm = cm;
    p.cm.stall = g_stall_next_fwd.exchange(0);
    const int n_work = P.BH * p.n_jq * p.groups * (p.q + 2 * p.h + 2 * p.k);
    if (g_.d < 512) return launch_mc<FwdMcOpT<8>>(TTT_KERNEL_FWD, p, p.cs, n_work, st_);
    return launch_mc<FwdMcOpT<4>>(TTT_KERNEL_FWD, p, p.cs, n_work, st_);
  }

  // O[s, s + valid) = H_q W2^T on stream `os`.
  int apply(int s, int valid, cudaStream_t os) {
    const int d = g_.d;
    const int mt = (valid + BM - 1) / BM, nt = (d + P.bn_o - 1) / P.bn_o;
    auto fill = [&](auto& p) {
      p.mH = mHq; p.mW2 = mW2o; p.O = static_cast<bf16*>(O_);
      p.d = d; p.dh = g_.dh; p.T = T_; p.chunk_start = s; p.valid = valid; p.m_tiles = mt; p.n_tiles = nt;
      p.cm = cm;
    };
#if TTT_HAS_MULTICAST
    if (mt >= 2) {
      OPairOp::Params p{};
      p.mH = mHq; p.mW2 = mW2p; p.O = static_cast<bf16*>(O_);
      p.d = d; p.dh = g_.dh; p.T = T_; p.chunk_start = s; p.valid = valid;
      p.m_pairs = (mt + 1) / 2; p.n_tiles = (d + 255) / 256; p.BH = P.BH;
      p.cm = cm;
      return launch_pair<OPairOp>(TTT_KERNEL_APPLY, p, P.BH * p.m_pairs * p.n_tiles, os);
    }
#endif
    const dim3 grid(mt * nt, P.BH);
    if (P.bn_o == 256) { typename OOp<256>::Params p{}; fill(p); return launch_op<OOp<256>>(TTT_KERNEL_APPLY, p, grid, os); }
    if (P.bn_o == 192) { typename OOp<192>::Params p{}; fill(p); return launch_op<OOp<192>>(TTT_KERNEL_APPLY, p, grid, os); }
    typename OOp<128>::Params p{}; fill(p); return launch_op<OOp<128>>(TTT_KERNEL_APPLY, p, grid, os);
  }

  // Chunk gradient of tokens [s, s + valid) (chunk ci) from E into `out`
  // ([Z][d][dh] fp32), or, when out is NULL: into the workspace's G, or (fused
  // Newton-Schulz) straight into the Muon step's input operands.
  int grad(int ci, int s, int valid, float* out = nullptr) {
    const int d = g_.d, dh = g_.dh, Z = P.Z;
    float* dst = out ? out : G;
    const bool to_ns = !out && fused_ns;
    const bool full = n_full > 0 && (s + P.C <= T_) && ci < n_full && s == ci * P.C;
    const int kbs = (valid + 31) / 32;  // 32-token k-blocks
    const int items = Z * P.g_nt * P.g_mg;
    auto launch = [&](auto op) -> int {
      using Op = decltype(op);
      const int max_cl = mc_max_clusters<Op>(P.g_cs);
      if (max_cl <= 0) return TTT_ERR_CUDA;
      int splits = std::max(1, std::min({P.g_splits_max, kbs / 16, max_cl / items}));
      const int kb_per_split = (kbs + splits - 1) / splits;
      splits = (kbs + kb_per_split - 1) / kb_per_split;
      typename Op::Params p{};
      p.mK4 = mK4; p.mV4 = mV4; p.mK3 = mK3; p.mV3 = mV3; p.mE = mE[0]; p.mEl = mE[1];
      p.G = dst; p.split_out = splitbuf;
      p.d = d; p.dh = dh; p.Z = Z; p.chunk_idx = ci; p.chunk_start = s; p.valid = valid; p.use4d = full ? 1 : 0;
      p.nt = P.g_nt; p.splits = splits; p.kb_per_split = kb_per_split; p.e_split = split_grad ? 1 : 0; p.cm = cm;
      p.mg = P.g_mg; p.cs = P.g_cs;
      if (mse) {
        p.mY = mYg[0];
        p.mYl = mYg[1];
      }
      if (to_ns) {
        p.Xh = static_cast<bf16*>(nsa.Xh[0]);
        p.Xl = static_cast<bf16*>(nsa.Xl[0]);
        p.mom = mom;
        p.mu = g_.momentum;
        p.nsq = nsqg;
      }
      const int r = launch_mc<Op>(TTT_KERNEL_GRAD, p, P.g_cs, items * splits, st_);
      if (r != TTT_OK || splits == 1) return r;
      const size_t n = (size_t)Z * d * dh;
      cudaStream_t st = st_;
      if (to_ns)
        return ns_input_launch(splitbuf, splits, Z, d, dh, P.g_bn, mom, g_.momentum, nsa.Xh[0], nsa.Xl[0], nsqg, st);
      TTT_LAUNCH(TTT_KERNEL_GRAD, st, gsplit_reduce_kernel<<<4 * kNumSmsHint, 256, 0, st>>>(splitbuf, dst, splits, n));
      return TTT_OK;
    };
#if TTT_HAS_MULTICAST
    // CTA pairs when the columns come in 256-wide tiles and the rows in pairs
    // of 128 (a pair half past d would idle; d = 640 runs faster on clusters)
    if (g_grad_pairs && P.g_bn == 256 && d % (2 * BM) == 0) {
      auto launch2 = [&](auto op) -> int {
        using Op = decltype(op);
        int max_pairs = 0;
        const int rc = pair_max<Op>(&max_pairs);
        if (rc != TTT_OK) return rc;
        const int mg2 = (d + 2 * BM - 1) / (2 * BM);
        const int items2 = Z * P.g_nt * mg2;
        int splits = std::max(1, std::min({P.g_splits_max, kbs / 16, max_pairs / items2}));
        const int kb_per_split = (kbs + splits - 1) / splits;
        splits = (kbs + kb_per_split - 1) / kb_per_split;
        typename Op::Params p{};
        p.mK4 = mK4; p.mV4 = mV4; p.mK3 = mK3; p.mV3 = mV3; p.mE = mE[0]; p.mEl = mE[1];
        p.G = dst; p.split_out = splitbuf;
        p.d = d; p.dh = dh; p.Z = Z; p.chunk_idx = ci; p.chunk_start = s; p.valid = valid; p.use4d = full ? 1 : 0;
        p.nt = P.g_nt; p.splits = splits; p.kb_per_split = kb_per_split; p.e_split = split_grad ? 1 : 0; p.cm = cm;
        p.mg = mg2; p.cs = 2;
        if (mse) {
          p.mY = mYg[0];
          p.mYl = mYg[1];
        }
        if (to_ns) {
          p.Xh = static_cast<bf16*>(nsa.Xh[0]);
          p.Xl = static_cast<bf16*>(nsa.Xl[0]);
          p.mom = mom;
          p.mu = g_.momentum;
          p.nsq = nsqg;
        }
        const int r = launch_pair<Op>(TTT_KERNEL_GRAD, p, items2 * splits, st_);
        if (r != TTT_OK || splits == 1) return r;
        const size_t n = (size_t)Z * d * dh;
        cudaStream_t st = st_;
        if (to_ns)
          return ns_input_launch(splitbuf, splits, Z, d, dh, P.g_bn, mom, g_.momentum, nsa.Xh[0], nsa.Xl[0], nsqg, st);
        TTT_LAUNCH(TTT_KERNEL_GRAD, st, gsplit_reduce_kernel<<<4 * kNumSmsHint, 256, 0, st>>>(splitbuf, dst, splits, n));
        return TTT_OK;
      };
      return mse ? launch2(GradPairOp<true>{}) : launch2(GradPairOp<false>{});
    }
#endif
    if (mse) return P.g_bn == 256 ? launch(GradMcOp<256, true>{}) : launch(GradMcOp<128, true>{});
    return P.g_bn == 256 ? launch(GradMcOp<256>{}) : launch(GradMcOp<128>{});
  }

  // The update from the gradient `u` ([Z][d][dh] fp32; the workspace's G when
  // NULL): Muon + update + weight norm in one launch, or without Muon the
  // plain update + weight norm.
  int step(const float* u = nullptr) {
    const int d = g_.d, dh = g_.dh;
    const float* src = u ? u : G;
    if (g_.muon) {
      NsFusedArgs a = nsa;
      a.X = const_cast<float*>(src);
      if (!u && fused_ns) {
        // the gradient kernel wrote the operands and advanced the momentum
        a.fused = true;
        a.nsqg = nsqg;
        a.nsq_n = g_.d * P.g_nt;
        a.mom = nullptr;
      }
      return ns_fused_run(a, st_);
    }
    cudaStream_t st = st_;
    const dim3 grid(std::max((dh + 31) / 32, (d + 7) / 8), P.Z);
    TTT_LAUNCH(TTT_KERNEL_UPDATE, st,
               update_kernel<<<grid, 256, 0, st>>>(M, Ms, Msl, src, mom, g_.momentum, n0, g_.step, g_.wnorm,
                                                   g_.wnorm_eps, d, dh));
    return TTT_OK;
  }

  Plan P;

 private:
  ttt_cfg g_;
  cudaStream_t st_;
  char* ws_;
  bool split_fwd, split_grad, split_ns, fused_ns, mse = false;
  bf16* Hk[2] = {nullptr, nullptr};
  bf16* Y[2] = {nullptr, nullptr};
  CUtensorMap mHk[2], sHk[2], mYf[2], mYg[2], mW2y[2];
  const bf16* V_ = nullptr;
  float *M, *n0, *G, *splitbuf, *mom, *nsqg;
  bf16 *Ms, *Msl, *Hq, *E, *El;
  TcCommon cm;
  NsFusedArgs nsa;
  CUtensorMap mW[2], mHq, mW2o, mW2p, mE[2], sHq, sE[2];
  CUtensorMap mQ, mK, mV, mK3, mV3, mK4, mV4;
  const float* lr_ = nullptr;
  void* O_ = nullptr;
  int T_ = 0, n_full = 0;
};

}  // namespace

int tc_run(const Call& c) {
  const ttt_cfg& g = c.cfg;
  TcLayer L;
  int rc = L.init(g, c.ws, c.stream);
  if (rc == TTT_OK) rc = L.bind_tokens(c.Q, c.K, c.V, c.lr, c.O, g.T);
  if (rc == TTT_OK) rc = L.import_w0(c.W0);
  if (rc != TTT_OK) return rc;
  const cudaStream_t st = c.stream;
  const int T = g.T;

  // In shifted mode the apply of a chunk (O = H_q W2^T) and its gradient are
  // independent: the apply runs on a side stream between the forward and the
  // Muon step (which rewrites the weights the apply reads).
  SideStream* side = side_stream();
  for (int ci = 0; ci < c.n_chunks; ++ci) {
    const int s = ci * g.chunk;
    const int valid = std::min(g.chunk, T - s);
    const bool upd = call_updates(c, ci);
    if (c.chunk_ready && cudaStreamWaitEvent(st, c.chunk_ready[ci], 0) != cudaSuccess) return TTT_ERR_CUDA;
    if (g.mode == TTT_MODE_SHIFTED) {
      rc = L.fwd(s, valid, true, upd);
      if (rc == TTT_OK && upd && side) {
        cudaStream_t os = side->stream;
        if (cudaEventRecord(side->fwd_done, st) != cudaSuccess || cudaStreamWaitEvent(os, side->fwd_done, 0) != cudaSuccess)
          return TTT_ERR_CUDA;
        rc = L.apply(s, valid, os);
        if (rc == TTT_OK && c.chunk_done && cudaEventRecord(c.chunk_done[ci], os) != cudaSuccess) rc = TTT_ERR_CUDA;
        if (rc == TTT_OK && cudaEventRecord(side->apply_done, os) != cudaSuccess) rc = TTT_ERR_CUDA;
        if (rc == TTT_OK) rc = L.grad(ci, s, valid);
        if (rc == TTT_OK && cudaStreamWaitEvent(st, side->apply_done, 0) != cudaSuccess) rc = TTT_ERR_CUDA;
        if (rc == TTT_OK) rc = L.step();
      } else {
        if (rc == TTT_OK) rc = L.apply(s, valid, st);
        if (rc == TTT_OK && c.chunk_done && cudaEventRecord(c.chunk_done[ci], st) != cudaSuccess) rc = TTT_ERR_CUDA;
        if (rc == TTT_OK && upd) rc = L.grad(ci, s, valid);
        if (rc == TTT_OK && upd) rc = L.step();
      }
    } else {
      rc = TTT_OK;
      if (upd) {
        rc = L.fwd(s, valid, false, true);
        if (rc == TTT_OK) rc = L.grad(ci, s, valid);
        if (rc == TTT_OK) rc = L.step();
      }
      if (rc == TTT_OK) rc = L.fwd(s, valid, true, false);
      if (rc == TTT_OK) rc = L.apply(s, valid, st);
      if (rc == TTT_OK && c.chunk_done && cudaEventRecord(c.chunk_done[ci], st) != cudaSuccess) rc = TTT_ERR_CUDA;
    }
    if (rc != TTT_OK) return rc;
  }
  return L.export_w(c.Wf);
}

// ============================================================ context parallelism
namespace {

bool cp_aligned(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks shared by the context-parallel calls; on success `L` is ready on the workspace.
int cp_open(const ttt_cfg* cfg, void* ws, size_t ws_bytes, void* stream, TcLayer& L) {
  int v = validate_cfg(cfg);
  if (v != TTT_OK) return v;
  if (cfg->impl != TTT_IMPL_AUTO && cfg->impl != TTT_IMPL_TC) return TTT_ERR_UNSUPPORTED;
  if (!tc_supported(*cfg)) return TTT_ERR_UNSUPPORTED;
  if (cfg->T < cfg->chunk) return TTT_ERR_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < tc_workspace_bytes(*cfg)) return TTT_ERR_WORKSPACE;
  const void* p[1] = {ws};
  v = check_device_ptrs(p, 1);
  if (v != TTT_OK) return v;
  ttt_cfg g = *cfg;
  if (g.timeout_us == 0) g.timeout_us = 2000000u;
  return L.init(g, static_cast<char*>(ws), static_cast<cudaStream_t>(stream));
}

int cp_range_ok(const ttt_cfg* cfg, int T_all, int start, int n) {
  return (start >= 0 && n >= 1 && n <= cfg->chunk && T_all >= 1 && (int64_t)start + n <= T_all) ? TTT_OK : TTT_ERR_ARG;
}

}  // namespace
}  // namespace ttt

using namespace ttt;

extern "C" int ttt_cp_workspace_bytes(const ttt_cfg* cfg, size_t* bytes) {
  if (!bytes || validate_cfg(cfg) != TTT_OK) return TTT_ERR_ARG;
  if ((cfg->impl != TTT_IMPL_AUTO && cfg->impl != TTT_IMPL_TC) || !tc_supported(*cfg)) return TTT_ERR_UNSUPPORTED;
  if (cfg->T < cfg->chunk) return TTT_ERR_ARG;
  *bytes = tc_workspace_bytes(*cfg);
  return TTT_OK;
}

extern "C" int ttt_cp_begin(const ttt_cfg* cfg, const float* W0_1, const float* W0_2, const float* W0_3,
                            void* workspace, size_t workspace_bytes, void* stream) {
  TcLayer L;
  if (!cp_aligned(W0_1) || !cp_aligned(W0_2) || !cp_aligned(W0_3)) return TTT_ERR_ARG;
  int rc = cp_open(cfg, workspace, workspace_bytes, stream, L);
  if (rc != TTT_OK) return rc;
  const void* p[3] = {W0_1, W0_2, W0_3};
  rc = check_device_ptrs(p, 3);
  if (rc != TTT_OK) return rc;
  if (cudaMemsetAsync(workspace, 0, sizeof(int), static_cast<cudaStream_t>(stream)) != cudaSuccess) return TTT_ERR_CUDA;
  const float* w0[3] = {W0_1, W0_2, W0_3};
  return L.import_w0(w0);
}

extern "C" int ttt_cp_grad(const ttt_cfg* cfg, const void* K, const void* V, const float* lr, int T_all, int start,
                           int n, float* G, void* workspace, size_t workspace_bytes, void* stream) {
  TcLayer L;
  if (!cp_aligned(K) || !cp_aligned(V) || !cp_aligned(lr) || !cp_aligned(G)) return TTT_ERR_ARG;
  int rc = cp_open(cfg, workspace, workspace_bytes, stream, L);
  if (rc != TTT_OK) return rc;
  if ((rc = cp_range_ok(cfg, T_all, start, n)) != TTT_OK) return rc;
  const void* p[4] = {K, V, lr, G};
  if ((rc = check_device_ptrs(p, 4)) != TTT_OK) return rc;
  if ((rc = L.bind_tokens(nullptr, K, V, lr, nullptr, T_all)) != TTT_OK) return rc;
  if ((rc = L.fwd(start, n, false, true)) != TTT_OK) return rc;
  return L.grad(start == 0 ? 0 : -1, start, n, G);
}

extern "C" int ttt_cp_update(const ttt_cfg* cfg, const float* G, void* workspace, size_t workspace_bytes,
                             void* stream) {
  TcLayer L;
  if (!cp_aligned(G)) return TTT_ERR_ARG;
  int rc = cp_open(cfg, workspace, workspace_bytes, stream, L);
  if (rc != TTT_OK) return rc;
  const void* p[1] = {G};
  if ((rc = check_device_ptrs(p, 1)) != TTT_OK) return rc;
  return L.step(G);
}

extern "C" int ttt_cp_apply(const ttt_cfg* cfg, const void* Q, int T_all, int start, int n, void* O,
                            void* workspace, size_t workspace_bytes, void* stream) {
  TcLayer L;
  if (!cp_aligned(Q) || !cp_aligned(O)) return TTT_ERR_ARG;
  int rc = cp_open(cfg, workspace, workspace_bytes, stream, L);
  if (rc != TTT_OK) return rc;
  if ((rc = cp_range_ok(cfg, T_all, start, n)) != TTT_OK) return rc;
  const void* p[2] = {Q, O};
  if ((rc = check_device_ptrs(p, 2)) != TTT_OK) return rc;
  if ((rc = L.bind_tokens(Q, nullptr, nullptr, nullptr, O, T_all)) != TTT_OK) return rc;
  if ((rc = L.fwd(start, n, true, false)) != TTT_OK) return rc;
  return L.apply(start, n, static_cast<cudaStream_t>(stream));
}

extern "C" int ttt_cp_end(const ttt_cfg* cfg, float* Wf_1, float* Wf_2, float* Wf_3, void* workspace,
                          size_t workspace_bytes, void* stream) {
  TcLayer L;
  if (!cp_aligned(Wf_1) || !cp_aligned(Wf_2) || !cp_aligned(Wf_3)) return TTT_ERR_ARG;
  int rc = cp_open(cfg, workspace, workspace_bytes, stream, L);
  if (rc != TTT_OK) return rc;
  const void* p[3] = {Wf_1, Wf_2, Wf_3};
  if ((rc = check_device_ptrs(p, 3)) != TTT_OK) return rc;
  float* wf[3] = {Wf_1, Wf_2, Wf_3};
  return L.export_w(wf);
}

// ============================================================ test hooks
extern "C" int ttt_dbg_ns_plan(const ttt_cfg* cfg, int* grid, int* resident) {
  using namespace ttt;
  if (!cfg || !grid || ttt_select_impl(cfg) != TTT_IMPL_TC || !ns_fused_supported(*cfg)) return TTT_ERR_ARG;
  const int G = ns_fused_plan(*cfg, resident);
  if (G <= 0) return TTT_ERR_CUDA;
  *grid = G;
  return TTT_OK;
}

extern "C" int ttt_dbg_split_mask(int mask) {
  if (mask < 0 || mask > 7) return TTT_ERR_ARG;
  ttt::g_split_mask = mask;
  return TTT_OK;
}

extern "C" int ttt_dbg_ns_force_grid(int ctas) {
  if (ctas < 0) return TTT_ERR_ARG;
  ttt::ns_force_grid(ctas);
  return TTT_OK;
}

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

extern "C" int ttt_build_features(void) { return TTT_HAS_MULTICAST ? TTT_FEATURE_CLUSTER_MULTICAST : 0; }

extern "C" void ttt_dbg_stall_next_fwd(void) { ttt::g_stall_next_fwd.store(1); }

extern "C" int ttt_thread_release(void) { return ttt::side_streams_release(); }

extern "C" int ttt_dbg_grad_pairs(int on) {
  if (on != 0 && on != 1) return TTT_ERR_ARG;
  ttt::g_grad_pairs = on != 0;
  return TTT_OK;
}

