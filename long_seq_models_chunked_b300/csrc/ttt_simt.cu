// SIMT fp32 path of the chunked TTT layer: every step in fp32 FMA.
//
// One CTA owns one (batch, head) and walks its chunks in order (LaCT page §2.1
// update/apply phases; §3.2 shifted block-causal order; §3.1 single-chunk
// update-then-apply). The fast weights, the chunk gradient and the token-block
// intermediates live in a per-head slice of the workspace. Reductions run in a
// fixed order, so two runs give bitwise identical results.
//
// This path covers every configuration (SwiGLU or linear net, inner-product or
// MSE loss, Muon or plain SGD, any d/dh/chunk, fp32 or bf16 storage) and is the
// fp32 tier (no TF32 or bf16 tensor-core rounding).
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kThreads = 256;
constexpr int kTokenBlock = 64;

struct SimtLayout {
  size_t W[3], G[3], N0[3], Mom[3];
  size_t A, Bm, Hh, Y;
  size_t Hq, KQ;  // inclusive order: the block's query hiddens, and q.k / h_q.h_k products
  size_t X, S, P, Xn;
  size_t total;
};

__host__ __device__ inline SimtLayout simt_layout(int fast_net, int d, int dh, int tb, bool mom) {
  SimtLayout L{};
  size_t off = 0;
  const int nw = fast_net == TTT_NET_SWIGLU ? 3 : 1;
  size_t sz[3], rows[3];
  if (nw == 3) {
    sz[0] = sz[1] = sz[2] = (size_t)d * dh;
    rows[0] = dh; rows[1] = d; rows[2] = dh;
  } else {
    sz[0] = (size_t)d * d; rows[0] = d;
  }
  for (int j = 0; j < nw; ++j) { L.W[j] = off; off += align_up(sz[j], 64); }
  for (int j = 0; j < nw; ++j) { L.G[j] = off; off += align_up(sz[j], 64); }
  for (int j = 0; j < nw; ++j) { L.N0[j] = off; off += align_up(rows[j], 64); }
  for (int j = 0; j < nw; ++j) { L.Mom[j] = off; off += mom ? align_up(sz[j], 64) : 0; }
  const int hid = nw == 3 ? dh : d;
  L.A = off;  off += align_up((size_t)tb * hid, 64);
  L.Bm = off; off += align_up((size_t)tb * hid, 64);
  L.Hh = off; off += align_up((size_t)tb * hid, 64);
  L.Y = off;  off += align_up((size_t)tb * d, 64);
  L.Hq = off; off += align_up((size_t)tb * hid, 64);
  L.KQ = off; off += align_up((size_t)tb * tb, 64);
  const size_t m = nw == 3 ? (d < dh ? d : dh) : d;
  const size_t n = nw == 3 ? (d < dh ? dh : d) : d;
  L.X = off;  off += align_up(m * n, 64);
  L.S = off;  off += align_up(m * m, 64);
  L.P = off;  off += align_up(m * m, 64);
  L.Xn = off; off += align_up(m * n, 64);
  L.total = off;
  return L;
}

struct SimtArgs {
  int B, H, T, d, dh, chunk, fast_net, loss, mode, dtype, muon, ns_iters, wnorm;
  int w0_per_batch, has_mask, tb;
  int lr_stride;   // 1: one rate per token; n_w: one per token and matrix
  float ns_a, ns_b, ns_c, ns_eps, wnorm_eps, step;
  float momentum;  // 0: no momentum buffer
  const void* Q;
  const void* K;
  const void* V;
  const float* lr;
  const float* W0[3];
  void* O;
  float* Wf[3];
  float* scratch;
  size_t head_floats;
  int* status;
  MaskBits mask;
};

// Deterministic block-wide sum: strided per-thread partials, then a fixed tree.
__device__ float block_sum(float v, float* red) {
  red[threadIdx.x] = v;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  float r = red[0];
  __syncthreads();
  return r;
}

// Warp-reduced row norms of a rows x cols matrix (lane-strided, butterfly).
__device__ void row_norms(const float* W, int rows, int cols, float* out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  for (int r = warp; r < rows; r += nwarp) {
    float s = 0.f;
    for (int c = lane; c < cols; c += 32) s = fmaf(W[(size_t)r * cols + c], W[(size_t)r * cols + c], s);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) out[r] = sqrtf(s);
  }
}

__device__ void renorm_rows(float* W, int rows, int cols, const float* n0, float floor_) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  for (int r = warp; r < rows; r += nwarp) {
    float s = 0.f;
    for (int c = lane; c < cols; c += 32) s = fmaf(W[(size_t)r * cols + c], W[(size_t)r * cols + c], s);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float scale = n0[r] / fmaxf(sqrtf(s), floor_);
    for (int c = lane; c < cols; c += 32) W[(size_t)r * cols + c] *= scale;
  }
}

// Muon: G (rows x cols) <- NS5(G), iterating on the wide orientation.
__device__ void newton_schulz(const SimtArgs& a, float* G, int rows, int cols, float* ws,
                              const SimtLayout& L, float* red) {
  const bool tall = rows > cols;
  const int m = tall ? cols : rows, n = tall ? rows : cols;
  float* X = ws + L.X;
  float* S = ws + L.S;
  float* P = ws + L.P;
  float* Xn = ws + L.Xn;
  float part = 0.f;
  for (int idx = threadIdx.x; idx < m * n; idx += blockDim.x) {
    const int r = idx / n, c = idx % n;
    const float g = tall ? G[(size_t)c * cols + r] : G[(size_t)r * cols + c];
    X[idx] = g;
    part = fmaf(g, g, part);
  }
  const float fro = block_sum(part, red);
  const float inv = 1.0f / (sqrtf(fro) + a.ns_eps);
  for (int idx = threadIdx.x; idx < m * n; idx += blockDim.x) X[idx] *= inv;
  __syncthreads();
  for (int it = 0; it < a.ns_iters; ++it) {
    for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) {
      const int r1 = idx / m, r2 = idx % m;
      float acc = 0.f;
      for (int c = 0; c < n; ++c) acc = fmaf(X[(size_t)r1 * n + c], X[(size_t)r2 * n + c], acc);
      S[idx] = acc;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) {
      const int r1 = idx / m, r2 = idx % m;
      float acc = 0.f;
      for (int k = 0; k < m; ++k) acc = fmaf(S[(size_t)r1 * m + k], S[(size_t)k * m + r2], acc);
      P[idx] = a.ns_b * S[idx] + a.ns_c * acc;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < m * n; idx += blockDim.x) {
      const int r = idx / n, c = idx % n;
      float acc = 0.f;
      for (int k = 0; k < m; ++k) acc = fmaf(P[(size_t)r * m + k], X[(size_t)k * n + c], acc);
      Xn[idx] = a.ns_a * X[idx] + acc;
    }
    __syncthreads();
    float* t = X; X = Xn; Xn = t;
  }
  for (int idx = threadIdx.x; idx < m * n; idx += blockDim.x) {
    const int r = idx / n, c = idx % n;
    if (tall) G[(size_t)c * cols + r] = X[idx];
    else G[(size_t)r * cols + c] = X[idx];
  }
  __syncthreads();
}

__device__ void apply_chunk(const SimtArgs& a, float* ws, const SimtLayout& L, size_t head,
                            int s, int e) {
  const int d = a.d, dh = a.dh;
  for (int t0 = s; t0 < e; t0 += a.tb) {
    const int nt = min(a.tb, e - t0);
    const size_t base = (head * a.T + t0) * (size_t)d;
    if (a.fast_net == TTT_NET_SWIGLU) {
      const float* W1 = ws + L.W[0];
      const float* W2 = ws + L.W[1];
      const float* W3 = ws + L.W[2];
      float* Hh = ws + L.Hh;
      for (int idx = threadIdx.x; idx < nt * dh; idx += blockDim.x) {
        const int t = idx / dh, j = idx % dh;
        float xa = 0.f, xb = 0.f;
        for (int i = 0; i < d; ++i) {
          const float q = ld_val(a.Q, base + (size_t)t * d + i, a.dtype);
          xa = fmaf(W1[(size_t)j * d + i], q, xa);
          xb = fmaf(W3[(size_t)j * d + i], q, xb);
        }
        Hh[idx] = xa * sigmoidf_(xa) * xb;
      }
      __syncthreads();
      for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
        const int t = idx / d, i = idx % d;
        float acc = 0.f;
        for (int j = 0; j < dh; ++j) acc = fmaf(W2[(size_t)i * dh + j], Hh[(size_t)t * dh + j], acc);
        st_val(a.O, base + idx, a.dtype, acc);
      }
      __syncthreads();
    } else {
      const float* W = ws + L.W[0];
      for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
        const int t = idx / d, i = idx % d;
        float acc = 0.f;
        for (int k = 0; k < d; ++k)
          acc = fmaf(W[(size_t)i * d + k], ld_val(a.Q, base + (size_t)t * d + k, a.dtype), acc);
        st_val(a.O, base + idx, a.dtype, acc);
      }
      __syncthreads();
    }
  }
}

// Inclusive order (tutorial page §3: update with a token, then output with the
// updated weights), one token block [t0, t0 + nt) of a chunk: query t sees
// W - step (G + sum_{s <= t in the block} G_s), G the gradient summed over the
// chunk's earlier blocks and G_s token s's gradient, all at the chunk's
// starting weights W. Each layer is linear in its weights and every G_s is an
// outer product, so the block's part is a causal dual form:
//   A_q = q (W1 - step G1)^T - step sum_{s<=t} (q.k_s) DA_s   (B_q likewise with DB)
//   o   = (W2 - step G2) h_q - step sum_{s<=t} (h_q.h_s) lr2_s y_s
// On entry A, Bm hold the block's DA, DB (rates applied), Hh its key hiddens,
// Y its dl/df without rates; G holds the earlier blocks' sums.
template <class Eta>
__device__ void inclusive_block_swiglu(const SimtArgs& a, float* ws, const SimtLayout& L, size_t head, int t0,
                                       int nt, Eta eta) {
  const int d = a.d, dh = a.dh;
  const size_t base = (head * a.T + t0) * (size_t)d;
  const float* W1 = ws + L.W[0];
  const float* W2 = ws + L.W[1];
  const float* W3 = ws + L.W[2];
  const float* G1 = ws + L.G[0];
  const float* G2 = ws + L.G[1];
  const float* G3 = ws + L.G[2];
  const float* DA = ws + L.A;
  const float* DB = ws + L.Bm;
  const float* Hk = ws + L.Hh;
  const float* Y = ws + L.Y;
  float* Hq = ws + L.Hq;
  float* KQ = ws + L.KQ;
  const float st = a.step;
  for (int idx = threadIdx.x; idx < nt * nt; idx += blockDim.x) {
    const int t = idx / nt, u = idx % nt;
    float acc = 0.f;
    if (u <= t)
      for (int i = 0; i < d; ++i)
        acc = fmaf(ld_val(a.Q, base + (size_t)t * d + i, a.dtype), ld_val(a.K, base + (size_t)u * d + i, a.dtype), acc);
    KQ[idx] = acc;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nt * dh; idx += blockDim.x) {
    const int t = idx / dh, j = idx % dh;
    float xa = 0.f, xb = 0.f;
    for (int i = 0; i < d; ++i) {
      const float q = ld_val(a.Q, base + (size_t)t * d + i, a.dtype);
      xa = fmaf(W1[(size_t)j * d + i] - st * G1[(size_t)j * d + i], q, xa);
      xb = fmaf(W3[(size_t)j * d + i] - st * G3[(size_t)j * d + i], q, xb);
    }
    for (int u = 0; u <= t; ++u) {
      xa = fmaf(-st * KQ[(size_t)t * nt + u], DA[(size_t)u * dh + j], xa);
      xb = fmaf(-st * KQ[(size_t)t * nt + u], DB[(size_t)u * dh + j], xb);
    }
    Hq[idx] = xa * sigmoidf_(xa) * xb;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nt * nt; idx += blockDim.x) {  // KQ now holds h_q . h_k
    const int t = idx / nt, u = idx % nt;
    float acc = 0.f;
    if (u <= t)
      for (int j = 0; j < dh; ++j) acc = fmaf(Hq[(size_t)t * dh + j], Hk[(size_t)u * dh + j], acc);
    KQ[idx] = acc;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
    const int t = idx / d, i = idx % d;
    float o = 0.f;
    for (int j = 0; j < dh; ++j) o = fmaf(W2[(size_t)i * dh + j] - st * G2[(size_t)i * dh + j], Hq[(size_t)t * dh + j], o);
    for (int u = 0; u <= t; ++u) o = fmaf(-st * KQ[(size_t)t * nt + u] * eta(u, 1), Y[(size_t)u * d + i], o);
    st_val(a.O, base + idx, a.dtype, o);
  }
  __syncthreads();
}

// The linear net's block: o = (W - step G) q - step sum_{s<=t} (q.k_s) y_s, with
// Y = lr * dl/df (rates applied) on entry.
__device__ void inclusive_block_linear(const SimtArgs& a, float* ws, const SimtLayout& L, size_t head, int t0,
                                       int nt) {
  const int d = a.d;
  const size_t base = (head * a.T + t0) * (size_t)d;
  const float* W = ws + L.W[0];
  const float* G = ws + L.G[0];
  const float* Y = ws + L.Y;
  float* KQ = ws + L.KQ;
  const float st = a.step;
  for (int idx = threadIdx.x; idx < nt * nt; idx += blockDim.x) {
    const int t = idx / nt, u = idx % nt;
    float acc = 0.f;
    if (u <= t)
      for (int i = 0; i < d; ++i)
        acc = fmaf(ld_val(a.Q, base + (size_t)t * d + i, a.dtype), ld_val(a.K, base + (size_t)u * d + i, a.dtype), acc);
    KQ[idx] = acc;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
    const int t = idx / d, i = idx % d;
    float o = 0.f;
    for (int k = 0; k < d; ++k)
      o = fmaf(W[(size_t)i * d + k] - st * G[(size_t)i * d + k], ld_val(a.Q, base + (size_t)t * d + k, a.dtype), o);
    for (int u = 0; u <= t; ++u) o = fmaf(-st * KQ[(size_t)t * nt + u], Y[(size_t)u * d + i], o);
    st_val(a.O, base + idx, a.dtype, o);
  }
  __syncthreads();
}

__device__ void update_chunk(const SimtArgs& a, float* ws, const SimtLayout& L, size_t head,
                             int s, int e, float* red) {
  const int d = a.d, dh = a.dh;
  const int nw = a.fast_net == TTT_NET_SWIGLU ? 3 : 1;
  const int rows[3] = {nw == 3 ? dh : d, d, dh};
  const int cols[3] = {d, nw == 3 ? dh : d, d};
  for (int j = 0; j < nw; ++j)
    for (int idx = threadIdx.x; idx < rows[j] * cols[j]; idx += blockDim.x) ws[L.G[j] + idx] = 0.f;
  __syncthreads();
  for (int t0 = s; t0 < e; t0 += a.tb) {
    const int nt = min(a.tb, e - t0);
    const size_t base = (head * a.T + t0) * (size_t)d;
    // rate of token t for matrix j (j = 0 when every matrix shares it)
    const float* lr = a.lr + (head * a.T + t0) * a.lr_stride;
    const int ls = a.lr_stride;
    auto eta = [&](int t, int j) { return lr[(size_t)t * ls + (ls > 1 ? j : 0)]; };
    float* Y = ws + L.Y;
    if (a.fast_net == TTT_NET_SWIGLU) {
      const float* W1 = ws + L.W[0];
      const float* W2 = ws + L.W[1];
      const float* W3 = ws + L.W[2];
      float* A = ws + L.A;
      float* Bm = ws + L.Bm;
      float* Hh = ws + L.Hh;
      for (int idx = threadIdx.x; idx < nt * dh; idx += blockDim.x) {
        const int t = idx / dh, j = idx % dh;
        float xa = 0.f, xb = 0.f;
        for (int i = 0; i < d; ++i) {
          const float k = ld_val(a.K, base + (size_t)t * d + i, a.dtype);
          xa = fmaf(W1[(size_t)j * d + i], k, xa);
          xb = fmaf(W3[(size_t)j * d + i], k, xb);
        }
        A[idx] = xa;
        Bm[idx] = xb;
        Hh[idx] = xa * sigmoidf_(xa) * xb;
      }
      __syncthreads();
      for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
        const int t = idx / d, i = idx % d;
        const float v = ld_val(a.V, base + idx, a.dtype);
        float y;  // dl/df of token t, without its rate
        if (a.loss == TTT_LOSS_MSE) {
          float f = 0.f;
          for (int j = 0; j < dh; ++j) f = fmaf(W2[(size_t)i * dh + j], Hh[(size_t)t * dh + j], f);
          y = f - v;
        } else {
          y = -v;
        }
        Y[idx] = y;
      }
      __syncthreads();
      for (int idx = threadIdx.x; idx < nt * dh; idx += blockDim.x) {
        const int t = idx / dh, j = idx % dh;
        float g = 0.f;
        for (int i = 0; i < d; ++i) g = fmaf(Y[(size_t)t * d + i], W2[(size_t)i * dh + j], g);
        const float xa = A[idx], xb = Bm[idx];
        const float sg = sigmoidf_(xa);
        A[idx] = eta(t, 0) * g * xb * sg * (1.f + xa * (1.f - sg));   // lr1 * dl/da
        Bm[idx] = eta(t, 2) * g * xa * sg;                             // lr3 * dl/db
      }
      __syncthreads();
      if (a.mode == TTT_MODE_INCLUSIVE) inclusive_block_swiglu(a, ws, L, head, t0, nt, eta);
      float* G1 = ws + L.G[0];
      float* G2 = ws + L.G[1];
      float* G3 = ws + L.G[2];
      for (int idx = threadIdx.x; idx < d * dh; idx += blockDim.x) {
        const int i = idx / dh, j = idx % dh;
        float acc = 0.f;
        for (int t = 0; t < nt; ++t) acc = fmaf(eta(t, 1) * Y[(size_t)t * d + i], Hh[(size_t)t * dh + j], acc);
        G2[idx] += acc;
      }
      for (int idx = threadIdx.x; idx < dh * d; idx += blockDim.x) {
        const int j = idx / d, i = idx % d;
        float acc1 = 0.f, acc3 = 0.f;
        for (int t = 0; t < nt; ++t) {
          const float k = ld_val(a.K, base + (size_t)t * d + i, a.dtype);
          acc1 = fmaf(A[(size_t)t * dh + j], k, acc1);
          acc3 = fmaf(Bm[(size_t)t * dh + j], k, acc3);
        }
        G1[idx] += acc1;
        G3[idx] += acc3;
      }
      __syncthreads();
    } else {
      const float* W = ws + L.W[0];
      for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
        const int t = idx / d, i = idx % d;
        const float v = ld_val(a.V, base + idx, a.dtype);
        float y;
        if (a.loss == TTT_LOSS_MSE) {
          float f = 0.f;
          for (int k = 0; k < d; ++k)
            f = fmaf(W[(size_t)i * d + k], ld_val(a.K, base + (size_t)t * d + k, a.dtype), f);
          y = eta(t, 0) * (f - v);
        } else {
          y = -eta(t, 0) * v;
        }
        Y[idx] = y;
      }
      __syncthreads();
      if (a.mode == TTT_MODE_INCLUSIVE) inclusive_block_linear(a, ws, L, head, t0, nt);
      float* G = ws + L.G[0];
      for (int idx = threadIdx.x; idx < d * d; idx += blockDim.x) {
        const int i = idx / d, k = idx % d;
        float acc = 0.f;
        for (int t = 0; t < nt; ++t)
          acc = fmaf(Y[(size_t)t * d + i], ld_val(a.K, base + (size_t)t * d + k, a.dtype), acc);
        G[idx] += acc;
      }
      __syncthreads();
    }
  }
  for (int j = 0; j < nw; ++j) {
    float* G = ws + L.G[j];
    float* W = ws + L.W[j];
    if (a.momentum != 0.f) {
      // B <- mu B + G; B is what Newton-Schulz (or the plain step) receives
      float* Mo = ws + L.Mom[j];
      for (int idx = threadIdx.x; idx < rows[j] * cols[j]; idx += blockDim.x) {
        const float b = fmaf(a.momentum, Mo[idx], G[idx]);
        Mo[idx] = b;
        G[idx] = b;
      }
      __syncthreads();
    }
    if (a.muon) newton_schulz(a, G, rows[j], cols[j], ws, L, red);
    for (int idx = threadIdx.x; idx < rows[j] * cols[j]; idx += blockDim.x) W[idx] -= a.step * G[idx];
    __syncthreads();
    if (a.wnorm) {
      renorm_rows(W, rows[j], cols[j], ws + L.N0[j], a.wnorm_eps);
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(kThreads) simt_layer_kernel(const __grid_constant__ SimtArgs a) {
  __shared__ float red[kThreads];
  const size_t head = blockIdx.x;
  const int b = (int)(head / a.H), h = (int)(head % a.H);
  const SimtLayout L = simt_layout(a.fast_net, a.d, a.dh, a.tb, a.momentum != 0.f);
  float* ws = a.scratch + head * a.head_floats;
  const int nw = a.fast_net == TTT_NET_SWIGLU ? 3 : 1;
  const int rows[3] = {nw == 3 ? a.dh : a.d, a.d, a.dh};
  const int cols[3] = {a.d, nw == 3 ? a.dh : a.d, a.d};
  for (int j = 0; j < nw; ++j) {
    const size_t n = (size_t)rows[j] * cols[j];
    const float* src = a.W0[j] + (a.w0_per_batch ? head : (size_t)h) * n;
    for (size_t idx = threadIdx.x; idx < n; idx += blockDim.x) ws[L.W[j] + idx] = src[idx];
  }
  __syncthreads();
  for (int j = 0; j < nw; ++j) row_norms(ws + L.W[j], rows[j], cols[j], ws + L.N0[j]);
  if (a.momentum != 0.f)
    for (int j = 0; j < nw; ++j)
      for (size_t idx = threadIdx.x; idx < (size_t)rows[j] * cols[j]; idx += blockDim.x) ws[L.Mom[j] + idx] = 0.f;
  __syncthreads();
  (void)b;
  const int n_chunks = (a.T + a.chunk - 1) / a.chunk;
  for (int c = 0; c < n_chunks; ++c) {
    const int s = c * a.chunk, e = min(a.T, s + a.chunk);
    const bool upd = !a.has_mask || mask_bit(a.mask, c);
    if (a.mode == TTT_MODE_SHIFTED) {
      apply_chunk(a, ws, L, head, s, e);
      if (upd) update_chunk(a, ws, L, head, s, e, red);
    } else if (a.mode == TTT_MODE_INCLUSIVE) {
      // the update writes the chunk's outputs on the way (each token block's
      // queries before the block's gradient joins the sum)
      if (upd)
        update_chunk(a, ws, L, head, s, e, red);
      else
        apply_chunk(a, ws, L, head, s, e);
    } else {
      if (upd) update_chunk(a, ws, L, head, s, e, red);
      apply_chunk(a, ws, L, head, s, e);
    }
  }
  for (int j = 0; j < nw; ++j) {
    const size_t n = (size_t)rows[j] * cols[j];
    for (size_t idx = threadIdx.x; idx < n; idx += blockDim.x) a.Wf[j][head * n + idx] = ws[L.W[j] + idx];
  }
}

}  // namespace

size_t simt_workspace_bytes(const ttt_cfg& cfg) {
  const int tb = cfg.chunk < kTokenBlock ? cfg.chunk : kTokenBlock;
  const SimtLayout L = simt_layout(cfg.fast_net, cfg.d, cfg.dh, tb, cfg.momentum != 0.f);
  return kStatusBytes + (size_t)cfg.B * cfg.H * L.total * sizeof(float);
}

int simt_run(const Call& c) {
  const ttt_cfg& g = c.cfg;
  if (!c.mask_all && c.n_chunks > kMaxMaskChunks) return TTT_ERR_UNSUPPORTED;
  SimtArgs a{};
  a.B = g.B; a.H = g.H; a.T = g.T; a.d = g.d; a.dh = g.dh; a.chunk = g.chunk;
  a.fast_net = g.fast_net; a.loss = g.loss; a.mode = g.mode; a.dtype = g.dtype;
  a.muon = g.muon; a.ns_iters = g.ns_iters; a.wnorm = g.wnorm; a.w0_per_batch = g.w0_per_batch;
  a.tb = g.chunk < kTokenBlock ? g.chunk : kTokenBlock;
  a.ns_a = g.ns_a; a.ns_b = g.ns_b; a.ns_c = g.ns_c; a.ns_eps = g.ns_eps;
  a.wnorm_eps = g.wnorm_eps; a.step = g.step;
  a.momentum = g.momentum;
  a.lr_stride = g.lr_per_matrix ? (g.fast_net == TTT_NET_SWIGLU ? 3 : 1) : 1;
  a.Q = c.Q; a.K = c.K; a.V = c.V; a.lr = c.lr;
  for (int j = 0; j < 3; ++j) { a.W0[j] = c.W0[j]; a.Wf[j] = c.Wf[j]; }
  a.O = c.O;
  a.status = reinterpret_cast<int*>(c.ws);
  a.scratch = reinterpret_cast<float*>(c.ws + kStatusBytes);
  a.head_floats = simt_layout(g.fast_net, g.d, g.dh, a.tb, g.momentum != 0.f).total;
  a.has_mask = c.mask_all ? 0 : 1;
  if (a.has_mask)
    for (int i = 0; i < c.n_chunks; ++i)
      if (c.mask[i]) a.mask.w[i >> 5] |= 1u << (i & 31);
  const unsigned heads = (unsigned)g.B * (unsigned)g.H;
  prof_before(TTT_KERNEL_SIMT, c.stream);
  simt_layer_kernel<<<heads, kThreads, 0, c.stream>>>(a);
  prof_after(TTT_KERNEL_SIMT, c.stream);
  return cudaGetLastError() == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

}  // namespace ttt
