// Outer-loop backward of the chunked TTT layer: the gradients of a scalar loss
// with respect to the layer's inputs, through the chunked updates (TTT-E2E
// news page §2.2: the model's loss is differentiated through the inner loop).
//
// Covered: the linear fast net with plain gradient steps (no Muon, momentum or
// weight norm) in shifted mode, inner-product or MSE loss, fp32 or bf16
// storage; the small-chunk regime of the LaCT page §1.1. Per chunk c of tokens
// t (rates lr_t, step s):
//   o_t = W_c q_t,  y_t = W_c k_t - v_t (MSE) or -v_t,  W_{c+1} = W_c - s sum_t lr_t y_t k_t^T.
// Reverse mode from the last chunk, with L_c = dL/dW_c and L_n = dL/dW_final:
//   a_t = -s L_{c+1} k_t,  e_t = lr_t a_t
//   dq_t = W_c^T dO_t,  dlr_t = y_t . a_t,  dv_t = -e_t,
//   dk_t = -s L_{c+1}^T (lr_t y_t) + [MSE] W_c^T e_t,
//   L_c = L_{c+1} + sum_t dO_t q_t^T + [MSE] sum_t e_t k_t^T,   dW0 = L_0.
//
// fp32 SIMT, one CTA per (batch, head), every reduction in a fixed order (two
// runs are bitwise equal). The forward pass keeps every chunk's starting
// weights in the workspace; the reverse pass reads them back. With W0 shared
// over the batch, a second kernel sums the per-(b, h) dW0 over b in order.
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kBwThreads = 256;
constexpr int kBwBlock = 64;  // tokens per block inside a chunk

struct BwArgs {
  int B, H, T, d, chunk, loss, dtype, w0_per_batch, has_mask, tb, lr_stride;
  float step;
  const void* Q;
  const void* K;
  const void* V;
  const float* lr;
  const float* W0;
  const void* dO;
  const float* dWf;
  void* dQ;
  void* dK;
  void* dV;
  float* dlr;
  float* dW;       // [B][H][d][d]: per-(b, h) dW0
  float* scratch;  // per head: W_c for every chunk, L (two), Y and A blocks
  size_t head_floats;
  MaskBits mask;
};

struct BwLayout {
  size_t Wc, L0, L1, Y, A, total;
};

__host__ __device__ inline BwLayout bw_layout(int d, int n_chunks, int tb) {
  BwLayout L{};
  const size_t dd = align_up((size_t)d * d, 64);
  L.Wc = 0;
  L.L0 = (size_t)n_chunks * dd;
  L.L1 = L.L0 + dd;
  L.Y = L.L1 + dd;
  L.A = L.Y + align_up((size_t)tb * d, 64);
  L.total = L.A + align_up((size_t)tb * d, 64);
  return L;
}

__global__ void __launch_bounds__(kBwThreads) linear_bwd_kernel(const __grid_constant__ BwArgs a) {
  const size_t head = blockIdx.x;
  const int h = (int)(head % a.H);
  const int d = a.d;
  const size_t dd = (size_t)d * d;
  const int n_chunks = (a.T + a.chunk - 1) / a.chunk;
  const BwLayout L = bw_layout(d, n_chunks, a.tb);
  float* ws = a.scratch + head * a.head_floats;
  const size_t ddp = align_up(dd, 64);
  auto Wc = [&](int c) { return ws + L.Wc + (size_t)c * ddp; };
  float* Y = ws + L.Y;
  float* A = ws + L.A;
  const float st = a.step;
  auto rate = [&](size_t t) { return a.lr[t * a.lr_stride]; };

  // ---- forward: every chunk's starting weights
  const float* w0 = a.W0 + (a.w0_per_batch ? head : (size_t)h) * dd;
  for (size_t i = threadIdx.x; i < dd; i += blockDim.x) Wc(0)[i] = w0[i];
  __syncthreads();
  for (int c = 0; c < n_chunks; ++c) {
    const int s = c * a.chunk, e = min(a.T, s + a.chunk);
    float* W = Wc(c);
    float* Wn = c + 1 < n_chunks ? Wc(c + 1) : ws + L.L1;  // the final weights are not needed
    for (size_t i = threadIdx.x; i < dd; i += blockDim.x) Wn[i] = W[i];
    __syncthreads();
    if (a.has_mask && !mask_bit(a.mask, c)) continue;
    for (int t0 = s; t0 < e; t0 += a.tb) {
      const int nt = min(a.tb, e - t0);
      const size_t base = (head * a.T + t0) * (size_t)d;
      for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
        const int t = idx / d, r = idx % d;
        float y = -ld_val(a.V, base + idx, a.dtype);
        if (a.loss == TTT_LOSS_MSE)
          for (int i = 0; i < d; ++i) y = fmaf(W[(size_t)r * d + i], ld_val(a.K, base + (size_t)t * d + i, a.dtype), y);
        Y[idx] = rate(head * a.T + t0 + t) * y;
      }
      __syncthreads();
      for (int idx = threadIdx.x; idx < d * d; idx += blockDim.x) {
        const int r = idx / d, i = idx % d;
        float g = 0.f;
        for (int t = 0; t < nt; ++t) g = fmaf(Y[(size_t)t * d + r], ld_val(a.K, base + (size_t)t * d + i, a.dtype), g);
        Wn[idx] -= st * g;
      }
      __syncthreads();
    }
  }

  // ---- reverse: L_next = dL/dW_{c+1}, L_cur accumulates dL/dW_c
  float* Lnext = ws + L.L0;
  float* Lcur = ws + L.L1;
  const float* dwf = a.dWf + head * dd;
  for (size_t i = threadIdx.x; i < dd; i += blockDim.x) Lnext[i] = dwf[i];
  __syncthreads();
  for (int c = n_chunks - 1; c >= 0; --c) {
    const int s = c * a.chunk, e = min(a.T, s + a.chunk);
    const float* W = Wc(c);
    const bool upd = !a.has_mask || mask_bit(a.mask, c);
    for (size_t i = threadIdx.x; i < dd; i += blockDim.x) Lcur[i] = Lnext[i];
    __syncthreads();
    for (int t0 = s; t0 < e; t0 += a.tb) {
      const int nt = min(a.tb, e - t0);
      const size_t base = (head * a.T + t0) * (size_t)d;
      // dq_t = W^T dO_t
      for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
        const int t = idx / d, i = idx % d;
        float g = 0.f;
        for (int r = 0; r < d; ++r) g = fmaf(W[(size_t)r * d + i], ld_val(a.dO, base + (size_t)t * d + r, a.dtype), g);
        st_val(a.dQ, base + idx, a.dtype, g);
      }
      if (upd) {
        // Y rows: lr_t y_t; A rows: a_t = -s L_next k_t
        for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
          const int t = idx / d, r = idx % d;
          float y = -ld_val(a.V, base + idx, a.dtype);
          float av = 0.f;
          for (int i = 0; i < d; ++i) {
            const float k = ld_val(a.K, base + (size_t)t * d + i, a.dtype);
            if (a.loss == TTT_LOSS_MSE) y = fmaf(W[(size_t)r * d + i], k, y);
            av = fmaf(Lnext[(size_t)r * d + i], k, av);
          }
          Y[idx] = y;  // y_t (the rate is applied below)
          A[idx] = -st * av;
        }
      }
      __syncthreads();
      if (upd) {
        // dlr_t = y_t . a_t, one warp per token (butterfly sum, fixed order)
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        for (int t = warp; t < nt; t += kBwThreads / 32) {
          float v = 0.f;
          for (int r = lane; r < d; r += 32) v = fmaf(Y[(size_t)t * d + r], A[(size_t)t * d + r], v);
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) a.dlr[(head * a.T + t0 + t) * a.lr_stride] = v;
        }
        // dv_t = -lr_t a_t;  dk_t = -s L_next^T (lr_t y_t) + [MSE] W^T (lr_t a_t)
        for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
          const int t = idx / d, i = idx % d;
          const float lt = rate(head * a.T + t0 + t);
          st_val(a.dV, base + idx, a.dtype, -lt * A[idx]);
          float g = 0.f;
          for (int r = 0; r < d; ++r) {
            g = fmaf(-st * Lnext[(size_t)r * d + i], lt * Y[(size_t)t * d + r], g);
            if (a.loss == TTT_LOSS_MSE) g = fmaf(W[(size_t)r * d + i], lt * A[(size_t)t * d + r], g);
          }
          st_val(a.dK, base + idx, a.dtype, g);
        }
      } else {
        for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
          const int t = idx / d;
          st_val(a.dV, base + idx, a.dtype, 0.f);
          st_val(a.dK, base + idx, a.dtype, 0.f);
          if (idx % d == 0) a.dlr[(head * a.T + t0 + t) * a.lr_stride] = 0.f;
        }
      }
      // L_cur += sum_t dO_t q_t^T + [MSE] sum_t (lr_t a_t) k_t^T
      for (int idx = threadIdx.x; idx < d * d; idx += blockDim.x) {
        const int r = idx / d, i = idx % d;
        float g = 0.f;
        for (int t = 0; t < nt; ++t) {
          g = fmaf(ld_val(a.dO, base + (size_t)t * d + r, a.dtype), ld_val(a.Q, base + (size_t)t * d + i, a.dtype), g);
          if (upd && a.loss == TTT_LOSS_MSE)
            g = fmaf(rate(head * a.T + t0 + t) * A[(size_t)t * d + r], ld_val(a.K, base + (size_t)t * d + i, a.dtype), g);
        }
        Lcur[idx] += g;
      }
      __syncthreads();
    }
    float* tmp = Lnext;
    Lnext = Lcur;
    Lcur = tmp;
    __syncthreads();
  }
  for (size_t i = threadIdx.x; i < dd; i += blockDim.x) a.dW[head * dd + i] = Lnext[i];
}

// dW0[h] = sum over b of the per-(b, h) gradients, b in order.
__global__ void sum_over_batch_kernel(const float* dW, float* dW0, int B, int H, size_t dd) {
  const size_t n = (size_t)H * dd;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    float acc = 0.f;
    for (int b = 0; b < B; ++b) acc += dW[(size_t)b * n + i];
    dW0[i] = acc;
  }
}

// ---------------------------------------------------------------- SwiGLU net
// The SwiGLU net f(x) = W2 (silu(W1 x) * (W3 x)) with plain gradient steps in
// shifted mode, the inner-product loss l = -<f(k), v> or the MSE loss
// l = |f(k) - v|^2 / 2; one rate per token (lr_t) for all three matrices. Per chunk c: o_t = f(q_t; W_c) for its
// queries and W_{c+1} = W_c - s sum_t lr_t grad_W l_t(W_c). With Lh = dL/dW_{c+1}
// (the adjoint reaching W_{c+1}) and phi_t = <Lh, grad_W l_t(W_c)>:
//   dL/dW_c = Lh - s sum_t lr_t grad_W phi_t + sum_t grad_W <dO_t, f(q_t; W_c)>
//   dlr_t = -s phi_t,  dk_t = -s lr_t grad_k phi_t,  dv_t = -s lr_t grad_v phi_t,
// phi_t being the derivative of l_t along Lh. With a = W1 k, b = W3 k, s = silu(a),
// h = s b, f = W2 h, the loss's dl/df = y (y = -v for the inner product, f - v for
// MSE) and the tangents along Lh (dots): a' = Lh1 k, b' = Lh3 k, s' = silu'(a) a',
// h' = s' b + s b', f' = Lh2 h + W2 h':
//   phi = y . f';  grad_v phi = -f';  grad_W2 phi = y h'^T [+ f' h^T for MSE];
//   gh = Lh2^T y [+ W2^T f' for MSE],  gh' = W2^T y,
//   gs = gh b + gh' b',  gb = gh s + gh' s',  gs' = gh' b,  gb' = gh' s,
//   ga = gs silu'(a) + gs' silu''(a) a',  ga' = gs' silu'(a),
//   grad_W1 phi = ga k^T,  grad_W3 phi = gb k^T,
//   grad_k phi = W1^T ga + W3^T gb + Lh1^T ga' + Lh3^T gb',
// with silu'(a) = sig (1 + a (1 - sig)) and silu''(a) = sig (1 - sig) (2 + a (1 - 2 sig)).
// fp32 SIMT, one CTA per (batch, head), every sum in a fixed order.
constexpr int kSwTb = 16;  // tokens per block

struct SwArgs {
  int B, H, T, d, dh, chunk, dtype, w0_per_batch, has_mask, loss;
  float step;
  const void* Q;
  const void* K;
  const void* V;
  const float* lr;
  const float* W0[3];
  const void* dO;
  const float* dWf[3];
  void* dQ;
  void* dK;
  void* dV;
  float* dlr;
  float* dW[3];    // per-(b, h) dW0 of each matrix
  float* scratch;  // per head: W_c of every chunk, two adjoints, the token block's vectors
  size_t head_floats;
  MaskBits mask;
};

struct SwLayout {
  size_t mat, Wc, L0, L1, vec, fd, cv, total;  // mat: floats of one matrix (padded)
};

__host__ __device__ inline SwLayout sw_layout(int d, int dh, int n_chunks) {
  SwLayout L{};
  L.mat = align_up((size_t)d * dh, 64);
  L.Wc = 0;
  L.L0 = (size_t)n_chunks * 3 * L.mat;
  L.L1 = L.L0 + 3 * L.mat;
  L.vec = L.L1 + 3 * L.mat;                                    // 13 vectors of [kSwTb][dh]
  L.fd = L.vec + 13 * align_up((size_t)kSwTb * dh, 64);       // f' of the block: [kSwTb][d]
  L.cv = L.fd + align_up((size_t)kSwTb * d, 64);               // y (dl/df) of the block: [kSwTb][d]
  L.total = L.cv + align_up((size_t)kSwTb * d, 64);
  return L;
}

__device__ __forceinline__ float sw_sig(float x) { return 1.f / (1.f + expf(-x)); }

__global__ void __launch_bounds__(kBwThreads) swiglu_bwd_kernel(const __grid_constant__ SwArgs a) {
  const size_t head = blockIdx.x;
  const int h = (int)(head % a.H);
  const int d = a.d, dh = a.dh;
  const size_t dd = (size_t)d * dh;
  const int n_chunks = (a.T + a.chunk - 1) / a.chunk;
  const SwLayout L = sw_layout(d, dh, n_chunks);
  float* ws = a.scratch + head * a.head_floats;
  // matrix j of the weights at the start of chunk c; W1, W3: [dh][d]; W2: [d][dh]
  auto Wc = [&](int c, int j) { return ws + L.Wc + ((size_t)c * 3 + j) * L.mat; };
  const size_t vs = align_up((size_t)kSwTb * dh, 64);
  auto vec = [&](int i) { return ws + L.vec + (size_t)i * vs; };
  float* FD = ws + L.fd;
  float* CV = ws + L.cv;
  const bool mse = a.loss == TTT_LOSS_MSE;
  const float st = a.step;
  auto tok = [&](const void* p, size_t t, int i) { return ld_val(p, (head * a.T + t) * (size_t)d + i, a.dtype); };

  // ---- forward: every chunk's starting weights
  for (int j = 0; j < 3; ++j) {
    const float* w0 = a.W0[j] + (a.w0_per_batch ? head : (size_t)h) * dd;
    for (size_t i = threadIdx.x; i < dd; i += blockDim.x) Wc(0, j)[i] = w0[i];
  }
  __syncthreads();
  for (int c = 0; c + 1 < n_chunks; ++c) {
    const int s = c * a.chunk, e = min(a.T, s + a.chunk);
    for (int j = 0; j < 3; ++j)
      for (size_t i = threadIdx.x; i < dd; i += blockDim.x) Wc(c + 1, j)[i] = Wc(c, j)[i];
    __syncthreads();
    if (a.has_mask && !mask_bit(a.mask, c)) continue;
    const float *W1 = Wc(c, 0), *W2 = Wc(c, 1), *W3 = Wc(c, 2);
    float *N1 = Wc(c + 1, 0), *N2 = Wc(c + 1, 1), *N3 = Wc(c + 1, 2);
    float *AA = vec(0), *BB = vec(1), *HH = vec(2), *DA = vec(3), *DB = vec(4);
    for (int t0 = s; t0 < e; t0 += kSwTb) {
      const int nt = min(kSwTb, e - t0);
      // a, b, h
      for (int idx = threadIdx.x; idx < nt * dh; idx += blockDim.x) {
        const int t = idx / dh, jj = idx % dh;
        float av = 0.f, bv = 0.f;
        for (int i = 0; i < d; ++i) {
          const float k = tok(a.K, t0 + t, i);
          av = fmaf(W1[(size_t)jj * d + i], k, av);
          bv = fmaf(W3[(size_t)jj * d + i], k, bv);
        }
        AA[idx] = av;
        BB[idx] = bv;
        HH[idx] = av * sw_sig(av) * bv;
      }
      __syncthreads();
      // CV = lr y: y = -v (inner product) or W2 h - v (MSE)
      for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
        const int t = idx / d, r = idx % d;
        float y = -tok(a.V, t0 + t, r);
        if (mse)
          for (int jj = 0; jj < dh; ++jj) y = fmaf(W2[(size_t)r * dh + jj], HH[(size_t)t * dh + jj], y);
        CV[idx] = a.lr[head * a.T + t0 + t] * y;
      }
      __syncthreads();
      // DA = (W2^T CV) b silu'(a),  DB = (W2^T CV) s
      for (int idx = threadIdx.x; idx < nt * dh; idx += blockDim.x) {
        const int t = idx / dh, jj = idx % dh;
        float dhv = 0.f;
        for (int r = 0; r < d; ++r) dhv = fmaf(W2[(size_t)r * dh + jj], CV[(size_t)t * d + r], dhv);
        const float av = AA[idx], sg = sw_sig(av);
        DA[idx] = dhv * BB[idx] * sg * (1.f + av * (1.f - sg));
        DB[idx] = dhv * av * sg;
      }
      __syncthreads();
      // W1 -= s sum_t DA k^T;  W3 -= s sum_t DB k^T;  W2 -= s sum_t CV h^T
      for (size_t idx = threadIdx.x; idx < dd; idx += blockDim.x) {
        const int jj = (int)(idx / d), i = (int)(idx % d);
        float g1 = 0.f, g3 = 0.f;
        for (int t = 0; t < nt; ++t) {
          const float k = tok(a.K, t0 + t, i);
          g1 = fmaf(DA[(size_t)t * dh + jj], k, g1);
          g3 = fmaf(DB[(size_t)t * dh + jj], k, g3);
        }
        N1[idx] -= st * g1;
        N3[idx] -= st * g3;
        const int r = (int)(idx / dh), jq = (int)(idx % dh);
        float g2 = 0.f;
        for (int t = 0; t < nt; ++t) g2 = fmaf(CV[(size_t)t * d + r], HH[(size_t)t * dh + jq], g2);
        N2[idx] -= st * g2;
      }
      __syncthreads();
    }
  }

  // ---- reverse: Ln = dL/dW_{c+1}, Lc accumulates dL/dW_c
  float* Ln[3] = {ws + L.L0, ws + L.L0 + L.mat, ws + L.L0 + 2 * L.mat};
  float* Lc[3] = {ws + L.L1, ws + L.L1 + L.mat, ws + L.L1 + 2 * L.mat};
  for (int j = 0; j < 3; ++j) {
    const float* dwf = a.dWf[j] + head * dd;
    for (size_t i = threadIdx.x; i < dd; i += blockDim.x) Ln[j][i] = dwf[i];
  }
  __syncthreads();
  for (int c = n_chunks - 1; c >= 0; --c) {
    const int s = c * a.chunk, e = min(a.T, s + a.chunk);
    const float *W1 = Wc(c, 0), *W2 = Wc(c, 1), *W3 = Wc(c, 2);
    const bool upd = !a.has_mask || mask_bit(a.mask, c);
    for (int j = 0; j < 3; ++j)
      for (size_t i = threadIdx.x; i < dd; i += blockDim.x) Lc[j][i] = Ln[j][i];
    __syncthreads();
    for (int t0 = s; t0 < e; t0 += kSwTb) {
      const int nt = min(kSwTb, e - t0);
      // -- queries: GA = gh b silu'(a), GB = gh s, HQ = h with gh = W2^T dO
      float *GA = vec(0), *GB = vec(1), *HQ = vec(2);
      for (int idx = threadIdx.x; idx < nt * dh; idx += blockDim.x) {
        const int t = idx / dh, jj = idx % dh;
        float av = 0.f, bv = 0.f, gh = 0.f;
        for (int i = 0; i < d; ++i) {
          const float q = tok(a.Q, t0 + t, i);
          av = fmaf(W1[(size_t)jj * d + i], q, av);
          bv = fmaf(W3[(size_t)jj * d + i], q, bv);
        }
        for (int r = 0; r < d; ++r) gh = fmaf(W2[(size_t)r * dh + jj], tok(a.dO, t0 + t, r), gh);
        const float sg = sw_sig(av), sa = av * sg;
        GA[idx] = gh * bv * sg * (1.f + av * (1.f - sg));
        GB[idx] = gh * sa;
        HQ[idx] = sa * bv;
      }
      __syncthreads();
      // dq = W1^T GA + W3^T GB
      for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
        const int t = idx / d, i = idx % d;
        float g = 0.f;
        for (int jj = 0; jj < dh; ++jj) {
          g = fmaf(W1[(size_t)jj * d + i], GA[(size_t)t * dh + jj], g);
          g = fmaf(W3[(size_t)jj * d + i], GB[(size_t)t * dh + jj], g);
        }
        st_val(a.dQ, (head * a.T + t0 + t) * (size_t)d + i, a.dtype, g);
      }
      // Lc1 += GA q^T, Lc3 += GB q^T, Lc2 += dO HQ^T
      for (size_t idx = threadIdx.x; idx < dd; idx += blockDim.x) {
        const int jj = (int)(idx / d), i = (int)(idx % d);
        float g1 = 0.f, g3 = 0.f;
        for (int t = 0; t < nt; ++t) {
          const float q = tok(a.Q, t0 + t, i);
          g1 = fmaf(GA[(size_t)t * dh + jj], q, g1);
          g3 = fmaf(GB[(size_t)t * dh + jj], q, g3);
        }
        Lc[0][idx] += g1;
        Lc[2][idx] += g3;
        const int r = (int)(idx / dh), jq = (int)(idx % dh);
        float g2 = 0.f;
        for (int t = 0; t < nt; ++t) g2 = fmaf(tok(a.dO, t0 + t, r), HQ[(size_t)t * dh + jq], g2);
        Lc[1][idx] += g2;
      }
      __syncthreads();
      if (!upd) {
        for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
          const int t = idx / d;
          const size_t o = (head * a.T + t0 + t) * (size_t)d + idx % d;
          st_val(a.dK, o, a.dtype, 0.f);
          st_val(a.dV, o, a.dtype, 0.f);
          if (idx % d == 0) a.dlr[head * a.T + t0 + t] = 0.f;
        }
        continue;
      }
      // -- keys: the vectors of phi_t along Ln
      float *AV = vec(0), *BV = vec(1), *AD = vec(2), *BD = vec(3), *U = vec(4), *UH = vec(5);
      float *HK = vec(6), *HD = vec(7), *XA = vec(8), *XB = vec(9), *XAD = vec(10), *XBD = vec(11), *WF = vec(12);
      for (int idx = threadIdx.x; idx < nt * dh; idx += blockDim.x) {
        const int t = idx / dh, jj = idx % dh;
        float av = 0.f, bv = 0.f, ad = 0.f, bd = 0.f;
        for (int i = 0; i < d; ++i) {
          const float k = tok(a.K, t0 + t, i);
          av = fmaf(W1[(size_t)jj * d + i], k, av);
          bv = fmaf(W3[(size_t)jj * d + i], k, bv);
          ad = fmaf(Ln[0][(size_t)jj * d + i], k, ad);
          bd = fmaf(Ln[2][(size_t)jj * d + i], k, bd);
        }
        AV[idx] = av; BV[idx] = bv; AD[idx] = ad; BD[idx] = bd;
        HK[idx] = av * sw_sig(av) * bv;
      }
      __syncthreads();
      // y = dl/df: -v, or W2 h - v (MSE)
      for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
        const int t = idx / d, r = idx % d;
        float y = -tok(a.V, t0 + t, r);
        if (mse)
          for (int jj = 0; jj < dh; ++jj) y = fmaf(W2[(size_t)r * dh + jj], HK[(size_t)t * dh + jj], y);
        CV[idx] = y;
      }
      __syncthreads();
      // u = W2^T y, u' = Ln2^T y; h' = s' b + s b'
      for (int idx = threadIdx.x; idx < nt * dh; idx += blockDim.x) {
        const int t = idx / dh, jj = idx % dh;
        float u = 0.f, uh = 0.f;
        for (int r = 0; r < d; ++r) {
          const float y = CV[(size_t)t * d + r];
          u = fmaf(W2[(size_t)r * dh + jj], y, u);
          uh = fmaf(Ln[1][(size_t)r * dh + jj], y, uh);
        }
        U[idx] = u;
        UH[idx] = uh;
        const float av = AV[idx], sg = sw_sig(av);
        const float s1 = sg * (1.f + av * (1.f - sg));
        HD[idx] = s1 * AD[idx] * BV[idx] + av * sg * BD[idx];
      }
      __syncthreads();
      // f' = Ln2 h + W2 h';  dv = -s lr (-f')
      for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
        const int t = idx / d, r = idx % d;
        float f = 0.f;
        for (int jj = 0; jj < dh; ++jj) {
          f = fmaf(Ln[1][(size_t)r * dh + jj], HK[(size_t)t * dh + jj], f);
          f = fmaf(W2[(size_t)r * dh + jj], HD[(size_t)t * dh + jj], f);
        }
        FD[idx] = f;
        const float lt = a.lr[head * a.T + t0 + t];
        st_val(a.dV, (head * a.T + t0 + t) * (size_t)d + r, a.dtype, st * lt * f);
      }
      __syncthreads();
      // gh = u' [+ W2^T f' for MSE], gh' = u: the gradients of phi along a, b, a', b'
      for (int idx = threadIdx.x; idx < nt * dh; idx += blockDim.x) {
        const int t = idx / dh, jj = idx % dh;
        float wf = 0.f;
        if (mse)
          for (int r = 0; r < d; ++r) wf = fmaf(W2[(size_t)r * dh + jj], FD[(size_t)t * d + r], wf);
        WF[idx] = wf;
        const float av = AV[idx], bv = BV[idx], ad = AD[idx], bd = BD[idx];
        const float sg = sw_sig(av), sa = av * sg;
        const float s1 = sg * (1.f + av * (1.f - sg));
        const float s2 = sg * (1.f - sg) * (2.f + av * (1.f - 2.f * sg));
        const float gh = UH[idx] + wf, ghd = U[idx];
        const float gs = gh * bv + ghd * bd, gsd = ghd * bv;
        XA[idx] = gs * s1 + gsd * s2 * ad;   // grad_a phi
        XB[idx] = gh * sa + ghd * s1 * ad;   // grad_b phi
        XAD[idx] = gsd * s1;                 // grad_a' phi
        XBD[idx] = ghd * sa;                 // grad_b' phi
      }
      __syncthreads();
      // dk = -s lr (W1^T XA + W3^T XB + Ln1^T XAD + Ln3^T XBD)
      for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
        const int t = idx / d, i = idx % d;
        float g = 0.f;
        for (int jj = 0; jj < dh; ++jj) {
          const size_t o = (size_t)t * dh + jj, w = (size_t)jj * d + i;
          g = fmaf(W1[w], XA[o], g);
          g = fmaf(W3[w], XB[o], g);
          g = fmaf(Ln[0][w], XAD[o], g);
          g = fmaf(Ln[2][w], XBD[o], g);
        }
        const float lt = a.lr[head * a.T + t0 + t];
        st_val(a.dK, (head * a.T + t0 + t) * (size_t)d + i, a.dtype, -st * lt * g);
      }
      // phi_t = y . f';  dlr = -s phi
      for (int t = threadIdx.x; t < nt; t += blockDim.x) {
        float ph = 0.f;
        for (int r = 0; r < d; ++r) ph = fmaf(CV[(size_t)t * d + r], FD[(size_t)t * d + r], ph);
        a.dlr[head * a.T + t0 + t] = -st * ph;
      }
      // Lc1 -= s sum lr XA k^T;  Lc3 -= s sum lr XB k^T;  Lc2 -= s sum lr (y h'^T [+ f' h^T])
      for (size_t idx = threadIdx.x; idx < dd; idx += blockDim.x) {
        const int jj = (int)(idx / d), i = (int)(idx % d);
        float g1 = 0.f, g3 = 0.f;
        for (int t = 0; t < nt; ++t) {
          const float lk = a.lr[head * a.T + t0 + t] * tok(a.K, t0 + t, i);
          g1 = fmaf(XA[(size_t)t * dh + jj], lk, g1);
          g3 = fmaf(XB[(size_t)t * dh + jj], lk, g3);
        }
        Lc[0][idx] -= st * g1;
        Lc[2][idx] -= st * g3;
        const int r = (int)(idx / dh), jq = (int)(idx % dh);
        float g2 = 0.f;
        for (int t = 0; t < nt; ++t) {
          const float lt = a.lr[head * a.T + t0 + t];
          float gw = CV[(size_t)t * d + r] * HD[(size_t)t * dh + jq];
          if (mse) gw = fmaf(FD[(size_t)t * d + r], HK[(size_t)t * dh + jq], gw);
          g2 = fmaf(lt, gw, g2);
        }
        Lc[1][idx] -= st * g2;
      }
      __syncthreads();
    }
    for (int j = 0; j < 3; ++j) {
      float* tmp = Ln[j];
      Ln[j] = Lc[j];
      Lc[j] = tmp;
    }
    __syncthreads();
  }
  for (int j = 0; j < 3; ++j)
    for (size_t i = threadIdx.x; i < dd; i += blockDim.x) a.dW[j][head * dd + i] = Ln[j][i];
}

}  // namespace

bool bwd_supported(const ttt_cfg& g) {
  return g.fast_net == TTT_NET_LINEAR && g.mode == TTT_MODE_SHIFTED && !g.muon && !g.wnorm && g.momentum == 0.f;
}

size_t bwd_workspace_bytes(const ttt_cfg& g) {
  const int n_chunks = (g.T + g.chunk - 1) / g.chunk;
  const int tb = g.chunk < kBwBlock ? g.chunk : kBwBlock;
  const size_t per_head = bw_layout(g.d, n_chunks, tb).total;
  const size_t heads = (size_t)g.B * g.H;
  // per-(b, h) dW0 (summed over b afterwards when W0 is shared), then the heads' scratch
  return kStatusBytes + align_up(heads * g.d * g.d * sizeof(float), 256) + heads * per_head * sizeof(float);
}

int bwd_run(const ttt_cfg& g, const void* Q, const void* K, const void* V, const float* lr, const float* W0,
            const void* dO, const float* dWf, void* dQ, void* dK, void* dV, float* dlr, float* dW0, char* ws,
            cudaStream_t st) {
  const int n_chunks = (g.T + g.chunk - 1) / g.chunk;
  if (g.update_mask && n_chunks > kMaxMaskChunks) return TTT_ERR_UNSUPPORTED;
  BwArgs a{};
  a.B = g.B; a.H = g.H; a.T = g.T; a.d = g.d; a.chunk = g.chunk; a.loss = g.loss; a.dtype = g.dtype;
  a.w0_per_batch = g.w0_per_batch;
  a.tb = g.chunk < kBwBlock ? g.chunk : kBwBlock;
  a.lr_stride = 1;  // one matrix: per-matrix rates have the per-token layout
  a.step = g.step;
  a.Q = Q; a.K = K; a.V = V; a.lr = lr; a.W0 = W0; a.dO = dO; a.dWf = dWf;
  a.dQ = dQ; a.dK = dK; a.dV = dV; a.dlr = dlr;
  const size_t heads = (size_t)g.B * g.H, dd = (size_t)g.d * g.d;
  a.dW = g.w0_per_batch ? dW0 : reinterpret_cast<float*>(ws + kStatusBytes);
  a.scratch = reinterpret_cast<float*>(ws + kStatusBytes + align_up(heads * dd * sizeof(float), 256));
  a.head_floats = bw_layout(g.d, n_chunks, a.tb).total;
  a.has_mask = 0;
  if (g.update_mask) {
    for (int i = 0; i < n_chunks; ++i)
      if (!g.update_mask[i]) a.has_mask = 1;
    for (int i = 0; i < n_chunks; ++i)
      if (g.update_mask[i]) a.mask.w[i >> 5] |= 1u << (i & 31);
  }
  prof_before(TTT_KERNEL_SIMT, st);
  linear_bwd_kernel<<<(unsigned)heads, kBwThreads, 0, st>>>(a);
  prof_after(TTT_KERNEL_SIMT, st);
  if (cudaGetLastError() != cudaSuccess) return TTT_ERR_CUDA;
  if (!g.w0_per_batch) {
    prof_before(TTT_KERNEL_AUX, st);
    sum_over_batch_kernel<<<256, 256, 0, st>>>(a.dW, dW0, g.B, g.H, dd);
    prof_after(TTT_KERNEL_AUX, st);
    if (cudaGetLastError() != cudaSuccess) return TTT_ERR_CUDA;
  }
  return TTT_OK;
}

}  // namespace ttt

namespace ttt {

bool bwd_swiglu_supported(const ttt_cfg& g) {
  return g.fast_net == TTT_NET_SWIGLU && g.mode == TTT_MODE_SHIFTED && !g.muon && !g.wnorm &&
         g.momentum == 0.f && !g.lr_per_matrix;
}

size_t bwd_swiglu_workspace_bytes(const ttt_cfg& g) {
  const int n_chunks = (g.T + g.chunk - 1) / g.chunk;
  const size_t heads = (size_t)g.B * g.H, dd = (size_t)g.d * g.dh;
  const size_t per_head = sw_layout(g.d, g.dh, n_chunks).total;
  return kStatusBytes + 3 * align_up(heads * dd * sizeof(float), 256) + heads * per_head * sizeof(float);
}

int bwd_swiglu_run(const ttt_cfg& g, const void* Q, const void* K, const void* V, const float* lr,
                   const float* const W0[3], const void* dO, const float* const dWf[3], void* dQ, void* dK, void* dV,
                   float* dlr, float* const dW0[3], char* ws, cudaStream_t st) {
  const int n_chunks = (g.T + g.chunk - 1) / g.chunk;
  if (g.update_mask && n_chunks > kMaxMaskChunks) return TTT_ERR_UNSUPPORTED;
  SwArgs a{};
  a.B = g.B; a.H = g.H; a.T = g.T; a.d = g.d; a.dh = g.dh; a.chunk = g.chunk; a.dtype = g.dtype; a.loss = g.loss;
  a.w0_per_batch = g.w0_per_batch;
  a.step = g.step;
  a.Q = Q; a.K = K; a.V = V; a.lr = lr; a.dO = dO;
  a.dQ = dQ; a.dK = dK; a.dV = dV; a.dlr = dlr;
  const size_t heads = (size_t)g.B * g.H, dd = (size_t)g.d * g.dh;
  const size_t per = align_up(heads * dd * sizeof(float), 256);
  for (int j = 0; j < 3; ++j) {
    a.W0[j] = W0[j];
    a.dWf[j] = dWf[j];
    a.dW[j] = g.w0_per_batch ? dW0[j] : reinterpret_cast<float*>(ws + kStatusBytes + j * per);
  }
  a.scratch = reinterpret_cast<float*>(ws + kStatusBytes + 3 * per);
  a.head_floats = sw_layout(g.d, g.dh, n_chunks).total;
  a.has_mask = 0;
  if (g.update_mask) {
    for (int i = 0; i < n_chunks; ++i)
      if (!g.update_mask[i]) a.has_mask = 1;
    for (int i = 0; i < n_chunks; ++i)
      if (g.update_mask[i]) a.mask.w[i >> 5] |= 1u << (i & 31);
  }
  prof_before(TTT_KERNEL_SIMT, st);
  swiglu_bwd_kernel<<<(unsigned)heads, kBwThreads, 0, st>>>(a);
  prof_after(TTT_KERNEL_SIMT, st);
  if (cudaGetLastError() != cudaSuccess) return TTT_ERR_CUDA;
  if (!g.w0_per_batch) {
    for (int j = 0; j < 3; ++j) {
      prof_before(TTT_KERNEL_AUX, st);
      sum_over_batch_kernel<<<256, 256, 0, st>>>(a.dW[j], dW0[j], g.B, g.H, dd);
      prof_after(TTT_KERNEL_AUX, st);
      if (cudaGetLastError() != cudaSuccess) return TTT_ERR_CUDA;
    }
  }
  return TTT_OK;
}

}  // namespace ttt
