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
