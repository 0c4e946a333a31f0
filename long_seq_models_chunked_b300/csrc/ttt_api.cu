// C-ABI front end: argument validation, kernel-family selection, workspace
// planning, the device status word and the host-buffer wrapper.
#include <algorithm>
#include <cmath>
#include <cstring>

#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kAbiVersion = 2;
constexpr int64_t kMaxElems = int64_t(1) << 40;
constexpr int kMaxPipelineChunks = 512;  // per-chunk events of ttt_fwd_host

int elem_bytes(int dtype) { return dtype == TTT_DTYPE_F32 ? 4 : 2; }

}  // namespace

int validate_cfg(const ttt_cfg* g) {
  if (!g) return TTT_ERR_ARG;
  if (g->B < 1 || g->H < 1 || g->T < 1 || g->d < 1 || g->chunk < 1) return TTT_ERR_ARG;
  if (g->fast_net != TTT_NET_SWIGLU && g->fast_net != TTT_NET_LINEAR) return TTT_ERR_ARG;
  if (g->fast_net == TTT_NET_SWIGLU && g->dh < 1) return TTT_ERR_ARG;
  if (g->loss != TTT_LOSS_IP && g->loss != TTT_LOSS_MSE) return TTT_ERR_ARG;
  if (g->mode != TTT_MODE_SHIFTED && g->mode != TTT_MODE_SINGLE && g->mode != TTT_MODE_INCLUSIVE)
    return TTT_ERR_ARG;
  if (g->dtype != TTT_DTYPE_F32 && g->dtype != TTT_DTYPE_BF16) return TTT_ERR_ARG;
  if ((g->muon != 0 && g->muon != 1) || (g->wnorm != 0 && g->wnorm != 1)) return TTT_ERR_ARG;
  if (g->ns_iters < 0 || g->ns_iters > 64) return TTT_ERR_ARG;
  if (!std::isfinite(g->ns_a) || !std::isfinite(g->ns_b) || !std::isfinite(g->ns_c)) return TTT_ERR_ARG;
  if (!std::isfinite(g->ns_eps) || g->ns_eps < 0.f) return TTT_ERR_ARG;
  if (!std::isfinite(g->wnorm_eps) || !(g->wnorm_eps > 0.f)) return TTT_ERR_ARG;
  if (!std::isfinite(g->step)) return TTT_ERR_ARG;
  if (g->w0_per_batch != 0 && g->w0_per_batch != 1) return TTT_ERR_ARG;
  if (g->check_finite != 0 && g->check_finite != 1) return TTT_ERR_ARG;
  if (g->impl < TTT_IMPL_AUTO || g->impl > TTT_IMPL_LINEAR) return TTT_ERR_ARG;
  if (g->precision != TTT_PREC_SPLIT && g->precision != TTT_PREC_SINGLE) return TTT_ERR_ARG;
  if (!std::isfinite(g->momentum)) return TTT_ERR_ARG;
  if (g->lr_per_matrix != 0 && g->lr_per_matrix != 1) return TTT_ERR_ARG;
  // the inclusive order takes plain gradient steps (a prefix of a chunk has no Muon, momentum or norm)
  if (g->mode == TTT_MODE_INCLUSIVE && (g->muon || g->wnorm || g->momentum != 0.f)) return TTT_ERR_ARG;
  const int64_t tok = (int64_t)g->B * g->H * g->T;
  if (tok * g->d > kMaxElems) return TTT_ERR_ARG;
  const int64_t wd = g->fast_net == TTT_NET_SWIGLU ? (int64_t)g->d * g->dh : (int64_t)g->d * g->d;
  if ((int64_t)g->B * g->H * wd > kMaxElems) return TTT_ERR_ARG;
  return TTT_OK;
}

namespace {

int select_impl(const ttt_cfg& g) {
  switch (g.impl) {
    case TTT_IMPL_SIMT: return TTT_IMPL_SIMT;
    case TTT_IMPL_TC: return tc_supported(g) ? TTT_IMPL_TC : TTT_ERR_UNSUPPORTED;
    case TTT_IMPL_LINEAR: return linear_supported(g) ? TTT_IMPL_LINEAR : TTT_ERR_UNSUPPORTED;
    default: break;
  }
  if (g.dtype == TTT_DTYPE_BF16) {
    if (tc_supported(g)) return TTT_IMPL_TC;
    if (linear_supported(g)) return TTT_IMPL_LINEAR;
  }
  return TTT_IMPL_SIMT;
}

size_t impl_workspace(const ttt_cfg& g, int impl) {
  switch (impl) {
    case TTT_IMPL_TC: return tc_workspace_bytes(g);
    case TTT_IMPL_LINEAR: return linear_workspace_bytes(g);
    default: return simt_workspace_bytes(g);
  }
}

struct Range {
  const char* p;
  size_t n;
};

bool overlap(const Range& a, const Range& b) {
  if (!a.p || !b.p || !a.n || !b.n) return false;
  return a.p < b.p + b.n && b.p < a.p + a.n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Sizes {
  size_t tok_bytes, lr_bytes, w0_bytes[3], wf_bytes[3];
  int nw;
};

Sizes tensor_sizes(const ttt_cfg& g) {
  Sizes s{};
  const size_t tok = (size_t)g.B * g.H * g.T;
  s.tok_bytes = tok * g.d * elem_bytes(g.dtype);
  s.nw = g.fast_net == TTT_NET_SWIGLU ? 3 : 1;
  s.lr_bytes = tok * sizeof(float) * (g.lr_per_matrix ? s.nw : 1);
  const size_t wsz = s.nw == 3 ? (size_t)g.d * g.dh : (size_t)g.d * g.d;
  for (int j = 0; j < s.nw; ++j) {
    s.w0_bytes[j] = (size_t)(g.w0_per_batch ? g.B : 1) * g.H * wsz * sizeof(float);
    s.wf_bytes[j] = (size_t)g.B * g.H * wsz * sizeof(float);
  }
  return s;
}

}  // namespace

// Every tensor pointer must be device memory of the calling thread's current
// device: the tensor-core kernels read it through TMA tensor maps (some of them
// shared by a cluster through multicast), which must only ever cover this GPU's
// own memory. Host memory (pinned or not), managed memory and memory of
// another device are rejected before anything is launched.
int check_device_ptrs(const void* const* ptrs, int n) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TTT_ERR_CUDA;
  for (int i = 0; i < n; ++i) {
    if (!ptrs[i]) continue;
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, ptrs[i]) != cudaSuccess) {
      cudaGetLastError();  // clear the sticky-free error of the failed query
      return TTT_ERR_ARG;
    }
    if (a.type != cudaMemoryTypeDevice || a.device != dev) return TTT_ERR_ARG;
  }
  return TTT_OK;
}

namespace {

__global__ void check_finite_kernel(const void* p, size_t n, int dtype, int* status) {
  bool bad = false;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const float v = ld_val(p, i, dtype);
    bad |= !isfinite(v);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) set_status(status, TTT_ERR_NONFINITE);
}

}  // namespace

int launch_check_finite(const Call& c) {
  const ttt_cfg& g = c.cfg;
  const Sizes s = tensor_sizes(g);
  int* st = reinterpret_cast<int*>(c.ws);
  const size_t ntok = s.tok_bytes / elem_bytes(g.dtype);
  const void* tp[3] = {c.Q, c.K, c.V};
  prof_before(TTT_KERNEL_AUX, c.stream);
  for (int i = 0; i < 3; ++i) check_finite_kernel<<<592, 256, 0, c.stream>>>(tp[i], ntok, g.dtype, st);
  check_finite_kernel<<<592, 256, 0, c.stream>>>(c.lr, s.lr_bytes / 4, TTT_DTYPE_F32, st);
  for (int j = 0; j < s.nw; ++j)
    check_finite_kernel<<<592, 256, 0, c.stream>>>(c.W0[j], s.w0_bytes[j] / 4, TTT_DTYPE_F32, st);
  prof_after(TTT_KERNEL_AUX, c.stream);
  return cudaGetLastError() == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

}  // namespace ttt

using namespace ttt;

extern "C" {

void ttt_cfg_default(ttt_cfg* cfg) {
  if (!cfg) return;
  std::memset(cfg, 0, sizeof(*cfg));
  cfg->fast_net = TTT_NET_SWIGLU;
  cfg->loss = TTT_LOSS_IP;
  cfg->mode = TTT_MODE_SHIFTED;
  cfg->dtype = TTT_DTYPE_BF16;
  cfg->muon = 1;
  cfg->ns_iters = 5;
  cfg->ns_a = 3.4445f;
  cfg->ns_b = -4.7750f;
  cfg->ns_c = 2.0315f;
  cfg->ns_eps = 1e-7f;
  cfg->wnorm = 1;
  cfg->wnorm_eps = 1e-12f;
  cfg->step = 1.0f;
  cfg->update_mask = nullptr;
  cfg->w0_per_batch = 0;
  cfg->check_finite = 0;
  cfg->timeout_us = 2000000u;
  cfg->impl = TTT_IMPL_AUTO;
  cfg->precision = TTT_PREC_SPLIT;
  cfg->momentum = 0.f;
  cfg->lr_per_matrix = 0;
}

int ttt_abi_version(void) { return kAbiVersion; }

size_t ttt_cfg_size(void) { return sizeof(ttt_cfg); }

int ttt_select_impl(const ttt_cfg* cfg) {
  const int v = validate_cfg(cfg);
  if (v != TTT_OK) return v;
  return select_impl(*cfg);
}

int ttt_workspace_bytes(const ttt_cfg* cfg, size_t* bytes) {
  if (!bytes) return TTT_ERR_ARG;
  const int v = validate_cfg(cfg);
  if (v != TTT_OK) return v;
  const int impl = select_impl(*cfg);
  if (impl < 0) return impl;
  *bytes = impl_workspace(*cfg, impl);
  return TTT_OK;
}

}  // extern "C"

namespace ttt {

// The layer on device buffers. With `ready` / `done` (one event per chunk) the
// tensor-core family waits for ready[c] before chunk c and records done[c]
// after it; the other families wait for every ready event first.
int fwd_device(const ttt_cfg* cfg, const void* Q, const void* K, const void* V, const float* lr,
               const float* W0_1, const float* W0_2, const float* W0_3, void* O, float* Wf_1, float* Wf_2,
               float* Wf_3, void* workspace, size_t workspace_bytes, void* stream, const cudaEvent_t* ready,
               const cudaEvent_t* done) {
  int v = validate_cfg(cfg);
  if (v != TTT_OK) return v;
  const ttt_cfg& g = *cfg;
  const int impl = select_impl(g);
  if (impl < 0) return impl;
  const Sizes s = tensor_sizes(g);
  const void* in[4] = {Q, K, V, lr};
  for (const void* p : in)
    if (!p || !aligned16(p)) return TTT_ERR_ARG;
  const float* w0[3] = {W0_1, W0_2, W0_3};
  float* wf[3] = {Wf_1, Wf_2, Wf_3};
  for (int j = 0; j < s.nw; ++j)
    if (!w0[j] || !wf[j] || !aligned16(w0[j]) || !aligned16(wf[j])) return TTT_ERR_ARG;
  if (!O || !aligned16(O)) return TTT_ERR_ARG;
  const size_t need = impl_workspace(g, impl);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return TTT_ERR_WORKSPACE;
  // outputs may not overlap inputs, the workspace or each other
  Range outs[4] = {{(const char*)O, s.tok_bytes}, {}, {}, {}};
  for (int j = 0; j < s.nw; ++j) outs[1 + j] = {(const char*)wf[j], s.wf_bytes[j]};
  Range others[8] = {{(const char*)Q, s.tok_bytes}, {(const char*)K, s.tok_bytes},
                     {(const char*)V, s.tok_bytes}, {(const char*)lr, s.lr_bytes},
                     {}, {}, {}, {(const char*)workspace, need}};
  for (int j = 0; j < s.nw; ++j) others[4 + j] = {(const char*)w0[j], s.w0_bytes[j]};
  for (int i = 0; i < 4; ++i) {
    for (const Range& r : others)
      if (overlap(outs[i], r)) return TTT_ERR_ARG;
    for (int k = i + 1; k < 4; ++k)
      if (overlap(outs[i], outs[k])) return TTT_ERR_ARG;
  }
  {
    const void* ptrs[12] = {Q, K, V, lr, O, workspace};
    int n = 6;
    for (int j = 0; j < s.nw; ++j) {
      ptrs[n++] = w0[j];
      ptrs[n++] = wf[j];
    }
    v = check_device_ptrs(ptrs, n);
    if (v != TTT_OK) return v;
  }
  Call c{};
  c.cfg = g;
  if (c.cfg.timeout_us == 0) c.cfg.timeout_us = 2000000u;
  c.n_chunks = (g.T + g.chunk - 1) / g.chunk;
  c.nw = s.nw;
  if (s.nw == 3) {
    c.rows[0] = g.dh; c.cols[0] = g.d;
    c.rows[1] = g.d;  c.cols[1] = g.dh;
    c.rows[2] = g.dh; c.cols[2] = g.d;
  } else {
    c.rows[0] = g.d; c.cols[0] = g.d;
  }
  c.Q = Q; c.K = K; c.V = V; c.lr = lr;
  for (int j = 0; j < 3; ++j) { c.W0[j] = j < s.nw ? w0[j] : nullptr; c.Wf[j] = j < s.nw ? wf[j] : nullptr; }
  c.O = O;
  c.ws = static_cast<char*>(workspace);
  c.ws_bytes = workspace_bytes;
  c.stream = static_cast<cudaStream_t>(stream);
  c.mask = g.update_mask;
  c.mask_all = true;
  if (g.update_mask)
    for (int i = 0; i < c.n_chunks; ++i)
      if (!g.update_mask[i]) { c.mask_all = false; break; }
  if (ready && (impl != TTT_IMPL_TC || g.check_finite)) {
    // no per-chunk pipelining: every input must have arrived before anything runs
    for (int i = 0; i < c.n_chunks; ++i)
      if (cudaStreamWaitEvent(c.stream, ready[i], 0) != cudaSuccess) return TTT_ERR_CUDA;
  } else {
    c.chunk_ready = ready;
  }
  c.chunk_done = impl == TTT_IMPL_TC ? done : nullptr;
  if (cudaMemsetAsync(workspace, 0, sizeof(int), c.stream) != cudaSuccess) return TTT_ERR_CUDA;
  if (g.check_finite) {
    v = launch_check_finite(c);
    if (v != TTT_OK) return v;
  }
  switch (impl) {
    case TTT_IMPL_TC: return tc_run(c);
    case TTT_IMPL_LINEAR: return linear_run(c);
    default: return simt_run(c);
  }
}

}  // namespace ttt

extern "C" {

int ttt_fwd(const ttt_cfg* cfg, const void* Q, const void* K, const void* V, const float* lr,
            const float* W0_1, const float* W0_2, const float* W0_3, void* O, float* Wf_1,
            float* Wf_2, float* Wf_3, void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_device(cfg, Q, K, V, lr, W0_1, W0_2, W0_3, O, Wf_1, Wf_2, Wf_3, workspace, workspace_bytes, stream,
                    nullptr, nullptr);
}

int ttt_status(void* workspace, void* stream) {
  if (!workspace) return TTT_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return TTT_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return TTT_ERR_CUDA;
  return word;
}

int ttt_host_arena_bytes(const ttt_cfg* cfg, size_t* bytes) {
  if (!bytes) return TTT_ERR_ARG;
  size_t ws = 0;
  const int v = ttt_workspace_bytes(cfg, &ws);
  if (v != TTT_OK) return v;
  const Sizes s = tensor_sizes(*cfg);
  size_t total = 4 * align_up(s.tok_bytes, 256) + align_up(s.lr_bytes, 256);
  for (int j = 0; j < s.nw; ++j) total += align_up(s.w0_bytes[j], 256) + align_up(s.wf_bytes[j], 256);
  *bytes = total + align_up(ws, 256);
  return TTT_OK;
}

int ttt_fwd_host(const ttt_cfg* cfg, const void* Q, const void* K, const void* V, const float* lr,
                 const float* W0_1, const float* W0_2, const float* W0_3, void* O, float* Wf_1,
                 float* Wf_2, float* Wf_3, void* arena, size_t arena_bytes, void* stream) {
  size_t need = 0;
  int v = ttt_host_arena_bytes(cfg, &need);
  if (v != TTT_OK) return v;
  if (!arena || (reinterpret_cast<uintptr_t>(arena) & 255u) || arena_bytes < need)
    return TTT_ERR_WORKSPACE;
  const ttt_cfg& g = *cfg;
  const Sizes s = tensor_sizes(g);
  const void* hin[3] = {Q, K, V};
  const float* hw0[3] = {W0_1, W0_2, W0_3};
  float* hwf[3] = {Wf_1, Wf_2, Wf_3};
  for (const void* p : hin)
    if (!p) return TTT_ERR_ARG;
  if (!lr || !O) return TTT_ERR_ARG;
  for (int j = 0; j < s.nw; ++j)
    if (!hw0[j] || !hwf[j]) return TTT_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* p = static_cast<char*>(arena);
  void* din[3];
  for (int i = 0; i < 3; ++i) { din[i] = p; p += align_up(s.tok_bytes, 256); }
  float* dlr = reinterpret_cast<float*>(p);
  p += align_up(s.lr_bytes, 256);
  float* dw0[3] = {nullptr, nullptr, nullptr};
  float* dwf[3] = {nullptr, nullptr, nullptr};
  for (int j = 0; j < s.nw; ++j) { dw0[j] = reinterpret_cast<float*>(p); p += align_up(s.w0_bytes[j], 256); }
  void* dO = p;
  p += align_up(s.tok_bytes, 256);
  for (int j = 0; j < s.nw; ++j) { dwf[j] = reinterpret_cast<float*>(p); p += align_up(s.wf_bytes[j], 256); }
  void* dws = p;
  size_t ws_bytes = 0;
  ttt_workspace_bytes(cfg, &ws_bytes);

  // Chunk-pipelined copies: chunk c's queries, keys and values go in on one
  // copy stream while earlier chunks compute, and chunk c's outputs come back
  // on another as soon as they are written. Every (b, h) row block of a chunk
  // is one strided 2D copy. With pageable host memory the copies still run,
  // but without overlap.
  const int n_chunks = (g.T + g.chunk - 1) / g.chunk;
  const size_t es = g.dtype == TTT_DTYPE_F32 ? 4 : 2;
  const size_t row_pitch = (size_t)g.T * g.d * es;  // one (b, h) block of Q, K, V or O
  const size_t BH = (size_t)g.B * g.H;
  const bool pipelined = select_impl(g) == TTT_IMPL_TC && n_chunks <= kMaxPipelineChunks;
  cudaStream_t cin = nullptr, cout = nullptr;
  cudaEvent_t ev[2 * kMaxPipelineChunks + 1];
  int n_ev = 0;
  int rc = TTT_OK;
  auto fail = [&](int code) { rc = code; };
  if (cudaMemcpyAsync(dlr, lr, s.lr_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) fail(TTT_ERR_CUDA);
  for (int j = 0; j < s.nw && rc == TTT_OK; ++j)
    if (cudaMemcpyAsync(dw0[j], hw0[j], s.w0_bytes[j], cudaMemcpyHostToDevice, st) != cudaSuccess)
      fail(TTT_ERR_CUDA);
  if (rc == TTT_OK && pipelined) {
    if (cudaStreamCreateWithFlags(&cin, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&cout, cudaStreamNonBlocking) != cudaSuccess)
      fail(TTT_ERR_CUDA);
    for (int i = 0; i < 2 * n_chunks + 1 && rc == TTT_OK; ++i) {
      if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) fail(TTT_ERR_CUDA);
      else n_ev = i + 1;
    }
  }
  if (rc == TTT_OK && pipelined) {
    cudaEvent_t* ready = ev;
    cudaEvent_t* done = ev + n_chunks;
    cudaEvent_t start = ev[2 * n_chunks];
    // the copy streams start after everything enqueued on `stream` so far
    if (cudaEventRecord(start, st) != cudaSuccess || cudaStreamWaitEvent(cin, start, 0) != cudaSuccess)
      fail(TTT_ERR_CUDA);
    for (int ci = 0; ci < n_chunks && rc == TTT_OK; ++ci) {
      const size_t off = (size_t)ci * g.chunk * g.d * es;
      const size_t width = (size_t)std::min(g.chunk, g.T - ci * g.chunk) * g.d * es;
      for (int i = 0; i < 3 && rc == TTT_OK; ++i)
        if (cudaMemcpy2DAsync(static_cast<char*>(din[i]) + off, row_pitch, static_cast<const char*>(hin[i]) + off,
                              row_pitch, width, BH, cudaMemcpyHostToDevice, cin) != cudaSuccess)
          fail(TTT_ERR_CUDA);
      if (rc == TTT_OK && cudaEventRecord(ready[ci], cin) != cudaSuccess) fail(TTT_ERR_CUDA);
    }
    if (rc == TTT_OK) {
      const int r = fwd_device(cfg, din[0], din[1], din[2], dlr, dw0[0], dw0[1], dw0[2], dO, dwf[0], dwf[1],
                               dwf[2], dws, ws_bytes, stream, ready, done);
      if (r != TTT_OK) fail(r);
    }
    for (int ci = 0; ci < n_chunks && rc == TTT_OK; ++ci) {
      const size_t off = (size_t)ci * g.chunk * g.d * es;
      const size_t width = (size_t)std::min(g.chunk, g.T - ci * g.chunk) * g.d * es;
      if (cudaStreamWaitEvent(cout, done[ci], 0) != cudaSuccess ||
          cudaMemcpy2DAsync(static_cast<char*>(O) + off, row_pitch, static_cast<const char*>(dO) + off, row_pitch,
                            width, BH, cudaMemcpyDeviceToHost, cout) != cudaSuccess)
        fail(TTT_ERR_CUDA);
    }
  } else if (rc == TTT_OK) {
    for (int i = 0; i < 3 && rc == TTT_OK; ++i)
      if (cudaMemcpyAsync(din[i], hin[i], s.tok_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
        fail(TTT_ERR_CUDA);
    if (rc == TTT_OK) {
      const int r = fwd_device(cfg, din[0], din[1], din[2], dlr, dw0[0], dw0[1], dw0[2], dO, dwf[0], dwf[1],
                               dwf[2], dws, ws_bytes, stream, nullptr, nullptr);
      if (r != TTT_OK) fail(r);
    }
    if (rc == TTT_OK && cudaMemcpyAsync(O, dO, s.tok_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
      fail(TTT_ERR_CUDA);
  }
  for (int j = 0; j < s.nw && rc == TTT_OK; ++j)
    if (cudaMemcpyAsync(hwf[j], dwf[j], s.wf_bytes[j], cudaMemcpyDeviceToHost, st) != cudaSuccess)
      fail(TTT_ERR_CUDA);
  // wait for everything this call enqueued, then release the streams and events
  if (cin && cudaStreamSynchronize(cin) != cudaSuccess) fail(TTT_ERR_CUDA);
  if (cout && cudaStreamSynchronize(cout) != cudaSuccess) fail(TTT_ERR_CUDA);
  const int status = ttt_status(dws, stream);
  for (int i = 0; i < n_ev; ++i) cudaEventDestroy(ev[i]);
  if (cin) cudaStreamDestroy(cin);
  if (cout) cudaStreamDestroy(cout);
  return rc != TTT_OK ? rc : status;
}

int ttt_bwd_workspace_bytes(const ttt_cfg* cfg, size_t* bytes) {
  if (!bytes) return TTT_ERR_ARG;
  const int v = validate_cfg(cfg);
  if (v != TTT_OK) return v;
  if (!bwd_supported(*cfg)) return TTT_ERR_UNSUPPORTED;
  *bytes = bwd_workspace_bytes(*cfg);
  return TTT_OK;
}

int ttt_bwd(const ttt_cfg* cfg, const void* Q, const void* K, const void* V, const float* lr, const float* W0,
            const void* dO, const float* dWf, void* dQ, void* dK, void* dV, float* dlr, float* dW0,
            void* workspace, size_t workspace_bytes, void* stream) {
  size_t need = 0;
  int v = ttt_bwd_workspace_bytes(cfg, &need);
  if (v != TTT_OK) return v;
  const ttt_cfg& g = *cfg;
  const Sizes s = tensor_sizes(g);
  const void* in[7] = {Q, K, V, lr, W0, dO, dWf};
  void* out[5] = {dQ, dK, dV, dlr, dW0};
  for (const void* p : in)
    if (!p || !aligned16(p)) return TTT_ERR_ARG;
  for (const void* p : out)
    if (!p || !aligned16(p)) return TTT_ERR_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return TTT_ERR_WORKSPACE;
  // outputs may not overlap the inputs, the workspace or each other
  const size_t in_n[7] = {s.tok_bytes, s.tok_bytes, s.tok_bytes, s.lr_bytes, s.w0_bytes[0], s.tok_bytes,
                          s.wf_bytes[0]};
  const size_t out_n[5] = {s.tok_bytes, s.tok_bytes, s.tok_bytes, s.lr_bytes, s.w0_bytes[0]};
  for (int i = 0; i < 5; ++i) {
    const Range o{(const char*)out[i], out_n[i]};
    for (int k = 0; k < 7; ++k)
      if (overlap(o, Range{(const char*)in[k], in_n[k]})) return TTT_ERR_ARG;
    if (overlap(o, Range{(const char*)workspace, need})) return TTT_ERR_ARG;
    for (int k = i + 1; k < 5; ++k)
      if (overlap(o, Range{(const char*)out[k], out_n[k]})) return TTT_ERR_ARG;
  }
  const void* ptrs[13] = {Q, K, V, lr, W0, dO, dWf, dQ, dK, dV, dlr, dW0, workspace};
  v = check_device_ptrs(ptrs, 13);
  if (v != TTT_OK) return v;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return TTT_ERR_CUDA;
  return bwd_run(g, Q, K, V, lr, W0, dO, dWf, dQ, dK, dV, dlr, dW0, static_cast<char*>(workspace), st);
}

int ttt_bwd_swiglu_workspace_bytes(const ttt_cfg* cfg, size_t* bytes) {
  if (!bytes) return TTT_ERR_ARG;
  const int v = validate_cfg(cfg);
  if (v != TTT_OK) return v;
  if (!bwd_swiglu_supported(*cfg)) return TTT_ERR_UNSUPPORTED;
  *bytes = bwd_swiglu_workspace_bytes(*cfg);
  return TTT_OK;
}

int ttt_bwd_swiglu(const ttt_cfg* cfg, const void* Q, const void* K, const void* V, const float* lr,
                   const float* W0_1, const float* W0_2, const float* W0_3, const void* dO, const float* dWf_1,
                   const float* dWf_2, const float* dWf_3, void* dQ, void* dK, void* dV, float* dlr, float* dW0_1,
                   float* dW0_2, float* dW0_3, void* workspace, size_t workspace_bytes, void* stream) {
  size_t need = 0;
  int v = ttt_bwd_swiglu_workspace_bytes(cfg, &need);
  if (v != TTT_OK) return v;
  const ttt_cfg& g = *cfg;
  const Sizes s = tensor_sizes(g);
  const void* in[11] = {Q, K, V, lr, W0_1, W0_2, W0_3, dO, dWf_1, dWf_2, dWf_3};
  void* out[7] = {dQ, dK, dV, dlr, dW0_1, dW0_2, dW0_3};
  for (const void* p : in)
    if (!p || !aligned16(p)) return TTT_ERR_ARG;
  for (const void* p : out)
    if (!p || !aligned16(p)) return TTT_ERR_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return TTT_ERR_WORKSPACE;
  // outputs may not overlap the inputs, the workspace or each other
  const size_t in_n[11] = {s.tok_bytes,    s.tok_bytes,    s.tok_bytes, s.lr_bytes,     s.w0_bytes[0], s.w0_bytes[1],
                           s.w0_bytes[2], s.tok_bytes,    s.wf_bytes[0], s.wf_bytes[1], s.wf_bytes[2]};
  const size_t out_n[7] = {s.tok_bytes, s.tok_bytes, s.tok_bytes, s.lr_bytes, s.w0_bytes[0], s.w0_bytes[1],
                           s.w0_bytes[2]};
  for (int i = 0; i < 7; ++i) {
    const Range o{(const char*)out[i], out_n[i]};
    for (int k = 0; k < 11; ++k)
      if (overlap(o, Range{(const char*)in[k], in_n[k]})) return TTT_ERR_ARG;
    if (overlap(o, Range{(const char*)workspace, need})) return TTT_ERR_ARG;
    for (int k = i + 1; k < 7; ++k)
      if (overlap(o, Range{(const char*)out[k], out_n[k]})) return TTT_ERR_ARG;
  }
  const void* ptrs[19] = {Q, K, V, lr, W0_1, W0_2, W0_3, dO, dWf_1, dWf_2, dWf_3,
                          dQ, dK, dV, dlr, dW0_1, dW0_2, dW0_3, workspace};
  v = check_device_ptrs(ptrs, 19);
  if (v != TTT_OK) return v;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return TTT_ERR_CUDA;
  const float* const w0[3] = {W0_1, W0_2, W0_3};
  const float* const dwf[3] = {dWf_1, dWf_2, dWf_3};
  float* const dw0[3] = {dW0_1, dW0_2, dW0_3};
  return bwd_swiglu_run(g, Q, K, V, lr, w0, dO, dwf, dQ, dK, dV, dlr, dw0, static_cast<char*>(workspace), st);
}

const char* ttt_strerror(int status) {
  switch (status) {
    case TTT_OK: return "ok";
    case TTT_ERR_ARG: return "invalid argument (shape, NULL or misaligned pointer, or overlapping buffers)";
    case TTT_ERR_UNSUPPORTED: return "configuration not covered by the selected kernel family";
    case TTT_ERR_WORKSPACE: return "workspace NULL, misaligned or smaller than ttt_workspace_bytes()";
    case TTT_ERR_CUDA: return "a CUDA runtime call failed";
    case TTT_ERR_TIMEOUT: return "a device-side wait exceeded timeout_us";
    case TTT_ERR_NONFINITE: return "an input holds NaN or Inf";
    case TTT_ERR_DEVICE: return "a device-side consistency check failed";
    case TTT_ERR_SCRATCH_LIMIT: return "request needs more scratch than TTT_STATIC_SCRATCH_BYTES";
    default: return "unknown status";
  }
}

}  // extern "C"
