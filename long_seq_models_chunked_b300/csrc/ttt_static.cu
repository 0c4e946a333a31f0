// Allocation-free entry point: the fp32 SIMT layer with its scratch memory in
// a file-scope device array instead of a caller-provided workspace.
//
// Who needs it: code that is handed its input and output buffers but may not
// allocate device memory itself - a plugin running inside a host application
// that reserves all device memory for its own pool, or a latency-bound loop in
// which cudaMalloc/cudaFree (which can synchronise the whole device) are not
// allowed. Such a caller cannot size and own the workspace ttt_fwd expects.
//
// The array is TTT_STATIC_SCRATCH_BYTES large and lives on every device that
// loads the library, until the process exits. Every call shares it.
#include "ttt_common.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

// The scratch of every ttt_fwd_static_scratch call: status word in the first
// kStatusBytes, then the SIMT family's per-head slices.
static __device__ __align__(256) unsigned char g_static_scratch[TTT_STATIC_SCRATCH_BYTES];

// Host code may not pass g_static_scratch to a kernel (on the host that name is
// only a stand-in for the device array). Its device address is looked up on
// every call, with the calling thread's device current: the lookup allocates
// nothing, and a stale address can never survive a cudaDeviceReset that
// reloads the module.
int static_scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return TTT_ERR_CUDA;
  *out = p;
  return TTT_OK;
}

bool aligned16_(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || !na || !nb) return false;
  const char* pa = static_cast<const char*>(a);
  const char* pb = static_cast<const char*>(b);
  return pa < pb + nb && pb < pa + na;
}

}  // namespace
}  // namespace ttt

using namespace ttt;

extern "C" int ttt_fwd_static_scratch(const ttt_cfg* cfg, const void* Q, const void* K, const void* V,
                                      const float* lr, const float* W0_1, const float* W0_2, const float* W0_3,
                                      void* O, float* Wf_1, float* Wf_2, float* Wf_3, int* status,
                                      void* stream) {
  const int sel = ttt_select_impl(cfg);  // validates *cfg
  if (sel < 0) return sel;
  const ttt_cfg& g = *cfg;
  if (g.impl != TTT_IMPL_AUTO && g.impl != TTT_IMPL_SIMT) return TTT_ERR_UNSUPPORTED;
  const size_t need = simt_workspace_bytes(g);
  if (need > (size_t)TTT_STATIC_SCRATCH_BYTES) return TTT_ERR_SCRATCH_LIMIT;

  const int nw = g.fast_net == TTT_NET_SWIGLU ? 3 : 1;
  const size_t es = g.dtype == TTT_DTYPE_F32 ? 4 : 2;
  const size_t tok = (size_t)g.B * g.H * g.T;
  const size_t tok_bytes = tok * g.d * es, lr_bytes = tok * sizeof(float) * (g.lr_per_matrix ? nw : 1);
  const size_t wsz = nw == 3 ? (size_t)g.d * g.dh : (size_t)g.d * g.d;
  const size_t w0_bytes = (size_t)(g.w0_per_batch ? g.B : 1) * g.H * wsz * sizeof(float);
  const size_t wf_bytes = (size_t)g.B * g.H * wsz * sizeof(float);
  const void* in[4] = {Q, K, V, lr};
  const size_t in_bytes[4] = {tok_bytes, tok_bytes, tok_bytes, lr_bytes};
  const float* w0[3] = {W0_1, W0_2, W0_3};
  float* wf[3] = {Wf_1, Wf_2, Wf_3};
  for (const void* p : in)
    if (!p || !aligned16_(p)) return TTT_ERR_ARG;
  if (!O || !aligned16_(O)) return TTT_ERR_ARG;
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return TTT_ERR_ARG;
  for (int j = 0; j < nw; ++j)
    if (!w0[j] || !wf[j] || !aligned16_(w0[j]) || !aligned16_(wf[j])) return TTT_ERR_ARG;
  // outputs may not overlap the inputs or each other
  const void* outs[4] = {O, wf[0], nw == 3 ? wf[1] : nullptr, nw == 3 ? wf[2] : nullptr};
  const size_t out_bytes[4] = {tok_bytes, wf_bytes, wf_bytes, wf_bytes};
  for (int i = 0; i < 4; ++i) {
    for (int k = 0; k < 4; ++k)
      if (overlaps(outs[i], out_bytes[i], in[k], in_bytes[k])) return TTT_ERR_ARG;
    for (int j = 0; j < nw; ++j)
      if (overlaps(outs[i], out_bytes[i], w0[j], w0_bytes)) return TTT_ERR_ARG;
    for (int k = i + 1; k < 4; ++k)
      if (overlaps(outs[i], out_bytes[i], outs[k], out_bytes[k])) return TTT_ERR_ARG;
    if (status && overlaps(outs[i], out_bytes[i], status, sizeof(int))) return TTT_ERR_ARG;
  }
  // the status word is written last: it may not overlap an input either
  if (status) {
    for (int k = 0; k < 4; ++k)
      if (overlaps(status, sizeof(int), in[k], in_bytes[k])) return TTT_ERR_ARG;
    for (int j = 0; j < nw; ++j)
      if (overlaps(status, sizeof(int), w0[j], w0_bytes)) return TTT_ERR_ARG;
  }

  {
    const void* ptrs[12] = {Q, K, V, lr, O, status};
    int n = 6;
    for (int j = 0; j < nw; ++j) {
      ptrs[n++] = w0[j];
      ptrs[n++] = wf[j];
    }
    const int v = check_device_ptrs(ptrs, n);
    if (v != TTT_OK) return v;
  }
  void* scratch = nullptr;
  int rc = static_scratch_address(&scratch);
  if (rc != TTT_OK) return rc;

  Call c{};
  c.cfg = g;
  if (c.cfg.timeout_us == 0) c.cfg.timeout_us = 2000000u;
  c.n_chunks = (g.T + g.chunk - 1) / g.chunk;
  c.nw = nw;
  if (nw == 3) {
    c.rows[0] = g.dh; c.cols[0] = g.d;
    c.rows[1] = g.d;  c.cols[1] = g.dh;
    c.rows[2] = g.dh; c.cols[2] = g.d;
  } else {
    c.rows[0] = g.d; c.cols[0] = g.d;
  }
  c.Q = Q; c.K = K; c.V = V; c.lr = lr;
  for (int j = 0; j < 3; ++j) {
    c.W0[j] = j < nw ? w0[j] : nullptr;
    c.Wf[j] = j < nw ? wf[j] : nullptr;
  }
  c.O = O;
  c.ws = static_cast<char*>(scratch);
  c.ws_bytes = TTT_STATIC_SCRATCH_BYTES;
  c.stream = static_cast<cudaStream_t>(stream);
  c.mask = g.update_mask;
  c.mask_all = true;
  if (g.update_mask)
    for (int i = 0; i < c.n_chunks; ++i)
      if (!g.update_mask[i]) { c.mask_all = false; break; }

  // the array keeps the previous call's contents: the status word must start at
  // zero (the SIMT kernel initialises every other byte it reads)
  if (cudaMemsetAsync(scratch, 0, sizeof(int), c.stream) != cudaSuccess) return TTT_ERR_CUDA;
  if (g.check_finite) {
    rc = launch_check_finite(c);
    if (rc != TTT_OK) return rc;
  }
  rc = simt_run(c);
  if (rc != TTT_OK) return rc;
  if (status && cudaMemcpyAsync(status, scratch, sizeof(int), cudaMemcpyDeviceToDevice, c.stream) != cudaSuccess)
    return TTT_ERR_CUDA;
  return TTT_OK;
}
