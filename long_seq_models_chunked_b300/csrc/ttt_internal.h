// Internal interface between the C-ABI front end and the kernel families.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ttt.h"
#include "../../include/ttt_debug.h"

namespace ttt {

// A validated ttt_fwd request (host side).
struct Call {
  ttt_cfg cfg;
  int n_chunks;
  int nw;                       // fast-weight matrices: 3 (SwiGLU) or 1 (linear)
  int rows[3], cols[3];         // out x in of each matrix
  const void *Q, *K, *V;
  const float* lr;
  const float* W0[3];
  void* O;
  float* Wf[3];
  char* ws;                     // workspace base (status word at offset 0)
  size_t ws_bytes;
  cudaStream_t stream;
  bool mask_all;                // every chunk updates
  const uint8_t* mask;          // host flags (may be NULL when mask_all)
  // host-buffer pipelining (tensor-core family): the stream waits for
  // chunk_ready[c] before chunk c reads its inputs and records chunk_done[c]
  // once chunk c's outputs are written (both NULL: no per-chunk events)
  const cudaEvent_t* chunk_ready;
  const cudaEvent_t* chunk_done;
};

inline bool call_updates(const Call& c, int chunk) {
  return c.mask_all || c.mask[chunk] != 0;
}

// ---- SIMT fp32 family (any shape, one CTA per head) -----------------------
size_t simt_workspace_bytes(const ttt_cfg& cfg);
int simt_run(const Call& c);

// ---- tensor-core bf16 family (tcgen05 / TMEM / TMA) ------------------------
bool tc_supported(const ttt_cfg& cfg);
size_t tc_workspace_bytes(const ttt_cfg& cfg);
int tc_run(const Call& c);

// ---- linear small-chunk family (persistent, W resident on chip) ------------
bool linear_supported(const ttt_cfg& cfg);
size_t linear_workspace_bytes(const ttt_cfg& cfg);
int linear_run(const Call& c);

// ---- outer-loop backward (linear net, plain steps, shifted mode) -----------
bool bwd_supported(const ttt_cfg& cfg);
size_t bwd_workspace_bytes(const ttt_cfg& cfg);
int bwd_run(const ttt_cfg& g, const void* Q, const void* K, const void* V, const float* lr, const float* W0,
            const void* dO, const float* dWf, void* dQ, void* dK, void* dV, float* dlr, float* dW0, char* ws,
            cudaStream_t st);
bool bwd_swiglu_supported(const ttt_cfg& cfg);
size_t bwd_swiglu_workspace_bytes(const ttt_cfg& cfg);
int bwd_swiglu_run(const ttt_cfg& g, const void* Q, const void* K, const void* V, const float* lr,
                   const float* const W0[3], const void* dO, const float* const dWf[3], void* dQ, void* dK, void* dV,
                   float* dlr, float* const dW0[3], char* ws, cudaStream_t st);

// ---- misc ------------------------------------------------------------------
// TTT_OK or TTT_ERR_ARG: field ranges and sizes of *cfg (host only).
int validate_cfg(const ttt_cfg* cfg);
int launch_check_finite(const Call& c);
// TTT_OK when every non-NULL pointer is device memory of the current device,
// else TTT_ERR_ARG (TTT_ERR_CUDA if the current device cannot be queried).
int check_device_ptrs(const void* const* ptrs, int n);

// Launch accounting (and optional event timing) around every kernel launch.
void prof_before(int kind, cudaStream_t st);
void prof_after(int kind, cudaStream_t st);

}  // namespace ttt
