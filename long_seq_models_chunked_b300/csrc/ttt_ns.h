// Fused Muon step (Newton-Schulz + update + weight norm) of the tensor-core path.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "../../include/ttt.h"
#include "tc_kernel.cuh"

namespace ttt {

struct NsFusedArgs {
  const ttt_cfg* cfg;
  int Z;                 // matrices: 3 per (batch, head)
  bool split;            // SPLIT (bf16 hi/lo operands) or SINGLE (fp16) precision
  float* X;              // [Z][d][dh] fp32: the chunk gradient (read only)
  void* Xh[2];           // operand ping-pong buffers (hi)
  void* Xl[2];           //                          (lo; SPLIT only)
  void* Rh; void* Rl;    // R = X X^T + beta I operand (hi, lo), [Z][d][d] each
  void* Ph; void* Pl;    // P operand (hi, lo)
  float* M;              // [Z][d][dh] fp32 master weights, updated in place
  void* Ms; void* Msl;   // bf16 shadows (hi, lo or nullptr)
  const float* n0;       // [Z][dh] reference row norms
  float* scratch;        // >= ns_fused_scratch_floats() floats (partial sums, barrier)
  float* mom;            // [Z][d][dh] momentum buffers (B <- mu B + G), or nullptr
  float mu;
  // fused normalisation: the gradient kernel wrote Xh[0] / Xl[0] from the
  // UNSCALED gradient (momentum already advanced) and per-z partial sums of
  // squares nsqg[z][nsq_n]; X and mom are then unused. Otherwise the call
  // prepares X0 from X (and mom) itself, with nsqg as scratch of
  // Z * d * (dh / 128) floats.
  bool fused;
  const float* nsqg;
  int nsq_n;
  TcCommon cm;
};

bool ns_fused_supported(const ttt_cfg& g);
size_t ns_fused_scratch_floats(const ttt_cfg& g, int Z);
// CTAs of the fused kernel's cooperative grid (<= 0: it cannot be launched);
// *resident (optional) receives how many CTAs fit on the device at once.
int ns_fused_plan(const ttt_cfg& g, int* resident);
// Test hook: cap the grid at `ctas` CTAs (0 = every SM).
void ns_force_grid(int ctas);
int ns_fused_run(const NsFusedArgs& a, cudaStream_t st);
// Newton-Schulz's input from fp32 gradients: sums `splits` partials
// [splits][Z][d][dh] in order, advances the momentum buffer (mom != NULL:
// B <- mu B + G), writes bf16 (hi, lo) operands (none when Xh is NULL) and the
// sums of squares nsq[(z d + m) (dh / bn) + tile] of bn-wide row tiles.
int ns_input_launch(const float* parts, int splits, int Z, int d, int dh, int bn, float* mom, float mu, void* Xh,
                    void* Xl, float* nsq, cudaStream_t st);

}  // namespace ttt
