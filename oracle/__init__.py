"""Independent fp64 CPU oracle of the chunked TTT fast-weight layer.

Test infrastructure only: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it; the product path never does.
It shares no code with the CUDA path.

Parity status of each function (what pins it is in tests/test_oracle_pins.py):
  swiglu_apply, linear_apply  - pinned (torch fp64 library forward; zero-update case)
  swiglu_grad, linear_grad    - pinned (central finite differences; torch autograd;
                                per-token sum)
  newton_schulz               - pinned (closed form through the SVD)
  weight_norm                 - pinned (row-norm and direction invariants)
  update (momentum buffer)    - pinned (geometric-series closed form of the linear
                                momentum optimiser; the buffer, not the gradient,
                                feeds Newton-Schulz)
  chunk_grad (rates [n, 3])   - pinned (brute-force weighted sum of per-token
                                gradients; equal columns = the shared rate; a zero
                                column leaves its matrix unchanged)
  ttt_head / ttt_layer        - pinned in the special cases with closed forms
                                (delta rule, block-shifted linear attention,
                                a chunk of orthonormal keys memorised under MSE,
                                single-chunk linear attention, zero update) and by
                                invariants (causality, resume, permutation);
                                the full SwiGLU + Muon + weight-norm chain (no page
                                prints values for it) by its equivariance under input
                                rotations, output sign-permutations and hidden-unit
                                permutations, with momentum and a mask, and by the
                                closed form of a one-token Muon step (the unit
                                rank-one gradient times the quintic iterated from 1).
  apply_inclusive (inclusive  - pinned (chunk-1 linear MSE = the delta rule read after
  order)                        the update; linear inner product = causal linear
                                attention for every chunk size; chunk-1 SwiGLU = the
                                per-token recurrence; the SwiGLU matrix dual form)
  linear_head_backward        - pinned (central finite differences of the forward
                                oracle, every input, inner product and MSE, masks and
                                ragged chunks)
  swiglu_head_backward        - pinned (central finite differences of the forward
                                oracle ttt_head, every input, inner product and MSE,
                                masks and ragged chunks)
"""
from .ttt_oracle import (OracleCfg, apply_inclusive, chunk_grad, linear_apply,  # noqa: F401
                         linear_grad, linear_head_backward, newton_schulz, row_norms, sigmoid,
                         swiglu_apply, swiglu_grad, swiglu_head_backward, ttt_head, ttt_layer,
                         update, weight_norm)
