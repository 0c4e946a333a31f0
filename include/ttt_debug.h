/*
 * ttt_debug.h - test hooks of the B300 TTT-layer library.
 *
 * These entry points expose single building blocks of the bf16 tensor-core
 * path so that tests can check them in isolation. They are not part of the
 * layer's API and no page defines them.
 */
#ifndef TTT_B300_DEBUG_H
#define TTT_B300_DEBUG_H

#include "ttt.h"

#ifdef __cplusplus
extern "C" {
#endif

/* D[z] = A[z] * B[z]^T for z < Z on the same warp-specialised tcgen05/TMEM/TMA
 * tile kernel the layer's GEMM phases use (bf16 operands, fp32 accumulation).
 *   A  bf16, DEVICE: [Z, M, K] when a_mn_major == 0 (K-major), else [Z, K, M]
 *   B  bf16, DEVICE: [Z, N, K] when b_mn_major == 0 (K-major), else [Z, K, N]
 *   D  fp32, DEVICE: [Z, M, N], written
 * M, N, K must be positive multiples of 64; pointers 16-byte aligned.
 * Enqueued on `stream`; returns TTT_OK, TTT_ERR_ARG or TTT_ERR_CUDA. */
TTT_API int ttt_dbg_gemm_bf16(const void* A, int a_mn_major, const void* B, int b_mn_major, float* D,
                              int Z, int M, int N, int K, void* stream);

/* CTAs of the fused Muon kernel's cooperative grid for *cfg on the current
 * device; *resident (may be NULL) receives how many of its CTAs fit at once.
 * Returns TTT_OK, TTT_ERR_ARG (cfg not on the tensor-core path) or TTT_ERR_CUDA. */
TTT_API int ttt_dbg_ns_plan(const ttt_cfg* cfg, int* grid, int* resident);

/* In TTT_PREC_SPLIT precision, which stages of the weight-update path carry
 * split (bf16 hi + lo) operands: bit 0 the keys' forward (W = hi + lo), bit 1
 * the gradient (E = hi + lo), bit 2 Newton-Schulz; a cleared bit gives that
 * stage single operands. Default 7 (all). Process-global, for precision
 * studies and tests. Returns TTT_OK or TTT_ERR_ARG. */
TTT_API int ttt_dbg_split_mask(int mask);

/* Caps the fused Muon kernel's grid at `ctas` CTAs (0 = one per SM, the
 * default) for every later launch in this process. For tuning sweeps and tests.
 * Returns TTT_OK or TTT_ERR_ARG. */
TTT_API int ttt_dbg_ns_force_grid(int ctas);

/* Whether the fused Muon kernel computes the symmetric d x d products
 * (R = X X^T + beta I and P = c R^2 + alpha I) on the tiles that meet the upper
 * triangle only, writing the missing lower blocks as transposes: 1 always,
 * 0 never, -1 (default) when an iteration has more than four tiles per SM.
 * Process-global, for comparisons and tests. Returns TTT_OK. */
TTT_API int ttt_dbg_ns_symmetric(int on);

/* Column-tile widths of the fused Muon kernel's d x d products (bns) and of its
 * X updates (bnx): 128 or 256, each dividing d (bns, or d <= bns) and dh (bnx);
 * 0 = chosen by the shape (the default). Process-global, for tuning sweeps and
 * tests. Returns TTT_OK or TTT_ERR_ARG. */
TTT_API int ttt_dbg_ns_tiles(int bns, int bnx);

/* Phase timeline of the fused Muon kernel. With tracing on, every later launch
 * records %globaltimer stamps (ns) into a device table: slot 0 the start,
 * slot 1 the last CTA's exit, and for phase i of the item list (0 norm1,
 * 1 norm2, 2 + 3 it + k the Gram / polynomial / X update of iteration it, then
 * the weight norm) slot 2 + 2i the earliest start and slot 3 + 2i the latest
 * finish of one of its items. A traced launch synchronises its stream first.
 * read copies the first n (<= 96) slots of the last traced launch to HOST
 * memory `out`. Return TTT_OK, TTT_ERR_ARG or TTT_ERR_CUDA. */
TTT_API int ttt_dbg_ns_trace(int on);
TTT_API int ttt_dbg_ns_trace_read(unsigned long long* out, int n);

/* Failure-detection test: the next launch of the linear small-chunk kernel
 * issues none of its loads, so its first wait (bounded by cfg->timeout_us)
 * runs out; the kernel records TTT_ERR_TIMEOUT in the status word and returns
 * with nothing in flight. Later launches are unaffected. */
TTT_API void ttt_dbg_stall_next_linear(void);

/* Failure-detection test: the next launch of the tensor-core forward (the
 * first kernel of a chunk) issues none of its TMA loads, so its MMA warps' first
 * wait runs out after cfg->timeout_us; the kernel records TTT_ERR_TIMEOUT and
 * every CTA returns with nothing in flight. The call's later kernels see the
 * status word and stop early or run on stale workspace data; the next call
 * starts from W0 again and is unaffected. */
TTT_API void ttt_dbg_stall_next_fwd(void);

/* Whether the chunk gradient runs on CTA pairs (1, the default; cta_group::2
 * MMAs of 256 x 256, each CTA holding half of E's columns) or on clusters of
 * one-CTA tiles that share E by multicast (0). Only the single-GPU build has
 * the pair kernel; the other build ignores the setting. Process-global, for
 * tests and tuning. Returns TTT_OK or TTT_ERR_ARG. */
TTT_API int ttt_dbg_grad_pairs(int on);

/* Failure-detection test: in the next launch of the fused Muon kernel CTA 0
 * never signals the completion of its first item, so the items of that
 * matrix's next phase wait until their bounded waits run out; TTT_ERR_TIMEOUT
 * is recorded, every CTA skips the remaining work, drains what it has in
 * flight, frees its TMEM and returns. Later launches are unaffected. */
TTT_API void ttt_dbg_stall_next_ns(void);

/* ---- launch accounting and per-kernel timing ------------------------------
 * Every kernel launch of the library is counted by class. With timing on, each
 * launch is bracketed by CUDA events recorded on its own stream (a few
 * microseconds of overhead per launch); the times resolve when read. */
enum {
  TTT_KERNEL_FWD = 0,     /* fused [A|B] = X[W1;W3]^T, Dm = V W2, SwiGLU (backward) epilogue */
  TTT_KERNEL_APPLY = 1,   /* O = H_q W2^T                                                   */
  TTT_KERNEL_GRAD = 2,    /* chunk gradients G1^T, G2, G3^T (+ split-K reduction)            */
  TTT_KERNEL_GRAM = 3,    /* Newton-Schulz R = X X^T + beta I  \  phases of TTT_KERNEL_NS;   */
  TTT_KERNEL_POLY = 4,    /* Newton-Schulz P = c R^2 + alpha I  > no launch of their own:    */
  TTT_KERNEL_XUPD = 5,    /* Newton-Schulz X <- P X            /  classes of the FLOP split   */
  TTT_KERNEL_UPDATE = 6,  /* W <- W - step U, row weight norm, shadows                        */
  TTT_KERNEL_AUX = 7,     /* import/export of the weights, normalisation, finiteness scan     */
  TTT_KERNEL_LINEAR = 8,  /* linear small-chunk persistent kernel                            */
  TTT_KERNEL_SIMT = 9,    /* fp32 SIMT layer kernel                                          */
  TTT_KERNEL_NS = 10,     /* fused Muon step: normalise, 5 Newton-Schulz iterations, update,
                             row weight norm (one dataflow launch over every matrix)        */
  TTT_KERNEL_COUNT = 11
};

TTT_API void ttt_prof_enable(int on);
/* Drops recorded timings and zeroes the launch counters. */
TTT_API void ttt_prof_reset(void);
/* Totals of one kernel class since the last reset: summed event time (ms), how
 * many launches were timed, how many were launched. Waits for the recorded
 * events. Returns TTT_OK or TTT_ERR_ARG. */
TTT_API int ttt_prof_read(int kind, double* total_ms, long long* timed_launches, long long* launches);
/* Kernel launches of every class since the last reset. */
TTT_API long long ttt_launch_count(void);
TTT_API const char* ttt_kernel_name(int kind);

#ifdef __cplusplus
}
#endif
#endif /* TTT_B300_DEBUG_H */
