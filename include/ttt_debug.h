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

#ifdef __cplusplus
}
#endif
#endif /* TTT_B300_DEBUG_H */
