/*
 * ttt.h - C ABI of the B300 (sm_103a) chunked test-time-training layer.
 *
 * The layer (LaCT page, "Large Chunk Test-Time Training", §2.1): per (batch,
 * head) a fast-weight net f_W is applied to each chunk's queries (apply phase,
 * the page's eq. 2) and updated from the gradient of a self-supervised inner
 * loss, summed over the chunk's tokens with per-token learning rates (update
 * phase, eq. 4-5). The update optionally goes through Muon's Newton-Schulz
 * orthogonalisation (§2.2.1, eq. 9-10) and an L2 row weight norm (§2.2.1,
 * eq. 8). Shifted mode applies chunk i with the weights left by chunks
 * 0..i-1 (§3.2, shifted block-causal mask); single mode updates on a chunk and
 * then applies to the same chunk (§3.1: one chunk = the whole image set).
 *
 *   fast nets: SwiGLU   f(x) = W2 (silu(W1 x) * (W3 x)),  W1,W3: [dh, d], W2: [d, dh]
 *              linear   f(x) = W x,                       W: [d, d]
 *   losses:    inner product  l = -f(k).v ;  MSE  l = 1/2 ||f(k) - v||^2
 *   update:    G = sum_t lr_t grad_W l_t ;  U = NS5(G) or G ;  W <- W - step * U ;
 *              (weight norm) W[r,:] <- W[r,:] * n0[r] / max(||W[r,:]||, wnorm_eps),
 *              n0 = the row norms of W0.
 *
 * Every call runs on the GPU. There is no CPU fallback: a build without the
 * device code cannot be loaded.
 */
#ifndef TTT_B300_H
#define TTT_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TTT_API __attribute__((visibility("default")))
#else
#define TTT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (0 = success, negative = error) ---------------------- */
#define TTT_OK               0
#define TTT_ERR_ARG         -1  /* bad shape, NULL or misaligned pointer, aliasing */
#define TTT_ERR_UNSUPPORTED -2  /* valid request that no built kernel covers       */
#define TTT_ERR_WORKSPACE   -3  /* workspace NULL, too small or misaligned         */
#define TTT_ERR_CUDA        -4  /* a CUDA runtime call failed                      */
#define TTT_ERR_TIMEOUT     -5  /* a device-side wait gave up (timeout_us)         */
#define TTT_ERR_NONFINITE   -6  /* check_finite found a NaN/Inf in the inputs      */
#define TTT_ERR_DEVICE      -7  /* a device-side consistency check failed          */
#define TTT_ERR_SCRATCH_LIMIT -8 /* request needs more than the static scratch array */

/* ---- enumerations -------------------------------------------------------- */
enum { TTT_NET_SWIGLU = 0, TTT_NET_LINEAR = 1 };
enum { TTT_LOSS_IP = 0, TTT_LOSS_MSE = 1 };
/* SHIFTED: chunk c is applied with the weights left by chunks 0..c-1, then
 *          updates (LaCT page §3.2);
 * SINGLE: every chunk updates, then applies to its own queries (§3.1);
 * INCLUSIVE: query t of a chunk sees the chunk's starting weights minus step
 *          times the gradients of the chunk's tokens up to and including t
 *          (each taken at the starting weights); the chunk then updates with
 *          all of them. With chunks of one token this is the per-token order
 *          of the TTT tutorial page (§3: update with x_t, then output with the
 *          updated weights). Plain gradient steps only: muon = wnorm = 0 and
 *          momentum = 0, else TTT_ERR_ARG. */
enum { TTT_MODE_SHIFTED = 0, TTT_MODE_SINGLE = 1, TTT_MODE_INCLUSIVE = 2 };
enum { TTT_DTYPE_F32 = 0, TTT_DTYPE_BF16 = 1 };
/* kernel family: AUTO picks the fastest one that covers the request */
enum { TTT_IMPL_AUTO = 0, TTT_IMPL_SIMT = 1, TTT_IMPL_TC = 2, TTT_IMPL_LINEAR = 3 };
/* operand precision of the tensor-core family on the weight-update path
 * (the forward of the keys, the gradient, Newton-Schulz):
 *   SPLIT  every operand computed inside the layer is carried as a bf16 pair
 *          (hi + lo) and every product takes the two or three bf16 MMAs that
 *          keep ~16 significant bits; the fast weights, whose updates feed back
 *          chunk after chunk, stay within the bf16 tier's tolerance of an exact
 *          computation over long sequences of updates (default);
 *   SINGLE one bf16 (fp16 inside Newton-Schulz) operand per product: fewer MMAs
 *          and half the traffic of the intermediate operands, but the rounding is
 *          amplified from chunk to chunk (about 1.3x per update on a 512 x 1024
 *          Muon layer), so it suits few updates, such as single-chunk mode. */
enum { TTT_PREC_SPLIT = 0, TTT_PREC_SINGLE = 1 };

/* Layer configuration. Fill it with ttt_cfg_default() and override fields. */
typedef struct ttt_cfg {
  int32_t B, H, T;        /* batch, heads, tokens per sequence; each >= 1 (an empty
                             sequence is TTT_ERR_ARG: there is nothing to apply) */
  int32_t d;              /* head dim (input and output width of f)             */
  int32_t dh;             /* SwiGLU hidden width (ignored for the linear net)    */
  int32_t chunk;          /* tokens per chunk; the last chunk may be shorter     */
  int32_t fast_net;       /* TTT_NET_*                                            */
  int32_t loss;           /* TTT_LOSS_*                                           */
  int32_t mode;           /* TTT_MODE_*                                           */
  int32_t dtype;          /* storage type of Q, K, V, O: TTT_DTYPE_*              */
  int32_t muon;           /* 1: Newton-Schulz orthogonalisation of each G         */
  int32_t ns_iters;       /* Newton-Schulz iterations (5)                         */
  float   ns_a, ns_b, ns_c; /* quintic coefficients (3.4445, -4.7750, 2.0315)     */
  float   ns_eps;         /* X0 = G / (||G||_F + ns_eps)  (1e-7)                  */
  int32_t wnorm;          /* 1: restore the row norms of W0 after every update    */
  float   wnorm_eps;      /* floor of the row norm in the rescale (1e-12)         */
  float   step;           /* W <- W - step * U  (1.0)                             */
  const uint8_t* update_mask; /* HOST array of n_chunks flags; NULL = every chunk
                             updates. Read during the ttt_fwd call only.        */
  int32_t w0_per_batch;   /* 0: W0 is [H, out, in] shared over B; 1: [B, H, out, in] */
  int32_t check_finite;   /* 1: scan the inputs first; NaN/Inf -> TTT_ERR_NONFINITE */
  uint32_t timeout_us;    /* limit of every device-side wait (default 2,000,000)  */
  int32_t impl;           /* TTT_IMPL_*                                           */
  int32_t precision;      /* TTT_PREC_* (tensor-core family only)                 */
  float   momentum;       /* mu of the momentum buffer B_j of each matrix (LaCT page
                             §2.2.1 compares Muon with a momentum optimiser):
                             B_j <- mu B_j + G_j at every update (B_j starts at 0),
                             then U_j = NS5(B_j) with Muon, or U_j = B_j without.
                             0 (default) = no buffer, U_j from G_j alone        */
  int32_t lr_per_matrix;  /* 0: lr is [B, H, T], one rate per token for every matrix;
                             1: lr is [B, H, T, n_w], one rate per token and matrix
                             (n_w = 3 for SwiGLU, in the order W1, W2, W3; 1 for
                             the linear net): G_j = sum_t lr[t, j] grad_Wj l_t   */
} ttt_cfg;

/* Fills *cfg with the defaults above (B = H = T = d = dh = chunk = 0, SwiGLU,
 * inner-product loss, shifted mode, bf16, Muon with 5 iterations, weight norm
 * on, step 1, AUTO, SPLIT precision, no momentum, one rate per token). */
TTT_API void ttt_cfg_default(ttt_cfg* cfg);

/* Bytes of device workspace ttt_fwd needs for *cfg (and the path AUTO picks).
 * Returns TTT_OK, TTT_ERR_ARG or TTT_ERR_UNSUPPORTED. */
TTT_API int ttt_workspace_bytes(const ttt_cfg* cfg, size_t* bytes);

/* The layer forward (LaCT page §2.1: apply + update over all chunks).
 *
 * All tensor pointers are DEVICE pointers, 16-byte aligned, row-major,
 * contiguous, owned by the caller:
 *   Q, K, V   [B, H, T, d]     fp32 or bf16 (cfg->dtype); read only
 *   lr        [B, H, T]        fp32 per-token learning rate ([B, H, T, n_w] with
 *                              lr_per_matrix); read only
 *   W0_1..3   SwiGLU: W1 [H, dh, d], W2 [H, d, dh], W3 [H, dh, d] fp32
 *             (each with a leading B when w0_per_batch); linear: W0_1 = W [H, d, d],
 *             W0_2 = W0_3 = NULL; read only
 *   O         [B, H, T, d]     cfg->dtype; written
 *   Wf_1..3   final fast weights [B, H, out, in] fp32; written (Wf_2, Wf_3 NULL for linear)
 *   workspace device scratch of >= ttt_workspace_bytes() bytes, 256-byte aligned;
 *             its first 256 bytes hold the device status word
 *   stream    a cudaStream_t (NULL = the legacy default stream)
 * Outputs must not overlap inputs or the workspace. Every tensor pointer and
 * the workspace must be device memory (cudaMalloc or a pool on top of it) of
 * the calling thread's current device: host, managed or another device's
 * memory is TTT_ERR_ARG, detected before any launch.
 *
 * The work is enqueued on `stream`; the call returns without waiting. Host-
 * detectable errors (TTT_ERR_ARG, _UNSUPPORTED, _WORKSPACE) return before any
 * launch. Device-side errors (TTT_ERR_TIMEOUT, _NONFINITE, _DEVICE) are
 * recorded in the workspace status word: read them with ttt_status(). */
TTT_API int ttt_fwd(const ttt_cfg* cfg,
            const void* Q, const void* K, const void* V, const float* lr,
            const float* W0_1, const float* W0_2, const float* W0_3,
            void* O, float* Wf_1, float* Wf_2, float* Wf_3,
            void* workspace, size_t workspace_bytes, void* stream);

/* Waits for `stream`, then returns the status word of the most recent
 * ttt_fwd on this workspace (every ttt_fwd clears it when it starts): TTT_OK,
 * a device-side error code, or TTT_ERR_CUDA if the stream reports an error. */
TTT_API int ttt_status(void* workspace, void* stream);

/* Bytes of one DEVICE arena that ttt_fwd_host needs: room for the inputs,
 * the outputs and the workspace, each 256-byte aligned. */
TTT_API int ttt_host_arena_bytes(const ttt_cfg* cfg, size_t* bytes);

/* The layer on HOST buffers (same shapes and types as ttt_fwd; pinned host
 * memory gives full copy bandwidth). Copies the inputs into `arena` (device,
 * >= ttt_host_arena_bytes(), caller-owned), runs ttt_fwd on `stream`, copies O
 * and the final weights back, waits for the stream and returns the status
 * (ttt_status folded in). */
TTT_API int ttt_fwd_host(const ttt_cfg* cfg,
                 const void* Q, const void* K, const void* V, const float* lr,
                 const float* W0_1, const float* W0_2, const float* W0_3,
                 void* O, float* Wf_1, float* Wf_2, float* Wf_3,
                 void* arena, size_t arena_bytes, void* stream);

/* ---- allocation-free variant ----------------------------------------------
 * The pages define no such call; it serves callers that are given their input
 * and output buffers but may not allocate device memory: a plugin running
 * inside a host application that keeps all device memory in its own pool, or a
 * latency-bound loop in which cudaMalloc/cudaFree (which can synchronise the
 * whole device) are not allowed. Such callers cannot provide the workspace
 * that ttt_fwd takes.
 *
 * ttt_fwd_static_scratch runs the fp32 SIMT kernel family (every
 * configuration; cfg->impl must be TTT_IMPL_AUTO or TTT_IMPL_SIMT) with its
 * scratch in one array of TTT_STATIC_SCRATCH_BYTES that the library holds in
 * device memory, on every GPU that loads the library, until the process exits.
 * Arguments are those of ttt_fwd without the workspace; `status` is an
 * optional DEVICE int (NULL = not wanted, 4-byte aligned, overlapping no
 * input or output) that receives the device-side status word (TTT_OK,
 * TTT_ERR_NONFINITE, ...) once the layer has run on `stream`.
 *
 * - The call allocates nothing: no cudaMalloc, cudaFree or allocating library
 *   routine. It runs on the calling thread's current device.
 * - Every call looks up the array's device address (cudaGetSymbolAddress,
 *   which allocates nothing) with the calling thread's device current. The
 *   first lookup on a device loads the library's device code there; make that
 *   first call before any stream capture.
 * - A request whose scratch (ttt_workspace_bytes with impl = SIMT) exceeds
 *   TTT_STATIC_SCRATCH_BYTES returns TTT_ERR_SCRATCH_LIMIT before any launch.
 * - Every call uses the same array, which keeps the previous call's contents
 *   (the call clears what has to start at zero). Calls that overlap on the GPU
 *   (other streams, other host threads) race on it: serialise them.
 * Returns TTT_OK or a host-detected error, as ttt_fwd does. */
#define TTT_STATIC_SCRATCH_BYTES (16u << 20)
TTT_API int ttt_fwd_static_scratch(const ttt_cfg* cfg,
            const void* Q, const void* K, const void* V, const float* lr,
            const float* W0_1, const float* W0_2, const float* W0_3,
            void* O, float* Wf_1, float* Wf_2, float* Wf_3,
            int* status, void* stream);

/* ---- outer-loop backward ---------------------------------------------------
 * Gradients of a scalar loss L through the layer (the outer loop that trains
 * the model around it differentiates through the inner updates: TTT-E2E news
 * page §2.2), for the linear fast net with plain gradient steps (muon = wnorm =
 * 0, momentum = 0) in shifted mode, inner-product or MSE loss: given
 * dO = dL/dO ([B, H, T, d], cfg->dtype) and dWf = dL/dW_final ([B, H, d, d]
 * fp32), writes dQ, dK, dV ([B, H, T, d], cfg->dtype), dlr ([B, H, T] fp32)
 * and dW0 (fp32, W0's layout: summed over the batch unless w0_per_batch).
 * Other configurations return TTT_ERR_UNSUPPORTED. Pointers, alignment,
 * device memory, workspace (>= ttt_bwd_workspace_bytes, 256-byte aligned) and
 * errors as for ttt_fwd; outputs overlap nothing. Enqueued on `stream`. */
TTT_API int ttt_bwd_workspace_bytes(const ttt_cfg* cfg, size_t* bytes);
TTT_API int ttt_bwd(const ttt_cfg* cfg, const void* Q, const void* K, const void* V, const float* lr,
                    const float* W0, const void* dO, const float* dWf, void* dQ, void* dK, void* dV,
                    float* dlr, float* dW0, void* workspace, size_t workspace_bytes, void* stream);

/* The same for the SwiGLU fast net with plain gradient steps (muon = wnorm = 0,
 * momentum = 0, one rate per token: lr_per_matrix = 0) in shifted mode,
 * inner-product or MSE loss: W0_j, dWf_j and dW0_j as the three matrices of
 * ttt_fwd (W1 [dh, d], W2 [d, dh], W3 [dh, d] per head; W0 and dW0 shared over
 * the batch unless w0_per_batch, dWf per (batch, head)). The second-order terms
 * of the inner updates (the derivative of each token's gradient along the
 * adjoint of the weights it updates) come out exactly. Other configurations
 * return TTT_ERR_UNSUPPORTED. Checks and errors as for ttt_bwd. */
TTT_API int ttt_bwd_swiglu_workspace_bytes(const ttt_cfg* cfg, size_t* bytes);
TTT_API int ttt_bwd_swiglu(const ttt_cfg* cfg, const void* Q, const void* K, const void* V, const float* lr,
                           const float* W0_1, const float* W0_2, const float* W0_3, const void* dO,
                           const float* dWf_1, const float* dWf_2, const float* dWf_3, void* dQ, void* dK,
                           void* dV, float* dlr, float* dW0_1, float* dW0_2, float* dW0_3, void* workspace,
                           size_t workspace_bytes, void* stream);

/* ---- context parallelism (LaCT page §2.2.2) -------------------------------
 * The tokens of one chunk are split into shards held by different GPUs (or
 * handled by different calls). Every shard computes its partial gradient with
 * the same fast weights; the caller sums the partials over the shards (an
 * all-reduce: the one exchange of the method); every shard then applies the
 * same update to its copy of the weights, and its own queries. These calls
 * run those steps one at a time on a state kept in the caller's workspace.
 * They cover the tensor-core family (bf16 SwiGLU, inner-product loss).
 *
 * cfg: B, H, d, dh and the update hyper-parameters as for ttt_fwd; cfg->chunk
 *      = the largest token count of one ttt_cp_grad / ttt_cp_apply call;
 *      cfg->T >= 1, cfg->mode and cfg->update_mask are not used (the caller
 *      orders apply, gradient and update).
 * Tokens: Q, K, V [B, H, T_all, d] bf16 and lr [B, H, T_all(, 3)] fp32 as for
 *      ttt_fwd, of which the call uses tokens [start, start + n) of every
 *      (b, h); O has Q's layout and gets those tokens written.
 * G:   per (b, h), the gradients of W1, W2, W3 as [B * H][3][d][dh] fp32, W1
 *      and W3 transposed (d x dh), W2 as is: the partial of one shard from
 *      ttt_cp_grad, the sum over the shards for ttt_cp_update.
 * All pointers are device memory of the current device, 16-byte aligned; the
 * workspace (>= ttt_cp_workspace_bytes, 256-byte aligned) holds the state from
 * ttt_cp_begin to ttt_cp_end and the status word (read it with ttt_status).
 * Work is enqueued on `stream`. Each call returns TTT_OK or a host-detected
 * error (TTT_ERR_ARG, _UNSUPPORTED, _WORKSPACE, _CUDA) before any launch. */
TTT_API int ttt_cp_workspace_bytes(const ttt_cfg* cfg, size_t* bytes);
/* Loads W0 (layouts of ttt_fwd) into the state; clears the status word. */
TTT_API int ttt_cp_begin(const ttt_cfg* cfg, const float* W0_1, const float* W0_2, const float* W0_3,
                         void* workspace, size_t workspace_bytes, void* stream);
/* The partial gradient of tokens [start, start + n) with the current weights. */
TTT_API int ttt_cp_grad(const ttt_cfg* cfg, const void* K, const void* V, const float* lr, int T_all,
                        int start, int n, float* G, void* workspace, size_t workspace_bytes, void* stream);
/* One update (momentum, Muon, step, weight norm) from the summed gradient. */
TTT_API int ttt_cp_update(const ttt_cfg* cfg, const float* G, void* workspace, size_t workspace_bytes,
                          void* stream);
/* O of tokens [start, start + n) with the current weights. */
TTT_API int ttt_cp_apply(const ttt_cfg* cfg, const void* Q, int T_all, int start, int n, void* O,
                         void* workspace, size_t workspace_bytes, void* stream);
/* Writes the current weights to Wf_1..3 ([B, H, out, in] fp32, as ttt_fwd). */
TTT_API int ttt_cp_end(const ttt_cfg* cfg, float* Wf_1, float* Wf_2, float* Wf_3, void* workspace,
                       size_t workspace_bytes, void* stream);

/* Which kernel family AUTO (or cfg->impl) resolves to for *cfg: TTT_IMPL_*,
 * or a negative status if none covers it. */
TTT_API int ttt_select_impl(const ttt_cfg* cfg);

/* Static description of a status code. */
TTT_API const char* ttt_strerror(int status);

/* Host-thread resources. In shifted mode the tensor-core path runs each
 * chunk's apply on a side stream beside that chunk's gradient (ordered by two
 * events after the forward and before the next weight update); the library
 * creates that stream and its events once per host thread and device, on the
 * thread's first such call, and keeps them for its later calls.
 * ttt_thread_release() waits for and destroys the calling thread's (every
 * device it used). Call it before a host thread that used the library exits
 * when the process outlives the thread; later calls create them again.
 * Returns TTT_OK (also when there is nothing to release) or TTT_ERR_CUDA. */
TTT_API int ttt_thread_release(void);

/* Build features, as bit flags.
 * TTT_FEATURE_CLUSTER_MULTICAST: the tensor-core kernels share operand tiles
 * across the CTAs of a thread-block cluster with TMA multicast loads (and
 * signal each other's barriers with multicast commits). Every such load reads
 * this GPU's own memory (ttt_fwd rejects pointers that are not), but this build
 * is meant for processes that use one GPU alone. The library built without it
 * (libttt_b300_local.so: clusters of one CTA, no multicast and no CTA pairs
 * anywhere) is the one a process that runs beside ranks on other GPUs loads. */
#define TTT_FEATURE_CLUSTER_MULTICAST 1
TTT_API int ttt_build_features(void);

/* ABI version (incremented on any incompatible change of this header). */
TTT_API int ttt_abi_version(void);

/* sizeof(ttt_cfg) as compiled into the library (lets bindings check layout). */
TTT_API size_t ttt_cfg_size(void);

#ifdef __cplusplus
}
#endif
#endif /* TTT_B300_H */
