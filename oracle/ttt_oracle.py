"""fp64 CPU oracle of the chunked test-time-training (TTT) fast-weight layer.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import or run this module. The product path
(the C-ABI library and its Python binding) never touches it and shares no code
with it.

It is a plain NumPy fp64 restatement of what the layer computes, step by step,
in the order the pages give. Sources:

* LaCT page ("Large Chunk Test-Time Training", peacm.com/news/1205172):
  - §2.1  the large-chunk TTT layer has an update phase (the gradient of the
          whole chunk, summed, updates the fast weights; eq. 4-5) and an apply
          phase (the updated weights process every query; eq. 2);
  - §1.2  "key implementation tricks": the fast-weight net is a SwiGLU MLP and
          the update goes through the Muon optimiser;
  - §2.2.1 weight normalisation (L2 normalisation of the fast weights, eq. 8)
          and Muon (the gradient turned into an approximately orthogonal matrix
          by an approximate SVD, eq. 9-10);
  - §3.1  image sets: the chunk is the whole sequence;
  - §3.2  language: fixed 2K/4K chunks with a shifted block-causal mask
          (chunk i only sees weights left by chunks 0..i-1);
  - §3.3  video: fast weights are updated only on the clean-frame chunks.
* TTT tutorial page ("Test-Time Training layers", aivaro.ru/zh/answers/718):
  - §3    the recurrence theta_t = theta_{t-1} - eta * grad L, then h_t = f(x_t),
          an MSE reconstruction loss, and a linear inner model.

The equations (2, 4-5, 8, 9-10) are referenced on the LaCT page but not printed.
The readings used here:

* inner loss per token: inner product  l_t = -f(k_t).v_t,
  or MSE  l_t = 1/2 ||f(k_t) - v_t||^2;
* chunk gradient G = sum_t eta_t * grad_W l_t  (a SUM, per-token lr inside);
* SwiGLU fast net f(x) = W2 (silu(W1 x) * (W3 x)); linear f(x) = W x;
* Muon (when on): Newton-Schulz quintic iteration of the public Muon method on
  the wide orientation, X0 = G / (||G||_F + eps), X <- aX + (bA + cA^2)X with
  A = X X^T, coefficients (a, b, c) given by the caller;
* momentum (off by default, mu = 0): a buffer per matrix, M <- mu M + G, carried
  from update to update and fed to Newton-Schulz (or, with Muon off, used as the
  step: the plain momentum optimiser the LaCT page compares Muon with, §2.2.1);
* update W <- W - step * U, U = NS(M) or M (M = G without momentum);
* per-token learning rates: one per token shared by the matrices ([T]), or one
  per token and matrix ([T, n_matrices]); G_j = sum_t eta_{t,j} grad_{W_j} l_t;
* weight norm (when on): each row of each out x in matrix is rescaled to the
  row norm it had in W0:  W[r,:] <- W[r,:] * n0[r] / max(||W[r,:]||, floor);
* shifted mode: for each chunk, apply with the current W, then (if the chunk's
  update flag is set) update; "single" mode: for each chunk, update first,
  then apply (with one chunk covering the whole sequence this is the image-set
  layer);
* "inclusive" mode (the tutorial page's per-token order, §3: update with x_t,
  then output with the updated weights), for chunks of any size: query t of a
  chunk sees the chunk's starting weights minus step times the summed
  gradients of the chunk's tokens up to and including t, each taken at the
  starting weights (mini-batch test-time training); the chunk then updates
  with the sum over all its tokens. With chunks of one token this is exactly
  the per-token recurrence. Plain gradient steps only (no Muon, momentum or
  weight norm: those act on a whole chunk's update, not on a prefix of it).

The sums over tokens of a whole-sequence chunk are taken over blocks of tokens
(``block`` argument) only to bound host memory; in fp64 the grouping of the
terms of a sum changes nothing that the tolerances see.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import numpy as np

Weights = Tuple[np.ndarray, ...]


# ------------------------------------------------------------------ fast nets
def sigmoid(x: np.ndarray) -> np.ndarray:
    """Logistic function, evaluated without overflow for either sign."""
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def swiglu_apply(W: Weights, X: np.ndarray) -> np.ndarray:
    """f(x) = W2 (silu(W1 x) * (W3 x)) for every row x of X (LaCT page §1.2)."""
    W1, W2, W3 = W
    A = X @ W1.T
    Bm = X @ W3.T
    H = A * sigmoid(A) * Bm
    return H @ W2.T


def linear_apply(W: Weights, X: np.ndarray) -> np.ndarray:
    """f(x) = W x (tutorial page §3-§4: a linear inner model)."""
    return X @ W[0].T


def swiglu_grad(W: Weights, K: np.ndarray, V: np.ndarray, eta: np.ndarray,
                loss: str) -> Weights:
    """Gradient of sum_t eta_t * l_t over the tokens (K, V) for the SwiGLU net.

    Returns (G1, G2, G3) shaped like (W1, W2, W3). Hand-derived backward:
      a = W1 k, b = W3 k, s = silu(a), h = s * b, f = W2 h
      dl/df = -v (inner product) or f - v (MSE), scaled by eta_t
      G2 = sum (dl/df) h^T,  dh = W2^T dl/df
      da = dh * b * silu'(a),  silu'(a) = sig(a) (1 + a (1 - sig(a)))
      db = dh * s
      G1 = sum da k^T,  G3 = sum db k^T
    """
    W1, W2, W3 = W
    A = K @ W1.T
    Bm = K @ W3.T
    sg = sigmoid(A)
    S = A * sg
    H = S * Bm
    if loss == "ip":
        Y = -V
    elif loss == "mse":
        Y = H @ W2.T - V
    else:
        raise ValueError(loss)
    Yh = eta[:, None] * Y
    G2 = Yh.T @ H
    DH = Yh @ W2
    DA = DH * Bm * sg * (1.0 + A * (1.0 - sg))
    DB = DH * S
    G1 = DA.T @ K
    G3 = DB.T @ K
    return G1, G2, G3


def linear_grad(W: Weights, K: np.ndarray, V: np.ndarray, eta: np.ndarray,
                loss: str) -> Weights:
    """Gradient of sum_t eta_t * l_t for f(x) = W x: G = sum_t eta_t (dl/df_t) k_t^T."""
    if loss == "ip":
        Y = -V
    elif loss == "mse":
        Y = K @ W[0].T - V
    else:
        raise ValueError(loss)
    return ((eta[:, None] * Y).T @ K,)


# ------------------------------------------------------------------ optimiser
def newton_schulz(G: np.ndarray, iters: int, a: float, b: float, c: float,
                  eps: float) -> np.ndarray:
    """Muon's orthogonalisation of one gradient matrix (LaCT page §2.2.1, eq. 9-10).

    Works on the wide orientation (rows <= cols) and maps back.
    """
    tall = G.shape[0] > G.shape[1]
    X = G.T if tall else G
    X = X / (np.sqrt((X * X).sum()) + eps)
    for _ in range(iters):
        A = X @ X.T
        X = a * X + (b * A + c * (A @ A)) @ X
    return X.T if tall else X


def row_norms(W: np.ndarray) -> np.ndarray:
    return np.sqrt((W * W).sum(axis=1))


def weight_norm(W: np.ndarray, n0: np.ndarray, floor: float) -> np.ndarray:
    """Rescale every row to its reference norm n0 (LaCT page §2.2.1, eq. 8)."""
    return W * (n0 / np.maximum(row_norms(W), floor))[:, None]


class OracleCfg:
    """Hyper-parameters of the layer, as plain attributes."""

    def __init__(self, chunk: int, fast_net: str = "swiglu", loss: str = "ip",
                 mode: str = "shifted", muon: bool = True, ns_iters: int = 5,
                 ns_coef: Tuple[float, float, float] = (3.4445, -4.7750, 2.0315),
                 ns_eps: float = 1e-7, wnorm: bool = True, wnorm_floor: float = 1e-12,
                 step: float = 1.0, mask: Optional[Sequence[int]] = None, momentum: float = 0.0):
        self.chunk = int(chunk)
        self.fast_net = fast_net
        self.loss = loss
        self.mode = mode
        self.muon = bool(muon)
        self.ns_iters = int(ns_iters)
        self.ns_coef = tuple(float(x) for x in ns_coef)
        self.ns_eps = float(ns_eps)
        self.wnorm = bool(wnorm)
        self.wnorm_floor = float(wnorm_floor)
        self.step = float(step)
        self.mask = None if mask is None else [int(m) for m in mask]
        self.momentum = float(momentum)

    @classmethod
    def from_spec(cls, spec) -> "OracleCfg":
        """Build from a workload description with LayerSpec-style attributes."""
        return cls(chunk=spec.chunk, fast_net=spec.fast_net, loss=spec.loss,
                   mode=spec.mode, muon=spec.muon, ns_iters=spec.ns_iters,
                   wnorm=spec.wnorm, step=spec.step, mask=list(spec.update_mask()),
                   momentum=getattr(spec, "momentum", 0.0))


def _apply(cfg: OracleCfg, W: Weights, X: np.ndarray) -> np.ndarray:
    return swiglu_apply(W, X) if cfg.fast_net == "swiglu" else linear_apply(W, X)


def chunk_grad(cfg: OracleCfg, W: Weights, K: np.ndarray, V: np.ndarray,
               eta: np.ndarray, block: int = 0) -> Weights:
    """Chunk gradient: the sum over the chunk's tokens (LaCT page §2.1).

    eta is [n] (one rate per token for every matrix) or [n, len(W)] (one per
    token and matrix): matrix j's gradient is then the sum weighted by column j.
    """
    eta = np.asarray(eta, dtype=np.float64)
    if eta.ndim == 2:
        # the gradient is linear in the token weights: G_j from column j alone
        return tuple(chunk_grad(cfg, W, K, V, eta[:, j], block)[j] for j in range(len(W)))
    fn = swiglu_grad if cfg.fast_net == "swiglu" else linear_grad
    n = K.shape[0]
    if block <= 0 or block >= n:
        return fn(W, K, V, eta, cfg.loss)
    total = None
    for s in range(0, n, block):
        e = min(n, s + block)
        g = fn(W, K[s:e], V[s:e], eta[s:e], cfg.loss)
        total = list(g) if total is None else [t + x for t, x in zip(total, g)]
    return tuple(total)


def update(cfg: OracleCfg, W: Weights, G: Weights, n0: Sequence[np.ndarray],
           mom: Optional[List[np.ndarray]] = None) -> Weights:
    """One fast-weight update: optional momentum, optional Muon, the step,
    optional weight norm. `mom` (the momentum buffers, one per matrix) is
    updated in place when given; without it the update has no momentum."""
    a, b, c = cfg.ns_coef
    new = []
    for j, (Wj, Gj, nj) in enumerate(zip(W, G, n0)):
        if mom is not None:
            mom[j] = cfg.momentum * mom[j] + Gj
            Gj = mom[j]
        Uj = newton_schulz(Gj, cfg.ns_iters, a, b, c, cfg.ns_eps) if cfg.muon else Gj
        Wj = Wj - cfg.step * Uj
        if cfg.wnorm:
            Wj = weight_norm(Wj, nj, cfg.wnorm_floor)
        new.append(Wj)
    return tuple(new)


def ttt_head(cfg: OracleCfg, Q: np.ndarray, K: np.ndarray, V: np.ndarray,
             lr: np.ndarray, W0: Weights, block: int = 0) -> Tuple[np.ndarray, Weights]:
    """The layer on one (batch, head): returns (O [T, d], final weights)."""
    T = Q.shape[0]
    C = cfg.chunk
    n = (T + C - 1) // C
    mask = cfg.mask if cfg.mask is not None else [1] * n
    if len(mask) < n:
        raise ValueError("update mask shorter than the number of chunks")
    W = tuple(np.asarray(w, dtype=np.float64) for w in W0)
    n0 = [row_norms(w) for w in W]
    lr = np.asarray(lr, dtype=np.float64)
    # momentum buffers start at zero; with mu = 0 the buffer is the gradient itself
    mom = [np.zeros_like(w) for w in W] if cfg.momentum != 0.0 else None
    O = np.empty((T, W[0].shape[0] if cfg.fast_net == "linear" else W[1].shape[0]))
    for ci in range(n):
        s, e = ci * C, min(T, (ci + 1) * C)
        if cfg.mode == "shifted":
            O[s:e] = _apply_blocks(cfg, W, Q[s:e], block)
            if mask[ci]:
                W = update(cfg, W, chunk_grad(cfg, W, K[s:e], V[s:e], lr[s:e], block), n0, mom)
        elif cfg.mode == "single":
            if mask[ci]:
                W = update(cfg, W, chunk_grad(cfg, W, K[s:e], V[s:e], lr[s:e], block), n0, mom)
            O[s:e] = _apply_blocks(cfg, W, Q[s:e], block)
        elif cfg.mode == "inclusive":
            if cfg.muon or cfg.wnorm or cfg.momentum != 0.0:
                raise ValueError("inclusive mode takes plain gradient steps only")
            if mask[ci]:
                O[s:e] = apply_inclusive(cfg, W, Q[s:e], K[s:e], V[s:e], lr[s:e])
                W = update(cfg, W, chunk_grad(cfg, W, K[s:e], V[s:e], lr[s:e], block), n0, mom)
            else:
                O[s:e] = _apply_blocks(cfg, W, Q[s:e], block)
        else:
            raise ValueError(cfg.mode)
    return O, W


def apply_inclusive(cfg: OracleCfg, W: Weights, Q: np.ndarray, K: np.ndarray, V: np.ndarray,
                    eta: np.ndarray) -> np.ndarray:
    """Outputs of one chunk in inclusive mode: for token t the weights
    W - step * sum_{s <= t} grad_s(W), then f(q_t) (tutorial page §3)."""
    acc = [np.zeros_like(w) for w in W]
    out = np.empty((Q.shape[0], W[0].shape[0] if cfg.fast_net == "linear" else W[1].shape[0]))
    for t in range(Q.shape[0]):
        g = chunk_grad(cfg, W, K[t:t + 1], V[t:t + 1], eta[t:t + 1])
        acc = [a + gj for a, gj in zip(acc, g)]
        Wt = tuple(w - cfg.step * a for w, a in zip(W, acc))
        out[t] = _apply(cfg, Wt, Q[t:t + 1])[0]
    return out


def _apply_blocks(cfg: OracleCfg, W: Weights, X: np.ndarray, block: int) -> np.ndarray:
    if block <= 0 or block >= X.shape[0]:
        return _apply(cfg, W, X)
    return np.concatenate([_apply(cfg, W, X[s:s + block])
                           for s in range(0, X.shape[0], block)])


def ttt_layer(cfg: OracleCfg, Q: np.ndarray, K: np.ndarray, V: np.ndarray,
              lr: np.ndarray, W0: Sequence[np.ndarray],
              heads: Optional[Sequence[Tuple[int, int]]] = None,
              w0_per_batch: bool = False, block: int = 0):
    """The layer on [B, H, T, d] inputs.

    W0 holds each matrix as [H, out, in] (shared over the batch) or, with
    ``w0_per_batch``, [B, H, out, in]. Returns (O, Wf) for the requested
    (b, h) heads (all by default): O as [B, H, T, d] when every head is
    computed, else a dict {(b, h): (O_bh, Wf_bh)}.
    """
    Bn, Hn = Q.shape[0], Q.shape[1]
    want = heads if heads is not None else [(b, h) for b in range(Bn) for h in range(Hn)]
    out = {}
    for (b, h) in want:
        w0 = tuple(np.asarray(w[b, h] if w0_per_batch else w[h], dtype=np.float64)
                   for w in W0)
        out[(b, h)] = ttt_head(cfg, np.asarray(Q[b, h], np.float64),
                               np.asarray(K[b, h], np.float64),
                               np.asarray(V[b, h], np.float64), lr[b, h], w0, block)
    if heads is not None:
        return out
    O = np.stack([np.stack([out[(b, h)][0] for h in range(Hn)]) for b in range(Bn)])
    Wf = [np.stack([np.stack([out[(b, h)][1][j] for h in range(Hn)]) for b in range(Bn)])
          for j in range(len(W0))]
    return O, Wf


# ------------------------------------------------------------------ backward (outer loop)
def linear_head_backward(cfg: OracleCfg, Q: np.ndarray, K: np.ndarray, V: np.ndarray, lr: np.ndarray,
                         W0: np.ndarray, dO: np.ndarray, dWf: np.ndarray):
    """Gradients of a scalar loss L through the layer on one head, given
    dL/dO (dO) and dL/dW_final (dWf): returns (dQ, dK, dV, dlr, dW0).

    The outer loop of the TTT-E2E news page (§2.2: the model's loss is
    differentiated through the inner updates), for the linear net with plain
    gradient steps in shifted mode (the small-chunk regime). Per chunk c of
    tokens t: o_t = W_c q_t; y_t = W_c k_t - v_t (MSE) or -v_t (inner product);
    W_{c+1} = W_c - step * sum_t lr_t y_t k_t^T. Reverse mode, chunk by chunk
    from the last, with L_c = dL/dW_c:
      L_c = L_{c+1} + sum_t dO_t q_t^T + [MSE] sum_t e_t k_t^T,
      with a_t = -step L_{c+1} k_t (the cotangent of lr_t y_t) and e_t = lr_t a_t;
      dq_t = W_c^T dO_t;  dlr_t = y_t . a_t;  dv_t = -e_t;
      dk_t = -step L_{c+1}^T (lr_t y_t) + [MSE] W_c^T e_t.
    """
    if cfg.fast_net != "linear" or cfg.muon or cfg.wnorm or cfg.momentum != 0.0 or cfg.mode != "shifted":
        raise ValueError("the backward covers the linear net, plain steps, shifted mode")
    T = Q.shape[0]
    C = cfg.chunk
    n = (T + C - 1) // C
    mask = cfg.mask if cfg.mask is not None else [1] * n
    lr = np.asarray(lr, dtype=np.float64)
    # forward, keeping every chunk's starting weights
    Ws = [np.asarray(W0, dtype=np.float64)]
    for ci in range(n):
        s, e = ci * C, min(T, (ci + 1) * C)
        W = Ws[-1]
        if mask[ci]:
            Y = (K[s:e] @ W.T - V[s:e]) if cfg.loss == "mse" else -V[s:e]
            W = W - cfg.step * (lr[s:e, None] * Y).T @ K[s:e]
        Ws.append(W)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    dlr = np.zeros(T)
    Lnext = np.asarray(dWf, dtype=np.float64).copy()   # dL/dW_{c+1}
    for ci in reversed(range(n)):
        s, e = ci * C, min(T, (ci + 1) * C)
        W = Ws[ci]
        Lc = Lnext.copy()
        dQ[s:e] = dO[s:e] @ W
        Lc += dO[s:e].T @ Q[s:e]
        if mask[ci]:
            Y = (K[s:e] @ W.T - V[s:e]) if cfg.loss == "mse" else -V[s:e]
            A = -cfg.step * K[s:e] @ Lnext.T                  # rows a_t = -step L_{c+1} k_t
            dlr[s:e] = (Y * A).sum(axis=1)
            E = lr[s:e, None] * A                             # rows e_t: cotangents of y_t
            dV[s:e] = -E
            dK[s:e] = -cfg.step * (lr[s:e, None] * Y) @ Lnext
            if cfg.loss == "mse":
                dK[s:e] += E @ W
                Lc += E.T @ K[s:e]
        Lnext = Lc
    return dQ, dK, dV, dlr, Lnext


def swiglu_head_backward(cfg: OracleCfg, Q: np.ndarray, K: np.ndarray, V: np.ndarray, lr: np.ndarray,
                         W0: Weights, dO: np.ndarray, dWf: Weights):
    """Gradients of a scalar loss L through the layer on one head for the
    SwiGLU net with plain gradient steps in shifted mode, given dL/dO (dO) and
    dL/dW_final (dWf, one per matrix): returns (dQ, dK, dV, dlr, dW0) with dW0 a
    tuple (dW1, dW2, dW3).

    The outer loop of the TTT-E2E news page (§2.2: the model's loss is
    differentiated through the inner updates). The forward is the same as
    ttt_head's for this configuration, written with fp64 torch operations so that
    reverse-mode automatic differentiation (a library routine) gives every
    gradient: per chunk c, O_t = f(q_t; W_c) for the chunk's queries, then
    W_{c+1} = W_c - step * sum_t lr_t grad_W l_t(W_c) with swiglu_grad's
    hand-derived gradient (which the automatic differentiation goes through, so
    the second-order terms of the update come out of it), and
    L = sum dO * O + sum_j <dWf_j, W_final_j>.
    """
    import torch  # fp64 CPU tensors only

    if cfg.fast_net != "swiglu" or cfg.muon or cfg.wnorm or cfg.momentum != 0.0 or cfg.mode != "shifted":
        raise ValueError("the SwiGLU backward covers plain steps in shifted mode")
    f64 = torch.float64
    tq, tk, tv = (torch.tensor(np.asarray(x, dtype=np.float64), dtype=f64, requires_grad=True) for x in (Q, K, V))
    tl = torch.tensor(np.asarray(lr, dtype=np.float64), dtype=f64, requires_grad=True)
    tw = [torch.tensor(np.asarray(w, dtype=np.float64), dtype=f64, requires_grad=True) for w in W0]

    def apply(W, X):
        A = X @ W[0].T
        return (A * torch.sigmoid(A) * (X @ W[2].T)) @ W[1].T

    def grad(W, Kc, Vc, eta):
        A = Kc @ W[0].T
        Bm = Kc @ W[2].T
        sg = torch.sigmoid(A)
        S = A * sg
        H = S * Bm
        Y = -Vc if cfg.loss == "ip" else H @ W[1].T - Vc
        Yh = eta[:, None] * Y
        DH = Yh @ W[1]
        DA = DH * Bm * sg * (1.0 + A * (1.0 - sg))
        DB = DH * S
        return DA.T @ Kc, Yh.T @ H, DB.T @ Kc

    T = Q.shape[0]
    C = cfg.chunk
    n = (T + C - 1) // C
    mask = cfg.mask if cfg.mask is not None else [1] * n
    W = list(tw)
    outs = []
    for ci in range(n):
        s, e = ci * C, min(T, (ci + 1) * C)
        outs.append(apply(W, tq[s:e]))
        if mask[ci]:
            G = grad(W, tk[s:e], tv[s:e], tl[s:e])
            W = [w - cfg.step * g for w, g in zip(W, G)]
    O = torch.cat(outs, dim=0)
    L = (O * torch.tensor(np.asarray(dO, dtype=np.float64), dtype=f64)).sum()
    for w, dw in zip(W, dWf):
        L = L + (w * torch.tensor(np.asarray(dw, dtype=np.float64), dtype=f64)).sum()
    gq, gk, gv, gl, g1, g2, g3 = torch.autograd.grad(L, [tq, tk, tv, tl] + tw, allow_unused=True)
    z = lambda g, like: (np.zeros_like(like) if g is None else g.detach().numpy())
    return (z(gq, Q), z(gk, K), z(gv, V), z(gl, np.asarray(lr, dtype=np.float64)),
            (z(g1, W0[0]), z(g2, W0[1]), z(g3, W0[2])))
