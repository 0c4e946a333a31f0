"""Emulation, on the CPU, of the tensor-core path's operand precision for one head of
the SwiGLU layer (shifted order, inner-product loss, Muon + weight norm), used to ask
which terms of the split (hi/lo) products the recurrence needs.

Test infrastructure, not the product: it shares no code with the CUDA path and
compares against the fp64 oracle. Each contraction is a float32 matrix product (fp32
accumulation, as in TMEM) of operands rounded the way the kernels store them:

  'x'   exact (already representable: the bf16 tokens)
  'b1'  one bf16 operand            'b2'  bf16 pair hi = bf16(x), lo = bf16(x - hi)
  'h1'  one fp16 operand            'h2'  fp16 pair
  (the fp16 modes scale by a power of two first so the largest entry sits near 2^14)

A product of two operands sums the selected terms among hi*hi, hi*lo and lo*hi.
The dataflow follows the kernels: the key forward [A|B] = K[M1|M3], Dm = V M2
(M1 = W1^T, M2 = W2, M3 = W3^T, fp32 masters); the SwiGLU backward in fp32 with the
token's rate folded in (E = DA, He, DB); the chunk gradient G1 = K^T DA, G2 = V^T He,
G3 = K^T DB; Newton-Schulz on the wide orientation with the square completed
(R = X X^T + beta I, P = c R R + alpha I, X <- P X; the first Gram and X update scaled
by 1/||G||^2 and 1/||G||); W <- W - step U; the row weight norm in fp64.

    python tests/precision_study.py [workload [n_chunks]]   # the study on head (0, 0)
"""
from __future__ import annotations

import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from long_seq_models_chunked_b300 import synth  # noqa: E402
from oracle import OracleCfg, ttt_head  # noqa: E402

F32 = np.float32
ALL = ("hh", "hl", "lh")


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest-even bf16, returned as fp32 (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=F32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(F32)


def fp16_round(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=F32).astype(np.float16).astype(F32)


def operand(x: np.ndarray, mode: str) -> list:
    """The parts (hi, or hi and lo) of x stored in `mode`, as fp32 arrays."""
    x = np.asarray(x, dtype=F32)
    if mode == "x":
        return [x]
    if mode in ("b1", "b2"):
        h = bf16_round(x)
        return [h] if mode == "b1" else [h, bf16_round(x - h)]
    if mode in ("h1", "h2"):
        mx = float(np.abs(x).max()) or 1.0
        sc = F32(2.0 ** np.floor(np.log2(16384.0 / mx)))
        h = fp16_round(x * sc)
        return [h / sc] if mode == "h1" else [h / sc, fp16_round(x * sc - h) / sc]
    if mode == "f32":
        return [x]
    raise ValueError(mode)


def product(a: list, b: list, terms=ALL) -> np.ndarray:
    out = None
    for t in terms:
        ia, ib = int(t[0] == "l"), int(t[1] == "l")
        if ia < len(a) and ib < len(b):
            r = np.matmul(a[ia], b[ib])
            out = r if out is None else out + r
    return out


def emulate_head(spec, n_chunks: int, fwd=("b2", "b2", "b2"), E=("b2", "b2", "b2"),
                 ns=("b2",) * 5, g0="b2", terms=None, x=None, block: int = 65536):
    """Final (W1, W2, W3) of head (0, 0) after n_chunks chunks, fp64 arrays.

    fwd: modes of the M1, M2, M3 shadows in the key forward; E: modes of DA, He, DB;
    ns: mode of R, P (and of X entering the next iteration) per iteration; g0: mode of
    the unscaled gradient entering the first iteration; terms: per phase ('gram',
    'poly', 'xup') the product terms used."""
    terms = terms or {}
    x = x if x is not None else synth.head_tokens(spec, 0, 0, 0, n_chunks * spec.chunk)
    w0 = [w[0].astype(np.float64) for w in synth.initial_weights(spec)]
    K, V, lr = x["K64"].astype(F32), x["V64"].astype(F32), x["lr"].astype(F32)
    a, b, c = OracleCfg(chunk=1).ns_coef
    beta, alpha = b / (2 * c), a - b * b / (4 * c)
    M = [w0[0].T.astype(F32), w0[1].astype(F32), w0[2].T.astype(F32)]
    n0 = [np.sqrt((w ** 2).sum(1)) for w in w0]
    mask = spec.update_mask()
    C = spec.chunk
    for ci in range(n_chunks):
        if not mask[ci]:
            continue
        sh = [operand(m, fwd[j]) for j, m in enumerate(M)]
        G = [np.zeros(M[0].shape, dtype=F32) for _ in range(3)]
        c0, c1 = ci * C, min(K.shape[0], (ci + 1) * C)
        for s0 in range(c0, c1, block):     # token blocks: fp32 partial sums of the gradient
            s1 = min(c1, s0 + block)
            Kc, Vc, lc = K[s0:s1], V[s0:s1], lr[s0:s1, None]
            A, Bm, Dm = product([Kc], sh[0]), product([Kc], sh[2]), product([Vc], sh[1])
            sg = (1.0 / (1.0 + np.exp(-A.astype(np.float64)))).astype(F32)
            S = A * sg
            # dl/df = -v: the rate-scaled cotangent of H is -lr * (V W2)
            DA = -lc * Dm * Bm * sg * (1.0 + A * (1.0 - sg))
            DB = -lc * Dm * S
            He = -lc * (S * Bm)
            # (the fp16 modes take their power-of-two scale per block)
            Eo = [operand(v, m) for v, m in zip((DA, He, DB), E)]
            for j, (tok, e) in enumerate(((Kc, Eo[0]), (Vc, Eo[1]), (Kc, Eo[2]))):
                G[j] += product([tok.T.copy()], e)
        for j in range(3):
            g = G[j]
            inv = 1.0 / (float(np.sqrt((g.astype(np.float64) ** 2).sum())) + 1e-7)
            X = operand(g, g0)
            eye = np.eye(g.shape[0], dtype=F32)
            for it in range(5):
                R = product(X, [p.T.copy() for p in X], terms.get("gram", ALL))
                R = R * F32(inv * inv) if it == 0 else R
                Ro = operand(R + F32(beta) * eye, ns[it])
                Po = operand(F32(c) * product(Ro, Ro, terms.get("poly", ALL)) + F32(alpha) * eye, ns[it])
                Xn = product(Po, X, terms.get("xup", ALL))
                Xn = Xn * F32(inv) if it == 0 else Xn
                X = operand(Xn, ns[it + 1]) if it < 4 else [Xn]
            M[j] = M[j] - F32(spec.step) * X[0]
        for j in range(3):
            m = M[j].astype(np.float64)
            ax = 1 if j == 1 else 0
            nr = np.sqrt((m ** 2).sum(ax))
            s = n0[j] / np.maximum(nr, 1e-12)
            M[j] = (m * (s[:, None] if j == 1 else s[None, :])).astype(F32)
    return M[0].T.astype(np.float64), M[1].astype(np.float64), M[2].T.astype(np.float64)


def oracle_head(spec, n_chunks: int, x=None):
    x = x if x is not None else synth.head_tokens(spec, 0, 0, 0, n_chunks * spec.chunk)
    w0 = tuple(w[0].astype(np.float64) for w in synth.initial_weights(spec))
    _, W = ttt_head(OracleCfg.from_spec(spec), x["Q64"], x["K64"], x["V64"], x["lr"], w0, block=65536)
    return W


def max_rel_err(W, Wr) -> float:
    return max(float(np.abs(p - q).max() / np.abs(q).max()) for p, q in zip(W, Wr))


F16_1 = ("h1",) * 5
STUDY = {
    "every operand split (the shipped SPLIT precision)": {},
    "every operand single (bf16; fp16 in Newton-Schulz)": dict(fwd=("b1",) * 3, E=("b1",) * 3, ns=F16_1, g0="h1"),
    "key forward: weights single bf16": dict(fwd=("b1",) * 3),
    "key forward: W1 only single bf16": dict(fwd=("b1", "b2", "b2")),
    "key forward: weights single fp16": dict(fwd=("h1",) * 3),
    "gradient: E single bf16": dict(E=("b1",) * 3),
    "gradient: DA only single bf16": dict(E=("b1", "b2", "b2")),
    "gradient: E single fp16": dict(E=("h1",) * 3),
    "key forward and E single fp16": dict(fwd=("h1",) * 3, E=("h1",) * 3),
    "Newton-Schulz single fp16": dict(ns=F16_1, g0="h1"),
    "Newton-Schulz single bf16": dict(ns=("b1",) * 5, g0="b1"),
    "Newton-Schulz: G single bf16": dict(g0="b1"),
    "Newton-Schulz: iteration 1 single fp16": dict(ns=("h1", "b2", "b2", "b2", "b2")),
    "Newton-Schulz: iteration 5 single fp16": dict(ns=("b2", "b2", "b2", "b2", "h1")),
    "Newton-Schulz: Gram without lo*hi": dict(terms={"gram": ("hh", "hl")}),
    "Newton-Schulz: polynomial without lo*hi": dict(terms={"poly": ("hh", "hl")}),
    "Newton-Schulz: X update without lo*hi": dict(terms={"xup": ("hh", "hl")}),
    "Newton-Schulz: X update without hi*lo": dict(terms={"xup": ("hh", "lh")}),
    "Newton-Schulz fp16 pairs": dict(ns=("h2",) * 5, g0="h2"),
    "Newton-Schulz fp16 pairs, Gram without lo*hi": dict(ns=("h2",) * 5, g0="h2", terms={"gram": ("hh", "hl")}),
    "Newton-Schulz fp16 pairs, polynomial without lo*hi": dict(ns=("h2",) * 5, g0="h2", terms={"poly": ("hh", "hl")}),
    "Newton-Schulz fp16 pairs, X update without lo*hi": dict(ns=("h2",) * 5, g0="h2", terms={"xup": ("hh", "hl")}),
}


def main():
    name = sys.argv[1] if len(sys.argv) > 1 else "lm_chunk2k"
    spec = synth.WORKLOADS[name]
    n = int(sys.argv[2]) if len(sys.argv) > 2 else spec.n_chunks
    x = synth.head_tokens(spec, 0, 0, 0, min(spec.T, n * spec.chunk))
    Wr = oracle_head(spec, n, x)
    print(f"{name} head (0, 0), {n} chunk(s): max relative error of the final W1, W2, W3")
    for name, kw in STUDY.items():
        t0 = time.time()
        e = max_rel_err(emulate_head(spec, n, x=x, **kw), Wr)
        print(f"  {e:9.3e}  {name}   ({time.time() - t0:.0f} s)", flush=True)


if __name__ == "__main__":
    main()
