"""Seeded synthetic inputs for the chunked TTT fast-weight layer.

This module is shared by the CUDA path's tests and benchmark and by the fp64
oracle's tests. It holds the workload table and the random-number recipe only:
none of the layer's arithmetic lives here.

Recipe (the LaCT page, "Large Chunk Test-Time Training", §3.1-§3.3 and §4.1
Table 1 give the workload shapes; the value distributions are the ones the
workload table below states):

* Q, K, V ~ N(0, 1) drawn in fp64; every token of Q and K is divided by its L2
  norm in fp64 (V is not normalised).
* The fp64 values are rounded to the storage type: fp32 (round to nearest even),
  or fp32 and then bf16 (round to nearest even on the fp32 bit pattern).
  Everyone downstream (oracle and kernels) consumes the ROUNDED values.
* Per-token learning rates: ``uniform(lo, hi)`` or ``scale * sigmoid(N(0, 1))``,
  computed in fp64 and rounded to fp32; with per-matrix rates, one such column
  per matrix (column 0 is the shared rate's stream).
* Initial fast weights (one set per head, shared by every batch row):
  W1, W3 ~ N(0, 1/d), W2 ~ N(0, 1/dh); linear W ~ N(0, 1/d); stored fp32.
* Streams: numpy PCG64 seeded by ``SeedSequence(entropy=ENTROPY,
  spawn_key=(seed, tensor, b, h, block))``; tokens come in blocks of
  ``TOKEN_BLOCK`` so any token range of any head can be regenerated on its own.
"""
from __future__ import annotations

import dataclasses
import functools
import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

ENTROPY = 20261202
TOKEN_BLOCK = 4096

# tensor ids inside the spawn key
_T_Q, _T_K, _T_V, _T_LR = 0, 1, 2, 3
_T_W = 10  # + matrix index
_T_LR_COL = 20  # + matrix index (per-matrix rates, columns 1 and 2)


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    """Shape and hyper-parameters of one TTT-layer workload."""

    name: str
    B: int
    H: int
    T: int
    d: int
    dh: int
    chunk: int
    fast_net: str = "swiglu"   # "swiglu" | "linear"
    loss: str = "ip"           # "ip" (-f(k).v) | "mse" (1/2 ||f(k)-v||^2)
    mode: str = "shifted"      # "shifted" | "single" (update-then-apply per chunk) | "inclusive"
    dtype: str = "bf16"        # storage type of Q, K, V, O: "bf16" | "fp32"
    muon: bool = True
    ns_iters: int = 5
    wnorm: bool = True
    step: float = 1.0
    update: str = "all"        # "all" | "odd" (0-based odd chunks update) | "none"
    lr_kind: str = "sigmoid"   # "sigmoid" | "uniform"
    lr_a: float = 0.01         # sigmoid: scale; uniform: low
    lr_b: float = 0.0          # uniform: high
    seed: int = 0
    momentum: float = 0.0      # mu of the per-matrix momentum buffer (0 = none)
    lr_per_matrix: bool = False  # lr [T, n_weights]: one rate per token and matrix

    @property
    def n_chunks(self) -> int:
        return (self.T + self.chunk - 1) // self.chunk

    @property
    def n_weights(self) -> int:
        return 3 if self.fast_net == "swiglu" else 1

    def weight_shapes(self) -> List[Tuple[int, int]]:
        """Out x in shapes of the fast-weight matrices (W1, W2, W3) or (W,)."""
        if self.fast_net == "swiglu":
            return [(self.dh, self.d), (self.d, self.dh), (self.dh, self.d)]
        return [(self.d, self.d)]

    def update_mask(self) -> np.ndarray:
        m = np.ones(self.n_chunks, dtype=np.uint8)
        if self.update == "odd":
            m[:] = 0
            m[1::2] = 1
        elif self.update == "none":
            m[:] = 0
        return m

    def replace(self, **kw) -> "LayerSpec":
        return dataclasses.replace(self, **kw)


# The five workloads. Sizes follow the LaCT page: language chunks of 2K tokens
# (§3.2, §4.1), one chunk of 128 images x (960/8) x (536/8) patches = 1,029,120
# tokens (§3.1), video chunks of three latent frames (§3.3, §4.1), and the
# small-chunk linear regime the page contrasts with (§1.1: 16-64 token updates).
WORKLOADS: Dict[str, LayerSpec] = {
    "tiny_fp32": LayerSpec(
        "tiny_fp32", B=1, H=2, T=256, d=32, dh=64, chunk=64, dtype="fp32",
        muon=False, wnorm=True, lr_kind="uniform", lr_a=0.0, lr_b=0.1, seed=1),
    "lm_chunk2k": LayerSpec(
        "lm_chunk2k", B=2, H=3, T=32768, d=512, dh=1024, chunk=2048,
        lr_a=0.01, seed=2),
    "imageset_1m": LayerSpec(
        "imageset_1m", B=1, H=4, T=1029120, d=192, dh=384, chunk=1029120,
        mode="single", lr_a=0.005, seed=3),
    "video_ar": LayerSpec(
        "video_ar", B=1, H=8, T=56160, d=640, dh=1280, chunk=5616,
        update="odd", lr_a=0.01, seed=4),
    "linear_chunk64": LayerSpec(
        "linear_chunk64", B=16, H=16, T=8192, d=64, dh=64, chunk=64,
        fast_net="linear", loss="mse", muon=False, wnorm=False, lr_a=0.1, seed=5),
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(
        np.random.SeedSequence(entropy=ENTROPY, spawn_key=tuple(int(k) for k in key))))


# ---------------------------------------------------------------- rounding
def round_fp32(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def fp32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def to_storage(x64: np.ndarray, dtype: str) -> Tuple[np.ndarray, np.ndarray]:
    """Round fp64 values to the storage type.

    Returns (stored, exact) where ``stored`` is float32 (fp32) or uint16 bf16
    bit patterns, and ``exact`` is the fp64 value of every stored element.
    """
    x32 = round_fp32(x64)
    if dtype == "fp32":
        return x32, x32.astype(np.float64)
    if dtype == "bf16":
        bits = fp32_to_bf16_bits(x32)
        return bits, bf16_bits_to_f64(bits)
    raise ValueError(dtype)


# ---------------------------------------------------------------- per-head draws
@functools.lru_cache(maxsize=6)
def _block_normals(seed: int, tensor: int, b: int, h: int, blk: int, width: int) -> np.ndarray:
    """One block of TOKEN_BLOCK tokens' standard normals (read-only). The last few
    blocks are kept, so walking a head chunk by chunk draws each block once."""
    z = _rng(seed, tensor, b, h, blk).standard_normal((TOKEN_BLOCK, width))
    z.setflags(write=False)
    return z


def _token_draw(spec: LayerSpec, tensor: int, b: int, h: int, t0: int, t1: int,
                width: int) -> np.ndarray:
    """Standard normals for tokens [t0, t1) of one head, shape [t1-t0, width]."""
    out = np.empty((t1 - t0, width), dtype=np.float64)
    blk0, blk1 = t0 // TOKEN_BLOCK, (t1 - 1) // TOKEN_BLOCK
    for blk in range(blk0, blk1 + 1):
        z = _block_normals(spec.seed, tensor, b, h, blk, width)
        s = max(t0, blk * TOKEN_BLOCK)
        e = min(t1, (blk + 1) * TOKEN_BLOCK)
        out[s - t0:e - t0] = z[s - blk * TOKEN_BLOCK:e - blk * TOKEN_BLOCK]
    return out


def _lr_draw(spec: LayerSpec, b: int, h: int, t0: int, t1: int, column: int = 0) -> np.ndarray:
    """Rates of tokens [t0, t1); column j > 0 (per-matrix rates) has its own stream."""
    out = np.empty(t1 - t0, dtype=np.float64)
    blk0, blk1 = t0 // TOKEN_BLOCK, (t1 - 1) // TOKEN_BLOCK
    for blk in range(blk0, blk1 + 1):
        g = _rng(spec.seed, _T_LR if column == 0 else _T_LR_COL + column, b, h, blk)
        if spec.lr_kind == "uniform":
            z = g.uniform(spec.lr_a, spec.lr_b, TOKEN_BLOCK)
        else:
            z = spec.lr_a / (1.0 + np.exp(-g.standard_normal(TOKEN_BLOCK)))
        s = max(t0, blk * TOKEN_BLOCK)
        e = min(t1, (blk + 1) * TOKEN_BLOCK)
        out[s - t0:e - t0] = z[s - blk * TOKEN_BLOCK:e - blk * TOKEN_BLOCK]
    return out


def _unit_rows(x: np.ndarray) -> np.ndarray:
    return x / np.sqrt((x * x).sum(axis=1, keepdims=True))


def head_tokens(spec: LayerSpec, b: int, h: int, t0: int = 0,
                t1: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Inputs of one (b, h) head for tokens [t0, t1).

    Q, K, V come back as (stored, exact) pairs; lr as fp32.
    """
    t1 = spec.T if t1 is None else t1
    q = _unit_rows(_token_draw(spec, _T_Q, b, h, t0, t1, spec.d))
    k = _unit_rows(_token_draw(spec, _T_K, b, h, t0, t1, spec.d))
    v = _token_draw(spec, _T_V, b, h, t0, t1, spec.d)
    out = {}
    for name, x in (("Q", q), ("K", k), ("V", v)):
        out[name], out[name + "64"] = to_storage(x, spec.dtype)
    if spec.lr_per_matrix:
        out["lr"] = round_fp32(np.stack([_lr_draw(spec, b, h, t0, t1, j) for j in range(spec.n_weights)],
                                        axis=1))
    else:
        out["lr"] = round_fp32(_lr_draw(spec, b, h, t0, t1))
    return out


def initial_weights(spec: LayerSpec) -> List[np.ndarray]:
    """Initial fast weights, fp32, each [H, out, in] (shared across the batch)."""
    ws = []
    for j, (o, i) in enumerate(spec.weight_shapes()):
        std = 1.0 / math.sqrt(i)
        w = np.stack([_rng(spec.seed, _T_W + j, h).standard_normal((o, i)) * std
                      for h in range(spec.H)])
        ws.append(round_fp32(w))
    return ws


def layer_inputs(spec: LayerSpec, exact: bool = True) -> Dict[str, object]:
    """All inputs of a workload.

    Returns a dict with Q, K, V (storage arrays [B, H, T, d]: float32 or uint16
    bf16 bits), lr (float32 [B, H, T]), W0 (list of float32 [H, out, in]),
    mask (uint8 [n_chunks]) and, when ``exact``, Q64/K64/V64 (fp64 values).
    """
    sdt = np.float32 if spec.dtype == "fp32" else np.uint16
    shp = (spec.B, spec.H, spec.T, spec.d)
    res: Dict[str, object] = {n: np.empty(shp, dtype=sdt) for n in ("Q", "K", "V")}
    if exact:
        for n in ("Q64", "K64", "V64"):
            res[n] = np.empty(shp, dtype=np.float64)
    res["lr"] = np.empty((spec.B, spec.H, spec.T) + ((spec.n_weights,) if spec.lr_per_matrix else ()),
                         dtype=np.float32)
    for b in range(spec.B):
        for h in range(spec.H):
            ht = head_tokens(spec, b, h)
            for n in ("Q", "K", "V"):
                res[n][b, h] = ht[n]
                if exact:
                    res[n + "64"][b, h] = ht[n + "64"]
            res["lr"][b, h] = ht["lr"]
    res["W0"] = initial_weights(spec)
    res["mask"] = spec.update_mask()
    return res
