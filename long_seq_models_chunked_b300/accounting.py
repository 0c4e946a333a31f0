"""Fixed FLOP and byte accounting of one TTT-layer call.

The counts are the work the method itself must do (the tutorial page's
O(n d^2) cost per token, "Test-Time Training layers" §6), independent of how a
kernel schedules it. They are what throughput and roofline fractions divide by.
"""
from __future__ import annotations

from .synth import LayerSpec


def algorithmic_flops(spec: LayerSpec) -> float:
    """Fixed FLOP accounting of one layer call (GEMM + Newton-Schulz).

    SwiGLU: 6*d*dh per applied token and 12*d*dh per updated token (inner-product
    loss; MSE adds 2*d*dh for the extra forward of W2); Newton-Schulz:
    3 * iters * (4 m^2 n + 2 m^3) per update with m = min(d, dh), n = max(d, dh).
    Linear: 2 d^2 per applied token and 4 d^2 per updated token.
    Elementwise, norm and activation work is not counted.
    """
    mask = spec.update_mask()
    upd_tokens = 0
    for c in range(spec.n_chunks):
        if mask[c]:
            upd_tokens += min(spec.T, (c + 1) * spec.chunk) - c * spec.chunk
    n_upd = int(mask.sum())
    heads = spec.B * spec.H
    if spec.fast_net == "swiglu":
        per_upd = 12 if spec.loss == "ip" else 14
        f = 6.0 * spec.d * spec.dh * spec.T + per_upd * spec.d * spec.dh * upd_tokens
        if spec.muon:
            m, n = min(spec.d, spec.dh), max(spec.d, spec.dh)
            f += n_upd * 3 * spec.ns_iters * (4.0 * m * m * n + 2.0 * m ** 3)
    else:
        f = 2.0 * spec.d ** 2 * spec.T + 4.0 * spec.d ** 2 * upd_tokens
        if spec.muon:
            f += n_upd * spec.ns_iters * (6.0 * spec.d ** 3)
    return heads * f
