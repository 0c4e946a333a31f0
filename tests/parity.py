"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded inputs, and compare them."""
from __future__ import annotations

import numpy as np

from long_seq_models_chunked_b300 import synth
from oracle import OracleCfg, ttt_layer


def rel_err(x: np.ndarray, y: np.ndarray) -> float:
    """max_i |x_i - y_i| / max_i |y_i|  (per output tensor)."""
    den = np.abs(y).max()
    return float(np.abs(x - y).max() / (den if den > 0 else 1.0))


def to_device(x: dict, spec, device="cuda"):
    import torch
    out = {}
    for n in ("Q", "K", "V"):
        t = torch.from_numpy(np.ascontiguousarray(x[n]))
        if spec.dtype == "bf16":
            t = t.view(torch.bfloat16)
        out[n] = t.to(device)
    out["lr"] = torch.from_numpy(x["lr"]).to(device)
    out["W0"] = [torch.from_numpy(w).to(device) for w in x["W0"]]
    return out


def to_f64(t, spec) -> np.ndarray:
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return synth.bf16_bits_to_f64(t.view(torch.int16).numpy().view(np.uint16))
    return t.double().numpy()


def run_gpu(spec, x: dict, impl: int = 0, **kw):
    from long_seq_models_chunked_b300 import abi
    dev = to_device(x, spec)
    holder = abi.cfg_from_spec(spec, impl=impl, **kw)
    O, Wf = abi.layer(holder, dev["Q"], dev["K"], dev["V"], dev["lr"], dev["W0"])
    return to_f64(O, spec), [w.double().cpu().numpy() for w in Wf]


def run_oracle(spec, x: dict, heads=None, block: int = 0):
    cfg = OracleCfg.from_spec(spec)
    return ttt_layer(cfg, x["Q64"], x["K64"], x["V64"], x["lr"], x["W0"], heads=heads,
                     block=block)


def compare(spec, gpu, ref, tol: float):
    """Per-tensor relative errors; asserts each is within tol."""
    O, Wf = gpu
    Or, Wr = ref
    errs = {"O": rel_err(O, Or)}
    for j, (a, b) in enumerate(zip(Wf, Wr)):
        errs[f"W{j + 1}"] = rel_err(a, b)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{spec.name}: {errs} (tol {tol})"
    return errs


def full_workload_check(spec, heads, tol: float, block: int = 0, **gpu_kw):
    """Run a full-size workload on the GPU and compare the sampled (b, h) heads
    with the oracle, head by head (the oracle regenerates only those heads' exact
    inputs). Returns {(b, h): errs}."""
    x = synth.layer_inputs(spec, exact=False)
    O, Wf = run_gpu(spec, x, **gpu_kw)
    cfg = OracleCfg.from_spec(spec)
    from oracle import ttt_head
    out = {}
    for (b, h) in heads:
        ht = synth.head_tokens(spec, b, h)
        w0 = [w[h].astype(np.float64) for w in x["W0"]]
        Or, Wr = ttt_head(cfg, ht["Q64"], ht["K64"], ht["V64"], ht["lr"], w0, block=block)
        out[(b, h)] = compare(spec, (O[b, h], [w[b, h] for w in Wf]), (Or, Wr), tol)
    return out
