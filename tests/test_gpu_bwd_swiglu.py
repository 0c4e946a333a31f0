"""The outer-loop backward of the SwiGLU net (ttt_bwd_swiglu) against the fp64
oracle's reverse mode (automatic differentiation of the forward, pinned to
central finite differences): plain gradient steps in shifted mode, the
inner-product and MSE losses, fp32 storage (tolerance 1e-4, max relative error
per tensor) and bf16 storage (2e-2); W0 shared over the batch or one per batch."""
import numpy as np
import pytest

from long_seq_models_chunked_b300 import abi, synth
from oracle import OracleCfg, swiglu_head_backward

pytestmark = pytest.mark.gpu

from parity import rel_err, to_device, to_f64  # noqa: E402

TINY = synth.WORKLOADS["tiny_fp32"].replace(wnorm=False, muon=False, loss="ip")
CASES = {
    "fp32": (TINY.replace(name="sbwd_fp32", B=2, H=2, T=150, chunk=32, d=16, dh=32, step=0.8, seed=111), 1e-4),
    "fp32_ragged_odd": (TINY.replace(name="sbwd_odd", B=1, H=2, T=97, chunk=20, d=8, dh=24, update="odd",
                                     step=0.8, seed=112), 1e-4),
    "fp32_chunk1": (TINY.replace(name="sbwd_c1", B=1, H=1, T=24, chunk=1, d=8, dh=16, step=0.5, seed=113), 1e-4),
    "bf16": (TINY.replace(name="sbwd_bf16", B=2, H=1, T=128, chunk=32, d=32, dh=64, dtype="bf16", step=0.8,
                          seed=114), 2e-2),
    "mse_fp32": (TINY.replace(name="sbwd_mse", B=2, H=2, T=150, chunk=32, d=16, dh=32, loss="mse", step=0.5,
                              seed=115), 1e-4),
    "mse_fp32_ragged_odd": (TINY.replace(name="sbwd_mse_odd", B=1, H=2, T=97, chunk=20, d=8, dh=24, loss="mse",
                                         update="odd", step=0.5, seed=116), 1e-4),
    "mse_bf16": (TINY.replace(name="sbwd_mse_bf16", B=1, H=2, T=128, chunk=32, d=32, dh=64, loss="mse",
                              dtype="bf16", step=0.5, seed=117), 2e-2),
}


def _run(spec, x, dO, dWf, per_batch):
    import torch
    dev = to_device(x, spec)
    holder = abi.cfg_from_spec(spec)
    cfg = holder.cfg
    cfg.w0_per_batch = 1 if per_batch else 0
    W0 = dev["W0"]
    if per_batch:
        W0 = [w.unsqueeze(0).expand(spec.B, -1, -1, -1).contiguous() for w in W0]
    tdt = torch.float32 if spec.dtype == "fp32" else torch.bfloat16
    dO_t = torch.from_numpy(dO.astype(np.float32)).to(tdt).cuda()
    dWf_t = [torch.from_numpy(w.astype(np.float32)).cuda() for w in dWf]
    dQ, dK, dV = (torch.empty_like(dev[n]) for n in ("Q", "K", "V"))
    dlr = torch.empty_like(dev["lr"])
    dW0 = [torch.empty_like(w) for w in W0]
    ws = torch.empty(abi.ttt_bwd_swiglu_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    abi.ttt_bwd_swiglu(cfg, dev["Q"], dev["K"], dev["V"], dev["lr"], W0, dO_t, dWf_t, dQ, dK, dV, dlr, dW0, ws)
    assert abi.ttt_status(ws) == abi.TTT_OK
    dO_exact = to_f64(dO_t, spec)
    return ([to_f64(t, spec) for t in (dQ, dK, dV)] + [dlr.double().cpu().numpy()] +
            [w.double().cpu().numpy() for w in dW0]), dO_exact


@pytest.mark.parametrize("per_batch", [False, True])
@pytest.mark.parametrize("name", list(CASES))
def test_swiglu_backward_matches_oracle(name, per_batch):
    spec, tol = CASES[name]
    x = synth.layer_inputs(spec)
    rng = np.random.default_rng(9)
    dO = rng.standard_normal((spec.B, spec.H, spec.T, spec.d))
    dWf = [rng.standard_normal((spec.B,) + w.shape) for w in x["W0"]]
    got, dO_exact = _run(spec, x, dO, dWf, per_batch)
    cfg = OracleCfg.from_spec(spec)
    ref_dW0 = [np.zeros((spec.B,) + w.shape) for w in x["W0"]]
    for b in range(spec.B):
        for h in range(spec.H):
            W0 = tuple(w[h].astype(np.float64) for w in x["W0"])
            r = swiglu_head_backward(cfg, x["Q64"][b, h], x["K64"][b, h], x["V64"][b, h], x["lr"][b, h], W0,
                                     dO_exact[b, h], tuple(w[b, h] for w in dWf))
            for k, name_k in enumerate(("dQ", "dK", "dV", "dlr")):
                err = rel_err(got[k][b, h], r[k])
                assert err <= tol, (name, name_k, b, h, err)
            for j in range(3):
                ref_dW0[j][b, h] = r[4][j]
    for j in range(3):
        want = ref_dW0[j] if per_batch else ref_dW0[j].sum(axis=0)
        assert rel_err(got[4 + j], want) <= tol, (name, "dW0_%d" % (j + 1), rel_err(got[4 + j], want))


def test_swiglu_backward_is_deterministic():
    spec, _ = CASES["fp32"]
    x = synth.layer_inputs(spec, exact=False)
    rng = np.random.default_rng(10)
    dO = rng.standard_normal((spec.B, spec.H, spec.T, spec.d))
    dWf = [rng.standard_normal((spec.B,) + w.shape) for w in x["W0"]]
    a, _ = _run(spec, x, dO, dWf, False)
    b, _ = _run(spec, x, dO, dWf, False)
    assert all(np.array_equal(p, q) for p, q in zip(a, b))
