"""The outer-loop backward (ttt_bwd) against the fp64 oracle's reverse mode,
which is itself pinned to central finite differences: the linear fast net with
plain gradient steps in shifted mode, inner-product and MSE loss, fp32 storage
(tolerance 1e-4, max relative error per tensor) and bf16 storage (2e-2)."""
import numpy as np
import pytest

from long_seq_models_chunked_b300 import abi, synth
from oracle import OracleCfg, linear_head_backward

pytestmark = pytest.mark.gpu

from parity import rel_err, to_device, to_f64  # noqa: E402

LIN = synth.WORKLOADS["linear_chunk64"]
CASES = {
    "mse_fp32": (LIN.replace(name="bwd_mse", B=2, H=2, T=300, chunk=64, dtype="fp32", seed=101), 1e-4),
    "ip_fp32_ragged_odd": (LIN.replace(name="bwd_ip", B=1, H=3, T=230, chunk=48, loss="ip", update="odd",
                                       dtype="fp32", step=0.7, seed=102), 1e-4),
    "mse_fp32_chunk1": (LIN.replace(name="bwd_c1", B=1, H=2, T=40, d=16, dh=16, chunk=1, dtype="fp32",
                                    seed=103), 1e-4),
    "mse_bf16_workload_shape": (LIN.replace(name="bwd_bf16", B=2, H=2, T=1024, seed=104), 2e-2),
}


def _run(spec, x, dO, dWf, per_batch):
    import torch
    dev = to_device(x, spec)
    holder = abi.cfg_from_spec(spec)
    cfg = holder.cfg
    cfg.w0_per_batch = 1 if per_batch else 0
    W0 = dev["W0"][0]
    if per_batch:
        W0 = W0.unsqueeze(0).expand(spec.B, -1, -1, -1).contiguous()
    tdt = torch.float32 if spec.dtype == "fp32" else torch.bfloat16
    dO_t = torch.from_numpy(dO.astype(np.float32)).to(tdt).cuda()
    dWf_t = torch.from_numpy(dWf.astype(np.float32)).cuda()
    dQ, dK, dV = (torch.empty_like(dev[n]) for n in ("Q", "K", "V"))
    dlr = torch.empty_like(dev["lr"])
    dW0 = torch.empty_like(W0)
    ws = torch.empty(abi.ttt_bwd_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    abi.ttt_bwd(cfg, dev["Q"], dev["K"], dev["V"], dev["lr"], W0, dO_t, dWf_t, dQ, dK, dV, dlr, dW0, ws)
    assert abi.ttt_status(ws) == abi.TTT_OK
    dO_exact = to_f64(dO_t, spec)
    return [to_f64(t, spec) for t in (dQ, dK, dV)] + [dlr.double().cpu().numpy(), dW0.double().cpu().numpy()], dO_exact


@pytest.mark.parametrize("per_batch", [False, True])
@pytest.mark.parametrize("name", list(CASES))
def test_backward_matches_oracle(name, per_batch):
    spec, tol = CASES[name]
    x = synth.layer_inputs(spec)
    rng = np.random.default_rng(7)
    dO = rng.standard_normal((spec.B, spec.H, spec.T, spec.d))
    dWf = rng.standard_normal((spec.B, spec.H, spec.d, spec.d))
    got, dO_exact = _run(spec, x, dO, dWf, per_batch)
    cfg = OracleCfg.from_spec(spec)
    ref_dW0 = np.zeros((spec.B, spec.H, spec.d, spec.d))
    for b in range(spec.B):
        for h in range(spec.H):
            r = linear_head_backward(cfg, x["Q64"][b, h], x["K64"][b, h], x["V64"][b, h], x["lr"][b, h],
                                     x["W0"][0][h].astype(np.float64), dO_exact[b, h], dWf[b, h])
            for k, name_k in enumerate(("dQ", "dK", "dV", "dlr")):
                err = rel_err(got[k][b, h], r[k])
                assert err <= tol, (name, name_k, b, h, err)
            ref_dW0[b, h] = r[4]
    want = ref_dW0 if per_batch else ref_dW0.sum(axis=0)
    assert rel_err(got[4], want) <= tol, (name, "dW0", rel_err(got[4], want))


def test_backward_is_deterministic():
    import torch
    spec, _ = CASES["mse_fp32"]
    x = synth.layer_inputs(spec, exact=False)
    rng = np.random.default_rng(8)
    dO = rng.standard_normal((spec.B, spec.H, spec.T, spec.d))
    dWf = rng.standard_normal((spec.B, spec.H, spec.d, spec.d))
    a, _ = _run(spec, x, dO, dWf, False)
    b, _ = _run(spec, x, dO, dWf, False)
    torch.cuda.synchronize()
    assert all(np.array_equal(p, q) for p, q in zip(a, b))
