"""The allocation-free entry point ttt_fwd_static_scratch.

It exists for callers that receive their input and output buffers but may not
allocate device memory (a plugin inside a host application that keeps all
device memory in its own pool, or a loop where cudaMalloc/cudaFree and the
device-wide synchronisation they can cause are not allowed). It runs the fp32
SIMT kernel family on a scratch array the library holds, and must give what
ttt_fwd gives with a caller-provided workspace.

Two calls in a row, on different workloads, check that the contents the first
call leaves in the shared array do not leak into the second. This file is
collected last so that a run stopping at the first failure has already run
every other test.
"""
import numpy as np
import pytest

from long_seq_models_chunked_b300 import abi, synth

pytestmark = pytest.mark.gpu

TOL = 1e-4   # the fp32 SIMT tier's tolerance


def _inputs(spec):
    import torch
    x = synth.layer_inputs(spec, exact=False)
    dev = {}
    for n in ("Q", "K", "V"):
        t = torch.from_numpy(np.ascontiguousarray(x[n]))
        if spec.dtype == "bf16":
            t = t.view(torch.bfloat16)
        dev[n] = t.cuda()
    dev["lr"] = torch.from_numpy(x["lr"]).cuda()
    dev["W0"] = [torch.from_numpy(w).cuda() for w in x["W0"]]
    return dev


def _outputs(cfg, like):
    import torch
    O = torch.full_like(like, float("nan"))
    Wf = [torch.full((cfg.B, cfg.H) + s, float("nan"), dtype=torch.float32, device=like.device)
          for s in abi.weight_shapes(cfg)]
    return O, Wf


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def _static_call(holder, x):
    import torch
    cfg = holder.cfg
    O, Wf = _outputs(cfg, x["Q"])
    status = torch.full((1,), -99, dtype=torch.int32, device="cuda")
    w0 = x["W0"] + [None] * (3 - len(x["W0"]))
    wf = Wf + [None] * (3 - len(Wf))
    abi.ttt_fwd_static_scratch(cfg, x["Q"], x["K"], x["V"], x["lr"], w0[0], w0[1], w0[2], O,
                               wf[0], wf[1], wf[2], status)
    torch.cuda.synchronize()
    assert int(status.item()) == abi.TTT_OK
    return O, Wf


SPECS = [
    synth.WORKLOADS["tiny_fp32"].replace(name="static_a", muon=True, seed=91),
    synth.WORKLOADS["tiny_fp32"].replace(name="static_b", T=230, chunk=48, update="odd", d=48, dh=96,
                                         muon=True, seed=92),
]


def test_static_scratch_matches_workspace_entry_point_twice_in_a_row():
    import torch
    for spec in SPECS:
        holder = abi.cfg_from_spec(spec, impl=abi.TTT_IMPL_SIMT)
        x = _inputs(spec)
        O_s, Wf_s = _static_call(holder, x)
        O_w, Wf_w = abi.layer(holder, x["Q"], x["K"], x["V"], x["lr"], x["W0"])
        torch.cuda.synchronize()
        errs = [_rel(O_s, O_w)] + [_rel(a, b) for a, b in zip(Wf_s, Wf_w)]
        assert max(errs) <= TOL, (spec.name, errs)


def test_static_scratch_matches_oracle():
    from parity import compare, run_oracle, to_f64
    for spec in SPECS:
        holder = abi.cfg_from_spec(spec, impl=abi.TTT_IMPL_SIMT)
        host = synth.layer_inputs(spec)
        O_s, Wf_s = _static_call(holder, _inputs(spec))
        gpu = (to_f64(O_s, spec), [w.double().cpu().numpy() for w in Wf_s])
        compare(spec, gpu, run_oracle(spec, host), TOL)


def test_static_scratch_rejects_requests_beyond_its_size():
    import torch
    spec = synth.WORKLOADS["lm_chunk2k"].replace(T=4096)
    holder = abi.cfg_from_spec(spec, impl=abi.TTT_IMPL_SIMT)
    assert abi.ttt_workspace_bytes(holder.cfg) > abi.TTT_STATIC_SCRATCH_BYTES
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    w = torch.empty(16, dtype=torch.float32, device="cuda")
    rc = abi.ttt_fwd_static_scratch(holder.cfg, t, t, t, w, w, w, w, t, w, w, w, None, check=False)
    assert rc == abi.TTT_ERR_SCRATCH_LIMIT
    assert "TTT_STATIC_SCRATCH_BYTES" in abi.ttt_strerror(rc)
