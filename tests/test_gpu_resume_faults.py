"""GPU checks of the host-visible contract around the layer:

* resume: the layer over tokens [0, T1) and then over [T1, T) with the first
  call's final weights as per-(b, h) initial weights (w0_per_batch) equals one
  call over [0, T), split at a chunk boundary (the fast weights are the whole
  state the pages' chunks share). The weight norm restores the row norms of the
  call's own W0, which after the first call are those of the original W0 up to
  fp32 rounding, so the two runs agree to fp32 rounding, not bit for bit;
* non-finite input: with check_finite the status word reports TTT_ERR_NONFINITE
  and the next call on clean inputs succeeds.
"""
import numpy as np
import pytest

from long_seq_models_chunked_b300 import abi, synth

pytestmark = pytest.mark.gpu

from parity import to_device  # noqa: E402


def _call(spec, dev, T0, T1, W0, per_batch, impl):
    import torch
    sub = spec.replace(T=T1 - T0)
    holder = abi.cfg_from_spec(sub, impl=impl)
    holder.cfg.w0_per_batch = 1 if per_batch else 0
    cut = {n: dev[n][:, :, T0:T1].contiguous() for n in ("Q", "K", "V")}
    lr = dev["lr"][:, :, T0:T1].contiguous()
    O, Wf = abi.layer(holder, cut["Q"], cut["K"], cut["V"], lr, W0)
    torch.cuda.synchronize()
    return O, Wf


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.abs(a - b).max() / np.abs(b).max())


@pytest.mark.parametrize("impl,spec", [
    (abi.TTT_IMPL_TC, synth.LayerSpec("resume_tc", B=2, H=2, T=768, d=64, dh=128, chunk=128, seed=71)),
    (abi.TTT_IMPL_LINEAR, synth.WORKLOADS["linear_chunk64"].replace(name="resume_lin", B=2, H=2, T=1024,
                                                                     seed=72)),
    (abi.TTT_IMPL_SIMT, synth.WORKLOADS["tiny_fp32"].replace(name="resume_simt", muon=True, seed=73)),
])
def test_resume_at_a_chunk_boundary_equals_one_call(impl, spec):
    x = synth.layer_inputs(spec, exact=False)
    dev = to_device(x, spec)
    T1 = (spec.T // spec.chunk // 2) * spec.chunk
    O_all, W_all = _call(spec, dev, 0, spec.T, dev["W0"], False, impl)
    O_a, W_a = _call(spec, dev, 0, T1, dev["W0"], False, impl)
    O_b, W_b = _call(spec, dev, T1, spec.T, [w.contiguous() for w in W_a], True, impl)
    import torch
    O_two = torch.cat([O_a, O_b], dim=2)
    w_errs = [_rel(b, a) for a, b in zip(W_all, W_b)]
    o_err = _rel(O_two.float(), O_all.float())
    if spec.dtype == "fp32":
        assert max(w_errs + [o_err]) <= 1e-4, (o_err, w_errs)
    else:
        # fp32 state; O is bf16, where a last-bit difference is 2^-8 of that element
        assert max(w_errs) <= 2e-3 and o_err <= 1e-2, (o_err, w_errs)


@pytest.mark.parametrize("impl,spec", [
    (abi.TTT_IMPL_TC, synth.LayerSpec("nan_tc", B=1, H=2, T=256, d=64, dh=128, chunk=128, seed=74)),
    (abi.TTT_IMPL_SIMT, synth.WORKLOADS["tiny_fp32"].replace(name="nan_simt", seed=75)),
])
def test_non_finite_input_is_reported_and_the_next_call_succeeds(impl, spec):
    import torch
    x = synth.layer_inputs(spec, exact=False)
    dev = to_device(x, spec)
    bad = dev["K"].clone()
    bad[0, 1, 17, 3] = float("nan")
    holder = abi.cfg_from_spec(spec, impl=impl, check_finite=True)
    with pytest.raises(abi.TTTError) as err:
        abi.layer(holder, dev["Q"], bad, dev["V"], dev["lr"], dev["W0"])
    assert err.value.code == abi.TTT_ERR_NONFINITE
    torch.cuda.synchronize()
    O, Wf = abi.layer(holder, dev["Q"], dev["K"], dev["V"], dev["lr"], dev["W0"])
    torch.cuda.synchronize()
    assert torch.isfinite(O.float()).all() and all(torch.isfinite(w).all() for w in Wf)


@pytest.mark.parametrize("where", ["pinned", "pageable"])
def test_host_memory_is_rejected_before_any_launch(where):
    """Every tensor must be device memory of the current device (the kernels
    read it through TMA tensor maps): host memory passed as Q is TTT_ERR_ARG,
    returned before anything is launched or written."""
    import torch
    spec = synth.LayerSpec("hostptr", B=1, H=2, T=256, d=64, dh=128, chunk=128, seed=76)
    x = synth.layer_inputs(spec, exact=False)
    dev = to_device(x, spec)
    holder = abi.cfg_from_spec(spec, impl=abi.TTT_IMPL_TC)
    cfg = holder.cfg
    hq = dev["Q"].cpu()
    if where == "pinned":
        hq = hq.pin_memory()
    O = torch.empty_like(dev["Q"])
    Wf = [torch.empty((cfg.B, cfg.H) + s, dtype=torch.float32, device="cuda") for s in abi.weight_shapes(cfg)]
    ws = torch.zeros(abi.ttt_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    n0 = abi.ttt_launch_count()
    rc = abi.ttt_fwd(cfg, hq, dev["K"], dev["V"], dev["lr"], *dev["W0"], O, *Wf, ws, check=False)
    assert rc == abi.TTT_ERR_ARG
    torch.cuda.synchronize()
    assert abi.ttt_launch_count() == n0
    assert int(ws[:4].view(torch.int32).item()) == 0
