"""ttt_fwd_host: the layer on host buffers (inputs copied in, outputs copied
back, chunk-pipelined on the tensor-core path) gives exactly what ttt_fwd gives
on device buffers: the same kernels run on the same values, so the results are
bitwise equal, with pinned and with pageable host memory."""
import numpy as np
import pytest

from long_seq_models_chunked_b300 import abi, synth

pytestmark = pytest.mark.gpu

from parity import to_device  # noqa: E402


def _host_call(holder, spec, x, pinned):
    import torch
    cfg = holder.cfg

    def host(a, bf=False):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if bf:
            t = t.view(torch.bfloat16)
        return t.pin_memory() if pinned else t

    bf = spec.dtype == "bf16"
    Q, K, V = (host(x[n], bf) for n in ("Q", "K", "V"))
    lr = host(x["lr"])
    W0 = [host(w) for w in x["W0"]]
    O = torch.empty(Q.shape, dtype=Q.dtype)
    Wf = [torch.empty((cfg.B, cfg.H) + s, dtype=torch.float32) for s in abi.weight_shapes(cfg)]
    if pinned:
        O = O.pin_memory()
        Wf = [w.pin_memory() for w in Wf]
    arena = torch.empty(abi.ttt_host_arena_bytes(cfg), dtype=torch.uint8, device="cuda")
    w0 = W0 + [None] * (3 - len(W0))
    wf = Wf + [None] * (3 - len(Wf))
    abi.ttt_fwd_host(cfg, Q, K, V, lr, w0[0], w0[1], w0[2], O, wf[0], wf[1], wf[2], arena)
    return O, Wf


CASES = [
    ("tc_ragged_odd", abi.TTT_IMPL_TC,
     synth.LayerSpec("host_tc", B=2, H=2, T=700, d=64, dh=128, chunk=200, update="odd", seed=81)),
    ("tc_single", abi.TTT_IMPL_TC,
     synth.LayerSpec("host_tc1", B=1, H=2, T=512, d=64, dh=128, chunk=512, mode="single", seed=82)),
    ("linear", abi.TTT_IMPL_LINEAR,
     synth.WORKLOADS["linear_chunk64"].replace(name="host_lin", B=2, H=2, T=640, seed=83)),
    ("simt", abi.TTT_IMPL_SIMT, synth.WORKLOADS["tiny_fp32"].replace(name="host_simt", muon=True, seed=84)),
]


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("name,impl,spec", CASES)
def test_host_entry_equals_device_entry(name, impl, spec, pinned):
    import torch
    x = synth.layer_inputs(spec, exact=False)
    holder = abi.cfg_from_spec(spec, impl=impl)
    dev = to_device(x, spec)
    O_d, Wf_d = abi.layer(holder, dev["Q"], dev["K"], dev["V"], dev["lr"], dev["W0"])
    torch.cuda.synchronize()
    O_h, Wf_h = _host_call(holder, spec, x, pinned)
    assert torch.equal(O_h.view(torch.int16) if O_h.dtype == torch.bfloat16 else O_h,
                       (O_d.cpu().view(torch.int16) if O_d.dtype == torch.bfloat16 else O_d.cpu())), name
    for a, b in zip(Wf_h, Wf_d):
        assert torch.equal(a, b.cpu()), name
