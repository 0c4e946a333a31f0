"""Context parallelism on the GPU (LaCT page, "Large Chunk Test-Time Training",
§2.2.2): every chunk's tokens split into shards, each shard's partial gradient
from the same weights, the partials summed, the same update everywhere.

One GPU stands in for the ranks: their steps run one after another in one
process (cp.run_lockstep), each rank on its own workspace, the partials summed
on the device. Nothing runs concurrently and no kernel waits on another."""
import numpy as np
import pytest

from long_seq_models_chunked_b300 import abi, cp, synth

pytestmark = pytest.mark.gpu

from parity import compare, run_oracle, to_device, to_f64  # noqa: E402

TOL = 2e-2


def _shard_tokens(t, C, R, r):
    """Rank r's local tensor: its 1/R slice of every chunk of C tokens (dim 2)."""
    import torch
    Cl = C // R
    T = t.shape[2]
    return torch.cat([t[:, :, c + r * Cl:c + (r + 1) * Cl] for c in range(0, T, C)], dim=2).contiguous()


def _run_cp(spec, x, R):
    import torch
    dev = to_device(x, spec)
    C = spec.chunk
    Cl = C // R
    local = spec.replace(chunk=Cl, T=(spec.T // C) * Cl)
    holder = abi.cfg_from_spec(local, impl=abi.TTT_IMPL_TC)
    shards, steps, outs, ins = [], [], [], []
    for r in range(R):
        Q, K, V, lr = (_shard_tokens(dev[n], C, R, r) for n in ("Q", "K", "V", "lr"))
        O = torch.empty_like(Q)
        sh = cp.Shard(holder, dev["W0"], local.T)
        shards.append(sh)
        outs.append(O)
        ins.append((Q, K, V, lr))
        steps.append(cp.rank_steps(sh, Q, K, V, lr, O, local.T, Cl, spec.mode == "shifted", spec.update_mask()))
    cp.run_lockstep(steps)
    Wfs = [sh.end() for sh in shards]
    torch.cuda.synchronize()
    for sh in shards:
        assert sh.status() == abi.TTT_OK
    # every rank holds the same weights
    for Wf in Wfs[1:]:
        for a, b in zip(Wf, Wfs[0]):
            assert torch.equal(a, b)
    O = torch.empty_like(dev["Q"])
    for r in range(R):
        for c0 in range(0, spec.T, C):
            O[:, :, c0 + r * Cl:c0 + (r + 1) * Cl] = outs[r][:, :, (c0 // C) * Cl:(c0 // C + 1) * Cl]
    return to_f64(O, spec), [w.double().cpu().numpy() for w in Wfs[0]]


CASES = {
    # one chunk over every token (the image-set layer's shape, scaled down)
    "single_2": (synth.LayerSpec("cp_single", B=1, H=2, T=8192, d=192, dh=384, chunk=8192, mode="single",
                                 lr_a=0.005, seed=81), 2),
    "single_4": (synth.LayerSpec("cp_single4", B=1, H=2, T=4096, d=64, dh=128, chunk=4096, mode="single",
                                 seed=82), 4),
    # shifted chunks, each split over the ranks; odd chunks update
    "shifted_2": (synth.LayerSpec("cp_shifted", B=2, H=2, T=1024, d=64, dh=128, chunk=256, update="odd",
                                  seed=83), 2),
    "shifted_3_momentum": (synth.LayerSpec("cp_shifted3", B=1, H=2, T=768, d=128, dh=256, chunk=384,
                                           momentum=0.9, lr_per_matrix=True, seed=84), 3),
    # the language-model layer's shapes over two chunks
    "lm_2": (synth.WORKLOADS["lm_chunk2k"].replace(name="cp_lm", B=1, H=2, T=4096, seed=85), 2),
}


@pytest.mark.parametrize("name", list(CASES))
def test_context_parallel_layer_matches_oracle(name):
    spec, R = CASES[name]
    x = synth.layer_inputs(spec)
    compare(spec, _run_cp(spec, x, R), run_oracle(spec, x), TOL)


def test_shard_gradients_sum_to_the_chunk_gradient():
    """The partials of three shards, from the same weights, sum to the gradient
    of the whole chunk (fp32 sums in another order)."""
    import torch
    spec = synth.LayerSpec("cp_sum", B=1, H=3, T=3 * 640, d=128, dh=256, chunk=3 * 640, seed=86)
    x = synth.layer_inputs(spec, exact=False)
    dev = to_device(x, spec)
    holder = abi.cfg_from_spec(spec, impl=abi.TTT_IMPL_TC)
    sh = cp.Shard(holder, dev["W0"], spec.T)
    whole = sh.grad(dev["K"], dev["V"], dev["lr"], 0, spec.T).clone()
    parts = torch.zeros_like(whole)
    for s in (0, 640, 1280):
        parts += sh.grad(dev["K"], dev["V"], dev["lr"], s, 640)
    torch.cuda.synchronize()
    err = ((parts - whole).abs().max() / whole.abs().max()).item()
    assert err <= 1e-5, err


def test_cp_calls_reject_bad_ranges_before_launch():
    import torch
    spec = synth.LayerSpec("cp_bad", B=1, H=2, T=512, d=64, dh=128, chunk=256, seed=87)
    x = synth.layer_inputs(spec, exact=False)
    dev = to_device(x, spec)
    holder = abi.cfg_from_spec(spec, impl=abi.TTT_IMPL_TC)
    sh = cp.Shard(holder, dev["W0"], spec.T)
    n0 = abi.ttt_launch_count()
    for start, n in ((0, 257), (-1, 10), (500, 20), (0, 0)):
        with pytest.raises(abi.TTTError) as err:
            sh.grad(dev["K"], dev["V"], dev["lr"], start, n)
        assert err.value.code == abi.TTT_ERR_ARG
    with pytest.raises(abi.TTTError) as err:
        abi.ttt_cp_update(holder.cfg, sh.G.cpu(), sh.ws)   # host memory
    assert err.value.code == abi.TTT_ERR_ARG
    assert abi.ttt_launch_count() == n0
    torch.cuda.synchronize()
