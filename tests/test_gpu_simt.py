"""GPU parity of the fp32 SIMT path against the fp64 oracle (tolerance 1e-4
for fp32 storage; bf16 outputs add the bf16 rounding of O)."""
import numpy as np
import pytest

from long_seq_models_chunked_b300 import synth

pytestmark = pytest.mark.gpu

from parity import compare, run_gpu, run_oracle  # noqa: E402

SIMT = 1
TINY = synth.WORKLOADS["tiny_fp32"]

CASES = {
    "tiny_fp32": TINY,
    "tiny_muon": TINY.replace(name="tiny_muon", muon=True, seed=31),
    "tiny_single": TINY.replace(name="tiny_single", mode="single", chunk=256, muon=True, seed=32),
    "tiny_mse": TINY.replace(name="tiny_mse", loss="mse", seed=33),
    "tiny_ragged_odd": TINY.replace(name="tiny_ragged_odd", T=230, chunk=48, update="odd",
                                    muon=True, seed=34),
    "tall_hidden": TINY.replace(name="tall_hidden", d=48, dh=24, B=2, H=1, T=96, chunk=32,
                                muon=True, seed=35),
    "linear_mse": synth.WORKLOADS["linear_chunk64"].replace(
        name="linear_mse", B=2, H=3, T=640, dtype="fp32", seed=36),
    "linear_ip_muon": synth.WORKLOADS["linear_chunk64"].replace(
        name="linear_ip_muon", B=1, H=2, T=256, d=32, dh=32, loss="ip", muon=True,
        wnorm=True, dtype="fp32", seed=37),
    # LaCT page §2.2.1: Muon against a momentum optimiser; per-matrix rates
    "momentum_muon": TINY.replace(name="momentum_muon", muon=True, momentum=0.9, seed=39),
    "momentum_sgd": TINY.replace(name="momentum_sgd", momentum=0.8, seed=40),
    "lr_per_matrix": TINY.replace(name="lr_per_matrix", muon=True, lr_per_matrix=True, seed=41),
    "momentum_lr_mse_odd": TINY.replace(name="momentum_lr_mse_odd", loss="mse", momentum=0.5,
                                        lr_per_matrix=True, T=230, chunk=48, update="odd", seed=42),
    "linear_momentum": synth.WORKLOADS["linear_chunk64"].replace(
        name="linear_momentum", B=1, H=2, T=512, dtype="fp32", momentum=0.9, lr_per_matrix=True, seed=43),
    # inclusive order (tutorial page §3): each query sees its own token's update
    "inclusive_mse": TINY.replace(name="inclusive_mse", mode="inclusive", loss="mse", wnorm=False, seed=44),
    "inclusive_ip_rates": TINY.replace(name="inclusive_ip_rates", mode="inclusive", wnorm=False,
                                       lr_per_matrix=True, T=230, chunk=48, update="odd", seed=45),
    "inclusive_chunk1": TINY.replace(name="inclusive_chunk1", mode="inclusive", wnorm=False, loss="mse",
                                     T=40, chunk=1, seed=46),
    "inclusive_block_tail": TINY.replace(name="inclusive_block_tail", mode="inclusive", wnorm=False, T=300,
                                         chunk=150, step=0.5, seed=47),   # blocks of 64 inside a chunk
    "inclusive_linear": synth.WORKLOADS["linear_chunk64"].replace(
        name="inclusive_linear", B=2, H=2, T=512, dtype="fp32", mode="inclusive", seed=48),
}


@pytest.mark.parametrize("name", list(CASES))
def test_simt_fp32_matches_oracle(name):
    spec = CASES[name]
    x = synth.layer_inputs(spec)
    compare(spec, run_gpu(spec, x, impl=SIMT), run_oracle(spec, x), 1e-4)


def test_simt_inclusive_bf16_linear_workload_heads():
    """The small-chunk linear workload's shape (64 x 64 weights, chunks of 64,
    MSE) in the inclusive order, bf16 storage, sampled heads against the oracle."""
    from parity import full_workload_check
    spec = synth.WORKLOADS["linear_chunk64"].replace(name="inclusive_lin_wl", B=2, H=4, T=2048, mode="inclusive")
    full_workload_check(spec, [(0, 0), (1, 3)], 2e-2, impl=SIMT)


def test_simt_bf16_storage_matches_oracle():
    spec = TINY.replace(name="tiny_bf16", dtype="bf16", muon=True, seed=38)
    x = synth.layer_inputs(spec)
    O, Wf = run_gpu(spec, x, impl=SIMT)
    Or, Wr = run_oracle(spec, x)
    errs = compare(spec, (O, Wf), (Or, Wr), 2e-2)
    assert max(errs[k] for k in errs if k != "O") <= 1e-4, errs
    assert errs["O"] <= 2.0 ** -8, errs          # bf16 rounding of the output only


def test_simt_is_deterministic():
    spec = CASES["tiny_muon"]
    x = synth.layer_inputs(spec)
    a = run_gpu(spec, x, impl=SIMT)
    b = run_gpu(spec, x, impl=SIMT)
    assert np.array_equal(a[0], b[0]) and all(np.array_equal(p, q) for p, q in zip(a[1], b[1]))
