"""GPU parity of the bf16 tensor-core path against the fp64 oracle on the same
seeded inputs (max relative error per output tensor <= 2e-2).

SPLIT precision (the default) carries every operand of the weight-update path
as a bf16 hi/lo pair; SINGLE precision uses one bf16 (fp16 in Newton-Schulz)
operand per product and is checked on short sequences only, where few updates
have compounded."""
import numpy as np
import pytest

from long_seq_models_chunked_b300 import abi, synth

pytestmark = pytest.mark.gpu

from parity import compare, full_workload_check, run_gpu, run_oracle  # noqa: E402

TC = abi.TTT_IMPL_TC
SINGLE = abi.TTT_PREC_SINGLE
TOL = 2e-2
BASE = synth.LayerSpec("tc_small", B=1, H=2, T=512, d=64, dh=128, chunk=128, seed=41)

CASES = {
    "small_muon": BASE,
    "small_sgd": BASE.replace(name="small_sgd", muon=False, seed=42),
    "small_single": BASE.replace(name="small_single", mode="single", chunk=512, seed=43),
    "small_odd_ragged": BASE.replace(name="small_odd_ragged", T=700, chunk=200, update="odd", seed=44),
    "small_no_wnorm": BASE.replace(name="small_no_wnorm", wnorm=False, step=0.5, seed=47),
    "d192_split_k": BASE.replace(name="d192_split_k", d=192, dh=384, T=8192, chunk=8192, mode="single",
                                 lr_a=0.005, seed=45),
    "multi_head_batch": BASE.replace(name="multi_head_batch", B=2, H=3, d=128, dh=256, T=384, seed=46),
    "long_small": BASE.replace(name="long_small", T=2048, chunk=128, seed=48),   # 16 updates
    # d and dh multiples of 256: Newton-Schulz on CTA-pair (cta_group::2) tiles
    "pair_d256": BASE.replace(name="pair_d256", B=2, H=2, d=256, dh=512, T=1024, chunk=256, seed=49),
}


@pytest.mark.parametrize("name", list(CASES))
def test_tc_matches_oracle(name):
    spec = CASES[name]
    x = synth.layer_inputs(spec)
    compare(spec, run_gpu(spec, x, impl=TC), run_oracle(spec, x), TOL)


@pytest.mark.parametrize("name", ["small_muon", "small_single", "small_odd_ragged", "pair_d256"])
def test_tc_single_precision_short(name):
    spec = CASES[name]
    x = synth.layer_inputs(spec)
    compare(spec, run_gpu(spec, x, impl=TC, precision=SINGLE), run_oracle(spec, x), TOL)


@pytest.mark.parametrize("wl,T", [("lm_chunk2k", 4096), ("video_ar", 2 * 5616)])
def test_tc_workload_shapes_short(wl, T):
    """The workloads' own d, dh, chunk and head counts over their first chunks;
    the oracle checks the first and the last (b, h) head."""
    spec = synth.WORKLOADS[wl].replace(T=T)
    full_workload_check(spec, [(0, 0), (spec.B - 1, spec.H - 1)], TOL, impl=TC)


@pytest.mark.parametrize("wl,heads,block", [
    ("lm_chunk2k", [(0, 0), (1, 2)], 0),
    ("video_ar", [(0, 0), (0, 7)], 0),
    ("imageset_1m", [(0, 1)], 65536),
])
def test_tc_full_workload_sampled_heads(wl, heads, block):
    """Full-size workloads in the configuration the benchmark times (all heads on
    the GPU); sampled heads compared element by element with the oracle."""
    spec = synth.WORKLOADS[wl]
    full_workload_check(spec, heads, TOL, block=block)


def test_tc_is_deterministic():
    spec = CASES["small_odd_ragged"]
    x = synth.layer_inputs(spec)
    a = run_gpu(spec, x, impl=TC)
    b = run_gpu(spec, x, impl=TC)
    assert np.array_equal(a[0], b[0]) and all(np.array_equal(p, q) for p, q in zip(a[1], b[1]))


@pytest.mark.parametrize("name", ["small_odd_ragged", "pair_d256", "d192_split_k"])
def test_forward_on_cta_pairs_equals_multicast_clusters(name):
    """The forward on CTA pairs (two token tiles as one M = 256 MMA, each CTA
    holding half of the weight slice) forms every product in the same order as
    the multicast-cluster forward, so the layer's outputs are bitwise equal."""
    spec = CASES[name]
    x = synth.layer_inputs(spec)
    try:
        abi.ttt_dbg_fwd_pairs(True)
        a = run_gpu(spec, x, impl=TC)
        abi.ttt_dbg_fwd_pairs(False)
        b = run_gpu(spec, x, impl=TC)
    finally:
        abi.ttt_dbg_fwd_pairs(True)
    assert np.array_equal(a[0], b[0]) and all(np.array_equal(p, q) for p, q in zip(a[1], b[1]))


def test_muon_on_cta_pairs_matches_oracle():
    """The Muon step's GEMM phases on CTA-pair tiles (cta_group::2, off by
    default; taken when d and dh are multiples of 256), with the update fused
    into the last X update: parity with the oracle, on a small case and on the
    lm workload's shapes."""
    spec = CASES["pair_d256"]
    x = synth.layer_inputs(spec)
    lm = synth.WORKLOADS["lm_chunk2k"].replace(T=4096)
    try:
        abi.ttt_dbg_ns_pairs(True)
        got = run_gpu(spec, x, impl=TC)
        full_workload_check(lm, [(0, 0), (lm.B - 1, lm.H - 1)], TOL, impl=TC)
    finally:
        abi.ttt_dbg_ns_pairs(False)
    compare(spec, got, run_oracle(spec, x), TOL)
