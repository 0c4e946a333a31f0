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
    # d and dh multiples of 256: 256-wide Newton-Schulz tiles
    "pair_d256": BASE.replace(name="pair_d256", B=2, H=2, d=256, dh=512, T=1024, chunk=256, seed=49),
    # degenerate cases: no chunk updates (O is the plain SwiGLU MLP of W0, Wf = W0),
    # and every learning rate zero (G = 0: Newton-Schulz of a zero matrix is zero)
    "no_update": BASE.replace(name="no_update", update="none", T=640, chunk=128, seed=50),
    "zero_lr": BASE.replace(name="zero_lr", lr_a=0.0, seed=51),
    "zero_lr_single": BASE.replace(name="zero_lr_single", lr_a=0.0, mode="single", chunk=512, seed=52),
    # LaCT page §2.2.1: a momentum buffer before Newton-Schulz (or as the step
    # without Muon), and one rate per token and matrix
    "momentum_muon": BASE.replace(name="momentum_muon", momentum=0.9, seed=53),
    "momentum_sgd": BASE.replace(name="momentum_sgd", muon=False, momentum=0.8, seed=54),
    "lr_per_matrix": BASE.replace(name="lr_per_matrix", lr_per_matrix=True, seed=55),
    "momentum_lr_odd_ragged": BASE.replace(name="momentum_lr_odd_ragged", T=700, chunk=200, update="odd",
                                           momentum=0.5, lr_per_matrix=True, seed=56),
    # MSE loss (tutorial page §3; the modular-TTT abstract's loss choice) on the
    # tensor-core path: Y = f(k) - v feeds the SwiGLU backward and G2
    "mse": BASE.replace(name="mse", loss="mse", seed=57),
    "mse_single_ragged": BASE.replace(name="mse_single_ragged", loss="mse", mode="single", T=700, chunk=700,
                                      seed=58),
    "mse_odd_momentum_rates": BASE.replace(name="mse_odd_momentum_rates", loss="mse", T=700, chunk=200,
                                           update="odd", momentum=0.9, lr_per_matrix=True, seed=59),
    "mse_d192_split_k": BASE.replace(name="mse_d192_split_k", loss="mse", d=192, dh=384, T=8192, chunk=8192,
                                     mode="single", lr_a=0.005, seed=60),
    "mse_sgd": BASE.replace(name="mse_sgd", loss="mse", muon=False, seed=61),
    # novel-view synthesis (LaCT page §3.1, fig. 3d): one chunk over a set of
    # views in which every fourth view is a target: its tokens only query
    # (rate 0), the input views' tokens update
    "nvs_strided": BASE.replace(name="nvs_strided", d=128, dh=256, T=4096, chunk=4096, mode="single",
                                lr_a=0.005, seed=62),
    # the chunk gradient on CTA pairs (256-wide column tiles, row pairs): MSE's
    # computed operand and token splits; d = 384 stays on the one-CTA tiles
    "mse_pair_d256": BASE.replace(name="mse_pair_d256", loss="mse", d=256, dh=512, T=1024, chunk=256, seed=63),
    "pair_d384_ragged": BASE.replace(name="pair_d384_ragged", d=384, dh=512, T=900, chunk=256, seed=64),
    "pair_split_k": BASE.replace(name="pair_split_k", d=256, dh=512, T=8192, chunk=8192, mode="single",
                                 lr_a=0.005, seed=65),
}

# token rate masks of the cases above (1 = the token updates)
RATE_MASKS = {"nvs_strided": lambda T: (np.arange(T) // 256) % 4 != 3}


def _inputs(name):
    spec = CASES[name]
    x = synth.layer_inputs(spec)
    if name in RATE_MASKS:
        x["lr"] = x["lr"] * RATE_MASKS[name](spec.T).astype(np.float32)
    return spec, x


@pytest.mark.parametrize("name", list(CASES))
def test_tc_matches_oracle(name):
    spec, x = _inputs(name)
    compare(spec, run_gpu(spec, x, impl=TC), run_oracle(spec, x), TOL)


@pytest.mark.parametrize("name", ["small_muon", "small_single", "small_odd_ragged", "pair_d256"])
def test_tc_single_precision_short(name):
    spec = CASES[name]
    x = synth.layer_inputs(spec)
    compare(spec, run_gpu(spec, x, impl=TC, precision=SINGLE), run_oracle(spec, x), TOL)


@pytest.mark.parametrize("wl,T,extra", [("lm_chunk2k", 4096, {}), ("video_ar", 2 * 5616, {}),
                                        ("lm_chunk2k", 6144, {"momentum": 0.9, "lr_per_matrix": True}),
                                        ("lm_chunk2k", 4096, {"loss": "mse"})])
def test_tc_workload_shapes_short(wl, T, extra):
    """The workloads' own d, dh, chunk and head counts over their first chunks;
    the oracle checks the first and the last (b, h) head."""
    spec = synth.WORKLOADS[wl].replace(T=T, **extra)
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


@pytest.mark.parametrize("name", ["no_update", "zero_lr"])
def test_tc_degenerate_cases_keep_w0(name):
    """With no update (mask all zero, or every rate zero) the final weights are
    W0 and the output is the plain SwiGLU MLP f_W0(Q) (LaCT page §2.1 with the
    update phase removed)."""
    spec = CASES[name]
    x = synth.layer_inputs(spec)
    O, Wf = run_gpu(spec, x, impl=TC)
    for j, w in enumerate(x["W0"]):
        for b in range(spec.B):
            assert np.abs(Wf[j][b] - w).max() <= 1e-6 * np.abs(w).max(), (name, j)
    W1, W2, W3 = (w.astype(np.float64) for w in x["W0"])
    for h in range(spec.H):
        q = x["Q64"][0, h]
        a, bm = q @ W1[h].T, q @ W3[h].T
        mlp = (a / (1.0 + np.exp(-a)) * bm) @ W2[h].T
        assert np.abs(O[0, h] - mlp).max() <= TOL * np.abs(mlp).max(), name


def test_tc_is_deterministic():
    spec = CASES["small_odd_ragged"]
    x = synth.layer_inputs(spec)
    a = run_gpu(spec, x, impl=TC)
    b = run_gpu(spec, x, impl=TC)
    assert np.array_equal(a[0], b[0]) and all(np.array_equal(p, q) for p, q in zip(a[1], b[1]))


@pytest.mark.parametrize("name", ["pair_d256", "mse_pair_d256", "pair_d384_ragged", "pair_split_k"])
def test_gradient_pairs_equal_one_cta_tiles(name):
    """The chunk gradient on CTA pairs (the default) gives bit for bit what the
    one-CTA tiles sharing E by multicast give: the same products, accumulated
    in the same order."""
    spec, x = _inputs(name)
    got = run_gpu(spec, x, impl=TC)
    try:
        abi.ttt_dbg_grad_pairs(False)
        ref = run_gpu(spec, x, impl=TC)
    finally:
        abi.ttt_dbg_grad_pairs(True)
    assert np.array_equal(got[0], ref[0]) and all(np.array_equal(p, q) for p, q in zip(got[1], ref[1])), name


def test_thread_release_between_calls():
    """ttt_thread_release destroys the side stream the shifted-mode apply runs
    on; the next call creates it again and gives the same bits."""
    spec, x = _inputs("small_odd_ragged")
    a = run_gpu(spec, x, impl=TC)
    assert abi.ttt_thread_release() == abi.TTT_OK
    assert abi.ttt_thread_release() == abi.TTT_OK  # nothing left to release
    b = run_gpu(spec, x, impl=TC)
    assert np.array_equal(a[0], b[0]) and all(np.array_equal(p, q) for p, q in zip(a[1], b[1]))


@pytest.mark.parametrize("ctas", [5, 37])
def test_muon_on_a_small_grid_matches_oracle(ctas):
    """The fused Muon kernel's item list on a grid far smaller than its items
    (each CTA walks many items of every phase, waiting on other CTAs' matrix
    counters): parity with the oracle on a small case and on the lm workload's
    shapes."""
    spec = CASES["pair_d256"]
    x = synth.layer_inputs(spec)
    lm = synth.WORKLOADS["lm_chunk2k"].replace(T=4096)
    try:
        abi.ttt_dbg_ns_force_grid(ctas)
        got = run_gpu(spec, x, impl=TC)
        full_workload_check(lm, [(0, 0), (lm.B - 1, lm.H - 1)], TOL, impl=TC)
    finally:
        abi.ttt_dbg_ns_force_grid(0)
    compare(spec, got, run_oracle(spec, x), TOL)


@pytest.mark.parametrize("sym", [0, 1])
@pytest.mark.parametrize("name", ["small_muon", "d192_split_k", "pair_d256", "small_odd_ragged", "momentum_muon"])
def test_muon_tile_sets_match_oracle(name, sym):
    """The fused Muon kernel with every tile of R = X X^T + beta I and
    P = c R^2 + alpha I computed (0), or only the tiles that meet the upper
    triangle, the missing lower blocks written as transposes (1); the default
    picks one by the shape."""
    spec = CASES[name]
    x = synth.layer_inputs(spec)
    try:
        abi.ttt_dbg_ns_symmetric(sym)
        got = run_gpu(spec, x, impl=TC)
    finally:
        abi.ttt_dbg_ns_symmetric(-1)
    compare(spec, got, run_oracle(spec, x), TOL)


def test_muon_split_mask_without_fused_normalisation():
    """With Newton-Schulz on single fp16 operands (precision-study hook), the
    Muon kernel normalises the fp32 gradient itself (its normalise phases);
    the short lm shape stays within the tolerance."""
    lm = synth.WORKLOADS["lm_chunk2k"].replace(T=4096)
    try:
        abi.ttt_dbg_split_mask(3)
        full_workload_check(lm, [(0, 0)], TOL, impl=TC)
    finally:
        abi.ttt_dbg_split_mask(7)


@pytest.mark.parametrize("hook", ["fwd", "ns"])
def test_bounded_wait_reports_timeout_and_the_next_call_succeeds(hook):
    """Failure detection without a GPU fault: the tensor-core forward withholds
    its loads (its MMA warp's mbarrier wait runs out), or one CTA of the fused
    Muon kernel never signals an item's completion (the waits of the items that
    need it run out).
    The status word says TTT_ERR_TIMEOUT, the context stays usable, and the
    next call matches the oracle."""
    import torch
    from parity import to_device
    spec = CASES["small_muon"]
    x = synth.layer_inputs(spec)
    dev = to_device(x, spec)
    holder = abi.cfg_from_spec(spec, impl=TC, timeout_us=20000)
    (abi.ttt_dbg_stall_next_fwd if hook == "fwd" else abi.ttt_dbg_stall_next_ns)()
    with pytest.raises(abi.TTTError) as err:
        abi.layer(holder, dev["Q"], dev["K"], dev["V"], dev["lr"], dev["W0"])
    assert err.value.code == abi.TTT_ERR_TIMEOUT
    torch.cuda.synchronize()
    compare(spec, run_gpu(spec, x, impl=TC), run_oracle(spec, x), TOL)


_LOCAL_BUILD_CHECK = """
import sys
sys.path.insert(0, {root!r})
sys.path.insert(0, {tests!r})
from long_seq_models_chunked_b300 import abi, synth
from parity import compare, run_gpu, run_oracle
assert abi.ttt_build_features() & abi.TTT_FEATURE_CLUSTER_MULTICAST == 0
for spec in [synth.LayerSpec("local_a", B=1, H=2, T=700, d=64, dh=128, chunk=200, update="odd", seed=61),
             synth.LayerSpec("local_b", B=1, H=2, T=4096, d=192, dh=384, chunk=4096, mode="single",
                             lr_a=0.005, seed=62)]:
    x = synth.layer_inputs(spec)
    print(spec.name, compare(spec, run_gpu(spec, x, impl=abi.TTT_IMPL_TC), run_oracle(spec, x), 2e-2))
"""


def test_build_without_multicast_matches_oracle():
    """The library a multi-GPU process loads (built without cluster multicast:
    clusters of one CTA; the gradient's row tiles become separate work items)
    runs the same tensor-core path and matches the oracle."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = _LOCAL_BUILD_CHECK.format(root=root, tests=os.path.join(root, "tests"))
    env = dict(os.environ, TTT_B300_LIBRARY="local")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
