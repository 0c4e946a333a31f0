"""Host-side measurement logic (no GPU): the fixed FLOP accounting, its split
over the kernel classes, the CPU baseline's scaling to layer tokens/s, the
reading of committed ncu traffic figures and the roofline object."""
import math

import pytest

from long_seq_models_chunked_b300 import accounting, synth


def _hand_count(B, H, T, C, d, dh, upd_chunks, muon=True, iters=5):
    """SwiGLU with the inner-product loss, counted by hand: 6 d dh per applied
    token (two forward GEMMs of 2 d dh each for [A|B], one for O), 12 d dh per
    updated token (keys' forward 6 d dh, three gradient outer products 6 d dh),
    and per update 3 matrices x iters x (Gram 2 m^2 n + X update 2 m^2 n + poly
    2 m^3), m = d, n = dh."""
    upd_tokens = sum(min(T, (c + 1) * C) - c * C for c in upd_chunks)
    f = 6 * d * dh * T + 12 * d * dh * upd_tokens
    if muon:
        f += len(upd_chunks) * 3 * iters * (4 * d * d * dh + 2 * d ** 3)
    return B * H * f


@pytest.mark.parametrize("name,expected", [
    ("lm_chunk2k", _hand_count(2, 3, 32768, 2048, 512, 1024, range(16))),          # 3.788e12
    ("imageset_1m", _hand_count(1, 4, 1029120, 1029120, 192, 384, [0])),           # 5.467e12
    ("video_ar", _hand_count(1, 8, 56160, 5616, 640, 1280, [1, 3, 5, 7, 9])),      # 5.989e12
])
def test_swiglu_workloads_match_a_hand_count(name, expected):
    assert math.isclose(accounting.algorithmic_flops(synth.WORKLOADS[name]), expected, rel_tol=1e-12)


def test_linear_workload_matches_a_hand_count():
    # 2 d^2 per applied token, 4 d^2 per updated token (R = K W^T and G = R^T K)
    B, H, T, d = 16, 16, 8192, 64
    assert math.isclose(accounting.algorithmic_flops(synth.WORKLOADS["linear_chunk64"]),
                        B * H * (2 * d * d * T + 4 * d * d * T), rel_tol=1e-12)


@pytest.mark.parametrize("name", ["lm_chunk2k", "imageset_1m", "video_ar"])
def test_kernel_classes_partition_the_layer(name):
    """The per-kernel FLOP that the roofline divides by add up to the layer's
    count: forward + apply + gradient + fused Muon step, and the Muon step is
    its Gram, polynomial and X-update parts."""
    import bench
    from long_seq_models_chunked_b300 import abi
    spec = synth.WORKLOADS[name]
    parts = [bench.kernel_flops_per_launch(spec, k, 1)
             for k in (abi.TTT_KERNEL_FWD, abi.TTT_KERNEL_APPLY, abi.TTT_KERNEL_GRAD, abi.TTT_KERNEL_NS)]
    assert math.isclose(sum(parts), accounting.algorithmic_flops(spec), rel_tol=1e-12)
    ns = sum(bench.kernel_flops_per_launch(spec, k, 1)
             for k in (abi.TTT_KERNEL_GRAM, abi.TTT_KERNEL_POLY, abi.TTT_KERNEL_XUPD))
    assert math.isclose(ns, parts[3], rel_tol=1e-12)
    # per launch: the class total divided by its launches
    assert math.isclose(bench.kernel_flops_per_launch(spec, abi.TTT_KERNEL_NS, 16), parts[3] / 16, rel_tol=1e-12)


def test_oracle_sample_is_scaled_per_layer_token(monkeypatch):
    """With a clock that advances 0.5 s per reading, each chunk the oracle runs
    costs 0.5 s; a 1 s budget runs two 64-token chunks of head (0, 0). At that
    rate the whole layer (B*H heads of T tokens) takes B*H*T/128 s for B*T
    tokens, i.e. 128 / H tokens/s."""
    import bench
    spec = synth.WORKLOADS["tiny_fp32"]
    t = [0.0]

    def clock():
        t[0] += 0.5
        return t[0]

    monkeypatch.setattr(bench.time, "perf_counter", clock)
    value, desc, spent = bench.oracle_sample(spec, 1.0)
    assert spent == pytest.approx(1.0)
    whole_layer_s = spec.B * spec.H * spec.T / 128.0
    assert value == pytest.approx(spec.B * spec.T / whole_layer_s)
    assert value == pytest.approx(128.0 / spec.H)
    assert desc.startswith("2 chunks")


def test_read_traffic_uses_committed_profiles():
    import bench
    v = bench.read_traffic("ns_fused", "lm_chunk2k")
    assert isinstance(v, float) and v > 1e8
    assert bench.read_traffic("no_such_kernel", "lm_chunk2k") is None


def test_roofline_of_the_top_kernel_class():
    """The benchmark's roofline object from per-kernel-class device times: the class
    with the most time, its algorithmic FLOP per launch over its mean launch time,
    against the burst bf16 peak (the sustained one beside it); the linear kernel's
    bytes against the copy bandwidth."""
    import bench
    from long_seq_models_chunked_b300 import abi
    peaks = {"hbm_gbs": 6500.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
    spec = synth.WORKLOADS["lm_chunk2k"]
    steps, per_step = 20, 16
    kinds = {"ns_fused": (abi.TTT_KERNEL_NS, 0.35 * per_step * steps, per_step * steps, per_step * steps),
             "fwd": (abi.TTT_KERNEL_FWD, 0.13 * per_step * steps, per_step * steps, per_step * steps)}
    r = bench.roofline(spec, kinds, steps, peaks, "test")
    fl = bench.kernel_flops_per_launch(spec, abi.TTT_KERNEL_NS, per_step)
    assert r["kernel"] == "ns_fused" and r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert math.isclose(r["achieved"], fl / 0.35e-3 / 1e12, rel_tol=1e-12)
    assert r["peak"] == 1800.0 and math.isclose(r["frac"], r["achieved"] / 1800.0, rel_tol=1e-12)
    assert math.isclose(r["frac_of_sustained"], r["achieved"] / 1400.0, rel_tol=1e-12)
    assert math.isclose(r["share"], 0.35 / 0.48, rel_tol=1e-12) and math.isclose(r["launch_ms"], 0.35)
    assert r["traffic"] == bench.read_traffic("ns_fused", "lm_chunk2k")

    lin = synth.WORKLOADS["linear_chunk64"]
    r = bench.roofline(lin, {"linear": (abi.TTT_KERNEL_LINEAR, 0.43 * steps, steps, steps)}, steps, peaks, "test")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6500.0
    assert math.isclose(r["achieved"], bench.linear_bytes_per_step(lin) / 0.43e-3 / 1e9, rel_tol=1e-12)
