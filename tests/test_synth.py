"""The seeded input generator: determinism, block access, rounding, recipe."""
import numpy as np

from long_seq_models_chunked_b300 import synth


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 3.0e-3],
                 dtype=np.float32)
    bits = synth.fp32_to_bf16_bits(x)
    back = synth.bf16_bits_to_f64(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: goes to the even mantissa (1.0)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.0 + 2 ** -6
    assert back[3] == 1.0 and back[4] == -2.5
    assert abs(back[5] - 3.0e-3) <= 3.0e-3 * 2 ** -8


def test_token_ranges_regenerate_identically():
    spec = synth.WORKLOADS["lm_chunk2k"].replace(T=9000)
    full = synth.head_tokens(spec, 1, 2)
    part = synth.head_tokens(spec, 1, 2, 4000, 8500)
    for n in ("Q", "K", "V", "lr"):
        assert np.array_equal(full[n][4000:8500], part[n])


def test_recipe_normalises_q_and_k_only():
    spec = synth.WORKLOADS["video_ar"].replace(T=300, dtype="fp32")
    x = synth.head_tokens(spec, 0, 3)
    assert np.abs(np.linalg.norm(x["Q64"], axis=1) - 1).max() < 1e-6
    assert np.abs(np.linalg.norm(x["K64"], axis=1) - 1).max() < 1e-6
    assert np.abs(np.linalg.norm(x["V64"], axis=1) - 1).max() > 0.1
    assert (x["lr"] > 0).all() and (x["lr"] < 0.01).all()


def test_masks_and_weights():
    v = synth.WORKLOADS["video_ar"]
    assert list(v.update_mask()) == [0, 1] * 5
    W = synth.initial_weights(synth.WORKLOADS["tiny_fp32"])
    assert [w.shape for w in W] == [(2, 64, 32), (2, 32, 64), (2, 64, 32)]
    assert abs(W[0].std() - 32 ** -0.5) < 0.02 and abs(W[1].std() - 64 ** -0.5) < 0.02
