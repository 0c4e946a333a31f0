"""Stored fixtures: the pages' workload figures and the oracle's own regression record."""
import json
import os

import numpy as np

from long_seq_models_chunked_b300.synth import WORKLOADS

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_workload_table_matches_the_pages_figures():
    g = json.load(open(os.path.join(HERE, "page_workloads.json")))
    img = WORKLOADS["imageset_1m"]
    # 8x8 patches of 128 images of 960x536
    assert img.T == g["imageset_views"]["value"] * (g["imageset_width"]["value"] // 8) * (
        g["imageset_height"]["value"] // 8)
    assert abs(img.T - g["imageset_tokens_approx"]["value"]) / 1e6 < 0.05
    assert img.chunk == img.T and img.mode == "single"
    assert WORKLOADS["lm_chunk2k"].chunk in g["text_chunk_tokens"]["value"]
    vid = WORKLOADS["video_ar"]
    assert abs(vid.T - g["video_tokens_approx"]["value"]) / 56000 < 0.02
    assert vid.chunk % g["video_chunk_frames"]["value"] == 0
    assert abs(vid.chunk - g["video_chunk_tokens_approx"]["value"]) / 5000 < 0.15
    lo, hi = g["small_chunk_tokens"]["value"]
    assert lo <= WORKLOADS["linear_chunk64"].chunk <= hi


def test_oracle_regression_record():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    stored = json.load(open(os.path.join(HERE, "oracle_tiny.json")))
    for name, s in mg.CASES.items():
        now = mg.compute(s)
        assert np.abs(np.array(now["O"]) - np.array(stored[name]["O"])).max() <= 1e-12
        for a, b in zip(now["Wf"], stored[name]["Wf"]):
            assert np.abs(np.array(a) - np.array(b)).max() <= 1e-12
