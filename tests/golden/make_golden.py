"""Writes tests/golden/oracle_tiny.json: the oracle's outputs on a tiny seeded case.

It calls only the oracle and the seeded input generator. The stored values are a
regression record of the oracle itself (so that an unintended change of its
arithmetic shows up); they are not used as a parity reference for the kernels.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from long_seq_models_chunked_b300.synth import LayerSpec, layer_inputs  # noqa: E402
from oracle import OracleCfg, ttt_layer  # noqa: E402

CASES = {
    "swiglu_muon_wnorm_shifted": LayerSpec("g1", B=1, H=1, T=12, d=4, dh=8, chunk=4,
                                           dtype="fp32", seed=101),
    "swiglu_sgd_single": LayerSpec("g2", B=1, H=1, T=10, d=4, dh=8, chunk=10, mode="single",
                                   muon=False, dtype="fp32", seed=102),
    "linear_mse_sgd": LayerSpec("g3", B=1, H=1, T=9, d=3, dh=3, chunk=3, fast_net="linear",
                                loss="mse", muon=False, wnorm=False, dtype="fp32",
                                lr_a=0.5, seed=103),
    "swiglu_muon_momentum_rates_odd": LayerSpec("g4", B=1, H=1, T=14, d=4, dh=8, chunk=4, update="odd",
                                                momentum=0.5, lr_per_matrix=True, dtype="fp32", seed=104),
    "swiglu_mse_inclusive": LayerSpec("g5", B=1, H=1, T=11, d=4, dh=8, chunk=4, loss="mse",
                                      mode="inclusive", muon=False, wnorm=False, dtype="fp32",
                                      seed=105),
}


def compute(spec):
    x = layer_inputs(spec)
    O, Wf = ttt_layer(OracleCfg.from_spec(spec), x["Q64"], x["K64"], x["V64"],
                      x["lr"], x["W0"])
    return {"O": O.ravel().tolist(), "Wf": [w.ravel().tolist() for w in Wf]}


if __name__ == "__main__":
    out = {name: compute(spec) for name, spec in CASES.items()}
    with open(os.path.join(HERE, "oracle_tiny.json"), "w") as f:
        json.dump(out, f, indent=0)
