"""The CPU emulation of the tensor-core path's operand precision
(tests/precision_study.py) follows the oracle's arithmetic: with fp32 operands it
lands on the fp64 oracle within fp32 rounding, and rounding the operands moves it
away in the order the stored precisions predict (pairs far closer than singles,
fp16 closer than bf16)."""
import pytest

from long_seq_models_chunked_b300 import synth
from precision_study import emulate_head, max_rel_err, oracle_head

SPEC = synth.LayerSpec("prec_small", B=1, H=1, T=1024, d=64, dh=128, chunk=256, seed=71)
F32 = dict(fwd=("f32",) * 3, E=("f32",) * 3, ns=("f32",) * 5, g0="f32")


@pytest.fixture(scope="module")
def ref():
    x = synth.head_tokens(SPEC, 0, 0)
    return x, oracle_head(SPEC, SPEC.n_chunks, x)


def test_fp32_operands_reproduce_the_oracle(ref):
    x, Wr = ref
    assert max_rel_err(emulate_head(SPEC, SPEC.n_chunks, x=x, **F32), Wr) <= 2e-5


def test_rounding_orders_as_the_stored_precision_predicts(ref):
    x, Wr = ref
    e = {name: max_rel_err(emulate_head(SPEC, SPEC.n_chunks, x=x, **kw), Wr) for name, kw in {
        "split": {},
        "single": dict(fwd=("b1",) * 3, E=("b1",) * 3, ns=("h1",) * 5, g0="h1"),
        "E_bf16": dict(E=("b1",) * 3),
        "E_fp16": dict(E=("h1",) * 3),
    }.items()}
    assert e["split"] * 10 < e["single"], e
    assert e["E_fp16"] < e["E_bf16"], e
    assert e["split"] < e["E_fp16"], e
