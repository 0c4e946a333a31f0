"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, and rejects bad requests before launching anything. No GPU needed:
every ttt_fwd call here fails validation, so no pointer is ever dereferenced."""
import ctypes
import os
import re
import subprocess

import pytest

from long_seq_models_chunked_b300 import abi, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"TTT_API\s+[\w\s\*]+?\b(\w+)\s*\(", txt)
    return names


def test_library_exports_every_declared_symbol():
    names = _declared()
    assert "ttt_fwd" in names and len(names) >= 10
    out = subprocess.run(["nm", "-D", "--defined-only", abi.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(abi.lib(), n)
    assert set(abi.EXPORTED) <= set(names)


def test_cfg_layout_and_defaults():
    assert abi.lib().ttt_cfg_size() == ctypes.sizeof(abi.ttt_cfg)
    c = abi.ttt_cfg_default()
    assert (c.fast_net, c.loss, c.mode, c.dtype, c.muon, c.ns_iters, c.wnorm) == (0, 0, 0, 1, 1, 5, 1)
    assert abs(c.ns_a - 3.4445) < 1e-6 and abs(c.ns_b + 4.775) < 1e-6 and abs(c.ns_c - 2.0315) < 1e-6
    assert c.step == 1.0 and c.timeout_us == 2000000 and abi.ttt_abi_version() >= 1


def test_workspace_query_and_selection():
    for name, spec in synth.WORKLOADS.items():
        h = abi.cfg_from_spec(spec)
        assert abi.ttt_select_impl(h.cfg) >= 1, name
        assert abi.ttt_workspace_bytes(h.cfg) >= 256, name
        assert abi.ttt_host_arena_bytes(h.cfg) > abi.ttt_workspace_bytes(h.cfg)
    tiny = abi.cfg_from_spec(synth.WORKLOADS["tiny_fp32"]).cfg
    assert abi.ttt_select_impl(tiny) == abi.TTT_IMPL_SIMT


@pytest.mark.parametrize("field,value", [("B", 0), ("T", -1), ("T", 0), ("H", 0), ("d", 0), ("chunk", 0),
                                         ("fast_net", 2), ("loss", 5), ("mode", 3),
                                         ("dtype", 7), ("ns_iters", -1), ("wnorm_eps", 0.0),
                                         ("impl", 9), ("muon", 2)])
def test_bad_cfg_is_rejected(field, value):
    c = abi.cfg_from_spec(synth.WORKLOADS["tiny_fp32"]).cfg
    setattr(c, field, value)
    assert abi.ttt_select_impl(c) == abi.TTT_ERR_ARG
    with pytest.raises(abi.TTTError):
        abi.ttt_workspace_bytes(c)


def _fake(n):  # distinct, 256-aligned, never dereferenced
    return 0x10000000 + n * 0x1000000


def _call(c, **over):
    p = dict(Q=_fake(1), K=_fake(2), V=_fake(3), lr=_fake(4), W1=_fake(5), W2=_fake(6),
             W3=_fake(7), O=_fake(8), F1=_fake(9), F2=_fake(10), F3=_fake(11), ws=_fake(12),
             ws_bytes=abi.ttt_workspace_bytes(c))
    p.update(over)
    return abi.lib().ttt_fwd(ctypes.byref(c), p["Q"], p["K"], p["V"], p["lr"], p["W1"],
                             p["W2"], p["W3"], p["O"], p["F1"], p["F2"], p["F3"], p["ws"],
                             p["ws_bytes"], None)


@pytest.mark.parametrize("over,code", [
    (dict(Q=0), abi.TTT_ERR_ARG),
    (dict(lr=_fake(4) + 4), abi.TTT_ERR_ARG),          # misaligned
    (dict(W2=0), abi.TTT_ERR_ARG),
    (dict(O=_fake(1)), abi.TTT_ERR_ARG),               # O aliases Q
    (dict(F2=_fake(9)), abi.TTT_ERR_ARG),              # two outputs alias
    (dict(O=_fake(12) + 256), abi.TTT_ERR_ARG),        # output inside the workspace
    (dict(ws=0), abi.TTT_ERR_WORKSPACE),
    (dict(ws=_fake(12) + 16), abi.TTT_ERR_WORKSPACE),  # not 256-aligned
    (dict(ws_bytes=255), abi.TTT_ERR_WORKSPACE),
])
def test_fwd_rejects_before_launch(over, code):
    c = abi.cfg_from_spec(synth.WORKLOADS["tiny_fp32"]).cfg
    assert _call(c, **over) == code


def test_strerror_covers_every_code():
    for code in range(0, abi.TTT_ERR_SCRATCH_LIMIT - 1, -1):
        assert abi.ttt_strerror(code) != "unknown status"
    assert abi.ttt_strerror(12345) == "unknown status"


def _static_call(c, **over):
    p = dict(Q=_fake(1), K=_fake(2), V=_fake(3), lr=_fake(4), W1=_fake(5), W2=_fake(6),
             W3=_fake(7), O=_fake(8), F1=_fake(9), F2=_fake(10), F3=_fake(11), st=_fake(12))
    p.update(over)
    return abi.lib().ttt_fwd_static_scratch(ctypes.byref(c), p["Q"], p["K"], p["V"], p["lr"], p["W1"],
                                            p["W2"], p["W3"], p["O"], p["F1"], p["F2"], p["F3"], p["st"],
                                            None)


@pytest.mark.parametrize("over", [
    dict(st=_fake(1) + 64),       # status word inside Q
    dict(st=_fake(4)),            # status word on the learning rates
    dict(st=_fake(6) + 128),      # status word inside W0_2
    dict(st=_fake(9) + 4),        # status word inside an output
    dict(st=_fake(12) + 2),       # misaligned
])
def test_static_scratch_rejects_a_bad_status_word_before_launch(over):
    c = abi.cfg_from_spec(synth.WORKLOADS["tiny_fp32"], impl=abi.TTT_IMPL_SIMT).cfg
    assert _static_call(c, **over) == abi.TTT_ERR_ARG


def test_backward_covers_the_linear_net_with_plain_steps():
    lin = abi.cfg_from_spec(synth.WORKLOADS["linear_chunk64"]).cfg
    assert abi.ttt_bwd_workspace_bytes(lin) > 0
    for spec in (synth.WORKLOADS["lm_chunk2k"], synth.WORKLOADS["linear_chunk64"].replace(mode="single")):
        c = abi.cfg_from_spec(spec).cfg
        with pytest.raises(abi.TTTError) as err:
            abi.ttt_bwd_workspace_bytes(c)
        assert err.value.code == abi.TTT_ERR_UNSUPPORTED

def test_test_hooks_reject_bad_arguments():
    assert abi.lib().ttt_dbg_grad_pairs(2) == abi.TTT_ERR_ARG
    assert abi.lib().ttt_dbg_grad_pairs(-1) == abi.TTT_ERR_ARG
    assert abi.lib().ttt_dbg_grad_pairs(1) == abi.TTT_OK
    assert abi.lib().ttt_dbg_ns_tiles(64, 0) == abi.TTT_ERR_ARG
    assert abi.lib().ttt_dbg_ns_tiles(0, 0) == abi.TTT_OK


def test_thread_release_with_nothing_to_release():
    assert abi.ttt_thread_release() == abi.TTT_OK


def test_swiglu_backward_support():
    spec = synth.WORKLOADS["tiny_fp32"].replace(wnorm=False, muon=False, loss="ip")
    assert abi.ttt_bwd_swiglu_workspace_bytes(abi.cfg_from_spec(spec).cfg) > 0
    assert abi.ttt_bwd_swiglu_workspace_bytes(abi.cfg_from_spec(spec.replace(loss="mse")).cfg) > 0
    for bad in (spec.replace(muon=True), spec.replace(wnorm=True), spec.replace(mode="single"),
                spec.replace(lr_per_matrix=True), spec.replace(momentum=0.5)):
        with pytest.raises(abi.TTTError) as e:
            abi.ttt_bwd_swiglu_workspace_bytes(abi.cfg_from_spec(bad).cfg)
        assert e.value.code == abi.TTT_ERR_UNSUPPORTED


def _swbwd_call(c, **over):
    # fake, well-separated device-like addresses (the checks here run before any CUDA call)
    p = {n: _fake(i + 1) for i, n in enumerate(
        ["Q", "K", "V", "lr", "W1", "W2", "W3", "dO", "F1", "F2", "F3",
         "dQ", "dK", "dV", "dlr", "G1", "G2", "G3", "ws"])}
    need = c_size = ctypes.c_size_t(0)
    assert abi.lib().ttt_bwd_swiglu_workspace_bytes(ctypes.byref(c), ctypes.byref(c_size)) == abi.TTT_OK
    p["ws_bytes"] = need.value
    p.update(over)
    return abi.lib().ttt_bwd_swiglu(ctypes.byref(c), p["Q"], p["K"], p["V"], p["lr"], p["W1"], p["W2"], p["W3"],
                                    p["dO"], p["F1"], p["F2"], p["F3"], p["dQ"], p["dK"], p["dV"], p["dlr"],
                                    p["G1"], p["G2"], p["G3"], p["ws"], p["ws_bytes"], None)


@pytest.mark.parametrize("over,code", [
    (dict(Q=0), abi.TTT_ERR_ARG),
    (dict(W2=_fake(6) + 4), abi.TTT_ERR_ARG),         # misaligned
    (dict(dQ=_fake(1)), abi.TTT_ERR_ARG),             # an output on an input
    (dict(G3=_fake(17)), abi.TTT_ERR_ARG),            # two outputs alias
    (dict(ws=0), abi.TTT_ERR_WORKSPACE),
    (dict(ws_bytes=255), abi.TTT_ERR_WORKSPACE),
])
def test_swiglu_backward_rejects_before_launch(over, code):
    spec = synth.WORKLOADS["tiny_fp32"].replace(wnorm=False, muon=False)
    c = abi.cfg_from_spec(spec).cfg
    assert _swbwd_call(c, **over) == code


def test_binding_refuses_a_strided_view_before_the_call():
    """The C ABI reads dense row-major memory: a transposed or sliced-with-step
    view is refused by the binding (ValueError) before any library call."""
    import torch
    c = abi.cfg_from_spec(synth.WORKLOADS["tiny_fp32"]).cfg
    dense = torch.zeros(4, 8)
    n0 = abi.ttt_launch_count()
    for view in (dense.t(), dense[:, ::2]):
        with pytest.raises(ValueError, match="not contiguous"):
            abi.ttt_fwd(c, view, dense, dense, dense, dense, dense, dense, dense, dense, dense, dense,
                        torch.zeros(256, dtype=torch.uint8), stream=0)
    assert abi.ttt_launch_count() == n0
    assert abi._ptr(dense) == dense.data_ptr() and abi._ptr(None) is None and abi._ptr(64) == 64


def test_layer_checks_shapes_and_dtypes_before_the_call():
    """abi.layer compares every input's shape, dtype and device with the
    configuration before it allocates or calls anything."""
    import torch
    spec = synth.WORKLOADS["tiny_fp32"]
    holder = abi.cfg_from_spec(spec)
    B, H, T, d, dh = spec.B, spec.H, spec.T, spec.d, spec.dh
    ok = dict(Q=torch.zeros(B, H, T, d), K=torch.zeros(B, H, T, d), V=torch.zeros(B, H, T, d),
              lr=torch.zeros(B, H, T), W0=[torch.zeros(H, dh, d), torch.zeros(H, d, dh), torch.zeros(H, dh, d)])
    abi._check_layer_tensors(holder.cfg, **ok)
    bad = [dict(Q=torch.zeros(B, H, T, d + 1)), dict(K=torch.zeros(B, H, T, d, dtype=torch.bfloat16)),
           dict(lr=torch.zeros(B, H, T, 3)), dict(W0=ok["W0"][:2]),
           dict(W0=[torch.zeros(H, d, dh)] * 3), dict(V=torch.zeros(B, H, T - 1, d))]
    n0 = abi.ttt_launch_count()
    for over in bad:
        with pytest.raises(ValueError):
            abi.layer(holder, **{**ok, **over})
    assert abi.ttt_launch_count() == n0
