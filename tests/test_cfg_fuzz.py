"""Host-side validation of layer configurations under random and extreme fields
(no GPU): the workspace query, the kernel-family choice and the backward's and
context-parallel queries answer every configuration with a defined status and
never crash; what they accept is consistent with what each family covers."""
import ctypes

from hypothesis import HealthCheck, given, settings
from hypothesis import strategies as st

from long_seq_models_chunked_b300 import abi

CODES = {abi.TTT_OK, abi.TTT_ERR_ARG, abi.TTT_ERR_UNSUPPORTED}
EXTREME_INT = st.sampled_from([-(2 ** 31), -1, 0, 2 ** 20 + 1, 2 ** 31 - 1])
EXTREME_FLOAT = st.sampled_from([float("inf"), float("-inf"), float("nan"), -1.0, 0.0])


@st.composite
def configs(draw):
    """Mostly well-formed configurations over the families' shapes and options,
    one field in four set to an extreme or invalid value."""
    c = abi.ttt_cfg_default()
    c.B, c.H = draw(st.integers(1, 4)), draw(st.integers(1, 8))
    c.T = draw(st.integers(1, 70000))
    c.d = draw(st.sampled_from([16, 32, 48, 64, 128, 192, 256, 512, 640, 1024, 2048]))
    c.dh = draw(st.sampled_from([16, 64, 128, 256, 384, 512, 1024, 1280, 2048, 16384, 32768]))
    c.chunk = draw(st.one_of(st.integers(1, c.T + 8), st.sampled_from([64, 2048])))
    c.fast_net = draw(st.sampled_from([abi.TTT_NET_SWIGLU, abi.TTT_NET_LINEAR]))
    c.loss = draw(st.sampled_from([abi.TTT_LOSS_IP, abi.TTT_LOSS_MSE]))
    c.mode = draw(st.sampled_from([abi.TTT_MODE_SHIFTED, abi.TTT_MODE_SINGLE, abi.TTT_MODE_INCLUSIVE]))
    c.dtype = draw(st.sampled_from([abi.TTT_DTYPE_F32, abi.TTT_DTYPE_BF16]))
    c.muon, c.wnorm = draw(st.integers(0, 1)), draw(st.integers(0, 1))
    if c.mode == abi.TTT_MODE_INCLUSIVE and draw(st.integers(0, 3)):
        c.muon = c.wnorm = 0
    c.ns_iters = draw(st.integers(0, 6))
    c.ns_c = draw(st.sampled_from([2.0315, 0.0]))
    c.impl = draw(st.sampled_from([abi.TTT_IMPL_AUTO, abi.TTT_IMPL_SIMT, abi.TTT_IMPL_TC, abi.TTT_IMPL_LINEAR]))
    c.precision = draw(st.sampled_from([abi.TTT_PREC_SPLIT, abi.TTT_PREC_SINGLE]))
    c.momentum = draw(st.sampled_from([0.0, 0.0, 0.5]))
    c.lr_per_matrix = draw(st.integers(0, 1))
    c.w0_per_batch = draw(st.integers(0, 1))
    shape = draw(st.sampled_from(["free", "tc", "linear"]))
    if shape == "tc":       # the tensor-core family's shapes
        c.fast_net, c.dtype = abi.TTT_NET_SWIGLU, abi.TTT_DTYPE_BF16
        c.d = draw(st.sampled_from([64, 128, 192, 256, 512, 640, 1024]))
        c.dh = c.d * draw(st.sampled_from([2, 4])) if c.d % 64 == 0 else 128
        c.mode = draw(st.sampled_from([abi.TTT_MODE_SHIFTED, abi.TTT_MODE_SINGLE]))
        c.ns_c, c.ns_iters = 2.0315, draw(st.integers(1, 6))
    elif shape == "linear":  # the linear kernel's shapes
        c.fast_net, c.dtype, c.d = abi.TTT_NET_LINEAR, abi.TTT_DTYPE_BF16, 64
        c.muon = c.wnorm = 0
        c.momentum = 0.0
        c.chunk = 64 * draw(st.integers(1, 4))
        c.T = 4 * draw(st.integers(1, 4096))
        c.mode = draw(st.sampled_from([abi.TTT_MODE_SHIFTED, abi.TTT_MODE_INCLUSIVE]))
    if draw(st.integers(0, 3)) == 0:
        f = draw(st.sampled_from(["B", "H", "T", "d", "dh", "chunk", "fast_net", "loss", "mode", "dtype", "muon",
                                  "ns_iters", "impl", "precision", "lr_per_matrix", "ns_eps", "wnorm_eps", "step",
                                  "momentum", "ns_a"]))
        if isinstance(getattr(c, f), float):
            setattr(c, f, draw(EXTREME_FLOAT))
        else:
            setattr(c, f, draw(EXTREME_INT))
    return c


def _size_query(fn, c):
    n = ctypes.c_size_t(0)
    rc = fn(ctypes.byref(c), ctypes.byref(n))
    assert rc in CODES, rc
    assert (rc == abi.TTT_OK) == (n.value > 0), (rc, n.value)
    return rc, n.value


@settings(max_examples=600, deadline=None, suppress_health_check=[HealthCheck.too_slow])
@given(configs())
def test_every_configuration_gets_a_defined_answer(c):
    lib = abi.lib()
    rc, nbytes = _size_query(lib.ttt_workspace_bytes, c)
    impl = lib.ttt_select_impl(ctypes.byref(c))
    assert impl in CODES | {abi.TTT_IMPL_SIMT, abi.TTT_IMPL_TC, abi.TTT_IMPL_LINEAR}, impl
    # the workspace query and the family choice agree on what is accepted
    assert (rc == abi.TTT_OK) == (impl > 0), (rc, impl)
    if impl == abi.TTT_IMPL_TC:
        assert c.fast_net == abi.TTT_NET_SWIGLU and c.dtype == abi.TTT_DTYPE_BF16
        assert c.d % 64 == 0 and c.dh % 128 == 0 and c.d <= c.dh and c.mode != abi.TTT_MODE_INCLUSIVE
    if impl == abi.TTT_IMPL_LINEAR:
        assert c.fast_net == abi.TTT_NET_LINEAR and c.d == 64 and not c.muon and not c.wnorm
    if rc == abi.TTT_OK:
        assert c.B >= 1 and c.H >= 1 and c.T >= 1 and c.d >= 1 and c.chunk >= 1
        assert nbytes >= 4  # at least the status word
    for q in (lib.ttt_bwd_workspace_bytes, lib.ttt_bwd_swiglu_workspace_bytes, lib.ttt_cp_workspace_bytes,
              lib.ttt_host_arena_bytes):
        qrc, _ = _size_query(q, c)
        if rc == abi.TTT_ERR_ARG:
            assert qrc == abi.TTT_ERR_ARG, (q.__name__, qrc)
