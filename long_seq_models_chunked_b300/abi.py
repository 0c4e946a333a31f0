"""Thin ctypes binding of the C ABI in include/ttt.h (argument marshalling only).

Functions keep the C names. Tensor arguments are torch tensors (device memory
for ttt_fwd, host memory for ttt_fwd_host); only their data pointers cross the
boundary. Every step of the layer runs in the CUDA library: if
the library is missing this module fails to import. The multicast build
(libttt_b300.so) is loaded unless TTT_B300_LIBRARY=local selects the build
without cluster multicast (libttt_b300_local.so).
"""
from __future__ import annotations

import ctypes
import os
from ctypes import c_float, c_int, c_int32, c_size_t, c_uint32, c_void_p
from typing import Optional, Sequence

import numpy as np

from .build_ext import LIB_PATH

# status codes and enums (mirrors of include/ttt.h)
TTT_OK = 0
TTT_ERR_ARG = -1
TTT_ERR_UNSUPPORTED = -2
TTT_ERR_WORKSPACE = -3
TTT_ERR_CUDA = -4
TTT_ERR_TIMEOUT = -5
TTT_ERR_NONFINITE = -6
TTT_ERR_DEVICE = -7
TTT_ERR_SCRATCH_LIMIT = -8
TTT_STATIC_SCRATCH_BYTES = 16 << 20
TTT_NET_SWIGLU, TTT_NET_LINEAR = 0, 1
TTT_LOSS_IP, TTT_LOSS_MSE = 0, 1
TTT_MODE_SHIFTED, TTT_MODE_SINGLE, TTT_MODE_INCLUSIVE = 0, 1, 2
TTT_DTYPE_F32, TTT_DTYPE_BF16 = 0, 1
TTT_IMPL_AUTO, TTT_IMPL_SIMT, TTT_IMPL_TC, TTT_IMPL_LINEAR = 0, 1, 2, 3
TTT_PREC_SPLIT, TTT_PREC_SINGLE = 0, 1

EXPORTED = ("ttt_cfg_default", "ttt_workspace_bytes", "ttt_fwd", "ttt_status",
            "ttt_host_arena_bytes", "ttt_fwd_host", "ttt_select_impl", "ttt_strerror",
            "ttt_abi_version", "ttt_cfg_size", "ttt_dbg_gemm_bf16", "ttt_prof_enable",
            "ttt_prof_reset", "ttt_prof_read", "ttt_launch_count", "ttt_kernel_name",
            "ttt_fwd_static_scratch", "ttt_dbg_ns_plan", "ttt_dbg_ns_force_grid",
            "ttt_dbg_split_mask", "ttt_dbg_stall_next_linear", "ttt_dbg_ns_trace",
            "ttt_dbg_ns_trace_read", "ttt_dbg_stall_next_fwd", "ttt_dbg_stall_next_ns", "ttt_build_features",
            "ttt_dbg_ns_symmetric", "ttt_cp_workspace_bytes", "ttt_cp_begin", "ttt_cp_grad", "ttt_cp_update",
            "ttt_cp_apply", "ttt_cp_end", "ttt_dbg_ns_tiles", "ttt_bwd_workspace_bytes", "ttt_bwd",
            "ttt_dbg_grad_pairs", "ttt_thread_release", "ttt_bwd_swiglu_workspace_bytes", "ttt_bwd_swiglu")
TTT_FEATURE_CLUSTER_MULTICAST = 1
TTT_KERNEL_FWD, TTT_KERNEL_APPLY, TTT_KERNEL_GRAD, TTT_KERNEL_GRAM, TTT_KERNEL_POLY = 0, 1, 2, 3, 4
TTT_KERNEL_XUPD, TTT_KERNEL_UPDATE, TTT_KERNEL_AUX, TTT_KERNEL_LINEAR, TTT_KERNEL_SIMT = 5, 6, 7, 8, 9
TTT_KERNEL_NS = 10
TTT_KERNEL_COUNT = 11


class ttt_cfg(ctypes.Structure):
    _fields_ = [
        ("B", c_int32), ("H", c_int32), ("T", c_int32), ("d", c_int32), ("dh", c_int32),
        ("chunk", c_int32), ("fast_net", c_int32), ("loss", c_int32), ("mode", c_int32),
        ("dtype", c_int32), ("muon", c_int32), ("ns_iters", c_int32),
        ("ns_a", c_float), ("ns_b", c_float), ("ns_c", c_float), ("ns_eps", c_float),
        ("wnorm", c_int32), ("wnorm_eps", c_float), ("step", c_float),
        ("update_mask", c_void_p), ("w0_per_batch", c_int32), ("check_finite", c_int32),
        ("timeout_us", c_uint32), ("impl", c_int32), ("precision", c_int32),
        ("momentum", c_float), ("lr_per_matrix", c_int32),
    ]


class TTTError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = code
        super().__init__(f"{where}: {ttt_strerror(code)} ({code})" if where else ttt_strerror(code))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -m long_seq_models_chunked_b300.build_ext` "
            "(the layer has no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(ttt_cfg)
    lib.ttt_cfg_default.argtypes = [P]
    lib.ttt_cfg_default.restype = None
    lib.ttt_workspace_bytes.argtypes = [P, ctypes.POINTER(c_size_t)]
    lib.ttt_host_arena_bytes.argtypes = [P, ctypes.POINTER(c_size_t)]
    ten = [c_void_p] * 11
    lib.ttt_fwd.argtypes = [P, *ten, c_void_p, c_size_t, c_void_p]
    lib.ttt_fwd_host.argtypes = [P, *ten, c_void_p, c_size_t, c_void_p]
    lib.ttt_status.argtypes = [c_void_p, c_void_p]
    lib.ttt_fwd_static_scratch.argtypes = [P, *ten, c_void_p, c_void_p]
    lib.ttt_fwd_static_scratch.restype = c_int
    lib.ttt_select_impl.argtypes = [P]
    lib.ttt_strerror.argtypes = [c_int]
    lib.ttt_strerror.restype = ctypes.c_char_p
    lib.ttt_abi_version.argtypes = []
    lib.ttt_cfg_size.argtypes = []
    lib.ttt_cfg_size.restype = c_size_t
    for name in ("ttt_workspace_bytes", "ttt_host_arena_bytes", "ttt_fwd", "ttt_fwd_host",
                 "ttt_status", "ttt_select_impl", "ttt_abi_version"):
        getattr(lib, name).restype = c_int
    lib.ttt_dbg_gemm_bf16.argtypes = [c_void_p, c_int, c_void_p, c_int, c_void_p, c_int, c_int, c_int,
                                      c_int, c_void_p]
    lib.ttt_dbg_gemm_bf16.restype = c_int
    lib.ttt_cp_workspace_bytes.argtypes = [P, ctypes.POINTER(c_size_t)]
    lib.ttt_cp_begin.argtypes = [P, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]
    lib.ttt_cp_grad.argtypes = [P, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p,
                                c_size_t, c_void_p]
    lib.ttt_cp_update.argtypes = [P, c_void_p, c_void_p, c_size_t, c_void_p]
    lib.ttt_cp_apply.argtypes = [P, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_size_t, c_void_p]
    lib.ttt_cp_end.argtypes = [P, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]
    for name in ("ttt_cp_workspace_bytes", "ttt_cp_begin", "ttt_cp_grad", "ttt_cp_update", "ttt_cp_apply",
                 "ttt_cp_end"):
        getattr(lib, name).restype = c_int
    lib.ttt_bwd_workspace_bytes.argtypes = [P, ctypes.POINTER(c_size_t)]
    lib.ttt_bwd_workspace_bytes.restype = c_int
    lib.ttt_bwd.argtypes = [P] + [c_void_p] * 12 + [c_void_p, c_size_t, c_void_p]
    lib.ttt_bwd.restype = c_int
    lib.ttt_bwd_swiglu_workspace_bytes.argtypes = [P, ctypes.POINTER(c_size_t)]
    lib.ttt_bwd_swiglu_workspace_bytes.restype = c_int
    lib.ttt_bwd_swiglu.argtypes = [P] + [c_void_p] * 18 + [c_void_p, c_size_t, c_void_p]
    lib.ttt_bwd_swiglu.restype = c_int
    lib.ttt_build_features.argtypes = []
    lib.ttt_build_features.restype = c_int
    lib.ttt_dbg_ns_tiles.argtypes = [c_int, c_int]
    lib.ttt_dbg_ns_tiles.restype = c_int
    lib.ttt_dbg_ns_symmetric.argtypes = [c_int]
    lib.ttt_dbg_ns_symmetric.restype = c_int
    lib.ttt_thread_release.argtypes = []
    lib.ttt_thread_release.restype = c_int
    lib.ttt_dbg_grad_pairs.argtypes = [c_int]
    lib.ttt_dbg_grad_pairs.restype = c_int
    lib.ttt_dbg_ns_trace.argtypes = [c_int]
    lib.ttt_dbg_ns_trace.restype = c_int
    lib.ttt_dbg_ns_trace_read.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), c_int]
    lib.ttt_dbg_ns_trace_read.restype = c_int
    lib.ttt_dbg_ns_plan.argtypes = [P, ctypes.POINTER(c_int), ctypes.POINTER(c_int)]
    lib.ttt_dbg_ns_plan.restype = c_int
    lib.ttt_dbg_ns_force_grid.argtypes = [c_int]
    lib.ttt_dbg_ns_force_grid.restype = c_int
    lib.ttt_dbg_split_mask.argtypes = [c_int]
    lib.ttt_dbg_split_mask.restype = c_int
    lib.ttt_dbg_stall_next_linear.argtypes = []
    lib.ttt_dbg_stall_next_linear.restype = None
    for name in ("ttt_dbg_stall_next_fwd", "ttt_dbg_stall_next_ns"):
        getattr(lib, name).argtypes = []
        getattr(lib, name).restype = None
    lib.ttt_prof_enable.argtypes = [c_int]
    lib.ttt_prof_enable.restype = None
    lib.ttt_prof_reset.argtypes = []
    lib.ttt_prof_reset.restype = None
    lib.ttt_prof_read.argtypes = [c_int, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_longlong),
                                  ctypes.POINTER(ctypes.c_longlong)]
    lib.ttt_prof_read.restype = c_int
    lib.ttt_launch_count.argtypes = []
    lib.ttt_launch_count.restype = ctypes.c_longlong
    lib.ttt_kernel_name.argtypes = [c_int]
    lib.ttt_kernel_name.restype = ctypes.c_char_p
    if lib.ttt_cfg_size() != ctypes.sizeof(ttt_cfg):
        raise ImportError("ttt_cfg layout mismatch between the binding and the library")
    return lib


_lib = _load()


def lib():
    return _lib


# ----------------------------------------------------------------- C names
def ttt_cfg_default() -> ttt_cfg:
    c = ttt_cfg()
    _lib.ttt_cfg_default(ctypes.byref(c))
    return c


def ttt_strerror(code: int) -> str:
    return _lib.ttt_strerror(int(code)).decode()


def ttt_abi_version() -> int:
    return _lib.ttt_abi_version()


def ttt_select_impl(cfg: ttt_cfg) -> int:
    return _lib.ttt_select_impl(ctypes.byref(cfg))


def ttt_workspace_bytes(cfg: ttt_cfg) -> int:
    n = c_size_t(0)
    rc = _lib.ttt_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n))
    if rc != TTT_OK:
        raise TTTError(rc, "ttt_workspace_bytes")
    return n.value


def ttt_host_arena_bytes(cfg: ttt_cfg) -> int:
    n = c_size_t(0)
    rc = _lib.ttt_host_arena_bytes(ctypes.byref(cfg), ctypes.byref(n))
    if rc != TTT_OK:
        raise TTTError(rc, "ttt_host_arena_bytes")
    return n.value


def _ptr(t) -> Optional[int]:
    """The address of a tensor's first element (None and plain ints pass through).
    The C ABI reads every tensor as dense row-major memory, so a strided view is
    refused here rather than read as if it were dense."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError(f"tensor of shape {tuple(t.shape)} and strides {tuple(t.stride())} is not "
                         "contiguous; the C ABI reads dense row-major memory (pass .contiguous())")
    return t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def ttt_fwd(cfg: ttt_cfg, Q, K, V, lr, W0_1, W0_2, W0_3, O, Wf_1, Wf_2, Wf_3,
            workspace, stream=None, check: bool = True) -> int:
    """Enqueue the layer on `stream` (torch tensors on the GPU). Returns the status."""
    nbytes = workspace.numel() * workspace.element_size()
    rc = _lib.ttt_fwd(ctypes.byref(cfg), _ptr(Q), _ptr(K), _ptr(V), _ptr(lr), _ptr(W0_1),
                      _ptr(W0_2), _ptr(W0_3), _ptr(O), _ptr(Wf_1), _ptr(Wf_2), _ptr(Wf_3),
                      _ptr(workspace), nbytes, _stream_handle(stream))
    if check and rc != TTT_OK:
        raise TTTError(rc, "ttt_fwd")
    return rc


def ttt_status(workspace, stream=None) -> int:
    return _lib.ttt_status(_ptr(workspace), _stream_handle(stream))


def ttt_fwd_host(cfg: ttt_cfg, Q, K, V, lr, W0_1, W0_2, W0_3, O, Wf_1, Wf_2, Wf_3,
                 arena, stream=None, check: bool = True) -> int:
    """The layer on host tensors (pinned for full bandwidth); synchronous."""
    nbytes = arena.numel() * arena.element_size()
    rc = _lib.ttt_fwd_host(ctypes.byref(cfg), _ptr(Q), _ptr(K), _ptr(V), _ptr(lr), _ptr(W0_1),
                           _ptr(W0_2), _ptr(W0_3), _ptr(O), _ptr(Wf_1), _ptr(Wf_2), _ptr(Wf_3),
                           _ptr(arena), nbytes, _stream_handle(stream))
    if check and rc != TTT_OK:
        raise TTTError(rc, "ttt_fwd_host")
    return rc


def ttt_fwd_static_scratch(cfg: ttt_cfg, Q, K, V, lr, W0_1, W0_2, W0_3, O, Wf_1, Wf_2, Wf_3,
                           status=None, stream=None, check: bool = True) -> int:
    """The allocation-free variant (fp32 SIMT family, library-held scratch):
    same tensors as ttt_fwd minus the workspace; `status` is an optional device
    int32 tensor that receives the device-side status word."""
    rc = _lib.ttt_fwd_static_scratch(ctypes.byref(cfg), _ptr(Q), _ptr(K), _ptr(V), _ptr(lr), _ptr(W0_1),
                                     _ptr(W0_2), _ptr(W0_3), _ptr(O), _ptr(Wf_1), _ptr(Wf_2), _ptr(Wf_3),
                                     _ptr(status), _stream_handle(stream))
    if check and rc != TTT_OK:
        raise TTTError(rc, "ttt_fwd_static_scratch")
    return rc


# ----------------------------------------------------------------- backward
def ttt_bwd_workspace_bytes(cfg: ttt_cfg) -> int:
    n = c_size_t(0)
    rc = _lib.ttt_bwd_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n))
    if rc != TTT_OK:
        raise TTTError(rc, "ttt_bwd_workspace_bytes")
    return n.value


def ttt_bwd(cfg: ttt_cfg, Q, K, V, lr, W0, dO, dWf, dQ, dK, dV, dlr, dW0, workspace, stream=None,
            check: bool = True) -> int:
    """Enqueue the outer-loop backward (include/ttt.h) on `stream`."""
    rc = _lib.ttt_bwd(ctypes.byref(cfg), _ptr(Q), _ptr(K), _ptr(V), _ptr(lr), _ptr(W0), _ptr(dO), _ptr(dWf),
                      _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(dlr), _ptr(dW0), _ptr(workspace),
                      workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if check and rc != TTT_OK:
        raise TTTError(rc, "ttt_bwd")
    return rc


def ttt_bwd_swiglu_workspace_bytes(cfg: ttt_cfg) -> int:
    n = c_size_t(0)
    rc = _lib.ttt_bwd_swiglu_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n))
    if rc != TTT_OK:
        raise TTTError(rc, "ttt_bwd_swiglu_workspace_bytes")
    return n.value


def ttt_bwd_swiglu(cfg: ttt_cfg, Q, K, V, lr, W0, dO, dWf, dQ, dK, dV, dlr, dW0, workspace, stream=None,
                   check: bool = True) -> int:
    """Enqueue the outer-loop backward of the SwiGLU net (include/ttt.h) on
    `stream`; W0, dWf and dW0 are sequences of the three matrices."""
    rc = _lib.ttt_bwd_swiglu(ctypes.byref(cfg), _ptr(Q), _ptr(K), _ptr(V), _ptr(lr), _ptr(W0[0]), _ptr(W0[1]),
                             _ptr(W0[2]), _ptr(dO), _ptr(dWf[0]), _ptr(dWf[1]), _ptr(dWf[2]), _ptr(dQ), _ptr(dK),
                             _ptr(dV), _ptr(dlr), _ptr(dW0[0]), _ptr(dW0[1]), _ptr(dW0[2]), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if check and rc != TTT_OK:
        raise TTTError(rc, "ttt_bwd_swiglu")
    return rc


# ----------------------------------------------------------------- context parallelism
def _cp_check(rc, where):
    if rc != TTT_OK:
        raise TTTError(rc, where)


def ttt_cp_workspace_bytes(cfg: ttt_cfg) -> int:
    n = c_size_t(0)
    _cp_check(_lib.ttt_cp_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)), "ttt_cp_workspace_bytes")
    return n.value


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def ttt_cp_begin(cfg: ttt_cfg, W0_1, W0_2, W0_3, workspace, stream=None) -> None:
    _cp_check(_lib.ttt_cp_begin(ctypes.byref(cfg), _ptr(W0_1), _ptr(W0_2), _ptr(W0_3), _ptr(workspace),
                                _nbytes(workspace), _stream_handle(stream)), "ttt_cp_begin")


def ttt_cp_grad(cfg: ttt_cfg, K, V, lr, T_all: int, start: int, n: int, G, workspace, stream=None) -> None:
    _cp_check(_lib.ttt_cp_grad(ctypes.byref(cfg), _ptr(K), _ptr(V), _ptr(lr), T_all, start, n, _ptr(G),
                               _ptr(workspace), _nbytes(workspace), _stream_handle(stream)), "ttt_cp_grad")


def ttt_cp_update(cfg: ttt_cfg, G, workspace, stream=None) -> None:
    _cp_check(_lib.ttt_cp_update(ctypes.byref(cfg), _ptr(G), _ptr(workspace), _nbytes(workspace),
                                 _stream_handle(stream)), "ttt_cp_update")


def ttt_cp_apply(cfg: ttt_cfg, Q, T_all: int, start: int, n: int, O, workspace, stream=None) -> None:
    _cp_check(_lib.ttt_cp_apply(ctypes.byref(cfg), _ptr(Q), T_all, start, n, _ptr(O), _ptr(workspace),
                                _nbytes(workspace), _stream_handle(stream)), "ttt_cp_apply")


def ttt_cp_end(cfg: ttt_cfg, Wf_1, Wf_2, Wf_3, workspace, stream=None) -> None:
    _cp_check(_lib.ttt_cp_end(ctypes.byref(cfg), _ptr(Wf_1), _ptr(Wf_2), _ptr(Wf_3), _ptr(workspace),
                              _nbytes(workspace), _stream_handle(stream)), "ttt_cp_end")


def ttt_dbg_gemm_bf16(A, a_mn_major: bool, B, b_mn_major: bool, D, Z: int, M: int, N: int, K: int,
                      stream=None) -> int:
    """Test hook: D[z] = A[z] B[z]^T on the tcgen05 tile kernel (include/ttt_debug.h)."""
    return _lib.ttt_dbg_gemm_bf16(_ptr(A), int(a_mn_major), _ptr(B), int(b_mn_major), _ptr(D), Z, M, N,
                                  K, _stream_handle(stream))


def ttt_build_features() -> int:
    """Bit flags of the loaded build (TTT_FEATURE_CLUSTER_MULTICAST)."""
    return _lib.ttt_build_features()


def ttt_dbg_ns_symmetric(on: int) -> int:
    """Test hook: symmetric (upper-triangle) tiles in the fused Muon kernel:
    1 always, 0 never, -1 chosen by the shape (the default)."""
    return _lib.ttt_dbg_ns_symmetric(int(on))


def ttt_thread_release() -> int:
    """Waits for and destroys the calling thread's side streams and events
    (created by the tensor-core path's shifted-mode calls); later calls create
    them again. Returns the status."""
    return _lib.ttt_thread_release()


def ttt_dbg_grad_pairs(on: bool) -> None:
    """Test hook: the chunk gradient on CTA pairs (on, the default in the
    single-GPU build) or on one-CTA clusters sharing E by multicast (off)."""
    rc = _lib.ttt_dbg_grad_pairs(int(bool(on)))
    if rc != TTT_OK:
        raise TTTError(rc, "ttt_dbg_grad_pairs")


def ttt_dbg_ns_tiles(bns: int, bnx: int) -> None:
    """Test hook: column-tile widths of the fused Muon kernel (0 = by shape)."""
    rc = _lib.ttt_dbg_ns_tiles(int(bns), int(bnx))
    if rc != TTT_OK:
        raise TTTError(rc, "ttt_dbg_ns_tiles")


def ttt_dbg_ns_trace(on: bool) -> int:
    """Test hook: record the fused Muon kernel's phase timeline (include/ttt_debug.h)."""
    return _lib.ttt_dbg_ns_trace(int(on))


def ttt_dbg_ns_trace_read(n: int = 96):
    """Test hook: the last traced launch's timestamps (ns) as a list of n ints."""
    buf = (ctypes.c_ulonglong * n)()
    rc = _lib.ttt_dbg_ns_trace_read(buf, n)
    if rc != TTT_OK:
        raise TTTError(rc, "ttt_dbg_ns_trace_read")
    return list(buf)


def ttt_dbg_ns_plan(cfg: ttt_cfg):
    """Test hook: (grid CTAs, CTAs resident at once) of the fused Muon kernel."""
    grid, res = c_int(0), c_int(0)
    rc = _lib.ttt_dbg_ns_plan(ctypes.byref(cfg), ctypes.byref(grid), ctypes.byref(res))
    if rc != TTT_OK:
        raise TTTError(rc, "ttt_dbg_ns_plan")
    return grid.value, res.value


def ttt_dbg_ns_force_grid(ctas: int) -> None:
    """Test hook: cap the fused Muon kernel's grid (0 = one CTA per SM)."""
    rc = _lib.ttt_dbg_ns_force_grid(int(ctas))
    if rc != TTT_OK:
        raise TTTError(rc, "ttt_dbg_ns_force_grid")


def ttt_dbg_split_mask(mask: int) -> None:
    """Test hook: stages with split operands in SPLIT precision (bit 0 keys'
    forward, bit 1 gradient, bit 2 Newton-Schulz; default 7)."""
    rc = _lib.ttt_dbg_split_mask(int(mask))
    if rc != TTT_OK:
        raise TTTError(rc, "ttt_dbg_split_mask")


def ttt_dbg_stall_next_linear() -> None:
    """Test hook: the next linear-kernel launch withholds its loads and times out."""
    _lib.ttt_dbg_stall_next_linear()


def ttt_dbg_stall_next_fwd() -> None:
    """Test hook: the next tensor-core forward launch withholds its loads and times out."""
    _lib.ttt_dbg_stall_next_fwd()


def ttt_dbg_stall_next_ns() -> None:
    """Test hook: the next fused Muon launch loses one item's completion signal."""
    _lib.ttt_dbg_stall_next_ns()


def ttt_prof_enable(on: bool) -> None:
    _lib.ttt_prof_enable(int(on))


def ttt_prof_reset() -> None:
    _lib.ttt_prof_reset()


def ttt_prof_read(kind: int):
    """(total event ms, timed launches, launches) of one kernel class since the last reset."""
    ms, timed, n = ctypes.c_double(0), ctypes.c_longlong(0), ctypes.c_longlong(0)
    rc = _lib.ttt_prof_read(kind, ctypes.byref(ms), ctypes.byref(timed), ctypes.byref(n))
    if rc != TTT_OK:
        raise TTTError(rc, "ttt_prof_read")
    return ms.value, timed.value, n.value


def ttt_launch_count() -> int:
    return _lib.ttt_launch_count()


def ttt_kernel_name(kind: int) -> str:
    return _lib.ttt_kernel_name(kind).decode()


# ----------------------------------------------------------------- helpers
class CfgHolder:
    """A ttt_cfg plus the host update-mask buffer it points to (kept alive)."""

    def __init__(self, cfg: ttt_cfg, mask: Optional[np.ndarray]):
        self.cfg = cfg
        self.mask = mask


def cfg_from_spec(spec, impl: int = TTT_IMPL_AUTO, check_finite: bool = False,
                  timeout_us: int = 0, T: Optional[int] = None,
                  precision: int = TTT_PREC_SPLIT) -> CfgHolder:
    """A ttt_cfg for a LayerSpec-like workload description."""
    c = ttt_cfg_default()
    c.B, c.H = spec.B, spec.H
    c.T = spec.T if T is None else T
    c.d, c.dh, c.chunk = spec.d, spec.dh, spec.chunk
    c.fast_net = TTT_NET_SWIGLU if spec.fast_net == "swiglu" else TTT_NET_LINEAR
    c.loss = TTT_LOSS_IP if spec.loss == "ip" else TTT_LOSS_MSE
    c.mode = {"shifted": TTT_MODE_SHIFTED, "single": TTT_MODE_SINGLE, "inclusive": TTT_MODE_INCLUSIVE}[spec.mode]
    c.dtype = TTT_DTYPE_F32 if spec.dtype == "fp32" else TTT_DTYPE_BF16
    c.muon = int(spec.muon)
    c.ns_iters = spec.ns_iters
    c.wnorm = int(spec.wnorm)
    c.step = spec.step
    c.impl = impl
    c.precision = precision
    c.check_finite = int(check_finite)
    c.timeout_us = timeout_us
    c.momentum = float(getattr(spec, "momentum", 0.0))
    c.lr_per_matrix = int(bool(getattr(spec, "lr_per_matrix", False)))
    n_chunks = (c.T + c.chunk - 1) // c.chunk
    mask = np.ascontiguousarray(spec.replace(T=c.T).update_mask(), dtype=np.uint8)
    assert mask.size == n_chunks
    if mask.all():
        mask = None
    else:
        c.update_mask = mask.ctypes.data
    return CfgHolder(c, mask)


def weight_shapes(cfg: ttt_cfg) -> Sequence[tuple]:
    if cfg.fast_net == TTT_NET_SWIGLU:
        return [(cfg.dh, cfg.d), (cfg.d, cfg.dh), (cfg.dh, cfg.d)]
    return [(cfg.d, cfg.d)]


def _check_layer_tensors(cfg: ttt_cfg, Q, K, V, lr, W0: Sequence) -> None:
    """Shapes, dtypes and device of the layer's inputs against the configuration
    (the C ABI sees only addresses): Q, K, V [B, H, T, d] in the storage type;
    lr [B, H, T] or [B, H, T, n_w] fp32; W0_j [H, out, in] (or [B, H, out, in]) fp32."""
    import torch
    tdt = torch.bfloat16 if cfg.dtype == TTT_DTYPE_BF16 else torch.float32
    shapes = weight_shapes(cfg)
    want = [("Q", Q, (cfg.B, cfg.H, cfg.T, cfg.d), tdt), ("K", K, (cfg.B, cfg.H, cfg.T, cfg.d), tdt),
            ("V", V, (cfg.B, cfg.H, cfg.T, cfg.d), tdt),
            ("lr", lr, (cfg.B, cfg.H, cfg.T) + ((len(shapes),) if cfg.lr_per_matrix else ()), torch.float32)]
    if len(W0) != len(shapes):
        raise ValueError(f"W0: {len(shapes)} matrices expected, got {len(W0)}")
    lead = (cfg.B, cfg.H) if cfg.w0_per_batch else (cfg.H,)
    want += [(f"W0_{j + 1}", w, lead + s, torch.float32) for j, (w, s) in enumerate(zip(W0, shapes))]
    for name, t, shape, dt in want:
        if tuple(t.shape) != shape or t.dtype != dt:
            raise ValueError(f"{name}: expected {shape} {dt}, got {tuple(t.shape)} {t.dtype}")
        if t.device != Q.device:
            raise ValueError(f"{name} is on {t.device}, Q on {Q.device}")


def layer(holder: CfgHolder, Q, K, V, lr, W0: Sequence, stream=None, sync: bool = True):
    """Allocate outputs and workspace (torch, on Q's device) and run ttt_fwd.

    Returns (O, [Wf...]). With ``sync`` the status word is read back and a
    device-side error raises TTTError.
    """
    import torch
    cfg = holder.cfg
    _check_layer_tensors(cfg, Q, K, V, lr, W0)
    dev = Q.device
    O = torch.empty_like(Q)
    Wf = [torch.empty((cfg.B, cfg.H) + s, dtype=torch.float32, device=dev)
          for s in weight_shapes(cfg)]
    ws = torch.empty(ttt_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    w0 = list(W0) + [None] * (3 - len(W0))
    wf = Wf + [None] * (3 - len(Wf))
    ttt_fwd(cfg, Q, K, V, lr, w0[0], w0[1], w0[2], O, wf[0], wf[1], wf[2], ws, stream)
    if sync:
        rc = ttt_status(ws, stream)
        if rc != TTT_OK:
            raise TTTError(rc, "ttt_fwd (device)")
    return O, Wf
