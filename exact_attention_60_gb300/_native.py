"""ctypes binding of libfa.so: the C ABI of include/fa.h under the same names.

Argument marshalling only -- every step of the attention runs in the CUDA
library.  Loading fails loudly (``RuntimeError``) when the library has not been
built; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_DTYPE_BF16 = 0
FA_DTYPE_FP16 = 1
FA_SCHED_WHOLE = 0
FA_SCHED_SPLIT = 1
FA_SCHED_BAND = 2
FA_SCHED_TABLE = 3

# Every symbol include/fa.h declares.
EXPORTED = ("fa_fwd", "fa_fwd_workspace_size", "fa_fwd_schedule", "fa_fwd_ws", "fa_fwd_window", "fa_fwd_strided",
            "fa_fwd_noalloc", "fa_fwd_host_workspace_size", "fa_fwd_host",
            "fa_bwd_workspace_size", "fa_bwd", "fa_bwd_masked", "fa_bwd_strided", "fa_status_string",
            "fa_last_device_status",
            "fa_debug_set")

_lib = None


def load(path: str = LIB) -> ctypes.CDLL:
    """Load libfa.so (once) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing: run __graft_entry__.build() "
                           "(or python -m exact_attention_60_gb300.build) first")
    lib = ctypes.CDLL(path)
    vp = ctypes.c_void_p
    lib.fa_fwd.restype = ctypes.c_int
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                           ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, vp]
    lib.fa_fwd_workspace_size.restype = ctypes.c_int
    lib.fa_fwd_workspace_size.argtypes = [ctypes.c_int] * 6 + [ctypes.POINTER(ctypes.c_size_t)]
    lib.fa_fwd_schedule.restype = ctypes.c_int
    lib.fa_fwd_schedule.argtypes = [ctypes.c_int] * 6 + [ctypes.POINTER(ctypes.c_int)]
    lib.fa_fwd_ws.restype = ctypes.c_int
    lib.fa_fwd_ws.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                              ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, vp,
                              ctypes.c_size_t, vp]
    lib.fa_fwd_window.restype = ctypes.c_int
    lib.fa_fwd_window.argtypes = [vp, vp, vp, vp, vp] + [ctypes.c_int] * 7 + [ctypes.c_float, vp]
    lp3 = ctypes.POINTER(ctypes.c_longlong)
    lib.fa_fwd_strided.restype = ctypes.c_int
    lib.fa_fwd_strided.argtypes = [vp, lp3, vp, lp3, vp, lp3, vp, lp3, vp, vp] + [ctypes.c_int] * 7 + \
        [ctypes.c_float, ctypes.c_int, vp, ctypes.c_size_t, vp]
    lib.fa_fwd_noalloc.restype = ctypes.c_int
    lib.fa_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, vp]
    lib.fa_fwd_host_workspace_size.restype = ctypes.c_int
    lib.fa_fwd_host_workspace_size.argtypes = [ctypes.c_int] * 7 + [ctypes.POINTER(ctypes.c_size_t)]
    lib.fa_fwd_host.restype = ctypes.c_int
    lib.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp] + [ctypes.c_int] * 7 + [ctypes.c_float, vp,
                                                                          ctypes.c_size_t, vp]
    lib.fa_bwd_workspace_size.restype = ctypes.c_int
    lib.fa_bwd_workspace_size.argtypes = [ctypes.c_int] * 6 + [ctypes.POINTER(ctypes.c_size_t)]
    lib.fa_bwd.restype = ctypes.c_int
    lib.fa_bwd.argtypes = [vp] * 9 + [ctypes.c_int] * 6 + [ctypes.c_float, vp, ctypes.c_size_t, vp]
    lib.fa_bwd_masked.restype = ctypes.c_int
    lib.fa_bwd_masked.argtypes = [vp] * 10 + [ctypes.c_int] * 7 + [ctypes.c_float, vp, ctypes.c_size_t, vp]
    lib.fa_bwd_strided.restype = ctypes.c_int
    lib.fa_bwd_strided.argtypes = [vp, lp3, vp, lp3, vp, lp3, vp, lp3, vp, lp3, vp, vp, lp3, vp, lp3,
                                   vp, lp3, vp] + [ctypes.c_int] * 7 + \
        [ctypes.c_float, ctypes.c_int, vp, ctypes.c_size_t, vp]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_status_string.argtypes = [ctypes.c_int]
    lib.fa_last_device_status.restype = ctypes.c_int
    lib.fa_last_device_status.argtypes = [vp]
    lib.fa_debug_set.restype = ctypes.c_int
    lib.fa_debug_set.argtypes = [ctypes.c_uint, ctypes.c_ulonglong]
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr() or None
    return int(x) or None


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream or None
    return int(s) or None


def fa_fwd(Q, K, V, O, LSE, B, H, Lq, Lk, D, causal, scale, stream=None) -> int:
    """C ``fa_fwd``.  Pointers may be ints or tensors (their ``data_ptr()``);
    ``stream`` may be an int handle, a torch stream, or None (torch's current stream)."""
    return load().fa_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), int(B), int(H),
                         int(Lq), int(Lk), int(D), int(bool(causal)), float(scale),
                         _stream(stream))


def fa_fwd_workspace_size(B, H, Lq, Lk, D, causal):
    """C ``fa_fwd_workspace_size``: returns (status, bytes)."""
    n = ctypes.c_size_t(0)
    st = load().fa_fwd_workspace_size(int(B), int(H), int(Lq), int(Lk), int(D),
                                      int(bool(causal)), ctypes.byref(n))
    return st, int(n.value)


def fa_fwd_schedule(B, H, Lq, Lk, D, causal):
    """C ``fa_fwd_schedule``: returns (status, FA_SCHED_* code)."""
    sc = ctypes.c_int(0)
    st = load().fa_fwd_schedule(int(B), int(H), int(Lq), int(Lk), int(D), int(bool(causal)),
                                ctypes.byref(sc))
    return st, int(sc.value)


def fa_fwd_ws(Q, K, V, O, LSE, B, H, Lq, Lk, D, causal, scale, workspace, workspace_bytes,
              stream=None) -> int:
    """C ``fa_fwd_ws``; ``workspace`` may be an int, a tensor or None."""
    return load().fa_fwd_ws(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), int(B), int(H),
                            int(Lq), int(Lk), int(D), int(bool(causal)), float(scale),
                            _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_fwd_window(Q, K, V, O, LSE, B, H, Lq, Lk, D, window_left, window_right, scale,
                  stream=None) -> int:
    """C ``fa_fwd_window``: keys i - window_left <= j <= i + window_right (-1: unbounded)."""
    return load().fa_fwd_window(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), int(B), int(H),
                                int(Lq), int(Lk), int(D), int(window_left), int(window_right),
                                float(scale), _stream(stream))


def _strides3(st):
    """Three element strides {batch, head, row} as a C array (None stays None)."""
    if st is None:
        return None
    a, b, c = (int(x) for x in st)
    return (ctypes.c_longlong * 3)(a, b, c)


def fa_fwd_strided(Q, q_stride, K, k_stride, V, v_stride, O, o_stride, LSE, kv_len, B, H, Lq, Lk,
                   D, window_left, window_right, scale, dtype, workspace=None, workspace_bytes=0,
                   stream=None) -> int:
    """C ``fa_fwd_strided``; strides are sequences of three element strides; ``kv_len`` a
    device int32 array of per-batch key counts, or None."""
    return load().fa_fwd_strided(_ptr(Q), _strides3(q_stride), _ptr(K), _strides3(k_stride),
                                 _ptr(V), _strides3(v_stride), _ptr(O), _strides3(o_stride),
                                 _ptr(LSE), _ptr(kv_len), int(B), int(H), int(Lq), int(Lk), int(D),
                                 int(window_left), int(window_right), float(scale), int(dtype),
                                 _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_fwd_noalloc(Q, K, V, O, LSE, B, H, Lq, Lk, D, causal, scale, stream=None) -> int:
    """C ``fa_fwd_noalloc``: fa_fwd_ws with the library's built-in scratch, for
    callers that cannot allocate device memory (see include/fa.h)."""
    return load().fa_fwd_noalloc(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), int(B), int(H),
                                 int(Lq), int(Lk), int(D), int(bool(causal)), float(scale),
                                 _stream(stream))


def fa_fwd_host_workspace_size(B, H, Lq, Lk, D, window_left, window_right):
    """C ``fa_fwd_host_workspace_size``: returns (status, bytes)."""
    n = ctypes.c_size_t(0)
    st = load().fa_fwd_host_workspace_size(int(B), int(H), int(Lq), int(Lk), int(D),
                                           int(window_left), int(window_right), ctypes.byref(n))
    return st, int(n.value)


def fa_fwd_host(Q, K, V, O, LSE, B, H, Lq, Lk, D, window_left, window_right, scale, workspace,
                workspace_bytes, stream=None) -> int:
    """C ``fa_fwd_host``: Q, K, V, O, LSE are HOST pointers (ints or CPU tensors, pinned for
    overlap); ``workspace`` is device memory of fa_fwd_host_workspace_size bytes."""
    return load().fa_fwd_host(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), int(B), int(H),
                              int(Lq), int(Lk), int(D), int(window_left), int(window_right),
                              float(scale), _ptr(workspace), int(workspace_bytes),
                              _stream(stream))


def fa_bwd_workspace_size(B, H, Lq, Lk, D, causal):
    """C ``fa_bwd_workspace_size``: returns (status, bytes)."""
    n = ctypes.c_size_t(0)
    st = load().fa_bwd_workspace_size(int(B), int(H), int(Lq), int(Lk), int(D),
                                      int(bool(causal)), ctypes.byref(n))
    return st, int(n.value)


def fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Lq, Lk, D, causal, scale, workspace,
           workspace_bytes, stream=None) -> int:
    """C ``fa_bwd``: gradients dQ, dK, dV of the forward attention given dO."""
    return load().fa_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ),
                         _ptr(dK), _ptr(dV), int(B), int(H), int(Lq), int(Lk), int(D),
                         int(bool(causal)), float(scale), _ptr(workspace), int(workspace_bytes),
                         _stream(stream))


def fa_bwd_masked(Q, K, V, O, dO, LSE, dQ, dK, dV, kv_len, B, H, Lq, Lk, D, window_left,
                  window_right, scale, workspace, workspace_bytes, stream=None) -> int:
    """C ``fa_bwd_masked``: fa_bwd under a band (-1 = unbounded side) and key padding."""
    return load().fa_bwd_masked(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ),
                                _ptr(dK), _ptr(dV), _ptr(kv_len), int(B), int(H), int(Lq), int(Lk),
                                int(D), int(window_left), int(window_right), float(scale),
                                _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd_strided(Q, q_stride, K, k_stride, V, v_stride, O, o_stride, dO, do_stride, LSE, dQ,
                   dq_stride, dK, dk_stride, dV, dv_stride, kv_len, B, H, Lq, Lk, D, window_left,
                   window_right, scale, dtype, workspace, workspace_bytes, stream=None) -> int:
    """C ``fa_bwd_strided``; strides are sequences of three element strides."""
    return load().fa_bwd_strided(_ptr(Q), _strides3(q_stride), _ptr(K), _strides3(k_stride), _ptr(V),
                                 _strides3(v_stride), _ptr(O), _strides3(o_stride), _ptr(dO),
                                 _strides3(do_stride), _ptr(LSE), _ptr(dQ), _strides3(dq_stride),
                                 _ptr(dK), _strides3(dk_stride), _ptr(dV), _strides3(dv_stride),
                                 _ptr(kv_len), int(B), int(H), int(Lq), int(Lk), int(D),
                                 int(window_left), int(window_right), float(scale), int(dtype),
                                 _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_status_string(status: int) -> str:
    return load().fa_status_string(int(status)).decode()


def fa_last_device_status(stream=None) -> int:
    return load().fa_last_device_status(_stream(stream))


def fa_debug_set(flags: int, wait_limit_ns: int) -> int:
    return load().fa_debug_set(int(flags), int(wait_limit_ns))
