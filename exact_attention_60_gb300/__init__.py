"""GB300-native FlashAttention-2 forward: a C-ABI CUDA library and its thin binding.

``fa_fwd`` and friends mirror include/fa.h one to one (see ``_native``);
``attention`` allocates the outputs with torch and raises on any error status.
"""
from __future__ import annotations

import math

from ._native import (FA_DTYPE_BF16, FA_DTYPE_FP16, FA_ERR_CUDA, FA_ERR_INVALID_ARG,
                      FA_ERR_TIMEOUT, FA_ERR_UNSUPPORTED, FA_OK, FA_SCHED_BAND, FA_SCHED_SPLIT,
                      FA_SCHED_TABLE, FA_SCHED_WHOLE, fa_bwd, fa_bwd_masked,
                      fa_bwd_strided, fa_bwd_workspace_size,
                      fa_debug_set, fa_fwd, fa_fwd_host, fa_fwd_host_workspace_size,
                      fa_fwd_noalloc, fa_fwd_schedule, fa_fwd_strided, fa_fwd_window,
                      fa_fwd_workspace_size,
                      fa_fwd_ws, fa_last_device_status, fa_status_string)


class FaError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(fa_status_string(status))
        self.status = status


_workspaces = {}


def workspace_for(B, H, Lq, Lk, D, causal, device):
    """A cached device workspace large enough for fa_fwd_ws on this problem (or None)."""
    import torch
    st, nbytes = fa_fwd_workspace_size(B, H, Lq, Lk, D, causal)
    if st != FA_OK:
        raise FaError(st)
    if nbytes == 0:
        return None, 0
    key = (torch.device(device).index, )
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws, ws.numel()


def attention(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
              stream=None, split: bool = True, window=None, kv_len=None):
    """O, LSE = exact attention of contiguous bf16 CUDA tensors q [B,H,Lq,D], k/v [B,H,Lk,D].

    Allocates ``out`` (bf16 [B,H,Lq,D]) and ``lse`` (fp32 [B,H,Lq]) if not given.  With
    ``split`` (default) it calls fa_fwd_ws with a cached workspace, so the library may
    split key ranges across SMs; ``split=False`` calls fa_fwd.  Calls that share the
    cached workspace (same device) must be ordered on one stream.

    ``window=(left, right)`` restricts row i to keys i - left <= j <= i + right (-1:
    unbounded side) and calls fa_fwd_window; with ``causal`` the band is cut at the
    diagonal (right = 0).

    q, k, v (and ``out``) may also be fp16, or strided views of shape [B, H, L, D] with a
    contiguous last dimension (for instance slices of a packed [B, L, 3, H, D] projection);
    those calls go to fa_fwd_strided.  ``out`` defaults to a contiguous tensor of q's dtype.

    ``kv_len`` (an int32 CUDA tensor of B key counts) masks keys j >= kv_len[b] of batch b
    (key padding, on top of ``causal`` / ``window``); a row left without keys gets O = 0
    and LSE = -inf.
    """
    import torch
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dtype = q.dtype
    if dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q, k, v must be bf16 or fp16")
    for t in (q, k, v):
        if t.dtype != dtype or not t.is_cuda or t.dim() != 4 or t.stride(3) != 1:
            raise ValueError("q, k, v must be CUDA tensors of one dtype, [B, H, L, D], last dim contiguous")
    if tuple(k.shape) != (B, H, Lk, D) or tuple(v.shape) != (B, H, Lk, D):
        raise ValueError("k and v must be [B, H, Lk, D] matching q")
    if out is None:
        out = torch.empty((B, H, Lq, D), device=q.device, dtype=dtype)
    if lse is None:
        lse = torch.empty((B, H, Lq), device=q.device, dtype=torch.float32)
    if lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor")
    if kv_len is not None and (kv_len.dtype != torch.int32 or not kv_len.is_cuda
                               or kv_len.numel() != B or not kv_len.is_contiguous()):
        raise ValueError("kv_len must be a contiguous int32 CUDA tensor of B entries")
    plain = (dtype == torch.bfloat16 and kv_len is None
             and all(t.is_contiguous() for t in (q, k, v, out)))
    if not plain:
        if out.dtype != dtype or out.shape != q.shape or out.stride(3) != 1:
            raise ValueError("out must have q's dtype and shape and a contiguous last dim")
        left, right = (-1, 0 if causal else -1) if window is None else (int(window[0]), int(window[1]))
        if window is not None and causal:
            right = 0
        ws, nbytes = (workspace_for(B, H, Lq, Lk, D, False, q.device)
                      if split and (left, right) == (-1, -1) else (None, 0))
        code = FA_DTYPE_FP16 if dtype == torch.float16 else FA_DTYPE_BF16
        if kv_len is not None:
            ws, nbytes = None, 0
        st = fa_fwd_strided(q, q.stride()[:3], k, k.stride()[:3], v, v.stride()[:3], out,
                            out.stride()[:3], lse, kv_len, B, H, Lq, Lk, D, left, right, scale,
                            code, ws, nbytes, stream)
        if st != FA_OK:
            raise FaError(st)
        return out, lse
    if window is not None:
        left, right = (int(x) for x in window)
        if causal:
            right = 0
        st = fa_fwd_window(q, k, v, out, lse, B, H, Lq, Lk, D, left, right, scale, stream)
    elif split:
        ws, nbytes = workspace_for(B, H, Lq, Lk, D, causal, q.device)
        st = fa_fwd_ws(q, k, v, out, lse, B, H, Lq, Lk, D, causal, scale, ws, nbytes, stream)
    else:
        st = fa_fwd(q, k, v, out, lse, B, H, Lq, Lk, D, causal, scale, stream)
    if st != FA_OK:
        raise FaError(st)
    return out, lse


_bwd_workspaces = {}


def attention_backward(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None,
                       dq=None, dk=None, dv=None, stream=None, window=None, kv_len=None):
    """dQ, dK, dV of ``attention`` given its inputs, its outputs ``o``/``lse`` and
    ``do`` = dLoss/dO (contiguous bf16 / fp32 CUDA tensors of the forward's shapes).
    Allocates the gradients if not given; uses a cached per-device workspace, so calls
    on one device must be ordered on one stream.  ``window`` and ``kv_len`` as for
    ``attention`` (fa_bwd_masked)."""
    import torch
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dtype = q.dtype
    if dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q, k, v, o, do must be bf16 or fp16")
    for t in (q, k, v, o, do):
        if t.dtype != dtype or not t.is_cuda or t.dim() != 4 or t.stride(3) != 1:
            raise ValueError("q, k, v, o, do must be CUDA tensors of one dtype, [B, H, L, D], last dim contiguous")
    if lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 CUDA tensor")
    dq = torch.empty((B, H, Lq, D), dtype=dtype, device=q.device) if dq is None else dq
    dk = torch.empty((B, H, Lk, D), dtype=dtype, device=q.device) if dk is None else dk
    dv = torch.empty((B, H, Lk, D), dtype=dtype, device=q.device) if dv is None else dv
    st, nbytes = fa_bwd_workspace_size(B, H, Lq, Lk, D, causal)
    if st != FA_OK:
        raise FaError(st)
    key = (torch.device(q.device).index, )
    ws = _bwd_workspaces.get(key)
    if ws is None or ws.numel() < max(nbytes, 256):
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
        _bwd_workspaces[key] = ws
    if kv_len is not None and (kv_len.dtype != torch.int32 or kv_len.numel() != B
                               or not kv_len.is_cuda or not kv_len.is_contiguous()):
        raise ValueError("kv_len must be a contiguous int32 CUDA tensor of B entries")
    plain = dtype == torch.bfloat16 and all(t.is_contiguous() for t in (q, k, v, o, do, dq, dk, dv))
    if not plain:
        left, right = (-1, 0 if causal else -1) if window is None else (int(window[0]), int(window[1]))
        if window is not None and causal:
            right = 0
        code = FA_DTYPE_FP16 if dtype == torch.float16 else FA_DTYPE_BF16
        st = fa_bwd_strided(q, q.stride()[:3], k, k.stride()[:3], v, v.stride()[:3], o, o.stride()[:3],
                            do, do.stride()[:3], lse, dq, dq.stride()[:3], dk, dk.stride()[:3], dv,
                            dv.stride()[:3], kv_len, B, H, Lq, Lk, D, left, right, scale, code, ws,
                            ws.numel(), stream)
    elif window is None and kv_len is None:
        st = fa_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, Lq, Lk, D, causal, scale, ws, ws.numel(),
                    stream)
    else:
        left, right = (-1, 0 if causal else -1) if window is None else (int(window[0]), int(window[1]))
        if window is not None and causal:
            right = 0
        st = fa_bwd_masked(q, k, v, o, do, lse, dq, dk, dv, kv_len, B, H, Lq, Lk, D, left, right,
                           scale, ws, ws.numel(), stream)
    if st != FA_OK:
        raise FaError(st)
    return dq, dk, dv


def flash_attention(q, k, v, causal: bool = False, scale: float | None = None, window=None,
                    kv_len=None):
    """Differentiable exact attention: ``attention`` forward, ``attention_backward``
    for the gradients (torch.autograd glue only)."""
    import torch

    class _Fn(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v):
            o, lse = attention(q, k, v, causal=causal, scale=scale, window=window, kv_len=kv_len)
            ctx.save_for_backward(q, k, v, o, lse)
            return o

        @staticmethod
        def backward(ctx, do):
            q, k, v, o, lse = ctx.saved_tensors
            return attention_backward(q, k, v, o, lse, do.contiguous(), causal=causal, scale=scale,
                                      window=window, kv_len=kv_len)

    return _Fn.apply(q, k, v)


_host_workspaces = {}


def attention_from_host(q, k, v, causal: bool = False, scale: float | None = None, out=None,
                        lse=None, device=None, window=None, stream=None):
    """Exact attention of host tensors through the C call fa_fwd_host.

    ``q`` [B,H,Lq,D], ``k``/``v`` [B,H,Lk,D] are contiguous bf16 CPU tensors (pinned for
    the copies to overlap the kernels).  The library cuts the (batch, head) slices into
    chunks and overlaps their uploads, kernels and downloads on three streams.  Returns
    host ``out`` (bf16) and ``lse`` (fp32), allocated pinned if not given, complete once
    ``stream`` (default: the device's current stream) has finished.  The device
    workspace is cached per device, so calls on one device must be ordered on one
    stream.  ``window`` as for ``attention``.
    """
    import torch
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 CPU tensors [B, H, L, D]")
    if tuple(k.shape) != (B, H, Lk, D) or tuple(v.shape) != (B, H, Lk, D):
        raise ValueError("k and v must be [B, H, Lk, D] matching q")
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    if lse is None:
        lse = torch.empty((B, H, Lq), dtype=torch.float32).pin_memory()
    if (out.dtype != torch.bfloat16 or out.is_cuda or tuple(out.shape) != tuple(q.shape)
            or not out.is_contiguous() or lse.dtype != torch.float32 or lse.is_cuda
            or tuple(lse.shape) != (B, H, Lq) or not lse.is_contiguous()):
        raise ValueError("out and lse must be contiguous CPU tensors: bf16 like q, fp32 [B, H, Lq]")
    if window is None:
        left, right = -1, (0 if causal else -1)
    else:
        left, right = int(window[0]), (0 if causal else int(window[1]))
    with torch.cuda.device(dev):
        st, nbytes = fa_fwd_host_workspace_size(B, H, Lq, Lk, D, left, right)
        if st != FA_OK:
            raise FaError(st)
        ws = _host_workspaces.get(dev.index)
        if ws is None or ws.numel() < max(nbytes, 256):
            ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
            _host_workspaces[dev.index] = ws
        if stream is None:
            stream = torch.cuda.current_stream(dev)
        st = fa_fwd_host(q, k, v, out, lse, B, H, Lq, Lk, D, left, right, scale, ws, ws.numel(),
                         stream)
    if st != FA_OK:
        raise FaError(st)
    return out, lse
