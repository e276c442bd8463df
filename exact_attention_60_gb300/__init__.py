"""GB300-native FlashAttention-2 forward: a C-ABI CUDA library and its thin binding.

``fa_fwd`` and friends mirror include/fa.h one to one (see ``_native``);
``attention`` allocates the outputs with torch and raises on any error status.
"""
from __future__ import annotations

import math

from ._native import (FA_DTYPE_BF16, FA_DTYPE_FP16, FA_ERR_CUDA, FA_ERR_INVALID_ARG,
                      FA_ERR_TIMEOUT, FA_ERR_UNSUPPORTED, FA_OK, fa_bwd, fa_bwd_masked,
                      fa_bwd_strided, fa_bwd_workspace_size,
                      fa_debug_set, fa_fwd, fa_fwd_noalloc, fa_fwd_strided, fa_fwd_window,
                      fa_fwd_workspace_size, fa_fwd_ws, fa_last_device_status, fa_status_string)


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


def attention_from_host(q, k, v, causal: bool = False, scale: float | None = None, out=None,
                        lse=None, chunks: int | None = None, device=None, window=None):
    """Exact attention of host tensors: copies in, computes, copies out, overlapped.

    ``q`` [B,H,Lq,D], ``k``/``v`` [B,H,Lk,D] are contiguous bf16 CPU tensors (pinned for
    the copies to overlap).  The (batch, head) slices are cut into ``chunks`` groups;
    group i+1 travels to the GPU while group i is computed and group i-1 travels back,
    on three streams ordered by events.  Returns host ``out`` (bf16) and ``lse`` (fp32),
    allocated pinned if not given.  Device buffers are allocated per call.  ``window``
    as for ``attention``.
    """
    import torch
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    BH = B * H
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    if lse is None:
        lse = torch.empty((B, H, Lq), dtype=torch.float32).pin_memory()
    if chunks is None:
        chunks = default_chunks(BH, Lq, Lk, causal)
    chunks = max(1, min(int(chunks), BH))
    dq = torch.empty((BH, Lq, D), dtype=torch.bfloat16, device=dev)
    dk = torch.empty((BH, Lk, D), dtype=torch.bfloat16, device=dev)
    dv = torch.empty((BH, Lk, D), dtype=torch.bfloat16, device=dev)
    do = torch.empty((BH, Lq, D), dtype=torch.bfloat16, device=dev)
    dl = torch.empty((BH, Lq), dtype=torch.float32, device=dev)
    hq, hk, hv = q.reshape(BH, Lq, D), k.reshape(BH, Lk, D), v.reshape(BH, Lk, D)
    ho, hl = out.view(BH, Lq, D), lse.view(BH, Lq)
    main = torch.cuda.current_stream(dev)
    # uploads on one stream (parallel upload streams measured slower: they make the
    # first chunk's tensors arrive later), kernels on a second, downloads on a third
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    for s in (s_in, s_cmp, s_out):
        s.wait_stream(main)
    bounds = [(BH * i // chunks, BH * (i + 1) // chunks) for i in range(chunks)]
    for a, b in bounds:
        if a == b:
            continue
        with torch.cuda.stream(s_in):
            dq[a:b].copy_(hq[a:b], non_blocking=True)
            dk[a:b].copy_(hk[a:b], non_blocking=True)
            dv[a:b].copy_(hv[a:b], non_blocking=True)
        s_cmp.wait_stream(s_in)
        with torch.cuda.stream(s_cmp):
            n = b - a
            attention(dq[a:b].view(1, n, Lq, D), dk[a:b].view(1, n, Lk, D), dv[a:b].view(1, n, Lk, D),
                      causal=causal, scale=scale, out=do[a:b].view(1, n, Lq, D),
                      lse=dl[a:b].view(1, n, Lq), stream=s_cmp, window=window)
        s_out.wait_stream(s_cmp)
        with torch.cuda.stream(s_out):
            ho[a:b].copy_(do[a:b], non_blocking=True)
            hl[a:b].copy_(dl[a:b], non_blocking=True)
    main.wait_stream(s_out)
    for t in (dq, dk, dv, do, dl):
        for s in (s_in, s_cmp, s_out):
            t.record_stream(s)
    return out, lse


def default_chunks(BH: int, Lq: int, Lk: int, causal: bool) -> int:
    """Chunks for attention_from_host: enough to overlap the copies with the kernels,
    few enough that each kernel still spreads over the GPU (at least 256 query-tile
    pairs per chunk, at most 8 chunks)."""
    units = BH * ((Lq + 255) // 256)
    return max(1, min(8, units // 256, BH))
