"""GB300-native FlashAttention-2 forward: a C-ABI CUDA library and its thin binding.

``fa_fwd`` and friends mirror include/fa.h one to one (see ``_native``);
``attention`` allocates the outputs with torch and raises on any error status.
"""
from __future__ import annotations

import math

from ._native import (FA_ERR_CUDA, FA_ERR_INVALID_ARG, FA_ERR_TIMEOUT, FA_ERR_UNSUPPORTED,
                      FA_OK, fa_debug_set, fa_fwd, fa_fwd_noalloc, fa_fwd_workspace_size,
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
              stream=None, split: bool = True):
    """O, LSE = exact attention of contiguous bf16 CUDA tensors q [B,H,Lq,D], k/v [B,H,Lk,D].

    Allocates ``out`` (bf16 [B,H,Lq,D]) and ``lse`` (fp32 [B,H,Lq]) if not given.  With
    ``split`` (default) it calls fa_fwd_ws with a cached workspace, so the library may
    split key ranges across SMs; ``split=False`` calls fa_fwd.  Calls that share the
    cached workspace (same device) must be ordered on one stream.
    """
    import torch
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    if tuple(k.shape) != (B, H, Lk, D) or tuple(v.shape) != (B, H, Lk, D):
        raise ValueError("k and v must be [B, H, Lk, D] matching q")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Lq), device=q.device, dtype=torch.float32)
    if split:
        ws, nbytes = workspace_for(B, H, Lq, Lk, D, causal, q.device)
        st = fa_fwd_ws(q, k, v, out, lse, B, H, Lq, Lk, D, causal, scale, ws, nbytes, stream)
    else:
        st = fa_fwd(q, k, v, out, lse, B, H, Lq, Lk, D, causal, scale, stream)
    if st != FA_OK:
        raise FaError(st)
    return out, lse
