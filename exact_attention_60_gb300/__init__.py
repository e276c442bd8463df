"""GB300-native FlashAttention-2 forward: a C-ABI CUDA library and its thin binding.

``fa_fwd`` and friends mirror include/fa.h one to one (see ``_native``);
``attention`` allocates the outputs with torch and raises on any error status.
"""
from __future__ import annotations

import math

from ._native import (FA_ERR_CUDA, FA_ERR_INVALID_ARG, FA_ERR_TIMEOUT, FA_ERR_UNSUPPORTED,
                      FA_OK, fa_debug_set, fa_fwd, fa_last_device_status, fa_status_string)


class FaError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(fa_status_string(status))
        self.status = status


def attention(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
              stream=None):
    """O, LSE = exact attention of contiguous bf16 CUDA tensors q [B,H,Lq,D], k/v [B,H,Lk,D].

    Allocates ``out`` (bf16 [B,H,Lq,D]) and ``lse`` (fp32 [B,H,Lq]) if not given.
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
    st = fa_fwd(q, k, v, out, lse, B, H, Lq, Lk, D, causal, scale, stream)
    if st != FA_OK:
        raise FaError(st)
    return out, lse
