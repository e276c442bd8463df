"""fp64 CPU oracle for exact softmax attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product (the CUDA library and its
Python binding in ``exact_attention_60_gb300``) never imports it.

The arithmetic lives in ``attn_oracle.c`` (plain loops, double precision,
materialised score and probability rows); this module only compiles it with
gcc, loads it with ctypes and marshals numpy arrays.  See that file's header
for the passages each step follows:

* "Triton Ascend Attention" (skillmd.com), section 标准 Attention 计算流程:
  the three-stage definition softmax(Q K^T / sqrt(d_k)) V.
* wsisp.com post "FlashAttention-2 forward in Triton", the passage that FA
  computes exactly S = QK^T, P = softmax(S), O = PV, and the outer-kernel
  epilogue storing m + log(l) per row.
* "flash-attention-kernel" skill card: causal keeps ``offs_m >= offs_n``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle source into a shared library (gcc, OpenMP, -O2)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _dptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> np.ndarray:
    """Exact widening to a contiguous float64 array (bf16 values are exact in fp64)."""
    if hasattr(a, "detach"):  # a torch tensor: widen through float32, which holds bf16 exactly
        a = a.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


class OracleLib:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lp = ctypes.POINTER(ctypes.c_long)
        lib.oracle_attn_head.restype = ctypes.c_int
        lib.oracle_attn_head.argtypes = [dp, dp, dp, ctypes.c_long, ctypes.c_long,
                                         ctypes.c_long, ctypes.c_int, ctypes.c_double,
                                         lp, ctypes.c_long, dp, dp, dp, ctypes.c_int]
        lib.oracle_attn_full.restype = ctypes.c_int
        lib.oracle_attn_full.argtypes = [dp, dp, dp, ctypes.c_long, ctypes.c_long,
                                         ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                         ctypes.c_int, ctypes.c_double, dp, dp, dp,
                                         ctypes.c_int]
        lib.oracle_attn_head_window.restype = ctypes.c_int
        lib.oracle_attn_head_window.argtypes = [dp, dp, dp, ctypes.c_long, ctypes.c_long,
                                                ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                                ctypes.c_double, lp, ctypes.c_long, dp, dp, dp,
                                                ctypes.c_int]
        lib.oracle_attn_head_keypad.restype = ctypes.c_int
        lib.oracle_attn_head_keypad.argtypes = [dp, dp, dp, ctypes.c_long, ctypes.c_long,
                                                ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                                ctypes.c_long, ctypes.c_double, lp, ctypes.c_long,
                                                dp, dp, dp, ctypes.c_int]
        lib.oracle_attn_bwd_head_masked.restype = ctypes.c_int
        lib.oracle_attn_bwd_head_masked.argtypes = [dp, dp, dp, dp, ctypes.c_long, ctypes.c_long,
                                                    ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                                    ctypes.c_long, ctypes.c_double, dp, dp, dp,
                                                    ctypes.c_int]
        lib.oracle_attn_bwd_head.restype = ctypes.c_int
        lib.oracle_attn_bwd_head.argtypes = [dp, dp, dp, dp, ctypes.c_long, ctypes.c_long,
                                             ctypes.c_long, ctypes.c_int, ctypes.c_double,
                                             dp, dp, dp, ctypes.c_int]
        lib.oracle_attn_bwd_rows.restype = ctypes.c_int
        lib.oracle_attn_bwd_rows.argtypes = [dp, dp, dp, dp, ctypes.c_long, ctypes.c_long,
                                             ctypes.c_long, ctypes.c_int, ctypes.c_double,
                                             lp, ctypes.c_long, lp, ctypes.c_long, dp, dp, dp,
                                             dp, dp, ctypes.c_int]
        lib.oracle_attn_bwd_rows_masked.restype = ctypes.c_int
        lib.oracle_attn_bwd_rows_masked.argtypes = [dp, dp, dp, dp, ctypes.c_long, ctypes.c_long,
                                                    ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                                    ctypes.c_long, ctypes.c_double, lp, ctypes.c_long,
                                                    lp, ctypes.c_long, dp, dp, dp, dp, dp, ctypes.c_int]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        self.lib = lib
        self.path = path

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def attn_head(self, q, k, v, causal: bool, scale: float, rows=None,
                  want_p: bool = False, nthreads: int = 0):
        """Attention of one (batch, head) slice.

        q: [Lq, D]; k, v: [Lk, D].  ``rows``: query indices to compute (default all).
        Returns (O [n, D], LSE [n]) or (O, LSE, P [n, Lk]) with ``want_p``.
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        Lq, D = q.shape
        Lk = k.shape[0]
        if k.shape != (Lk, D) or v.shape != (Lk, D):
            raise ValueError("k and v must be [Lk, D] with the same D as q")
        if rows is None:
            n, rp = Lq, None
        else:
            rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
            n = rows_arr.shape[0]
            rp = rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_long))
        O = np.empty((n, D), dtype=np.float64)
        L = np.empty((n,), dtype=np.float64)
        P = np.empty((n, Lk), dtype=np.float64) if want_p else None
        rc = self.lib.oracle_attn_head(_dptr(q), _dptr(k), _dptr(v), Lq, Lk, D,
                                       int(bool(causal)), float(scale), rp, n,
                                       _dptr(O), _dptr(L), _dptr(P), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_attn_head failed with code {rc}")
        return (O, L, P) if want_p else (O, L)

    def attn_head_window(self, q, k, v, left: int, right: int, scale: float, rows=None,
                         want_p: bool = False, nthreads: int = 0):
        """Local attention of one (batch, head) slice: key j allowed for row i iff
        i - left <= j <= i + right (-1: unbounded).  Returns (O, LSE[, P])."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        Lq, D = q.shape
        Lk = k.shape[0]
        if k.shape != (Lk, D) or v.shape != (Lk, D):
            raise ValueError("k and v must be [Lk, D] with the same D as q")
        if rows is None:
            n, rp = Lq, None
        else:
            rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
            n = rows_arr.shape[0]
            rp = rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_long))
        O = np.empty((n, D), dtype=np.float64)
        L = np.empty((n,), dtype=np.float64)
        P = np.empty((n, Lk), dtype=np.float64) if want_p else None
        rc = self.lib.oracle_attn_head_window(_dptr(q), _dptr(k), _dptr(v), Lq, Lk, D, int(left),
                                              int(right), float(scale), rp, n, _dptr(O),
                                              _dptr(L), _dptr(P), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_attn_head_window failed with code {rc}")
        return (O, L, P) if want_p else (O, L)

    def attn_full_window(self, q, k, v, left: int, right: int, scale: float, nthreads: int = 0):
        """Local attention over contiguous [B, H, L, D] tensors: returns (O, LSE)."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, Lq, D = q.shape
        O = np.empty((B, H, Lq, D))
        L = np.empty((B, H, Lq))
        for b in range(B):
            for h in range(H):
                O[b, h], L[b, h] = self.attn_head_window(q[b, h], k[b, h], v[b, h], left, right,
                                                         scale, nthreads=nthreads)
        return O, L

    def attn_head_keypad(self, q, k, v, left: int, right: int, kv_len: int, scale: float,
                         rows=None, want_p: bool = False, nthreads: int = 0):
        """Band plus key padding (keys j >= kv_len masked) for one (batch, head) slice;
        rows without any allowed key give O = 0, LSE = -inf.  Returns (O, LSE[, P])."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        Lq, D = q.shape
        Lk = k.shape[0]
        if k.shape != (Lk, D) or v.shape != (Lk, D):
            raise ValueError("k and v must be [Lk, D] with the same D as q")
        if rows is None:
            n, rp = Lq, None
        else:
            rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
            n = rows_arr.shape[0]
            rp = rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_long))
        O = np.empty((n, D), dtype=np.float64)
        L = np.empty((n,), dtype=np.float64)
        P = np.empty((n, Lk), dtype=np.float64) if want_p else None
        rc = self.lib.oracle_attn_head_keypad(_dptr(q), _dptr(k), _dptr(v), Lq, Lk, D, int(left),
                                              int(right), int(kv_len), float(scale), rp, n,
                                              _dptr(O), _dptr(L), _dptr(P), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_attn_head_keypad failed with code {rc}")
        return (O, L, P) if want_p else (O, L)

    def attn_full_keypad(self, q, k, v, left: int, right: int, kv_len, scale: float,
                         nthreads: int = 0):
        """Band plus per-batch key padding over [B, H, L, D] tensors: (O, LSE)."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, Lq, D = q.shape
        O = np.empty((B, H, Lq, D))
        L = np.empty((B, H, Lq))
        for b in range(B):
            for h in range(H):
                O[b, h], L[b, h] = self.attn_head_keypad(q[b, h], k[b, h], v[b, h], left, right,
                                                         int(kv_len[b]), scale, nthreads=nthreads)
        return O, L

    def attn_bwd_head(self, q, k, v, do, causal: bool, scale: float, nthreads: int = 0):
        """Gradients (dQ, dK, dV) of one (batch, head) slice given dO = dLoss/dO."""
        q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
        Lq, D = q.shape
        Lk = k.shape[0]
        if k.shape != (Lk, D) or v.shape != (Lk, D) or do.shape != (Lq, D):
            raise ValueError("k, v must be [Lk, D] and do [Lq, D] with the same D as q")
        dq = np.empty((Lq, D))
        dk = np.empty((Lk, D))
        dv = np.empty((Lk, D))
        rc = self.lib.oracle_attn_bwd_head(_dptr(q), _dptr(k), _dptr(v), _dptr(do), Lq, Lk, D,
                                           int(bool(causal)), float(scale), _dptr(dq), _dptr(dk),
                                           _dptr(dv), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_attn_bwd_head failed with code {rc}")
        return dq, dk, dv

    def attn_bwd_rows(self, q, k, v, do, causal: bool, scale: float, qrows, krows,
                      nthreads: int = 0):
        """Gradients of one (batch, head) slice at sampled outputs: dQ at query rows
        ``qrows``, dK and dV at key rows ``krows``.  Returns (dQ_rows, dK_rows, dV_rows,
        LSE, Delta), the last two over every query row."""
        return self._bwd_rows(q, k, v, do, scale, qrows, krows, nthreads, causal=causal)

    def attn_bwd_rows_masked(self, q, k, v, do, left: int, right: int, kv_len: int,
                             scale: float, qrows, krows, nthreads: int = 0):
        """attn_bwd_rows under the band and key-padding mask of attn_bwd_head_masked."""
        return self._bwd_rows(q, k, v, do, scale, qrows, krows, nthreads, band=(left, right, kv_len))

    def _bwd_rows(self, q, k, v, do, scale, qrows, krows, nthreads, causal=None, band=None):
        q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
        Lq, D = q.shape
        Lk = k.shape[0]
        if k.shape != (Lk, D) or v.shape != (Lk, D) or do.shape != (Lq, D):
            raise ValueError("k, v must be [Lk, D] and do [Lq, D] with the same D as q")
        qr = np.ascontiguousarray(np.asarray(qrows, dtype=np.int64)).astype(ctypes.c_long)
        kr = np.ascontiguousarray(np.asarray(krows, dtype=np.int64)).astype(ctypes.c_long)
        if (qr.size and (qr.min() < 0 or qr.max() >= Lq)) or (kr.size and (kr.min() < 0 or kr.max() >= Lk)):
            raise ValueError("sampled rows out of range")
        dq, dk, dv = np.empty((qr.size, D)), np.empty((kr.size, D)), np.empty((kr.size, D))
        lse, delta = np.empty(Lq), np.empty(Lq)
        lp = ctypes.POINTER(ctypes.c_long)
        head = (_dptr(q), _dptr(k), _dptr(v), _dptr(do), Lq, Lk, D)
        tail = (qr.ctypes.data_as(lp), qr.size, kr.ctypes.data_as(lp), kr.size, _dptr(dq), _dptr(dk),
                _dptr(dv), _dptr(lse), _dptr(delta), int(nthreads))
        if band is None:
            rc = self.lib.oracle_attn_bwd_rows(*head, int(bool(causal)), float(scale), *tail)
        else:
            left, right, kv_len = (int(x) for x in band)
            rc = self.lib.oracle_attn_bwd_rows_masked(*head, left, right, kv_len, float(scale), *tail)
        if rc != 0:
            raise ValueError(f"oracle_attn_bwd_rows failed with code {rc}")
        return dq, dk, dv, lse, delta

    def attn_bwd_head_masked(self, q, k, v, do, left: int, right: int, kv_len: int,
                             scale: float, nthreads: int = 0):
        """Gradients (dQ, dK, dV) under the band and key-padding mask of attn_head_keypad."""
        q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
        Lq, D = q.shape
        Lk = k.shape[0]
        if k.shape != (Lk, D) or v.shape != (Lk, D) or do.shape != (Lq, D):
            raise ValueError("k, v must be [Lk, D] and do [Lq, D] with the same D as q")
        dq, dk, dv = np.empty((Lq, D)), np.empty((Lk, D)), np.empty((Lk, D))
        rc = self.lib.oracle_attn_bwd_head_masked(_dptr(q), _dptr(k), _dptr(v), _dptr(do), Lq, Lk,
                                                  D, int(left), int(right), int(kv_len),
                                                  float(scale), _dptr(dq), _dptr(dk), _dptr(dv),
                                                  int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_attn_bwd_head_masked failed with code {rc}")
        return dq, dk, dv

    def attn_bwd_full(self, q, k, v, do, causal: bool, scale: float, nthreads: int = 0):
        """Gradients over contiguous [B, H, L, D] tensors: returns (dQ, dK, dV)."""
        q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
        B, H = q.shape[:2]
        dq, dk, dv = np.empty(q.shape), np.empty(k.shape), np.empty(v.shape)
        for b in range(B):
            for h in range(H):
                dq[b, h], dk[b, h], dv[b, h] = self.attn_bwd_head(q[b, h], k[b, h], v[b, h],
                                                                  do[b, h], causal, scale, nthreads)
        return dq, dk, dv

    def attn_full(self, q, k, v, causal: bool, scale: float, want_p: bool = False,
                  nthreads: int = 0):
        """Attention over contiguous [B, H, L, D] tensors: returns (O, LSE[, P])."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, Lq, D = q.shape
        Lk = k.shape[2]
        if k.shape != (B, H, Lk, D) or v.shape != (B, H, Lk, D):
            raise ValueError("k and v must be [B, H, Lk, D] matching q")
        O = np.empty((B, H, Lq, D), dtype=np.float64)
        L = np.empty((B, H, Lq), dtype=np.float64)
        P = np.empty((B, H, Lq, Lk), dtype=np.float64) if want_p else None
        rc = self.lib.oracle_attn_full(_dptr(q), _dptr(k), _dptr(v), B, H, Lq, Lk, D,
                                       int(bool(causal)), float(scale), _dptr(O),
                                       _dptr(L), _dptr(P), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_attn_full failed with code {rc}")
        return (O, L, P) if want_p else (O, L)


_default = None


def _get() -> OracleLib:
    global _default
    if _default is None:
        _default = OracleLib(build())
    return _default


def max_threads() -> int:
    return _get().max_threads()


def attn_head(*args, **kwargs):
    return _get().attn_head(*args, **kwargs)


def attn_full(*args, **kwargs):
    return _get().attn_full(*args, **kwargs)


def attn_head_window(*args, **kwargs):
    return _get().attn_head_window(*args, **kwargs)


def attn_full_window(*args, **kwargs):
    return _get().attn_full_window(*args, **kwargs)


def attn_bwd_head(*args, **kwargs):
    return _get().attn_bwd_head(*args, **kwargs)


def attn_head_keypad(*args, **kwargs):
    return _get().attn_head_keypad(*args, **kwargs)


def attn_full_keypad(*args, **kwargs):
    return _get().attn_full_keypad(*args, **kwargs)


def attn_bwd_full(*args, **kwargs):
    return _get().attn_bwd_full(*args, **kwargs)


def attn_bwd_head_masked(*args, **kwargs):
    return _get().attn_bwd_head_masked(*args, **kwargs)


def attn_bwd_rows(*args, **kwargs):
    return _get().attn_bwd_rows(*args, **kwargs)


def attn_bwd_rows_masked(*args, **kwargs):
    return _get().attn_bwd_rows_masked(*args, **kwargs)
