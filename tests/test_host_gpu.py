"""fa_fwd_host: the forward pass on host buffers, called through the C ABI.

Q, K, V go in from host memory and O, LSE come back to host memory, with the copies and
the kernels overlapped by chunks of heads inside the library.  Results are compared
with the fp64 oracle (every row, the specification's tolerances) and, where the chunks
run on whole units, bit for bit with fa_fwd on device buffers: each query tile's
arithmetic does not depend on which other heads share its launch.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_60_gb300 as fa
from exact_attention_60_gb300.workloads import make_qkv

pytestmark = pytest.mark.gpu

TOL_O = 2e-2
TOL_LSE = 1e-3
DEV = torch.device("cuda:0")


class many_chunks:
    """fa_debug_set bit 3: cut the heads into as many chunks as possible."""

    def __init__(self, on):
        self.on = on

    def __enter__(self):
        if self.on:
            fa.fa_debug_set(8, 0)

    def __exit__(self, *exc):
        fa.fa_debug_set(0, 0)


def run_host(q, k, v, left, right, scale, pinned=True, stream=None):
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    st, nbytes = fa.fa_fwd_host_workspace_size(B, H, Lq, Lk, D, left, right)
    assert st == fa.FA_OK
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=DEV)
    if pinned:
        q, k, v = (t.pin_memory() for t in (q, k, v))
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16)
    lse = torch.full((B, H, Lq), float("nan"), dtype=torch.float32)
    if pinned:
        o, lse = o.pin_memory(), lse.pin_memory()
    s = stream or torch.cuda.current_stream(DEV)
    st = fa.fa_fwd_host(q, k, v, o, lse, B, H, Lq, Lk, D, left, right, scale, ws, ws.numel(), s)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    s.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    return o, lse, nbytes


def oracle_full(oracle_mod, q, k, v, left, right, scale):
    if (left, right) == (-1, -1):
        return oracle_mod.attn_full(q, k, v, False, scale)
    if (left, right) == (-1, 0):
        return oracle_mod.attn_full(q, k, v, True, scale)
    return oracle_mod.attn_full_window(q, k, v, left, right, scale)


@pytest.mark.parametrize("chunked", [False, True])
@pytest.mark.parametrize("B,H,Lq,Lk,D,left,right", [
    (2, 5, 300, 520, 128, -1, -1),     # ragged, full mask
    (2, 5, 300, 520, 128, -1, 0),      # ragged, causal
    (1, 7, 257, 129, 64, -1, 0),       # causal with Lq > Lk, D = 64
    (2, 3, 700, 650, 128, 100, 20),    # band
])
def test_host_matches_oracle(oracle_mod, chunked, B, H, Lq, Lk, D, left, right):
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=B * 1000 + Lq + Lk + D)
    scale = 1.0 / math.sqrt(D)
    with many_chunks(chunked):
        o, lse, _ = run_host(q, k, v, left, right, scale)
    ref_o, ref_l = oracle_full(oracle_mod, q, k, v, left, right, scale)
    assert np.abs(o.float().numpy() - ref_o).max() <= TOL_O
    assert np.abs(lse.numpy() - ref_l).max() <= TOL_LSE


@pytest.mark.parametrize("left,right", [(-1, 0), (100, 20)])
def test_host_bit_identical_to_device_call(left, right):
    """Causal and band masks always run whole units, in the chunks as in one launch, so the
    chunked host call gives the bits of fa_fwd_window on device buffers.  (With the full
    mask a small chunk may take the split-key schedule, whose merge sums in another order;
    that case is checked against the oracle above.)"""
    B, H, Lq, Lk, D = 3, 4, 1000, 1000, 128
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=77)
    scale = 1.0 / math.sqrt(D)
    with many_chunks(True):
        o, lse, _ = run_host(q, k, v, left, right, scale)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    od = torch.empty_like(qd)
    ld = torch.empty((B, H, Lq), device=DEV)
    assert fa.fa_fwd_window(qd, kd, vd, od, ld, B, H, Lq, Lk, D, left, right, scale) == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())


def test_host_split_schedule_inside_chunks(oracle_mod):
    """Few query tiles over long key ranges: each chunk runs the split-key schedule with
    its part of the workspace, chunk after chunk."""
    B, H, Lq, Lk, D = 1, 6, 256, 8191, 128
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=5)
    scale = 1.0 / math.sqrt(D)
    with many_chunks(True):
        o, lse, nbytes = run_host(q, k, v, -1, -1, scale)
    inputs = 2 * B * H * (2 * Lq + 2 * Lk) * D + 4 * B * H * Lq
    assert nbytes > inputs   # the split workspace is part of it
    ref_o, ref_l = oracle_mod.attn_full(q, k, v, False, scale)
    assert np.abs(o.float().numpy() - ref_o).max() <= TOL_O
    assert np.abs(lse.numpy() - ref_l).max() <= TOL_LSE


def test_host_pageable_memory(oracle_mod):
    """Plain (pageable) host memory works too; the copies are then serialised."""
    B, H, Lq, Lk, D = 1, 3, 200, 300, 64
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=9)
    with many_chunks(True):
        o, lse, _ = run_host(q, k, v, -1, 0, 0.125, pinned=False)
    ref_o, ref_l = oracle_mod.attn_full(q, k, v, True, 0.125)
    assert np.abs(o.float().numpy() - ref_o).max() <= TOL_O
    assert np.abs(lse.numpy() - ref_l).max() <= TOL_LSE


def test_host_call_is_ordered_on_the_stream():
    """The call starts after the work already queued on its stream (here a delay and then
    the device-to-host copy that fills the pinned Q), and the stream completes only once
    O and LSE are back in host memory."""
    B, H, Lq, Lk, D = 2, 4, 512, 512, 128
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=13)
    scale = 1.0 / math.sqrt(D)
    s = torch.cuda.Stream(DEV)
    qp = torch.zeros(q.shape, dtype=torch.bfloat16).pin_memory()
    kp, vp = k.pin_memory(), v.pin_memory()
    qd = q.to(DEV)
    st, nbytes = fa.fa_fwd_host_workspace_size(B, H, Lq, Lk, D, -1, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    o = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    lse = torch.empty((B, H, Lq), dtype=torch.float32).pin_memory()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        torch.cuda._sleep(20_000_000)           # keeps the stream busy for a while
        qp.copy_(qd, non_blocking=True)         # Q reaches the host buffer only then
    with many_chunks(True):
        assert fa.fa_fwd_host(qp, kp, vp, o, lse, B, H, Lq, Lk, D, -1, 0, scale, ws, nbytes, s) == fa.FA_OK
    s.synchronize()
    od = torch.empty_like(qd)
    ld = torch.empty((B, H, Lq), device=DEV)
    assert fa.fa_fwd(qd, k.to(DEV), v.to(DEV), od, ld, B, H, Lq, Lk, D, 1, scale) == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())


def test_host_argument_errors():
    B, H, Lq, Lk, D = 1, 2, 64, 64, 64
    q, k, v = (t.pin_memory() for t in make_qkv(B, H, Lq, Lk, D, seed=1))
    o = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    lse = torch.empty((B, H, Lq), dtype=torch.float32).pin_memory()
    st, nbytes = fa.fa_fwd_host_workspace_size(B, H, Lq, Lk, D, -1, -1)
    assert st == fa.FA_OK and nbytes >= 2 * (2 * q.numel() + 2 * k.numel()) + 4 * lse.numel()
    ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=DEV)

    def call(Q=q, K=k, V=v, O=o, L=lse, D=D, left=-1, right=-1, scale=0.125, W=ws, n=nbytes):
        return fa.fa_fwd_host(Q, K, V, O, L, B, H, Lq, Lk, D, left, right, scale, W, n)

    assert call(D=96) == fa.FA_ERR_UNSUPPORTED
    assert call(left=-2) == fa.FA_ERR_INVALID_ARG
    assert call(scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert call(Q=None) == fa.FA_ERR_INVALID_ARG
    assert call(O=q) == fa.FA_ERR_INVALID_ARG                    # O overlaps Q
    assert call(L=o) == fa.FA_ERR_INVALID_ARG                    # LSE inside O
    assert call(W=None) == fa.FA_ERR_INVALID_ARG
    assert call(n=nbytes - 1) == fa.FA_ERR_INVALID_ARG           # too small
    assert call(W=ws.data_ptr() + 16) == fa.FA_ERR_INVALID_ARG   # not 256-byte aligned
    assert fa.fa_fwd_host_workspace_size(B, H, Lq, 0, D, -1, -1)[0] == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_host_workspace_size(0, H, Lq, Lk, D, -1, -1) == (fa.FA_OK, 0)
    lib = fa._native.load()
    assert lib.fa_fwd_host_workspace_size(B, H, Lq, Lk, D, -1, -1, None) == fa.FA_ERR_INVALID_ARG
    assert call() == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK


def test_attention_from_host_wrapper(oracle_mod):
    """The Python helper is a thin call of fa_fwd_host."""
    B, H, Lq, Lk, D = 2, 5, 300, 520, 128
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=41)
    o, lse = fa.attention_from_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), causal=True)
    torch.cuda.synchronize()
    assert o.device.type == "cpu" and lse.device.type == "cpu"
    ref_o, ref_l = oracle_mod.attn_full(q, k, v, True, 1.0 / math.sqrt(D))
    assert np.abs(o.float().numpy() - ref_o).max() <= TOL_O
    assert np.abs(lse.numpy() - ref_l).max() <= TOL_LSE


@pytest.mark.parametrize("D", [128, 64])
def test_host_long_causal_in_chunks(oracle_mod, D):
    """A causal problem large enough for the library to cut into chunks of heads on its own
    (no test hook): the chunks' kernels compute each row exactly as one launch does, so the
    bits match fa_fwd on device buffers; sampled rows are checked against the oracle."""
    B, H, L = 2, 32, 2048
    q, k, v = make_qkv(B, H, L, L, D, seed=D + 7)
    scale = 1.0 / math.sqrt(D)
    o, lse, _ = run_host(q, k, v, -1, 0, scale)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    od = torch.empty_like(qd)
    ld = torch.empty((B, H, L), device=DEV)
    assert fa.fa_fwd(qd, kd, vd, od, ld, B, H, L, L, D, 1, scale) == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())
    rows = np.unique(np.concatenate([np.arange(0, 4), np.arange(250, 262), [L // 8 - 1, L // 8],
                                     np.random.default_rng(1).integers(0, L, 40), [L - 1]]))
    for b, h in ((0, 0), (1, H - 1), (0, 17)):
        ref_o, ref_l = oracle_mod.attn_head(q[b, h], k[b, h], v[b, h], True, scale, rows=rows)
        assert np.abs(o[b, h][rows].float().numpy() - ref_o).max() <= TOL_O
        assert np.abs(lse[b, h][rows].numpy() - ref_l).max() <= TOL_LSE
