"""GPU tests of fa_fwd_strided: strided layouts and fp16 I/O.

Strided inputs and outputs change only the addressing, so their results must equal
the contiguous bf16 calls bit for bit.  fp16 changes the arithmetic (P and O rounded
to fp16), so fp16 results are compared with the fp64 oracle on the fp16 input values,
at the forward's tolerances (max-abs 2e-2 on O, 1e-3 on LSE).
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_60_gb300 as fa
from exact_attention_60_gb300.workloads import WORKLOADS, make_qkv, make_workload_inputs, sample_rows

pytestmark = pytest.mark.gpu

TOL_O = 2e-2
TOL_LSE = 1e-3
DEV = torch.device("cuda:0")


def packed_qkv(B, H, Lq, D, seed, dtype=torch.bfloat16):
    """Q, K, V as views of one [B, L, 3, H, D] projection output (Lq == Lk)."""
    q, k, v = make_qkv(B, H, Lq, Lq, D, seed)
    packed = torch.empty((B, Lq, 3, H, D), dtype=dtype, device=DEV)
    for i, t in enumerate((q, k, v)):
        packed[:, :, i] = t.to(dtype).to(DEV).transpose(1, 2)
    views = tuple(packed[:, :, i].transpose(1, 2) for i in range(3))   # [B, H, L, D], strided
    return views, (q, k, v)


@pytest.mark.parametrize("B,H,L,D,causal", [(2, 3, 300, 128, True), (1, 4, 257, 64, False),
                                            (3, 1, 129, 128, False), (1, 1, 1000, 64, True),
                                            (2, 8, 640, 128, True)])
def test_packed_qkv_equals_contiguous(B, H, L, D, causal):
    (qv, kv, vv), (q, k, v) = packed_qkv(B, H, L, D, seed=L + D)
    assert not qv.is_contiguous()
    o_ref, l_ref = fa.attention(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, split=False)
    o, lse = fa.attention(qv, kv, vv, causal=causal, split=False)
    assert fa.fa_last_device_status() == fa.FA_OK
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_strided_output_equals_contiguous():
    q, k, v = (t.to(DEV) for t in make_qkv(2, 4, 500, 700, 128, seed=3))
    o_ref, l_ref = fa.attention(q, k, v, causal=True, split=False)
    buf = torch.full((2, 500, 4, 128), 7.0, dtype=torch.bfloat16, device=DEV)   # [B, L, H, D]
    out = buf.transpose(1, 2)
    o, lse = fa.attention(q, k, v, causal=True, out=out)
    assert o.data_ptr() == buf.data_ptr()
    assert torch.equal(out, o_ref) and torch.equal(lse, l_ref)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("layout", ["offset16", "rowpad8"])
def test_output_aligned_to_16_bytes_only(layout, causal):
    """At D = 128 the epilogue stores O 32 bytes a time when O's base and strides allow it;
    an output that is only 16-byte aligned (its base 16 bytes into a buffer, or rows
    padded by 8 elements) takes the 16-byte stores.  Same bits as the contiguous call, and
    nothing outside the output written."""
    B, H, L, D = 2, 3, 300, 128
    q, k, v = (t.to(DEV) for t in make_qkv(B, H, L, L, D, seed=17))
    o_ref, l_ref = fa.attention(q, k, v, causal=causal, split=False)
    n = B * H * L * D
    if layout == "offset16":
        buf = torch.full((n + 16,), 7.0, dtype=torch.bfloat16, device=DEV)
        out = buf[8:8 + n].view(B, H, L, D)
        assert out.data_ptr() % 32 == 16
    else:
        buf = torch.full((B, H, L, D + 8), 7.0, dtype=torch.bfloat16, device=DEV)
        out = buf[..., :D]
        assert out.stride(2) * 2 % 32 == 16
    o, lse = fa.attention(q, k, v, causal=causal, out=out, split=False)
    assert fa.fa_last_device_status() == fa.FA_OK
    assert torch.equal(out, o_ref) and torch.equal(lse, l_ref)
    if layout == "offset16":
        assert bool((buf[:8] == 7.0).all()) and bool((buf[8 + n:] == 7.0).all())
    else:
        assert bool((buf[..., D:] == 7.0).all())


@pytest.mark.parametrize("window", [(100, 0), (64, 64), (-1, 3)])
def test_strided_band_equals_contiguous(window):
    (qv, kv, vv), (q, k, v) = packed_qkv(2, 2, 700, 128, seed=11)
    o_ref, l_ref = fa.attention(q.to(DEV), k.to(DEV), v.to(DEV), window=window)
    o, lse = fa.attention(qv, kv, vv, window=window)
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_strided_split_schedule_equals_contiguous():
    """Few query tiles, long keys: the split schedule with a workspace, strided inputs."""
    q, k, v = (t.to(DEV) for t in make_qkv(1, 4, 512, 8192, 128, seed=5))
    o_ref, l_ref = fa.attention(q, k, v, causal=False)   # fa_fwd_ws, split
    st, ws_bytes = fa.fa_fwd_workspace_size(1, 4, 512, 8192, 128, 0)
    assert ws_bytes > 0
    kt = k.transpose(1, 2).contiguous().transpose(1, 2)   # [B, L, H, D] memory, [B, H, L, D] view
    vt = v.transpose(1, 2).contiguous().transpose(1, 2)
    o, lse = fa.attention(q, kt, vt, causal=False)
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def fp16_inputs(B, H, Lq, Lk, D, seed, sigma_qk=1.0):
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed, sigma_qk=sigma_qk)   # bf16 draws, exact in fp16 too
    return tuple(t.to(torch.float16) for t in (q, k, v))


@pytest.mark.parametrize("B,H,Lq,Lk,D,causal", [(1, 2, 128, 128, 64, False), (2, 2, 300, 260, 128, True),
                                                (1, 3, 257, 500, 64, True), (2, 1, 700, 129, 128, False)])
def test_fp16_against_oracle(oracle_mod, B, H, Lq, Lk, D, causal):
    q, k, v = fp16_inputs(B, H, Lq, Lk, D, seed=Lq + Lk)
    o, lse = fa.attention(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal)
    assert o.dtype == torch.float16 and fa.fa_last_device_status() == fa.FA_OK
    ref_o, ref_l = oracle_mod.attn_full(q.float(), k.float(), v.float(), causal, 1.0 / math.sqrt(D))
    assert np.abs(o.float().cpu().numpy() - ref_o).max() <= TOL_O
    assert np.abs(lse.cpu().numpy() - ref_l).max() <= TOL_LSE


def test_fp16_is_more_accurate_than_bf16(oracle_mod):
    """fp16 keeps 3 more significand bits for P and O: its error is smaller."""
    q, k, v = fp16_inputs(1, 4, 512, 512, 128, seed=17)
    ref_o, _ = oracle_mod.attn_full(q.float(), k.float(), v.float(), True, 128 ** -0.5)
    o16, _ = fa.attention(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    ob, _ = fa.attention(q.to(DEV).bfloat16(), k.to(DEV).bfloat16(), v.to(DEV).bfloat16(), causal=True)
    e16 = np.abs(o16.float().cpu().numpy() - ref_o).max()
    eb = np.abs(ob.float().cpu().numpy() - ref_o).max()
    assert e16 < eb / 2, (e16, eb)


def test_fp16_band_and_split_against_oracle(oracle_mod):
    q, k, v = fp16_inputs(1, 2, 600, 600, 128, seed=23)
    o, lse = fa.attention(q.to(DEV), k.to(DEV), v.to(DEV), window=(200, 50))
    ref_o, ref_l = oracle_mod.attn_full_window(q.float(), k.float(), v.float(), 200, 50, 128 ** -0.5)
    assert np.abs(o.float().cpu().numpy() - ref_o).max() <= TOL_O
    assert np.abs(lse.cpu().numpy() - ref_l).max() <= TOL_LSE
    q, k, v = fp16_inputs(1, 2, 256, 4000, 64, seed=29, sigma_qk=2.0)
    st, ws_bytes = fa.fa_fwd_workspace_size(1, 2, 256, 4000, 64, 0)
    assert ws_bytes > 0   # the split schedule runs
    o, lse = fa.attention(q.to(DEV), k.to(DEV), v.to(DEV), causal=False)
    ref_o, ref_l = oracle_mod.attn_full(q.float(), k.float(), v.float(), False, 0.125)
    assert np.abs(o.float().cpu().numpy() - ref_o).max() <= TOL_O
    assert np.abs(lse.cpu().numpy() - ref_l).max() <= TOL_LSE


def test_fp16_packed_strided_equals_fp16_contiguous():
    (qv, kv, vv), (q, k, v) = packed_qkv(2, 2, 400, 128, seed=31, dtype=torch.float16)
    o_ref, l_ref = fa.attention(*(t.to(torch.float16).to(DEV) for t in (q, k, v)), causal=True)
    o, lse = fa.attention(qv, kv, vv, causal=True)
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_strided_guard_band_untouched():
    """Strided O inside a larger buffer: nothing outside O's elements is written."""
    q, k, v = (t.to(DEV) for t in make_qkv(1, 2, 300, 300, 64, seed=37))
    buf = torch.full((1, 300, 2, 96), 5.0, dtype=torch.bfloat16, device=DEV)   # 32 spare features per row
    out = buf[..., :64].transpose(1, 2)
    fa.attention(q, k, v, causal=True, out=out)
    torch.cuda.synchronize()
    assert (buf[..., 64:] == 5.0).all()
    o_ref, _ = fa.attention(q, k, v, causal=True, split=False)
    assert torch.equal(out, o_ref)


def bshd(t):
    """The same [B, H, L, D] values stored [B, L, H, D] (a strided view)."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


def test_workload_bshd_equals_contiguous_both_passes():
    """The benchmark's [B, L, H, D] variant of the 16K causal workload: forward and backward
    results identical to the contiguous calls, bit for bit (only addressing changes)."""
    w = WORKLOADS["seq16k_d128_causal"]
    q, k, v = (t.to(DEV) for t in make_workload_inputs(w))
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(w.seed + 99)).to(torch.bfloat16).to(DEV)
    o, lse = fa.attention(q, k, v, causal=True)
    grads = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    qb, kb, vb, dob = (bshd(t) for t in (q, k, v, do))
    assert not qb.is_contiguous()
    o_b, lse_b = fa.attention(qb, kb, vb, causal=True)
    dq_b, dk_b, dv_b = (bshd(torch.empty_like(t)) for t in (q, k, v))
    fa.attention_backward(qb, kb, vb, o_b, lse_b, dob, causal=True, dq=dq_b, dk=dk_b, dv=dv_b)
    assert fa.fa_last_device_status() == fa.FA_OK
    assert torch.equal(o_b, o) and torch.equal(lse_b, lse)
    for a, b in zip(grads, (dq_b, dk_b, dv_b)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("D", [64, 128])
def test_gradients_aligned_to_16_bytes_only(D):
    """The backward's epilogues store dQ, dK and dV 32 bytes a time when their bases and
    strides allow it; gradients whose buffers start 16 bytes in (or whose rows are padded by
    8 elements) take 16-byte stores.  Same bits as the contiguous call; the padding untouched."""
    B, H, Lq, Lk = 2, 3, 300, 260
    q, k, v = (t.to(DEV) for t in make_qkv(B, H, Lq, Lk, D, seed=23))
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16).to(DEV)
    o, lse = fa.attention(q, k, v, causal=True)
    grads = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    n_q, n_k = B * H * Lq * D, B * H * Lk * D
    buf_q = torch.full((n_q + 16,), 7.0, dtype=torch.bfloat16, device=DEV)
    dq = buf_q[8:8 + n_q].view(B, H, Lq, D)                  # base 16 bytes into the buffer
    buf_k = torch.full((B, H, Lk, D + 8), 7.0, dtype=torch.bfloat16, device=DEV)
    dk = buf_k[..., :D]                                      # rows padded by 8 elements
    buf_v = torch.full((n_k + 16,), 7.0, dtype=torch.bfloat16, device=DEV)
    dv = buf_v[8:8 + n_k].view(B, H, Lk, D)
    assert dq.data_ptr() % 32 == 16 and dv.data_ptr() % 32 == 16 and dk.stride(2) * 2 % 32 == 16
    fa.attention_backward(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv)
    assert fa.fa_last_device_status() == fa.FA_OK
    for a, b in zip(grads, (dq, dk, dv)):
        assert torch.equal(a, b)
    assert bool((buf_q[:8] == 7.0).all()) and bool((buf_q[8 + n_q:] == 7.0).all())
    assert bool((buf_v[:8] == 7.0).all()) and bool((buf_v[8 + n_k:] == 7.0).all())
    assert bool((buf_k[..., D:] == 7.0).all())


def test_workload_fp16_sampled(oracle_mod):
    """The benchmark's fp16 variant of the 16K causal workload against the oracle at
    sampled rows (the bf16 draws are exact in fp16)."""
    w = WORKLOADS["seq16k_d128_causal"]
    q, k, v = (t.to(torch.float16) for t in make_workload_inputs(w))
    o, lse = fa.attention(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    assert o.dtype == torch.float16 and fa.fa_last_device_status() == fa.FA_OK
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    pairs = sample_rows(w, 256)
    for bh in np.unique(pairs[:, 0]):
        rows = pairs[pairs[:, 0] == bh, 1]
        b, h = divmod(int(bh), w.H)
        ref_o, ref_l = oracle_mod.attn_head(q[b, h].float(), k[b, h].float(), v[b, h].float(), True,
                                            w.scale, rows=rows)
        assert np.abs(o[b, h][rows] - ref_o).max() <= TOL_O
        assert np.abs(lse[b, h][rows] - ref_l).max() <= TOL_LSE
