"""The host-computed unit order for large causal problems (kSchedTable).

When the heads' K/V outgrow the L2 cache, causal units run in an order computed on the
host: heads in groups whose K/V fit in L2, each group's units heaviest first, each unit
to the CTA with the least work so far.  Every unit still computes its two query tiles
exactly as before, so the results must be bit-identical to the formula order
(fa_debug_set bit 4 turns the table off) -- and both must match the oracle, which the
full-size parity tests of the 4K and 16K causal workloads check on the table path.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_60_gb300 as fa
from exact_attention_60_gb300.workloads import make_qkv

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def run(q, k, v, fn, flags):
    fa.fa_debug_set(flags, 0)
    try:
        out = fn(q, k, v)
        torch.cuda.synchronize()
        assert fa.fa_last_device_status() == fa.FA_OK
    finally:
        fa.fa_debug_set(0, 0)
    return out


@pytest.mark.parametrize("B,H,L,D", [(1, 32, 4096, 128),    # 64 MiB of K/V: table order
                                     (1, 48, 3000, 128),    # ragged last query tile
                                     (2, 32, 4096, 64),     # D = 64, 64 MiB
                                     (3, 12, 2900, 128)])   # head groups of 22 and 14 heads
def test_table_order_is_bit_identical_to_formula_order(B, H, L, D):
    assert B * H * 4 * L * D > 48 << 20
    q, k, v = (t.to(DEV) for t in make_qkv(B, H, L, L, D, seed=L + H))
    scale = 1.0 / math.sqrt(D)

    def call(q, k, v):
        o = torch.empty_like(q)
        lse = torch.empty((B, H, L), device=DEV)
        assert fa.fa_fwd(q, k, v, o, lse, B, H, L, L, D, 1, scale) == fa.FA_OK
        return o, lse

    o_tab, l_tab = run(q, k, v, call, 0)
    o_ref, l_ref = run(q, k, v, call, 16)
    assert torch.equal(o_tab, o_ref) and torch.equal(l_tab, l_ref)


def test_table_order_on_strided_fp16_and_window_entry_points():
    """The same order behind fa_fwd_strided (fp16, [B, L, H, D]) and fa_fwd_window's
    causal band."""
    B, H, L, D = 1, 32, 4096, 128
    q, k, v = (t.to(DEV) for t in make_qkv(B, H, L, L, D, seed=3))
    scale = 1.0 / math.sqrt(D)

    def strided(q, k, v):
        qs, ks, vs = (t.to(torch.float16).transpose(1, 2).contiguous().transpose(1, 2) for t in (q, k, v))
        o, lse = fa.attention(qs, ks, vs, causal=True, scale=scale)
        return o, lse

    def window(q, k, v):
        o = torch.empty_like(q)
        lse = torch.empty((B, H, L), device=DEV)
        assert fa.fa_fwd_window(q, k, v, o, lse, B, H, L, L, D, -1, 0, scale) == fa.FA_OK
        return o, lse

    for fn in (strided, window):
        a = run(q, k, v, fn, 0)
        b = run(q, k, v, fn, 16)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("B,H,L,D,causal,expect", [
    (1, 16, 16384, 128, 1, fa.FA_SCHED_TABLE),   # 128 MiB of K/V
    (2, 32, 4096, 128, 1, fa.FA_SCHED_TABLE),
    (1, 1, 16384, 128, 1, fa.FA_SCHED_SPLIT),    # one long head: key ranges split
    (4, 16, 1024, 64, 1, fa.FA_SCHED_WHOLE),     # 16 MiB of K/V stay in L2
    (4, 16, 1024, 64, 0, fa.FA_SCHED_WHOLE),
    (1, 4, 2048, 128, 0, fa.FA_SCHED_SPLIT)])    # 16 units on 152 SMs
def test_schedule_query_names_the_schedule_taken(B, H, L, D, causal, expect):
    """fa_fwd_schedule agrees with the workspace query (split iff a workspace is needed)
    and reports the table order exactly when it is on (debug bit 4 turns it off)."""
    st, sc = fa.fa_fwd_schedule(B, H, L, L, D, causal)
    assert st == fa.FA_OK and sc == expect
    st, ws = fa.fa_fwd_workspace_size(B, H, L, L, D, causal)
    assert st == fa.FA_OK and (ws > 0) == (sc == fa.FA_SCHED_SPLIT)
    fa.fa_debug_set(16, 0)
    try:
        st, sc_off = fa.fa_fwd_schedule(B, H, L, L, D, causal)
    finally:
        fa.fa_debug_set(0, 0)
    assert st == fa.FA_OK
    assert sc_off == (fa.FA_SCHED_WHOLE if expect == fa.FA_SCHED_TABLE else expect)
