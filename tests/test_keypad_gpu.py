"""GPU parity of the key-padding mask (fa_fwd_strided with kv_len) against the oracle.

Keys j >= kv_len[b] of batch b are masked for every head and query, on top of the
full, causal or band mask.  Rows left without any allowed key must come back as
O = 0 and LSE = -inf (the oracle's reading); every other row within the forward's
tolerances (max-abs 2e-2 on O, 1e-3 on LSE).
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_60_gb300 as fa
from exact_attention_60_gb300.workloads import WORKLOADS, make_qkv, make_workload_inputs

pytestmark = pytest.mark.gpu

TOL_O = 2e-2
TOL_LSE = 1e-3
DEV = torch.device("cuda:0")


def run_keypad(q, k, v, kv_len, window, dtype=torch.bfloat16):
    qd, kd, vd = (t.to(dtype).to(DEV) for t in (q, k, v))
    kl = torch.tensor(kv_len, dtype=torch.int32, device=DEV)
    o, lse = fa.attention(qd, kd, vd, window=window, kv_len=kl)
    st = fa.fa_last_device_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return o.float().cpu().numpy(), lse.cpu().numpy()


def compare(oracle_mod, q, k, v, kv_len, window, scale, dtype=torch.bfloat16):
    o, lse = run_keypad(q, k, v, kv_len, window, dtype)
    qq, kk, vv = (t.to(dtype).float() for t in (q, k, v))
    ref_o, ref_l = oracle_mod.attn_full_keypad(qq, kk, vv, window[0], window[1], kv_len, scale)
    empty = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(lse), empty), "rows without keys must have LSE = -inf"
    assert np.all(o[empty] == 0.0), "rows without keys must have O = 0"
    assert np.isfinite(o).all()
    assert np.abs(o - ref_o).max() <= TOL_O
    if (~empty).any():
        assert np.abs(lse[~empty] - ref_l[~empty]).max() <= TOL_LSE
    return int(empty.sum())


WINDOWS = [(-1, -1), (-1, 0), (200, 0), (50, 50)]


@pytest.mark.parametrize("window", WINDOWS)
@pytest.mark.parametrize("D", [64, 128])
def test_keypad_against_oracle(oracle_mod, window, D):
    B, H, Lq, Lk = 5, 2, 600, 700
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=D + window[0] * 3 + window[1])
    kv_len = [700, 0, 1, 333, 129]
    compare(oracle_mod, q, k, v, kv_len, window, 1.0 / math.sqrt(D))


def test_keypad_ragged_and_lq_beyond_lk(oracle_mod):
    q, k, v = make_qkv(3, 3, 1000, 300, 128, seed=41)
    n_empty = compare(oracle_mod, q, k, v, [300, 128, 257], (-1, 0), 128 ** -0.5)
    assert n_empty == 0   # causal rows always keep key 0
    n_empty = compare(oracle_mod, q, k, v, [300, 128, 257], (10, 10), 128 ** -0.5)
    assert n_empty > 0    # bands past the padding


def test_keypad_fp16(oracle_mod):
    q, k, v = make_qkv(2, 2, 400, 500, 64, seed=43)
    compare(oracle_mod, q, k, v, [450, 77], (-1, 0), 0.125, dtype=torch.float16)


def test_keypad_without_padding_equals_unpadded():
    """kv_len = Lk everywhere: the band kernel gives the whole-unit kernels' bits."""
    q, k, v = (t.to(DEV) for t in make_qkv(2, 3, 700, 900, 128, seed=47))
    kl = torch.full((2,), 900, dtype=torch.int32, device=DEV)
    for causal in (False, True):
        o_ref, l_ref = fa.attention(q, k, v, causal=causal, split=False)
        o, lse = fa.attention(q, k, v, causal=causal, kv_len=kl)
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_keypad_out_of_range_lengths_are_clamped(oracle_mod):
    q, k, v = make_qkv(3, 1, 300, 256, 64, seed=53)
    a = run_keypad(q, k, v, [-5, 10_000, 256], (-1, -1))
    b = run_keypad(q, k, v, [0, 256, 256], (-1, -1))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def bench_kv_len(w, pad):
    """The per-batch key counts ``bench.py --kv-pad pad`` draws for workload w."""
    g = np.random.default_rng(0xCAFE + w.index)
    lo = max(1, int(round(w.Lk * (1.0 - 2.0 * pad))))
    return g.integers(lo, w.Lk + 1, size=w.B).astype(np.int32)


def test_keypad_workload_sampled(oracle_mod):
    """The key-padding benchmark variant (16K causal, a quarter of the keys padded on
    average) at sampled rows of every head, rows at the padding edge included."""
    w = WORKLOADS["seq16k_d128_causal"]
    kv_len = bench_kv_len(w, 0.25)
    q, k, v = make_workload_inputs(w)
    o, lse = run_keypad(q, k, v, kv_len.tolist(), (-1, 0))
    rng = np.random.default_rng(0x5EED + 99)
    for b in range(w.B):
        kv = int(kv_len[b])
        rows = sorted({0, 1, 127, 128, kv - 2, kv - 1, kv, kv + 1, w.Lq - 1} & set(range(w.Lq))
                      | set(rng.integers(0, w.Lq, 24).tolist()))
        for h in (0, w.H // 2, w.H - 1):
            ref_o, ref_l = oracle_mod.attn_head_keypad(q[b, h], k[b, h], v[b, h], -1, 0, kv, w.scale,
                                                       rows=rows)
            assert np.abs(o[b, h][rows] - ref_o).max() <= TOL_O
            assert np.abs(lse[b, h][rows] - ref_l).max() <= TOL_LSE
