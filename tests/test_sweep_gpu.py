"""A seeded sweep of random problems through the public entry points, each compared in
full against the fp64 oracle.

The fixed-shape tests pin each schedule and mask at chosen sizes; this sweep draws
sizes, masks, element types and layouts together, so that combinations nobody wrote
down (a ragged key tail under a band, a causal problem with Lq > Lk split across SMs,
key padding in a strided fp16 call, ...) go through whichever schedule the library
picks.  The cases are drawn once from a fixed seed, so every run checks the same ones.

Forward: O within 2e-2 and LSE within 1e-3 of the oracle (the bar the specification
sets); a row left without keys by key padding must give O = 0 and LSE = -inf.
Backward: the per-element bound of the backward tests (derived there from where the
kernels round).
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_60_gb300 as fa
from exact_attention_60_gb300.workloads import make_qkv

from test_backward_gpu import check as bwd_check, check_masked as bwd_check_masked, make_do

pytestmark = pytest.mark.gpu

TOL_O = 2e-2
TOL_LSE = 1e-3


def _length(rng, hi):
    """A sequence length: tile multiples, one off a tile edge either way, or arbitrary."""
    kind = rng.integers(0, 4)
    if kind == 0:
        return int(128 * rng.integers(1, hi // 128 + 1))
    if kind == 1:
        return int(128 * rng.integers(1, hi // 128 + 1) + 1)
    if kind == 2:
        return max(1, int(128 * rng.integers(1, hi // 128 + 1) - 1))
    return int(rng.integers(1, hi + 1))


def _mask(rng, Lq, Lk, B, allow_pad=True):
    """(left, right, kv_len): the full mask, causal, a band or key padding.  A band never
    leaves a row without keys (the library rejects that as an argument error); key
    padding may (those rows are defined: O = 0, LSE = -inf)."""
    kind = rng.integers(0, 5 if allow_pad else 3)
    kv_len = None
    if kind == 0:
        left, right = -1, -1
    elif kind == 1:
        left, right = -1, 0
    elif kind == 2:
        left = -1 if rng.random() < 0.3 else int(rng.integers(max(0, Lq - Lk), max(Lq - Lk, 0) + 300))
        right = -1 if rng.random() < 0.3 else int(rng.integers(0, 300))
    else:
        left, right = (-1, -1) if kind == 3 else (-1, 0)
        kv_len = [int(rng.integers(0, Lk + 1)) if rng.random() < 0.8 else Lk for _ in range(B)]
    return left, right, kv_len


def _forward_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        B, H = int(rng.integers(1, 4)), int(rng.integers(1, 5))
        D = int(rng.choice([64, 128]))
        Lq, Lk = _length(rng, 2100), _length(rng, 2100)
        left, right, kv_len = _mask(rng, Lq, Lk, B)
        dtype = "fp16" if rng.random() < 0.25 else "bf16"
        layout = "bshd" if rng.random() < 0.25 else "bhld"
        cases.append((i, B, H, Lq, Lk, D, left, right, kv_len, dtype, layout))
    return cases


def _as_layout(t, layout, dtype):
    """t [B, H, L, D] on the device, in the element type and memory layout asked for
    ("bshd": a [B, H, L, D] view of a contiguous [B, L, H, D] tensor)."""
    t = t.to(torch.float16 if dtype == "fp16" else torch.bfloat16)
    if layout == "bshd":
        t = t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    return t


def _call(q, k, v, left, right, kv_len, scale):
    dev = q.device
    kl = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int32, device=dev)
    if kl is None and left == -1 and right in (-1, 0):
        return fa.attention(q, k, v, causal=(right == 0), scale=scale)
    return fa.attention(q, k, v, window=(left, right), kv_len=kl, scale=scale)


@pytest.mark.parametrize("case", _forward_cases(120, 2026), ids=lambda c: f"f{c[0]}")
def test_forward_sweep_against_oracle(oracle_mod, case):
    i, B, H, Lq, Lk, D, left, right, kv_len, dtype, layout = case
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=7000 + i)
    if dtype == "fp16":   # the bf16 draws are exact in fp16: the oracle sees the same values
        q, k, v = (t.to(torch.float16) for t in (q, k, v))
    scale = 1.0 / math.sqrt(D)
    dev = torch.device("cuda:0")
    qd, kd, vd = (_as_layout(t.to(dev), layout, dtype) for t in (q, k, v))
    o, lse = _call(qd, kd, vd, left, right, kv_len, scale)
    st = fa.fa_last_device_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    kvl = [Lk] * B if kv_len is None else kv_len
    ref_o, ref_l = oracle_mod.attn_full_keypad(q, k, v, left, right, kvl, scale)
    empty = np.isneginf(ref_l)   # rows without an allowed key
    assert (np.isneginf(lse) == empty).all(), "rows without keys must be exactly those with LSE = -inf"
    assert (o[empty] == 0).all()
    assert np.isfinite(o).all() and np.isfinite(lse[~empty]).all()
    err_o = np.abs(o - ref_o).max()
    err_l = np.abs(lse[~empty] - ref_l[~empty]).max() if (~empty).any() else 0.0
    assert err_o <= TOL_O, f"max|dO| = {err_o}"
    assert err_l <= TOL_LSE, f"max|dLSE| = {err_l}"


def _backward_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        D = int(rng.choice([64, 128]))
        Lq, Lk = _length(rng, 1100), _length(rng, 1100)
        left, right, kv_len = _mask(rng, Lq, Lk, B)
        cases.append((i, B, H, Lq, Lk, D, left, right, kv_len))
    return cases


@pytest.mark.parametrize("case", _backward_cases(48, 2027), ids=lambda c: f"b{c[0]}")
def test_backward_sweep_against_oracle(oracle_mod, case):
    i, B, H, Lq, Lk, D, left, right, kv_len = case
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=8000 + i)
    do = make_do(B, H, Lq, D, seed=8000 + i)
    scale = 1.0 / math.sqrt(D)
    if kv_len is None and left == -1 and right in (-1, 0):   # fa_bwd itself
        bwd_check(oracle_mod, q, k, v, do, right == 0, scale)
    else:                                                    # fa_bwd_masked
        bwd_check_masked(oracle_mod, q, k, v, do, left, right, kv_len, scale)
