"""The split-key schedule for causal problems with few long units.

With the causal mask the units (pairs of query tiles of one head) grow along the sequence,
so whole units finish no sooner than the longest one.  When that unit is far above an
even share of all key-tile steps (at least twice it) -- a few heads of long sequences -- fa_fwd_ws cuts the key
ranges across CTAs: each unit's steps are the key tiles up to the diagonal of its last
tile, parts park their rows' partial state and a second kernel merges them.  A part may
hold no key tile of the pair's first (shorter) tile; it then parks an empty state.
Checked against the oracle on sampled rows (tile and unit edges included) and against the
whole-unit launch of fa_fwd.
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

SHAPES = [(1, 1, 16384, 16384, 128),  # one head of 16K tokens: 64 units for 152 SMs
          (1, 1, 16384, 16384, 64),
          (1, 1, 32768, 32768, 128),  # longest unit 2.4x the even share: split since it is >= 2x
          (1, 2, 16384, 16384, 128),  # 2.3x
          (1, 4, 8192, 8192, 128),    # 2.3x
          (1, 2, 8192, 8192, 64),
          (2, 2, 4096, 4096, 128),
          (1, 3, 3900, 3900, 128),    # last pair without its second tile
          (1, 4, 2500, 5000, 128),    # Lq < Lk (top-left causal: keys j <= i)
          (1, 4, 2400, 5000, 128),    # Lq < Lk, last pair without its second tile: one step fewer
          (1, 2, 5000, 2500, 64)]     # Lq > Lk (rows past Lk see every key)


def sample(Lq, seed):
    rng = np.random.default_rng(seed)
    edges = [0, 1, 127, 128, 129, 255, 256, Lq // 2, Lq - 129, Lq - 128, Lq - 2, Lq - 1]
    return np.unique(np.clip(np.concatenate([rng.integers(0, Lq, 160), edges]), 0, Lq - 1))


@pytest.mark.parametrize("B,H,Lq,Lk,D", SHAPES)
def test_causal_split_matches_oracle_and_whole_units(oracle_mod, B, H, Lq, Lk, D):
    st, nbytes = fa.fa_fwd_workspace_size(B, H, Lq, Lk, D, True)
    assert st == fa.FA_OK and nbytes > 0, "expected the split schedule for this shape"
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=Lq + 3 * Lk + H)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, Lq), float("nan"), device=DEV)
    assert fa.fa_fwd_ws(qd, kd, vd, o, lse, B, H, Lq, Lk, D, 1, scale, ws, nbytes) == fa.FA_OK
    o_w = torch.empty_like(qd)
    l_w = torch.empty((B, H, Lq), device=DEV)
    assert fa.fa_fwd(qd, kd, vd, o_w, l_w, B, H, Lq, Lk, D, 1, scale) == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    # whole-unit launch: the same values up to the merge's summation order
    assert (o.float() - o_w.float()).abs().max().item() <= TOL_O
    assert (lse - l_w).abs().max().item() <= TOL_LSE
    o, lse = o.cpu(), lse.cpu()
    rows = sample(Lq, Lq + Lk)
    for b, h in {(0, 0), (B - 1, H - 1)}:
        ref_o, ref_l = oracle_mod.attn_head(q[b, h], k[b, h], v[b, h], True, scale, rows=rows)
        assert np.abs(o[b, h][rows].float().numpy() - ref_o).max() <= TOL_O
        assert np.abs(lse[b, h][rows].numpy() - ref_l).max() <= TOL_LSE


def test_causal_split_through_strided_fp16(oracle_mod):
    """fa_fwd_strided takes the same schedule given a workspace (fp16, [B, L, H, D])."""
    B, H, L, D = 1, 1, 16384, 128
    assert fa.fa_fwd_workspace_size(B, H, L, L, D, True)[1] > 0
    q, k, v = make_qkv(B, H, L, L, D, seed=17)
    scale = 1.0 / math.sqrt(D)
    qs, ks, vs = (t.to(torch.float16).to(DEV).transpose(1, 2).contiguous().transpose(1, 2)
                  for t in (q, k, v))
    o, lse = fa.attention(qs, ks, vs, causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    rows = sample(L, 5)
    ref_o, ref_l = oracle_mod.attn_head(q[0, 0].half().float(), k[0, 0].half().float(),
                                        v[0, 0].half().float(), True, scale, rows=rows)
    assert np.abs(o[0, 0].cpu()[rows].float().numpy() - ref_o).max() <= TOL_O
    assert np.abs(lse[0, 0].cpu()[rows].numpy() - ref_l).max() <= TOL_LSE
