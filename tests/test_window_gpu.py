"""GPU parity of local (sliding-window) attention, fa_fwd_window, against the oracle.

Row i keeps keys i - left <= j <= i + right (-1: unbounded side).  The oracle is
oracle_attn_head_window (fp64, the definition applied to each row's band).
Tolerances as for fa_fwd: max-abs 2e-2 on O, 1e-3 on LSE.  The band kernel is
also compared bit for bit with fa_fwd's kernels on the two bands they compute
((-1, 0) causal, (-1, -1) full), with the debug flag that routes those bands to it.
"""
import numpy as np
import pytest
import torch

import exact_attention_60_gb300 as fa
from exact_attention_60_gb300.workloads import WORKLOADS, make_qkv, make_workload_inputs, sample_rows

pytestmark = pytest.mark.gpu

TOL_O = 2e-2
TOL_LSE = 1e-3
FORCE_BAND = 4   # fa_debug_set flag: bands (-1, 0) and (-1, -1) also run the band kernel


def run_window(q, k, v, window, causal=False, scale=None):
    dev = torch.device("cuda:0")
    o, lse = fa.attention(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale,
                          window=window)
    st = fa.fa_last_device_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return o.cpu(), lse.cpu()


def check_window_full(oracle_mod, q, k, v, window, scale):
    o, lse = run_window(q, k, v, window, scale=scale)
    ref_o, ref_l = oracle_mod.attn_full_window(q, k, v, window[0], window[1], scale)
    o, lse = o.float().numpy(), lse.numpy()
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    err_o, err_l = np.abs(o - ref_o).max(), np.abs(lse - ref_l).max()
    assert err_o <= TOL_O, f"max|dO| = {err_o}"
    assert err_l <= TOL_LSE, f"max|dLSE| = {err_l}"


# (B, H, Lq, Lk, D, left, right): bands at and off tile edges, one-sided, ragged,
# a band of one key, Lq > Lk and Lq < Lk.
WINDOW_SHAPES = [
    (1, 2, 1000, 1000, 128, 300, 0),
    (1, 2, 777, 900, 64, 129, 200),
    (2, 3, 513, 513, 128, 0, 0),
    (1, 2, 640, 384, 64, -1, 130),
    (1, 2, 300, 1000, 128, 127, -1),
    (1, 1, 257, 257, 64, 128, 127),
    (1, 2, 700, 700, 128, 255, 0),
    (1, 2, 129, 4000, 64, 5, 3000),
    (1, 3, 1100, 640, 128, 600, 1),
    (2, 2, 384, 384, 64, 1, 1),
]


@pytest.mark.parametrize("shape", WINDOW_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_window_against_oracle(oracle_mod, shape):
    B, H, Lq, Lk, D, left, right = shape
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=Lq * 13 + Lk + left * 7 + right)
    check_window_full(oracle_mod, q, k, v, (left, right), 1.0 / D ** 0.5)


@pytest.mark.parametrize("Lq,Lk", [(1, 1), (1, 300), (127, 127), (129, 200), (255, 129), (256, 256)])
@pytest.mark.parametrize("window", [(0, 0), (1, 0), (0, 1), (128, 128), (60, -1), (-1, 60)])
def test_window_edge_shapes(oracle_mod, Lq, Lk, window):
    left, right = window
    if left >= 0 and Lq - 1 - left > Lk - 1:
        pytest.skip("some row has no key in its band (rejected, tested separately)")
    q, k, v = make_qkv(1, 2, Lq, Lk, 64, seed=Lq * 7 + Lk + 3 * left + right)
    check_window_full(oracle_mod, q, k, v, window, 0.125)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Lq,Lk", [(1000, 1000), (700, 300), (300, 900), (129, 129)])
def test_band_kernel_equals_causal_and_full_kernels(D, Lq, Lk):
    """Bands (-1, 0) and (-1, -1) through the band kernel give fa_fwd's bits."""
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(2, 3, Lq, Lk, D, seed=Lq + Lk + D))
    for causal, window in ((True, (-1, 0)), (False, (-1, -1))):
        o_ref, l_ref = fa.attention(q, k, v, causal=causal, split=False)
        fa.fa_debug_set(FORCE_BAND, 0)
        try:
            o_band, l_band = fa.attention(q, k, v, window=window)
        finally:
            fa.fa_debug_set(0, 0)
        assert fa.fa_last_device_status() == fa.FA_OK
        assert torch.equal(o_band, o_ref) and torch.equal(l_band, l_ref)


def test_normalised_bands_route_to_the_same_result():
    """A side as wide as every key is unbounded: (Lq-1+x, Lk-1+y) == (-1, -1), and
    causal=True with a window cuts the band at the diagonal."""
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(1, 2, 600, 500, 128, seed=5))
    o_full, l_full = fa.attention(q, k, v, causal=False, split=False)
    o_w, l_w = fa.attention(q, k, v, window=(599, 499))
    assert torch.equal(o_w, o_full) and torch.equal(l_w, l_full)
    o_w, l_w = fa.attention(q, k, v, window=(10_000, 10_000))
    assert torch.equal(o_w, o_full) and torch.equal(l_w, l_full)
    o_c, l_c = fa.attention(q, k, v, causal=True, split=False)
    o_w, l_w = fa.attention(q, k, v, causal=True, window=(-1, 77))
    assert torch.equal(o_w, o_c) and torch.equal(l_w, l_c)
    o_a, l_a = fa.attention(q, k, v, window=(100, 0))
    o_b, l_b = fa.attention(q, k, v, causal=True, window=(100, 33))
    assert torch.equal(o_a, o_b) and torch.equal(l_a, l_b)


def test_window_rows_without_keys_are_rejected():
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(1, 1, 300, 200, 64, seed=1))
    with pytest.raises(fa.FaError) as e:
        fa.attention(q, k, v, window=(50, 0))
    assert e.value.status == fa.FA_ERR_INVALID_ARG


def test_window_deterministic():
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(2, 4, 2000, 2000, 128, seed=11))
    o1, l1 = fa.attention(q, k, v, window=(700, 50))
    o2, l2 = fa.attention(q, k, v, window=(700, 50))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("name", ["seq16k_d128_window4k", "seq4k_d64_local256"])
def test_window_workload_sampled(oracle_mod, name):
    w = WORKLOADS[name]
    left, right = w.window
    q, k, v = make_workload_inputs(w)
    o, lse = run_window(q, k, v, w.window, scale=w.scale)
    # rows where the band's edges cross tile boundaries, plus a seeded sample
    extra = (left - 1, left, left + 1, left + 127, left + 128, w.Lq - 129)
    pairs = sample_rows(w, 384, extra)
    worst_o = worst_l = 0.0
    H = w.H
    for bh in np.unique(pairs[:, 0]):
        rows = pairs[pairs[:, 0] == bh, 1]
        b, h = divmod(int(bh), H)
        ref_o, ref_l = oracle_mod.attn_head_window(q[b, h], k[b, h], v[b, h], left, right,
                                                   w.scale, rows=rows)
        worst_o = max(worst_o, float(np.abs(o[b, h][rows].float().numpy() - ref_o).max()))
        worst_l = max(worst_l, float(np.abs(lse[b, h][rows].numpy() - ref_l).max()))
    assert worst_o <= TOL_O, f"max|dO| = {worst_o}"
    assert worst_l <= TOL_LSE, f"max|dLSE| = {worst_l}"
    # any size: finite, and |O| within the head's largest |V| (a convex combination)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    vmax = v.float().abs().amax(dim=(2, 3), keepdim=True)
    assert (o.float().abs() <= vmax + 1e-2).all()


def test_window_from_host(oracle_mod):
    q, k, v = make_qkv(2, 4, 900, 900, 128, seed=21)
    fa.fa_debug_set(8, 0)   # as many chunks as there are heads (overlapped pipeline)
    try:
        o, lse = fa.attention_from_host(q.pin_memory(), k.pin_memory(), v.pin_memory(),
                                        window=(200, 10))
        torch.cuda.synchronize()
    finally:
        fa.fa_debug_set(0, 0)
    ref_o, ref_l = oracle_mod.attn_full_window(q, k, v, 200, 10, 128 ** -0.5)
    assert np.abs(o.float().numpy() - ref_o).max() <= TOL_O
    assert np.abs(lse.numpy() - ref_l).max() <= TOL_LSE
