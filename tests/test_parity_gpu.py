"""GPU parity: fa_fwd (through the C ABI) against the fp64 oracle.

Tolerances: max-abs 2e-2 on O (bf16 output) and 1e-3 on LSE (fp32), the bar
the method's specification sets.  Small cases are compared element by element
on every row; the full-size workloads on a seeded sample of rows (plus rows at
tile edges), computed one by one by the oracle.
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


def run_fa(q, k, v, causal, scale=None):
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o, lse = fa.attention(qd, kd, vd, causal=causal, scale=scale)
    st = fa.fa_last_device_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check_full(oracle_mod, q, k, v, causal, scale):
    o, lse = run_fa(q, k, v, causal, scale)
    ref_o, ref_l = oracle_mod.attn_full(q, k, v, causal, scale)
    err_o = np.abs(o - ref_o).max()
    err_l = np.abs(lse - ref_l).max()
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert err_o <= TOL_O, f"max|dO| = {err_o}"
    assert err_l <= TOL_LSE, f"max|dLSE| = {err_l}"
    return err_o, err_l


def check_rows(oracle_mod, q, k, v, causal, scale, pairs, o, lse):
    """Compare sampled (bh, i) rows of a GPU result with the oracle, row by row."""
    B, H = q.shape[0], q.shape[1]
    worst_o = worst_l = 0.0
    for bh in np.unique(pairs[:, 0]):
        rows = pairs[pairs[:, 0] == bh, 1]
        b, h = divmod(int(bh), H)
        ref_o, ref_l = oracle_mod.attn_head(q[b, h], k[b, h], v[b, h], causal, scale, rows=rows)
        got_o = o[b, h][rows].float().numpy()
        got_l = lse[b, h][rows].numpy()
        worst_o = max(worst_o, float(np.abs(got_o - ref_o).max()))
        worst_l = max(worst_l, float(np.abs(got_l - ref_l).max()))
    assert worst_o <= TOL_O, f"max|dO| = {worst_o}"
    assert worst_l <= TOL_LSE, f"max|dLSE| = {worst_l}"
    return worst_o, worst_l


@pytest.mark.parametrize("name", ["tiny_d64", "seq1k_d64", "seq1k_d64_causal"])
def test_workload_full(oracle_mod, name):
    w = WORKLOADS[name]
    q, k, v = make_workload_inputs(w)
    check_full(oracle_mod, q, k, v, w.causal, w.scale)


@pytest.mark.parametrize("name", ["seq4k_d128_causal", "seq16k_d128_causal",
                                  "cross_q500_k8191_d128", "seq16k_d128_causal_h1"])
def test_workload_sampled(oracle_mod, name):
    w = WORKLOADS[name]
    q, k, v = make_workload_inputs(w)
    dev = torch.device("cuda:0")
    o, lse = fa.attention(q.to(dev), k.to(dev), v.to(dev), causal=w.causal, scale=w.scale)
    assert fa.fa_last_device_status() == fa.FA_OK
    o, lse = o.cpu(), lse.cpu()
    extra = (383, 384, 499) if w.Lq == 500 else ()
    pairs = sample_rows(w, 512, extra)
    check_rows(oracle_mod, q, k, v, w.causal, w.scale, pairs, o, lse)
    # properties that hold at any size, on every row: finite outputs, and
    # |O| bounded by the largest |V| entry of the head (a convex combination).
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    vmax = v.float().abs().amax(dim=(2, 3), keepdim=True)
    assert (o.float().abs() <= vmax + 1e-2).all()


EDGE_LQ = [1, 127, 128, 129, 255, 257, 500]
EDGE_LK = [1, 2, 128, 129, 255, 500]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Lk", EDGE_LK)
@pytest.mark.parametrize("Lq", EDGE_LQ)
def test_edge_shapes(oracle_mod, Lq, Lk, causal, D):
    q, k, v = make_qkv(1, 2, Lq, Lk, D, seed=Lq * 1000 + Lk + D)
    check_full(oracle_mod, q, k, v, causal, 1.0 / math.sqrt(D))


@pytest.mark.parametrize("Lq,Lk,causal,D", [(8191, 8191, True, 128), (1000, 3000, True, 64),
                                             (3000, 1000, True, 128), (777, 4099, False, 64)])
def test_larger_ragged(oracle_mod, Lq, Lk, causal, D):
    q, k, v = make_qkv(2, 3, Lq, Lk, D, seed=Lq + 7 * Lk)
    dev = torch.device("cuda:0")
    o, lse = fa.attention(q.to(dev), k.to(dev), v.to(dev), causal=causal)
    assert fa.fa_last_device_status() == fa.FA_OK
    rng = np.random.default_rng(Lq * 31 + Lk)
    pairs = np.stack([rng.integers(0, 6, 96), rng.integers(0, Lq, 96)], axis=1)
    edge = np.array([[0, 0], [5, Lq - 1], [1, min(127, Lq - 1)], [2, min(128, Lq - 1)],
                     [3, min(255, Lq - 1)], [4, min(256, Lq - 1)]])
    check_rows(oracle_mod, q, k, v, causal, 1.0 / math.sqrt(D), np.concatenate([pairs, edge]),
               o.cpu(), lse.cpu())


def test_non_default_scale(oracle_mod):
    q, k, v = make_qkv(2, 2, 300, 260, 128, seed=99, sigma_qk=2.0)
    for scale in (0.02, 0.3):
        check_full(oracle_mod, q, k, v, True, scale)
        check_full(oracle_mod, q, k, v, False, scale)


BF16_U = 2.0 ** -8   # unit roundoff of bf16 (8-bit significand, round to nearest)


def test_large_logits(oracle_mod):
    """Scores spread over hundreds of units: the lazy rescale has to fire often.

    The softmax is then almost one-hot, so |O| approaches max|V| (about 5 here)
    and the bf16 rounding of P and of O dominates the error.  The bound used is
    the one the arithmetic gives per element:
        |dO| <= u * max|V| (P rounded to bf16) + u * |O| (O rounded to bf16) + 1e-3,
    u = 2^-8.  The workloads of the specification keep the flat 2e-2 bound.
    """
    q, k, v = make_qkv(1, 2, 384, 640, 128, seed=5, sigma_qk=6.0)
    scale = 1.0 / math.sqrt(128)
    vmax = v.float().abs().amax(dim=(2, 3)).numpy()[:, :, None, None]
    for causal in (False, True):
        o, lse = run_fa(q, k, v, causal, scale)
        ref_o, ref_l = oracle_mod.attn_full(q, k, v, causal, scale)
        bound = BF16_U * (vmax + np.abs(ref_o)) + 1e-3
        assert (np.abs(o - ref_o) <= bound).all(), float((np.abs(o - ref_o) - bound).max())
        assert np.abs(lse - ref_l).max() <= TOL_LSE


def test_increasing_scores(oracle_mod):
    """Keys whose scores grow along the sequence force a new row max on every tile."""
    Lk, D = 1024, 64
    q = torch.ones(1, 1, 256, D)
    ramp = torch.linspace(0.0, 40.0, Lk)[:, None] / D
    k = (ramp * torch.ones(1, D)).reshape(1, 1, Lk, D)
    v = torch.randn(1, 1, Lk, D, generator=torch.Generator().manual_seed(3))
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    check_full(oracle_mod, q, k, v, False, 1.0)
    check_full(oracle_mod, q, k, v, True, 1.0)


def test_guard_bands_untouched():
    """O and LSE sit inside larger buffers whose margins hold a sentinel; the
    kernel must write exactly [B,H,Lq,D] and [B,H,Lq] (ragged Lq included)."""
    dev = torch.device("cuda:0")
    B, H, Lq, Lk, D = 2, 3, 300, 200, 128
    q, k, v = (t.to(dev) for t in make_qkv(B, H, Lq, Lk, D, seed=11))
    pad = 4096
    n_o, n_l = B * H * Lq * D, B * H * Lq
    o_buf = torch.full((n_o + 2 * pad,), float("nan"), device=dev, dtype=torch.bfloat16)
    l_buf = torch.full((n_l + 2 * pad,), float("nan"), device=dev, dtype=torch.float32)
    o = o_buf[pad:pad + n_o].view(B, H, Lq, D)
    lse = l_buf[pad:pad + n_l].view(B, H, Lq)
    for causal in (False, True):
        fa.attention(q, k, v, causal=causal, out=o, lse=lse)
        assert fa.fa_last_device_status() == fa.FA_OK
        assert torch.isnan(o_buf[:pad].float()).all() and torch.isnan(o_buf[pad + n_o:].float()).all()
        assert torch.isnan(l_buf[:pad]).all() and torch.isnan(l_buf[pad + n_l:]).all()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_deterministic():
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(2, 4, 700, 900, 128, seed=12))
    o1, l1 = fa.attention(q, k, v, causal=True)
    o2, l2 = fa.attention(q, k, v, causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_empty_batch_is_noop():
    dev = torch.device("cuda:0")
    q = torch.empty(0, 2, 16, 64, device=dev, dtype=torch.bfloat16)
    k = torch.empty(0, 2, 16, 64, device=dev, dtype=torch.bfloat16)
    o, lse = fa.attention(q, k, k, causal=False)
    assert o.numel() == 0 and lse.numel() == 0
    assert fa.fa_last_device_status() == fa.FA_OK


def test_stream_argument():
    """fa_fwd runs on the stream it is given."""
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(1, 2, 256, 256, 64, seed=13))
    ref_o, ref_l = fa.attention(q, k, v, split=False)
    s = torch.cuda.Stream()
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 256, device=dev)
    s.wait_stream(torch.cuda.current_stream())
    st = fa.fa_fwd(q, k, v, o, lse, 1, 2, 256, 256, 64, 0, 0.125, s)
    assert st == fa.FA_OK
    assert fa.fa_last_device_status(s) == fa.FA_OK
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)


@pytest.mark.parametrize("B,H,Lq,Lk,D,causal", [
    (8, 64, 384, 384, 128, True),      # 1024 units: several rounds per CTA, absent tile 1 in every second unit
    (1, 2, 32768, 32768, 128, True),   # long sequence: 256 key tiles for the last query tiles
    (1, 4096, 1, 1, 64, False),        # thousands of one-row heads
    (2, 300, 130, 70, 64, True),       # more units than CTAs, ragged query and key tails
])
def test_scheduler_shapes(oracle_mod, B, H, Lq, Lk, causal, D):
    """Shapes that exercise the persistent unit schedule: many rounds per CTA,
    very long rows, and many tiny units."""
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=B * 7 + H + Lq)
    dev = torch.device("cuda:0")
    o, lse = fa.attention(q.to(dev), k.to(dev), v.to(dev), causal=causal)
    assert fa.fa_last_device_status() == fa.FA_OK
    o, lse = o.cpu(), lse.cpu()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    BH = B * H
    rng = np.random.default_rng(B + H + Lq + Lk)
    pairs = np.stack([rng.integers(0, BH, 160), rng.integers(0, Lq, 160)], axis=1)
    edge = np.array([[0, 0], [BH - 1, Lq - 1], [BH // 2, Lq // 2], [BH - 1, 0], [0, Lq - 1]])
    check_rows(oracle_mod, q, k, v, causal, 1.0 / math.sqrt(D), np.concatenate([pairs, edge]),
               o, lse)


@pytest.mark.parametrize("B,H,Lq,Lk,D,causal,sched", [
    (4, 64, 4096, 4096, 64, True, fa.FA_SCHED_TABLE),      # 4096 units: the host table's limit
    (5, 64, 4096, 4096, 64, True, fa.FA_SCHED_WHOLE),      # 5120 units: past it, fixed order
    (1, 1, 131072, 131072, 128, True, fa.FA_SCHED_TABLE),  # one head of 128K tokens (64 MiB of K/V)
    (1, 2, 256, 1 << 20, 64, False, fa.FA_SCHED_SPLIT),    # a million keys per row
    (1, 65536, 64, 64, 64, False, fa.FA_SCHED_WHOLE),      # 65,536 heads of one short tile
])
def test_size_limits(oracle_mod, B, H, Lq, Lk, D, causal, sched):
    """The largest shapes each schedule is built for, and one past the host table's limit:
    the schedule the library reports, then sampled rows (first, last, tile edges) against
    the oracle."""
    assert fa.fa_fwd_schedule(B, H, Lq, Lk, D, causal) == (fa.FA_OK, sched)
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=(B * H + Lq + Lk) % 100003)
    dev = torch.device("cuda:0")
    o, lse = fa.attention(q.to(dev), k.to(dev), v.to(dev), causal=causal)
    assert fa.fa_last_device_status() == fa.FA_OK
    o, lse = o.cpu(), lse.cpu()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    BH = B * H
    rng = np.random.default_rng(BH + Lq)
    n = 24 if Lk >= 1 << 17 else 96
    pairs = np.stack([rng.integers(0, BH, n), rng.integers(0, Lq, n)], axis=1)
    edge = np.array([[0, 0], [BH - 1, Lq - 1], [BH - 1, 0], [0, Lq - 1],
                     [BH // 2, min(Lq - 1, 127)], [BH // 2, min(Lq - 1, 128)]])
    check_rows(oracle_mod, q, k, v, causal, 1.0 / math.sqrt(D), np.concatenate([pairs, edge]),
               o, lse)


@pytest.mark.parametrize("B,H,Lq,Lk,D,causal", [(1, 2, 300, 300, 64, True),
                                                 (2, 1, 129, 1000, 128, False),
                                                 (1, 3, 600, 600, 128, True)])
@pytest.mark.parametrize("level", [0.0, 64.0])
def test_equal_scores_give_the_mean_of_v(B, H, Lq, Lk, D, causal, level):
    """Degenerate softmax: every allowed key of a row has the same score s, so the row's
    weights are uniform.  Closed form (no oracle): O_i = the mean of the allowed V rows,
    LSE_i = s + ln(n_i), n_i = i + 1 (causal) or Lk.  With level 64 the scores are
    64 * 64 / sqrt(D) (362 at D = 128), whose exponentials overflow fp32 unless the row
    maximum is subtracted first."""
    g = torch.Generator().manual_seed(Lq + Lk + D)
    q = torch.zeros(B, H, Lq, D)
    k = torch.zeros(B, H, Lk, D)
    q[..., 0] = level
    k[..., 0] = level
    v = torch.randn(B, H, Lk, D, generator=g).to(torch.bfloat16)
    q, k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    dev = torch.device("cuda:0")
    o, lse = fa.attention(q.to(dev), k.to(dev), v.to(dev), causal=causal)
    assert fa.fa_last_device_status() == fa.FA_OK
    o, lse = o.float().cpu().double(), lse.cpu().double()
    vd = v.double()
    if causal:
        n = torch.arange(1, Lq + 1, dtype=torch.float64)
        ref_o = vd[:, :, :Lq].cumsum(2) / n[:, None]
    else:
        n = torch.full((Lq,), float(Lk), dtype=torch.float64)
        ref_o = vd.mean(2, keepdim=True).expand(B, H, Lq, D)
    s = level * level / math.sqrt(D)
    ref_l = (s + torch.log(n)).expand(B, H, Lq)
    assert float((o - ref_o).abs().max()) <= TOL_O
    assert float((lse - ref_l).abs().max()) <= TOL_LSE


# non-causal shapes with few units (query-tile pairs) per SM: the split-key schedule
SPLIT_SHAPES = [(1, 4, 2048, 32768, 128), (1, 8, 2048, 16384, 128), (1, 4, 2048, 32768, 64),
                (1, 2, 256, 256, 64), (3, 5, 700, 1300, 128), (1, 1, 128, 40000, 128),
                (2, 3, 500, 8191, 64)]


@pytest.mark.parametrize("B,H,Lq,Lk,D", SPLIT_SHAPES)
def test_split_schedule_matches(oracle_mod, B, H, Lq, Lk, D):
    """Non-causal shapes that take the split-key schedule: the merged result agrees
    with the whole-unit schedule (fa_fwd) and with the oracle on sampled rows."""
    st, nbytes = fa.fa_fwd_workspace_size(B, H, Lq, Lk, D, False)
    assert st == fa.FA_OK and nbytes > 0
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=B + H + Lq + Lk, sigma_qk=2.0)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o1, l1 = fa.attention(qd, kd, vd, split=False)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=dev)   # arbitrary contents
    o2 = torch.empty_like(qd)
    l2 = torch.empty(B, H, Lq, device=dev)
    for _ in range(2):   # the workspace is reused as left by the previous call
        st = fa.fa_fwd_ws(qd, kd, vd, o2, l2, B, H, Lq, Lk, D, 0, 1.0 / math.sqrt(D), ws, nbytes)
        assert st == fa.FA_OK
        assert fa.fa_last_device_status() == fa.FA_OK
        assert (o2.float() - o1.float()).abs().max().item() <= TOL_O
        assert (l2 - l1).abs().max().item() <= TOL_LSE
    rng = np.random.default_rng(Lk)
    pairs = np.stack([rng.integers(0, B * H, 64), rng.integers(0, Lq, 64)], axis=1)
    pairs = np.concatenate([pairs, [[0, 0], [B * H - 1, Lq - 1]]])
    check_rows(oracle_mod, q, k, v, False, 1.0 / math.sqrt(D), pairs, o2.cpu(), l2.cpu())


def test_no_split_for_causal_or_full_rounds():
    assert fa.fa_fwd_workspace_size(2, 32, 4096, 4096, 128, True) == (fa.FA_OK, 0)
    assert fa.fa_fwd_workspace_size(1, 16, 16384, 16384, 128, True) == (fa.FA_OK, 0)
    assert fa.fa_fwd_workspace_size(1, 2, 128, 128, 64, False) == (fa.FA_OK, 0)   # one key tile
    assert fa.fa_fwd_workspace_size(8, 16, 500, 8191, 128, False) == (fa.FA_OK, 0)  # 84 % fill
    assert fa.fa_fwd_workspace_size(0, 2, 128, 512, 64, False) == (fa.FA_OK, 0)   # empty


def test_workspace_argument_errors():
    dev = torch.device("cuda:0")
    B, H, Lq, Lk, D = 2, 4, 300, 1000, 128
    q, k, v = (t.to(dev) for t in make_qkv(B, H, Lq, Lk, D, seed=31))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Lq, device=dev)
    st, nbytes = fa.fa_fwd_workspace_size(B, H, Lq, Lk, D, False)
    assert st == fa.FA_OK and nbytes > 0
    ws = torch.empty(nbytes + 512, dtype=torch.uint8, device=dev)
    call = lambda w, n: fa.fa_fwd_ws(q, k, v, o, lse, B, H, Lq, Lk, D, 0, 0.1, w, n)
    assert call(None, 0) == fa.FA_ERR_INVALID_ARG                   # needed but missing
    assert call(ws, nbytes - 1) == fa.FA_ERR_INVALID_ARG            # too small
    assert call(ws.data_ptr() + 16, nbytes) == fa.FA_ERR_INVALID_ARG   # not 256-aligned
    assert call(o.data_ptr(), nbytes) == fa.FA_ERR_INVALID_ARG      # overlaps O
    assert call(ws, nbytes) == fa.FA_OK
    assert fa.fa_last_device_status() == fa.FA_OK


@pytest.mark.parametrize("shape,kw,feed", [((4, 16, 1024, 1024, 64), dict(causal=True), "q"),   # dependent launches
                                           ((1, 4, 512, 8192, 128), dict(causal=False), "q"),   # split + combine
                                           ((2, 8, 700, 700, 128), dict(window=(100, 0)), "q"),  # band
                                           ((4, 16, 1024, 1024, 64), dict(causal=True), "kv"),
                                           ((2, 16, 2048, 2048, 128), dict(causal=False), "kv")])
def test_chained_calls_see_previous_results(shape, kw, feed):
    """Each call's output is the next call's Q (or K and V: read after write, including the
    tiles a kernel prefetches into L2 while the previous one finishes) and the previous
    call's input buffer is the next call's output (write after read): back-to-back launches,
    which may overlap their set-up, must give the same bits as calls separated by a device
    sync."""
    B, H, Lq, Lk, D = shape
    dev = torch.device("cuda:0")
    q0, k, v = (t.to(dev) for t in make_qkv(B, H, Lq, Lk, D, seed=61))
    def chain(sync):
        bufs = [(q0 if feed == "q" else k).clone(), torch.empty_like(q0)]
        lse = torch.empty((B, H, Lq), device=dev, dtype=torch.float32)
        for i in range(6):
            src, dst = bufs[i % 2], bufs[(i + 1) % 2]
            if feed == "q":
                fa.attention(src, k, v, out=dst, lse=lse, **kw)
            else:
                fa.attention(q0, src, src, out=dst, lse=lse, **kw)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return bufs[0].clone(), lse.clone()
    a = chain(sync=True)
    b = chain(sync=False)
    assert fa.fa_last_device_status() == fa.FA_OK
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("name", ["seq16k_d128_causal", "cross_q500_k8191_d128"])
def test_workload_through_host_call(oracle_mod, name):
    """The end-to-end path the benchmark times: pinned host Q, K, V through the C call
    fa_fwd_host (chunks of heads, copies overlapped with the kernels) at full size, on the
    seeded row sample of the workload."""
    w = WORKLOADS[name]
    q, k, v = make_workload_inputs(w)
    dev = torch.device("cuda:0")
    left, right = -1, (0 if w.causal else -1)
    st, nbytes = fa.fa_fwd_host_workspace_size(w.B, w.H, w.Lq, w.Lk, w.D, left, right)
    assert st == fa.FA_OK
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    qp, kp, vp = (t.pin_memory() for t in (q, k, v))
    o = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    lse = torch.empty((w.B, w.H, w.Lq), dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream(dev)
    assert fa.fa_fwd_host(qp, kp, vp, o, lse, w.B, w.H, w.Lq, w.Lk, w.D, left, right, w.scale, ws,
                          nbytes, stream) == fa.FA_OK
    stream.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    extra = (383, 384, 499) if w.Lq == 500 else ()
    check_rows(oracle_mod, q, k, v, w.causal, w.scale, sample_rows(w, 512, extra), o, lse)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    # every row against one launch on device buffers (equal up to the summation order where
    # a chunk takes the split-key schedule)
    od, ld = fa.attention(q.to(dev), k.to(dev), v.to(dev), causal=w.causal, scale=w.scale)
    assert (o.float() - od.float().cpu()).abs().max().item() <= TOL_O
    assert (lse - ld.cpu()).abs().max().item() <= TOL_LSE


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_rows_past_lq_untouched_between_heads(D, causal):
    """O written into a strided view whose heads are separated by sentinel rows: rows at and
    past Lq of every head (the ragged last query tile; at D = 64 the epilogue stores whole
    tiles with TMA, clipped by the tensor's bounds) must stay untouched, and the values must
    equal the contiguous call's bit for bit."""
    dev = torch.device("cuda:0")
    B, H, Lq, Lk, D_ = 2, 3, 300, 520, D
    q, k, v = (t.to(dev) for t in make_qkv(B, H, Lq, Lk, D_, seed=29 + D))
    gap = 77   # sentinel rows after each head's Lq rows
    o_buf = torch.full((B, H, Lq + gap, D_), float("nan"), device=dev, dtype=torch.bfloat16)
    o = o_buf[:, :, :Lq, :]
    o_ref, l_ref = fa.attention(q, k, v, causal=causal)
    _, lse = fa.attention(q, k, v, causal=causal, out=o)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    assert torch.isnan(o_buf[:, :, Lq:, :].float()).all()
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
