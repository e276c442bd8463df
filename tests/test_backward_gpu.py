"""GPU parity of the backward pass (fa_bwd through the C ABI) against the fp64 oracle.

The method states no tolerance for gradients, so the bound used is derived from
where the kernels round, per element, with u = 2^-8 (bf16 unit roundoff):
  * P is rounded to bf16 before dV = P^T dO:        u * sum_i P_ij |dO_i|
  * Delta = rowsum(dO * O) uses the bf16 output O:   e_i = 2u * sum_d |dO_id O_id|
    (the forward's own rounding of O plus the kernel's deviation from exact O)
  * dS is rounded to bf16 before dK = dS^T Q and dQ = dS K:
        scale * sum (P_ij e_i + u |dS_ij|) |Q_i|   (dK),   ... |K_j| (dQ)
  * every output is rounded to bf16:                  u * |result|
plus 1e-3 for fp32 accumulation and the approximate exp2.  The test asserts
|GPU - oracle| <= 2 x that bound element by element (the factor covers the
fp32 P, LSE and the bound's first-order nature), and also reports the error
relative to the largest gradient entry.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_60_gb300 as fa
from exact_attention_60_gb300.workloads import WORKLOADS, make_qkv, make_workload_inputs

pytestmark = pytest.mark.gpu

U = 2.0 ** -8


def make_do(B, H, Lq, D, seed):
    g = torch.Generator().manual_seed(int(seed) + 99)
    return torch.randn((B, H, Lq, D), generator=g).to(torch.bfloat16)


def gpu_grads(q, k, v, do, causal, scale):
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.attention(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    st = fa.fa_last_device_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return o.float().cpu().numpy(), dq.float().cpu().numpy(), dk.float().cpu().numpy(), dv.float().cpu().numpy()


def bounds_head(q, k, v, do, o, causal, scale, oracle_mod):
    """Per-element error bounds (dQ, dK, dV) for one head, from the rounding points."""
    P = oracle_mod.attn_head(q, k, v, causal, scale, want_p=True)[2]
    dP = do @ v.T
    delta = (P * dP).sum(axis=1)
    dS = P * (dP - delta[:, None])
    e = 2 * U * np.abs(do * o).sum(axis=1)                # Delta from the bf16 O
    w = P * e[:, None] + U * np.abs(dS)                    # dS error per pair
    bq = scale * w @ np.abs(k)
    bk = scale * w.T @ np.abs(q)
    bv = U * P.T @ np.abs(do)
    return bq, bk, bv


def check(oracle_mod, q, k, v, do, causal, scale, heads=None):
    o_g, dq_g, dk_g, dv_g = gpu_grads(q, k, v, do, causal, scale)
    B, H = q.shape[:2]
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    f64 = lambda t: t.double().numpy()
    worst_rel = 0.0
    for (b, h) in heads:
        qh, kh, vh, doh = (f64(t[b, h]) for t in (q, k, v, do))
        rq, rk, rv = oracle_mod.attn_bwd_head(qh, kh, vh, doh, causal, scale)
        bq, bk, bv = bounds_head(qh, kh, vh, doh, o_g[b, h].astype(np.float64), causal, scale, oracle_mod)
        for name, got, ref, bnd in (("dQ", dq_g[b, h], rq, bq), ("dK", dk_g[b, h], rk, bk),
                                    ("dV", dv_g[b, h], rv, bv)):
            assert np.isfinite(got).all(), name
            tol = 2.0 * (bnd + U * np.abs(ref)) + 1e-3
            err = np.abs(got - ref)
            bad = err > tol
            assert not bad.any(), (f"{name} head {(b, h)}: {bad.sum()} elements over the bound, "
                                   f"worst excess {np.max(err - tol):.3e}, max err {err.max():.3e}")
            worst_rel = max(worst_rel, float(err.max() / max(np.abs(ref).max(), 1e-30)))
    return worst_rel


SHAPES = [
    (1, 2, 128, 128, 64, False), (1, 2, 128, 128, 64, True),
    (1, 2, 300, 300, 128, True), (1, 2, 300, 300, 128, False),
    (2, 2, 257, 129, 64, False), (1, 3, 129, 500, 128, True),    # Lq < Lk causal: keys past Lq get 0
    (1, 2, 500, 200, 128, True), (1, 1, 1, 1, 64, False), (1, 1, 1, 300, 128, True),
    (2, 1, 640, 640, 64, True), (1, 2, 1000, 1000, 128, True),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_backward_against_oracle(oracle_mod, shape):
    B, H, Lq, Lk, D, causal = shape
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=Lq * 3 + Lk + D + causal)
    do = make_do(B, H, Lq, D, seed=Lq + Lk)
    check(oracle_mod, q, k, v, do, causal, 1.0 / math.sqrt(D))


def test_backward_large_logits(oracle_mod):
    q, k, v = make_qkv(1, 2, 384, 384, 128, seed=7, sigma_qk=3.0)
    do = make_do(1, 2, 384, 128, seed=7)
    check(oracle_mod, q, k, v, do, True, 128 ** -0.5)
    check(oracle_mod, q, k, v, do, False, 0.05)


@pytest.mark.parametrize("name", ["seq4k_d128_causal", "seq1k_d64", "cross_q500_k8191_d128"])
def test_backward_workload_sampled_heads(oracle_mod, name):
    """Full workload on the GPU, two heads compared in full against the oracle (the
    cross-attention workload draws Q and K with standard deviation 3: large logits)."""
    w = WORKLOADS[name]
    q, k, v = make_workload_inputs(w)
    do = make_do(w.B, w.H, w.Lq, w.D, seed=w.seed)
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    check(oracle_mod, q, k, v, do, w.causal, w.scale, heads=heads)


@pytest.mark.parametrize("H,L", [(20, 4096), (10, 8192)])
def test_backward_grouped_units_cover_every_head(H, L):
    """Causal problems hand their units out by groups of heads sized to L2 (Q and dO, or K
    and V, of 16 heads at L = 4096, D = 128; of 8 heads at L = 8192), so H = 20 and H = 10 end
    on a partial group.  Every head, written into NaN-filled gradients, must equal the same
    head computed as a one-head problem."""
    dev = torch.device("cuda:0")
    D = 128
    q, k, v = (t.to(dev) for t in make_qkv(1, H, L, L, D, seed=91 + H))
    do = make_do(1, H, L, D, seed=91 + H).to(dev)
    o, lse = fa.attention(q, k, v, causal=True)
    grads = [torch.full_like(t, float("nan")) for t in (q, k, v)]
    fa.attention_backward(q, k, v, o, lse, do, causal=True, dq=grads[0], dk=grads[1], dv=grads[2])
    assert fa.fa_last_device_status() == fa.FA_OK
    for g in grads:
        assert torch.isfinite(g).all()
    for h in sorted({0, H // 2, H - 2, H - 1}):
        sl = lambda t: t[:, h:h + 1].contiguous()
        one = fa.attention_backward(sl(q), sl(k), sl(v), sl(o), sl(lse), sl(do), causal=True)
        for a, b in zip(grads, one):
            assert torch.equal(a[:, h:h + 1], b), h


@pytest.mark.parametrize("name,kv_pad,dtype", [("seq16k_d128_causal", 0.0, torch.bfloat16),
                                               ("seq16k_d128_window4k", 0.0, torch.bfloat16),
                                               ("seq4k_d64_local256", 0.0, torch.bfloat16),
                                               ("seq16k_d128_causal", 0.25, torch.bfloat16),
                                               ("seq16k_d128_causal", 0.0, torch.float16)])
def test_backward_workload_sampled_rows(oracle_mod, name, kv_pad, dtype):
    """Long workloads of the backward benchmark at sampled outputs of two heads: dQ at
    sampled query rows and dK, dV at sampled key rows against the oracle's row-sampled
    backward (band masks through its masked form), under the element-wise bound of
    ``check`` computed for those rows and columns only (the full-head matrices would take
    up to 2 GB each).  With kv_pad > 0 the keys past each batch's count (drawn as
    ``bench.py --kv-pad`` draws them) are masked too; their dK and dV must be zero.  fp16
    runs on the same values (the bf16 draws are exact in fp16) under the same bound, which
    assumes bf16 rounding and so holds for fp16 too."""
    w = WORKLOADS[name]
    dev = torch.device("cuda:0")
    q, k, v = make_workload_inputs(w)
    do = make_do(w.B, w.H, w.Lq, w.D, seed=w.seed)
    qd, kd, vd, dod = (t.to(dtype).to(dev) for t in (q, k, v, do))
    kv_len = np.full(w.B, w.Lk, dtype=np.int32)
    if kv_pad > 0:
        g = np.random.default_rng(0xCAFE + w.index)
        kv_len = g.integers(max(1, int(round(w.Lk * (1.0 - 2.0 * kv_pad)))), w.Lk + 1, size=w.B).astype(np.int32)
    kl = torch.from_numpy(kv_len).to(dev) if kv_pad > 0 else None
    o, lse_g = fa.attention(qd, kd, vd, causal=w.causal, scale=w.scale, window=w.window, kv_len=kl)
    dq_g, dk_g, dv_g = (t.float().cpu().numpy() for t in
                        fa.attention_backward(qd, kd, vd, o, lse_g, dod, causal=w.causal, scale=w.scale,
                                              window=w.window, kv_len=kl))
    assert fa.fa_last_device_status() == fa.FA_OK
    o_g = o.float().cpu().numpy()
    left, right = w.window if w.window is not None else (-1, 0 if w.causal else -1)
    rng = np.random.default_rng(0x5EED + w.index)
    rows = sorted({0, 1, 127, 128, 129, w.Lq // 2, w.Lq - 1} | set(rng.integers(0, w.Lq, 9).tolist()))
    keys = sorted({0, 1, 127, 128, w.Lk // 2, w.Lk - 1} | set(rng.integers(0, w.Lk, 9).tolist()))
    i_all = np.arange(w.Lq)
    lo_all = np.array([w.key_range(int(i))[0] for i in i_all])
    hi_band = np.array([w.key_range(int(i))[1] for i in i_all])
    check_sampled(oracle_mod, q, k, v, do, o_g, (dq_g, dk_g, dv_g), [(0, 0), (w.B - 1, w.H - 1)],
                  (left, right), kv_len if kv_pad > 0 else None, w.scale, rows, keys, lo_all, hi_band)


def check_sampled(oracle_mod, q, k, v, do, o_g, grads, heads, band, kv_len, sc, rows, keys, lo_all, hi_band):
    """dQ at query rows ``rows`` and dK, dV at key rows ``keys`` of the given heads against
    the oracle's row-sampled backward, under the element-wise bound of ``check`` computed
    for those rows and columns.  Query row i may see keys lo_all[i]..hi_band[i] below the
    batch's key count (``kv_len``, None for all keys); padded keys' gradients must be 0."""
    dq_g, dk_g, dv_g = grads
    left, right = band
    Lk = k.shape[2]
    for (b, h) in heads:
        kv = Lk if kv_len is None else int(kv_len[b])
        keys_b = keys if kv_len is None else sorted(set(keys) | {kv - 1, kv} & set(range(Lk)))
        hi_all = np.minimum(hi_band, kv - 1)
        qh, kh, vh, doh = (t[b, h].double().numpy() for t in (q, k, v, do))
        rq, rk, rv, lse, delta = oracle_mod.attn_bwd_rows_masked(qh, kh, vh, doh, left, right, kv, sc,
                                                                 rows, keys_b)
        e = 2 * U * np.abs(doh * o_g[b, h].astype(np.float64)).sum(axis=1)   # Delta from bf16 O
        for r, i in enumerate(rows):          # query row i sees keys lo..hi
            lo, hi = lo_all[i], hi_all[i]
            p = np.exp(sc * (kh[lo:hi + 1] @ qh[i]) - lse[i])
            ds = p * (vh[lo:hi + 1] @ doh[i] - delta[i])
            bq = sc * (p * e[i] + U * np.abs(ds)) @ np.abs(kh[lo:hi + 1])
            err = np.abs(dq_g[b, h, i] - rq[r])
            assert (err <= 2 * (bq + U * np.abs(rq[r])) + 1e-3).all(), (b, h, i, err.max())
        for r, j in enumerate(keys_b):        # key j is seen by the queries whose range holds it
            sel = (lo_all <= j) & (j <= hi_all)
            qs, dos = qh[sel], doh[sel]
            p = np.exp(sc * (qs @ kh[j]) - lse[sel])
            ds = p * (dos @ vh[j] - delta[sel])
            wgt = p * e[sel] + U * np.abs(ds)
            bk = sc * wgt @ np.abs(qs)
            bv = U * p @ np.abs(dos)
            for nm, got, ref, bnd in (("dK", dk_g[b, h, j], rk[r], bk), ("dV", dv_g[b, h, j], rv[r], bv)):
                err = np.abs(got - ref)
                assert (err <= 2 * (bnd + U * np.abs(ref)) + 1e-3).all(), (nm, b, h, j, err.max())


@pytest.mark.parametrize("B,H,Lq,Lk,D,causal", [(1, 2, 8191, 8191, 128, True), (2, 1, 5000, 12345, 64, False),
                                                (1, 1, 12000, 3000, 128, True)])
def test_backward_large_ragged_sampled(oracle_mod, B, H, Lq, Lk, D, causal):
    """Large problems whose lengths are not tile multiples (causal with Lq > Lk included:
    query rows past Lk see every key), at sampled outputs of the first and last head."""
    dev = torch.device("cuda:0")
    q, k, v = make_qkv(B, H, Lq, Lk, D, seed=Lq + Lk + D)
    do = make_do(B, H, Lq, D, seed=Lq + D)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.attention(qd, kd, vd, causal=causal, scale=scale)
    grads = tuple(t.float().cpu().numpy() for t in fa.attention_backward(qd, kd, vd, o, lse, dod,
                                                                         causal=causal, scale=scale))
    assert fa.fa_last_device_status() == fa.FA_OK
    rng = np.random.default_rng(Lq * 7 + Lk)
    edges = lambda L: {0, 1, 127, 128, 129, L // 2, L - 2, L - 1, (L - 1) // 128 * 128, (L - 1) // 128 * 128 - 1}
    rows = sorted({i for i in edges(Lq) | {Lk - 1, Lk} if 0 <= i < Lq} | set(rng.integers(0, Lq, 8).tolist()))
    keys = sorted({j for j in edges(Lk) if 0 <= j < Lk} | set(rng.integers(0, Lk, 8).tolist()))
    i_all = np.arange(Lq)
    hi_band = np.minimum(i_all, Lk - 1) if causal else np.full(Lq, Lk - 1)
    check_sampled(oracle_mod, q, k, v, do, o.float().cpu().numpy(), grads, [(0, 0), (B - 1, H - 1)],
                  (-1, 0 if causal else -1), None, scale, rows, keys, np.zeros(Lq, dtype=np.int64), hi_band)


def test_backward_unattended_keys_are_zero():
    """Causal with Lq < Lk: keys j >= Lq are seen by no query; their gradients are 0."""
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(1, 2, 200, 700, 64, seed=3))
    do = make_do(1, 2, 200, 64, seed=3).to(dev)
    o, lse = fa.attention(q, k, v, causal=True)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    assert fa.fa_last_device_status() == fa.FA_OK
    assert (dk[:, :, 200:] == 0).all() and (dv[:, :, 200:] == 0).all()
    assert (dk[:, :, :200].abs().sum() > 0) and (dv[:, :, :200].abs().sum() > 0)


def test_backward_empty_query_zero_fills():
    dev = torch.device("cuda:0")
    q = torch.empty((1, 2, 0, 64), dtype=torch.bfloat16, device=dev)
    k = torch.randn((1, 2, 50, 64), device=dev).to(torch.bfloat16)
    dk = torch.full_like(k, 7.0)
    dv = torch.full_like(k, 7.0)
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    st = fa.fa_bwd(q, k, k, q, q, None, None, dk, dv, 1, 2, 0, 50, 64, 0, 0.125, ws, 256, None)
    torch.cuda.synchronize()
    assert st == fa.FA_OK and (dk == 0).all() and (dv == 0).all()


def test_backward_deterministic():
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(2, 4, 1500, 1500, 128, seed=5))
    do = make_do(2, 4, 1500, 128, seed=5).to(dev)
    o, lse = fa.attention(q, k, v, causal=True)
    g1 = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    g2 = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


@pytest.mark.parametrize("B,H,L,D", [(4, 16, 1024, 64), (2, 8, 700, 128)])
def test_backward_chained_calls_see_previous_results(B, H, L, D):
    """Short backward problems launch their kernels as programmatic dependents.  Each call
    here consumes the previous call's dK as its dO and overwrites the buffers the call before
    read (the workspace included): back to back they must give the bits of calls separated
    by a device sync."""
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(B, H, L, L, D, seed=9))
    o, lse = fa.attention(q, k, v, causal=True)
    do0 = make_do(B, H, L, D, seed=9).to(dev)

    def chain(sync):
        do = do0.clone()
        outs = []
        for i in range(5):
            dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, causal=True)
            if sync:
                torch.cuda.synchronize()
            outs.append((dq, dk, dv))
            do = dk   # [B, H, L, D] with Lq == Lk: the next call reads what this one wrote
        torch.cuda.synchronize()
        return outs

    a, b = chain(True), chain(False)
    assert fa.fa_last_device_status() == fa.FA_OK
    for ga, gb in zip(a, b):
        for x, y in zip(ga, gb):
            assert torch.equal(x, y)


@pytest.mark.parametrize("B,H,L,D", [(4, 16, 1024, 64), (1, 16, 8192, 64)])
def test_forward_after_backward_sees_its_gradients(B, H, L, D):
    """The dQ kernel runs beside the dK/dV kernel's last units and waits for that kernel
    only before it exits.  Forward and backward calls alternate here, each forward taking
    the previous backward's dQ, dK, dV as its Q, K, V (a short problem, whose backward
    kernels all launch as dependents, and a long one, whose Delta and dK/dV kernels launch
    plainly): back to back they must give the bits of calls separated by a device sync."""
    dev = torch.device("cuda:0")
    q0, k0, v0 = (t.to(dev) for t in make_qkv(B, H, L, L, D, seed=13))
    do = make_do(B, H, L, D, seed=13).to(dev)

    def chain(sync):
        q, k, v = q0, k0, v0
        outs = []
        for i in range(3):
            o, lse = fa.attention(q, k, v, causal=True)
            if sync:
                torch.cuda.synchronize()
            dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, causal=True)
            if sync:
                torch.cuda.synchronize()
            outs.append((o, lse, dq, dk, dv))
            q, k, v = dq, dk, dv   # the next forward follows the dQ kernel directly
        torch.cuda.synchronize()
        return outs

    a, b = chain(True), chain(False)
    assert fa.fa_last_device_status() == fa.FA_OK
    for ga, gb in zip(a, b):
        for x, y in zip(ga, gb):
            assert torch.isfinite(x.float()).all()
            assert torch.equal(x, y)


def test_few_key_tiles_fork_and_join():
    """With fewer key tiles than SMs the dQ kernel runs on the library's own stream beside
    the dK/dV kernel, and the caller's stream waits for it.  One causal head of 16K tokens
    (128 key tiles; its dQ kernel takes about 0.1 ms) on a side stream, with a reduction
    of each gradient queued on that stream right behind the call: the sums and the bits
    must be those of the same call followed by a device sync."""
    dev = torch.device("cuda:0")
    B, H, L, D = 1, 1, 16384, 128
    q, k, v = (t.to(dev) for t in make_qkv(B, H, L, L, D, seed=21))
    do = make_do(B, H, L, D, seed=21).to(dev)
    o, lse = fa.attention(q, k, v, causal=True)
    ref = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    ref_sums = torch.stack([r.float().sum() for r in ref])
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        grads = fa.attention_backward(q, k, v, o, lse, do, causal=True)
        sums = torch.stack([g.float().sum() for g in grads])
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    for g, r in zip(grads, ref):
        assert torch.isfinite(g.float()).all()
        assert torch.equal(g, r)
    assert torch.equal(sums, ref_sums)


def test_few_key_tiles_backward_in_a_cuda_graph():
    """The forked backward captured into a CUDA graph (the library's stream joins the
    capture through the fork event and leaves it through the join event): replays give
    the bits of an eager call.  The first call, which creates the library's stream and
    the cached workspace, is made before the capture."""
    dev = torch.device("cuda:0")
    B, H, L, D = 1, 2, 8192, 128   # 128 key tiles and 128 query tiles against 152 SMs
    q, k, v = (t.to(dev) for t in make_qkv(B, H, L, L, D, seed=23))
    do = make_do(B, H, L, D, seed=23).to(dev)
    o, lse = fa.attention(q, k, v, causal=True)
    ref = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    grads = tuple(torch.empty_like(t) for t in (q, k, v))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.attention_backward(q, k, v, o, lse, do, causal=True, dq=grads[0], dk=grads[1], dv=grads[2])
    for _ in range(2):
        for t in grads:
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert fa.fa_last_device_status() == fa.FA_OK
        for x, r in zip(grads, ref):
            assert torch.equal(x, r)


def test_few_key_tiles_from_two_threads():
    """Two host threads, each on its own stream, call the backward of few-key-tile
    problems (both take the library's second stream: 128 key tiles and 128 query tiles
    against 152 SMs) while the other does: every result must equal the same call made
    alone."""
    import threading
    dev = torch.device("cuda:0")
    cases = [(1, 1, 16384, 64, 31), (1, 2, 8192, 128, 32)]
    inputs, refs = [], []
    for B, H, L, D, seed in cases:
        q, k, v = (t.to(dev) for t in make_qkv(B, H, L, L, D, seed=seed))
        do = make_do(B, H, L, D, seed=seed).to(dev)
        o, lse = fa.attention(q, k, v, causal=True)
        inputs.append((q, k, v, o, lse, do))
        refs.append(fa.attention_backward(q, k, v, o, lse, do, causal=True))
    torch.cuda.synchronize()
    out = {}

    def work(i):
        try:   # the C entry point with this thread's own workspace and outputs
            q, k, v, o, lse, do = inputs[i]
            B, H, L, D = q.shape
            st, nb = fa.fa_bwd_workspace_size(B, H, L, L, D, 1)
            assert st == fa.FA_OK
            ws = torch.empty(nb, dtype=torch.uint8, device=dev)
            s = torch.cuda.Stream(dev)
            res = []
            for _ in range(4):
                g = tuple(torch.empty_like(t) for t in (q, k, v))
                st = fa.fa_bwd(q, k, v, o, do, lse, *g, B, H, L, L, D, 1, 1.0 / math.sqrt(D), ws, nb, s)
                assert st == fa.FA_OK, fa.fa_status_string(st)
                res.append(g)
            s.synchronize()
            out[i] = res
        except Exception as e:   # reported in the main thread
            out[f"err{i}"] = e

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not [k for k in out if str(k).startswith("err")], out
    assert fa.fa_last_device_status() == fa.FA_OK
    for i in range(2):
        for grads in out[i]:
            for g, r in zip(grads, refs[i]):
                assert torch.equal(g, r)


def test_autograd_function_matches_direct_calls():
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev).requires_grad_(True) for t in make_qkv(1, 2, 300, 400, 64, seed=9))
    do = make_do(1, 2, 300, 64, seed=9).to(dev)
    o = fa.flash_attention(q, k, v, causal=True)
    o.backward(do)
    o2, lse = fa.attention(q.detach(), k.detach(), v.detach(), causal=True)
    dq, dk, dv = fa.attention_backward(q.detach(), k.detach(), v.detach(), o2, lse, do, causal=True)
    assert torch.equal(o, o2)
    assert torch.equal(q.grad, dq) and torch.equal(k.grad, dk) and torch.equal(v.grad, dv)


def test_calls_from_a_fresh_thread():
    """A thread that never touched CUDA before (as autograd's backward thread): the
    library makes the device's context current itself."""
    import threading
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(1, 2, 200, 200, 128, seed=4))
    do = make_do(1, 2, 200, 128, seed=4).to(dev)
    o_ref, l_ref = fa.attention(q, k, v, causal=True)
    g_ref = fa.attention_backward(q, k, v, o_ref, l_ref, do, causal=True)
    torch.cuda.synchronize()
    out = {}

    def work():
        try:
            o, lse = fa.attention(q, k, v, causal=True, stream=0)
            out["g"] = fa.attention_backward(q, k, v, o, lse, do, causal=True, stream=0)
            torch.cuda.synchronize()
            out["o"] = o
        except Exception as e:   # reported in the main thread
            out["err"] = e

    t = threading.Thread(target=work)
    t.start()
    t.join()
    assert "err" not in out, out.get("err")
    assert torch.equal(out["o"], o_ref)
    for a, b in zip(out["g"], g_ref):
        assert torch.equal(a, b)


# ---------------------------------------------------------------- band and key padding
def check_masked(oracle_mod, q, k, v, do, left, right, kv_len, scale):
    """fa_bwd_masked against oracle_attn_bwd_head_masked, with the per-element bound of
    ``check`` (P from the key-padding forward oracle)."""
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    kl = None if kv_len is None else torch.tensor(kv_len, dtype=torch.int32, device=dev)
    o, lse = fa.attention(qd, kd, vd, window=(left, right), kv_len=kl, scale=scale)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, window=(left, right), kv_len=kl, scale=scale)
    assert fa.fa_last_device_status() == fa.FA_OK
    got = [t.float().cpu().numpy() for t in (dq, dk, dv)]
    o_g = o.float().cpu().numpy()
    B, H, Lq, D = q.shape
    Lk = k.shape[2]
    f64 = lambda t: t.double().numpy()
    for b in range(B):
        kvb = Lk if kv_len is None else kv_len[b]
        for h in range(H):
            qh, kh, vh, doh = (f64(t[b, h]) for t in (q, k, v, do))
            refs = oracle_mod.attn_bwd_head_masked(qh, kh, vh, doh, left, right, kvb, scale)
            P = oracle_mod.attn_head_keypad(qh, kh, vh, left, right, kvb, scale, want_p=True)[2]
            dP = doh @ vh.T
            dS = P * (dP - (P * dP).sum(axis=1)[:, None])
            e = 2 * U * np.abs(doh * o_g[b, h]).sum(axis=1)
            w = P * e[:, None] + U * np.abs(dS)
            bnds = (scale * w @ np.abs(kh), scale * w.T @ np.abs(qh), U * P.T @ np.abs(doh))
            for name, g_, ref, bnd in zip(("dQ", "dK", "dV"), got, refs, bnds):
                gh = g_[b, h]
                assert np.isfinite(gh).all(), name
                tol = 2.0 * (bnd + U * np.abs(ref)) + 1e-3
                bad = np.abs(gh - ref) > tol
                assert not bad.any(), f"{name} {(b, h)}: {bad.sum()} over the bound, max err {np.abs(gh - ref).max():.3e}"


@pytest.mark.parametrize("left,right", [(100, 0), (64, 64), (-1, 30), (200, -1), (0, 0)])
@pytest.mark.parametrize("D", [64, 128])
def test_backward_band_against_oracle(oracle_mod, left, right, D):
    q, k, v = make_qkv(1, 2, 500, 500, D, seed=left + 3 * right + D)
    do = make_do(1, 2, 500, D, seed=left + right)
    check_masked(oracle_mod, q, k, v, do, left, right, None, 1.0 / math.sqrt(D))


@pytest.mark.parametrize("left,right", [(-1, -1), (-1, 0), (50, 50)])
def test_backward_key_padding_against_oracle(oracle_mod, left, right):
    q, k, v = make_qkv(4, 2, 300, 420, 128, seed=71 + left)
    do = make_do(4, 2, 300, 128, seed=71)
    check_masked(oracle_mod, q, k, v, do, left, right, [420, 0, 1, 257], 128 ** -0.5)


def test_backward_masked_full_and_causal_equal_fa_bwd():
    """(-1, -1) and (-1, 0) with no padding through fa_bwd_masked give fa_bwd's bits."""
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(2, 2, 600, 700, 128, seed=73))
    do = make_do(2, 2, 600, 128, seed=73).to(dev)
    for causal, win in ((False, (-1, -1)), (True, (-1, 0))):
        o, lse = fa.attention(q, k, v, causal=causal, split=False)
        a = fa.attention_backward(q, k, v, o, lse, do, causal=causal)
        st, nb = fa.fa_bwd_workspace_size(2, 2, 600, 700, 128, causal)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        b = [torch.empty_like(t) for t in (q, k, v)]
        assert fa.fa_bwd_masked(q, k, v, o, do, lse, *b, None, 2, 2, 600, 700, 128, win[0], win[1],
                                128 ** -0.5, ws, nb, None) == fa.FA_OK
        torch.cuda.synchronize()
        for x, y in zip(a, b):
            assert torch.equal(x, y)


def test_autograd_with_window_and_padding(oracle_mod):
    dev = torch.device("cuda:0")
    q, k, v = make_qkv(2, 2, 256, 256, 64, seed=79)
    do = make_do(2, 2, 256, 64, seed=79)
    kl = torch.tensor([256, 100], dtype=torch.int32, device=dev)
    qg, kg, vg = (t.to(dev).requires_grad_(True) for t in (q, k, v))
    o = fa.flash_attention(qg, kg, vg, window=(40, 0), kv_len=kl)
    o.backward(do.to(dev))
    for b, kvb in enumerate((256, 100)):
        for h in range(2):
            ref = oracle_mod.attn_bwd_head_masked(q[b, h].double().numpy(), k[b, h].double().numpy(),
                                                  v[b, h].double().numpy(), do[b, h].double().numpy(),
                                                  40, 0, kvb, 0.125)
            for g_, r in zip((qg.grad, kg.grad, vg.grad), ref):
                assert np.abs(g_[b, h].float().cpu().numpy() - r).max() < 5e-2


# ---------------------------------------------------------------- strided layouts and fp16
def _packed(B, H, L, D, dtype, seed):
    q, k, v = make_qkv(B, H, L, L, D, seed)
    dev = torch.device("cuda:0")
    packed = torch.empty((B, L, 3, H, D), dtype=dtype, device=dev)
    for i, t in enumerate((q, k, v)):
        packed[:, :, i] = t.to(dtype).to(dev).transpose(1, 2)
    return tuple(packed[:, :, i].transpose(1, 2) for i in range(3)), (q, k, v)


@pytest.mark.parametrize("causal,D", [(True, 128), (False, 64)])
def test_backward_strided_equals_contiguous(causal, D):
    """Q, K, V from a packed [B, L, 3, H, D] projection, gradients written into a
    [B, L, H, D] buffer: the bits of the contiguous call."""
    dev = torch.device("cuda:0")
    (qv, kv, vv), (q, k, v) = _packed(2, 3, 400, D, torch.bfloat16, seed=81 + D)
    qc, kc, vc = (t.to(dev) for t in (q, k, v))
    do = make_do(2, 3, 400, D, seed=81).to(dev)
    o, lse = fa.attention(qc, kc, vc, causal=causal, split=False)
    ref = fa.attention_backward(qc, kc, vc, o, lse, do, causal=causal)
    bufs = [torch.full((2, 400, 3, D), 9.0, dtype=torch.bfloat16, device=dev) for _ in range(3)]
    outs = [b.transpose(1, 2) for b in bufs]
    got = fa.attention_backward(qv, kv, vv, o, lse, do, causal=causal, dq=outs[0], dk=outs[1], dv=outs[2])
    assert fa.fa_last_device_status() == fa.FA_OK
    for g_, r in zip(got, ref):
        assert torch.equal(g_, r)


@pytest.mark.parametrize("causal,D,window", [(True, 128, None), (False, 64, None), (False, 128, (100, 20))])
def test_backward_fp16_against_oracle(oracle_mod, causal, D, window):
    dev = torch.device("cuda:0")
    q, k, v = make_qkv(1, 2, 300, 300, D, seed=91 + D)
    do = make_do(1, 2, 300, D, seed=91)
    q16, k16, v16, do16 = (t.to(torch.float16).to(dev) for t in (q, k, v, do))
    o, lse = fa.attention(q16, k16, v16, causal=causal, window=window)
    dq, dk, dv = fa.attention_backward(q16, k16, v16, o, lse, do16, causal=causal, window=window)
    assert dq.dtype == torch.float16 and fa.fa_last_device_status() == fa.FA_OK
    left, right = window if window is not None else (-1, 0 if causal else -1)
    for h in range(2):
        ref = oracle_mod.attn_bwd_head_masked(q[0, h].double().numpy(), k[0, h].double().numpy(),
                                              v[0, h].double().numpy(), do[0, h].double().numpy(),
                                              left, right, 300, 1.0 / math.sqrt(D))
        for g_, r in zip((dq, dk, dv), ref):
            err = np.abs(g_[0, h].float().cpu().numpy() - r).max()
            assert err <= 2e-2 * max(1.0, np.abs(r).max()), err


def test_fp16_autograd_through_packed_views():
    dev = torch.device("cuda:0")
    (qv, kv, vv), _ = _packed(1, 2, 256, 64, torch.float16, seed=97)
    leaf = qv._base if qv._base is not None else qv
    leaf.requires_grad_(True)
    q, k, v = (leaf[:, :, i].transpose(1, 2) for i in range(3))
    o = fa.flash_attention(q, k, v, causal=True)
    o.float().sum().backward()
    assert leaf.grad is not None and torch.isfinite(leaf.grad.float()).all()
    assert leaf.grad.abs().sum() > 0
