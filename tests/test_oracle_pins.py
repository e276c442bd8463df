"""Pins for the fp64 oracle: facts fixed by the pages and by the mathematics.

None of these compares the oracle with itself or with the CUDA path.  They use
closed forms, invariants, special cases that reduce to a library routine
(torch fp64 softmax / logsumexp), an independent online-softmax recurrence, and
hand-worked fixtures under tests/golden/.  The last test plants plausible
mistakes in a copy of the oracle source and checks that the pins catch each.
"""
import json
import math
import os
import shutil

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _allowed(i, Lk, causal):
    return min(i + 1, Lk) if causal else Lk


# --------------------------------------------------------------------------
# The individual pins, each taking an oracle library so the mutation test can
# run them against a deliberately broken copy.
# --------------------------------------------------------------------------

def pin_rows_sum_to_one(lib):
    """Every probability row sums to 1 and is exactly 0 on masked keys."""
    for causal, (Lq, Lk) in [(False, (7, 11)), (True, (9, 9)), (True, (12, 5)), (True, (4, 10))]:
        q, k, v = _rand((Lq, 16), 1), _rand((Lk, 16), 2), _rand((Lk, 16), 3)
        _, _, P = lib.attn_head(q, k, v, causal, 0.25, want_p=True)
        assert np.allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
        for i in range(Lq):
            n = _allowed(i, Lk, causal)
            assert np.all(P[i, n:] == 0.0)
            assert np.all(P[i, :n] > 0.0)


def pin_single_key(lib):
    """Lk = 1: O is exactly V's only row; LSE is that row's scaled score."""
    q, k, v = _rand((6, 32), 4), _rand((1, 32), 5), _rand((1, 32), 6)
    for causal in (False, True):
        O, L = lib.attn_head(q, k, v, causal, 0.3)
        assert np.array_equal(O, np.repeat(v, 6, axis=0))
        np.testing.assert_allclose(L, 0.3 * (q @ k[0]), rtol=0, atol=1e-12)


def pin_constant_v(lib):
    """All value rows equal c: every output row is c."""
    q, k = _rand((10, 8), 7), _rand((13, 8), 8)
    c = _rand((8,), 9)
    v = np.tile(c, (13, 1))
    for causal in (False, True):
        O, _ = lib.attn_head(q, k, v, causal, 0.5)
        np.testing.assert_allclose(O, np.tile(c, (10, 1)), rtol=0, atol=1e-12)


def pin_causal_row0(lib):
    """Causal row 0 sees only key 0: O_0 = V_0, LSE_0 = scale * q_0 . k_0."""
    q, k, v = _rand((5, 8), 10), _rand((7, 8), 11), _rand((7, 8), 12)
    O, L = lib.attn_head(q, k, v, True, 0.7)
    np.testing.assert_allclose(O[0], v[0], rtol=0, atol=1e-12)
    assert abs(L[0] - 0.7 * (q[0] @ k[0])) < 1e-12


def pin_uniform_scores(lib):
    """Q = 0 makes every score 0: O_i is the mean of the allowed value rows and
    LSE_i = ln(number of allowed keys).  Pins the causal key count per row."""
    for causal, (Lq, Lk) in [(False, (5, 9)), (True, (9, 9)), (True, (11, 6)), (True, (3, 8))]:
        q, k, v = np.zeros((Lq, 4)), _rand((Lk, 4), 13), _rand((Lk, 4), 14)
        O, L = lib.attn_head(q, k, v, causal, 1.0)
        for i in range(Lq):
            n = _allowed(i, Lk, causal)
            np.testing.assert_allclose(O[i], v[:n].mean(axis=0), rtol=0, atol=1e-12)
            assert abs(L[i] - math.log(n)) < 1e-12


def pin_permutation(lib):
    """Non-causal attention is invariant under one permutation of K and V rows."""
    q, k, v = _rand((6, 8), 15), _rand((10, 8), 16), _rand((10, 8), 17)
    perm = np.random.default_rng(18).permutation(10)
    O1, L1 = lib.attn_head(q, k, v, False, 0.4)
    O2, L2 = lib.attn_head(q, k[perm], v[perm], False, 0.4)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L1, L2, rtol=0, atol=1e-12)


def pin_key_shift(lib):
    """Adding u to every key row leaves O unchanged and moves LSE_i by scale*q_i.u."""
    q, k, v = _rand((6, 8), 19), _rand((9, 8), 20), _rand((9, 8), 21)
    u = _rand((8,), 22)
    for causal in (False, True):
        O1, L1 = lib.attn_head(q, k, v, causal, 0.35)
        O2, L2 = lib.attn_head(q, k + u, v, causal, 0.35)
        np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-11)
        np.testing.assert_allclose(L2 - L1, 0.35 * (q @ u), rtol=0, atol=1e-11)


def pin_torch_f64(lib):
    """Brute force on tiny shapes: torch fp64 softmax / logsumexp with a mask."""
    cases = [(1, 1, 3, 3, 4, False), (2, 3, 5, 7, 8, True), (1, 2, 9, 4, 16, True),
             (2, 1, 6, 6, 8, False), (1, 1, 4, 11, 8, True)]
    for (B, H, Lq, Lk, D, causal) in cases:
        g = torch.Generator().manual_seed(Lq * 100 + Lk)
        q = torch.randn(B, H, Lq, D, generator=g, dtype=torch.float64)
        k = torch.randn(B, H, Lk, D, generator=g, dtype=torch.float64)
        v = torch.randn(B, H, Lk, D, generator=g, dtype=torch.float64)
        scale = 1.0 / math.sqrt(D)
        s = torch.einsum("bhid,bhjd->bhij", q, k) * scale
        if causal:
            keep = torch.arange(Lq)[:, None] >= torch.arange(Lk)[None, :]
            s = s.masked_fill(~keep, float("-inf"))
        ref_o = torch.softmax(s, dim=-1) @ v
        ref_l = torch.logsumexp(s, dim=-1)
        O, L = lib.attn_full(q.numpy(), k.numpy(), v.numpy(), causal, scale)
        np.testing.assert_allclose(O, ref_o.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(L, ref_l.numpy(), rtol=0, atol=1e-12)


def _online(q, k, v, causal, scale, block):
    """Online softmax over key blocks of size ``block``, as the "Triton Ascend
    Attention" page's 在线 Softmax 算法 sketch states it (running max m, running
    exp-sum l, accumulator rescaled by alpha = exp(m_old - m_new)), applied to
    rows of scores, with the final divide by l and the statistic m + log(l)."""
    Lq, Lk = q.shape[0], k.shape[0]
    O = np.zeros((Lq, v.shape[1]))
    L = np.zeros(Lq)
    for i in range(Lq):
        n = _allowed(i, Lk, causal)
        m, l, acc = -np.inf, 0.0, np.zeros(v.shape[1])
        for j0 in range(0, n, block):
            j1 = min(n, j0 + block)
            s = scale * (k[j0:j1] @ q[i])
            m_new = max(m, s.max())
            p = np.exp(s - m_new)
            alpha = math.exp(m - m_new)
            l = l * alpha + p.sum()
            acc = acc * alpha + p @ v[j0:j1]
            m = m_new
        O[i] = acc / l
        L[i] = m + math.log(l)
    return O, L


def pin_online_recurrence(lib):
    """The online recurrence, for every key-block size, equals the definition."""
    q, k, v = _rand((6, 8), 23, 2.0), _rand((9, 8), 24, 2.0), _rand((9, 8), 25)
    for causal in (False, True):
        O, L = lib.attn_head(q, k, v, causal, 0.6)
        for block in range(1, 10):
            O2, L2 = _online(q, k, v, causal, 0.6, block)
            np.testing.assert_allclose(O, O2, rtol=0, atol=1e-12)
            np.testing.assert_allclose(L, L2, rtol=0, atol=1e-12)


def pin_golden(lib):
    """Hand-worked closed forms (tests/golden/closed_forms.json)."""
    with open(os.path.join(HERE, "golden", "closed_forms.json")) as f:
        cases = json.load(f)["cases"]
    env = {"e": math.e, "exp": math.exp, "log": math.log, "sqrt": math.sqrt, "__builtins__": {}}
    for c in cases:
        q, k, v = (np.array(c[x], dtype=np.float64) for x in ("Q", "K", "V"))
        O, L = lib.attn_head(q, k, v, c["causal"], c["scale"])
        exp_o = np.array([[eval(x, env) for x in row] for row in c["O"]])
        exp_l = np.array([eval(x, env) for x in c["LSE"]])
        np.testing.assert_allclose(O, exp_o, rtol=0, atol=1e-14, err_msg=c["name"])
        np.testing.assert_allclose(L, exp_l, rtol=0, atol=1e-14, err_msg=c["name"])


def pin_row_subset(lib):
    """Computing a subset of rows gives exactly those rows of the full result."""
    q, k, v = _rand((20, 8), 26), _rand((17, 8), 27), _rand((17, 8), 28)
    for causal in (False, True):
        O, L = lib.attn_head(q, k, v, causal, 0.5)
        rows = [19, 0, 7, 7, 16]
        Os, Ls = lib.attn_head(q, k, v, causal, 0.5, rows=rows)
        assert np.array_equal(Os, O[rows]) and np.array_equal(Ls, L[rows])


PINS = [pin_rows_sum_to_one, pin_single_key, pin_constant_v, pin_causal_row0,
        pin_uniform_scores, pin_permutation, pin_key_shift, pin_torch_f64,
        pin_online_recurrence, pin_golden, pin_row_subset]


# --------------------------------------------------------------------------
# Local (sliding-window) attention: key j allowed for row i iff
# i - left <= j <= i + right (-1 = unbounded).
# --------------------------------------------------------------------------

def _window(i, Lk, left, right):
    lo = 0 if left < 0 else max(0, i - left)
    hi = Lk - 1 if right < 0 else min(Lk - 1, i + right)
    return lo, hi


WINDOW_CASES = [(9, 9, 3, 0), (12, 9, 4, 2), (6, 15, 2, 5), (10, 10, -1, 1), (8, 20, 0, -1),
                (5, 5, 1, 1)]


def pin_window_torch_f64(lib):
    """Brute force with torch fp64 and an explicit window mask."""
    for (Lq, Lk, left, right) in WINDOW_CASES:
        g = torch.Generator().manual_seed(Lq * 31 + Lk + left)
        q = torch.randn(Lq, 8, generator=g, dtype=torch.float64)
        k = torch.randn(Lk, 8, generator=g, dtype=torch.float64)
        v = torch.randn(Lk, 8, generator=g, dtype=torch.float64)
        i = torch.arange(Lq)[:, None]
        j = torch.arange(Lk)[None, :]
        keep = torch.ones(Lq, Lk, dtype=torch.bool)
        if left >= 0:
            keep &= j >= i - left
        if right >= 0:
            keep &= j <= i + right
        s = (q @ k.T * 0.4).masked_fill(~keep, float("-inf"))
        O, L = lib.attn_head_window(q.numpy(), k.numpy(), v.numpy(), left, right, 0.4)
        np.testing.assert_allclose(O, (torch.softmax(s, -1) @ v).numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(L, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def pin_window_uniform(lib):
    """Q = 0: each row averages exactly the value rows in its window, LSE = ln(width)."""
    for (Lq, Lk, left, right) in WINDOW_CASES:
        q, k, v = np.zeros((Lq, 4)), _rand((Lk, 4), 50), _rand((Lk, 4), 51)
        O, L = lib.attn_head_window(q, k, v, left, right, 1.0)
        for i in range(Lq):
            lo, hi = _window(i, Lk, left, right)
            np.testing.assert_allclose(O[i], v[lo:hi + 1].mean(axis=0), rtol=0, atol=1e-12)
            assert abs(L[i] - math.log(hi - lo + 1)) < 1e-12


def pin_window_single_key(lib):
    """left = right = 0: row i sees only key i: O_i = V_i, LSE_i = scale q_i . k_i."""
    q, k, v = _rand((6, 8), 52), _rand((9, 8), 53), _rand((9, 8), 54)
    O, L = lib.attn_head_window(q, k, v, 0, 0, 0.7)
    np.testing.assert_allclose(O, v[:6], rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, 0.7 * np.einsum("id,id->i", q, k[:6]), rtol=0, atol=1e-12)


def pin_window_rows(lib):
    """Probability rows sum to 1, are positive inside the window and 0 outside."""
    for (Lq, Lk, left, right) in WINDOW_CASES:
        q, k, v = _rand((Lq, 8), 55), _rand((Lk, 8), 56), _rand((Lk, 8), 57)
        _, _, P = lib.attn_head_window(q, k, v, left, right, 0.5, want_p=True)
        for i in range(Lq):
            lo, hi = _window(i, Lk, left, right)
            assert abs(P[i].sum() - 1.0) < 1e-12
            assert np.all(P[i, lo:hi + 1] > 0) and np.all(P[i, :lo] == 0) and np.all(P[i, hi + 1:] == 0)


def pin_window_online(lib):
    """The online recurrence over the window's keys, for every block size."""
    q, k, v = _rand((7, 8), 58, 2.0), _rand((12, 8), 59, 2.0), _rand((12, 8), 60)
    left, right = 3, 2
    O, L = lib.attn_head_window(q, k, v, left, right, 0.6)
    for block in range(1, 8):
        for i in range(7):
            lo, hi = _window(i, 12, left, right)
            o2, l2 = _online(q[i:i + 1], k[lo:hi + 1], v[lo:hi + 1], False, 0.6, block)
            np.testing.assert_allclose(O[i], o2[0], rtol=0, atol=1e-12)
            assert abs(L[i] - l2[0]) < 1e-12


WINDOW_PINS = [pin_window_torch_f64, pin_window_uniform, pin_window_single_key, pin_window_rows,
               pin_window_online]
PINS.extend(WINDOW_PINS)


# --------------------------------------------------------------------------
# Backward pass (gradients): pinned by central finite differences of the forward
# oracle, which shares no arithmetic with the gradient formulas.
# --------------------------------------------------------------------------

def _fd_grads(lib, q, k, v, g, causal, scale, eps=1e-6):
    def loss(**kw):
        a = dict(q=q, k=k, v=v)
        a.update(kw)
        return float((lib.attn_head(a["q"], a["k"], a["v"], causal, scale)[0] * g).sum())
    out = []
    for name, x in (("q", q), ("k", k), ("v", v)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            fd[idx] = (loss(**{name: xp}) - loss(**{name: xm})) / (2 * eps)
        out.append(fd)
    return out


def pin_bwd_finite_differences(lib):
    """dQ, dK, dV equal the central differences of sum(G * O) to 1e-7."""
    for (Lq, Lk, D, causal) in [(5, 6, 3, False), (5, 6, 3, True), (7, 4, 2, True), (3, 8, 4, False)]:
        q, k, v = _rand((Lq, D), 70 + Lq, 1.5), _rand((Lk, D), 71 + Lk, 1.5), _rand((Lk, D), 72)
        g = _rand((Lq, D), 73)
        dq, dk, dv = lib.attn_bwd_head(q, k, v, g, causal, 0.7)
        for got, fd in zip((dq, dk, dv), _fd_grads(lib, q, k, v, g, causal, 0.7)):
            np.testing.assert_allclose(got, fd, rtol=0, atol=1e-7)


def pin_bwd_constant_v(lib):
    """Every value row equal: O does not depend on Q or K, so dQ = dK = 0."""
    q, k = _rand((6, 4), 74), _rand((9, 4), 75)
    v = np.tile(_rand((1, 4), 76), (9, 1))
    for causal in (False, True):
        dq, dk, _ = lib.attn_bwd_head(q, k, v, _rand((6, 4), 77), causal, 0.5)
        assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12


def pin_bwd_sums(lib):
    """Rows of P sum to 1 and rows of dS to 0: sum_j dV_j = sum_i dO_i, sum_j dK_j = 0."""
    q, k, v, g = _rand((8, 5), 78), _rand((11, 5), 79), _rand((11, 5), 80), _rand((8, 5), 81)
    for causal in (False, True):
        dq, dk, dv = lib.attn_bwd_head(q, k, v, g, causal, 0.9)
        np.testing.assert_allclose(dv.sum(axis=0), g.sum(axis=0), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dk.sum(axis=0), 0.0, rtol=0, atol=1e-12)


def pin_bwd_single_key(lib):
    """Lk = 1: P = 1, so dV_0 = sum_i dO_i and dQ = dK = 0."""
    q, k, v, g = _rand((5, 3), 82), _rand((1, 3), 83), _rand((1, 3), 84), _rand((5, 3), 85)
    dq, dk, dv = lib.attn_bwd_head(q, k, v, g, False, 1.0)
    np.testing.assert_allclose(dv[0], g.sum(axis=0), rtol=0, atol=1e-12)
    assert np.abs(dq).max() == 0.0 and np.abs(dk).max() == 0.0


def pin_bwd_rows_finite_differences(lib):
    """The row-sampled backward at its sampled rows equals central differences of
    sum(G * O) (to 1e-7), and its LSE equals the forward's."""
    for (Lq, Lk, D, causal) in [(5, 6, 3, False), (6, 6, 3, True), (7, 4, 2, True), (3, 8, 4, False)]:
        q, k, v = _rand((Lq, D), 90 + Lq, 1.5), _rand((Lk, D), 91 + Lk, 1.5), _rand((Lk, D), 92)
        g = _rand((Lq, D), 93)
        qr, kr = [0, Lq - 1, Lq // 2], [0, Lk - 1, Lk // 2]
        dq, dk, dv, lse, _ = lib.attn_bwd_rows(q, k, v, g, causal, 0.7, qr, kr)
        fq, fk, fv = _fd_grads(lib, q, k, v, g, causal, 0.7)
        for got, fd in ((dq, fq[qr]), (dk, fk[kr]), (dv, fv[kr])):
            np.testing.assert_allclose(got, fd, rtol=0, atol=1e-7)
        np.testing.assert_allclose(lse, lib.attn_head(q, k, v, causal, 0.7)[1], rtol=0, atol=1e-12)


def pin_bwd_rows_match_full_head(lib):
    """On heads small enough for both: the row-sampled backward equals the full-head one at
    the sampled rows, and Delta_i = sum_j P_ij dP_ij equals dO_i . O_i (the identity the
    kernels' Delta uses)."""
    for (Lq, Lk, D, causal) in [(37, 53, 8, True), (37, 53, 8, False), (60, 20, 5, True), (1, 1, 4, False)]:
        q, k, v, g = (_rand(sh, 100 + Lq + i) for i, sh in enumerate(((Lq, D), (Lk, D), (Lk, D), (Lq, D))))
        qr, kr = sorted({0, Lq - 1, Lq // 2, Lq // 3}), sorted({0, Lk - 1, Lk // 2, Lk // 5})
        dq, dk, dv, _, delta = lib.attn_bwd_rows(q, k, v, g, causal, 0.6, qr, kr)
        fq, fk, fv = lib.attn_bwd_head(q, k, v, g, causal, 0.6)
        for got, ref in ((dq, fq[qr]), (dk, fk[kr]), (dv, fv[kr])):
            np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
        o, _ = lib.attn_head(q, k, v, causal, 0.6)
        np.testing.assert_allclose(delta, (g * o).sum(axis=1), rtol=0, atol=1e-12)


BWD_PINS = [pin_bwd_finite_differences, pin_bwd_constant_v, pin_bwd_sums, pin_bwd_single_key,
            pin_bwd_rows_finite_differences, pin_bwd_rows_match_full_head]
PINS.extend(BWD_PINS)


# --------------------------------------------------------------------------
# Key padding: keys j >= kv_len masked on top of the band; empty rows give
# O = 0, LSE = -inf.
# --------------------------------------------------------------------------

KEYPAD_CASES = [(9, 12, -1, -1, 7), (10, 10, -1, 0, 4), (8, 15, 3, 2, 11), (6, 6, 0, 0, 3),
                (7, 9, -1, -1, 0), (12, 20, 2, -1, 20)]


def pin_keypad_torch_f64(lib):
    """Brute force with torch fp64 and explicit band and padding masks."""
    for (Lq, Lk, left, right, kv) in KEYPAD_CASES:
        g = torch.Generator().manual_seed(Lq * 13 + Lk + kv)
        q = torch.randn(Lq, 6, generator=g, dtype=torch.float64)
        k = torch.randn(Lk, 6, generator=g, dtype=torch.float64)
        v = torch.randn(Lk, 6, generator=g, dtype=torch.float64)
        i = torch.arange(Lq)[:, None]
        j = torch.arange(Lk)[None, :]
        keep = (j < kv) & (i >= 0)   # [Lq, Lk]
        if left >= 0:
            keep = keep & (j >= i - left)
        if right >= 0:
            keep = keep & (j <= i + right)
        s = (q @ k.T * 0.3).masked_fill(~keep, float("-inf"))
        O, L = lib.attn_head_keypad(q.numpy(), k.numpy(), v.numpy(), left, right, kv, 0.3)
        full = keep.any(dim=1)
        ref_o = torch.where(full[:, None], torch.softmax(s, -1).nan_to_num(0.0) @ v, torch.zeros(1, dtype=torch.float64))
        np.testing.assert_allclose(O, ref_o.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(L[full.numpy()], torch.logsumexp(s, -1)[full].numpy(), rtol=0, atol=1e-12)
        assert np.all(np.isneginf(L[~full.numpy()])) and np.all(O[~full.numpy()] == 0.0)


def pin_keypad_uniform(lib):
    """Q = 0: the mean of the values of the unpadded part of the band, LSE = ln(count)."""
    for (Lq, Lk, left, right, kv) in KEYPAD_CASES:
        q, k, v = np.zeros((Lq, 4)), _rand((Lk, 4), 90), _rand((Lk, 4), 91)
        O, L = lib.attn_head_keypad(q, k, v, left, right, kv, 1.0)
        for i in range(Lq):
            lo, hi = _window(i, Lk, left, right)
            hi = min(hi, kv - 1)
            if lo > hi:
                assert np.isneginf(L[i]) and np.all(O[i] == 0.0)
            else:
                np.testing.assert_allclose(O[i], v[lo:hi + 1].mean(axis=0), rtol=0, atol=1e-12)
                assert abs(L[i] - math.log(hi - lo + 1)) < 1e-12


def pin_keypad_no_padding_is_window(lib):
    """kv_len >= Lk: exactly the band oracle."""
    q, k, v = _rand((11, 5), 92), _rand((13, 5), 93), _rand((13, 5), 94)
    for (left, right) in ((-1, -1), (-1, 0), (4, 2)):
        a = lib.attn_head_keypad(q, k, v, left, right, 13, 0.6)
        b = lib.attn_head_window(q, k, v, left, right, 0.6)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
        c = lib.attn_head_keypad(q, k, v, left, right, 99, 0.6)   # clamped to Lk
        assert np.array_equal(c[0], b[0])


KEYPAD_PINS = [pin_keypad_torch_f64, pin_keypad_uniform, pin_keypad_no_padding_is_window]
PINS.extend(KEYPAD_PINS)


def pin_bwd_masked_finite_differences(lib):
    """Band + key padding gradients equal central differences of the key-padding forward
    (rows without keys have O = 0 and no gradient)."""
    for (Lq, Lk, D, left, right, kv) in [(6, 7, 3, 2, 1, 7), (7, 5, 2, -1, 0, 3), (5, 8, 3, 1, 3, 4),
                                         (6, 6, 2, 0, 0, 2)]:
        q, k, v = _rand((Lq, D), 95 + Lq, 1.5), _rand((Lk, D), 96 + Lk, 1.5), _rand((Lk, D), 97)
        g = _rand((Lq, D), 98)
        dq, dk, dv = lib.attn_bwd_head_masked(q, k, v, g, left, right, kv, 0.7)

        def loss(**kw):
            a = dict(q=q, k=k, v=v)
            a.update(kw)
            return float((lib.attn_head_keypad(a["q"], a["k"], a["v"], left, right, kv, 0.7)[0] * g).sum())
        for name, x, got in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            fd = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += 1e-6
                xm[idx] -= 1e-6
                fd[idx] = (loss(**{name: xp}) - loss(**{name: xm})) / 2e-6
            np.testing.assert_allclose(got, fd, rtol=0, atol=1e-7)


def pin_bwd_rows_masked_match_full_head(lib):
    """The row-sampled backward under band and key padding equals the masked full-head
    backward at the sampled rows (rows without keys included: dQ = 0, LSE = -inf,
    Delta = 0), and Delta_i = dO_i . O_i with the masked forward's O."""
    for n, (Lq, Lk, left, right, kv) in enumerate(KEYPAD_CASES):
        D = 4
        q, k, v, g = (_rand(sh, 140 + 7 * n + i) for i, sh in enumerate(((Lq, D), (Lk, D), (Lk, D), (Lq, D))))
        qr, kr = list(range(Lq)), list(range(Lk))
        dq, dk, dv, lse, delta = lib.attn_bwd_rows_masked(q, k, v, g, left, right, kv, 0.8, qr, kr)
        fq, fk, fv = lib.attn_bwd_head_masked(q, k, v, g, left, right, kv, 0.8)
        for got, ref in ((dq, fq), (dk, fk), (dv, fv)):
            np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
        o, l = lib.attn_head_keypad(q, k, v, left, right, kv, 0.8)
        assert np.array_equal(np.isinf(lse), np.isinf(l))
        np.testing.assert_allclose(lse[np.isfinite(l)], l[np.isfinite(l)], rtol=0, atol=1e-12)
        np.testing.assert_allclose(delta, (g * o).sum(axis=1), rtol=0, atol=1e-12)


def pin_bwd_masked_reduces_to_causal_and_full(lib):
    q, k, v, g = _rand((9, 4), 99), _rand((11, 4), 100), _rand((11, 4), 101), _rand((9, 4), 102)
    for causal, (left, right) in ((False, (-1, -1)), (True, (-1, 0))):
        a = lib.attn_bwd_head(q, k, v, g, causal, 0.8)
        b = lib.attn_bwd_head_masked(q, k, v, g, left, right, 11, 0.8)
        for x, y in zip(a, b):
            np.testing.assert_allclose(x, y, rtol=0, atol=1e-13)


BWD_PINS.extend([pin_bwd_masked_finite_differences, pin_bwd_masked_reduces_to_causal_and_full,
                 pin_bwd_rows_masked_match_full_head])
PINS.extend([pin_bwd_masked_finite_differences, pin_bwd_masked_reduces_to_causal_and_full,
             pin_bwd_rows_masked_match_full_head])


def test_window_rejects_empty_rows(oracle_mod):
    q, k, v = _rand((5, 4), 1), _rand((3, 4), 2), _rand((3, 4), 3)
    with pytest.raises(ValueError):   # row 4 would need key 4 >= Lk
        oracle_mod.attn_head_window(q, k, v, 0, 0, 1.0)


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pin(oracle_mod, pin):
    pin(oracle_mod._get())


def test_bad_arguments_rejected(oracle_mod):
    q, k, v = _rand((3, 4), 1), _rand((2, 4), 2), _rand((2, 4), 3)
    with pytest.raises(ValueError):
        oracle_mod.attn_head(q, k, v, False, 1.0, rows=[3])
    with pytest.raises(ValueError):
        oracle_mod.attn_head(q, k[:0], v[:0], False, 1.0)


# --------------------------------------------------------------------------
# Planted mistakes: each textual mutation of the oracle source must make at
# least one pin fail.  The mutated copies are built in a temporary directory.
# --------------------------------------------------------------------------

MUTATIONS = {
    "dropped_scale": ("S[j] = scale * dot;", "S[j] = dot;"),
    "max_sign_flip": ("P[j] = exp(S[j] - m);", "P[j] = exp(S[j] + m);"),
    "diagonal_excluded": ("return (i + 1 < Lk) ? (i + 1) : Lk;", "return (i < Lk) ? i : Lk;"),
    "keys_as_values": ("o[d] += w * V[j * D + d];", "o[d] += w * K[j * D + d];"),
    "reversed_feature_index": ("dot += q[d] * K[j * D + d];", "dot += q[d] * K[j * D + (D - 1 - d)];"),
    "lse_missing_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "no_normalisation": ("for (long j = 0; j < n_allowed; ++j) P[j] /= l;", ";"),
    "causal_ignored": ("if (!causal) return Lk;", "return Lk;"),
    "window_drops_last_key": ("double *p_row = P ? P + r * Lk : NULL;\n                attend_row(Q + i * D, K + lo * D, V + lo * D, hi - lo + 1, D, hi - lo + 1, scale,",
                              "double *p_row = P ? P + r * Lk : NULL;\n                attend_row(Q + i * D, K + lo * D, V + lo * D, hi - lo, D, hi - lo, scale,"),
    "keypad_empty_row_not_zeroed": ("for (long d = 0; d < D; ++d) O[r * D + d] = 0.0;\n                    LSE[r] = -INFINITY;",
                                    "for (long d = 0; d < D; ++d) O[r * D + d] = 0.0;\n                    LSE[r] = 0.0;"),
    "bwd_softmax_jacobian_without_row_term": ("ds[j] = p[j] * (ds[j] - pdp);", "ds[j] = p[j] * ds[j];", 0),
    "bwd_dk_missing_scale": ("dK[j * D + d] = scale * ak;", "dK[j * D + d] = ak;", 0),
    "bwd_dv_from_queries": ("av += P[i * Lk + j] * dO[i * D + d];", "av += P[i * Lk + j] * Q[i * D + d];", 0),
    "bwd_masked_jacobian_without_row_term": ("ds[j] = p[j] * (ds[j] - pdp);", "ds[j] = p[j] * ds[j];", 1),
    "bwd_masked_dk_missing_scale": ("dK[j * D + d] = scale * ak;", "dK[j * D + d] = ak;", 1),
    "bwd_masked_padding_ignored": ("if (hi > kv - 1) hi = kv - 1;", ";", 1),
    "keypad_last_key_kept": ("if (hi > kv - 1) hi = kv - 1;", "if (hi > kv) hi = kv;", 0),
    "bwd_rows_dq_without_row_term": ("const double ds = p * (dp - delta[i]);", "const double ds = p * dp;", 0),
    "bwd_rows_dk_without_row_term": ("const double ds = p * (dp - delta[i]);", "const double ds = p * dp;", 1),
    "bwd_rows_dk_missing_scale": ("for (long d = 0; d < D; ++d) ok[d] *= scale;", ";"),
    "bwd_rows_dv_from_queries": ("ov[d] += p * dO[i * D + d];", "ov[d] += p * Q[i * D + d];"),
    "bwd_rows_delta_unnormalised": ("pdp += exp(srow[j] - lse_i) * dot;", "pdp += exp(srow[j] - m) * dot;"),
    "bwd_rows_padding_ignored": ("if (h > kv - 1) h = kv - 1;", ";"),
    "window_shifted_values": ("double *p_row = P ? P + r * Lk : NULL;\n                attend_row(Q + i * D, K + lo * D, V + lo * D,",
                              "double *p_row = P ? P + r * Lk : NULL;\n                attend_row(Q + i * D, K + lo * D, V + (lo > 0 ? lo - 1 : 0) * D,"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    src = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")
    text = open(src).read()
    old, new, *which = MUTATIONS[name]
    which = which[0] if which else None   # occurrence to mutate when the text repeats
    if which is None:
        assert text.count(old) == 1, f"mutation anchor for {name} not found exactly once"
        at = text.index(old)
    else:
        at = -1
        for _ in range(which + 1):
            at = text.index(old, at + 1)
    mutated = tmp_path / f"oracle_{name}.c"
    mutated.write_text(text[:at] + new + text[at + len(old):])
    lib = oracle.OracleLib(oracle.build(force=True, src=str(mutated),
                                        out=str(tmp_path / f"lib_{name}.so")))
    failures = 0
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(lib)
        except (AssertionError, ValueError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake {name}"
    shutil.rmtree(tmp_path, ignore_errors=True)
