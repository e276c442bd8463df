"""The split-key schedule's step space, checked on the host.

The forward kernel, its merge kernel and the host planner each walk the same step space:
units (pairs of 128-row query tiles) head after head, each taking `cost` virtual steps and
then its key-tile steps, and CTA g taking the steps [T g / G, T (g + 1) / G).  A part is the
intersection of a CTA's range with a unit's key-tile steps, numbered per CTA; a cut part
parks its rows in slot 2 g (the CTA's first part) or 2 g + 1 (its last); and the merge
kernel's boundary b finishes a unit when it is the first boundary that cuts the unit's key
tiles.  This file restates those rules (`pair_steps`, `head_prefix`, `split_locate`, the
split branch of `unit_of`, `split_max_parts` and `fa_combine_kernel` in csrc/fa_fwd.cu) and
checks, for costs 0-5, that every unit's key tiles are covered exactly once, that only cut
units have cut parts, and that each cut unit is merged by exactly one boundary which lists
exactly its parts' slots.  The kernels' results on these schedules are checked on the GPU
(test_causal_split_gpu.py, test_sweep_gpu.py, test_parity_gpu.py).
"""
import random

import pytest


def pair_steps(pair, nkv, Lq, causal):
    if not causal:
        return nkv
    last = 2 * pair + 2 if pair * 256 + 128 < Lq else 2 * pair + 1
    return min(last, nkv)


def head_prefix(P, nkv, Lq, n_pairs, causal, cost):
    virt = P * cost
    if not causal:
        return P * nkv + virt
    c = nkv // 2
    s = P * (P + 1) if P <= c else c * (c + 1) + (P - c) * nkv
    if P == n_pairs and n_pairs > 0:
        full = min(2 * (n_pairs - 1) + 2, nkv)
        s -= full - pair_steps(n_pairs - 1, nkv, Lq, causal)
    return s + virt


def locate(x, nkv, Lq, n_pairs, causal, cost):
    per = head_prefix(n_pairs, nkv, Lq, n_pairs, causal, cost)
    h, xh = divmod(x, per)
    lo, hi = 0, n_pairs - 1
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if head_prefix(mid, nkv, Lq, n_pairs, causal, cost) <= xh:
            lo = mid
        else:
            hi = mid - 1
    return h, lo, h * per + head_prefix(lo, nkv, Lq, n_pairs, causal, cost), pair_steps(lo, nkv, Lq, causal)


def check(bh, Lq, Lk, causal, cost, sm=152):
    nkv, n_pairs = (Lk + 127) // 128, (Lq + 255) // 256
    G = min(bh * head_prefix(n_pairs, nkv, Lq, n_pairs, causal, 0), sm)
    T = bh * head_prefix(n_pairs, nkv, Lq, n_pairs, causal, cost)
    lo = lambda g: T * g // G
    parts = {}
    most = 0
    for g in range(G):
        a, b, x, k = lo(g), lo(g + 1), lo(g), 0
        while x < b:
            h, pair, start, steps = locate(x, nkv, Lq, n_pairs, causal, cost)
            ks, ke = start + cost, start + cost + steps
            ra, rb = max(x, ks), min(ke, b)
            if ra < rb:
                cut = (rb - ra) != steps
                parts.setdefault((h, pair), []).append((ra, rb, (2 * g + (k > 0)) if cut else None, cut, ks, ke))
                k += 1
            x = min(ke, b)
        most = max(most, k)
    owners = {}
    for b in range(1, G):
        xb = lo(b)
        h, pair, start, steps = locate(xb, nkv, Lq, n_pairs, causal, cost)
        ks, ke = start + cost, start + cost + steps
        if xb > ks and not (b >= 2 and lo(b - 1) > ks):
            g, slots = b - 1, []
            while g < G and lo(g) < ke:
                slots.append(2 * g + (0 if lo(g) >= start else 1))
                g += 1
            assert (h, pair) not in owners, "a unit with two merging boundaries"
            owners[(h, pair)] = sorted(slots)
    for h in range(bh):
        for pair in range(n_pairs):
            ps = sorted(parts.get((h, pair), []))
            assert ps, "a unit with no part"
            assert ps[0][0] == ps[0][4] and ps[-1][1] == ps[-1][5], "key tiles not covered to the ends"
            assert all(u[1] == v[0] for u, v in zip(ps, ps[1:])), "key tiles covered twice or not at all"
            if len(ps) == 1:
                assert not ps[0][3] and (h, pair) not in owners
            else:
                assert all(p[3] for p in ps)
                assert owners.get((h, pair)) == sorted(p[2] for p in ps), "merge slots differ from the parts"
    return most


SHAPES = [(1, 16384, 16384, 1), (2, 16384, 16384, 1), (4, 8192, 8192, 1), (1, 32768, 32768, 1),
          (4, 2048, 32768, 0), (2, 4096, 65536, 0), (1, 3900, 3900, 1), (1, 2400, 5000, 1),
          (1, 5000, 2500, 1), (3, 700, 1300, 0), (1, 128, 40000, 0)]
_rng = random.Random(7)
SHAPES += [(_rng.randint(1, 6), _rng.randint(1, 9000), _rng.randint(1, 9000), _rng.randint(0, 1))
           for _ in range(12)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("cost", [0, 3, 5])
def test_split_step_space(shape, cost):
    assert check(*shape, cost=cost) <= 24   # the kernel's per-CTA part list holds 24
