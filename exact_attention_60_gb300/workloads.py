"""Seeded synthetic workloads: shapes, input generators, row samples, work counts.

This module holds no attention arithmetic.  It is the one module that both the
CUDA path (tests, benchmark) and the fp64 oracle's callers draw inputs from, so
the two sides always see the same bits.

The first five workloads are the ones the method is measured on: a tiny head
pair, a 1K-token D=64 batch (non-causal and causal), a 4K-token and a 16K-token
causal D=128 batch, and a ragged cross-attention case whose query/key
logits are scaled up (standard deviation 3) to stress the softmax.  Two more
exercise local (sliding-window) attention: 16K tokens with a causal window of
4096 keys, and 4K tokens with a symmetric band of 256 keys on each side.  Inputs
are i.i.d. normal draws rounded to bf16, contiguous ``[B, H, L, D]``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Lq: int
    Lk: int
    D: int
    causal: bool
    sigma_qk: float = 1.0   # standard deviation of Q and K draws
    sigma_v: float = 1.0    # standard deviation of V draws
    index: int = 0          # position in the workload list (fixes the seed)
    window: tuple | None = None   # (left, right): keys i-left <= j <= i+right (-1: unbounded)

    @property
    def scale(self) -> float:
        """1/sqrt(D), the scale every workload uses."""
        return 1.0 / math.sqrt(self.D)

    @property
    def seed(self) -> int:
        return 1234 + self.index

    def key_range(self, i: int):
        """First and last allowed key of query row i."""
        if self.window is not None:
            left, right = self.window
            lo = 0 if left < 0 else max(0, i - left)
            hi = self.Lk - 1 if right < 0 else min(self.Lk - 1, i + right)
            return lo, hi
        return 0, (min(i, self.Lk - 1) if self.causal else self.Lk - 1)

    def pairs_per_head(self) -> int:
        """Unmasked (query, key) pairs of one head."""
        if self.window is not None:
            i = np.arange(self.Lq, dtype=np.int64)
            left, right = self.window
            lo = np.zeros_like(i) if left < 0 else np.maximum(0, i - left)
            hi = np.full_like(i, self.Lk - 1) if right < 0 else np.minimum(self.Lk - 1, i + right)
            return int(np.sum(hi - lo + 1))
        if not self.causal:
            return self.Lq * self.Lk
        # top-left aligned causal: row i keeps keys 0..min(i, Lk-1)
        n = min(self.Lq, self.Lk)
        full = n * (n + 1) // 2
        return full + max(0, self.Lq - self.Lk) * self.Lk

    def flops(self) -> int:
        """4 * D flops per unmasked pair (two GEMMs, forward only)."""
        return 4 * self.D * self.B * self.H * self.pairs_per_head()

    def algorithmic_bytes(self) -> int:
        """Q, K, V read once, O written once (bf16), LSE written once (fp32)."""
        bh = self.B * self.H
        return 2 * bh * self.D * (2 * self.Lq + 2 * self.Lk) + 4 * bh * self.Lq

    def describe(self) -> str:
        kind = "causal" if self.causal else "non-causal"
        if self.window is not None:
            kind = f"window=({self.window[0]},{self.window[1]})"
        return (f"B={self.B},H={self.H},Lq={self.Lq},Lk={self.Lk},D={self.D},{kind},"
                f"sigma_qk={self.sigma_qk:g},sigma_v={self.sigma_v:g}")


WORKLOADS = {
    "tiny_d64": Workload("tiny_d64", 1, 2, 128, 128, 64, False, index=0),
    "seq1k_d64": Workload("seq1k_d64", 4, 16, 1024, 1024, 64, False, index=1),
    "seq1k_d64_causal": Workload("seq1k_d64_causal", 4, 16, 1024, 1024, 64, True, index=1),
    "seq4k_d128_causal": Workload("seq4k_d128_causal", 2, 32, 4096, 4096, 128, True, index=2),
    "seq16k_d128_causal": Workload("seq16k_d128_causal", 1, 16, 16384, 16384, 128, True, index=3),
    "cross_q500_k8191_d128": Workload("cross_q500_k8191_d128", 8, 16, 500, 8191, 128, False,
                                      sigma_qk=3.0, sigma_v=1.0, index=4),
    "seq16k_d128_window4k": Workload("seq16k_d128_window4k", 1, 16, 16384, 16384, 128, False,
                                     index=5, window=(4095, 0)),
    "seq4k_d64_local256": Workload("seq4k_d64_local256", 2, 16, 4096, 4096, 64, False,
                                   index=6, window=(256, 256)),
    # one causal head of 16K tokens: too few units for whole units to fill the GPU, so
    # fa_fwd_ws cuts key ranges across CTAs (the split-key schedule)
    "seq16k_d128_causal_h1": Workload("seq16k_d128_causal_h1", 1, 1, 16384, 16384, 128, True,
                                      index=7),
}


def make_qkv(B, H, Lq, Lk, D, seed, sigma_qk=1.0, sigma_v=1.0):
    """Seeded bf16 Q, K, V on the CPU, contiguous [B, H, L, D].

    One torch CPU generator, seeded once, draws Q, then K, then V as
    ``randn * sigma`` in fp32, each rounded to bf16 (round to nearest even).
    """
    g = torch.Generator().manual_seed(int(seed))

    def draw(L, sigma):
        x = torch.randn((B, H, L, D), generator=g, dtype=torch.float32)
        if sigma != 1.0:
            x.mul_(float(sigma))
        return x.to(torch.bfloat16)

    q = draw(Lq, sigma_qk)
    k = draw(Lk, sigma_qk)
    v = draw(Lk, sigma_v)
    return q, k, v


def make_workload_inputs(w: Workload):
    return make_qkv(w.B, w.H, w.Lq, w.Lk, w.D, w.seed, w.sigma_qk, w.sigma_v)


def sample_rows(w: Workload, n_random: int = 512, extra_rows=()):
    """Seeded sample of (bh, i) query rows, plus forced rows at tile edges.

    Returns a sorted int64 array of unique pairs, shape [n, 2].  The forced rows
    are rows 0, 1, 127, 128, 129 and Lq-1 of the first and last (batch, head),
    plus ``extra_rows`` of those two heads, clipped to [0, Lq).
    """
    rng = np.random.default_rng(0x5EED + w.index)
    BH = w.B * w.H
    bh = rng.integers(0, BH, size=n_random)
    ii = rng.integers(0, w.Lq, size=n_random)
    pairs = set(zip(bh.tolist(), ii.tolist()))
    forced = [0, 1, 127, 128, 129, w.Lq - 1, *extra_rows]
    for h in {0, BH - 1}:
        for i in forced:
            if 0 <= i < w.Lq:
                pairs.add((h, i))
    return np.array(sorted(pairs), dtype=np.int64).reshape(-1, 2)
