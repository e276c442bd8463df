"""Failure detection without a GPU fault.

The load warp can be told (test hook) to withhold the first value-tile load.
The MMA warp's bounded wait then runs out, the kernel records FA_ERR_TIMEOUT
in the library's status word, every role stops and frees its resources, and
the host reads the status.  A normal call afterwards must still be exact, so
the context stays usable.  A second hook makes the host report a launch
failure without launching.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_60_gb300 as fa
from exact_attention_60_gb300.workloads import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture
def restore_hooks():
    yield
    fa.fa_debug_set(0, 0)


@pytest.mark.parametrize("D,causal", [(64, False), (128, True)])
def test_withheld_load_times_out_and_context_survives(oracle_mod, restore_hooks, D, causal):
    dev = torch.device("cuda:0")
    q, k, v = make_qkv(1, 2, 384, 512, D, seed=21)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    assert fa.fa_last_device_status() == fa.FA_OK
    fa.fa_debug_set(1, 20_000_000)   # withhold V_0; 20 ms per wait
    fa.attention(qd, kd, vd, causal=causal)
    assert fa.fa_last_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_last_device_status() == fa.FA_OK   # reading clears the word
    fa.fa_debug_set(0, 0)
    o, lse = fa.attention(qd, kd, vd, causal=causal)
    assert fa.fa_last_device_status() == fa.FA_OK
    ref_o, ref_l = oracle_mod.attn_full(q, k, v, causal, 1.0 / math.sqrt(D))
    assert np.abs(o.float().cpu().numpy() - ref_o).max() <= 2e-2
    assert np.abs(lse.cpu().numpy() - ref_l).max() <= 1e-3


def test_simulated_launch_failure(restore_hooks):
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(1, 1, 128, 128, 64, seed=22))
    o = torch.full_like(q, 7.0)
    lse = torch.full((1, 1, 128), 7.0, device=dev)
    fa.fa_debug_set(2, 0)
    st = fa.fa_fwd(q, k, v, o, lse, 1, 1, 128, 128, 64, 0, 0.125)
    assert st == fa.FA_ERR_CUDA
    torch.cuda.synchronize()
    assert (o.float() == 7.0).all() and (lse == 7.0).all()


def test_backward_withheld_load_times_out_and_context_survives(oracle_mod, restore_hooks):
    """The dK/dV kernel's first V tile is withheld: its waits run out, the status word says
    FA_ERR_TIMEOUT, and the next backward is exact again."""
    dev = torch.device("cuda:0")
    q, k, v = make_qkv(1, 2, 300, 300, 128, seed=23)
    g = torch.Generator().manual_seed(5)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.attention(qd, kd, vd, causal=True)
    assert fa.fa_last_device_status() == fa.FA_OK
    fa.fa_debug_set(1, 20_000_000)
    fa.attention_backward(qd, kd, vd, o, lse, dod, causal=True)
    assert fa.fa_last_device_status() == fa.FA_ERR_TIMEOUT
    fa.fa_debug_set(0, 0)
    dq, dk, dv = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=True)
    assert fa.fa_last_device_status() == fa.FA_OK
    ref = oracle_mod.attn_bwd_head(q[0, 1].double().numpy(), k[0, 1].double().numpy(),
                                   v[0, 1].double().numpy(), do[0, 1].double().numpy(), True, 128 ** -0.5)
    for got, r in zip((dq, dk, dv), ref):
        assert np.abs(got[0, 1].float().cpu().numpy() - r).max() < 5e-2


def test_backward_simulated_launch_failure(restore_hooks):
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(1, 1, 128, 128, 64, seed=24))
    o, lse = fa.attention(q, k, v)
    fa.fa_debug_set(2, 0)
    with pytest.raises(fa.FaError) as e:
        fa.attention_backward(q, k, v, o, lse, torch.randn_like(q))
    assert e.value.status == fa.FA_ERR_CUDA
