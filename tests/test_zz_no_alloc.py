"""fa_fwd_noalloc: the forward pass for callers that cannot allocate device memory.

Some callers cannot get device memory when they call attention: a plugin that is
handed only its input and output pointers through a fixed interface, with no
allocator behind it, or a latency-critical path that must not call cudaMalloc
because it can synchronize the device.  fa_fwd_noalloc serves them with scratch
memory built into the library instead of a caller-provided workspace.

Each test calls it through the C ABI twice in a row (the second call finds the
scratch as the first call left it) and compares the results with the existing
entry points -- fa_fwd_ws given its own workspace, or fa_fwd when no scratch is
involved.  The results must lie within the tolerances of the other parity tests
and, since both calls run the same kernels on the same schedule and inputs, be
bit-identical: a stale or partly overwritten scratch slot would show there.  One
test also checks the property the entry point exists for: a call changes the
device's free memory by nothing.  The file is named so that pytest collects it
after every other test file.
"""
import math

import pytest
import torch

import exact_attention_60_gb300 as fa
from exact_attention_60_gb300.workloads import make_qkv

pytestmark = pytest.mark.gpu

TOL_O = 2e-2
TOL_LSE = 1e-3


def _buffers(B, H, Lq, Lk, D, seed):
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(B, H, Lq, Lk, D, seed=seed))
    return q, k, v, torch.empty_like(q), torch.empty(B, H, Lq, device=dev)


@pytest.mark.parametrize("B,H,Lq,Lk,D", [(1, 4, 2048, 32768, 128), (2, 3, 500, 8191, 64),
                                          (1, 1, 128, 40000, 128)])
def test_noalloc_matches_workspace_entry_point(B, H, Lq, Lk, D):
    """Shapes that take the split-key schedule, i.e. that use scratch memory."""
    st, nbytes = fa.fa_fwd_workspace_size(B, H, Lq, Lk, D, False)
    assert st == fa.FA_OK and nbytes > 0
    q, k, v, o_ref, l_ref = _buffers(B, H, Lq, Lk, D, seed=Lq + Lk)
    scale = 1.0 / math.sqrt(D)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    assert fa.fa_fwd_ws(q, k, v, o_ref, l_ref, B, H, Lq, Lk, D, 0, scale, ws, nbytes) == fa.FA_OK
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(l_ref, float("nan"))
        assert fa.fa_fwd_noalloc(q, k, v, o, lse, B, H, Lq, Lk, D, 0, scale) == fa.FA_OK
        assert fa.fa_last_device_status() == fa.FA_OK
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        assert (o.float() - o_ref.float()).abs().max().item() <= TOL_O
        assert (lse - l_ref).abs().max().item() <= TOL_LSE
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_noalloc_call_allocates_no_device_memory():
    """After a first call (which looks up the scratch address), a call on a split
    shape leaves the device's free memory exactly as it was."""
    B, H, Lq, Lk, D = 1, 4, 2048, 32768, 128
    # The workspace it replaces: 2 slots x 2 tiles x 128 rows per CTA (one CTA per SM
    # here) of D partial-O floats, then (m, l) per row, each rounded up to 256 bytes.
    rows = torch.cuda.get_device_properties(0).multi_processor_count * 2 * 2 * 128
    r256 = lambda x: (x + 255) & ~255
    assert fa.fa_fwd_workspace_size(B, H, Lq, Lk, D, False) == (
        fa.FA_OK, r256(rows * D * 4) + r256(rows * 2 * 4))
    q, k, v, o, lse = _buffers(B, H, Lq, Lk, D, seed=3)
    scale = 1.0 / math.sqrt(D)
    assert fa.fa_fwd_noalloc(q, k, v, o, lse, B, H, Lq, Lk, D, 0, scale) == fa.FA_OK
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    assert fa.fa_fwd_noalloc(q, k, v, o, lse, B, H, Lq, Lk, D, 0, scale) == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert fa.fa_last_device_status() == fa.FA_OK


def test_noalloc_causal_split_matches_workspace_entry_point():
    """A causal problem of one long head also takes the split schedule, and its scratch."""
    B, H, Lq, Lk, D = 1, 1, 16384, 16384, 128
    st, nbytes = fa.fa_fwd_workspace_size(B, H, Lq, Lk, D, True)
    assert st == fa.FA_OK and nbytes > 0
    q, k, v, o_ref, l_ref = _buffers(B, H, Lq, Lk, D, seed=23)
    scale = 1.0 / math.sqrt(D)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    assert fa.fa_fwd_ws(q, k, v, o_ref, l_ref, B, H, Lq, Lk, D, 1, scale, ws, nbytes) == fa.FA_OK
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(l_ref, float("nan"))
        assert fa.fa_fwd_noalloc(q, k, v, o, lse, B, H, Lq, Lk, D, 1, scale) == fa.FA_OK
        assert fa.fa_last_device_status() == fa.FA_OK
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_noalloc_without_scratch_matches_fa_fwd():
    """A causal shape runs on whole units and needs no scratch."""
    B, H, Lq, Lk, D = 2, 4, 700, 700, 128
    assert fa.fa_fwd_workspace_size(B, H, Lq, Lk, D, True) == (fa.FA_OK, 0)
    q, k, v, o_ref, l_ref = _buffers(B, H, Lq, Lk, D, seed=5)
    scale = 1.0 / math.sqrt(D)
    assert fa.fa_fwd(q, k, v, o_ref, l_ref, B, H, Lq, Lk, D, 1, scale) == fa.FA_OK
    for _ in range(2):
        o = torch.empty_like(o_ref)
        lse = torch.empty_like(l_ref)
        assert fa.fa_fwd_noalloc(q, k, v, o, lse, B, H, Lq, Lk, D, 1, scale) == fa.FA_OK
        assert fa.fa_last_device_status() == fa.FA_OK
        assert (o.float() - o_ref.float()).abs().max().item() <= TOL_O
        assert (lse - l_ref).abs().max().item() <= TOL_LSE
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_noalloc_rejects_bad_arguments():
    q, k, v, o, lse = _buffers(1, 1, 16, 16, 64, seed=1)
    assert fa.fa_fwd_noalloc(q, k, v, o, lse, 1, 1, 16, 16, 96, 0, 0.1) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_noalloc(q, k, v, o, lse, 1, 1, 16, 0, 64, 0, 0.1) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_noalloc(None, k, v, o, lse, 1, 1, 16, 16, 64, 0, 0.1) == fa.FA_ERR_INVALID_ARG
