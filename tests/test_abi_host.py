"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the GPU.

No test here launches a kernel, so the file runs on a machine without a GPU.
Only argument errors that the library rejects before any CUDA call are used.
"""
import ctypes
import os
import re
import subprocess

import pytest

import exact_attention_60_gb300 as fa
from exact_attention_60_gb300 import _native
from exact_attention_60_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return _native.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    return set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\*?\s+\*?(fa_[a-z_]+)\s*\(", text, re.M))


def test_header_declares_the_binding_names():
    assert header_functions() == set(_native.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", fa_build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (fa_\w+)$", out, re.M))
    assert header_functions() <= exported


def test_status_strings(lib):
    for code in range(5):
        s = fa.fa_status_string(code)
        assert s.startswith("FA_"), s
    assert "unknown" in fa.fa_status_string(99)


# Every case below is rejected by argument checks that run before any CUDA call.
ALIGNED = 1 << 20   # a non-null, 16-byte aligned dummy address (never dereferenced)


def call(Q=ALIGNED, K=2 * ALIGNED, V=3 * ALIGNED, O=4 * ALIGNED, LSE=5 * ALIGNED, B=1, H=1,
         Lq=16, Lk=16, D=64, causal=0, scale=0.125):
    return fa.fa_fwd(Q, K, V, O, LSE, B, H, Lq, Lk, D, causal, scale, 0)


@pytest.mark.parametrize("kw,expect", [
    (dict(D=96), fa.FA_ERR_UNSUPPORTED),
    (dict(D=256), fa.FA_ERR_UNSUPPORTED),
    (dict(D=0), fa.FA_ERR_INVALID_ARG),
    (dict(B=-1), fa.FA_ERR_INVALID_ARG),
    (dict(H=-2), fa.FA_ERR_INVALID_ARG),
    (dict(Lq=-1), fa.FA_ERR_INVALID_ARG),
    (dict(Lk=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-0.5), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(Q=0), fa.FA_ERR_INVALID_ARG),
    (dict(LSE=0), fa.FA_ERR_INVALID_ARG),
    (dict(K=2 * ALIGNED + 8), fa.FA_ERR_INVALID_ARG),
    (dict(O=4 * ALIGNED + 2), fa.FA_ERR_INVALID_ARG),
    (dict(O=ALIGNED), fa.FA_ERR_INVALID_ARG),                  # O overlaps Q
    (dict(LSE=4 * ALIGNED + 64), fa.FA_ERR_INVALID_ARG),       # LSE inside O
    (dict(O=3 * ALIGNED + 1024), fa.FA_ERR_INVALID_ARG),       # O inside V
])
def test_bad_arguments_rejected(lib, kw, expect):
    assert call(**kw) == expect


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0), dict(Lq=0),
                                dict(B=0, Q=0, K=0, V=0, O=0, LSE=0),
                                dict(Lq=0, Lk=0)])
def test_empty_problem_is_ok_without_launch(lib, kw):
    assert call(**kw) == fa.FA_OK


def test_binding_is_argument_marshalling_only():
    """The binding module holds no attention arithmetic and imports no oracle."""
    src = open(_native.__file__).read() + open(fa.__file__).read()
    assert "oracle" not in src
    code = "\n".join(line for line in src.splitlines() if not line.strip().startswith("@"))  # decorators
    for word in ("softmax", "exp(", "exp2", "matmul", "einsum", "@"):
        assert word not in code, word


def test_missing_library_fails_loudly(tmp_path):
    missing = str(tmp_path / "libfa_missing.so")
    saved = _native._lib
    _native._lib = None
    try:
        with pytest.raises(RuntimeError):
            _native.load(missing)
    finally:
        _native._lib = saved


def test_workspace_size_rejects_bad_arguments(lib):
    assert fa.fa_fwd_workspace_size(1, 1, 16, 16, 96, 0)[0] == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_workspace_size(-1, 1, 16, 16, 64, 0)[0] == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_workspace_size(1, 1, 16, 0, 64, 0)[0] == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_workspace_size(0, 1, 16, 16, 64, 0) == (fa.FA_OK, 0)
    assert lib.fa_fwd_workspace_size(1, 1, 16, 16, 64, 0, None) == fa.FA_ERR_INVALID_ARG


def test_schedule_query_rejects_bad_arguments(lib):
    assert fa.fa_fwd_schedule(1, 1, 16, 16, 96, 1)[0] == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_schedule(1, -1, 16, 16, 64, 1)[0] == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_schedule(1, 1, 16, 0, 64, 1)[0] == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_schedule(2, 3, 0, 16, 128, 1) == (fa.FA_OK, fa.FA_SCHED_WHOLE)
    assert lib.fa_fwd_schedule(1, 1, 16, 16, 64, 0, None) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,expect", [(dict(D=96), fa.FA_ERR_UNSUPPORTED), (dict(Lk=0), fa.FA_ERR_INVALID_ARG),
                                       (dict(Q=0), fa.FA_ERR_INVALID_ARG), (dict(scale=0.0), fa.FA_ERR_INVALID_ARG)])
def test_fwd_ws_rejects_bad_arguments_before_any_cuda_call(lib, kw, expect):
    args = dict(Q=ALIGNED, K=2 * ALIGNED, V=3 * ALIGNED, O=4 * ALIGNED, LSE=5 * ALIGNED, B=1, H=1,
                Lq=16, Lk=16, D=64, causal=0, scale=0.125)
    args.update(kw)
    assert fa.fa_fwd_ws(args["Q"], args["K"], args["V"], args["O"], args["LSE"], args["B"],
                        args["H"], args["Lq"], args["Lk"], args["D"], args["causal"],
                        args["scale"], None, 0, 0) == expect


def call_window(left, right, Lq=16, Lk=16, **kw):
    args = dict(Q=ALIGNED, K=2 * ALIGNED, V=3 * ALIGNED, O=4 * ALIGNED, LSE=5 * ALIGNED, B=1, H=1,
                D=64, scale=0.125)
    args.update(kw)
    return fa.fa_fwd_window(args["Q"], args["K"], args["V"], args["O"], args["LSE"], args["B"],
                            args["H"], Lq, Lk, args["D"], left, right, args["scale"], 0)


@pytest.mark.parametrize("left,right,Lq,Lk,kw,expect", [
    (-2, 0, 16, 16, {}, fa.FA_ERR_INVALID_ARG),          # a side below -1
    (3, -5, 16, 16, {}, fa.FA_ERR_INVALID_ARG),
    (0, 0, 17, 16, {}, fa.FA_ERR_INVALID_ARG),           # row 16 would need key 16
    (3, -1, 300, 200, {}, fa.FA_ERR_INVALID_ARG),        # rows 204.. start past the last key
    (4, 4, 16, 16, dict(D=96), fa.FA_ERR_UNSUPPORTED),
    (4, 4, 16, 0, {}, fa.FA_ERR_INVALID_ARG),
    (4, 4, 16, 16, dict(Q=0), fa.FA_ERR_INVALID_ARG),
    (4, 4, 16, 16, dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (4, 4, 16, 16, dict(O=ALIGNED), fa.FA_ERR_INVALID_ARG),
])
def test_fwd_window_rejects_bad_arguments_before_any_cuda_call(lib, left, right, Lq, Lk, kw, expect):
    assert call_window(left, right, Lq, Lk, **kw) == expect


def test_fwd_window_empty_problem_is_ok_without_launch(lib):
    assert call_window(2, 2, Lq=0, Lk=16) == fa.FA_OK
    assert call_window(2, 2, B=0, Q=0, K=0, V=0, O=0, LSE=0) == fa.FA_OK


def test_bwd_rejects_bad_arguments_before_any_cuda_call(lib):
    A = ALIGNED
    def call(**kw):
        a = dict(Q=A, K=2 * A, V=3 * A, O=4 * A, dO=5 * A, LSE=6 * A, dQ=7 * A, dK=8 * A, dV=9 * A,
                 B=1, H=1, Lq=16, Lk=16, D=64, causal=0, scale=0.125, ws=10 * A, wsb=1 << 16)
        a.update(kw)
        return fa.fa_bwd(a["Q"], a["K"], a["V"], a["O"], a["dO"], a["LSE"], a["dQ"], a["dK"], a["dV"],
                         a["B"], a["H"], a["Lq"], a["Lk"], a["D"], a["causal"], a["scale"], a["ws"],
                         a["wsb"], 0)
    assert call(D=96) == fa.FA_ERR_UNSUPPORTED
    assert call(Lk=0) == fa.FA_ERR_INVALID_ARG
    assert call(B=-1) == fa.FA_ERR_INVALID_ARG
    assert call(scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert call(dO=0) == fa.FA_ERR_INVALID_ARG
    assert call(dQ=7 * A + 8) == fa.FA_ERR_INVALID_ARG          # misaligned
    assert call(ws=0) == fa.FA_ERR_INVALID_ARG                  # workspace missing
    assert call(wsb=16) == fa.FA_ERR_INVALID_ARG                # workspace too small
    assert call(wsb=2 * 128 * 4) == fa.FA_ERR_INVALID_ARG       # no room for the work counters
    assert call(ws=10 * A + 16) == fa.FA_ERR_INVALID_ARG        # workspace not 256-byte aligned
    assert call(dK=A) == fa.FA_ERR_INVALID_ARG                  # dK overlaps Q
    assert call(dV=8 * A) == fa.FA_ERR_INVALID_ARG              # dV overlaps dK
    assert call(ws=5 * A) == fa.FA_ERR_INVALID_ARG              # workspace overlaps dO
    assert call(B=0, Lk=0) == fa.FA_OK                           # nothing to do
    st, n = fa.fa_bwd_workspace_size(2, 3, 100, 50, 128, 1)
    # Delta and LSE * log2(e), each over whole 128-row tiles (2*3 heads x 1 tile x 128 rows),
    # then 256 bytes of work counters
    assert st == fa.FA_OK and n == 2 * (2 * 3 * 128 * 4) + 256
    assert fa.fa_bwd_workspace_size(1, 1, 16, 16, 96, 0)[0] == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_bwd_workspace_size(1, 1, 16, 16, 64, 0, None) == fa.FA_ERR_INVALID_ARG


def call_strided(qs=(32768, 2048, 64), ks=(32768, 2048, 64), vs=(32768, 2048, 64),
                 os_=(32768, 2048, 64), dtype=0, **kw):
    a = dict(Q=ALIGNED, K=2 * ALIGNED, V=3 * ALIGNED, O=4 * ALIGNED, LSE=5 * ALIGNED, B=2, H=16,
             Lq=32, Lk=32, D=64, left=-1, right=-1, scale=0.125, ws=None, wsb=0)
    a.update(kw)
    return fa.fa_fwd_strided(a["Q"], qs, a["K"], ks, a["V"], vs, a["O"], os_, a["LSE"], a.get("kv"), a["B"], a["H"],
                             a["Lq"], a["Lk"], a["D"], a["left"], a["right"], a["scale"], dtype,
                             a["ws"], a["wsb"], 0)


@pytest.mark.parametrize("kw,expect", [
    (dict(dtype=2), fa.FA_ERR_INVALID_ARG),                                  # unknown dtype
    (dict(qs=(32768, 2048, 60)), fa.FA_ERR_INVALID_ARG),                     # row stride not 16 bytes
    (dict(ks=(32768, -2048, 64)), fa.FA_ERR_INVALID_ARG),                    # negative stride
    (dict(os_=(32768, 2048, 32)), fa.FA_ERR_INVALID_ARG),                    # O rows overlap (stride < D)
    (dict(os_=(32768, 1024, 64)), fa.FA_ERR_INVALID_ARG),                    # O heads overlap
    (dict(O=ALIGNED + 4096), fa.FA_ERR_INVALID_ARG),                        # O inside Q's span
    (dict(LSE=4 * ALIGNED + 256), fa.FA_ERR_INVALID_ARG),                   # LSE inside O's span
    (dict(left=-3), fa.FA_ERR_INVALID_ARG),
    (dict(left=0, right=0, Lq=40, Lk=32), fa.FA_ERR_INVALID_ARG),           # rows without keys
    (dict(D=96), fa.FA_ERR_UNSUPPORTED),
    (dict(Q=ALIGNED + 8), fa.FA_ERR_INVALID_ARG),                           # misaligned
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(kv=6 * ALIGNED + 2), fa.FA_ERR_INVALID_ARG),                      # kv_len misaligned
])
def test_fwd_strided_rejects_bad_arguments_before_any_cuda_call(lib, kw, expect):
    assert call_strided(**kw) == expect


def test_fwd_strided_accepts_shared_inputs_and_empty(lib):
    # empty problems need no pointers
    assert fa.fa_fwd_strided(None, None, None, None, None, None, None, None, None, None, 0, 4, 16, 16,
                             64, -1, -1, 0.125, 0, None, 0, 0) == fa.FA_OK
    # a missing stride array with work to do is an argument error
    assert call_strided(qs=None) == fa.FA_ERR_INVALID_ARG


def split_workspace_bytes(grid: int, D: int) -> int:
    """The split schedule's workspace as fa_fwd_workspace_size documents it: 2 slots x
    2 query tiles x 128 rows per CTA of D partial-O floats, then (m, l) per row, each
    array rounded up to 256 bytes."""
    r256 = lambda x: (x + 255) & ~255
    rows = grid * 2 * 2 * 128
    return r256(rows * D * 4) + r256(rows * 2 * 4)


def test_noalloc_documented_limits_follow_from_the_scratch_size():
    """The largest grid whose split workspace fits fa_fwd_noalloc's built-in scratch,
    for each head dimension, is the SM count that the header and the source state."""
    src = open(os.path.join(ROOT, "exact_attention_60_gb300", "csrc", "fa_fwd.cu")).read()
    m = re.search(r"kNoAllocScratchBytes = (\d+)ull << (\d+);", src)
    assert m, "scratch size constant not found"
    cap = int(m.group(1)) << int(m.group(2))
    limits = {}
    for D in (128, 64):
        g = 1
        while split_workspace_bytes(g + 1, D) <= cap:
            g += 1
        limits[D] = g
    header = open(os.path.join(ROOT, "include", "fa.h")).read()
    stated = f"{limits[128]} SMs (D = 64: {limits[64]} SMs)"
    assert stated in " ".join(header.split()), stated
    assert (f"D = 128 on up to {limits[128]} SMs" in src
            and f"at D = 64 on up to {limits[64]} SMs" in src)


def test_host_entry_point_rejects_bad_arguments_before_cuda(lib):
    """fa_fwd_host and its workspace query check sizes, masks and head dimensions before
    they touch the device."""
    host = dict(Q=ALIGNED, K=2 * ALIGNED, V=3 * ALIGNED, O=4 * ALIGNED, LSE=5 * ALIGNED)

    def call(B=1, H=1, Lq=16, Lk=16, D=64, left=-1, right=-1, scale=0.125):
        return fa.fa_fwd_host(host["Q"], host["K"], host["V"], host["O"], host["LSE"], B, H, Lq,
                              Lk, D, left, right, scale, 6 * ALIGNED, 1 << 20, 0)

    assert call(D=96) == fa.FA_ERR_UNSUPPORTED
    assert call(B=-1) == fa.FA_ERR_INVALID_ARG
    assert call(left=-2) == fa.FA_ERR_INVALID_ARG
    assert call(right=-5) == fa.FA_ERR_INVALID_ARG
    assert call(Lk=0) == fa.FA_ERR_INVALID_ARG
    assert call(scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert call(Lq=300, Lk=100, left=10, right=0) == fa.FA_ERR_INVALID_ARG   # rows without keys
    assert call(B=0) == fa.FA_OK                                             # nothing to do
    assert fa.fa_fwd_host_workspace_size(1, 1, 16, 16, 96, -1, -1)[0] == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_host_workspace_size(1, 1, 16, 16, 64, -3, -1)[0] == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_host_workspace_size(0, 1, 16, 16, 64, -1, -1) == (fa.FA_OK, 0)
    assert lib.fa_fwd_host_workspace_size(1, 1, 16, 16, 64, -1, -1, None) == fa.FA_ERR_INVALID_ARG
