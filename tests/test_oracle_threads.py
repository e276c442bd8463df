"""The oracle's OpenMP use: results independent of the thread count, and an
allocation failure in one thread reported as an error rather than a hang.

Each query row of the oracle is computed on its own, in index order, so any
thread count must give bit-identical results, including teams with more threads
than rows.  The second test builds a copy of the oracle whose row buffers fail to
allocate in thread 1 only and checks that every forward entry point returns
ORACLE_NO_MEMORY: every thread of the team must still meet the worksharing loop,
or the others would wait for it at the loop's closing barrier.  That test runs in a
child process under a timeout, so a deadlock fails it instead of stalling the suite.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import oracle

THREADS = (2, 3, 8, 16)


def _qkv(Lq, Lk, D, seed):
    g = np.random.default_rng(seed)
    return g.standard_normal((Lq, D)), g.standard_normal((Lk, D)), g.standard_normal((Lk, D))


@pytest.mark.parametrize("Lq,Lk", [(1, 1), (3, 5), (5, 3), (17, 9)])
def test_thread_count_does_not_change_results(oracle_mod, Lq, Lk):
    q, k, v = _qkv(Lq, Lk, 8, seed=Lq * 31 + Lk)
    calls = [
        lambda n: oracle.attn_head(q, k, v, False, 0.3, nthreads=n),
        lambda n: oracle.attn_head(q, k, v, True, 0.3, nthreads=n),
        lambda n: oracle.attn_head(q, k, v, True, 0.3, rows=[Lq - 1, 0], nthreads=n),
        lambda n: oracle.attn_head_window(q, k, v, -1, 1, 0.3, nthreads=n),
        lambda n: oracle.attn_head_keypad(q, k, v, -1, -1, max(1, Lk - 1), 0.3, nthreads=n),
        lambda n: oracle.attn_head_keypad(q, k, v, 0, -1, 0, 0.3, nthreads=n),
    ]
    for call in calls:
        ref = call(1)
        for n in THREADS:
            got = call(n)
            for a, b in zip(ref, got):
                np.testing.assert_array_equal(a, b)


_FAILING_MALLOC = """
/* test build: the row buffers of OpenMP thread 1 cannot be allocated */
static void *oracle_test_malloc(size_t n) { return omp_get_thread_num() == 1 ? NULL : malloc(n); }
#define malloc(n) oracle_test_malloc(n)
"""


def test_allocation_failure_in_one_thread_is_reported(tmp_path):
    src = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")
    text = open(src).read()
    anchor = "#include <omp.h>\n#endif\n"
    assert text.count(anchor) == 1
    mutated = tmp_path / "oracle_failing_malloc.c"
    mutated.write_text(text.replace(anchor, anchor + _FAILING_MALLOC))
    lib = oracle.build(force=True, src=str(mutated), out=str(tmp_path / "lib_failing_malloc.so"))
    script = textwrap.dedent(f"""
        import sys
        import numpy as np
        sys.path.insert(0, {os.path.dirname(os.path.dirname(oracle.__file__))!r})
        import oracle
        lib = oracle.OracleLib({lib!r})
        g = np.random.default_rng(0)
        q, k, v = (g.standard_normal((64, 8)) for _ in range(3))
        calls = [lambda: lib.attn_head(q, k, v, True, 0.3, nthreads=4),
                 lambda: lib.attn_head_window(q, k, v, 2, 2, 0.3, nthreads=4),
                 lambda: lib.attn_head_keypad(q, k, v, -1, -1, 40, 0.3, nthreads=4)]
        for call in calls:
            try:
                call()
            except ValueError as e:
                assert "code 2" in str(e), str(e)
            else:
                raise AssertionError("allocation failure not reported")
        print("reported")
    """)
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "reported" in r.stdout, r.stdout + r.stderr
