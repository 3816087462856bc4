"""The oracle pools' BLAS thread limit, with and without threadpoolctl."""

import subprocess
import sys

import pytest

CODE = """
import sys
if {hide}:
    sys.modules["threadpoolctl"] = None          # import fails as if not installed
from oracle.threads import _openblas, blas_threads
fns = _openblas()
assert fns is not None, "numpy's OpenBLAS exports its thread-count functions"
get = fns[1]
before = get()
with blas_threads(1):
    assert get() == 1, get()
assert get() == before
print("ok", before)
"""


@pytest.mark.parametrize("hide", [False, True])
def test_blas_threads_limits_and_restores(hide):
    r = subprocess.run([sys.executable, "-c", CODE.format(hide=hide)], capture_output=True,
                       text=True, cwd=__file__.rsplit("/tests/", 1)[0], timeout=120,
                       env={"OPENBLAS_NUM_THREADS": "4", "PATH": "/usr/bin:/bin"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.startswith("ok 4")


def test_children_inherit_one_blas_thread():
    import os
    from oracle.threads import SINGLE_THREAD_ENV, single_thread_children
    before = {k: os.environ.get(k) for k in SINGLE_THREAD_ENV}
    with single_thread_children():
        out = subprocess.run([sys.executable, "-c",
                              "import os; print(os.environ['OPENBLAS_NUM_THREADS'])"],
                             capture_output=True, text=True, timeout=60).stdout.strip()
        assert out == "1"
    assert {k: os.environ.get(k) for k in SINGLE_THREAD_ENV} == before
