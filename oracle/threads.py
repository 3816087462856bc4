"""BLAS threads of the oracle's thread and process pools (test infrastructure).

Only the tests and the oracle legs of ``bench.py`` use this; it holds none of
the attention arithmetic.  The oracle runs one plane per thread or process,
each with one BLAS thread: a BLAS that starts its own thread per core inside
every worker oversubscribes the host many times over (16 workers x 16 BLAS
threads on a 16-core host ran slower than one worker).

``threadpoolctl`` does this where it is installed; where it is not, the
OpenBLAS that numpy loaded is asked directly through its exported
thread-count functions.  Spawned workers also get ``OPENBLAS_NUM_THREADS=1``
(and the OpenMP/MKL equivalents) in their environment, which every BLAS reads
when it loads.
"""

from __future__ import annotations

import contextlib
import ctypes
import os

_SET = ("openblas_set_num_threads", "scipy_openblas_set_num_threads64_",
        "openblas_set_num_threads64_", "scipy_openblas_set_num_threads")
_GET = ("openblas_get_num_threads", "scipy_openblas_get_num_threads64_",
        "openblas_get_num_threads64_", "scipy_openblas_get_num_threads")

SINGLE_THREAD_ENV = {"OPENBLAS_NUM_THREADS": "1", "OMP_NUM_THREADS": "1",
                     "MKL_NUM_THREADS": "1"}


def _openblas():
    """(set, get) thread-count functions of the OpenBLAS loaded in this process, or None."""
    import numpy  # noqa: F401 - makes sure numpy's BLAS is loaded
    try:
        maps = open("/proc/self/maps").read().splitlines()
    except OSError:
        return None
    paths = sorted({ln.split()[-1] for ln in maps if "openblas" in ln.lower() and "/" in ln})
    for path in paths:
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        set_fn = next((getattr(lib, n) for n in _SET if hasattr(lib, n)), None)
        get_fn = next((getattr(lib, n) for n in _GET if hasattr(lib, n)), None)
        if set_fn is not None and get_fn is not None:
            set_fn.argtypes, set_fn.restype = [ctypes.c_int], None
            get_fn.argtypes, get_fn.restype = [], ctypes.c_int
            return set_fn, get_fn
    return None


def set_blas_threads(n: int) -> bool:
    """Set this process's BLAS thread count for good (worker initialisers)."""
    try:
        from threadpoolctl import threadpool_limits
        threadpool_limits(limits=n)
        return True
    except ImportError:
        pass
    fns = _openblas()
    if fns is None:
        return False
    fns[0](n)
    return True


@contextlib.contextmanager
def blas_threads(n: int):
    """BLAS limited to n threads inside the block, restored afterwards."""
    try:
        from threadpoolctl import threadpool_limits
    except ImportError:
        threadpool_limits = None
    if threadpool_limits is not None:
        with threadpool_limits(limits=n):
            yield
        return
    fns = _openblas()
    if fns is None:
        yield
        return
    set_fn, get_fn = fns
    old = get_fn()
    set_fn(n)
    try:
        yield
    finally:
        set_fn(old)


@contextlib.contextmanager
def single_thread_children():
    """Environment inherited by processes started inside the block: one BLAS thread."""
    old = {k: os.environ.get(k) for k in SINGLE_THREAD_ENV}
    os.environ.update(SINGLE_THREAD_ENV)
    try:
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
