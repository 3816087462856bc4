"""ctypes binding of the C ABI declared in include/attn_b300.h.

Argument marshalling only: every step of the attention forward runs in the
CUDA library.  The functions keep the C names and argument order; tensors
are passed as raw device pointers (``tensor.data_ptr()``) and the stream as a
``cudaStream_t`` handle (``torch.cuda.current_stream().cuda_stream``).
There is no CPU fallback: if the library cannot be loaded, :func:`load`
raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn_b300.so")

ATTN_OK = 0
ATTN_ERR_NULL = -1
ATTN_ERR_SHAPE = -2
ATTN_ERR_HEADDIM = -3
ATTN_ERR_ALIGN = -4
ATTN_ERR_ARCH = -5
ATTN_ERR_LAUNCH = -6
ATTN_ERR_TIMEOUT = -7
ATTN_ERR_BOUNDS = -8
ATTN_ERR_SCALE = -9
ATTN_ERR_SCRATCH = -10
ATTN_ERR_DTYPE = -11
ATTN_BF16 = 0
ATTN_F16 = 1
ATTN_F32 = 2
NOALLOC_SCRATCH_BYTES = 2 << 20

# Every symbol include/attn_b300.h declares, with its ctypes signature.
_SIGNATURES = {
    "attn_fwd": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4
                 + [ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p]),
    "attn_fwd_f16": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4
                     + [ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p]),
    "attn_fwd_f32": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4
                     + [ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p]),
    "attn_fwd_cross": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5
                       + [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_float,
                          ctypes.c_int, ctypes.c_void_p]),
    "attn_fwd_host": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5
                      + [ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_ulonglong,
                         ctypes.c_void_p]),
    "attn_fwd_host_workspace_bytes": (ctypes.c_int, [ctypes.c_int] * 5
                                      + [ctypes.POINTER(ctypes.c_ulonglong)]),
    "attn_bwd": (ctypes.c_int, [ctypes.c_void_p] * 9 + [ctypes.c_int] * 5
                 + [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                    ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_void_p]),
    "attn_bwd_workspace_bytes": (ctypes.c_int, [ctypes.c_int] * 5
                                 + [ctypes.POINTER(ctypes.c_ulonglong)]),
    "attn_decode": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5
                    + [ctypes.c_float, ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_void_p]),
    "attn_decode_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5
                            + [ctypes.c_float, ctypes.c_void_p]),
    "attn_decode_workspace_bytes": (ctypes.c_int, [ctypes.c_int] * 5
                                    + [ctypes.POINTER(ctypes.c_ulonglong)]),
    "attn_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "attn_get_device_error": (ctypes.c_int, [ctypes.c_void_p]),
    "attn_set_wait_timeout_ns": (ctypes.c_int, [ctypes.c_ulonglong]),
    "attn_set_fault_injection": (ctypes.c_int, [ctypes.c_int]),
    "attn_wait_selftest": (ctypes.c_int, [ctypes.c_ulonglong, ctypes.c_void_p]),
    "attn_hbm_read_probe": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_void_p,
                                           ctypes.c_void_p]),
    "attn_version": (ctypes.c_int, []),
}

_lib = None
_lock = threading.Lock()


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {strerror(status)} (status {status})")


def load(path: str = LIB_PATH):
    """Load the library (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path) or path == LIB_PATH:
                from . import build as _build
                if _build.needs_build():
                    _build.build()
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def strerror(status: int) -> str:
    return load().attn_strerror(int(status)).decode()


def attn_fwd(q, k, v, o, lse, B, H, N, D, cu_seqlens, causal, scale, stream) -> int:
    """bf16 forward; pointers are ints (device addresses) or None."""
    return load().attn_fwd(q, k, v, o, lse, int(B), int(H), int(N), int(D), cu_seqlens,
                           int(causal), float(scale), stream)


def attn_fwd_f16(q, k, v, o, lse, B, H, N, D, cu_seqlens, causal, scale, stream) -> int:
    """fp16 forward; pointers are ints (device addresses) or None."""
    return load().attn_fwd_f16(q, k, v, o, lse, int(B), int(H), int(N), int(D), cu_seqlens,
                               int(causal), float(scale), stream)


def attn_fwd_f32(q, k, v, o, lse, B, H, N, D, cu_seqlens, causal, scale, stream) -> int:
    """fp32 forward; pointers are ints (device addresses) or None."""
    return load().attn_fwd_f32(q, k, v, o, lse, int(B), int(H), int(N), int(D), cu_seqlens,
                               int(causal), float(scale), stream)


def attn_fwd_cross(q, k, v, o, lse, B, H, Nq, Nk, D, cu_seqlens_q, cu_seqlens_k, causal, scale,
                   dtype, stream) -> int:
    """Forward with Nq queries and Nk keys (ATTN_BF16 / ATTN_F16 / ATTN_F32)."""
    return load().attn_fwd_cross(q, k, v, o, lse, int(B), int(H), int(Nq), int(Nk), int(D),
                                 cu_seqlens_q, cu_seqlens_k, int(causal), float(scale),
                                 int(dtype), stream)


def attn_fwd_host(q, k, v, o, lse, B, H, N, D, causal, scale, dtype, workspace, workspace_bytes,
                  stream) -> int:
    """Forward from host buffers (q, k, v, o, lse are host addresses)."""
    return load().attn_fwd_host(q, k, v, o, lse, int(B), int(H), int(N), int(D), int(causal),
                                float(scale), int(dtype), workspace, int(workspace_bytes), stream)


def attn_fwd_host_workspace_bytes(B, H, N, D, dtype):
    """(status, bytes) for the host-buffer forward's device workspace."""
    n = ctypes.c_ulonglong(0)
    rc = load().attn_fwd_host_workspace_bytes(int(B), int(H), int(N), int(D), int(dtype),
                                              ctypes.byref(n))
    return rc, n.value


def attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, D, cu_seqlens_q, cu_seqlens_k,
             causal, scale, dtype, workspace, workspace_bytes, stream) -> int:
    """Backward pass (dQ, dK, dV); pointers are ints (device addresses) or None."""
    return load().attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, int(B), int(H), int(Nq), int(Nk),
                           int(D), cu_seqlens_q, cu_seqlens_k, int(causal), float(scale),
                           int(dtype), workspace, int(workspace_bytes), stream)


def attn_bwd_workspace_bytes(B, H, Nq, D, packed):
    """(status, bytes) for the backward workspace."""
    n = ctypes.c_ulonglong(0)
    rc = load().attn_bwd_workspace_bytes(int(B), int(H), int(Nq), int(D), int(bool(packed)),
                                         ctypes.byref(n))
    return rc, n.value


def attn_decode(q, k, v, o, lse, B, H, Nq, Nk, D, scale, workspace, workspace_bytes,
                stream) -> int:
    """bf16 KV-cache decode; pointers are ints (device addresses) or None."""
    return load().attn_decode(q, k, v, o, lse, int(B), int(H), int(Nq), int(Nk), int(D),
                              float(scale), workspace, int(workspace_bytes), stream)


def attn_decode_noalloc(q, k, v, o, lse, B, H, Nq, Nk, D, scale, stream) -> int:
    """Decode without a caller workspace (the library's built-in scratch is used)."""
    return load().attn_decode_noalloc(q, k, v, o, lse, int(B), int(H), int(Nq), int(Nk), int(D),
                                      float(scale), stream)


def attn_decode_workspace_bytes(B, H, Nq, Nk, D):
    """(status, bytes) for the decode workspace on the current device."""
    n = ctypes.c_ulonglong(0)
    rc = load().attn_decode_workspace_bytes(int(B), int(H), int(Nq), int(Nk), int(D),
                                            ctypes.byref(n))
    return rc, n.value


def attn_get_device_error(stream) -> int:
    return load().attn_get_device_error(stream)


def attn_set_wait_timeout_ns(ns: int) -> int:
    return load().attn_set_wait_timeout_ns(int(ns))


def attn_set_fault_injection(on: int) -> int:
    return load().attn_set_fault_injection(int(on))


def attn_wait_selftest(timeout_ns: int, stream) -> int:
    return load().attn_wait_selftest(int(timeout_ns), stream)


def attn_hbm_read_probe(buf, nbytes, out, stream) -> int:
    """Read-only stream over `nbytes` of device memory (bandwidth measurement)."""
    return load().attn_hbm_read_probe(buf, int(nbytes), out, stream)


def attn_version() -> int:
    return load().attn_version()
