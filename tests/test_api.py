"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, and rejects bad arguments before touching a device."""

import os
import re

import pytest

from exact_io_aware_107_b300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("attn_fwd", "attn_fwd_f32", "attn_strerror", "attn_get_device_error"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert name in B._SIGNATURES, f"{name} has no ctypes signature"


def test_version_and_strerror(lib):
    assert B.attn_version() >= 100
    for code in range(-11, 1):
        s = B.strerror(code)
        assert s and s != "unknown status"
    assert B.strerror(-1234) == "unknown status"


BUF_BYTES = 8 << 20


@pytest.fixture(scope="module")
def buffers():
    """Addresses for the argument-error cases, inside buffers this module owns.

    Every shape these tests pass fits in BUF_BYTES, so a call that got past
    its checks by mistake would still only touch memory it may touch.  With a
    CUDA device the device address is a real device allocation; without one
    no call can launch, and a host buffer serves for both.
    """
    import numpy as np
    import torch
    host = np.zeros(BUF_BYTES + 256, dtype=np.uint8)
    hp = (host.ctypes.data + 255) // 256 * 256
    dev = torch.zeros(BUF_BYTES, dtype=torch.uint8, device="cuda") \
        if torch.cuda.is_available() else None
    yield (dev.data_ptr() if dev is not None else hp), hp
    if dev is not None:
        torch.cuda.synchronize()


@pytest.fixture
def P(buffers):
    """A 256-byte aligned device address (see `buffers`)."""
    return buffers[0]


@pytest.fixture
def HP(buffers):
    """A 256-byte aligned host address (see `buffers`)."""
    return buffers[1]


@pytest.mark.parametrize("fn", [B.attn_fwd, B.attn_fwd_f16, B.attn_fwd_f32])
def test_argument_errors_return_before_launch(lib, fn, P):
    good = dict(q=P, k=P, v=P, o=P, lse=P, B=1, H=1, N=16, D=64, cu_seqlens=None, causal=1,
                scale=0.125, stream=None)

    def call(**kw):
        a = dict(good, **kw)
        return fn(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["D"],
                  a["cu_seqlens"], a["causal"], a["scale"], a["stream"])

    assert call(B=0) == B.ATTN_ERR_SHAPE
    assert call(H=0) == B.ATTN_ERR_SHAPE
    assert call(N=-1) == B.ATTN_ERR_SHAPE
    assert call(scale=0.0) == B.ATTN_ERR_SCALE
    assert call(scale=-1.0) == B.ATTN_ERR_SCALE
    assert call(scale=float("inf")) == B.ATTN_ERR_SCALE
    assert call(scale=float("nan")) == B.ATTN_ERR_SCALE
    assert call(q=None) == B.ATTN_ERR_NULL
    assert call(lse=None) == B.ATTN_ERR_NULL
    assert call(o=P + 8) == B.ATTN_ERR_ALIGN
    assert call(lse=P + 2) == B.ATTN_ERR_ALIGN
    assert call(cu_seqlens=P + 1) == B.ATTN_ERR_ALIGN
    assert call(D=0) == B.ATTN_ERR_HEADDIM
    assert call(D=129) == B.ATTN_ERR_HEADDIM
    # N == 0 is a no-op even with NULL pointers
    assert call(N=0, q=None, k=None, v=None, o=None, lse=None) == B.ATTN_OK


@pytest.mark.parametrize("dtype", [B.ATTN_BF16, B.ATTN_F16, B.ATTN_F32])
def test_cross_argument_errors(lib, dtype, P):
    def call(**kw):
        a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, H=2, Nq=16, Nk=40, D=64, cq=None, ck=None,
                 causal=1, scale=0.125, dtype=dtype)
        a.update(kw)
        return B.attn_fwd_cross(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"],
                                a["Nq"], a["Nk"], a["D"], a["cq"], a["ck"], a["causal"],
                                a["scale"], a["dtype"], None)
    assert call(Nq=-1) == B.ATTN_ERR_SHAPE
    assert call(Nk=-1) == B.ATTN_ERR_SHAPE
    assert call(B=0) == B.ATTN_ERR_SHAPE
    assert call(cq=P) == B.ATTN_ERR_NULL          # only one of the two offset arrays
    assert call(ck=P) == B.ATTN_ERR_NULL
    assert call(k=None) == B.ATTN_ERR_NULL
    assert call(v=None) == B.ATTN_ERR_NULL
    assert call(cq=P, ck=P + 2) == B.ATTN_ERR_ALIGN
    assert call(k=P + 8) == B.ATTN_ERR_ALIGN
    assert call(scale=0.0) == B.ATTN_ERR_SCALE
    assert call(D=129) == B.ATTN_ERR_HEADDIM
    assert call(dtype=3) == B.ATTN_ERR_DTYPE
    assert call(dtype=-1) == B.ATTN_ERR_DTYPE
    # Nq == 0 is a no-op; Nk == 0 accepts NULL k and v (then fails only for want of a GPU)
    assert call(Nq=0, q=None, k=None, v=None, o=None, lse=None) == B.ATTN_OK
    assert call(Nk=0, k=None, v=None) in (B.ATTN_OK, B.ATTN_ERR_LAUNCH)


def test_host_forward_argument_errors(lib, P, HP):
    # q, k, v, o, lse are host addresses here, the workspace a device address
    def call(**kw):
        a = dict(q=HP, k=HP, v=HP, o=HP, lse=HP, B=2, H=3, N=100, D=128, causal=1, scale=0.1,
                 dtype=B.ATTN_BF16, ws=P, wsb=BUF_BYTES)
        a.update(kw)
        return B.attn_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"],
                               a["D"], a["causal"], a["scale"], a["dtype"], a["ws"], a["wsb"], None)
    assert call(B=0) == B.ATTN_ERR_SHAPE
    assert call(N=-1) == B.ATTN_ERR_SHAPE
    assert call(scale=0.0) == B.ATTN_ERR_SCALE
    assert call(dtype=7) == B.ATTN_ERR_DTYPE
    assert call(D=96) == B.ATTN_ERR_HEADDIM
    assert call(D=96, dtype=B.ATTN_F32) != B.ATTN_ERR_HEADDIM
    assert call(o=None) == B.ATTN_ERR_NULL
    assert call(ws=None) == B.ATTN_ERR_NULL
    assert call(ws=P + 128) == B.ATTN_ERR_ALIGN
    rc, need = B.attn_fwd_host_workspace_bytes(2, 3, 100, 128, B.ATTN_BF16)
    # 6 planes in 6 chunks of 1: two slots of q, k, v, o (100 x 128 bf16) and lse, 256-byte rounded
    assert rc == B.ATTN_OK and need == 2 * (4 * 25600 + 512)
    assert call(wsb=need - 1) == B.ATTN_ERR_SCRATCH
    assert call(N=0, q=None, k=None, v=None, o=None, lse=None, ws=None) == B.ATTN_OK


def test_backward_argument_errors(lib, P):
    def call(**kw):
        a = dict(q=P, k=P, v=P, o=P, lse=P, do=P, dq=P, dk=P, dv=P, B=1, H=2, Nq=16, Nk=40, D=64,
                 cq=None, ck=None, causal=1, scale=0.125, dtype=B.ATTN_BF16, ws=P, wsb=BUF_BYTES)
        a.update(kw)
        return B.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"],
                          a["dv"], a["B"], a["H"], a["Nq"], a["Nk"], a["D"], a["cq"], a["ck"],
                          a["causal"], a["scale"], a["dtype"], a["ws"], a["wsb"], None)
    assert call(B=0) == B.ATTN_ERR_SHAPE
    assert call(Nk=-1) == B.ATTN_ERR_SHAPE
    assert call(scale=0.0) == B.ATTN_ERR_SCALE
    assert call(dtype=B.ATTN_F32) == B.ATTN_ERR_DTYPE
    assert call(D=96) == B.ATTN_ERR_HEADDIM
    assert call(do=None) == B.ATTN_ERR_NULL
    assert call(dq=None) == B.ATTN_ERR_NULL
    assert call(dk=None) == B.ATTN_ERR_NULL
    assert call(ws=None) == B.ATTN_ERR_NULL
    assert call(cq=P) == B.ATTN_ERR_NULL
    assert call(dv=P + 8) == B.ATTN_ERR_ALIGN
    assert call(ws=P + 4) == B.ATTN_ERR_ALIGN
    rc, need = B.attn_bwd_workspace_bytes(1, 2, 16, 64, 0)
    assert rc == B.ATTN_OK and need == 256 + 2 * 16 * 64 * 4
    assert call(wsb=need - 1) == B.ATTN_ERR_SCRATCH
    assert B.attn_bwd_workspace_bytes(1, 2, 16, 80, 0)[0] == B.ATTN_ERR_HEADDIM
    assert B.attn_bwd_workspace_bytes(3, 2, 100, 128, 1)[1] == 1024 + 2 * 100 * 128 * 4
    assert call(Nq=0, Nk=0, q=None, k=None, v=None, o=None, lse=None, do=None, dq=None,
                dk=None, dv=None, ws=None) == B.ATTN_OK


def test_16bit_head_dims(lib, P):
    for fn in (B.attn_fwd, B.attn_fwd_f16):
        for d in (32, 96, 256):
            assert fn(P, P, P, P, P, 1, 1, 16, d, None, 1, 0.1, None) == B.ATTN_ERR_HEADDIM


def test_timeout_setter(lib):
    assert B.attn_set_wait_timeout_ns(0) == B.ATTN_ERR_SHAPE
    assert B.attn_set_wait_timeout_ns(999_999) == B.ATTN_ERR_SHAPE   # below one millisecond
    assert B.attn_set_wait_timeout_ns(1_000_000) == B.ATTN_OK
    assert B.attn_set_wait_timeout_ns(10**9) == B.ATTN_OK
    assert B.attn_wait_selftest(0, None) == B.ATTN_ERR_SHAPE


def test_fault_injection_switch(lib):
    assert B.attn_set_fault_injection(2) == B.ATTN_ERR_SHAPE
    assert B.attn_set_fault_injection(-1) == B.ATTN_ERR_SHAPE
    assert B.attn_set_fault_injection(1) == B.ATTN_OK
    assert B.attn_set_fault_injection(0) == B.ATTN_OK


def test_no_device_means_loud_failure(lib, P):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    # valid arguments with no GPU: the call fails, it never computes on the CPU
    assert B.attn_fwd(P, P, P, P, P, 1, 1, 16, 64, None, 1, 0.125, None) == B.ATTN_ERR_LAUNCH
    assert B.attn_fwd_f16(P, P, P, P, P, 1, 1, 16, 64, None, 1, 0.125, None) == B.ATTN_ERR_LAUNCH
    assert B.attn_fwd_f32(P, P, P, P, P, 1, 1, 16, 64, None, 1, 0.125, None) == B.ATTN_ERR_LAUNCH
    for dt in (B.ATTN_BF16, B.ATTN_F16, B.ATTN_F32):
        assert B.attn_fwd_cross(P, P, P, P, P, 1, 1, 16, 48, 64, None, None, 1, 0.125, dt,
                                None) == B.ATTN_ERR_LAUNCH


def test_decode_argument_errors(lib, P):
    def call(**kw):
        a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, H=2, Nq=1, Nk=100, D=128, scale=0.1, ws=None,
                 wsb=0)
        a.update(kw)
        return B.attn_decode(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"],
                             a["Nk"], a["D"], a["scale"], a["ws"], a["wsb"], None)
    assert call(Nq=0) == B.ATTN_ERR_SHAPE
    assert call(Nq=9) == B.ATTN_ERR_SHAPE
    assert call(Nk=0) == B.ATTN_ERR_SHAPE
    assert call(B=0) == B.ATTN_ERR_SHAPE
    assert call(D=96) == B.ATTN_ERR_HEADDIM
    assert call(scale=0.0) == B.ATTN_ERR_SCALE
    assert call(v=None) == B.ATTN_ERR_NULL
    assert call(o=P + 2) == B.ATTN_ERR_ALIGN
    assert call(ws=P + 4, wsb=1024) == B.ATTN_ERR_ALIGN
    rc, _ = B.attn_decode_workspace_bytes(1, 1, 9, 10, 128)
    assert rc == B.ATTN_ERR_SHAPE
    rc, _ = B.attn_decode_workspace_bytes(1, 1, 1, 10, 80)
    assert rc == B.ATTN_ERR_HEADDIM
    # B * H beyond 2^24 planes (and beyond the int range) is refused, not wrapped
    rc, _ = B.attn_decode_workspace_bytes(1 << 16, 1 << 16, 1, 10, 128)
    assert rc == B.ATTN_ERR_SHAPE
    rc, _ = B.attn_decode_workspace_bytes(1 << 12, (1 << 12) + 1, 1, 10, 128)
    assert rc == B.ATTN_ERR_SHAPE


def test_read_probe_argument_errors(lib, P):
    assert B.attn_hbm_read_probe(None, 16, P, None) == B.ATTN_ERR_NULL
    assert B.attn_hbm_read_probe(P, 16, None, None) == B.ATTN_ERR_NULL
    assert B.attn_hbm_read_probe(P, 0, P, None) == B.ATTN_ERR_SHAPE
    assert B.attn_hbm_read_probe(P, 24, P, None) == B.ATTN_ERR_SHAPE
    assert B.attn_hbm_read_probe(P + 8, 16, P, None) == B.ATTN_ERR_ALIGN
    assert B.attn_hbm_read_probe(P, 16, P + 2, None) == B.ATTN_ERR_ALIGN
