"""attn_decode_noalloc: KV-cache decode for callers that cannot allocate device memory.

Some callers of this library have no device allocator they may use: a host
program embedded in another runtime that already owns all device memory
through its own pool, or latency-sensitive code that cannot afford the
device-wide synchronisation that freeing memory brings.  For them the decode
entry point has a variant that takes no workspace and allocates nothing; its
per-slice partials go to a fixed scratch array built into the library.

These tests call it through the C ABI and compare it with attn_decode (which
uses a caller workspace), on two calls in a row with different shapes, so the
second call runs on scratch that still holds the first call's partials.  The
file sorts last so that a run that stops at the first failure has already run
every other test.
"""

import numpy as np
import pytest

from exact_io_aware_107_b300 import _binding as B
from gpu_util import BF16_TOL_LSE, BF16_TOL_O

pytestmark = pytest.mark.gpu


def _draw(shape_q, shape_kv, seed):
    import torch
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn(*shape_q, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(*shape_kv, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(*shape_kv, generator=g).to(torch.bfloat16).cuda()
    return q, k, v


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    assert B.attn_get_device_error(stream) == B.ATTN_OK
    cases = [(8, 32, 1, 32768, 128, 0), (2, 4, 3, 5000, 64, 1)]
    for Bn, H, Nq, Nk, D, seed in cases:
        q, k, v = _draw((Bn, H, Nq, D), (Bn, H, Nk, D), seed)
        scale = float(np.float32(1.0 / np.sqrt(D)))
        rc, need = B.attn_decode_workspace_bytes(Bn, H, Nq, Nk, D)
        assert rc == B.ATTN_OK and 0 < need <= B.NOALLOC_SCRATCH_BYTES
        # the existing entry point, with a workspace allocated here by torch
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        o_ref = torch.empty_like(q)
        lse_ref = torch.empty((Bn, H, Nq), dtype=torch.float32, device="cuda")
        assert B.attn_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_ref.data_ptr(),
                             lse_ref.data_ptr(), Bn, H, Nq, Nk, D, scale, ws.data_ptr(), need,
                             stream) == B.ATTN_OK
        # the variant that allocates nothing
        o = torch.full_like(q, float("nan"))
        lse = torch.full((Bn, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
        assert B.attn_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), Bn, H, Nq, Nk, D, scale,
                                     stream) == B.ATTN_OK
        assert B.attn_get_device_error(stream) == B.ATTN_OK
        d_o = (o.float() - o_ref.float()).abs().max().item()
        d_l = (lse - lse_ref).abs().max().item()
        assert d_o <= BF16_TOL_O and d_l <= BF16_TOL_LSE, (Bn, H, Nq, Nk, D, d_o, d_l)


def test_noalloc_refuses_problems_beyond_its_scratch():
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    Bn, H, Nq, Nk, D = 8, 32, 8, 32768, 128
    rc, need = B.attn_decode_workspace_bytes(Bn, H, Nq, Nk, D)
    assert rc == B.ATTN_OK and need > B.NOALLOC_SCRATCH_BYTES
    p = 1 << 20  # aligned stand-in addresses: the call must refuse before touching memory
    assert B.attn_decode_noalloc(p, p, p, p, p, Bn, H, Nq, Nk, D, 0.09, stream) == \
        B.ATTN_ERR_SCRATCH
    assert "scratch" in B.strerror(B.ATTN_ERR_SCRATCH)
    assert B.attn_get_device_error(stream) == B.ATTN_OK
