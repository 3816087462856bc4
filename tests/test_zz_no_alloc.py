"""attn_decode_noalloc: KV-cache decode for callers that cannot allocate device memory.

Some callers of this library have no device allocator they may use: a host
program embedded in another runtime that already owns all device memory
through its own pool, or latency-sensitive code that cannot afford the
device-wide synchronisation that freeing memory brings.  For them the decode
entry point has a variant that takes no workspace and allocates nothing; its
per-slice partials go to a fixed scratch array built into the library.

These tests call it through the C ABI and compare it with attn_decode (which
uses a caller workspace).  Both run the same split of the keys through the
same kernels, so their results must agree bit for bit; the new entry point
is also checked against the fp64 oracle.  Four calls run in a row: a small
problem, one with more partials, one at the other head size, and the first
again, so that the later calls find the earlier calls' partials still in the
scratch array.  The file
sorts last so that a run that stops at the first failure has already run
every other test.
"""

import numpy as np
import pytest

import oracle
from exact_io_aware_107_b300 import _binding as B
from exact_io_aware_107_b300 import workloads as W
from gpu_util import BF16_TOL_LSE, BF16_TOL_O, max_err

pytestmark = pytest.mark.gpu


def _draw(shape_q, shape_kv, seed):
    import torch
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn(*shape_q, generator=g).to(torch.bfloat16)
    k = torch.randn(*shape_kv, generator=g).to(torch.bfloat16)
    v = torch.randn(*shape_kv, generator=g).to(torch.bfloat16)
    return q, k, v


def test_noalloc_decode_matches_workspace_decode_on_consecutive_calls():
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    assert B.attn_get_device_error(stream) == B.ATTN_OK
    # (B, H, Nq, Nk, D, seed): 264 KB of partials, then 1.06 MB, then 250 KB
    # at D = 64, then the first shape again on top of the others' partials
    cases = [(8, 32, 1, 32768, 128, 0), (2, 4, 8, 20000, 128, 1), (2, 4, 3, 5000, 64, 2),
             (8, 32, 1, 32768, 128, 3)]
    partials = []
    for Bn, H, Nq, Nk, D, seed in cases:
        hq, hk, hv = _draw((Bn, H, Nq, D), (Bn, H, Nk, D), seed)
        q, k, v = hq.cuda(), hk.cuda(), hv.cuda()
        scale = float(np.float32(1.0 / np.sqrt(D)))
        rc, need = B.attn_decode_workspace_bytes(Bn, H, Nq, Nk, D)
        assert rc == B.ATTN_OK and 0 < need <= B.NOALLOC_SCRATCH_BYTES
        partials.append(need)
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
        assert torch.equal(o, o_ref), (Bn, H, Nq, Nk, D)
        assert torch.equal(lse, lse_ref), (Bn, H, Nq, Nk, D)
        # and against the oracle, at the bf16 bars
        ro, rl = oracle.attention(W.as_f64(hq), W.as_f64(hk), W.as_f64(hv), scale, False)
        eo = max_err(o.float().cpu().numpy(), ro)
        el = max_err(lse.cpu().numpy(), rl)
        assert eo <= BF16_TOL_O and el <= BF16_TOL_LSE, (Bn, H, Nq, Nk, D, eo, el)
    assert partials[1] > partials[0] == partials[3]


def test_noalloc_refuses_problems_beyond_its_scratch():
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    # 256 planes of 256 keys split in two slices, 8 query rows: 2.1 MB of partials
    Bn, H, Nq, Nk, D = 8, 32, 8, 256, 128
    rc, need = B.attn_decode_workspace_bytes(Bn, H, Nq, Nk, D)
    assert rc == B.ATTN_OK and need > B.NOALLOC_SCRATCH_BYTES
    # real buffers of the problem's size: the call must refuse before launching,
    # but if it did not, it would still only touch memory it owns
    q = torch.zeros((Bn, H, Nq, D), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((Bn, H, Nk, D), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    o = torch.zeros_like(q)
    lse = torch.zeros((Bn, H, Nq), dtype=torch.float32, device="cuda")
    assert B.attn_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), Bn, H, Nq, Nk, D, 0.09, stream) == \
        B.ATTN_ERR_SCRATCH
    assert "scratch" in B.strerror(B.ATTN_ERR_SCRATCH)
    assert B.attn_get_device_error(stream) == B.ATTN_OK
