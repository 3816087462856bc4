"""Cross-attention (Nq != Nk) on the GPU: parity with the fp64 oracle and
identities that need no oracle.

The causal mask aligns the last query with the last key (key j allowed for
query i when j <= i + Nk - Nq); a query with no allowed key gets O = 0 and
LSE = -inf.
"""

import numpy as np
import pytest

import oracle
from exact_io_aware_107_b300 import workloads as W
from gpu_util import (BF16_TOL_LSE, BF16_TOL_O, F16_TOL_LSE, F16_TOL_O, F32_TOL_LSE, F32_TOL_O,
                      max_err, run_cuda)

pytestmark = pytest.mark.gpu

TOL = {"bf16": (BF16_TOL_O, BF16_TOL_LSE), "f16": (F16_TOL_O, F16_TOL_LSE),
       "f32": (F32_TOL_O, F32_TOL_LSE)}


def _compare(w):
    x = W.generate(w)
    o, lse = run_cuda(x["q"], x["k"], x["v"], w.causal, w.scale, x["cu_seqlens"],
                      cu_seqlens_k=x["cu_seqlens_k"])
    ro, rl = oracle.attention(W.as_f64(x["q"]), W.as_f64(x["k"]), W.as_f64(x["v"]), w.scale,
                              w.causal, cu_seqlens=x["cu_seqlens"],
                              cu_seqlens_k=x["cu_seqlens_k"])
    tol_o, tol_l = TOL[w.dtype]
    eo, el = max_err(o, ro), max_err(lse, rl)
    assert eo <= tol_o and el <= tol_l, (w, eo, el)
    # rows without a key: exactly zero and -inf
    dead = np.isneginf(rl)
    assert (o[dead] == 0).all() and np.isneginf(lse[dead]).all()
    return o, lse, x


SHAPES = [(1, 300), (77, 300), (128, 1000), (129, 257), (300, 77), (1000, 128), (257, 1),
          (5, 700), (640, 640)]


@pytest.mark.parametrize("nq,nk", SHAPES)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_cross_dense(nq, nk, D, causal):
    _compare(W.custom("bf16", B=1, H=2, N=nq, D=D, causal=causal, seed=nq * 3 + nk, Nk=nk))


@pytest.mark.parametrize("nq,nk", [(77, 300), (300, 77), (1, 129), (640, 640)])
@pytest.mark.parametrize("causal", [False, True])
def test_f16_cross_dense(nq, nk, causal):
    _compare(W.custom("f16", B=2, H=1, N=nq, D=128, causal=causal, seed=nq + nk, Nk=nk))


@pytest.mark.parametrize("nq,nk", [(1, 300), (77, 300), (300, 77), (33, 1), (64, 64)])
@pytest.mark.parametrize("D", [16, 100, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_f32_cross_dense(nq, nk, D, causal):
    _compare(W.custom("f32", B=1, H=2, N=nq, D=D, causal=causal, seed=nq + 7 * nk, Nk=nk))


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("f16", 64), ("f32", 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_packed_cross(dtype, D, causal):
    # includes a sequence without keys, one without queries, and ragged tiles
    lq = [1, 300, 0, 129, 513, 7, 256]
    lk = [40, 130, 9, 0, 600, 7, 1000]
    _compare(W.custom(dtype, H=3, D=D, causal=causal, seed=11, varlen=lq, varlen_k=lk))


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("f16", 128), ("f32", 64)])
def test_causal_cross_is_the_tail_of_self_attention(dtype, D):
    # queries = the last Nq positions: every output row equals the matching row
    # of causal self-attention, bit for bit (the same key tiles and mask reach
    # each row; the extra fully masked tiles of a self-attention tile add zeros)
    import torch
    n = 1000
    x = W.generate(W.custom(dtype, B=1, H=2, N=n, D=D, causal=True, seed=21))
    o, lse = run_cuda(x["q"], x["k"], x["v"], True, 0.1)
    for nq in (1, 100, 128, 129, 999):
        qt = x["q"][:, :, n - nq:].contiguous()
        oc, lc = run_cuda(qt, x["k"], x["v"], True, 0.1)
        np.testing.assert_array_equal(oc, o[:, :, n - nq:])
        np.testing.assert_array_equal(lc, lse[:, :, n - nq:])
    del torch


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_cross_entry_with_equal_lengths_matches_self_entry(dtype):
    import torch
    from exact_io_aware_107_b300 import _binding, device_error
    w = W.custom(dtype, B=2, H=3, N=700, D=64, causal=True, seed=5)
    x = W.generate(w)
    o_self, l_self = run_cuda(x["q"], x["k"], x["v"], True, w.scale)
    q, k, v = (t.cuda() for t in (x["q"], x["k"], x["v"]))
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    kind = {"bf16": _binding.ATTN_BF16, "f16": _binding.ATTN_F16, "f32": _binding.ATTN_F32}[dtype]
    rc = _binding.attn_fwd_cross(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), 2, 3, 700, 700, 64, None, None, 1, w.scale, kind,
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == 0 and device_error() == 0
    np.testing.assert_array_equal(o.float().cpu().numpy(), o_self)
    np.testing.assert_array_equal(lse.cpu().numpy(), l_self)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
def test_no_keys_at_all(dtype, causal):
    import torch
    from exact_io_aware_107_b300 import attention_forward, device_error
    x = W.generate(W.custom(dtype, B=2, H=2, N=300, D=64, seed=3))
    q = x["q"].cuda()
    k = torch.empty((2, 2, 0, 64), dtype=q.dtype, device="cuda")
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    attention_forward(q, k, k, causal=causal, out=o, lse=lse)
    assert device_error() == 0
    assert (o == 0).all() and torch.isneginf(lse).all()


def test_bad_cu_seqlens_k_reported_on_device():
    import torch
    from exact_io_aware_107_b300 import _binding, attention_forward, device_error
    x = W.generate(W.custom("bf16", B=1, H=2, N=256, D=64, seed=6))
    q = x["q"][0].contiguous().cuda()
    k = x["k"][0].contiguous().cuda()
    cu = torch.tensor([0, 100, 256], dtype=torch.int32, device="cuda")
    for bad in ([0, 300, 256], [0, 200, 100]):       # beyond Nk; decreasing
        cuk = torch.tensor(bad, dtype=torch.int32, device="cuda")
        attention_forward(q, k, k, causal=True, cu_seqlens=cu, cu_seqlens_k=cuk)
        assert device_error() == _binding.ATTN_ERR_BOUNDS
    assert device_error() == 0


def _rows(n, rng):
    base = {0, 1, n - 1, n - 2} | {t + d for t in range(128, n, 128) for d in (-1, 0)}
    base = sorted(r for r in base if 0 <= r < n)
    pick = rng.choice(base, min(48, len(base)), replace=False).tolist()
    return np.array(sorted(set(pick) | set(rng.integers(0, n, 32).tolist()) | {0, n - 1}))


@pytest.mark.parametrize("name", sorted(W.CROSS_WORKLOADS))
def test_cross_workloads_sampled(name):
    w = W.CROSS_WORKLOADS[name]
    x = W.generate(w)
    o, lse = run_cuda(x["q"], x["k"], x["v"], w.causal, w.scale)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    rng = np.random.default_rng(99)
    worst_o = worst_l = 0.0
    for b, h in ((0, 0), (1, 31), (0, 13)):
        rows = _rows(w.N, rng)
        ro, rl = oracle.attention_rows(W.as_f64(x["q"][b, h]), W.as_f64(x["k"][b, h]),
                                       W.as_f64(x["v"][b, h]), w.scale, w.causal, rows)
        worst_o = max(worst_o, max_err(o[b, h][rows], ro))
        worst_l = max(worst_l, max_err(lse[b, h][rows], rl))
    assert worst_o <= BF16_TOL_O and worst_l <= BF16_TOL_LSE, (worst_o, worst_l)
