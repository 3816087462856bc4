"""Backward pass on the GPU (dQ, dK, dV) against the fp64 oracle.

Each gradient is compared element by element with the bound of
``gpu_util.bwd_bound_plane``: twice the first-order rounding error of the
16-bit arithmetic the kernel performs (P and dS rounded for the MMAs, Delta
from the 16-bit forward output, each gradient rounded once).
"""

import numpy as np
import pytest

from exact_io_aware_107_b300 import workloads as W
from gpu_util import UNIT, bwd_bound_plane, run_cuda_bwd

pytestmark = pytest.mark.gpu


def _dout(w, seed):
    """dO: standard normal, rounded to the workload's dtype, shaped like q."""
    import torch
    x = W.generate(W.custom(w.dtype, B=w.B, H=w.H, N=w.N, D=w.D, seed=seed, varlen=w.varlen))
    return x["q"].to(torch.float32).to(x["q"].dtype)


def _check_plane(got, q, k, v, do, scale, causal, unit, where):
    (rq, rk, rv), (bq, bk, bv) = bwd_bound_plane(q, k, v, do, scale, causal, unit)
    for name, g, r, b in (("dQ", got[0], rq, bq), ("dK", got[1], rk, bk), ("dV", got[2], rv, bv)):
        assert not np.isnan(g).any(), (where, name, "NaN")
        if g.size == 0:
            continue
        excess = np.abs(g - r) - b
        assert excess.max() <= 0, (where, name, float(np.abs(g - r).max()), float(excess.max()))
        # The bound above adds rounding errors as if they never cancelled.  Taken
        # together they do: each is at most u relative to its term and the terms'
        # signs vary, so the error of a whole gradient relative to the gradient
        # stays near u.  The test asks for 2u (Frobenius norms, planes of 64 or
        # more elements, whose gradient is not identically zero).
        nr = np.linalg.norm(r)
        if g.size >= 64 and nr > 1e-3:
            rel = np.linalg.norm(g - r) / nr
            assert rel <= 2 * unit, (where, name, "relative Frobenius error", rel)


def _compare(w, seed=100):
    x = W.generate(w)
    do = _dout(w, seed)
    dq, dk, dv = run_cuda_bwd(x["q"], x["k"], x["v"], do, w.causal, w.scale, x["cu_seqlens"],
                              x["cu_seqlens_k"])
    f = W.as_f64
    q, k, v, g = f(x["q"]), f(x["k"]), f(x["v"]), f(do)
    unit = UNIT[w.dtype]
    if x["cu_seqlens"] is None:
        for b in range(w.B):
            for h in range(w.H):
                _check_plane((dq[b, h], dk[b, h], dv[b, h]), q[b, h], k[b, h], v[b, h], g[b, h],
                             w.scale, w.causal, unit, (w.name, b, h))
    else:
        cu = x["cu_seqlens"]
        cuk = x["cu_seqlens_k"] if x["cu_seqlens_k"] is not None else cu
        for s in range(len(cu) - 1):
            a, e, ak, ek = int(cu[s]), int(cu[s + 1]), int(cuk[s]), int(cuk[s + 1])
            for h in range(w.H):
                _check_plane((dq[h, a:e], dk[h, ak:ek], dv[h, ak:ek]), q[h, a:e], k[h, ak:ek],
                             v[h, ak:ek], g[h, a:e], w.scale, w.causal, unit, (w.name, s, h))
    return dq, dk, dv, x, do


@pytest.mark.parametrize("N", [1, 7, 128, 129, 300, 700])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_backward_sweep(N, D, causal):
    _compare(W.custom("bf16", B=1, H=2, N=N, D=D, causal=causal, seed=N * 3 + D))


@pytest.mark.parametrize("N", [1, 129, 300])
@pytest.mark.parametrize("causal", [False, True])
def test_f16_backward_sweep(N, causal):
    _compare(W.custom("f16", B=1, H=2, N=N, D=128, causal=causal, seed=N + 1))


def test_bf16_backward_multi_batch_head():
    _compare(W.custom("bf16", B=2, H=3, N=513, D=128, causal=True, seed=8))


@pytest.mark.parametrize("nq,nk", [(77, 300), (300, 77), (1, 129), (130, 1), (256, 1000)])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_backward_cross(nq, nk, causal):
    _compare(W.custom("bf16", B=1, H=2, N=nq, D=128, causal=causal, seed=nq + nk, Nk=nk))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_bf16_backward_packed(causal, D):
    _compare(W.custom("bf16", H=2, D=D, causal=causal, seed=4,
                      varlen=[1, 127, 129, 300, 0, 257]))


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_backward_packed_cross(causal):
    _compare(W.custom("bf16", H=2, D=128, causal=causal, seed=5, varlen=[3, 200, 0, 130, 64],
                      varlen_k=[40, 130, 9, 0, 300]))


def test_backward_sum_identities_on_gpu():
    # sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i hold for any inputs; the GPU
    # sums are compared with the same bounds summed over the keys
    w = W.custom("bf16", B=1, H=2, N=1000, D=128, causal=True, seed=12)
    dq, dk, dv, x, do = _compare(w)
    g = W.as_f64(do)
    for h in range(2):
        (_, _, _), (bq, bk, bv) = bwd_bound_plane(W.as_f64(x["q"][0, h]), W.as_f64(x["k"][0, h]),
                                                 W.as_f64(x["v"][0, h]), g[0, h], w.scale, True,
                                                 UNIT["bf16"])
        assert (np.abs(dk[0, h].sum(0)) <= bk.sum(0)).all()
        assert (np.abs(dv[0, h].sum(0) - g[0, h].sum(0)) <= bv.sum(0)).all()


def test_backward_no_keys_and_no_queries():
    import torch
    from exact_io_aware_107_b300 import attention_backward, device_error
    x = W.generate(W.custom("bf16", B=1, H=2, N=200, D=64, seed=3))
    q = x["q"].cuda()
    empty = torch.empty((1, 2, 0, 64), dtype=q.dtype, device="cuda")
    lse = torch.full((1, 2, 200), float("-inf"), device="cuda")
    o = torch.zeros_like(q)
    dq, dk, dv = attention_backward(q, empty, empty, o, lse, q.clone(), causal=True)
    assert device_error() == 0
    assert (dq == 0).all() and dk.numel() == 0
    k = x["k"].cuda()
    qe = torch.empty((1, 2, 0, 64), dtype=q.dtype, device="cuda")
    lse0 = torch.empty((1, 2, 0), device="cuda")
    dq, dk, dv = attention_backward(qe, k, k, qe, lse0, qe, causal=False,
                                    dk=torch.full_like(k, float("nan")),
                                    dv=torch.full_like(k, float("nan")))
    assert device_error() == 0
    assert (dk == 0).all() and (dv == 0).all()


def test_backward_dk_dv_deterministic():
    w = W.custom("bf16", B=1, H=4, N=777, D=128, causal=True, seed=14)
    x = W.generate(w)
    do = _dout(w, 7)
    a = run_cuda_bwd(x["q"], x["k"], x["v"], do, True, w.scale)
    b = run_cuda_bwd(x["q"], x["k"], x["v"], do, True, w.scale)
    np.testing.assert_array_equal(a[1], b[1])
    np.testing.assert_array_equal(a[2], b[2])
    # dQ sums key tiles in a free order: equal up to fp32 reassociation before the rounding
    assert np.abs(a[0] - b[0]).max() <= 2.0 ** -7 * max(1.0, np.abs(a[0]).max())


def test_backward_bf16_causal_b2_h32_n8192_d128_one_plane():
    # the full-size workload; the oracle checks two planes completely
    w = W.WORKLOADS["bf16_causal_b2_h32_n8192_d128"]
    x = W.generate(w)
    do = _dout(w, 1)
    dq, dk, dv = run_cuda_bwd(x["q"], x["k"], x["v"], do, True, w.scale)
    assert np.isfinite(dq).all() and np.isfinite(dk).all() and np.isfinite(dv).all()
    f = W.as_f64
    for b, h in ((0, 0), (1, 31)):
        _check_plane((dq[b, h], dk[b, h], dv[b, h]), f(x["q"][b, h]), f(x["k"][b, h]),
                     f(x["v"][b, h]), f(do[b, h]), w.scale, True, UNIT["bf16"], (b, h))


def test_backward_long_plane_tail_and_sampled_rows():
    # One causal plane of 2^16 rows.  The full fp64 gradient is out of reach,
    # but two parts of it are exact on slices: the last 256 query rows are the
    # only ones that see the last 256 keys, so the oracle on those rows (the
    # cross alignment: last query with last key) gives dQ of those rows and
    # dK, dV of those keys completely; and row r's dQ needs only keys 0..r.
    n, d = 1 << 16, 128
    w = W.custom("bf16", B=1, H=1, N=n, D=d, causal=True, seed=15)
    x = W.generate(w)
    do = _dout(w, 16)
    dq, dk, dv = run_cuda_bwd(x["q"], x["k"], x["v"], do, True, w.scale)
    assert np.isfinite(dq).all() and np.isfinite(dk).all() and np.isfinite(dv).all()
    q, k, v, g = (W.as_f64(t[0, 0]) for t in (x["q"], x["k"], x["v"], do))
    u = UNIT["bf16"]
    tail = 256
    (rq, rk, rv), (bq, bk, bv) = bwd_bound_plane(q[n - tail:], k, v, g[n - tail:], w.scale,
                                                 True, u)
    assert (np.abs(dq[0, 0, n - tail:] - rq) <= bq).all()
    assert (np.abs(dk[0, 0, n - tail:] - rk[n - tail:]) <= bk[n - tail:]).all()
    assert (np.abs(dv[0, 0, n - tail:] - rv[n - tail:]) <= bv[n - tail:]).all()
    rng = np.random.default_rng(16)
    for r in sorted({0, 1, 127, 128, 129, n // 2, n - tail - 1} | set(rng.integers(0, n, 8))):
        r = int(r)
        (rq1, _, _), (bq1, _, _) = bwd_bound_plane(q[r:r + 1], k[:r + 1], v[:r + 1], g[r:r + 1],
                                                   w.scale, True, u)
        assert (np.abs(dq[0, 0, r] - rq1[0]) <= bq1[0]).all(), r
