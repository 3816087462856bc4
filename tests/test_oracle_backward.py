"""Pins of the fp64 backward oracle (dQ, dK, dV) against facts that do not
come from its own formula: central finite differences of the forward oracle,
the sum identities of the softmax gradient, special cases with a closed
form, and torch autograd through an independently written forward."""

import numpy as np
import pytest

from oracle import exact as A


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _loss(q, k, v, do, scale, causal):
    o, _ = A.attention_plane(q, k, v, scale, causal)
    return float((o * do).sum())


def _finite_diff(q, k, v, do, scale, causal, h=1e-6):
    out = []
    for which in range(3):
        args = [q, k, v]
        g = np.zeros_like(args[which])
        for idx in np.ndindex(*g.shape):
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[which][idx] += h
            minus[which][idx] -= h
            g[idx] = (_loss(*plus, do, scale, causal) - _loss(*minus, do, scale, causal)) / (2 * h)
        out.append(g)
    return out


CASES = [(1, 1), (2, 2), (4, 4), (5, 5), (3, 6), (6, 3), (1, 4)]


@pytest.mark.parametrize("nq,nk", CASES)
@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(nq, nk, causal):
    rng = np.random.default_rng(nq * 10 + nk + (100 if causal else 0))
    d = 3
    q, k, v, do = _rand(rng, nq, d), _rand(rng, nk, d), _rand(rng, nk, d), _rand(rng, nq, d)
    dq, dk, dv = A.attention_backward_plane(q, k, v, do, 0.8, causal)
    nq_, nk_, nv_ = _finite_diff(q, k, v, do, 0.8, causal)
    np.testing.assert_allclose(dq, nq_, rtol=0, atol=1e-7)
    np.testing.assert_allclose(dk, nk_, rtol=0, atol=1e-7)
    np.testing.assert_allclose(dv, nv_, rtol=0, atol=1e-7)


@pytest.mark.parametrize("nq,nk", [(40, 40), (17, 60), (60, 17)])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_sum_identities(nq, nk, causal):
    # each row of dS sums to zero over its keys, so sum_j dK_j = 0; rows of P
    # sum to one, so sum_j dV_j = sum of dO over the rows that see a key
    rng = np.random.default_rng(nq + nk)
    q, k, v, do = _rand(rng, nq, 8), _rand(rng, nk, 8), _rand(rng, nk, 8), _rand(rng, nq, 8)
    dq, dk, dv = A.attention_backward_plane(q, k, v, do, 0.4, causal)
    np.testing.assert_allclose(dk.sum(0), 0.0, atol=1e-12)
    live = np.arange(nq) + (nk - nq) >= 0 if causal else np.ones(nq, dtype=bool)
    np.testing.assert_allclose(dv.sum(0), do[live].sum(0), atol=1e-12)
    if causal and nq > nk:
        # the first nq - nk queries see no key: their gradient is zero
        assert (dq[:nq - nk] == 0).all()


def test_backward_special_cases():
    rng = np.random.default_rng(3)
    # one query, one key: P = 1, O = v, so dV = dO and dQ = dK = 0
    q, k, v, do = _rand(rng, 1, 4), _rand(rng, 1, 4), _rand(rng, 1, 4), _rand(rng, 1, 4)
    dq, dk, dv = A.attention_backward_plane(q, k, v, do, 0.5, True)
    np.testing.assert_array_equal(dv, do)
    assert (dq == 0).all() and (dk == 0).all()
    # causal: the last key is seen only by the last query
    q, k, v, do = _rand(rng, 6, 4), _rand(rng, 6, 4), _rand(rng, 6, 4), _rand(rng, 6, 4)
    dq, dk, dv = A.attention_backward_plane(q, k, v, do, 0.5, True)
    p = A.softmax_probs(q, k, 0.5, True)
    np.testing.assert_allclose(dv[5], p[5, 5] * do[5], atol=1e-14)
    # equal keys: P is uniform over the allowed keys and does not depend on Q,
    # so dQ = 0; with equal values too, O = v and dK = 0
    kk = np.tile(_rand(rng, 1, 4), (6, 1))
    vv = np.tile(_rand(rng, 1, 4), (6, 1))
    dq, dk, dv = A.attention_backward_plane(q, kk, vv, do, 0.5, False)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    np.testing.assert_allclose(dk, 0.0, atol=1e-13)
    np.testing.assert_allclose(dv, np.tile(do.sum(0) / 6, (6, 1)), atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk", [(50, 50), (30, 70)])
def test_backward_matches_autograd_of_a_separate_forward(causal, nq, nk):
    import torch
    rng = np.random.default_rng(9)
    q, k, v, do = _rand(rng, nq, 16), _rand(rng, nk, 16), _rand(rng, nk, 16), _rand(rng, nq, 16)
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    s = 0.3 * tq @ tk.T
    if causal:
        keep = torch.arange(nk)[None, :] <= torch.arange(nq)[:, None] + (nk - nq)
        s = s.masked_fill(~keep, float("-inf"))
    o = torch.softmax(s, dim=-1) @ tv
    o.backward(torch.tensor(do))
    dq, dk, dv = A.attention_backward_plane(q, k, v, do, 0.3, causal)
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)


def test_backward_slabs_equal_full(monkeypatch):
    rng = np.random.default_rng(12)
    q, k, v, do = _rand(rng, 300, 8), _rand(rng, 300, 8), _rand(rng, 300, 8), _rand(rng, 300, 8)
    full = A.attention_backward_plane(q, k, v, do, 0.3, True)
    monkeypatch.setattr(A, "FULL_MATRIX_MAX_N", 64)
    monkeypatch.setattr(A, "SLAB_ROWS", 37)
    slab = A.attention_backward_plane(q, k, v, do, 0.3, True)
    for a, b in zip(full, slab):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_backward_packed_equals_per_sequence():
    rng = np.random.default_rng(13)
    lq, lk = [3, 0, 40, 7], [5, 2, 30, 0]
    cq, ck = np.cumsum([0] + lq), np.cumsum([0] + lk)
    q, do = _rand(rng, 2, cq[-1], 8), _rand(rng, 2, cq[-1], 8)
    k, v = _rand(rng, 2, ck[-1], 8), _rand(rng, 2, ck[-1], 8)
    dq, dk, dv = A.attention_backward(q, k, v, do, 0.3, True, cu_seqlens=cq, cu_seqlens_k=ck)
    for s in range(4):
        for h in range(2):
            a, e, ak, ek = cq[s], cq[s + 1], ck[s], ck[s + 1]
            r = A.attention_backward_plane(q[h, a:e], k[h, ak:ek], v[h, ak:ek], do[h, a:e], 0.3,
                                           True)
            np.testing.assert_array_equal(dq[h, a:e], r[0])
            np.testing.assert_array_equal(dk[h, ak:ek], r[1])
            np.testing.assert_array_equal(dv[h, ak:ek], r[2])


# Plausible mistakes, planted in a copy of the oracle on the CPU: each must fail a pin.
def _mutant(kind):
    def bwd(qp, kp, vp, dop, scale, causal):
        n = qp.shape[0]
        p = A._probs_rows(qp, kp, scale, causal, kp.shape[0] - n, 0, n)
        o = p @ vp
        dv = p.T @ dop
        dp = dop @ vp.T
        delta = (dop * o).sum(axis=1, keepdims=True)
        if kind == "no_delta":
            delta = 0 * delta
        ds = p * (dp - delta)
        if kind == "ds_transposed" and ds.shape[0] == ds.shape[1]:
            ds = ds.T
        dq = scale * (ds @ kp)
        dk = scale * (ds.T @ qp)
        if kind == "no_scale":
            dq, dk = dq / scale, dk / scale
        if kind == "dv_uses_dp":
            dv = p.T @ (dop + 0.01 * dp @ vp)
        return dq, dk, dv
    return bwd


@pytest.mark.parametrize("kind", ["no_delta", "ds_transposed", "no_scale", "dv_uses_dp"])
def test_backward_mutants_are_caught(kind):
    rng = np.random.default_rng(5)
    q, k, v, do = _rand(rng, 4, 3), _rand(rng, 4, 3), _rand(rng, 4, 3), _rand(rng, 4, 3)
    dq, dk, dv = _mutant(kind)(q, k, v, do, 0.8, True)
    fq, fk, fv = _finite_diff(q, k, v, do, 0.8, True)
    err = max(np.abs(dq - fq).max(), np.abs(dk - fk).max(), np.abs(dv - fv).max())
    assert err > 1e-4
    # and the unmutated form passes the same check
    dq, dk, dv = _mutant("none")(q, k, v, do, 0.8, True)
    assert max(np.abs(dq - fq).max(), np.abs(dk - fk).max(), np.abs(dv - fv).max()) < 1e-7
