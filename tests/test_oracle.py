"""Pins for the fp64 oracle: closed forms, invariants and brute force.

Each check fixes the oracle against something other than itself, so that a
plausible slip (a dropped scale, a causal mask that drops or flips the
diagonal, a transposed operand, a wrong log base, a missing max shift, an
off-by-one in the slab loop) fails at least one of them.  ``test_mutants_are_caught``
plants exactly those slips in copies of the oracle and checks that the pins
reject every one.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import exact as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


# ---------------------------------------------------------------------------
# Individual pins, written as functions of an attention implementation so the
# same checks can be run against planted mistakes.
# ---------------------------------------------------------------------------

def pin_golden(fn):
    """Hand-derived three-token example with rational probabilities."""
    fx = json.load(open(os.path.join(GOLDEN, "closed_form_n3_d2.json")))
    q, k, v = (np.array(fx[n]) for n in ("q", "k", "v"))
    for causal, key in ((True, "causal"), (False, "noncausal")):
        o, lse = fn(q, k, v, fx["scale"], causal)
        np.testing.assert_allclose(o, np.array(fx[key]["o"]), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse, np.array(fx[key]["lse"]), rtol=0, atol=1e-14)


def pin_brute_force(fn):
    """Scalar loops with math.exp / math.fsum on tiny shapes, independent of numpy BLAS."""
    rng = np.random.default_rng(11)
    for n in (1, 2, 3, 5, 8):
        for d in (1, 2, 4):
            q, k, v = _rand(rng, n, d), _rand(rng, n, d), _rand(rng, n, d)
            scale = 0.7
            for causal in (False, True):
                o, lse = fn(q, k, v, scale, causal)
                for i in range(n):
                    keys = range(i + 1) if causal else range(n)
                    s = [scale * math.fsum(q[i, t] * k[j, t] for t in range(d)) for j in keys]
                    mx = max(s)
                    e = [math.exp(x - mx) for x in s]
                    den = math.fsum(e)
                    for t in range(d):
                        ref = math.fsum(e[c] * v[j, t] for c, j in enumerate(keys)) / den
                        assert abs(o[i, t] - ref) <= 1e-13 * (1 + abs(ref)), (n, d, causal, i, t)
                    assert abs(lse[i] - (mx + math.log(den))) <= 1e-13 * (1 + abs(mx)), (n, d, i)


def pin_causal_row0(fn):
    """Causal row 0 sees only key 0: O_0 = V_0, LSE_0 = scale * q_0 . k_0."""
    rng = np.random.default_rng(3)
    q, k, v = _rand(rng, 40, 16), _rand(rng, 40, 16), _rand(rng, 40, 16)
    o, lse = fn(q, k, v, 0.25, True)
    np.testing.assert_array_equal(o[0], v[0])
    assert abs(lse[0] - 0.25 * math.fsum(q[0] * k[0])) < 1e-14


def pin_zero_query(fn):
    """Q = 0 makes every allowed score 0: O is the (prefix) mean of V, LSE = ln(count)."""
    rng = np.random.default_rng(4)
    n, d = 37, 8
    q = np.zeros((n, d))
    k, v = _rand(rng, n, d), _rand(rng, n, d)
    o, lse = fn(q, k, v, 0.3, True)
    counts = np.arange(1, n + 1)[:, None]
    np.testing.assert_allclose(o, np.cumsum(v, axis=0) / counts, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.log(np.arange(1, n + 1)), rtol=0, atol=1e-14)
    o, lse = fn(q, k, v, 0.3, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=0), o.shape), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.full(n, math.log(n)), rtol=0, atol=1e-14)


def pin_value_ones(fn):
    rng = np.random.default_rng(5)
    q, k = _rand(rng, 33, 8), _rand(rng, 33, 8)
    for causal in (False, True):
        o, _ = fn(q, k, np.ones((33, 8)), 0.5, causal)
        np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-14)


def pin_permutation(fn):
    """Non-causal: permuting K and V rows together changes nothing."""
    rng = np.random.default_rng(6)
    q, k, v = _rand(rng, 29, 8), _rand(rng, 29, 8), _rand(rng, 29, 8)
    perm = rng.permutation(29)
    o1, l1 = fn(q, k, v, 0.4, False)
    o2, l2 = fn(q, k[perm], v[perm], 0.4, False)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def pin_key_shift(fn):
    """K_j -> K_j + u: every score of row i moves by scale*q_i.u, so O is unchanged
    and LSE_i moves by exactly that amount (the softmax shift invariance)."""
    rng = np.random.default_rng(7)
    q, k, v = _rand(rng, 31, 8), _rand(rng, 31, 8), _rand(rng, 31, 8)
    u = _rand(rng, 8)
    for causal in (False, True):
        o1, l1 = fn(q, k, v, 0.35, causal)
        o2, l2 = fn(q, k + u, v, 0.35, causal)
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l2 - l1, 0.35 * (q @ u), rtol=0, atol=1e-12)


def pin_causality(fn):
    """Causal: changing keys/values j > i leaves row i untouched (bit for bit)."""
    rng = np.random.default_rng(8)
    n = 50
    q, k, v = _rand(rng, n, 8), _rand(rng, n, 8), _rand(rng, n, 8)
    o1, l1 = fn(q, k, v, 0.3, True)
    i = 20
    k2, v2 = k.copy(), v.copy()
    k2[i + 1:] = _rand(rng, n - i - 1, 8) * 5
    v2[i + 1:] = _rand(rng, n - i - 1, 8) * 5
    o2, l2 = fn(q, k2, v2, 0.3, True)
    np.testing.assert_allclose(o1[:i + 1], o2[:i + 1], rtol=0, atol=1e-14)
    np.testing.assert_allclose(l1[:i + 1], l2[:i + 1], rtol=0, atol=1e-14)
    assert np.abs(o1[i + 1:] - o2[i + 1:]).max() > 1e-3


def pin_large_scores(fn):
    """Scores near +-700 overflow exp unless the row max is subtracted first."""
    rng = np.random.default_rng(9)
    q, k, v = _rand(rng, 16, 4), _rand(rng, 16, 4), _rand(rng, 16, 4)
    o1, l1 = fn(q, k, v, 0.5, False)
    q2 = q * 400.0
    o2, l2 = fn(q2, k, v, 0.5 / 400.0, False)      # identical scores, bigger operands
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    big = np.zeros((16, 4))
    big[:, 0] = 900.0
    kk = np.ones((16, 4))
    o3, l3 = fn(big, kk, v, 1.0, False)            # every score 900: uniform weights
    assert np.all(np.isfinite(o3)) and np.all(np.isfinite(l3))
    np.testing.assert_allclose(o3, np.broadcast_to(v.mean(axis=0), o3.shape), atol=1e-12)
    np.testing.assert_allclose(l3, 900.0 + math.log(16), rtol=0, atol=1e-10)


ALL_PINS = [pin_golden, pin_brute_force, pin_causal_row0, pin_zero_query, pin_value_ones,
            pin_permutation, pin_key_shift, pin_causality, pin_large_scores]


def _oracle_plane(q, k, v, scale, causal):
    return A.attention_plane(q, k, v, scale, causal)


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pins(pin):
    pin(_oracle_plane)


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_online_tiled_pins(pin):
    pin(lambda q, k, v, s, c: A.online_tiled(q, k, v, s, c, br=4, bc=3))


# ---------------------------------------------------------------------------
# Structural checks of the oracle's own code paths
# ---------------------------------------------------------------------------

def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(1)
    for causal in (False, True):
        p = A.softmax_probs(_rand(rng, 70, 16), _rand(rng, 70, 16), 0.25, causal)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
        if causal:
            assert np.all(np.triu(p, 1) == 0.0)
            assert np.all(np.diag(p) > 0)


@pytest.mark.parametrize("n", [1, 2, 3, 17, 128, 129, 300])
@pytest.mark.parametrize("tile", [1, 16, 32, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_online_tiled_equals_materialised(n, tile, causal):
    if tile == 1 and n > 129:
        pytest.skip("tile 1 at n=300 is slow and adds nothing")
    rng = np.random.default_rng(n * 7 + tile)
    q, k, v = _rand(rng, n, 16), _rand(rng, n, 16), _rand(rng, n, 16)
    o1, l1 = A.attention_plane(q, k, v, 0.25, causal)
    o2, l2 = A.online_tiled(q, k, v, 0.25, causal, br=tile, bc=tile)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def test_slab_path_equals_full_matrix(monkeypatch):
    rng = np.random.default_rng(2)
    n = 1100
    q, k, v = _rand(rng, n, 8), _rand(rng, n, 8), _rand(rng, n, 8)
    for causal in (False, True):
        o1, l1 = A.attention_plane(q, k, v, 0.3, causal)
        monkeypatch.setattr(A, "FULL_MATRIX_MAX_N", 100)
        monkeypatch.setattr(A, "SLAB_ROWS", 97)        # ragged slabs
        o2, l2 = A.attention_plane(q, k, v, 0.3, causal)
        monkeypatch.undo()
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
        np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def test_attention_rows_equal_plane():
    rng = np.random.default_rng(12)
    n = 300
    q, k, v = _rand(rng, n, 8), _rand(rng, n, 8), _rand(rng, n, 8)
    rows = [0, 1, 127, 128, 129, 299]
    for causal in (False, True):
        o, l = A.attention_plane(q, k, v, 0.3, causal)
        o2, l2 = A.attention_rows(q, k, v, 0.3, causal, rows)
        np.testing.assert_allclose(o[rows], o2, rtol=0, atol=1e-14)
        np.testing.assert_allclose(l[rows], l2, rtol=0, atol=1e-14)


def test_varlen_equals_per_sequence_dense():
    rng = np.random.default_rng(13)
    lens = [1, 5, 130, 64]
    cu = np.concatenate([[0], np.cumsum(lens)])
    H, D = 3, 8
    q, k, v = (_rand(rng, H, cu[-1], D) for _ in range(3))
    o, lse = A.attention(q, k, v, 0.3, True, cu_seqlens=cu)
    for s in range(len(lens)):
        a, e = cu[s], cu[s + 1]
        od, ld = A.attention(q[None, :, a:e], k[None, :, a:e], v[None, :, a:e], 0.3, True)
        np.testing.assert_array_equal(o[:, a:e], od[0])
        np.testing.assert_array_equal(lse[:, a:e], ld[0])
        # first row of each sequence is its own first value row
        np.testing.assert_array_equal(o[:, a], v[:, a])


def test_dense_batch_layout():
    rng = np.random.default_rng(14)
    q, k, v = (_rand(rng, 2, 3, 20, 4) for _ in range(3))
    o, lse = A.attention(q, k, v, 0.5, True)
    assert o.shape == (2, 3, 20, 4) and lse.shape == (2, 3, 20)
    for b in range(2):
        for h in range(3):
            op, lp = A.attention_plane(q[b, h], k[b, h], v[b, h], 0.5, True)
            np.testing.assert_array_equal(o[b, h], op)
            np.testing.assert_array_equal(lse[b, h], lp)


def test_single_token_closed_form():
    rng = np.random.default_rng(15)
    q, k, v = _rand(rng, 1, 8), _rand(rng, 1, 8), _rand(rng, 1, 8)
    for causal in (False, True):
        o, lse = A.attention_plane(q, k, v, 0.125, causal)
        np.testing.assert_array_equal(o[0], v[0])
        assert abs(lse[0] - 0.125 * math.fsum(q[0] * k[0])) < 1e-15


# ---------------------------------------------------------------------------
# Planted mistakes: each mutant must fail at least one pin.
# ---------------------------------------------------------------------------

def _mutant(kind):
    def fn(q, k, v, scale, causal):
        q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
        n = q.shape[0]
        sc = 1.0 if kind == "no_scale" else scale
        s = sc * (q @ k.T) if kind != "transpose" else sc * (k @ q.T)
        i = np.arange(n)[:, None]
        j = np.arange(n)[None, :]
        if causal:
            keep = {"no_diag": j < i, "flipped": j >= i}.get(kind, j <= i)
            if kind == "no_diag":
                keep = keep | ((i == 0) & (j == 0))      # keep row 0 defined
            s = np.where(keep, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        if kind == "no_max":
            m = np.zeros_like(m)
        e = np.exp(s - m)
        l = e.sum(axis=1, keepdims=True)
        o = (e / l) @ v
        if kind == "value_transpose":
            o = (e / l) @ v[::-1]
        lse = m[:, 0] + (np.log2(l[:, 0]) if kind == "log2" else np.log(l[:, 0]))
        if kind == "lse_no_max":
            lse = np.log(l[:, 0])
        return o, lse
    return fn


MUTANTS = ["no_scale", "transpose", "no_diag", "flipped", "no_max", "value_transpose", "log2",
           "lse_no_max"]


def test_reference_implementation_of_mutant_harness_passes():
    # the harness itself, with no mistake planted, passes every pin
    for pin in ALL_PINS:
        pin(_mutant("none"))


@pytest.mark.parametrize("kind", MUTANTS)
def test_mutants_are_caught(kind):
    fn = _mutant(kind)
    failed = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(fn)
        except (AssertionError, FloatingPointError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {kind} passed every pin"


# ---------------------------------------------------------------------------
# Rectangular (decode) form: fewer query rows than keys, no mask
# ---------------------------------------------------------------------------

def test_rectangular_noncausal_brute_force():
    rng = np.random.default_rng(31)
    for nq in (1, 2, 5):
        for nk in (1, 3, 9):
            q, k, v = _rand(rng, nq, 4), _rand(rng, nk, 4), _rand(rng, nk, 3)
            o, lse = A.attention_plane(q, k, v, 0.6, False)
            assert o.shape == (nq, 3) and lse.shape == (nq,)
            for i in range(nq):
                s = [0.6 * math.fsum(q[i, t] * k[j, t] for t in range(4)) for j in range(nk)]
                mx = max(s)
                e = [math.exp(x - mx) for x in s]
                den = math.fsum(e)
                for t in range(3):
                    ref = math.fsum(e[j] * v[j, t] for j in range(nk)) / den
                    assert abs(o[i, t] - ref) <= 1e-13 * (1 + abs(ref))
                assert abs(lse[i] - (mx + math.log(den))) <= 1e-13 * (1 + abs(mx))


def test_key_slices_merge_by_log_sum_exp():
    # The split-key form: attention over key slices, merged with weights
    # exp(LSE_c - LSE), LSE = ln sum_c exp(LSE_c), equals attention over all keys.
    rng = np.random.default_rng(32)
    q, k, v = _rand(rng, 3, 8), _rand(rng, 1000, 8), _rand(rng, 1000, 8)
    o, lse = A.attention_plane(q, k, v, 0.4, False)
    bounds = [0, 128, 129, 512, 999, 1000]
    parts = [A.attention_plane(q, k[a:b], v[a:b], 0.4, False) for a, b in zip(bounds, bounds[1:])]
    lses = np.stack([pl for _, pl in parts])
    lse_m = np.log(np.exp(lses - lses.max(0)).sum(0)) + lses.max(0)
    o_m = sum(np.exp(pl - lse_m)[:, None] * po for po, pl in parts)
    np.testing.assert_allclose(lse_m, lse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o_m, o, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Causal cross form: Nq != Nk, query i aligned to key i + (Nk - Nq)
# ---------------------------------------------------------------------------

def _brute_causal_cross(q, k, v, scale):
    nq, nk = q.shape[0], k.shape[0]
    o = np.zeros((nq, v.shape[1]))
    lse = np.full(nq, -np.inf)
    for i in range(nq):
        allowed = [j for j in range(nk) if j - (nk - nq) <= i]
        if not allowed:
            continue
        s = {j: scale * math.fsum(q[i, t] * k[j, t] for t in range(q.shape[1])) for j in allowed}
        mx = max(s.values())
        e = {j: math.exp(s[j] - mx) for j in allowed}
        den = math.fsum(e.values())
        for t in range(v.shape[1]):
            o[i, t] = math.fsum(e[j] * v[j, t] for j in allowed) / den
        lse[i] = mx + math.log(den)
    return o, lse


@pytest.mark.parametrize("nq,nk", [(1, 1), (1, 7), (3, 7), (7, 7), (9, 4), (5, 1), (4, 6)])
def test_causal_cross_brute_force(nq, nk):
    rng = np.random.default_rng(nq * 17 + nk)
    q, k, v = _rand(rng, nq, 5), _rand(rng, nk, 5), _rand(rng, nk, 3)
    o, lse = A.attention_plane(q, k, v, 0.7, True)
    ro, rl = _brute_causal_cross(q, k, v, 0.7)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-13)
    assert np.array_equal(np.isinf(lse), np.isinf(rl))
    fin = np.isfinite(rl)
    np.testing.assert_allclose(lse[fin], rl[fin], rtol=0, atol=1e-13)


def test_causal_cross_is_the_tail_of_self_attention():
    # With Nq < Nk the queries are the last Nq positions: their output equals
    # the last Nq rows of causal self-attention over all Nk positions.
    rng = np.random.default_rng(41)
    n, d = 300, 16
    q, k, v = _rand(rng, n, d), _rand(rng, n, d), _rand(rng, n, d)
    o, lse = A.attention_plane(q, k, v, 0.25, True)
    for nq in (1, 2, 129, 299):
        oc, lc = A.attention_plane(q[n - nq:], k, v, 0.25, True)
        # same arithmetic up to the BLAS blocking of a different row count
        np.testing.assert_allclose(oc, o[n - nq:], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lc, lse[n - nq:], rtol=0, atol=1e-13)


def test_causal_cross_more_queries_than_keys():
    # With Nq > Nk the first Nq - Nk queries see no key (O = 0, LSE = -inf)
    # and query Nq - Nk + t sees keys 0..t: its output is V[0] when t = 0.
    rng = np.random.default_rng(42)
    q, k, v = _rand(rng, 10, 8), _rand(rng, 4, 8), _rand(rng, 4, 8)
    o, lse = A.attention_plane(q, k, v, 0.5, True)
    assert (o[:6] == 0).all() and np.isneginf(lse[:6]).all()
    np.testing.assert_array_equal(o[6], v[0])
    assert lse[6] == pytest.approx(0.5 * float(q[6] @ k[0]), abs=1e-14)
    # the last query sees every key: the non-causal result for that row
    on, ln_ = A.attention_plane(q[9:], k, v, 0.5, False)
    np.testing.assert_allclose(o[9], on[0], rtol=0, atol=1e-14)


@pytest.mark.parametrize("nq,nk", [(1, 300), (77, 300), (300, 77), (200, 200), (130, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_online_tiled_cross_equals_materialised(nq, nk, causal):
    rng = np.random.default_rng(nq + 3 * nk)
    q, k, v = _rand(rng, nq, 8), _rand(rng, nk, 8), _rand(rng, nk, 8)
    o, lse = A.attention_plane(q, k, v, 0.35, causal)
    ot, lt = A.online_tiled(q, k, v, 0.35, causal, br=64, bc=32)
    np.testing.assert_allclose(ot, o, rtol=0, atol=1e-12)
    assert np.array_equal(np.isneginf(lt), np.isneginf(lse))
    fin = np.isfinite(lse)
    np.testing.assert_allclose(lt[fin], lse[fin], rtol=0, atol=1e-12)


def test_cross_rows_equal_plane():
    rng = np.random.default_rng(43)
    q, k, v = _rand(rng, 50, 8), _rand(rng, 180, 8), _rand(rng, 180, 8)
    o, lse = A.attention_plane(q, k, v, 0.3, True)
    rows = [0, 1, 17, 49]
    ro, rl = A.attention_rows(q, k, v, 0.3, True, rows)
    np.testing.assert_allclose(ro, o[rows], rtol=0, atol=1e-13)
    np.testing.assert_allclose(rl, lse[rows], rtol=0, atol=1e-13)


def test_packed_cross_equals_per_sequence_dense():
    rng = np.random.default_rng(44)
    lq, lk = [3, 0, 130, 5, 1], [7, 4, 100, 0, 1]
    cq, ck = np.cumsum([0] + lq), np.cumsum([0] + lk)
    H, d = 2, 8
    q, k, v = _rand(rng, H, cq[-1], d), _rand(rng, H, ck[-1], d), _rand(rng, H, ck[-1], d)
    for causal in (False, True):
        o, lse = A.attention(q, k, v, 0.3, causal, cu_seqlens=cq, cu_seqlens_k=ck)
        for s in range(len(lq)):
            for h in range(H):
                qa, qe, ka, ke = cq[s], cq[s + 1], ck[s], ck[s + 1]
                ro, rl = _brute_causal_cross(q[h, qa:qe], k[h, ka:ke], v[h, ka:ke], 0.3) if causal \
                    else A.attention_plane(q[h, qa:qe], k[h, ka:ke], v[h, ka:ke], 0.3, False)
                np.testing.assert_allclose(o[h, qa:qe], ro, rtol=0, atol=1e-12)
                assert np.array_equal(np.isneginf(lse[h, qa:qe]), np.isneginf(rl))
        # a sequence with no keys: its queries get O = 0, LSE = -inf
        assert (o[:, cq[3]:cq[4]] == 0).all() and np.isneginf(lse[:, cq[3]:cq[4]]).all()
