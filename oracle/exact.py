"""fp64 CPU oracle for the exact attention forward (test infrastructure only).

This module is the correctness reference for the CUDA path.  Only the tests,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference legs of
``bench.py`` may import it; the product path never does.  It shares no code
with the CUDA library: it imports numpy alone.

What it computes
----------------
For one attention plane (one (batch, head) pair, or one packed sequence of
one head) with queries q_i, keys k_j and values v_j, and the allowed key set
J(i) = {j : j <= i + (Nk - Nq)} when causal (j <= i for self-attention),
else every key:

    s_ij   = scale * sum_d q_id k_jd                          (j in J(i))
    m_i    = max_j s_ij
    p_ij   = exp(s_ij - m_i) / sum_j' exp(s_ij' - m_i)
    O_i    = sum_j p_ij v_j
    LSE_i  = m_i + ln sum_j exp(s_ij - m_i)

Sources
-------
* The materialised form ``softmax(Q K^T / sqrt(d)) V`` with the max
  subtracted before ``exp``: "Building a FlashAttention-2 forward kernel in
  pure NumPy", section "Step 2: Naive attention as the reference"; the same
  matmul -> mask -> softmax -> matmul chain is "Build a FlashAttention kernel
  from scratch with Python and NumPy", sections "Step 3" to "Step 5".
* The causal mask keeps the diagonal (j <= i).  That page's comment says the
  lower triangle *including* the diagonal is kept while its printed ``np.tri``
  call drops it; the comment, the decoder reading of "Causal Masking and
  Incremental Decoding" ("Python Attention Mechanisms Explained: From
  Self-Attention to Flash Attention") and the requirement that row 0 is
  defined all agree on j <= i, so that is the reading taken.
* LSE: the invariant ``l * exp(m) = sum exp(scores seen)`` of the FA-2 page,
  section "Step 3: Online softmax core", read as LSE = m + ln l with natural
  log of the scaled, masked scores.
* Row slabs for long sequences: the row-block form of the first page's
  "Step 6" (full-row softmax per query block); it is still the plain
  definition above, not an online update.
* ``online_tiled`` restates the online-softmax update rule of the FA-2 page
  ("Architecture Overview" bullets and "Step 3"/"Step 4"), in the
  query-tile-outer, key/value-streamed order of "Hands-on build guide: tiled
  self-attention kernel with online softmax in pure NumPy" ("Architecture
  Overview", steps 1-3).  It is used only to check that the tiled form equals
  the materialised one.

Cross-attention (fewer or more query rows than keys) uses the causal
reading where the queries are the last Nq positions of an Nk-long sequence:
key j is allowed for query i when j <= i + (Nk - Nq).  The pages mention
cross-attention (Nq != Nk) without a mask convention ("Python Attention
Mechanisms Explained", "The Core Idea"); this bottom-right alignment makes a
cross call on the last Nq queries equal the last Nq rows of self-attention.
A row with no allowed key has O = 0 and LSE = -inf.

The backward pass (dQ, dK, dV for an upstream gradient dO) is the plain
gradient of the same definition; see the section "Backward pass" below.

Layouts match the CUDA boundary: dense tensors are (B, H, N, D); packed
variable-length tensors are (H, N_total, D) with ``cu_seqlens`` of length
nseq+1, each sequence attending only to itself with positions relative to its
own start.
"""

from __future__ import annotations

import numpy as np

# Rows per slab when a full N x N score matrix would be too large.
SLAB_ROWS = 512
FULL_MATRIX_MAX_N = 4096


def _plane_rows(qp, kp, vp, scale, causal, r0, r1, offset=0):
    """O and LSE of query rows [r0, r1) of one plane, materialising those score rows.

    Causal: key j is allowed for query i when j <= i + offset.
    """
    n_keys = kp.shape[0]
    kmax = max(0, min(n_keys, r1 + offset)) if causal else n_keys   # later keys are masked
    o = np.zeros((r1 - r0, vp.shape[1]))
    lse = np.full(r1 - r0, -np.inf)
    if kmax == 0:
        return o, lse
    s = scale * (qp[r0:r1] @ kp[:kmax].T)                 # (rows, kmax) fp64
    if causal:
        i = np.arange(r0, r1)[:, None]
        j = np.arange(kmax)[None, :]
        s = np.where(j <= i + offset, s, -np.inf)
    live = np.isfinite(s).any(axis=1)                     # rows with at least one allowed key
    sl = s[live]
    m = sl.max(axis=1, keepdims=True)
    e = np.exp(sl - m)
    l = e.sum(axis=1, keepdims=True)
    o[live] = (e / l) @ vp[:kmax]
    lse[live] = m[:, 0] + np.log(l[:, 0])
    return o, lse


def attention_plane(qp, kp, vp, scale, causal, offset=None):
    """Naive materialised attention for one plane in fp64.

    qp: (Nq, D), kp: (Nk, D), vp: (Nk, Dv).  The causal offset defaults to
    Nk - Nq (0 for self-attention).
    """
    qp, kp, vp = (np.asarray(a, dtype=np.float64) for a in (qp, kp, vp))
    n = qp.shape[0]
    if offset is None:
        offset = kp.shape[0] - n
    o = np.empty((n, vp.shape[1]), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    if n == 0:
        return o, lse
    step = n if n <= FULL_MATRIX_MAX_N else SLAB_ROWS
    for r0 in range(0, n, step):
        r1 = min(n, r0 + step)
        o[r0:r1], lse[r0:r1] = _plane_rows(qp, kp, vp, scale, causal, r0, r1, offset)
    return o, lse


def _planes(q, k, v, cu_seqlens, cu_seqlens_k):
    """Yield (index, q-plane, k-plane, v-plane) views for dense or packed layouts."""
    if cu_seqlens is None:
        B, H = q.shape[0], q.shape[1]
        for b in range(B):
            for h in range(H):
                yield (b, h, slice(None)), q[b, h], k[b, h], v[b, h]
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        cuk = cu if cu_seqlens_k is None else np.asarray(cu_seqlens_k, dtype=np.int64)
        H = q.shape[0]
        for s in range(len(cu) - 1):
            a, e = int(cu[s]), int(cu[s + 1])
            ak, ek = int(cuk[s]), int(cuk[s + 1])
            for h in range(H):
                yield (None, h, slice(a, e)), q[h, a:e], k[h, ak:ek], v[h, ak:ek]


def attention(q, k, v, scale, causal, cu_seqlens=None, cu_seqlens_k=None):
    """Exact attention forward in fp64.

    q, k, v: float arrays, (B, H, N, D) dense or (H, N_total, D) packed; k and
    v may hold a different number of rows (Nk) than q, and in the packed form
    their own offsets ``cu_seqlens_k`` (default: ``cu_seqlens``).
    Returns (O, LSE): O with q's shape, LSE with q's shape minus the last axis.
    """
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    o = np.empty(q.shape[:-1] + (v.shape[-1],), dtype=np.float64)
    lse = np.empty(q.shape[:-1], dtype=np.float64)
    for (b, h, sl), qp, kp, vp in _planes(q, k, v, cu_seqlens, cu_seqlens_k):
        po, pl = attention_plane(qp, kp, vp, scale, causal)
        if b is None:
            o[h, sl], lse[h, sl] = po, pl
        else:
            o[b, h], lse[b, h] = po, pl
    return o, lse


def attention_rows(qp, kp, vp, scale, causal, rows, offset=None):
    """O and LSE for selected query rows of one plane (same definition, row by row).

    Used to check full-size outputs on a sample of rows.
    """
    qp, kp, vp = (np.asarray(a, dtype=np.float64) for a in (qp, kp, vp))
    if offset is None:
        offset = kp.shape[0] - qp.shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    o = np.empty((len(rows), vp.shape[1]), dtype=np.float64)
    lse = np.empty(len(rows), dtype=np.float64)
    for t, r in enumerate(rows):
        o[t:t + 1], lse[t:t + 1] = _plane_rows(qp, kp, vp, scale, causal, int(r), int(r) + 1,
                                               offset)
    return o, lse


def softmax_probs(qp, kp, scale, causal):
    """The materialised probability matrix P of one plane (for the row-sum pin)."""
    qp, kp = (np.asarray(a, dtype=np.float64) for a in (qp, kp))
    s = scale * (qp @ kp.T)
    if causal:
        n, nk = s.shape
        s = np.where(np.arange(nk)[None, :] <= np.arange(n)[:, None] + (nk - n), s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=1, keepdims=True)


def online_tiled(qp, kp, vp, scale, causal, br=128, bc=128):
    """Tiled forward with the online-softmax update, fp64, for one plane.

    Query tiles are outer; key/value tiles stream past each one.  Per query
    row the state is a running max m, a running sum l (so that l * exp(m)
    is the sum of exp over the scores seen so far) and an unnormalised output
    accumulator.  For each key tile: m_new = max(m, rowmax S); alpha =
    exp(m - m_new); l = alpha * l + rowsum exp(S - m_new); acc = alpha * acc
    + exp(S - m_new) @ V_tile.  At the end O = acc / l and LSE = m + ln l.
    """
    qp, kp, vp = (np.asarray(a, dtype=np.float64) for a in (qp, kp, vp))
    n, nk, dv = qp.shape[0], kp.shape[0], vp.shape[1]
    off = nk - n                                  # causal alignment of the last query to the last key
    o = np.empty((n, dv))
    lse = np.empty(n)
    for i0 in range(0, n, br):
        i1 = min(n, i0 + br)
        m = np.full(i1 - i0, -np.inf)
        l = np.zeros(i1 - i0)
        acc = np.zeros((i1 - i0, dv))
        kend = max(0, min(nk, i1 + off)) if causal else nk
        for j0 in range(0, kend, bc):
            j1 = min(kend, j0 + bc)
            s = scale * (qp[i0:i1] @ kp[j0:j1].T)
            if causal:
                s = np.where(np.arange(j0, j1)[None, :] <= np.arange(i0, i1)[:, None] + off,
                             s, -np.inf)
            m_new = np.maximum(m, s.max(axis=1))
            # a row whose keys in this tile are all masked and that has seen
            # nothing yet keeps m = -inf; exp(-inf - -inf) would be NaN
            ref = np.where(np.isfinite(m_new), m_new, 0.0)
            alpha = np.exp(m - ref)
            p = np.exp(s - ref[:, None])
            l = alpha * l + p.sum(axis=1)
            acc = alpha[:, None] * acc + p @ vp[j0:j1]
            m = m_new
        live = l > 0                              # rows that saw no allowed key: O = 0, LSE = -inf
        o[i0:i1] = np.where(live[:, None], acc / np.where(live, l, 1.0)[:, None], 0.0)
        lse[i0:i1] = np.where(live, m + np.log(np.where(live, l, 1.0)), -np.inf)
    return o, lse


# ---------------------------------------------------------------------------
# Backward pass
# ---------------------------------------------------------------------------
#
# The pages name the backward pass as the next extension of the forward
# kernel: keep the forward's softmax statistics and output, and rebuild the
# probabilities tile by tile while the gradients stream back ("Building a
# FlashAttention-2 forward kernel in pure NumPy", section "Extending It: Your
# Roadmap to Senior-Level").  What it computes is the plain gradient of the forward
# above for a scalar loss whose gradient with respect to O is dO:
#
#     dV   = P^T dO
#     dP   = dO V^T
#     dS   = P * (dP - Delta),   Delta_i = sum_j P_ij dP_ij = dO_i . O_i
#     dQ   = scale * dS K
#     dK   = scale * dS^T Q
#
# (the softmax Jacobian applied row by row; masked entries have P = 0 and so
# dS = 0; a query with no allowed key has a constant O = 0 and contributes
# nothing).  The oracle materialises P from the definition, as the forward
# does; it is pinned by central finite differences of the forward and by
# the identities sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i.


def _probs_rows(qp, kp, scale, causal, offset, r0, r1):
    """Rows [r0, r1) of the probability matrix P of one plane (zeros for rows with no key)."""
    n_keys = kp.shape[0]
    s = scale * (qp[r0:r1] @ kp.T)
    if causal:
        i = np.arange(r0, r1)[:, None]
        j = np.arange(n_keys)[None, :]
        s = np.where(j <= i + offset, s, -np.inf)
    p = np.zeros_like(s)
    live = np.isfinite(s).any(axis=1) if n_keys else np.zeros(r1 - r0, dtype=bool)
    if live.any():
        sl = s[live]
        e = np.exp(sl - sl.max(axis=1, keepdims=True))
        p[live] = e / e.sum(axis=1, keepdims=True)
    return p


def attention_backward_plane(qp, kp, vp, dop, scale, causal, offset=None):
    """dQ, dK, dV of one plane in fp64 (qp, dop: (Nq, D); kp, vp: (Nk, D)).

    Long planes are processed in query-row slabs; every slab's contribution
    to dK and dV is summed, which is the same matrix product split by rows.
    """
    qp, kp, vp, dop = (np.asarray(a, dtype=np.float64) for a in (qp, kp, vp, dop))
    n = qp.shape[0]
    if offset is None:
        offset = kp.shape[0] - n
    dq = np.zeros_like(qp)
    dk = np.zeros_like(kp)
    dv = np.zeros_like(vp)
    step = max(1, n if n <= FULL_MATRIX_MAX_N else SLAB_ROWS)
    for r0 in range(0, n, step):
        r1 = min(n, r0 + step)
        p = _probs_rows(qp, kp, scale, causal, offset, r0, r1)     # (rows, Nk)
        o = p @ vp
        dv += p.T @ dop[r0:r1]
        dp = dop[r0:r1] @ vp.T
        delta = (dop[r0:r1] * o).sum(axis=1, keepdims=True)
        ds = p * (dp - delta)
        dq[r0:r1] = scale * (ds @ kp)
        dk += scale * (ds.T @ qp[r0:r1])
    return dq, dk, dv


def attention_backward(q, k, v, do, scale, causal, cu_seqlens=None, cu_seqlens_k=None):
    """dQ, dK, dV in fp64 for dense (B, H, N, D) or packed (H, N_total, D) tensors
    (the layouts of :func:`attention`)."""
    q, k, v, do = (np.asarray(a, dtype=np.float64) for a in (q, k, v, do))
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    if cu_seqlens is None:
        for b in range(q.shape[0]):
            for h in range(q.shape[1]):
                dq[b, h], dk[b, h], dv[b, h] = attention_backward_plane(
                    q[b, h], k[b, h], v[b, h], do[b, h], scale, causal)
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        cuk = cu if cu_seqlens_k is None else np.asarray(cu_seqlens_k, dtype=np.int64)
        for s in range(len(cu) - 1):
            a, e, ak, ek = int(cu[s]), int(cu[s + 1]), int(cuk[s]), int(cuk[s + 1])
            for h in range(q.shape[0]):
                dq[h, a:e], dk[h, ak:ek], dv[h, ak:ek] = attention_backward_plane(
                    q[h, a:e], k[h, ak:ek], v[h, ak:ek], do[h, a:e], scale, causal)
    return dq, dk, dv
