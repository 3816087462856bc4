"""Parity of the CUDA path against the fp64 oracle, element by element.

Small shapes are compared in full (they span several 128-row tiles and a
ragged tail); the full-size workloads are compared on sampled rows that the
oracle computes one by one (row 0, tile edges, the last rows, random rows).
"""

import os

import numpy as np
import pytest

import oracle
from exact_io_aware_107_b300 import workloads as W
from gpu_util import (BF16_TOL_LSE, BF16_TOL_O, F16_TOL_LSE, F16_TOL_O, F32_TOL_LSE, F32_TOL_O,
                      max_err, run_cuda)

pytestmark = pytest.mark.gpu


def _full_compare(w, tol_o, tol_lse):
    x = W.generate(w)
    o, lse = run_cuda(x["q"], x["k"], x["v"], w.causal, w.scale, x["cu_seqlens"])
    ro, rl = oracle.attention(W.as_f64(x["q"]), W.as_f64(x["k"]), W.as_f64(x["v"]), w.scale,
                              w.causal, cu_seqlens=x["cu_seqlens"])
    eo, el = max_err(o, ro), max_err(lse, rl)
    assert eo <= tol_o and el <= tol_lse, (w, eo, el)
    return eo, el


# ---------------------------------------------------------------- fp32 path

def test_f32_config_exact_small():
    w = W.WORKLOADS["f32_causal_b2_h4_n128_d64"]
    _full_compare(w, F32_TOL_O, F32_TOL_LSE)


@pytest.mark.parametrize("N", [1, 2, 31, 32, 33, 100, 257])
@pytest.mark.parametrize("D", [16, 64, 100, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_f32_sweep(N, D, causal):
    w = W.custom("f32", B=2, H=2, N=N, D=D, causal=causal, seed=N * 31 + D)
    _full_compare(w, F32_TOL_O, F32_TOL_LSE)


@pytest.mark.parametrize("causal", [False, True])
def test_f32_varlen(causal):
    w = W.custom("f32", H=3, D=64, causal=causal, seed=5, varlen=[1, 31, 32, 33, 90, 7])
    _full_compare(w, F32_TOL_O, F32_TOL_LSE)


# ---------------------------------------------------------------- bf16 path

@pytest.mark.parametrize("N", [1, 2, 3, 7, 8, 127, 128, 129, 255, 256, 257, 300, 511, 700])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_sweep(N, D, causal):
    w = W.custom("bf16", B=1, H=2, N=N, D=D, causal=causal, seed=N * 7 + D)
    _full_compare(w, BF16_TOL_O, BF16_TOL_LSE)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_multi_batch_head(D, causal):
    w = W.custom("bf16", B=3, H=5, N=600, D=D, causal=causal, seed=17)
    _full_compare(w, BF16_TOL_O, BF16_TOL_LSE)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_bf16_varlen_small(causal, D):
    lens = [1, 127, 128, 129, 300, 513, 7, 256, 257]
    w = W.custom("bf16", H=3, D=D, causal=causal, seed=9, varlen=lens)
    _full_compare(w, BF16_TOL_O, BF16_TOL_LSE)


@pytest.mark.parametrize("nseq", [256, 300])
def test_bf16_varlen_many_sequences(nseq):
    # up to 256 sequences are taken longest first (sorted inside the kernel);
    # more are taken in the order given: both orders against the oracle
    rng = np.random.default_rng(nseq)
    lens = rng.integers(0, 700, nseq).tolist()
    lens[::37] = [0] * len(lens[::37])                  # some empty sequences
    w = W.custom("bf16", H=2, D=64, causal=True, seed=nseq, varlen=lens)
    _full_compare(w, BF16_TOL_O, BF16_TOL_LSE)


def test_bf16_peaked_small():
    # Q, K ~ N(0, 2^2): scores with std 4, rows near one-hot, many reference-max moves
    w = W.custom("bf16", B=1, H=4, N=1500, D=128, causal=True, seed=3, qk_std=2.0)
    _full_compare(w, BF16_TOL_O, BF16_TOL_LSE)


def test_bf16_growing_max_forces_rescale():
    # scores grow along the key axis so the running max keeps rising by more
    # than the lazy-rescale threshold from tile to tile
    import torch
    N, D = 1024, 128
    rng = np.random.default_rng(21)
    q = rng.standard_normal((1, 2, N, D)).astype(np.float32) * 0.1
    q[..., 0] = 4.0
    k = rng.standard_normal((1, 2, N, D)).astype(np.float32) * 0.1
    k[..., 0] = np.linspace(0.0, 16.0, N, dtype=np.float32)
    v = rng.standard_normal((1, 2, N, D)).astype(np.float32)
    tq, tk, tv = (torch.from_numpy(a).to(torch.bfloat16) for a in (q, k, v))
    scale = float(np.float32(1 / np.sqrt(D)))
    for causal in (False, True):
        o, lse = run_cuda(tq, tk, tv, causal, scale)
        ro, rl = oracle.attention(W.as_f64(tq), W.as_f64(tk), W.as_f64(tv), scale, causal)
        assert max_err(o, ro) <= BF16_TOL_O and max_err(lse, rl) <= BF16_TOL_LSE


# ---------------------------------------------------------------- fp16 path

@pytest.mark.parametrize("N", [1, 7, 128, 129, 300, 700])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_f16_sweep(N, D, causal):
    w = W.custom("f16", B=1, H=2, N=N, D=D, causal=causal, seed=N * 5 + D)
    _full_compare(w, F16_TOL_O, F16_TOL_LSE)


@pytest.mark.parametrize("causal", [False, True])
def test_f16_varlen_small(causal):
    w = W.custom("f16", H=3, D=128, causal=causal, seed=19, varlen=[1, 127, 129, 300, 513])
    _full_compare(w, F16_TOL_O, F16_TOL_LSE)


def test_f16_peaked_small():
    w = W.custom("f16", B=1, H=4, N=1500, D=128, causal=True, seed=23, qk_std=2.0)
    _full_compare(w, F16_TOL_O, F16_TOL_LSE)


def test_f16_causal_b2_h32_n8192_d128_sampled():
    w = W.custom("f16", B=2, H=32, N=8192, D=128, causal=True, seed=0,
                 name="f16_causal_b2_h32_n8192_d128")
    x = W.generate(w)
    o, lse = run_cuda(x["q"], x["k"], x["v"], w.causal, w.scale)
    rng = np.random.default_rng(5)
    worst_o = worst_l = 0.0
    for b, h in ((0, 0), (1, 31), (0, 17)):
        rows = _sample_rows(w.N, rng)
        ro, rl = oracle.attention_rows(W.as_f64(x["q"][b, h]), W.as_f64(x["k"][b, h]),
                                       W.as_f64(x["v"][b, h]), w.scale, w.causal, rows)
        worst_o = max(worst_o, max_err(o[b, h][rows], ro))
        worst_l = max(worst_l, max_err(lse[b, h][rows], rl))
    assert worst_o <= F16_TOL_O and worst_l <= F16_TOL_LSE, (worst_o, worst_l)


# ---------------------------------------------------------------- the named workloads

def test_workload_bf16_b4_h16_n2048_d64_full():
    _full_compare(W.WORKLOADS["bf16_b4_h16_n2048_d64"], BF16_TOL_O, BF16_TOL_LSE)


def _sample_rows(n, rng, extra=48, target=None):
    """Row 0, the last rows, every 128-row tile edge +-1, then random rows (up
    to ``target`` rows in all when it is given)."""
    base = {0, 1, 2, n - 1, n - 2}
    for t in range(128, n, 128):
        base |= {t - 1, t, t + 1}
    base = {r for r in base if 0 <= r < n}
    if target is None:
        if len(base) > 96:
            base = set(rng.choice(sorted(base), 96, replace=False)) | {0, n - 1}
        base |= set(rng.integers(0, n, extra).tolist())
    else:
        want = min(n, target)
        rest = np.setdiff1d(np.arange(n), np.array(sorted(base)))
        if len(base) < want and len(rest):
            base |= set(rng.choice(rest, min(len(rest), want - len(base)), replace=False).tolist())
    return np.array(sorted(base))


# ---------------------------------------------------------------- every element
#
# The three large workloads are compared with the oracle on every output
# element: one fp64 plane (or packed sequence of one head) per task, on a
# thread per host core with one BLAS thread each (the oracle's matrix products
# and exponentials release the interpreter lock).  The test prints the largest
# errors and the host time.  The exact identities ride along: causal row 0 of
# every plane (and the first row of every packed sequence) is V's row 0 bit
# for bit, and every output row is a convex combination of value rows.

def _oracle_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 4


@pytest.mark.parametrize("name", ["bf16_causal_b2_h32_n8192_d128",
                                  "bf16_causal_b1_h16_n32768_d128_peaked",
                                  "bf16_varlen_causal_h32_d128"])
def test_workload_every_element(name):
    import time
    from concurrent.futures import ThreadPoolExecutor
    from oracle.threads import blas_threads
    w = W.WORKLOADS[name]
    x = W.generate(w)
    o, lse = run_cuda(x["q"], x["k"], x["v"], w.causal, w.scale, x["cu_seqlens"])
    assert not np.isnan(o).any() and not np.isnan(lse).any()
    q, k, v = (W.as_f64(t) for t in (x["q"], x["k"], x["v"]))
    if w.varlen is None:
        jobs = [((b, h), q[b, h], k[b, h], v[b, h]) for b in range(w.B) for h in range(w.H)]
        np.testing.assert_array_equal(o[:, :, 0], v[:, :, 0])
    else:
        cu = x["cu_seqlens"]
        jobs = [((h, slice(int(cu[s]), int(cu[s + 1]))), q[h, cu[s]:cu[s + 1]],
                 k[h, cu[s]:cu[s + 1]], v[h, cu[s]:cu[s + 1]])
                for s in range(len(w.varlen)) for h in range(w.H)]
        for s in range(len(cu) - 1):
            np.testing.assert_array_equal(o[:, cu[s]], v[:, cu[s]])
    assert float(np.abs(o).max()) <= float(np.abs(v).max()) + BF16_TOL_O
    # heaviest jobs first, so that the last ones to finish are short
    jobs.sort(key=lambda j: -j[1].shape[0] * j[2].shape[0])

    def one(job):
        idx, qp, kp, vp = job
        ro, rl = oracle.attention_plane(qp, kp, vp, w.scale, w.causal)
        return max_err(o[idx], ro), max_err(lse[idx], rl)

    t0 = time.perf_counter()
    with blas_threads(1):
        with ThreadPoolExecutor(max_workers=_oracle_threads()) as ex:
            errs = list(ex.map(one, jobs))
    secs = time.perf_counter() - t0
    eo = max(e[0] for e in errs)
    el = max(e[1] for e in errs)
    print(f"every element of {name}: max|dO| = {eo:.3e}, max|dLSE| = {el:.3e} over {o.size} "
          f"outputs in {len(jobs)} planes ({secs:.1f} s of oracle on {_oracle_threads()} threads)")
    assert eo <= BF16_TOL_O and el <= BF16_TOL_LSE, (name, eo, el)


# ---------------------------------------------------------------- size limits
#
# One long plane (2^18 rows causal; a ragged 200003 rows non-causal) on sampled
# rows, and many short planes (4096 of them) on every row of a subset: the
# index arithmetic at the far end of the row and plane ranges.

@pytest.mark.parametrize("N,D,causal", [(262144, 128, True), (200003, 64, False)])
def test_long_plane_sampled(N, D, causal):
    w = W.custom("bf16", B=1, H=1, N=N, D=D, causal=causal, seed=N % 97)
    x = W.generate(w)
    o, lse = run_cuda(x["q"], x["k"], x["v"], causal, w.scale)
    assert not np.isnan(o).any() and not np.isnan(lse).any()
    rows = _sample_rows(N, np.random.default_rng(5), extra=48)
    rows = np.union1d(rows, np.arange(N - 130, N))  # the whole last tile and its edge
    q, k, v = (W.as_f64(t[0, 0]) for t in (x["q"], x["k"], x["v"]))
    ro, rl = oracle.attention_rows(q, k, v, w.scale, causal, rows)
    eo, el = max_err(o[0, 0][rows], ro), max_err(lse[0, 0][rows], rl)
    assert eo <= BF16_TOL_O and el <= BF16_TOL_LSE, (N, eo, el)
    if causal:
        np.testing.assert_array_equal(o[0, 0, 0], v[0])


@pytest.mark.parametrize("N", [1280, 1100])
@pytest.mark.parametrize("causal", [False, True])
def test_many_planes_several_blocks_every_element(N, causal):
    # 160 planes of 5 blocks of 256 rows over the 148 persistent CTAs, every
    # plane compared in full.  Causal: 330 mirror pairs of 110 planes, then
    # the 250 single blocks of the last 50, handed out by the launch's work
    # counter; non-causal: 800 single blocks in static rounds, the last one
    # split into query tiles
    from concurrent.futures import ThreadPoolExecutor
    from oracle.threads import blas_threads
    B, H, D = 4, 40, 128
    w = W.custom("bf16", B=B, H=H, N=N, D=D, causal=causal, seed=N + causal)
    x = W.generate(w)
    o, lse = run_cuda(x["q"], x["k"], x["v"], causal, w.scale)
    q, k, v = (W.as_f64(t) for t in (x["q"], x["k"], x["v"]))

    def one(bh):
        b, h = bh
        ro, rl = oracle.attention_plane(q[b, h], k[b, h], v[b, h], w.scale, causal)
        return max_err(o[b, h], ro), max_err(lse[b, h], rl)

    with blas_threads(1):
        with ThreadPoolExecutor(max_workers=_oracle_threads()) as ex:
            errs = list(ex.map(one, [(b, h) for b in range(B) for h in range(H)]))
    eo, el = max(e[0] for e in errs), max(e[1] for e in errs)
    assert eo <= BF16_TOL_O and el <= BF16_TOL_LSE, (N, causal, eo, el)


@pytest.mark.parametrize("causal", [False, True])
def test_many_planes(causal):
    B, H, N, D = 64, 64, 80, 128
    w = W.custom("bf16", B=B, H=H, N=N, D=D, causal=causal, seed=17)
    x = W.generate(w)
    o, lse = run_cuda(x["q"], x["k"], x["v"], causal, w.scale)
    rng = np.random.default_rng(6)
    picks = {(0, 0), (B - 1, H - 1), (B - 1, 0), (0, H - 1)}
    picks |= {(int(b), int(h)) for b, h in zip(rng.integers(0, B, 12), rng.integers(0, H, 12))}
    for b, h in sorted(picks):
        ro, rl = oracle.attention_plane(W.as_f64(x["q"][b, h]), W.as_f64(x["k"][b, h]),
                                        W.as_f64(x["v"][b, h]), w.scale, causal)
        eo, el = max_err(o[b, h], ro), max_err(lse[b, h], rl)
        assert eo <= BF16_TOL_O and el <= BF16_TOL_LSE, (b, h, eo, el)


# ---------------------------------------------------------------- scale extremes
#
# A tiny scale makes every row nearly uniform (LSE -> ln of the key count); a
# large one makes rows one-hot, with most exponentials underflowing to zero and
# a new row maximum far above the old one in many tiles.  Both are compared with
# the oracle on every element.

@pytest.mark.parametrize("scale", [1e-3, 2.0])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("f16", 128), ("f32", 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_extreme_scales(scale, dtype, D, causal):
    w = W.custom(dtype, B=1, H=2, N=700, D=D, causal=causal, seed=23)
    x = W.generate(w)
    o, lse = run_cuda(x["q"], x["k"], x["v"], causal, scale)
    ro, rl = oracle.attention(W.as_f64(x["q"]), W.as_f64(x["k"]), W.as_f64(x["v"]), scale, causal)
    tol_o, tol_l = {"bf16": (BF16_TOL_O, BF16_TOL_LSE), "f16": (F16_TOL_O, F16_TOL_LSE),
                    "f32": (F32_TOL_O, F32_TOL_LSE)}[dtype]
    eo, el = max_err(o, ro), max_err(lse, rl)
    assert eo <= tol_o and el <= tol_l, (scale, dtype, D, causal, eo, el)
