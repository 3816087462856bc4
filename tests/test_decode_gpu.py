"""Parity of the KV-cache decode path (attn_decode) against the fp64 oracle."""

import numpy as np
import pytest

import oracle
from exact_io_aware_107_b300 import workloads as W
from gpu_util import BF16_TOL_LSE, BF16_TOL_O, max_err

pytestmark = pytest.mark.gpu


def _draw(B, H, Nq, Nk, D, seed, qk_std=1.0):
    import torch
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, Nq, D), dtype=np.float32) * np.float32(qk_std)
    k = rng.standard_normal((B, H, Nk, D), dtype=np.float32) * np.float32(qk_std)
    v = rng.standard_normal((B, H, Nk, D), dtype=np.float32)
    return tuple(torch.from_numpy(a).to(torch.bfloat16) for a in (q, k, v))


def _run(q, k, v, scale, workspace=True):
    import torch
    from exact_io_aware_107_b300 import attention_decode, device_error
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    o = torch.full_like(dq, float("nan"))
    lse = torch.full(dq.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    ws = None if workspace else torch.empty(16, dtype=torch.uint8, device="cuda")
    attention_decode(dq, dk, dv, scale=scale, workspace=ws, out=o, lse=lse)
    assert device_error() == 0
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("Nk", [1, 127, 128, 129, 1000, 5000])
@pytest.mark.parametrize("Nq", [1, 3, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_decode_matches_oracle(Nk, Nq, D):
    q, k, v = _draw(2, 3, Nq, Nk, D, seed=Nk + 7 * Nq + D)
    scale = float(np.float32(1 / np.sqrt(D)))
    o, lse = _run(q, k, v, scale)
    ro, rl = oracle.attention(W.as_f64(q), W.as_f64(k), W.as_f64(v), scale, False)
    assert max_err(o, ro) <= BF16_TOL_O and max_err(lse, rl) <= BF16_TOL_LSE


@pytest.mark.parametrize("D", [64, 128])
def test_decode_without_workspace_agrees(D):
    q, k, v = _draw(1, 2, 2, 20000, D, seed=3)
    scale = float(np.float32(1 / np.sqrt(D)))
    o1, l1 = _run(q, k, v, scale, workspace=True)
    o2, l2 = _run(q, k, v, scale, workspace=False)
    ro, rl = oracle.attention(W.as_f64(q), W.as_f64(k), W.as_f64(v), scale, False)
    for o, l in ((o1, l1), (o2, l2)):
        assert max_err(o, ro) <= BF16_TOL_O and max_err(l, rl) <= BF16_TOL_LSE


def test_decode_peaked_scores():
    q, k, v = _draw(2, 2, 4, 3000, 128, seed=11, qk_std=2.0)
    scale = float(np.float32(1 / np.sqrt(128)))
    o, lse = _run(q, k, v, scale)
    ro, rl = oracle.attention(W.as_f64(q), W.as_f64(k), W.as_f64(v), scale, False)
    assert max_err(o, ro) <= BF16_TOL_O and max_err(lse, rl) <= BF16_TOL_LSE


def test_decode_long_cache_sampled_heads():
    # B=8, H=32, one new token against a 32768-key cache; oracle on a few heads
    q, k, v = _draw(8, 32, 1, 32768, 128, seed=0)
    scale = float(np.float32(1 / np.sqrt(128)))
    o, lse = _run(q, k, v, scale)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    for b, h in ((0, 0), (3, 17), (7, 31)):
        ro, rl = oracle.attention_plane(W.as_f64(q[b, h]), W.as_f64(k[b, h]), W.as_f64(v[b, h]),
                                        scale, False)
        assert max_err(o[b, h], ro) <= BF16_TOL_O and max_err(lse[b, h], rl) <= BF16_TOL_LSE


def test_decode_single_key_is_that_value():
    q, k, v = _draw(2, 2, 3, 1, 128, seed=4)
    o, lse = _run(q, k, v, 0.125)
    np.testing.assert_array_equal(o, np.broadcast_to(W.as_f64(v), o.shape))


# 2..8 query rows take the warp-level MMA path: every row count, both head
# dims, ragged and long caches, and the score regimes at both ends.

@pytest.mark.parametrize("Nq", [2, 4, 5, 6, 7])
@pytest.mark.parametrize("Nk", [129, 5000])
@pytest.mark.parametrize("D", [64, 128])
def test_decode_every_row_count(Nq, Nk, D):
    q, k, v = _draw(2, 2, Nq, Nk, D, seed=100 + Nq + Nk + D)
    scale = float(np.float32(1 / np.sqrt(D)))
    o, lse = _run(q, k, v, scale)
    ro, rl = oracle.attention(W.as_f64(q), W.as_f64(k), W.as_f64(v), scale, False)
    assert max_err(o, ro) <= BF16_TOL_O and max_err(lse, rl) <= BF16_TOL_LSE


@pytest.mark.parametrize("scale", [1e-3, 2.0])
@pytest.mark.parametrize("Nq", [1, 4, 8])
def test_decode_extreme_scales(scale, Nq):
    # near-uniform rows, and one-hot rows whose weight of 1 is exact in bf16
    q, k, v = _draw(2, 3, Nq, 3000, 128, seed=200 + Nq)
    o, lse = _run(q, k, v, scale)
    ro, rl = oracle.attention(W.as_f64(q), W.as_f64(k), W.as_f64(v), scale, False)
    assert max_err(o, ro) <= BF16_TOL_O and max_err(lse, rl) <= BF16_TOL_LSE


def test_decode_eight_rows_long_cache_sampled_heads():
    q, k, v = _draw(8, 32, 8, 32768, 128, seed=9)
    scale = float(np.float32(1 / np.sqrt(128)))
    o, lse = _run(q, k, v, scale)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    for b, h in ((0, 0), (5, 9), (7, 31)):
        ro, rl = oracle.attention_plane(W.as_f64(q[b, h]), W.as_f64(k[b, h]), W.as_f64(v[b, h]),
                                        scale, False)
        assert max_err(o[b, h], ro) <= BF16_TOL_O and max_err(lse[b, h], rl) <= BF16_TOL_LSE
