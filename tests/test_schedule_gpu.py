"""The work counters of the persistent kernels.

The forward's causal and packed layouts hand their work items (pairs of
256-row blocks, then single blocks) to whichever persistent CTA asks first,
and so does the backward with its key tiles, from a counter in device memory
that the last CTA of each launch resets to zero.  What must hold: every call
covers every query row (forward) and every key row (backward), whatever
launches came before it on the same counter; repeated calls, CUDA-graph
replays and more launches than the library has counters give the same bits
as one call (dQ of the backward, summed over key tiles in a free order, up to
fp32 reassociation); and that call matches the oracle in every element.
Outputs are filled with NaN before every call, so a skipped item cannot pass.
"""

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
from exact_io_aware_107_b300 import workloads as W
from gpu_util import BF16_TOL_LSE, BF16_TOL_O, UNIT, bwd_bound_plane, max_err, run_cuda_bwd

pytestmark = pytest.mark.gpu

# dense causal, 100 planes of 4 blocks: 52 pairs of 26 planes, then 296
# single blocks (more items than CTAs); packed causal and non-causal sequences
CASES = {
    "dense_causal": dict(B=4, H=25, N=1024, D=64, causal=True, varlen=None),
    "packed_causal": dict(H=6, N=None, D=128, causal=True,
                          varlen=[3000, 17, 256, 1000, 2500, 700, 129, 4100]),
    "packed_noncausal": dict(H=5, N=None, D=64, causal=False,
                             varlen=[2000, 1, 300, 900, 1280]),
}


def _workload(name):
    c = dict(CASES[name])
    varlen = c.pop("varlen")
    if varlen is None:
        return W.custom("bf16", seed=77, **c)
    c.pop("N")
    return W.custom("bf16", seed=78, varlen=varlen, **c)


def _device_inputs(x):
    import torch
    q, k, v = (t.cuda() for t in (x["q"], x["k"], x["v"]))
    cu = None if x["cu_seqlens"] is None else torch.as_tensor(x["cu_seqlens"]).cuda()
    return q, k, v, cu


def _call(w, q, k, v, cu, o, lse, stream=None):
    from exact_io_aware_107_b300 import attention_forward
    o.fill_(float("nan"))
    lse.fill_(float("nan"))
    attention_forward(q, k, v, causal=w.causal, scale=w.scale, cu_seqlens=cu, out=o, lse=lse,
                      stream=stream)


def _oracle_errors(w, x, o, lse):
    from oracle.threads import blas_threads
    q, k, v = (W.as_f64(t) for t in (x["q"], x["k"], x["v"]))
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    if x["cu_seqlens"] is None:
        jobs = [(b, h) for b in range(w.B) for h in range(w.H)]

        def one(bh):
            b, h = bh
            ro, rl = oracle.attention_plane(q[b, h], k[b, h], v[b, h], w.scale, w.causal)
            return max_err(o[b, h], ro), max_err(lse[b, h], rl)
    else:
        cu = np.asarray(x["cu_seqlens"])
        jobs = [(h, s) for h in range(w.H) for s in range(len(cu) - 1)]

        def one(hs):
            h, s = hs
            a, e = cu[s], cu[s + 1]
            ro, rl = oracle.attention_plane(q[h, a:e], k[h, a:e], v[h, a:e], w.scale, w.causal)
            return max_err(o[h, a:e], ro), max_err(lse[h, a:e], rl)
    with blas_threads(1):
        with ThreadPoolExecutor(max_workers=8) as ex:
            errs = list(ex.map(one, jobs))
    return max(e[0] for e in errs), max(e[1] for e in errs)


@pytest.mark.parametrize("name", sorted(CASES))
def test_repeated_calls_bit_identical_and_match_oracle(name):
    import torch
    from exact_io_aware_107_b300 import device_error
    w = _workload(name)
    x = W.generate(w)
    q, k, v, cu = _device_inputs(x)
    outs = []
    for _ in range(4):
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")
        _call(w, q, k, v, cu, o, lse)
        outs.append((o, lse))
    torch.cuda.synchronize()
    assert device_error() == 0
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])
    eo, el = _oracle_errors(w, x, *outs[0])
    print(f"{name}: max|dO| {eo:.3g} max|dLSE| {el:.3g}")
    assert eo <= BF16_TOL_O and el <= BF16_TOL_LSE, (name, eo, el)


@pytest.mark.parametrize("name", ["dense_causal", "packed_causal"])
def test_graph_replays_equal_eager_calls(name):
    # one captured launch replayed on new inputs: it reuses one counter, which
    # each replay must find at zero
    import torch
    from exact_io_aware_107_b300 import device_error
    w = _workload(name)
    x = W.generate(w)
    q, k, v, cu = _device_inputs(x)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")
    ref_o, ref_lse = torch.empty_like(o), torch.empty_like(lse)
    _call(w, q, k, v, cu, ref_o, ref_lse)  # set-up of the library before the capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        _call(w, q, k, v, cu, o, lse, stream=torch.cuda.current_stream())
    torch.cuda.current_stream().wait_stream(side)
    gen = torch.Generator(device="cpu").manual_seed(3)
    for _ in range(3):
        for t in (q, k, v):
            t.copy_(torch.randn(t.shape, generator=gen).to(t.dtype))
        g.replay()
        _call(w, q, k, v, cu, ref_o, ref_lse)
        torch.cuda.synchronize()
        assert device_error() == 0
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)


def test_more_launches_than_counters():
    # 600 launches on two streams, more than the library's counters: each
    # counter is reused many times, and every launch must still cover every row
    import torch
    from exact_io_aware_107_b300 import device_error
    w = W.custom("bf16", B=2, H=3, N=600, D=64, causal=True, seed=79)
    x = W.generate(w)
    q, k, v, cu = _device_inputs(x)
    ref_o = torch.empty_like(q)
    ref_lse = torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")
    _call(w, q, k, v, cu, ref_o, ref_lse)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [(torch.empty_like(ref_o), torch.empty_like(ref_lse)) for _ in range(8)]
    for i in range(600):
        s = streams[i % 2]
        o, lse = outs[i % 8]
        with torch.cuda.stream(s):
            _call(w, q, k, v, cu, o, lse, stream=s)
        if i % 8 == 7:
            torch.cuda.synchronize()
            for o2, lse2 in outs:
                assert torch.equal(o2, ref_o) and torch.equal(lse2, ref_lse), i
    assert device_error() == 0
    eo, el = _oracle_errors(w, x, ref_o, ref_lse)
    assert eo <= BF16_TOL_O and el <= BF16_TOL_LSE, (eo, el)


# ---------------------------------------------------------------- backward

def _dout_like(q, seed):
    import torch
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randn(q.shape, generator=g).to(q.dtype)


@pytest.mark.parametrize("causal,D", [(True, 128), (False, 64)])
def test_backward_several_key_tiles_per_cta_every_plane(causal, D):
    # 80 planes of 10 key tiles: 800 work items over the persistent CTAs, so
    # each CTA runs five or six key tiles back to back (the phases of every
    # barrier carried from one key tile to the next); every plane is compared
    # with the oracle's gradient within the error bound
    B, H, N = 4, 20, 1280
    w = W.custom("bf16", B=B, H=H, N=N, D=D, causal=causal, seed=90 + D)
    x = W.generate(w)
    do = _dout_like(x["q"], 91)
    dq, dk, dv = run_cuda_bwd(x["q"], x["k"], x["v"], do, causal, w.scale)
    f = W.as_f64
    q, k, v, g = f(x["q"]), f(x["k"]), f(x["v"]), f(do)
    u = UNIT["bf16"]

    def one(bh):
        b, h = bh
        (rq, rk, rv), (bq, bk, bv) = bwd_bound_plane(q[b, h], k[b, h], v[b, h], g[b, h], w.scale,
                                                     causal, u)
        return max(float((np.abs(dq[b, h] - rq) - bq).max()),
                   float((np.abs(dk[b, h] - rk) - bk).max()),
                   float((np.abs(dv[b, h] - rv) - bv).max()))

    from oracle.threads import blas_threads
    with blas_threads(1):
        with ThreadPoolExecutor(max_workers=8) as ex:
            excess = list(ex.map(one, [(b, h) for b in range(B) for h in range(H)]))
    assert max(excess) <= 0, max(excess)


def test_backward_more_launches_than_counters():
    # 300 backward calls on two streams: every call finds its counter at zero,
    # dK and dV equal the first call's bit for bit, dQ up to reassociation
    import torch
    from exact_io_aware_107_b300 import attention_backward, attention_forward, device_error
    w = W.custom("bf16", B=2, H=3, N=700, D=128, causal=True, seed=92)
    x = W.generate(w)
    q, k, v = (t.cuda() for t in (x["q"], x["k"], x["v"]))
    do = _dout_like(x["q"], 93).cuda()
    o, lse = attention_forward(q, k, v, causal=True)
    ref = attention_backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [tuple(torch.empty_like(t) for t in ref) for _ in range(4)]
    wss = [None, None]
    for i in range(300):
        s = streams[i % 2]
        dq, dk, dv = outs[i % 4]
        with torch.cuda.stream(s):
            for t in (dq, dk, dv):
                t.fill_(float("nan"))
            attention_backward(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv, stream=s)
        if i % 4 == 3:
            torch.cuda.synchronize()
            for dq, dk, dv in outs:
                assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2]), i
                assert (dq.float() - ref[0].float()).abs().max() <= 2.0 ** -7 * max(
                    1.0, ref[0].float().abs().max().item()), i
    assert device_error() == 0


def test_malformed_offsets_late_in_the_list_are_reported():
    # the bad offsets come after 199 good sequences, so only a work item taken
    # late (decoded by the producer warp alone, not at a CTA's start) meets them
    import torch
    from exact_io_aware_107_b300 import (_binding, attention_backward, attention_forward,
                                         device_error)
    n = 200 * 256
    x = W.generate(W.custom("bf16", B=1, H=1, N=n, D=128, seed=94))
    q, k, v = (t[0].contiguous().cuda() for t in (x["q"], x["k"], x["v"]))
    cu = torch.arange(0, n + 1, 256, dtype=torch.int32)
    cu[-1] = cu[-2] - 10  # decreasing: the last sequence is malformed
    cu = cu.cuda()
    assert device_error() == 0
    for causal in (True, False):
        o, lse = attention_forward(q, k, v, causal=causal, cu_seqlens=cu)
        assert device_error() == _binding.ATTN_ERR_BOUNDS
        o = torch.zeros_like(q)
        lse = torch.zeros(q.shape[:-1], dtype=torch.float32, device="cuda")
        attention_backward(q, k, v, o, lse, q, causal=causal, cu_seqlens=cu)
        assert device_error() == _binding.ATTN_ERR_BOUNDS
    assert device_error() == 0


@pytest.mark.parametrize("dtype,causal", [("bf16", True), ("f16", False)])
def test_backward_packed_many_sequences_every_sequence(dtype, causal):
    # 40 packed sequences of 1..700 rows over 4 heads: several hundred key
    # tiles, so each persistent CTA walks several sequences' key tiles; every
    # (sequence, head) is compared with the oracle's gradient within the bound
    rng = np.random.default_rng(95)
    lens = [int(x) for x in rng.integers(1, 701, 40)]
    w = W.custom(dtype, H=4, D=128, causal=causal, seed=96, varlen=lens)
    x = W.generate(w)
    do = _dout_like(x["q"], 97)
    dq, dk, dv = run_cuda_bwd(x["q"], x["k"], x["v"], do, causal, w.scale, x["cu_seqlens"])
    f = W.as_f64
    q, k, v, g = f(x["q"]), f(x["k"]), f(x["v"]), f(do)
    cu = np.asarray(x["cu_seqlens"])
    u = UNIT[dtype]

    def one(hs):
        h, s = hs
        a, e = int(cu[s]), int(cu[s + 1])
        (rq, rk, rv), (bq, bk, bv) = bwd_bound_plane(q[h, a:e], k[h, a:e], v[h, a:e], g[h, a:e],
                                                     w.scale, causal, u)
        return max(float((np.abs(dq[h, a:e] - rq) - bq).max()),
                   float((np.abs(dk[h, a:e] - rk) - bk).max()),
                   float((np.abs(dv[h, a:e] - rv) - bv).max()))

    from oracle.threads import blas_threads
    with blas_threads(1):
        with ThreadPoolExecutor(max_workers=8) as ex:
            excess = list(ex.map(one, [(h, s) for h in range(w.H) for s in range(len(lens))]))
    assert max(excess) <= 0, max(excess)
