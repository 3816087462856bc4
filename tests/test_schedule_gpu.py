"""The forward's work counter.

The causal and the packed layouts hand their work items (pairs of 256-row
blocks, then single blocks) to whichever persistent CTA asks first, from a
counter in device memory that the last CTA of each launch resets to zero.
What must hold: every call covers every query row, whatever launches came
before it on the same counter; repeated calls, CUDA-graph replays and more
launches than the library has counters give the same bits as one call; and
that call matches the oracle in every element.  Outputs are filled with NaN
before every call, so a skipped item cannot pass.
"""

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
from exact_io_aware_107_b300 import workloads as W
from gpu_util import BF16_TOL_LSE, BF16_TOL_O, max_err

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
