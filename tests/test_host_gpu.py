"""The host-buffer forward (attn_fwd_host): chunked copies and kernels on
internal streams give the same O and LSE as the device-buffer call."""

import numpy as np
import pytest

import oracle
from exact_io_aware_107_b300 import workloads as W
from gpu_util import BF16_TOL_LSE, BF16_TOL_O, max_err

pytestmark = pytest.mark.gpu


def _both(w, causal):
    import torch
    from exact_io_aware_107_b300 import attention_forward, attention_forward_host, device_error
    x = W.generate(w)
    hq, hk, hv = (t.pin_memory() for t in (x["q"], x["k"], x["v"]))
    o_h = torch.full_like(hq, float("nan")).pin_memory()
    l_h = torch.full(hq.shape[:-1], float("nan"), dtype=torch.float32).pin_memory()
    attention_forward_host(hq, hk, hv, causal=causal, scale=w.scale, out=o_h, lse=l_h)
    torch.cuda.synchronize()
    assert device_error() == 0
    o_d, l_d = attention_forward(*(t.cuda() for t in (x["q"], x["k"], x["v"])), causal=causal,
                                 scale=w.scale)
    torch.cuda.synchronize()
    return x, o_h, l_h, o_d.cpu(), l_d.cpu()


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("f16", 128), ("f32", 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_host_equals_device_call(dtype, D, causal):
    # 2 x 9 = 18 planes: chunks of 3 planes through two slots (each slot reused)
    w = W.custom(dtype, B=2, H=9, N=300, D=D, causal=causal, seed=31)
    x, o_h, l_h, o_d, l_d = _both(w, causal)
    assert (o_h.float() == o_d.float()).all() and (l_h == l_d).all()


def test_host_single_plane_and_oracle():
    w = W.custom("bf16", B=1, H=1, N=1000, D=128, causal=True, seed=32)
    x, o_h, l_h, o_d, l_d = _both(w, True)
    assert (o_h.float() == o_d.float()).all()
    ro, rl = oracle.attention(W.as_f64(x["q"]), W.as_f64(x["k"]), W.as_f64(x["v"]), w.scale, True)
    assert max_err(o_h.float().numpy().astype(np.float64), ro) <= BF16_TOL_O
    assert max_err(l_h.numpy().astype(np.float64), rl) <= BF16_TOL_LSE


def test_host_orders_after_and_before_the_callers_stream():
    # the call follows work already on the stream and the stream waits for the copies back
    import torch
    from exact_io_aware_107_b300 import attention_forward_host
    w = W.custom("bf16", B=2, H=8, N=512, D=128, causal=True, seed=33)
    x = W.generate(w)
    hq, hk, hv = (t.pin_memory() for t in (x["q"], x["k"], x["v"]))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, l1 = attention_forward_host(hq, hk, hv, causal=True, scale=w.scale, non_blocking=True)
        hq2 = (hq.float() * 0.5).to(hq.dtype).pin_memory()
        o2, l2 = attention_forward_host(hq2, hk, hv, causal=True, scale=w.scale,
                                        non_blocking=True)
        done = torch.cuda.Event()
        done.record(s)
    done.synchronize()
    assert torch.isfinite(o1.float()).all() and torch.isfinite(o2.float()).all()
    assert not torch.equal(l1, l2)
