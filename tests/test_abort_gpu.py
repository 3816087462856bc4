"""The abort path of the real forward, backward and decode kernels.

Every wait inside the kernels is bounded.  With the library's fault-injection
switch on, the first thread block of each launch waits on an mbarrier phase
that nothing completes; its wait runs out of the (shortened) budget, the block
raises its abort flag, its other roles stop waiting, copies and MMAs already
issued drain, tensor memory is freed and the block exits.  The call must then
report ATTN_ERR_TIMEOUT, and the next ordinary call must be correct: the
context survives.  Nothing here faults or hangs the GPU: the wait that runs
out is the bounded one, and the drains it triggers wait for work that was
actually issued.
"""

import numpy as np
import pytest

import oracle
from exact_io_aware_107_b300 import workloads as W
from gpu_util import BF16_TOL_LSE, BF16_TOL_O, max_err

pytestmark = pytest.mark.gpu

BUDGET_NS = 5_000_000   # 5 ms: far above any legitimate wait of these small problems


@pytest.fixture
def injected():
    """Short wait budget and the stall switch on; both restored afterwards."""
    from exact_io_aware_107_b300 import _binding, device_error
    assert device_error() == 0
    assert _binding.attn_set_wait_timeout_ns(BUDGET_NS) == _binding.ATTN_OK
    assert _binding.attn_set_fault_injection(1) == _binding.ATTN_OK
    try:
        yield _binding
    finally:
        _binding.attn_set_fault_injection(0)
        _binding.attn_set_wait_timeout_ns(1_000_000_000)
        device_error()


def _inputs(dtype, B, H, N, D, seed, causal=True):
    w = W.custom(dtype, B=B, H=H, N=N, D=D, causal=causal, seed=seed)
    x = W.generate(w)
    return w, x


@pytest.mark.parametrize("dtype,D,N,causal", [("bf16", 128, 700, True), ("bf16", 64, 1300, False),
                                              ("f16", 128, 300, True)])
def test_forward_stall_reports_timeout_then_recovers(injected, dtype, D, N, causal):
    import torch
    from exact_io_aware_107_b300 import attention_forward, device_error
    B = injected
    w, x = _inputs(dtype, 2, 3, N, D, seed=N + D, causal=causal)
    q, k, v = (t.cuda() for t in (x["q"], x["k"], x["v"]))
    attention_forward(q, k, v, causal=causal, scale=w.scale)
    assert device_error() == B.ATTN_ERR_TIMEOUT
    assert device_error() == 0                       # the word was cleared
    B.attn_set_fault_injection(0)
    o, lse = attention_forward(q, k, v, causal=causal, scale=w.scale)
    assert device_error() == 0
    ro, rl = oracle.attention(W.as_f64(x["q"]), W.as_f64(x["k"]), W.as_f64(x["v"]), w.scale,
                              causal)
    tol_o = BF16_TOL_O if dtype == "bf16" else 5e-3
    assert max_err(o.float().cpu().numpy(), ro) <= tol_o
    assert max_err(lse.cpu().numpy(), rl) <= BF16_TOL_LSE
    torch.cuda.synchronize()


@pytest.mark.parametrize("D,N", [(128, 300), (64, 520)])
def test_backward_stall_reports_timeout_then_recovers(injected, D, N):
    from exact_io_aware_107_b300 import attention_backward, attention_forward, device_error
    from gpu_util import UNIT, bwd_bound_plane
    B = injected
    w, x = _inputs("bf16", 1, 2, N, D, seed=N)
    q, k, v = (t.cuda() for t in (x["q"], x["k"], x["v"]))
    do = W.generate(W.custom("bf16", B=1, H=2, N=N, D=D, seed=N + 1))["q"]
    ddo = do.cuda()
    B.attn_set_fault_injection(0)
    o, lse = attention_forward(q, k, v, causal=True, scale=w.scale)
    assert device_error() == 0
    B.attn_set_fault_injection(1)
    attention_backward(q, k, v, o, lse, ddo, causal=True, scale=w.scale)
    assert device_error() == B.ATTN_ERR_TIMEOUT
    B.attn_set_fault_injection(0)
    dq, dk, dv = attention_backward(q, k, v, o, lse, ddo, causal=True, scale=w.scale)
    assert device_error() == 0
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    for h in range(2):
        ref, bound = bwd_bound_plane(W.as_f64(x["q"][0, h]), W.as_f64(x["k"][0, h]),
                                     W.as_f64(x["v"][0, h]), W.as_f64(do[0, h]), w.scale, True,
                                     UNIT["bf16"])
        for g, r, b in zip((dq, dk, dv), ref, bound):
            assert (np.abs(f(g)[0, h] - r) <= b).all()


@pytest.mark.parametrize("workspace", [True, False])
def test_decode_stall_reports_timeout_then_recovers(injected, workspace):
    import torch
    from exact_io_aware_107_b300 import attention_decode, device_error
    from exact_io_aware_107_b300 import _binding
    B = injected
    Bn, H, Nq, Nk, D = 2, 4, 3, 5000, 128
    q = W.generate(W.custom("bf16", B=Bn, H=H, N=Nq, D=D, seed=31))["q"]
    kv = W.generate(W.custom("bf16", B=Bn, H=H, N=Nk, D=D, seed=32))
    dq, dk, dv = q.cuda(), kv["k"].cuda(), kv["v"].cuda()
    ws = None
    if workspace:
        rc, need = _binding.attn_decode_workspace_bytes(Bn, H, Nq, Nk, D)
        assert rc == 0 and need > 0          # several key slices per plane, then a merge
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    else:
        ws = torch.empty(0, dtype=torch.uint8, device="cuda")   # one slice per plane
    scale = float(np.float32(1 / np.sqrt(D)))
    attention_decode(dq, dk, dv, scale=scale, workspace=ws)
    assert device_error() == B.ATTN_ERR_TIMEOUT
    B.attn_set_fault_injection(0)
    o, lse = attention_decode(dq, dk, dv, scale=scale, workspace=ws)
    assert device_error() == 0
    ro, rl = oracle.attention(W.as_f64(q), W.as_f64(kv["k"]), W.as_f64(kv["v"]), scale, False)
    assert max_err(o.float().cpu().numpy(), ro) <= BF16_TOL_O
    assert max_err(lse.cpu().numpy(), rl) <= BF16_TOL_LSE
