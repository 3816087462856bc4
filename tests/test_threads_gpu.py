"""Calls from several host threads at once, each thread on its own stream.

The library's host state (per-device set-up, the error word, the host-buffer
pipeline) is shared between threads; the kernels themselves are deterministic
except for dQ's summation order.  So every concurrent forward must equal, bit
for bit, the same call made alone, and so must dK and dV of the backward.
"""

import threading

import pytest

from exact_io_aware_107_b300 import workloads as W

pytestmark = pytest.mark.gpu

SHAPES = [("bf16", 1, 4, 700, 128, True), ("bf16", 2, 2, 300, 64, False),
          ("f16", 1, 8, 1024, 128, False), ("f32", 3, 1, 129, 64, True),
          ("bf16", 1, 2, 4096, 128, True), ("f32", 1, 2, 257, 128, False)]


def _inputs():
    out = []
    for i, (dt, B, H, N, D, causal) in enumerate(SHAPES):
        x = W.generate(W.custom(dt, B=B, H=H, N=N, D=D, causal=causal, seed=40 + i))
        out.append((x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal))
    return out


def _run_threads(n, body):
    errors = []

    def wrap(i):
        try:
            body(i)
        except BaseException as e:  # noqa: BLE001 - surfaced by the assert below
            errors.append((i, repr(e)))

    ts = [threading.Thread(target=wrap, args=(i,)) for i in range(n)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in ts), "a thread did not finish"
    assert not errors, errors


def test_concurrent_forwards_equal_serial_calls():
    import torch
    from exact_io_aware_107_b300 import attention_forward, device_error
    inputs = _inputs()
    serial = []
    for q, k, v, causal in inputs:
        o, lse = attention_forward(q, k, v, causal=causal)
        serial.append((o.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert device_error() == 0
    results = [None] * len(inputs)

    def body(i):
        q, k, v, causal = inputs[i]
        s = torch.cuda.Stream()
        outs = []
        with torch.cuda.stream(s):
            for _ in range(8):
                outs.append(attention_forward(q, k, v, causal=causal))
        s.synchronize()
        results[i] = outs

    _run_threads(len(inputs), body)
    assert device_error() == 0
    for i, outs in enumerate(results):
        for o, lse in outs:
            assert torch.equal(o, serial[i][0]) and torch.equal(lse, serial[i][1]), SHAPES[i]


def test_concurrent_backwards_equal_serial_calls():
    import torch
    from exact_io_aware_107_b300 import attention_backward, attention_forward, device_error
    cases = []
    for i, (dt, B, H, N, D, causal) in enumerate(SHAPES):
        if dt == "f32":
            continue                                   # the backward is 16-bit only
        x = W.generate(W.custom(dt, B=B, H=H, N=N, D=D, causal=causal, seed=60 + i))
        q, k, v = (t.cuda() for t in (x["q"], x["k"], x["v"]))
        do = W.generate(W.custom(dt, B=B, H=H, N=N, D=D, seed=80 + i))["q"].cuda()
        o, lse = attention_forward(q, k, v, causal=causal)
        dq, dk, dv = attention_backward(q, k, v, o, lse, do, causal=causal)
        cases.append((q, k, v, o, lse, do, causal, dq.clone(), dk.clone(), dv.clone()))
    torch.cuda.synchronize()
    assert device_error() == 0
    results = [None] * len(cases)

    def body(i):
        q, k, v, o, lse, do, causal = cases[i][:7]
        s = torch.cuda.Stream()
        outs = []
        with torch.cuda.stream(s):
            for _ in range(4):
                outs.append(attention_backward(q, k, v, o, lse, do, causal=causal))
        s.synchronize()
        results[i] = outs

    _run_threads(len(cases), body)
    assert device_error() == 0
    for i, outs in enumerate(results):
        dq0, dk0, dv0 = cases[i][7:]
        for dq, dk, dv in outs:
            assert torch.equal(dk, dk0) and torch.equal(dv, dv0)
            # dQ is summed over key tiles in a free order: equal up to that order
            assert torch.allclose(dq.float(), dq0.float(), rtol=2e-2, atol=2e-3)


def test_concurrent_host_buffer_calls():
    import torch
    from exact_io_aware_107_b300 import attention_forward, attention_forward_host, device_error
    ins = []
    for i in range(3):
        x = W.generate(W.custom("bf16", B=1, H=8, N=1000, D=128, causal=True, seed=90 + i))
        ins.append((x["q"].pin_memory(), x["k"].pin_memory(), x["v"].pin_memory()))
    ref = []
    for q, k, v in ins:
        o, lse = attention_forward(q.cuda(), k.cuda(), v.cuda(), causal=True)
        ref.append((o.cpu(), lse.cpu()))
    results = [None] * len(ins)

    def body(i):
        q, k, v = ins[i]
        outs = []
        for _ in range(3):
            o, lse = attention_forward_host(q, k, v, causal=True)
            outs.append((o.clone(), lse.clone()))
        results[i] = outs

    _run_threads(len(ins), body)
    torch.cuda.synchronize()
    assert device_error() == 0
    for i, outs in enumerate(results):
        for o, lse in outs:
            assert torch.equal(o, ref[i][0]) and torch.equal(lse, ref[i][1])


def test_explicit_stream_keeps_the_workspace_until_the_work_is_done():
    # The wrappers allocate their workspace on torch's current stream.  When
    # the work goes to another stream that is still busy, that memory must not
    # be handed out again on the current stream when the call returns: a
    # same-size allocation made right after the call gets other memory.
    import torch
    from exact_io_aware_107_b300 import attention_backward, attention_decode, attention_forward
    from exact_io_aware_107_b300 import device_error
    w = W.custom("bf16", B=2, H=8, N=2048, D=128, causal=True, seed=71)
    x = W.generate(w)
    q, k, v = (t.cuda() for t in (x["q"], x["k"], x["v"]))
    do = W.generate(W.custom("bf16", B=2, H=8, N=2048, D=128, seed=72))["q"].cuda()
    o, lse = attention_forward(q, k, v, causal=True)
    ref = attention_backward(q, k, v, o, lse, do, causal=True)
    kv = W.generate(W.custom("bf16", B=2, H=8, N=65536, D=128, seed=73))
    kc, vc = kv["k"].cuda(), kv["v"].cuda()
    qd = q[:, :, :2].contiguous()      # inputs stay alive until the work is done
    ref_dec = attention_decode(qd, kc, vc)
    torch.cuda.synchronize()
    big = torch.zeros(1 << 28, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def call_and_spy(fn):
        # the byte-typed workspace the wrapper allocates: its address and size
        seen = []
        orig = torch.empty

        def spy(*a, **kw):
            t = orig(*a, **kw)
            if kw.get("dtype") == torch.uint8 and t.is_cuda:
                seen.append((t.data_ptr(), t.numel()))
            return t

        torch.empty = spy
        try:
            res = fn()
        finally:
            torch.empty = orig
        assert len(seen) == 1
        return res, seen[0]

    for _ in range(2):
        with torch.cuda.stream(s):
            for _ in range(8):        # keep s busy well past the checks below
                big.add_(1.0)
        got, (ptr, n) = call_and_spy(
            lambda: attention_backward(q, k, v, o, lse, do, causal=True, stream=s))
        junk = torch.full((n,), 0x7f, dtype=torch.uint8, device="cuda")
        assert junk.data_ptr() != ptr
        got_dec, (ptr2, n2) = call_and_spy(lambda: attention_decode(qd, kc, vc, stream=s))
        junk2 = torch.full((n2,), 0x7f, dtype=torch.uint8, device="cuda")
        assert junk2.data_ptr() != ptr2
        s.synchronize()
        torch.cuda.synchronize()
        del junk, junk2
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
        assert torch.allclose(got[0].float(), ref[0].float(), rtol=2e-2, atol=2e-3)
        assert torch.equal(got_dec[0], ref_dec[0]) and torch.equal(got_dec[1], ref_dec[1])
    assert device_error() == 0
