"""GPU checks that need no oracle: exact special cases, causality, packed-vs-dense
equality, determinism, untouched guard rows, device error reporting."""

import numpy as np
import pytest

from exact_io_aware_107_b300 import workloads as W
from gpu_util import run_cuda

pytestmark = pytest.mark.gpu


def _gen(dtype, B, H, N, D, seed, causal=True):
    x = W.generate(W.custom(dtype, B=B, H=H, N=N, D=D, causal=causal, seed=seed))
    return x["q"], x["k"], x["v"]


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("bf16", 128), ("f16", 128), ("f32", 64)])
def test_causal_row0_is_v0_bit_exact(dtype, D):
    q, k, v = _gen(dtype, 2, 3, 333, D, 1)
    o, lse = run_cuda(q, k, v, True, 0.125)
    np.testing.assert_array_equal(o[:, :, 0], W.as_f64(v[:, :, 0]))
    s0 = (W.as_f64(q[:, :, 0]) * W.as_f64(k[:, :, 0])).sum(-1) * 0.125
    assert np.abs(lse[:, :, 0] - s0).max() < 1e-4


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("f32", 128)])
def test_future_keys_do_not_leak(dtype, D):
    import torch
    q, k, v = _gen(dtype, 1, 2, 700, D, 2)
    o1, l1 = run_cuda(q, k, v, True, 0.1)
    i = 300
    k2, v2 = k.clone(), v.clone()
    k2[:, :, i + 1:] = (torch.randn_like(k2[:, :, i + 1:].float()) * 3).to(k.dtype)
    v2[:, :, i + 1:] = (torch.randn_like(v2[:, :, i + 1:].float()) * 3).to(v.dtype)
    o2, l2 = run_cuda(q, k2, v2, True, 0.1)
    np.testing.assert_array_equal(o1[:, :, :i + 1], o2[:, :, :i + 1])
    np.testing.assert_array_equal(l1[:, :, :i + 1], l2[:, :, :i + 1])
    assert np.abs(o1[:, :, i + 1:] - o2[:, :, i + 1:]).max() > 1e-2


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("f16", 128), ("f32", 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_packed_equals_dense_per_sequence(dtype, D, causal):
    lens = [5, 128, 300, 1, 257, 640]
    w = W.custom(dtype, H=2, D=D, causal=causal, seed=4, varlen=lens)
    x = W.generate(w)
    o, lse = run_cuda(x["q"], x["k"], x["v"], causal, w.scale, x["cu_seqlens"])
    cu = x["cu_seqlens"]
    for s in range(len(lens)):
        a, e = int(cu[s]), int(cu[s + 1])
        sl = lambda t: t[:, a:e].unsqueeze(0).contiguous()
        od, ld = run_cuda(sl(x["q"]), sl(x["k"]), sl(x["v"]), causal, w.scale)
        np.testing.assert_array_equal(o[:, a:e], od[0])
        np.testing.assert_array_equal(lse[:, a:e], ld[0])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_run_to_run_deterministic(dtype):
    q, k, v = _gen(dtype, 2, 4, 1000, 128 if dtype == "bf16" else 64, 3)
    a = run_cuda(q, k, v, True, 0.09)
    b = run_cuda(q, k, v, True, 0.09)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_rows_outside_every_sequence_stay_untouched(dtype):
    # cu_seqlens covers tokens [0, 260); rows 260..299 belong to no sequence
    x = W.generate(W.custom(dtype, B=1, H=2, N=300, D=64, seed=6))
    q, k, v = (t[0].contiguous() for t in (x["q"], x["k"], x["v"]))
    cu = np.array([0, 5, 133, 260], dtype=np.int32)
    o, lse = run_cuda(q, k, v, True, 0.125, cu)
    assert not np.isnan(o[:, :260]).any() and not np.isnan(lse[:, :260]).any()
    assert np.isnan(o[:, 260:]).all() and np.isnan(lse[:, 260:]).all()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bad_cu_seqlens_reported_on_device(dtype):
    import torch
    from exact_io_aware_107_b300 import attention_forward, device_error, _binding
    x = W.generate(W.custom(dtype, B=1, H=2, N=256, D=64, seed=6))
    q, k, v = (t[0].contiguous().cuda() for t in (x["q"], x["k"], x["v"]))
    assert device_error() == 0
    for bad in ([0, 100, 50, 256], [0, 100, 300]):     # decreasing; beyond N
        cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
        attention_forward(q, k, v, causal=True, cu_seqlens=cu)
        assert device_error() == _binding.ATTN_ERR_BOUNDS
    assert device_error() == 0   # the word was cleared
    # the context is still usable
    o, lse = run_cuda(x["q"], x["k"], x["v"], True, 0.125)
    assert np.isfinite(o).all()


def test_bounded_wait_times_out_and_context_survives():
    import torch
    from exact_io_aware_107_b300 import _binding, device_error
    s = torch.cuda.current_stream().cuda_stream
    assert device_error() == 0
    assert _binding.attn_wait_selftest(20_000_000, s) == 0          # 20 ms budget
    assert device_error() == _binding.ATTN_ERR_TIMEOUT
    assert device_error() == 0
    x = W.generate(W.custom("bf16", B=1, H=2, N=256, D=128, seed=8))
    o, lse = run_cuda(x["q"], x["k"], x["v"], True, 0.09)
    assert np.isfinite(o).all() and np.isfinite(lse).all()


def test_library_allocates_no_device_memory():
    import torch
    from exact_io_aware_107_b300 import attention_forward
    x = W.generate(W.custom("bf16", B=1, H=4, N=4096, D=128, seed=8))
    q, k, v = (t.cuda() for t in (x["q"], x["k"], x["v"]))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device="cuda")
    attention_forward(q, k, v, causal=True, out=o, lse=lse)     # first call: one-time set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    peak0 = torch.cuda.max_memory_allocated()
    for _ in range(5):
        attention_forward(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.max_memory_allocated() == peak0
    assert abs(free1 - free0) < (2 << 20)


@pytest.mark.parametrize("nbytes", [16, 16 * 12345, 64 << 20])
def test_hbm_read_probe_reads_every_word(nbytes):
    # the probe folds every 32-bit word it reads with XOR: the fold must equal
    # the host's, so the bandwidth it times is the bandwidth of reading it all
    import torch
    from exact_io_aware_107_b300 import _binding
    rng = np.random.default_rng(nbytes % 1000)
    host = rng.integers(0, 2**32, nbytes // 4, dtype=np.uint32)
    buf = torch.from_numpy(host.view(np.int32)).cuda()
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream()
    assert _binding.attn_hbm_read_probe(buf.data_ptr(), nbytes, out.data_ptr(), s.cuda_stream) == 0
    torch.cuda.synchronize()
    assert int(out.cpu().numpy().view(np.uint32)[0]) == int(np.bitwise_xor.reduce(host))
    assert _binding.attn_hbm_read_probe(buf.data_ptr(), 8, out.data_ptr(), s.cuda_stream) == \
        _binding.ATTN_ERR_SHAPE
