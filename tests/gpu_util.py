"""Helpers shared by the GPU tests: run the CUDA path, run the oracle, compare."""

import numpy as np

# Tolerances (max absolute error against the fp64 oracle on the same inputs).
F32_TOL_O = 1e-4
F32_TOL_LSE = 1e-4
BF16_TOL_O = 2e-2
BF16_TOL_LSE = 1e-3
# fp16 keeps three more mantissa bits than bf16: O is rounded with a half-ulp of
# at most 2^-9 for |O| < 8 and P with a relative 2^-11, so 5e-3 bounds O.
F16_TOL_O = 5e-3
F16_TOL_LSE = 1e-3


def run_cuda(q, k, v, causal, scale, cu_seqlens=None, poison=True, cu_seqlens_k=None):
    """Run the CUDA path on host tensors; returns fp64 numpy O and LSE."""
    import torch
    from exact_io_aware_107_b300 import attention_forward, device_error
    dq, dk, dv = (t.to("cuda") for t in (q, k, v))
    dcu = None if cu_seqlens is None else torch.as_tensor(cu_seqlens, dtype=torch.int32).cuda()
    dcuk = None if cu_seqlens_k is None else torch.as_tensor(cu_seqlens_k, dtype=torch.int32).cuda()
    o = torch.empty_like(dq)
    lse = torch.empty(dq.shape[:-1], dtype=torch.float32, device="cuda")
    if poison:
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
    attention_forward(dq, dk, dv, causal=causal, scale=scale, cu_seqlens=dcu, out=o, lse=lse,
                      cu_seqlens_k=dcuk)
    assert device_error() == 0
    return (o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64))


def max_err(a, b):
    """Largest |a - b|; equal infinities (LSE = -inf of a row with no key) count as 0."""
    if a.size == 0:
        return 0.0
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    same_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        d = np.where(same_inf, 0.0, np.abs(a - b))
    if np.isnan(d).any():
        return float("inf")
    return float(d.max())
