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


# ---------------------------------------------------------------- backward
#
# Error bound of the 16-bit backward, element by element (first order in the
# unit roundoff u: 2^-8 for bf16, 2^-11 for fp16 -- half an ulp at 1).  Every
# product the kernel feeds to the tensor cores has at most two 16-bit roundings
# in it (P, then dS = P (dP - Delta)), the fp32 sums add nothing of that order,
# and each gradient is rounded once at the end.  Delta is computed from the
# forward's 16-bit O, whose error is bounded the same way.  With T = 2u:
#   |dV err| <= T * P^T |dO| + u |dV|
#   |dS err| <= T * |dS| + P * |Delta err|,  |Delta err| <= |dO| . (T P|V| + u |O|)
#   |dK err| <= scale * |dS err|^T |Q| + u |dK|,   |dQ err| <= scale * |dS err| |K| + u |dQ|
# The bound below is twice that, plus 1e-6 absolute.

def bwd_bound_plane(q, k, v, do, scale, causal, unit):
    import oracle
    q, k, v, do = (np.asarray(a, dtype=np.float64) for a in (q, k, v, do))
    dq, dk, dv = oracle.attention_backward_plane(q, k, v, do, scale, causal)
    if q.shape[0] == 0 or k.shape[0] == 0:
        z = lambda a: np.full_like(a, 1e-6)
        return (dq, dk, dv), (z(dq), z(dk), z(dv))
    with np.errstate(invalid="ignore"):
        p = np.nan_to_num(oracle.softmax_probs(q, k, scale, causal))   # rows with no key: 0
    o = p @ v
    delta = (do * o).sum(1, keepdims=True)
    ds = p * (do @ v.T - delta)
    t = 2 * unit
    d_err = (np.abs(do) * (t * (p @ np.abs(v)) + unit * np.abs(o))).sum(1, keepdims=True)
    ds_err = t * np.abs(ds) + p * d_err
    b_dv = t * (p.T @ np.abs(do)) + unit * np.abs(dv)
    b_dk = scale * (ds_err.T @ np.abs(q)) + unit * np.abs(dk)
    b_dq = scale * (ds_err @ np.abs(k)) + unit * np.abs(dq)
    return (dq, dk, dv), (2 * b_dq + 1e-6, 2 * b_dk + 1e-6, 2 * b_dv + 1e-6)


def run_cuda_bwd(q, k, v, do, causal, scale, cu_seqlens=None, cu_seqlens_k=None):
    """Forward then backward on the GPU from host tensors; fp64 numpy dQ, dK, dV."""
    import torch
    from exact_io_aware_107_b300 import attention_backward, attention_forward, device_error
    dq_, dk_, dv_, ddo = (t.to("cuda") for t in (q, k, v, do))
    cu = None if cu_seqlens is None else torch.as_tensor(cu_seqlens, dtype=torch.int32).cuda()
    cuk = None if cu_seqlens_k is None else torch.as_tensor(cu_seqlens_k, dtype=torch.int32).cuda()
    o, lse = attention_forward(dq_, dk_, dv_, causal=causal, scale=scale, cu_seqlens=cu,
                               cu_seqlens_k=cuk)
    gq = torch.full_like(dq_, float("nan"))
    gk = torch.full_like(dk_, float("nan"))
    gv = torch.full_like(dv_, float("nan"))
    attention_backward(dq_, dk_, dv_, o, lse, ddo, causal=causal, scale=scale, cu_seqlens=cu,
                       cu_seqlens_k=cuk, dq=gq, dk=gk, dv=gv)
    assert device_error() == 0
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    return f(gq), f(gk), f(gv)


UNIT = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}
