"""Exact IO-aware attention forward for B300 (sm_103a).

The compute runs in the CUDA library ``libattn_b300.so`` (C ABI in
``include/attn_b300.h``); this package marshals torch tensors into it.  torch
is used for device memory and streams only.  There is no CPU fallback: if
the library or a CUDA device is missing, the calls raise.

    from exact_io_aware_107_b300 import attention_forward
    o, lse = attention_forward(q, k, v, causal=True)             # (B,H,N,D) bf16
    o, lse = attention_forward(q, k, v, causal=True,
                               cu_seqlens=cu)                     # packed (H,N,D)
"""

from __future__ import annotations

import math

from . import _binding
from ._binding import AttnError

__all__ = ["attention_forward", "attention_forward_host", "attention_backward",
           "attention_decode", "AttnError", "device_error", "load_library"]


def load_library():
    return _binding.load()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _keep_for(stream, device, tensors):
    """Tensors this module allocated on torch's current stream but handed to
    work on another ``stream``: tell torch's allocator not to reuse their
    memory before that work is done."""
    import torch
    if stream != torch.cuda.current_stream(device):
        for t in tensors:
            t.record_stream(stream)


def attention_forward(q, k, v, causal=False, scale=None, cu_seqlens=None, out=None, lse=None,
                      stream=None, cu_seqlens_k=None):
    """O and LSE of softmax(scale * Q K^T + causal mask) V.

    q, k, v: CUDA tensors, bf16 or fp16 (D in {64, 128}) or fp32 (D <= 128), contiguous,
    (B, H, N, D), or (H, N_total, D) with ``cu_seqlens`` (int32 CUDA tensor of
    nseq+1 offsets).  Returns (O, LSE) with O like q and LSE fp32 (B, H, N) or
    (H, N_total).  Enqueued on ``stream`` (default: torch's current stream).

    Cross-attention: k and v may have a different sequence length Nk than q
    (dense), or their own offsets ``cu_seqlens_k`` (packed).  The causal mask
    then allows key j for query i when j <= i + (Nk - Nq) (the last query sees
    every key); a query with no allowed key gets O = 0 and LSE = -inf.
    """
    import torch

    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must share a dtype")
    if k.shape != v.shape:
        raise ValueError("k and v must share a shape")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    cus = []
    for c in (cu_seqlens, cu_seqlens_k):
        if c is not None and (c.dtype != torch.int32 or not c.is_cuda or c.dim() != 1):
            raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
        cus.append(None if c is None else c.contiguous())
    cu_q, cu_k = cus
    if cu_q is None:
        if cu_k is not None:
            raise ValueError("cu_seqlens_k needs cu_seqlens")
        if q.dim() != 4 or k.dim() != 4:
            raise ValueError("dense layout is (B, H, N, D)")
        B, H, N, D = q.shape
        Nk = k.shape[2]
        if k.shape != (B, H, Nk, D):
            raise ValueError("k, v must be (B, H, Nk, D) with q's B, H, D")
    else:
        if q.dim() != 3 or k.dim() != 3:
            raise ValueError("packed layout is (H, N_total, D)")
        H, N, D = q.shape
        B = cu_q.numel() - 1
        Nk = k.shape[1]
        if k.shape != (H, Nk, D):
            raise ValueError("k, v must be (H, Nk_total, D) with q's H, D")
        if cu_k is not None and cu_k.numel() != cu_q.numel():
            raise ValueError("cu_seqlens and cu_seqlens_k must have the same length")
    cross = Nk != N or cu_k is not None
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    # offsets copied by .contiguous() above belong to this call too
    own = [c for c, orig in ((cu_q, cu_seqlens), (cu_k, cu_seqlens_k))
           if c is not None and c is not orig]
    if out is None:
        out = torch.empty_like(q)
        own.append(out)
    if lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
        own.append(lse)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    _keep_for(stream, q.device, own)
    handle = stream.cuda_stream
    kinds = {torch.bfloat16: (_binding.attn_fwd, _binding.ATTN_BF16),
             torch.float16: (_binding.attn_fwd_f16, _binding.ATTN_F16),
             torch.float32: (_binding.attn_fwd_f32, _binding.ATTN_F32)}
    if q.dtype not in kinds:
        raise TypeError("dtype must be bfloat16, float16 or float32")
    fn, dtype = kinds[q.dtype]
    if cross:
        if cu_q is not None and cu_k is None:
            cu_k = cu_q
        rc = _binding.attn_fwd_cross(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, Nk,
                                     D, _ptr(cu_q), _ptr(cu_k), causal, scale, dtype, handle)
        where = "attention_forward (cross)"
    else:
        rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, D, _ptr(cu_q), causal,
                scale, handle)
        where = "attention_forward"
    if rc != _binding.ATTN_OK:
        raise AttnError(rc, where)
    return out, lse


def attention_forward_host(q, k, v, causal=False, scale=None, out=None, lse=None, workspace=None,
                           stream=None, device=None, non_blocking=False):
    """The forward on host tensors (B, H, N, D): bf16, fp16 or fp32 CPU tensors,
    page-locked (``pin_memory()``) for the copies to overlap the compute.

    Copies in, computes and copies back chunk by chunk on the current CUDA
    device, ordered after the work already on ``stream`` (default: torch's
    current stream).  By default the call returns once O and LSE are in the
    returned host tensors (it synchronises ``stream``).  With
    ``non_blocking=True`` it only enqueues the work, like the C call: the host
    tensors hold the result once ``stream`` has synchronised, and the inputs
    must not change before then.
    ``workspace``: a CUDA tensor of at least ``attn_fwd_host_workspace_bytes``
    bytes (256-byte aligned), or None to let torch allocate one here.
    """
    import torch

    kinds = {torch.bfloat16: _binding.ATTN_BF16, torch.float16: _binding.ATTN_F16,
             torch.float32: _binding.ATTN_F32}
    if q.dtype not in kinds or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share a dtype: bfloat16, float16 or float32")
    for t in (q, k, v):
        if t.is_cuda or not t.is_contiguous() or t.dim() != 4 or t.shape != q.shape:
            raise ValueError("q, k, v must be contiguous (B, H, N, D) host tensors of one shape")
    B, H, N, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q, pin_memory=True)
    if lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, pin_memory=True)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    if workspace is None:
        rc, nbytes = _binding.attn_fwd_host_workspace_bytes(B, H, N, D, kinds[q.dtype])
        if rc != _binding.ATTN_OK:
            raise AttnError(rc, "attention_forward_host")
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    rc = _binding.attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, D,
                                causal, scale, kinds[q.dtype], _ptr(workspace),
                                workspace.numel() * workspace.element_size(), stream.cuda_stream)
    if rc != _binding.ATTN_OK:
        raise AttnError(rc, "attention_forward_host")
    if non_blocking:
        # the library's copy and compute streams use the workspace until
        # ``stream`` has passed the call: keep torch from handing it out before
        workspace.record_stream(stream)
    else:
        stream.synchronize()
    return out, lse


def attention_backward(q, k, v, o, lse, dout, causal=False, scale=None, cu_seqlens=None,
                       cu_seqlens_k=None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """dQ, dK, dV of the forward for the upstream gradient ``dout``.

    q, k, v, causal, scale, cu_seqlens, cu_seqlens_k: as passed to
    :func:`attention_forward`; o, lse: its outputs.  bf16 or fp16, D in {64, 128}.
    ``workspace``: a CUDA tensor of at least ``attn_bwd_workspace_bytes``
    bytes, or None to let torch allocate one here (the library itself never
    allocates).  Returns (dQ, dK, dV).
    """
    import torch

    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("the backward takes bfloat16 or float16 tensors")
    for t in (q, k, v, o, dout):
        if t.dtype != q.dtype or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v, o, dout must be contiguous CUDA tensors of one dtype")
    if o.shape != q.shape or dout.shape != q.shape or k.shape != v.shape:
        raise ValueError("o and dout must be shaped like q, v like k")
    if lse.dtype != torch.float32 or lse.shape != q.shape[:-1] or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 shaped like q without its last axis")
    cu_q = None if cu_seqlens is None else cu_seqlens.contiguous()
    cu_k = None if cu_seqlens_k is None else cu_seqlens_k.contiguous()
    if cu_q is None:
        if cu_k is not None:
            raise ValueError("cu_seqlens_k needs cu_seqlens")
        B, H, N, D = q.shape
        Nk = k.shape[2]
        if k.shape != (B, H, Nk, D):
            raise ValueError("k, v must be (B, H, Nk, D) with q's B, H, D")
    else:
        H, N, D = q.shape
        B = cu_q.numel() - 1
        Nk = k.shape[1]
        if k.shape != (H, Nk, D):
            raise ValueError("k, v must be (H, Nk_total, D) with q's H, D")
        if cu_k is None:
            cu_k = cu_q
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    # offsets copied by .contiguous() above belong to this call too
    own = [c for c, orig in ((cu_q, cu_seqlens), (cu_k, cu_seqlens_k))
           if c is not None and c is not orig]
    if dq is None:
        dq = torch.empty_like(q)
        own.append(dq)
    if dk is None:
        dk = torch.empty_like(k)
        own.append(dk)
    if dv is None:
        dv = torch.empty_like(v)
        own.append(dv)
    if workspace is None:
        rc, nbytes = _binding.attn_bwd_workspace_bytes(B, H, N, D, cu_q is not None)
        if rc != _binding.ATTN_OK:
            raise AttnError(rc, "attention_backward")
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
        own.append(workspace)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    _keep_for(stream, q.device, own)
    dtype = _binding.ATTN_BF16 if q.dtype == torch.bfloat16 else _binding.ATTN_F16
    rc = _binding.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                           _ptr(dk), _ptr(dv), B, H, N, Nk, D, _ptr(cu_q), _ptr(cu_k), causal,
                           scale, dtype, _ptr(workspace),
                           workspace.numel() * workspace.element_size(), stream.cuda_stream)
    if rc != _binding.ATTN_OK:
        raise AttnError(rc, "attention_backward")
    return dq, dk, dv


def attention_decode(q, k, v, scale=None, workspace=None, out=None, lse=None, stream=None):
    """KV-cache decode: O and LSE of Nq new rows against all cached keys, no mask.

    q: bf16 (B, H, Nq, D) with 1 <= Nq <= 8; k, v: bf16 (B, H, Nk, D) CUDA tensors.
    ``workspace``: a CUDA tensor of at least ``decode_workspace_bytes`` bytes, or
    None to let torch allocate one here (the library itself never allocates).
    """
    import torch

    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16 or t.dim() != 4:
            raise ValueError("q, k, v must be contiguous 4-D bf16 CUDA tensors")
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, D) or v.shape != k.shape:
        raise ValueError("k, v must be (B, H, Nk, D) with q's B, H, D")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    own = []
    if out is None:
        out = torch.empty_like(q)
        own.append(out)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
        own.append(lse)
    if workspace is None:
        rc, nbytes = _binding.attn_decode_workspace_bytes(B, H, Nq, Nk, D)
        if rc != _binding.ATTN_OK:
            raise AttnError(rc, "attention_decode")
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
        own.append(workspace)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    _keep_for(stream, q.device, own)
    rc = _binding.attn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nk, D,
                              scale, _ptr(workspace), workspace.numel() * workspace.element_size(),
                              stream.cuda_stream)
    if rc != _binding.ATTN_OK:
        raise AttnError(rc, "attention_decode")
    return out, lse


def device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return _binding.attn_get_device_error(stream.cuda_stream)
