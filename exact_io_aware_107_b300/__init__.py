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

__all__ = ["attention_forward", "attention_decode", "AttnError", "device_error", "load_library"]


def load_library():
    return _binding.load()


def _ptr(t):
    return None if t is None else t.data_ptr()


def attention_forward(q, k, v, causal=False, scale=None, cu_seqlens=None, out=None, lse=None,
                      stream=None):
    """O and LSE of softmax(scale * Q K^T + causal mask) V.

    q, k, v: CUDA tensors, bf16 or fp16 (D in {64, 128}) or fp32 (D <= 128), contiguous,
    (B, H, N, D), or (H, N_total, D) with ``cu_seqlens`` (int32 CUDA tensor of
    nseq+1 offsets).  Returns (O, LSE) with O like q and LSE fp32 (B, H, N) or
    (H, N_total).  Enqueued on ``stream`` (default: torch's current stream).
    """
    import torch

    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must share a dtype")
    if q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share a shape")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    if cu_seqlens is None:
        if q.dim() != 4:
            raise ValueError("dense layout is (B, H, N, D)")
        B, H, N, D = q.shape
    else:
        if q.dim() != 3:
            raise ValueError("packed layout is (H, N_total, D)")
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
            raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
        H, N, D = q.shape
        B = cu_seqlens.numel() - 1
        cu_seqlens = cu_seqlens.contiguous()
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream
    if q.dtype == torch.bfloat16:
        rc = _binding.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, D,
                               _ptr(cu_seqlens), causal, scale, handle)
    elif q.dtype == torch.float16:
        rc = _binding.attn_fwd_f16(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, D,
                                   _ptr(cu_seqlens), causal, scale, handle)
    elif q.dtype == torch.float32:
        rc = _binding.attn_fwd_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, D,
                                   _ptr(cu_seqlens), causal, scale, handle)
    else:
        raise TypeError("dtype must be bfloat16, float16 or float32")
    if rc != _binding.ATTN_OK:
        raise AttnError(rc, "attention_forward")
    return out, lse


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
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if workspace is None:
        rc, nbytes = _binding.attn_decode_workspace_bytes(B, H, Nq, Nk, D)
        if rc != _binding.ATTN_OK:
            raise AttnError(rc, "attention_decode")
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
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
