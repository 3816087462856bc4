"""Seeded synthetic inputs for the attention forward workloads.

This module only draws random numbers and rounds them to the storage dtype.
It holds none of the attention arithmetic, so both the CUDA path (through
the tests and the bench) and the CPU oracle can read the very same buffers.

Shapes follow the (batch, heads, seq_len, dim) problem statement of
"Build a FlashAttention kernel from scratch with Python and NumPy"
(section "Architecture Overview"); the packed variable-length layout is
(heads, total_tokens, dim) with a cu_seqlens offset vector, the un-padded
form described in "Flash Attention vs Standard Attention" (section
"Critical Implementation Details").

Recipes
-------
* ``f32_causal_small``: B=2, H=4, N=128, D=64, causal, fp32.  Q, K, V are
  drawn with the legacy global generator, ``np.random.seed(0)`` then three
  ``randn`` calls, exactly the call sequence of the first page's "Step 2".
* ``bf16_*`` dense: ``np.random.default_rng(seed).standard_normal(shape,
  dtype=float32)`` for Q, K, V in that order (the generator call of
  "Building a FlashAttention-2 forward kernel in pure NumPy", "Step 5");
  Q and K are multiplied by ``qk_std`` in fp32; every tensor is then rounded
  to bfloat16 with round-to-nearest-even.
* ``bf16_varlen_causal``: ``default_rng(7)``; 16 lengths from
  ``integers(256, 8193)``, then Q, K, V of shape (H, sum(lengths), D).
* Cross-attention workloads (``Nk`` set, keys of another length than the
  queries): the same ``default_rng`` draw order Q, K, V, with K and V of
  shape (B, H, Nk, D), or (H, sum(varlen_k), D) when packed.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "f32", "bf16" or "f16"
    B: int                # batch (number of sequences for varlen)
    H: int
    N: int                # seq_len (total tokens for varlen)
    D: int
    causal: bool
    seed: int
    qk_std: float = 1.0
    generator: str = "default_rng"   # or "legacy"
    varlen: Optional[tuple] = None   # sequence lengths for the packed layout
    len_draw: Optional[tuple] = None  # (nseq, lo, hi) when the lengths came from the same generator
    Nk: Optional[int] = None         # keys per plane (total keys for varlen); None: Nk == N
    varlen_k: Optional[tuple] = None  # key lengths per sequence (packed cross-attention)

    @property
    def n_keys(self) -> int:
        return self.N if self.Nk is None else self.Nk

    @property
    def is_cross(self) -> bool:
        return self.Nk is not None

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(D), rounded to fp32 so both sides use the same value."""
        return float(np.float32(1.0 / math.sqrt(self.D)))

    def flops(self) -> float:
        """Attention-forward FLOPs: 4*D per (query, key) pair, N^2 pairs per (b,h),
        halved when causal.

        For varlen the sum runs over sequences.  The causal halving is the
        usual convention (it counts N^2/2 pairs, not N(N+1)/2).  With Nq
        queries and Nk keys the pairs are Nq*Nk, and under the causal mask
        (last query aligned with the last key) Nq*Nk - Nq^2/2 when Nq <= Nk,
        else Nk^2/2: the same convention, which gives N^2/2 at Nq == Nk.
        """
        def pairs(nq, nk):
            if not self.causal:
                return float(nq) * nk
            return float(nq) * nk - nq * nq / 2.0 if nq <= nk else nk * nk / 2.0
        if self.varlen is not None:
            lk = self.varlen_k if self.varlen_k is not None else self.varlen
            return 4.0 * self.H * self.D * sum(pairs(a, b) for a, b in zip(self.varlen, lk))
        return 4.0 * self.B * self.H * self.D * pairs(self.N, self.n_keys)

    def hbm_bytes(self) -> float:
        """Algorithmic HBM bytes: Q, K, V read once, O and LSE written once."""
        elt = 4 if self.dtype == "f32" else 2
        planes = self.H if self.varlen is not None else self.B * self.H
        rows, keys = planes * self.N, planes * self.n_keys
        return (2.0 * rows + 2.0 * keys) * self.D * elt + rows * 4.0


def _varlen_lengths(seed: int, nseq: int, lo: int, hi: int) -> tuple:
    rng = np.random.default_rng(seed)
    return tuple(int(x) for x in rng.integers(lo, hi + 1, size=nseq))


def _mk(name, dtype, B, H, N, D, causal, seed, qk_std=1.0, generator="default_rng", varlen=None,
        len_draw=None, Nk=None, varlen_k=None):
    return Workload(name, dtype, B, H, N, D, causal, seed, qk_std, generator, varlen, len_draw,
                    Nk, varlen_k)


def _varlen_workload() -> Workload:
    lens = _varlen_lengths(7, 16, 256, 8192)
    return _mk("bf16_varlen_causal_h32_d128", "bf16", len(lens), 32, sum(lens), 128, True, 7,
               varlen=lens, len_draw=(16, 256, 8192))


WORKLOADS = {
    "f32_causal_b2_h4_n128_d64": _mk("f32_causal_b2_h4_n128_d64", "f32", 2, 4, 128, 64, True, 0,
                                     generator="legacy"),
    "bf16_b4_h16_n2048_d64": _mk("bf16_b4_h16_n2048_d64", "bf16", 4, 16, 2048, 64, False, 0),
    "bf16_causal_b2_h32_n8192_d128": _mk("bf16_causal_b2_h32_n8192_d128", "bf16", 2, 32, 8192,
                                         128, True, 0),
    "bf16_causal_b1_h16_n32768_d128_peaked": _mk("bf16_causal_b1_h16_n32768_d128_peaked", "bf16",
                                                 1, 16, 32768, 128, True, 0, qk_std=2.0),
    "bf16_varlen_causal_h32_d128": _varlen_workload(),
}

# The workload the throughput line is quoted on (bf16, causal, D=128, N=8192).
HEADLINE = "bf16_causal_b2_h32_n8192_d128"

# Cross-attention cases: a 2048-token chunk of queries against 8192 keys
# (the chunk's own keys are the last 2048, so causal alignment is bottom-right),
# and 8192 queries against a 1024-key memory without a mask.
CROSS_WORKLOADS = {
    "bf16_cross_causal_b2_h32_nq2048_nk8192_d128": _mk(
        "bf16_cross_causal_b2_h32_nq2048_nk8192_d128", "bf16", 2, 32, 2048, 128, True, 0,
        Nk=8192),
    "bf16_cross_b2_h32_nq8192_nk1024_d128": _mk(
        "bf16_cross_b2_h32_nq8192_nk1024_d128", "bf16", 2, 32, 8192, 128, False, 0, Nk=1024),
}


def custom(dtype="bf16", B=1, H=1, N=128, D=128, causal=True, seed=0, qk_std=1.0,
           varlen=None, name="custom", Nk=None, varlen_k=None) -> Workload:
    """A workload of arbitrary shape drawn with the default_rng recipe.

    ``Nk`` (dense) or ``varlen_k`` (packed, one key length per sequence) gives
    the keys another length than the queries.
    """
    if varlen is not None:
        varlen = tuple(int(x) for x in varlen)
        B, N = len(varlen), int(sum(varlen))
        if varlen_k is not None:
            varlen_k = tuple(int(x) for x in varlen_k)
            if len(varlen_k) != len(varlen):
                raise ValueError("varlen_k needs one length per sequence")
            Nk = int(sum(varlen_k))
    elif varlen_k is not None:
        raise ValueError("varlen_k needs varlen")
    return _mk(name, dtype, B, H, N, D, causal, seed, qk_std, "default_rng", varlen, Nk=Nk,
               varlen_k=varlen_k)


def cu_seqlens_of(lengths) -> np.ndarray:
    """Offsets [0, L0, L0+L1, ...] as int32 (the packed-sequence index)."""
    out = np.zeros(len(lengths) + 1, dtype=np.int32)
    out[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return out


def _round_f16(x32: np.ndarray):
    """fp32 -> IEEE fp16 with round-to-nearest-even."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x32)).to(torch.float16)


def _round_bf16(x32: np.ndarray):
    """fp32 -> bf16 with round-to-nearest-even (torch's conversion)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16)


def generate(w: Workload, as_torch=True):
    """Draw Q, K, V for workload ``w`` on the host.

    Returns a dict with ``q``, ``k``, ``v`` as CPU torch tensors in the
    storage dtype (bf16 or fp32), ``cu_seqlens`` (int32 numpy or None) and
    ``shape`` (the tensor shape).  The oracle reads the same tensors through
    :func:`as_f64`.
    """
    import torch
    shape = (w.H, w.N, w.D) if w.varlen is not None else (w.B, w.H, w.N, w.D)
    kshape = shape[:-2] + (w.n_keys, w.D)
    if w.generator == "legacy":
        np.random.seed(w.seed)
        q = np.random.randn(*shape).astype(np.float32)
        k = np.random.randn(*kshape).astype(np.float32)
        v = np.random.randn(*kshape).astype(np.float32)
    else:
        rng = np.random.default_rng(w.seed)
        if w.len_draw is not None:
            # the lengths were drawn first from the same generator
            nseq, lo, hi = w.len_draw
            rng.integers(lo, hi + 1, size=nseq)
        q = rng.standard_normal(shape, dtype=np.float32)
        k = rng.standard_normal(kshape, dtype=np.float32)
        v = rng.standard_normal(kshape, dtype=np.float32)
    if w.qk_std != 1.0:
        q *= np.float32(w.qk_std)
        k *= np.float32(w.qk_std)
    if w.dtype == "bf16":
        tq, tk, tv = _round_bf16(q), _round_bf16(k), _round_bf16(v)
    elif w.dtype == "f16":
        tq, tk, tv = _round_f16(q), _round_f16(k), _round_f16(v)
    else:
        tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(a)) for a in (q, k, v))
    cu = cu_seqlens_of(w.varlen) if w.varlen is not None else None
    cuk = cu_seqlens_of(w.varlen_k) if w.varlen_k is not None else None
    return {"q": tq, "k": tk, "v": tv, "cu_seqlens": cu, "cu_seqlens_k": cuk, "shape": shape}


def as_f64(t) -> np.ndarray:
    """Exact widening of a CPU torch tensor (bf16 or fp32) to a float64 array."""
    import torch
    return t.detach().to("cpu").to(torch.float32).numpy().astype(np.float64)
