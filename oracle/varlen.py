"""fp64 oracle for packed variable-length batches ("varlen").

Test infrastructure only: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline leg. The product path never uses it.

Source: "FlashAttention: making attention IO-aware", section "In practice",
the note on variable lengths without padding. A packed kernel takes one flat
batch of concatenated sequences plus the offsets at which each sequence
starts, so that padding tokens cost nothing.

Readings where that note is silent:

* Layout: token-major packing. q, k, v, o are [total, H, d]. Tokens
  cu_seqlens[b] .. cu_seqlens[b+1]-1 form sequence b, with
  cu_seqlens[0] = 0 and cu_seqlens[B] = total. L is [H, total], the same
  packing per head.
* Self-attention within each sequence: queries and keys share the offsets,
  and a sequence attends only to its own tokens. The causal mask is aligned
  at the start of each sequence, so key j is visible to query i iff j <= i,
  both counted from the sequence start.
* Within one sequence the result is the plain definition (the dense oracle
  of ``attention.py`` applied to that sequence alone). An empty sequence has
  no rows.
"""

from __future__ import annotations

import numpy as np

from .attention import _f64, backward, forward


def _bounds(cu_seqlens):
    cu = np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64)
    if cu.ndim != 1 or cu.size < 1 or cu[0] != 0 or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0 and be non-decreasing")
    return cu


def _seq(x, s, e):
    """Packed [total, H, d] slice of one sequence as a [1, H, n, d] batch."""
    return np.ascontiguousarray(x[s:e].transpose(1, 0, 2))[None]


def forward_varlen(q, k, v, cu_seqlens, scale: float, causal: bool = False):
    """Exact attention over a packed batch. Returns (O [total,H,d], L [H,total])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu = _bounds(cu_seqlens)
    total, H, d = q.shape
    if cu[-1] != total:
        raise ValueError("cu_seqlens[-1] must equal the packed length")
    O = np.zeros((total, H, d))
    L = np.zeros((H, total))
    for b in range(cu.size - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        if e == s:
            continue
        o, lse = forward(_seq(q, s, e), _seq(k, s, e), _seq(v, s, e), scale, causal=causal)
        O[s:e] = o[0].transpose(1, 0, 2)
        L[:, s:e] = lse[0]
    return O, L


def backward_varlen(q, k, v, do, cu_seqlens, scale: float, causal: bool = False):
    """Gradients of <dO, O> over a packed batch. Returns (dQ, dK, dV), each [total,H,d]."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    cu = _bounds(cu_seqlens)
    total, H, d = q.shape
    if cu[-1] != total:
        raise ValueError("cu_seqlens[-1] must equal the packed length")
    dq = np.zeros((total, H, d))
    dk = np.zeros((total, H, d))
    dv = np.zeros((total, H, d))
    for b in range(cu.size - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        if e == s:
            continue
        g = backward(_seq(q, s, e), _seq(k, s, e), _seq(v, s, e), _seq(do, s, e), scale, causal=causal)
        for out, x in zip((dq, dk, dv), g):
            out[s:e] = x[0].transpose(1, 0, 2)
    return dq, dk, dv
