"""fp64 oracle for decoding: a few query rows against a long key/value cache,
and the split-key procedure (Flash-Decoding) that computes it.

Test infrastructure only: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline leg. The product path never uses it.

Sources:

* "FlashAttention: making attention IO-aware", section "In practice", the
  note on decoding: with one query row against a long KV cache the
  query-block parallelism has nothing to split, so Flash-Decoding splits the
  keys across thread blocks and merges the partial results with the same
  logsumexp rescaling that the online softmax uses.
* "Why is FlashAttention faster?", section "FlashAttention is not KV-cache
  compression": one-token decode reads the cache and builds no N x N matrix.

Readings where the pages are silent:

* Shapes: q [B, H, Nq, d] (Nq new query rows, usually 1); the cache k, v
  [B, H, Nk, d]; cache_len[b] valid keys of batch element b (0 <= cache_len[b]
  <= Nk), the rest of the cache being unused capacity.
* Every query row of batch element b sees every valid key (no mask among
  the cache keys). With Nq = 1 this is the decode step the note describes.
* A split holds ``split`` consecutive keys. Its partial result is the
  running maximum m, the sum l of exp(s - m) and the unnormalised output
  o = sum exp(s - m) v over its valid keys; a split with no valid key has
  m = -inf, l = 0, o = 0 and drops out of the merge. The merge takes
  M = max m, l = sum exp(m_c - M) l_c, O = sum exp(m_c - M) o_c / l and
  L = M + log l (natural log), as in the online-softmax update.
* A row with no valid key has O = 0 and L = -inf.
"""

from __future__ import annotations

import numpy as np

from .attention import _f64


def _cache_len(cache_len, B, Nk):
    if cache_len is None:
        return np.full(B, Nk, dtype=np.int64)
    c = np.asarray(cache_len.cpu() if hasattr(cache_len, "cpu") else cache_len, dtype=np.int64)
    if c.shape != (B,) or np.any(c < 0) or np.any(c > Nk):
        raise ValueError("cache_len must hold B values in [0, Nk]")
    return c


def decode_forward(q, k, v, scale: float, cache_len=None):
    """Direct definition. Returns (O [B,H,Nq,d], L [B,H,Nq]) in fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    cl = _cache_len(cache_len, B, Nk)
    O = np.zeros((B, H, Nq, d))
    L = np.full((B, H, Nq), -np.inf)
    for b in range(B):
        n = int(cl[b])
        if n == 0:
            continue
        s = scale * (q[b] @ k[b, :, :n].transpose(0, 2, 1))   # [H, Nq, n]
        m = s.max(axis=-1, keepdims=True)
        e = np.exp(s - m)
        lsum = e.sum(axis=-1, keepdims=True)
        O[b] = (e / lsum) @ v[b, :, :n]
        L[b] = (m + np.log(lsum))[..., 0]
    return O, L


def split_partials(q, k, v, scale: float, split: int, cache_len=None):
    """Per-split partial results over key blocks of ``split`` keys.

    Returns (m, l, o) with shapes [B,H,Nq,S], [B,H,Nq,S], [B,H,Nq,S,d] for
    S = ceil(Nk / split) splits."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    cl = _cache_len(cache_len, B, Nk)
    S = -(-Nk // split)
    m = np.full((B, H, Nq, S), -np.inf)
    lsum = np.zeros((B, H, Nq, S))
    o = np.zeros((B, H, Nq, S, d))
    for b in range(B):
        for c in range(S):
            j0, j1 = c * split, min(Nk, (c + 1) * split, int(cl[b]))
            if j1 <= j0:
                continue
            s = scale * (q[b] @ k[b, :, j0:j1].transpose(0, 2, 1))
            mc = s.max(axis=-1)
            e = np.exp(s - mc[..., None])
            m[b, :, :, c] = mc
            lsum[b, :, :, c] = e.sum(axis=-1)
            o[b, :, :, c] = e @ v[b, :, j0:j1]
    return m, lsum, o


def merge_partials(m, lsum, o):
    """Logsumexp merge of split partials. Returns (O, L)."""
    M = m.max(axis=-1)
    seen = np.isfinite(M)
    shift = np.where(seen, M, 0.0)
    w = np.exp(m - shift[..., None])  # exp(m_c - M); 0 for empty splits
    lt = (w * lsum).sum(axis=-1)
    ot = (w[..., None] * o).sum(axis=-2)
    ok = lt > 0
    O = np.where(ok[..., None], ot / np.where(ok, lt, 1.0)[..., None], 0.0)
    with np.errstate(divide="ignore"):
        L = np.where(ok, shift + np.log(np.where(ok, lt, 1.0)), -np.inf)
    return O, L


def split_decode(q, k, v, scale: float, split: int, cache_len=None):
    """Flash-Decoding in fp64: split partials followed by the merge."""
    return merge_partials(*split_partials(q, k, v, scale, split, cache_len))
