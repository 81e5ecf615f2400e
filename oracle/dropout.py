"""fp64 oracle for attention with fused dropout on the probabilities.

Test infrastructure only: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline leg. The product path never uses it.

Sources: "Why is FlashAttention faster?", section "Kernel fusion removes
stage boundaries" (masking, softmax and dropout become stages of one fused
kernel instead of separate passes), and "FlashAttention: making attention
IO-aware", section "Attention is memory-bound" (dropout is one of the
elementwise steps a standard implementation runs as its own pass). The
backward pass regenerates the same dropout decisions instead of storing the
N x N mask ("The backward pass: recompute, don't store").

What is computed, for dropout rate p and keep mask Z (1 = kept):

    O = (softmax(S) * Z / (1 - p)) V,   L = logsumexp(S)  (dropout after softmax)

and the gradients of <dO, O>, with P = softmax(S):

    dV = (P * Z / (1 - p))^T dO,  dP = (dO V^T) * Z / (1 - p),
    D = rowsum(dO * O) = rowsum(P * dP),  dS = P * (dP - D),
    dQ = scale * dS K,  dK = scale * dS^T Q.

Readings where the pages are silent:

* Random numbers: a counter-based generator, Philox-4x32-10 (Salmon,
  Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3",
  SC 2011), implemented here from that definition; the CUDA side has its
  own implementation.
* One generator call covers a block of 4 query rows x 4 keys of one (b, h):
  key = (seed mod 2^32, seed div 2^32), counter = (i div 4, j div 4, h, b);
  output word (i mod 4) holds the four keys' bytes, key (j mod 4) in byte
  (j mod 4) counted from the least significant.
* A byte u in 0..255 keeps its element iff u >= t with t = round(256 p)
  (0 <= t <= 255): the effective rate is t / 256, and 1 / (1 - t / 256)
  rescales the kept elements.
* Masks (causal, key padding) apply before the softmax as in the dense
  oracle; dropout acts on the probabilities of the visible keys.
"""

from __future__ import annotations

import numpy as np

from .attention import _f64, backward as dense_backward, forward as dense_forward, probabilities, scores, visible

PHILOX_M0, PHILOX_M1 = 0xD2511F53, 0xCD9E8D57
PHILOX_W0, PHILOX_W1 = 0x9E3779B9, 0xBB67AE85


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox-4x32 with 10 rounds on arrays of 32-bit counters (uint64
    arrays holding 32-bit values); returns the four output words."""
    M = np.uint64(0xFFFFFFFF)
    c0, c1, c2, c3 = (np.asarray(x, dtype=np.uint64) & M for x in (c0, c1, c2, c3))
    k0 = np.asarray(k0, dtype=np.uint64) & M
    k1 = np.asarray(k1, dtype=np.uint64) & M
    for _ in range(10):
        p0 = np.uint64(PHILOX_M0) * c0          # < 2^64: exact in uint64
        p1 = np.uint64(PHILOX_M1) * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & M
        hi1, lo1 = p1 >> np.uint64(32), p1 & M
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & M, lo1, (hi0 ^ c3 ^ k1) & M, lo0
        k0 = (k0 + np.uint64(PHILOX_W0)) & M
        k1 = (k1 + np.uint64(PHILOX_W1)) & M
    return c0, c1, c2, c3


def threshold(p: float) -> int:
    """Byte threshold t = round(256 p), clamped to 0..255."""
    return int(min(255, max(0, round(256.0 * float(p)))))


def keep_mask(b: int, h: int, rows, N: int, seed: int, p: float) -> np.ndarray:
    """Keep mask Z [len(rows), N] (bool) of head (b, h) for the given query rows."""
    rows = np.asarray(rows)
    t = threshold(p)
    i = rows[:, None].astype(np.uint64)
    j = np.arange(N, dtype=np.uint64)[None, :]
    words = philox4x32_10(i >> np.uint64(2), j >> np.uint64(2), np.uint64(h), np.uint64(b),
                          np.uint64(seed & 0xFFFFFFFF), np.uint64((seed >> 32) & 0xFFFFFFFF))
    w = np.select([(i & np.uint64(3)) == np.uint64(k) for k in range(4)], list(words))
    byte = (w >> ((j & np.uint64(3)) * np.uint64(8))) & np.uint64(0xFF)
    return byte >= np.uint64(t)


def forward(q, k, v, scale: float, p: float, seed: int, causal: bool = False, kv_len=None, heads=None,
            chunk: int = 1024, rows=None):
    """Attention with dropout on P. Returns (O [B,H,N,d], L [B,H,N]) in fp64.
    ``heads`` optionally restricts the work to a list of (b, h) pairs (the
    other heads are left as NaN) and ``rows`` = (r0, r1) to those query
    rows; query rows are processed in chunks of ``chunk`` rows, each holding
    whole rows of S, P and Z."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    keep = 1.0 - threshold(p) / 256.0
    O = np.full((B, H, N, d), np.nan)
    _, L = dense_forward(q, k, v, scale, causal=causal, kv_len=kv_len, heads=heads, chunk=chunk, rows=rows)
    lo, hi = (0, N) if rows is None else rows
    kl = None if kv_len is None else np.asarray(kv_len.cpu() if hasattr(kv_len, "cpu") else kv_len)
    want = None if heads is None else set(heads)
    for b in range(B):
        for h in range(H):
            if want is not None and (b, h) not in want:
                continue
            for r0 in range(lo, hi, chunk):
                rr = np.arange(r0, min(hi, r0 + chunk))
                vis = visible(N, causal, None if kl is None else int(kl[b]), None, rr)
                P, _, _ = probabilities(scores(q[b, h, rr], k[b, h], scale, vis))
                Z = keep_mask(b, h, rr, N, seed, p)
                O[b, h, rr] = (P * Z / keep) @ v[b, h]
    return O, L


def backward(q, k, v, do, scale: float, p: float, seed: int, causal: bool = False, kv_len=None, heads=None,
             chunk: int = 1024, rows=None):
    """Gradients of <dO, O> for the dropout forward. Returns (dQ, dK, dV);
    ``heads``, ``rows`` and ``chunk`` as for `forward` (dK and dV sum the
    contributions of the rows taken)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, d = q.shape
    keep = 1.0 - threshold(p) / 256.0
    dq, dk, dv = np.full_like(q, np.nan), np.full_like(k, np.nan), np.full_like(v, np.nan)
    kl = None if kv_len is None else np.asarray(kv_len.cpu() if hasattr(kv_len, "cpu") else kv_len)
    want = None if heads is None else set(heads)
    for b in range(B):
        for h in range(H):
            if want is not None and (b, h) not in want:
                continue
            dk_bh, dv_bh = np.zeros((N, d)), np.zeros((N, d))
            lo, hi = (0, N) if rows is None else rows
            for r0 in range(lo, hi, chunk):
                rr = np.arange(r0, min(hi, r0 + chunk))
                vis = visible(N, causal, None if kl is None else int(kl[b]), None, rr)
                P, _, _ = probabilities(scores(q[b, h, rr], k[b, h], scale, vis))
                Zs = keep_mask(b, h, rr, N, seed, p) / keep
                dv_bh += (P * Zs).T @ do[b, h, rr]
                dP = (do[b, h, rr] @ v[b, h].T) * Zs
                dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
                dq[b, h, rr] = scale * dS @ k[b, h]
                dk_bh += scale * dS.T @ q[b, h, rr]
            dk[b, h], dv[b, h] = dk_bh, dv_bh
    return dq, dk, dv


__all__ = ["philox4x32_10", "threshold", "keep_mask", "forward", "backward", "dense_backward"]
