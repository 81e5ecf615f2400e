"""FLOP and byte accounting for exact attention (used by the benchmark).

FLOPs count the dense products of visible (query, key) pairs only:
  forward  4 * d per pair (S = Q K^T and O = P V, 2 flops per multiply-add)
  backward 10 * d per pair (S recomputed, dP = dO V^T, dV, dK, dQ)
Pair counts: N^2 without a mask; N^2 / 2 with a causal mask (the usual
"causal FLOPs halved" convention); N * kv_len[b] with key padding; 128^2 per
kept tile with a tile mask. Work that a mask removes is not counted.

Algorithmic bytes are the unavoidable HBM traffic of each pass: the forward
reads Q, K, V and writes O and L; the backward reads Q, K, V, O, dO, L and
writes dQ, dK, dV.

The "standard attention" helpers restate the worked example of "Why is
FlashAttention faster?" (section "The 4K-token traffic FlashAttention
avoids"): materialising S and P for one head costs a write and a re-read of
two N x N matrices.
"""

from __future__ import annotations

TILE = 128


def pairs_per_batch(N: int, causal: bool = False, kv_len=None, blockmask=None, B: int = 1):
    """Visible (query, key) pairs of one head, for each batch element."""
    out = []
    for b in range(B):
        if blockmask is None and kv_len is None:
            out.append(N * N / 2 if causal else float(N * N))
            continue
        if blockmask is not None and kv_len is None and not causal:
            kept = int((blockmask != 0).sum())
            out.append(float(kept * TILE * TILE))
            continue
        if kv_len is not None and blockmask is None and not causal:
            out.append(float(N * int(kv_len[b])))
            continue
        # mixtures: exact count of visible pairs
        import numpy as np
        i = np.arange(N)[:, None]
        j = np.arange(N)[None, :]
        vis = np.ones((N, N), dtype=bool)
        if causal:
            vis &= j <= i
        if kv_len is not None:
            vis &= j < int(kv_len[b])
        if blockmask is not None:
            bm = np.asarray(blockmask) != 0
            vis &= bm[i // TILE, j // TILE]
        out.append(float(vis.sum()))
    return out


def flops(B: int, H: int, N: int, d: int, causal=False, kv_len=None, blockmask=None):
    """(forward flops, backward flops) summed over all B * H heads."""
    pairs = sum(pairs_per_batch(N, causal, kv_len, blockmask, B)) * H
    return 4.0 * d * pairs, 10.0 * d * pairs


def tensor_bytes(B: int, H: int, N: int, d: int, elem: int) -> int:
    """Bytes of one [B, H, N, d] tensor."""
    return B * H * N * d * elem


def fwd_bytes(B, H, N, d, elem=2) -> int:
    return 4 * tensor_bytes(B, H, N, d, elem) + B * H * N * 4


def bwd_bytes(B, H, N, d, elem=2) -> int:
    return 8 * tensor_bytes(B, H, N, d, elem) + B * H * N * 4


def standard_square_bytes(N: int, elem: int) -> int:
    """Bytes of one materialised N x N score or probability matrix."""
    return N * N * elem


def standard_intermediate_traffic(N: int, elem: int, heads: int = 1) -> int:
    """HBM traffic of writing and re-reading both S and P (per the heads)."""
    return 4 * standard_square_bytes(N, elem) * heads
