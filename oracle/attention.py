"""fp64 CPU oracle for exact softmax attention, forward and backward.

Test infrastructure only: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline leg. The product path never uses it.

Sources (web pages on IO-aware exact attention):

* "FlashAttention: making attention IO-aware", section "Attention is memory-bound":
  attention for one head is S = Q K^T, P = softmax(S), O = P V.
* same page, section "Online softmax": softmax subtracts the row maximum; the
  running max / running sum / unnormalised output recurrence gives exactly
  the same result; O = o / l after the last tile.
* same page, section "The backward pass: recompute, don't store": the forward
  saves O and the per-row logsumexp L = m + log l (natural log, as in the
  page's forward listing), and the softmax gradient needs the row sum
  D = rowsum(dO * O).
* same page, forward listing (``flashForward``): the scale 1/sqrt(d) multiplies
  the dot product before the maximum is taken.
* same page, section "FlashAttention-2": causal masking skips tiles above the
  diagonal; section "Counting the IO": block-sparse attention skips tiles a
  sparsity mask zeroes out.
* "Why is FlashAttention faster?", section "Extra computation can still finish
  sooner": the key-padding mask.

What is computed here is the plain definition with S and P materialised
(chunked over query rows only to bound memory; every chunk holds whole rows).
The backward pass is the textbook derivative of that definition, which the
pages do not write out:

    dV = P^T dO,  dP = dO V^T,  dS = P * (dP - rowsum(P * dP)),
    dQ = scale * dS K,  dK = scale * dS^T Q.

Readings where the pages are silent (each is pinned by a test):

* Mask semantics: key j is visible to query i iff (not causal or j <= i) and
  (no key padding or j < kv_len[b]) and (no tile mask or
  blockmask[i // 128][j // 128] != 0). Query rows past kv_len are computed
  normally (they attend to the valid keys).
* A row with no visible key has O = 0, L = -inf, and contributes no gradient.
"""

from __future__ import annotations

import numpy as np

TILE = 128


def _f64(x):
    """Convert a numpy array or torch tensor to a float64 numpy array."""
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if str(x.dtype) in ("torch.bfloat16", "torch.float16"):
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def visible(N: int, causal: bool = False, kv_len_b=None, blockmask=None,
            rows=None, tile: int = TILE) -> np.ndarray:
    """Boolean [len(rows), N]: True where key j is visible to query i.

    Causal (FlashAttention-2 section): j <= i. Key padding ("Why is
    FlashAttention faster?", "Extra computation..."): j < kv_len. Tile mask
    ("Counting the IO", block-sparse): blockmask[i // tile][j // tile] != 0.
    """
    i = np.arange(N) if rows is None else np.asarray(rows)
    j = np.arange(N)
    vis = np.ones((i.size, N), dtype=bool)
    if causal:
        vis &= j[None, :] <= i[:, None]
    if kv_len_b is not None:
        vis &= j[None, :] < int(kv_len_b)
    if blockmask is not None:
        bm = np.asarray(blockmask.cpu() if hasattr(blockmask, "cpu") else blockmask) != 0
        vis &= bm[(i // tile)[:, None], (j // tile)[None, :]]
    return vis


def scores(q, k, scale: float, vis: np.ndarray) -> np.ndarray:
    """S = scale * Q K^T with invisible entries set to -inf (one head)."""
    s = scale * (q @ k.T)
    s[~vis] = -np.inf
    return s


def probabilities(s: np.ndarray):
    """Row softmax with the row maximum subtracted ("Online softmax":
    softmax(s)_k = exp(s_k - m) / sum exp(s - m)).

    Returns (P, m, lsum) where m is the row max and lsum = sum exp(s - m).
    Rows with no finite score give P = 0, m = -inf, lsum = 0.
    """
    m = s.max(axis=1)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe[:, None])          # exp(-inf) = 0 for masked entries
    lsum = e.sum(axis=1)
    p = e / np.where(empty, 1.0, lsum)[:, None]
    p[empty] = 0.0
    return p, m, lsum


def _heads(q, kv_len):
    B, H = q.shape[0], q.shape[1]
    for b in range(B):
        kb = None if kv_len is None else int(np.asarray(kv_len.cpu() if hasattr(kv_len, "cpu") else kv_len)[b])
        for h in range(H):
            yield b, h, kb


def forward(q, k, v, scale: float, causal: bool = False, kv_len=None,
            blockmask=None, chunk: int = 1024, heads=None, tile: int = TILE, rows=None):
    """Exact attention forward on [B, H, N, d] inputs, in fp64.

    O = softmax(scale * Q K^T + mask) V and L = m + log(sum exp(S - m))
    per row (natural log). ``heads`` optionally restricts the work to a list
    of (b, h) pairs; the other heads of the outputs are left as NaN.
    ``tile`` is the edge of the square tiles that ``blockmask`` describes.
    ``rows`` = (r0, r1) optionally restricts the work to those query rows.
    Returns (O [B,H,N,d], L [B,H,N]) as float64 numpy arrays.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    O = np.full((B, H, N, d), np.nan)
    L = np.full((B, H, N), np.nan)
    want = None if heads is None else set(heads)
    for b, h, kb in _heads(q, kv_len):
        if want is not None and (b, h) not in want:
            continue
        lo, hi = (0, N) if rows is None else rows
        for r0 in range(lo, hi, chunk):
            rr = np.arange(r0, min(hi, r0 + chunk))
            vis = visible(N, causal, kb, blockmask, rr, tile)
            s = scores(q[b, h, rr], k[b, h], scale, vis)
            p, m, lsum = probabilities(s)
            O[b, h, rr] = p @ v[b, h]
            with np.errstate(divide="ignore"):
                L[b, h, rr] = np.where(lsum > 0, m + np.log(np.where(lsum > 0, lsum, 1.0)), -np.inf)
    return O, L


def row_stat_D(do, o) -> np.ndarray:
    """D = rowsum(dO * O), the closed form of the softmax-gradient row sum
    ("The backward pass: recompute, don't store")."""
    return (_f64(do) * _f64(o)).sum(axis=-1)


def backward(q, k, v, do, scale: float, causal: bool = False, kv_len=None,
             blockmask=None, chunk: int = 1024, heads=None, tile: int = TILE, rows=None):
    """Gradients of <dO, O> with respect to Q, K, V, in fp64.

    Plain derivative of the definition (not written on the pages):
    dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(P * dP)),
    dQ = scale * dS K, dK = scale * dS^T Q. Masked entries have P = 0 and so
    carry no gradient. ``rows`` = (r0, r1) restricts the sum to those query
    rows (dK, dV then hold only their contribution). Returns (dQ, dK, dV) as
    float64 numpy arrays.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, d = q.shape
    dq = np.full_like(q, np.nan)
    dk = np.full_like(k, np.nan)
    dv = np.full_like(v, np.nan)
    want = None if heads is None else set(heads)
    for b, h, kb in _heads(q, kv_len):
        if want is not None and (b, h) not in want:
            continue
        dk_bh = np.zeros((N, d))
        dv_bh = np.zeros((N, d))
        lo, hi = (0, N) if rows is None else rows
        for r0 in range(lo, hi, chunk):
            rr = np.arange(r0, min(hi, r0 + chunk))
            vis = visible(N, causal, kb, blockmask, rr, tile)
            s = scores(q[b, h, rr], k[b, h], scale, vis)
            p, _, _ = probabilities(s)
            do_c = do[b, h, rr]
            dp = do_c @ v[b, h].T
            ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dq[b, h, rr] = scale * (ds @ k[b, h])
            dk_bh += scale * (ds.T @ q[b, h, rr])
            dv_bh += p.T @ do_c
        dk[b, h] = dk_bh
        dv[b, h] = dv_bh
    return dq, dk, dv


def tiled_forward(q, k, v, scale: float, Br: int, Bc: int, vis: np.ndarray):
    """Tiled forward for one head by the online-softmax recurrence.

    Restates the page's tiled forward ("FlashAttention: making attention
    IO-aware", forward listing and "Online softmax"): for each block of Br
    query rows, stream blocks of Bc keys; keep a running maximum m, a running
    sum l of exp(s - m) and an unnormalised output o; when a block raises the
    maximum, multiply l and o by exp(m_old - m_new); divide once at the end and
    keep L = m + log l. Used only to check that this recurrence reproduces the
    direct definition. ``vis`` is the [N, N] visibility matrix.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, d = q.shape
    O = np.zeros((N, d))
    L = np.zeros(N)
    for i0 in range(0, N, Br):
        rows = slice(i0, min(N, i0 + Br))
        nr = rows.stop - rows.start
        m = np.full(nr, -np.inf)
        lsum = np.zeros(nr)
        o = np.zeros((nr, d))
        for j0 in range(0, N, Bc):
            cols = slice(j0, min(N, j0 + Bc))
            s = scale * (q[rows] @ k[cols].T)
            s[~vis[rows, cols]] = -np.inf
            m_new = np.maximum(m, s.max(axis=1))
            # rows that have seen no visible key yet have m_new = -inf; shift
            # them by 0 instead so that exp() gives 0 rather than NaN
            seen = np.isfinite(m_new)
            shift = np.where(seen, m_new, 0.0)
            corr = np.exp(m - shift)                 # exp(m_old - m_new)
            pt = np.exp(s - shift[:, None])          # masked entries give 0
            lsum = corr * lsum + pt.sum(axis=1)
            o = corr[:, None] * o + pt @ v[cols]
            m = m_new
        ok = lsum > 0
        O[rows] = np.where(ok[:, None], o / np.where(ok, lsum, 1.0)[:, None], 0.0)
        with np.errstate(divide="ignore"):
            L[rows] = np.where(ok, m + np.log(np.where(ok, lsum, 1.0)), -np.inf)
    return O, L
