"""fp64 oracle for the FP8 forward pass with block scales and a Hadamard
rotation of Q and K.

Test infrastructure only: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline leg. The product path never uses it.

Source: "FlashAttention: making attention IO-aware", section
"FlashAttention-3", the bullet on FP8 with incoherent processing: FP8 doubles
throughput again but is fragile with outliers, so FA3 quantises per block and
first multiplies Q and K by a random orthogonal (Hadamard) matrix, which
spreads outliers across dimensions.

This is an approximation of attention, not an exact method, so the oracle
states the algorithm's steps in order (each in plain fp64 arithmetic on the
values the FP8 format can hold), with these readings where the page is
silent:

1. Rotation. R = diag(s) H_d / sqrt(d), with H_d the Sylvester Hadamard
   matrix (H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]]) and s a vector of
   random signs drawn once and passed in. R is orthogonal, so
   (Q R)(K R)^T = Q K^T: the rotation changes only the quantisation error.
   The values quantised are Q diag(s) H_d = sqrt(d) Q R (and the same for K),
   with the factor 1/d folded into the score scale. Each output is a signed
   sum of bf16 inputs, which fp32 holds exactly unless their exponents span
   more than about 16 binades; a rounding there (2^-24 relative) can change
   an E4M3 code only for a value that close to a rounding boundary, so the
   CUDA side's fp32 transform quantises to the same codes in practice.
2. Format. OCP FP8 E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits;
   normal values 2^(e-7) (1 + m/8), subnormals 2^-6 m/8, largest finite 448,
   no infinities. Conversion rounds to nearest, ties to even, and saturates
   at +-448.
3. Block scales. Each block of 128 rows of one head of the rotated Q and K
   of step 1 gets one scale, and V one scale per head (its P V product sums over every key
   block in one accumulator, so a per-block V scale cannot be applied). A
   scale is the power of two 2^ceil(log2(amax / 448)) (1 for an all-zero
   block), so that x / scale fits the format and every rescaling is exact.
4. Scores. S = (scale_attn / d) * deq(Q8) deq(K8)^T with
   deq(x8) = x8 * scale (1/d undoes the sqrt(d) of step 1 on both sides;
   without the rotation it is 1), masked as in the dense oracle.
5. Probabilities. With x = S log2(e) and M = floor(max_j x_j) over the
   row's visible keys, the weights are p_j = 2^(x_j - M) (in [0, 2)),
   rounded to E4M3 (p8_j). This is the definition `fp8_forward` computes:
   it depends on the row's scores only, not on the order in which a kernel
   visits the keys.
6. Output. O = sum_j p8_j deq(V8_j) / sum_j p8_j (a convex combination of
   the dequantised values), and L = logsumexp_j S_j (natural log) from the
   unrounded weights.

A single-pass kernel cannot know M before it has seen every key, so it
rounds relative to a running integer reference r instead (the online
softmax of "Online softmax"). Rounding to E4M3 commutes with multiplication
by 2^(M - r) except in E4M3's subnormal range (weights below 2^-6), so such a
kernel differs from the definition only through weights p_j < 2^-6. If every
key's weight is rounded relative to some integer r <= M (r may differ from
key to key, as a running reference rises) with 2^(x_j - r) <= 448, each such
weight moves by at most 2^-9 on the scale of M (half a subnormal step,
2^-10, on either side), and O moves by at most
2^-9 sum_{j: p_j < 2^-6} |deq(V8_j) - O| / sum_{j: p_j >= 2^-6} p8_j per
element; `fp8_shift_bound` returns that bound. `fp8_forward_online` models
one such procedure (128-key tiles in order; r set on the first visible tile
and moved to floor(tile maximum) whenever a tile exceeds it by more than 7;
sums rescaled by 2^(r_old - r_new), exactly).
"""

from __future__ import annotations

import numpy as np

from .attention import _f64, visible

E4M3_MAX = 448.0
BLOCK = 128           # rows per quantisation block of Q and K
TILE_KEYS = 128       # keys per tile of the online softmax
RESCALE_LOG2 = 7.0    # move the reference when a tile exceeds it by more than this


def e4m3_round(x) -> np.ndarray:
    """Round to the nearest E4M3 value (ties to even), saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # binade exponent, floored at the subnormal range (spacing 2^-9 below 2^-6)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    step = np.exp2(e - 3.0)
    r = np.round(a / step) * step  # numpy rounds halves to even
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, x)


def hadamard(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order d (a power of two), entries +-1."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def rotation(signs) -> np.ndarray:
    """R = diag(signs) H_d / sqrt(d)."""
    s = np.asarray(signs, dtype=np.float64)
    d = s.size
    return (s[:, None] * hadamard(d)) / np.sqrt(d)


def pow2_scale(amax: float) -> float:
    """Smallest power of two 2^k with amax / 2^k <= 448 (1 for amax = 0)."""
    if amax <= 0:
        return 1.0
    return float(np.exp2(np.ceil(np.log2(amax / E4M3_MAX))))


def quantize_rows(x, rows: int = BLOCK):
    """Block quantisation of a [N, d] matrix: blocks of `rows` rows.

    Returns (x8 [N, d] on the E4M3 grid, scales [ceil(N / rows)])."""
    x = np.asarray(x, dtype=np.float64)
    N = x.shape[0]
    nb = -(-N // rows)
    x8 = np.zeros_like(x)
    sc = np.ones(nb)
    for b in range(nb):
        blk = x[b * rows:(b + 1) * rows]
        sc[b] = pow2_scale(float(np.abs(blk).max()) if blk.size else 0.0)
        x8[b * rows:(b + 1) * rows] = e4m3_round(blk / sc[b])
    return x8, sc


def dequantize_rows(x8, sc, rows: int = BLOCK):
    return x8 * np.repeat(sc, rows)[: x8.shape[0], None]


def quantized_inputs(q, k, v, signs, rows: int = BLOCK, rotate: bool = True):
    """Steps 1-3 for one head ([N, d] arrays): (q8, q scales, k8, k scales,
    v8, v scale), the values on the E4M3 grid as fp64 (``rotate=False``
    skips step 1)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    d = q.shape[-1]
    T = rotation(signs) * np.sqrt(d) if rotate else np.eye(d)
    q8, sq = quantize_rows(q @ T, rows)
    k8, sk = quantize_rows(k @ T, rows)
    sv = pow2_scale(float(np.abs(v).max()))
    return q8, sq, k8, sk, e4m3_round(v / sv), sv


def _heads_fp8(q, k, v, scale, signs, causal, rotate, rows, kv_len):
    """Steps 1-4 per head: yields (b, h, x = S log2 e [N, N] with -inf on
    invisible keys, deq(V8) [N, d])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    # sqrt(d) R = diag(s) H_d: the transform applied to Q and K
    T = rotation(signs) * np.sqrt(d) if rotate else np.eye(d)
    s_fold = scale / d if rotate else scale
    kl = None if kv_len is None else np.asarray(kv_len.cpu() if hasattr(kv_len, "cpu") else kv_len)
    for b in range(B):
        vis = visible(N, causal, None if kl is None else int(kl[b]))
        for h in range(H):
            q8, sq = quantize_rows(q[b, h] @ T, rows)
            k8, sk = quantize_rows(k[b, h] @ T, rows)
            sv = pow2_scale(float(np.abs(v[b, h]).max()))
            v8 = e4m3_round(v[b, h] / sv)
            s = s_fold * (dequantize_rows(q8, sq, rows) @ dequantize_rows(k8, sk, rows).T)
            yield b, h, np.where(vis, s, -np.inf) * np.log2(np.e), v8 * sv


def _definition_weights(x):
    """Step 5 for one head: M = floor(row max) (0 on rows with no visible
    key), unrounded weights w = 2^(x - M) and their E4M3 roundings."""
    xm = x.max(axis=1)
    M = np.floor(np.where(np.isfinite(xm), xm, 0.0))
    w = np.exp2(x - M[:, None])   # invisible keys give 0
    return M, w, e4m3_round(w)


def fp8_forward(q, k, v, scale: float, signs, causal: bool = False, rotate: bool = True, rows: int = BLOCK,
                kv_len=None):
    """FP8 forward of [B, H, N, d] inputs by steps 1-6 (the weights rounded
    relative to the floor of each row's final maximum). Returns (O, L) in
    fp64.

    ``kv_len`` (optional, [B]) masks keys j >= kv_len[b] as in the dense
    oracle; the quantisation of steps 1-3 still covers every row.

    ``rotate=False`` skips step 1 (plain block-quantised FP8), for comparing
    the error with and without the rotation."""
    B, H, N, d = np.shape(q)
    O = np.zeros((B, H, N, d))
    L = np.zeros((B, H, N))
    for b, h, x, vd in _heads_fp8(q, k, v, scale, signs, causal, rotate, rows, kv_len):
        M, w, p8 = _definition_weights(x)
        l8, lx = p8.sum(axis=1), w.sum(axis=1)
        seen = l8 > 0
        O[b, h] = np.where(seen[:, None], (p8 @ vd) / np.where(seen, l8, 1.0)[:, None], 0.0)
        with np.errstate(divide="ignore"):
            L[b, h] = np.where(lx > 0, (M + np.log2(np.where(lx > 0, lx, 1.0))) * np.log(2.0), -np.inf)
    return O, L


def fp8_shift_bound(q, k, v, scale: float, signs, causal: bool = False, rotate: bool = True, rows: int = BLOCK,
                    kv_len=None):
    """Per-element bound [B, H, N, d] on |O' - O| for any computation that
    differs from `fp8_forward` only in rounding each weight relative to an
    integer reference r <= M (any r per key, with 2^(x - r) <= 448) instead
    of M (see the module notes):
    2^-9 sum_{j: w_j < 2^-6} |deq(V8_j) - O| / sum_{j: w_j >= 2^-6} p8_j."""
    B, H, N, d = np.shape(q)
    out = np.zeros((B, H, N, d))
    for b, h, x, vd in _heads_fp8(q, k, v, scale, signs, causal, rotate, rows, kv_len):
        M, w, p8 = _definition_weights(x)
        l8 = p8.sum(axis=1)
        seen = l8 > 0
        O = np.where(seen[:, None], (p8 @ vd) / np.where(seen, l8, 1.0)[:, None], 0.0)
        sub = np.isfinite(x) & (w < 2.0 ** -6)
        lnorm = np.where(sub, 0.0, p8).sum(axis=1)
        for i in range(N):
            if not seen[i]:
                continue
            out[b, h, i] = 2.0 ** -9 * np.abs(vd[sub[i]] - O[i]).sum(axis=0) / lnorm[i]
    return out


def fp8_forward_online(q, k, v, scale: float, signs, causal: bool = False, rotate: bool = True, rows: int = BLOCK,
                       kv_len=None):
    """Steps 1-6 with step 5 done by one single-pass procedure (a model of
    how a kernel that visits 128-key tiles in order can round its weights):
    an integer reference r per row, set to floor(tile maximum) on the first
    tile with a visible key and moved there whenever a tile's maximum
    exceeds r by more than 7; the sums so far are multiplied by
    2^(r_old - r_new) (exact). Weights relative to r are <= 2^8 (inside
    E4M3). It differs from `fp8_forward` within `fp8_shift_bound`.
    Returns (O, L) in fp64."""
    B, H, N, d = np.shape(q)
    O = np.zeros((B, H, N, d))
    L = np.zeros((B, H, N))
    for b, h, x, vd in _heads_fp8(q, k, v, scale, signs, causal, rotate, rows, kv_len):
        m = np.full(N, -np.inf)    # integer reference exponent r per row
        l8 = np.zeros(N)           # sum of the rounded weights
        lx = np.zeros(N)           # sum of the unrounded weights
        o = np.zeros((N, d))
        err = np.seterr(invalid="ignore")  # -inf - (-inf) on rows that have seen no key yet
        for j0 in range(0, N, TILE_KEYS):
            xt = x[:, j0:j0 + TILE_KEYS]
            tmax = xt.max(axis=1)
            first = np.isneginf(m)
            upd = np.isfinite(tmax) & (first | (tmax - m > RESCALE_LOG2))
            m_new = np.where(upd, np.floor(np.where(np.isfinite(tmax), tmax, 0.0)), m)
            alpha = np.where(upd & ~first, np.exp2(np.where(upd & ~first, m - m_new, 0.0)), 1.0)
            m = m_new
            l8 *= alpha
            lx *= alpha
            o *= alpha[:, None]
            mu = np.where(np.isfinite(m), m, 0.0)
            pt = np.exp2(xt - mu[:, None])   # masked keys give 0
            p8 = e4m3_round(pt)
            l8 += p8.sum(axis=1)
            lx += pt.sum(axis=1)
            o += p8 @ vd[j0:j0 + TILE_KEYS]
        np.seterr(**err)
        seen = l8 > 0
        O[b, h] = np.where(seen[:, None], o / np.where(seen, l8, 1.0)[:, None], 0.0)
        with np.errstate(divide="ignore"):
            L[b, h] = np.where(lx > 0, (np.where(np.isfinite(m), m, 0.0) + np.log2(np.where(lx > 0, lx, 1.0)))
                               * np.log(2.0), -np.inf)
    return O, L
