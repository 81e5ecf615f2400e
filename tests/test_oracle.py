"""Pins for the fp64 CPU oracle (no GPU).

The oracle is only trusted because these tests tie it to things other than
itself: a hand-derived worked example, closed forms (identical keys, causal
row 0), the softmax invariants, the online-softmax recurrence, the
D = rowsum(dO * O) identity, central finite differences, and an independent
library routine (torch's scaled_dot_product_attention in fp64 with autograd).
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def mask_cases(N, tile):
    """(causal, kv_len per batch, blockmask) combinations used below."""
    T = -(-N // tile)
    rng = np.random.default_rng(7)
    bm = (rng.random((T, T)) < 0.5).astype(np.uint8)
    np.fill_diagonal(bm, 1)
    bm[0, -1] = 1  # make the mask clearly asymmetric
    bm[-1, 0] = 0 if T > 1 else 1
    return [
        (False, None, None),
        (True, None, None),
        (False, [max(1, N // 2), N], None),
        (False, None, bm),
        (True, [max(1, N - 3), max(1, N // 3)], bm),
    ]


# --------------------------------------------------------------------------
# Hand-derived worked example (tests/golden/two_keys.json)
# --------------------------------------------------------------------------

def test_golden_two_keys():
    g = json.load(open(os.path.join(GOLDEN, "two_keys.json")))
    q, k, v, do = (np.array(g[n]) for n in ("q", "k", "v", "do"))
    s = g["scale"]
    O, L = oracle.forward(q, k, v, s)
    e = g["expect"]
    np.testing.assert_allclose(O[0, 0], e["O"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(L[0, 0], e["L"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(oracle.row_stat_D(do, O)[0, 0], e["D"], atol=1e-13)
    dq, dk, dv = oracle.backward(q, k, v, do, s)
    np.testing.assert_allclose(dq[0, 0], e["dQ"], atol=1e-13)
    np.testing.assert_allclose(dk[0, 0], e["dK"], atol=1e-13)
    np.testing.assert_allclose(dv[0, 0], e["dV"], atol=1e-13)


def test_scale_applied_before_max():
    # Doubling the scale must square the softmax odds exp(s1 - s2).
    q = np.array([[[[1.0, 0.0]]]]).repeat(2, axis=2)
    k = np.array([[[[1.0, 0.0], [0.0, 1.0]]]])
    v = np.array([[[[1.0, 0.0], [0.0, 1.0]]]])
    for scale in (0.5, 1.0, 2.0):
        O, L = oracle.forward(q, k, v, scale)
        # O = [p1, p2] with p1 / p2 = exp(scale)
        assert O[0, 0, 0, 0] / O[0, 0, 0, 1] == pytest.approx(math.exp(scale), rel=1e-12)
        assert L[0, 0, 0] == pytest.approx(math.log(math.exp(scale) + 1.0), rel=1e-12)


# --------------------------------------------------------------------------
# Softmax invariants
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N,tile", [(37, 8), (64, 16)])
def test_rows_sum_to_one_and_masks_exact(N, tile):
    d = 5
    q, k = rnd((N, d), 1), rnd((N, d), 2)
    for causal, kvl, bm in mask_cases(N, tile):
        kb = None if kvl is None else kvl[0]
        vis = A.visible(N, causal, kb, bm, tile=tile)
        p, _, _ = A.probabilities(A.scores(q, k, 0.3, vis))
        has = vis.any(axis=1)
        np.testing.assert_allclose(p.sum(axis=1)[has], 1.0, atol=1e-12)
        assert (p >= 0).all()
        assert (p[~vis] == 0.0).all()
        assert (p[~has] == 0.0).all()


def test_visible_definition():
    N, tile = 12, 4
    bm = np.array([[1, 0, 1], [0, 1, 0], [1, 1, 1]], dtype=np.uint8)
    vis = A.visible(N, causal=True, kv_len_b=10, blockmask=bm, tile=tile)
    for i in range(N):
        for j in range(N):
            want = (j <= i) and (j < 10) and bm[i // tile][j // tile] == 1
            assert vis[i, j] == want, (i, j)


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal,kvl,use_bm", [
    (False, None, False), (True, None, False), (False, 9, False), (False, None, True), (True, 11, True)])
def test_identical_keys_give_mean_of_visible_values(causal, kvl, use_bm):
    N, d, tile = 16, 3, 4
    T = N // tile
    bm = None
    if use_bm:
        bm = np.zeros((T, T), np.uint8)
        np.fill_diagonal(bm, 1)
        bm[0, 3] = 1   # row block 0 sees column block 3, not the reverse
        bm[2, 1] = 1
    krow = rnd((1, d), 3)
    k = np.repeat(krow, N, axis=0)[None, None]
    q = rnd((1, 1, N, d), 4)
    v = rnd((1, 1, N, d), 5)
    scale = 0.7
    O, L = oracle.forward(q, k, v, scale, causal=causal,
                          kv_len=None if kvl is None else [kvl], blockmask=bm, tile=tile)
    for i in range(N):
        js = [j for j in range(N)
              if (not causal or j <= i) and (kvl is None or j < kvl)
              and (bm is None or bm[i // tile][j // tile])]
        s = scale * float(q[0, 0, i] @ krow[0])
        if not js:
            assert (O[0, 0, i] == 0).all() and L[0, 0, i] == -np.inf
            continue
        np.testing.assert_allclose(O[0, 0, i], v[0, 0, js].mean(axis=0), atol=1e-12)
        assert L[0, 0, i] == pytest.approx(s + math.log(len(js)), abs=1e-12)


def test_causal_row0_is_v0():
    N, d = 9, 4
    q, k, v = rnd((1, 2, N, d), 6), rnd((1, 2, N, d), 7), rnd((1, 2, N, d), 8)
    O, L = oracle.forward(q, k, v, 0.4, causal=True)
    np.testing.assert_allclose(O[:, :, 0], v[:, :, 0], atol=1e-14)
    np.testing.assert_allclose(L[:, :, 0], 0.4 * (q[:, :, 0] * k[:, :, 0]).sum(-1), atol=1e-14)


def test_fully_masked_rows():
    N, d, tile = 8, 3, 4
    bm = np.array([[0, 0], [1, 1]], np.uint8)     # query block 0 sees nothing
    q, k, v, do = (rnd((1, 1, N, d), s) for s in (9, 10, 11, 12))
    O, L = oracle.forward(q, k, v, 1.0, blockmask=bm, chunk=3, tile=tile)
    assert (O[0, 0, :4] == 0).all() and (L[0, 0, :4] == -np.inf).all()
    assert np.isfinite(O[0, 0, 4:]).all()
    dq, dk, dv = oracle.backward(q, k, v, do, 1.0, blockmask=bm, chunk=3, tile=tile)
    assert (dq[0, 0, :4] == 0).all()
    Ot, Lt = A.tiled_forward(q[0, 0], k[0, 0], v[0, 0], 1.0, 4, 4, A.visible(N, blockmask=bm, tile=tile))
    np.testing.assert_allclose(Ot, O[0, 0], atol=1e-13)
    assert (Lt[:4] == -np.inf).all()


# --------------------------------------------------------------------------
# Online softmax recurrence = direct definition
# --------------------------------------------------------------------------

@pytest.mark.parametrize("Br,Bc", [(16, 16), (64, 16), (16, 64), (128, 128), (64, 128)])
def test_tiled_online_softmax_equals_direct(Br, Bc):
    N, d, tile = 200, 8, 16          # ragged last tile for every block size
    q, k, v = rnd((N, d), 20), 3.0 * rnd((N, d), 21), rnd((N, d), 22)
    for causal, kvl, bm in mask_cases(N, tile):
        kb = None if kvl is None else kvl[0]
        vis = A.visible(N, causal, kb, bm, tile=tile)
        Ot, Lt = A.tiled_forward(q, k, v, 0.35, Br, Bc, vis)
        Od, Ld = oracle.forward(q[None, None], k[None, None], v[None, None], 0.35,
                                causal=causal, kv_len=None if kb is None else [kb],
                                blockmask=bm, chunk=64, tile=tile)
        np.testing.assert_allclose(Ot, Od[0, 0], atol=1e-12)
        np.testing.assert_allclose(Lt, Ld[0, 0], atol=1e-12)


def test_tiled_with_128_tiles_matches_forward_blockmask():
    N, d = 384, 16
    q, k, v = rnd((N, d), 30), rnd((N, d), 31), rnd((N, d), 32)
    bm = np.array([[1, 0, 1], [1, 1, 0], [0, 0, 1]], np.uint8)
    vis = A.visible(N, blockmask=bm)
    Ot, Lt = A.tiled_forward(q, k, v, 0.25, 128, 128, vis)
    Od, Ld = oracle.forward(q[None, None], k[None, None], v[None, None], 0.25, blockmask=bm)
    np.testing.assert_allclose(Ot, Od[0, 0], atol=1e-12)
    np.testing.assert_allclose(Lt, Ld[0, 0], atol=1e-12)


def test_chunking_does_not_change_result():
    N, d = 70, 6
    q, k, v, do = (rnd((2, 2, N, d), s) for s in (40, 41, 42, 43))
    a = oracle.forward(q, k, v, 0.5, causal=True, kv_len=[50, 70], chunk=1024)
    b = oracle.forward(q, k, v, 0.5, causal=True, kv_len=[50, 70], chunk=7)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-13)
    ga = oracle.backward(q, k, v, do, 0.5, causal=True, kv_len=[50, 70], chunk=1024)
    gb = oracle.backward(q, k, v, do, 0.5, causal=True, kv_len=[50, 70], chunk=9)
    for x, y in zip(ga, gb):
        np.testing.assert_allclose(x, y, atol=1e-12)


# --------------------------------------------------------------------------
# Backward: D identity and finite differences
# --------------------------------------------------------------------------

def test_D_equals_rowsum_P_dP():
    N, d = 48, 7
    q, k, v, do = (rnd((N, d), s) for s in (50, 51, 52, 53))
    for causal, kvl, bm in mask_cases(N, 16):
        kb = None if kvl is None else kvl[0]
        vis = A.visible(N, causal, kb, bm, tile=16)
        p, _, _ = A.probabilities(A.scores(q, k, 0.4, vis))
        O = p @ v
        dP = do @ v.T
        np.testing.assert_allclose(A.row_stat_D(do, O), (p * dP).sum(axis=1), atol=1e-12)


def _loss(q, k, v, do, scale, **kw):
    O, _ = oracle.forward(q, k, v, scale, **kw)
    return float((np.nan_to_num(O) * do).sum())


@pytest.mark.parametrize("N,d", [(5, 3), (8, 4), (16, 3)])
def test_finite_difference_gradients(N, d):
    B, H = 1, 2
    scale = 0.6
    q, k, v, do = (rnd((B, H, N, d), s) for s in (60 + N, 61 + N, 62 + N, 63 + N))
    cases = [dict(), dict(causal=True), dict(kv_len=[max(2, N - 2)])]
    if N > 8:
        cases.append(dict(blockmask=np.array([[1, 1], [0, 1]], np.uint8), tile=8))
        cases.append(dict(causal=True, kv_len=[N - 3], blockmask=np.array([[1, 0], [1, 1]], np.uint8), tile=8))
    h = 1e-6
    for kw in cases:
        dq, dk, dv = oracle.backward(q, k, v, do, scale, **kw)
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp = x.copy(); xp[idx] += h
                xm = x.copy(); xm[idx] -= h
                args = {"q": q, "k": k, "v": v}
                args[name] = xp
                lp = _loss(args["q"], args["k"], args["v"], do, scale, **kw)
                args[name] = xm
                lm = _loss(args["q"], args["k"], args["v"], do, scale, **kw)
                num[idx] = (lp - lm) / (2 * h)
            err = np.abs(num - g).max() / max(1e-12, np.abs(g).max())
            assert err < 1e-6, (name, kw, err)


def test_finite_difference_gradients_blockmask():
    # tile-masked case on a 256-row problem with 128-row tiles (the oracle's tile)
    N, d = 256, 2
    rng = np.random.default_rng(70)
    q, k, v, do = (rng.standard_normal((1, 1, N, d)) for _ in range(4))
    bm = np.array([[1, 1], [0, 1]], np.uint8)
    scale = 0.8
    dq, dk, dv = oracle.backward(q, k, v, do, scale, blockmask=bm)
    h = 1e-6
    # probe a handful of entries in each tensor, on both sides of the mask
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in [(0, 0, 3, 0), (0, 0, 130, 1), (0, 0, 200, 0), (0, 0, 127, 1)]:
            args = {"q": q, "k": k, "v": v}
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], do, scale, blockmask=bm)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], do, scale, blockmask=bm)
            num = (lp - lm) / (2 * h)
            assert abs(num - g[idx]) < 1e-6 * max(1.0, abs(g[idx])), (name, idx, num, g[idx])


# --------------------------------------------------------------------------
# Independent library routine: torch SDPA in fp64 + autograd
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N,d", [(33, 8), (130, 16)])
def test_against_torch_sdpa_fp64(N, d):
    B, H = 2, 3
    scale = 1.0 / math.sqrt(d)
    g = torch.Generator().manual_seed(N)
    q, k, v, do = (torch.randn(B, H, N, d, generator=g, dtype=torch.float64) for _ in range(4))
    T = -(-N // 128)
    bm = torch.ones(T, T, dtype=torch.uint8)
    if T > 1:
        bm[0, 1] = 0
    for causal, kv_len, blockmask in [(False, None, None), (True, None, None),
                                      (False, [N // 2, N], None), (True, [N, N - 5], bm)]:
        mask = torch.ones(B, 1, N, N, dtype=torch.bool)
        i = torch.arange(N)[:, None]
        j = torch.arange(N)[None, :]
        if causal:
            mask &= (j <= i)
        if kv_len is not None:
            for b in range(B):
                mask[b] &= (j < kv_len[b])
        if blockmask is not None:
            mask &= blockmask.bool()[i // 128, j // 128]
        qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
        out = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
        out.backward(do)
        O, L = oracle.forward(q, k, v, scale, causal=causal, kv_len=kv_len, blockmask=blockmask)
        dq, dk, dv = oracle.backward(q, k, v, do, scale, causal=causal, kv_len=kv_len, blockmask=blockmask)
        np.testing.assert_allclose(O, out.detach().numpy(), atol=1e-10)
        np.testing.assert_allclose(dq, qq.grad.numpy(), atol=1e-10)
        np.testing.assert_allclose(dk, kk.grad.numpy(), atol=1e-10)
        np.testing.assert_allclose(dv, vv.grad.numpy(), atol=1e-10)
        s = scale * (q @ k.transpose(-1, -2))
        s = s.masked_fill(~mask, float("-inf"))
        np.testing.assert_allclose(L, torch.logsumexp(s, dim=-1).numpy(), atol=1e-10)


def test_heads_subset():
    q, k, v, do = (rnd((2, 3, 20, 4), s) for s in (80, 81, 82, 83))
    O, L = oracle.forward(q, k, v, 0.5, heads=[(1, 2)])
    Of, Lf = oracle.forward(q, k, v, 0.5)
    np.testing.assert_allclose(O[1, 2], Of[1, 2], atol=0)
    assert np.isnan(O[0, 0]).all()
    dq, dk, dv = oracle.backward(q, k, v, do, 0.5, heads=[(0, 1)])
    gq, gk, gv = oracle.backward(q, k, v, do, 0.5)
    np.testing.assert_allclose(dk[0, 1], gk[0, 1], atol=0)


def test_row_subsets_partition_the_work():
    q, k, v, do = (rnd((1, 2, 300, 5), s) for s in (90, 91, 92, 93))
    kw = dict(causal=True, kv_len=[250])
    O, L = oracle.forward(q, k, v, 0.5, **kw)
    dq, dk, dv = oracle.backward(q, k, v, do, 0.5, **kw)
    parts = [(0, 128), (128, 200), (200, 300)]
    acc_k, acc_v = 0, 0
    for r in parts:
        Os, Ls = oracle.forward(q, k, v, 0.5, rows=r, chunk=50, **kw)
        np.testing.assert_allclose(Os[:, :, r[0]:r[1]], O[:, :, r[0]:r[1]], atol=1e-13)
        gq, gk, gv = oracle.backward(q, k, v, do, 0.5, rows=r, chunk=50, **kw)
        np.testing.assert_allclose(gq[:, :, r[0]:r[1]], dq[:, :, r[0]:r[1]], atol=1e-13)
        acc_k = acc_k + gk
        acc_v = acc_v + gv
    np.testing.assert_allclose(acc_k, dk, atol=1e-12)
    np.testing.assert_allclose(acc_v, dv, atol=1e-12)
