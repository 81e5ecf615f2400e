"""Pins for the dropout oracle (no GPU).

The generator is pinned to the published Philox-4x32-10 known-answer
vectors (Salmon et al., SC 2011), the element-to-bits mapping to a scalar
restatement in plain Python integers, the keep rate to its binomial
expectation, p = 0 to the dense oracle, and the backward to central finite
differences of <dO, O> and to the D = rowsum(P * dP) identity.
"""

import numpy as np
import pytest

from oracle import attention as A
from oracle import dropout as DR

KAT = [((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
       ((0xFFFFFFFF,) * 4, (0xFFFFFFFF, 0xFFFFFFFF), (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
       ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
        (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1))]


@pytest.mark.parametrize("ctr,key,expect", KAT)
def test_philox_known_answers(ctr, key, expect):
    out = DR.philox4x32_10(*ctr, *key)
    assert tuple(int(x) for x in out) == expect


def _scalar_philox(c, k):
    c0, c1, c2, c3 = c
    k0, k1 = k
    for _ in range(10):
        p0, p1 = 0xD2511F53 * c0, 0xCD9E8D57 * c2
        c0, c1, c2, c3 = ((p1 >> 32) ^ c1 ^ k0) & 0xFFFFFFFF, p1 & 0xFFFFFFFF, ((p0 >> 32) ^ c3 ^ k1) & 0xFFFFFFFF, \
            p0 & 0xFFFFFFFF
        k0, k1 = (k0 + 0x9E3779B9) & 0xFFFFFFFF, (k1 + 0xBB67AE85) & 0xFFFFFFFF
    return c0, c1, c2, c3


def test_mask_layout_matches_scalar_restatement():
    seed, p = 0x0123456789ABCDEF, 0.3
    b, h, N = 2, 5, 40
    Z = DR.keep_mask(b, h, np.arange(N), N, seed, p)
    t = DR.threshold(p)
    # every element of the first 16 x 16 block (all four row words and key
    # bytes of 16 generator calls) and the last rows and columns
    points = [(i, j) for i in range(16) for j in range(16)] + [(i, j) for i in (36, 39) for j in range(24, 40)]
    for i, j in points:
        words = _scalar_philox((i // 4, j // 4, h, b), (seed & 0xFFFFFFFF, seed >> 32))
        byte = (words[i % 4] >> (8 * (j % 4))) & 0xFF
        assert Z[i, j] == (byte >= t), (i, j)


def test_threshold_is_the_nearest_byte_rate():
    """The reading t = round(256 p): the effective rate t / 256 is the byte
    rate nearest to p (at most half a step, 1/512, away), for p below the
    last step."""
    for p in np.linspace(0.0, 0.99, 397):
        t = DR.threshold(p)
        assert isinstance(t, int) and 0 <= t <= 255
        assert abs(t / 256 - p) <= 1 / 512 + 1e-12, (p, t)
    assert DR.threshold(0.0) == 0 and DR.threshold(1.0) == 255


def test_keep_rate_is_binomial():
    p = 0.1
    Z = DR.keep_mask(0, 0, np.arange(512), 512, 7, p)
    keep = 1.0 - DR.threshold(p) / 256.0
    n = Z.size
    assert abs(Z.mean() - keep) < 4 * np.sqrt(keep * (1 - keep) / n)
    # heads draw different masks
    assert (DR.keep_mask(0, 1, np.arange(64), 64, 7, p) != DR.keep_mask(0, 0, np.arange(64), 64, 7, p)).any()


def test_zero_rate_is_the_dense_definition():
    rng = np.random.default_rng(0)
    q, k, v, do = (rng.standard_normal((1, 2, 40, 8)) for _ in range(4))
    O, L = DR.forward(q, k, v, 0.4, 0.0, 11, causal=True)
    Od, Ld = A.forward(q, k, v, 0.4, causal=True)
    np.testing.assert_allclose(O, Od, atol=1e-13)
    np.testing.assert_allclose(L, Ld, atol=1e-13)
    g = DR.backward(q, k, v, do, 0.4, 0.0, 11, causal=True)
    gd = A.backward(q, k, v, do, 0.4, causal=True)
    for a, b in zip(g, gd):
        np.testing.assert_allclose(a, b, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences(causal):
    rng = np.random.default_rng(1)
    B, H, N, d = 1, 2, 9, 3
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    args = dict(scale=0.7, p=0.25, seed=99, causal=causal, kv_len=np.array([7]))

    def loss(q_, k_, v_):
        return float((DR.forward(q_, k_, v_, **args)[0] * do).sum())

    g = DR.backward(q, k, v, do, **args)
    h = 1e-6
    for idx, x in enumerate((q, k, v)):
        num = np.zeros_like(x)
        for pos in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[pos] += h
            xm[pos] -= h
            a = [q, k, v]
            a[idx] = xp
            fp = loss(*a)
            a[idx] = xm
            num[pos] = (fp - loss(*a)) / (2 * h)
        assert np.linalg.norm(num - g[idx]) / np.linalg.norm(g[idx]) < 1e-6


def test_D_identity_with_dropout():
    rng = np.random.default_rng(2)
    q, k, v, do = (rng.standard_normal((1, 1, 33, 6)) for _ in range(4))
    O, _ = DR.forward(q, k, v, 0.5, 0.2, 5)
    vis = A.visible(33)
    P, _, _ = A.probabilities(A.scores(q[0, 0], k[0, 0], 0.5, vis))
    Zs = DR.keep_mask(0, 0, np.arange(33), 33, 5, 0.2) / (1 - DR.threshold(0.2) / 256)
    dP = (do[0, 0] @ v[0, 0].T) * Zs
    np.testing.assert_allclose((do[0, 0] * O[0, 0]).sum(axis=1), (P * dP).sum(axis=1), atol=1e-12)


def test_row_chunks_and_head_subsets_do_not_change_the_result():
    """Chunking the query rows and restricting the heads only reorders the
    sums: the chosen heads equal the whole computation's."""
    rng = np.random.default_rng(3)
    B, H, N, d = 1, 3, 100, 8
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    full = DR.forward(q, k, v, 0.3, 0.2, 99, causal=True)
    part = DR.forward(q, k, v, 0.3, 0.2, 99, causal=True, heads=[(0, 2)], chunk=7)
    np.testing.assert_allclose(part[0][0, 2], full[0][0, 2], rtol=0, atol=1e-12)
    gf = DR.backward(q, k, v, do, 0.3, 0.2, 99, causal=True)
    gp = DR.backward(q, k, v, do, 0.3, 0.2, 99, causal=True, heads=[(0, 2)], chunk=7)
    for a, b in zip(gp, gf):
        np.testing.assert_allclose(a[0, 2], b[0, 2], rtol=0, atol=1e-12)
        assert np.isnan(a[0, 0]).all()
