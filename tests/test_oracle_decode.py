"""Pins for the decoding oracle (no GPU).

Ties the direct decode definition and the split-and-merge procedure of
Flash-Decoding ("FlashAttention: making attention IO-aware", section "In
practice") to things outside their own code: closed forms (identical keys,
a single cached key, an empty cache), torch's scaled_dot_product_attention
with an explicit mask, the dense oracle on a square case, and the equality
of split-and-merge with the direct result for every split size.
"""

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import decode as DEC


def inputs(B, H, Nq, Nk, d, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, Nq, d))
    k = rng.standard_normal((B, H, Nk, d))
    v = rng.standard_normal((B, H, Nk, d))
    return q, k, v


def test_identical_keys_give_mean_of_valid_values():
    q, k, v = inputs(3, 2, 2, 40, 8, 0)
    k[:] = k[:, :, :1]
    cl = np.array([40, 7, 1])
    O, L = DEC.decode_forward(q, k, v, 0.3, cl)
    for b in range(3):
        n = cl[b]
        np.testing.assert_allclose(O[b], np.broadcast_to(v[b, :, :n].mean(axis=1)[:, None], O[b].shape), atol=1e-12)
        s = 0.3 * np.einsum("hqd,hd->hq", q[b], k[b, :, 0])
        np.testing.assert_allclose(L[b], s + np.log(n), atol=1e-12)


def test_single_key_and_empty_cache():
    q, k, v = inputs(2, 1, 3, 5, 4, 1)
    O, L = DEC.decode_forward(q, k, v, 0.5, np.array([1, 0]))
    np.testing.assert_allclose(O[0], np.broadcast_to(v[0, :, :1], O[0].shape), atol=1e-14)
    np.testing.assert_allclose(L[0, 0], 0.5 * q[0, 0] @ k[0, 0, 0], atol=1e-13)
    assert np.all(O[1] == 0) and np.all(np.isneginf(L[1]))


def test_against_torch_sdpa_with_mask():
    B, H, Nq, Nk, d = 2, 3, 4, 50, 16
    q, k, v = inputs(B, H, Nq, Nk, d, 2)
    cl = np.array([50, 23])
    O, _ = DEC.decode_forward(q, k, v, 1 / np.sqrt(d), cl)
    mask = torch.zeros(B, 1, Nq, Nk, dtype=torch.bool)
    for b in range(B):
        mask[b, :, :, :cl[b]] = True
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), attn_mask=mask)
    np.testing.assert_allclose(O, ref.numpy(), atol=1e-12)


def test_square_case_equals_dense_oracle_with_key_padding():
    B, H, N, d = 2, 2, 12, 4
    q, k, v = inputs(B, H, N, N, d, 3)
    cl = np.array([12, 5])
    O, L = DEC.decode_forward(q, k, v, 0.7, cl)
    Od, Ld = A.forward(q, k, v, 0.7, kv_len=cl)
    np.testing.assert_allclose(O, Od, atol=1e-12)
    np.testing.assert_allclose(L, Ld, atol=1e-12)


@pytest.mark.parametrize("split", [1, 7, 16, 64, 200])
def test_split_and_merge_equals_direct(split):
    q, k, v = inputs(3, 2, 2, 200, 8, 4)
    cl = np.array([200, 33, 0])
    O, L = DEC.decode_forward(q, k, v, 0.25, cl)
    Os, Ls = DEC.split_decode(q, k, v, 0.25, split, cl)
    np.testing.assert_allclose(Os, O, atol=1e-12)
    with np.errstate(invalid="ignore"):
        np.testing.assert_allclose(np.where(np.isneginf(L), 0, Ls - L), 0, atol=1e-12)
    assert np.array_equal(np.isneginf(Ls), np.isneginf(L))


def test_merge_ignores_empty_splits_and_is_order_free():
    q, k, v = inputs(1, 1, 1, 64, 4, 5)
    m, l, o = DEC.split_partials(q, k, v, 1.0, 16, np.array([20]))
    assert np.isneginf(m[0, 0, 0, 2]) and l[0, 0, 0, 3] == 0
    perm = [3, 1, 0, 2]
    O1, L1 = DEC.merge_partials(m, l, o)
    O2, L2 = DEC.merge_partials(m[..., perm], l[..., perm], o[..., perm, :])
    np.testing.assert_allclose(O1, O2, atol=1e-14)
    np.testing.assert_allclose(L1, L2, atol=1e-14)


def test_rejects_bad_cache_len():
    q, k, v = inputs(1, 1, 1, 8, 4, 6)
    with pytest.raises(ValueError):
        DEC.decode_forward(q, k, v, 1.0, np.array([9]))
