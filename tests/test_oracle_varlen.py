"""Pins for the packed variable-length oracle (no GPU).

The varlen oracle restates "FlashAttention: making attention IO-aware",
section "In practice" (variable lengths without padding), on top of the dense
oracle. These tests tie it to things other than its own code path:
per-sequence closed forms (identical keys give the mean of the visible
values), isolation between sequences, agreement with a padded batch and its
key-padding mask, finite differences of the packed loss, and
torch's scaled_dot_product_attention run on each sequence by hand.
"""

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import varlen as VL


def packed(lens, H, d, seed):
    rng = np.random.default_rng(seed)
    total = int(sum(lens))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    q, k, v, do = (rng.standard_normal((total, H, d)) for _ in range(4))
    return cu, q, k, v, do


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_visible_values(causal):
    lens = [5, 1, 9, 0, 3]
    H, d = 2, 4
    cu, q, k, v, _ = packed(lens, H, d, 0)
    for b in range(len(lens)):
        k[cu[b]:cu[b + 1]] = k[cu[b]]  # every key of a sequence is the same vector
    O, L = VL.forward_varlen(q, k, v, cu, 0.5, causal=causal)
    for b in range(len(lens)):
        s, e = cu[b], cu[b + 1]
        for i in range(s, e):
            n_vis = (i - s + 1) if causal else (e - s)
            np.testing.assert_allclose(O[i], v[s:s + n_vis].mean(axis=0), atol=1e-12)
            sc = 0.5 * (q[i] * k[s]).sum(axis=-1)  # [H]
            np.testing.assert_allclose(L[:, i], sc + np.log(n_vis), atol=1e-12)


def test_sequences_do_not_see_each_other():
    lens = [7, 4, 6]
    cu, q, k, v, _ = packed(lens, 2, 3, 1)
    O, L = VL.forward_varlen(q, k, v, cu, 0.7, causal=False)
    k2, v2 = k.copy(), v.copy()
    k2[cu[1]:cu[2]] += 3.0
    v2[cu[1]:cu[2]] -= 2.0
    O2, L2 = VL.forward_varlen(q, k2, v2, cu, 0.7, causal=False)
    for b in (0, 2):
        sl = slice(cu[b], cu[b + 1])
        np.testing.assert_array_equal(O[sl], O2[sl])
        np.testing.assert_array_equal(L[:, sl], L2[:, sl])
    assert not np.allclose(O[cu[1]:cu[2]], O2[cu[1]:cu[2]])


@pytest.mark.parametrize("causal", [False, True])
def test_matches_padded_batch_with_key_padding(causal):
    """Sequence b of the packed batch equals rows < len_b of a zero-padded
    [B, H, Nmax, d] batch with the key-padding mask kv_len = len_b (and, for
    causal, the same top-left causal mask)."""
    lens = [6, 13, 1, 9]
    H, d = 2, 5
    cu, q, k, v, do = packed(lens, H, d, 2)
    Nmax = max(lens)
    B = len(lens)

    def pad(x):
        out = np.zeros((B, H, Nmax, d))
        for b in range(B):
            out[b, :, :lens[b]] = x[cu[b]:cu[b + 1]].transpose(1, 0, 2)
        return out

    O, L = VL.forward_varlen(q, k, v, cu, 0.4, causal=causal)
    Od, Ld = A.forward(pad(q), pad(k), pad(v), 0.4, causal=causal, kv_len=np.array(lens))
    dq, dk, dv = VL.backward_varlen(q, k, v, do, cu, 0.4, causal=causal)
    # rows past len_b of the padded batch must not feed dK, dV: their dO is 0
    gq, gk, gv = A.backward(pad(q), pad(k), pad(v), pad(do), 0.4, causal=causal, kv_len=np.array(lens))
    for b in range(B):
        n = lens[b]
        sl = slice(cu[b], cu[b + 1])
        np.testing.assert_allclose(O[sl], Od[b, :, :n].transpose(1, 0, 2), atol=1e-12)
        np.testing.assert_allclose(L[:, sl], Ld[b, :, :n], atol=1e-12)
        np.testing.assert_allclose(dq[sl], gq[b, :, :n].transpose(1, 0, 2), atol=1e-12)
        np.testing.assert_allclose(dk[sl], gk[b, :, :n].transpose(1, 0, 2), atol=1e-12)
        np.testing.assert_allclose(dv[sl], gv[b, :, :n].transpose(1, 0, 2), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_finite_difference_gradients(causal):
    lens = [3, 0, 5, 2]
    H, d = 2, 3
    cu, q, k, v, do = packed(lens, H, d, 3)
    scale = 0.6

    def loss(q_, k_, v_):
        O, _ = VL.forward_varlen(q_, k_, v_, cu, scale, causal=causal)
        return float((O * do).sum())

    dq, dk, dv = VL.backward_varlen(q, k, v, do, cu, scale, causal=causal)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            pos = "qkv".index(name)
            args_p[pos], args_m[pos] = xp, xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.linalg.norm(num - g) / max(np.linalg.norm(g), 1e-30)
        assert err < 1e-6, (name, err)


def test_against_torch_sdpa_per_sequence():
    lens = [17, 4, 30]
    H, d = 3, 8
    cu, q, k, v, _ = packed(lens, H, d, 4)
    O, _ = VL.forward_varlen(q, k, v, cu, 1 / np.sqrt(d), causal=True)
    for b in range(len(lens)):
        sl = slice(cu[b], cu[b + 1])
        t = [torch.from_numpy(x[sl].transpose(1, 0, 2).copy())[None] for x in (q, k, v)]
        ref = torch.nn.functional.scaled_dot_product_attention(*t, is_causal=True)
        np.testing.assert_allclose(O[sl], ref[0].numpy().transpose(1, 0, 2), atol=1e-12)


def test_rejects_bad_offsets():
    _, q, k, v, _ = packed([3, 2], 1, 2, 5)
    with pytest.raises(ValueError):
        VL.forward_varlen(q, k, v, np.array([0, 4, 3]), 1.0)
    with pytest.raises(ValueError):
        VL.forward_varlen(q, k, v, np.array([0, 3, 6]), 1.0)
