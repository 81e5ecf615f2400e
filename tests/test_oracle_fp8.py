"""Pins for the FP8 forward oracle (no GPU).

The FP8 path approximates attention, so the oracle restates the algorithm's
steps ("FlashAttention: making attention IO-aware", section
"FlashAttention-3", FP8 with incoherent processing). These tests tie each
step to something outside the oracle: the E4M3 rounding to torch's own
float8_e4m3fn conversion, the Hadamard matrix to its defining identities,
the block scales to their bounds, the whole forward to closed forms (values
already on the FP8 grid, identical keys), to exact attention within the
format's error, and the rotation to its stated purpose (lower error when Q
and K carry outlier channels). The weights of the definition are checked
against torch's own E4M3 conversion, and the single-pass model of step 5
(`fp8_forward_online`) against the definition: equal when no weight is in
E4M3's subnormal range, within `fp8_shift_bound` otherwise.
"""

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import fp8 as F8


def test_e4m3_round_matches_torch_float8():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 200.0)])
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    # x is fp64 here; torch rounds from fp32, so compare on values exact in fp32
    x32 = x.astype(np.float32).astype(np.float64)
    np.testing.assert_array_equal(F8.e4m3_round(x32), ref)


def test_e4m3_grid_points_and_ties():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    grid = codes[np.isfinite(codes)]
    np.testing.assert_array_equal(F8.e4m3_round(grid), grid)           # representable values are fixed points
    assert F8.e4m3_round(np.array([448.0, 500.0, -1e6])).tolist() == [448.0, 448.0, -448.0]  # saturation
    # ties go to the even mantissa: 1 + 1/16 lies between 1 and 1.125
    assert F8.e4m3_round(np.array([1.0625, 1.1875]))[0] == 1.0
    assert F8.e4m3_round(np.array([1.1875]))[0] == 1.25
    assert F8.e4m3_round(np.array([2.0 ** -10]))[0] == 0.0            # half the smallest subnormal, ties to 0
    assert F8.e4m3_round(np.array([3 * 2.0 ** -10]))[0] == 2.0 ** -8


def test_power_of_two_invariance_of_rounding():
    """Reading 5: scaling by 2^k commutes with the rounding in the normal range."""
    rng = np.random.default_rng(1)
    p = rng.uniform(2.0 ** -5, 1.9, 5000)
    for k in range(0, 8):
        np.testing.assert_array_equal(F8.e4m3_round(p * 2.0 ** k), F8.e4m3_round(p) * 2.0 ** k)


@pytest.mark.parametrize("d", [1, 2, 8, 64, 128])
def test_hadamard_and_rotation(d):
    h = F8.hadamard(d)
    np.testing.assert_array_equal(h @ h.T, d * np.eye(d))
    signs = np.where(np.random.default_rng(d).random(d) < 0.5, -1.0, 1.0)
    R = F8.rotation(signs)
    np.testing.assert_allclose(R @ R.T, np.eye(d), atol=1e-14)
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal((5, d)), rng.standard_normal((7, d))
    np.testing.assert_allclose((q @ R) @ (k @ R).T, q @ k.T, atol=1e-12)


@pytest.mark.parametrize("d", [2, 8, 128])
def test_hadamard_is_the_sylvester_matrix(d):
    """Reading 1 names Sylvester's construction: its entry (i, j) is
    (-1)^popcount(i AND j), a closed form independent of the recursion (and
    the order of the fast Walsh-Hadamard butterflies)."""
    i, j = np.meshgrid(np.arange(d), np.arange(d), indexing="ij")
    odd = np.vectorize(lambda x: bin(int(x)).count("1") & 1)(i & j)
    np.testing.assert_array_equal(F8.hadamard(d), np.where(odd == 1, -1.0, 1.0))


def test_block_scales_are_tight_powers_of_two():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((300, 16)) * np.repeat([0.01, 5.0, 900.0], 100)[:, None]
    x8, sc = F8.quantize_rows(x, 128)
    assert sc.shape == (3,)
    for b, s in enumerate(sc):
        blk = x[b * 128:(b + 1) * 128]
        assert np.log2(s) == np.round(np.log2(s))
        assert np.abs(blk).max() / s <= 448.0 < 2 * np.abs(blk).max() / s
    deq = F8.dequantize_rows(x8, sc, 128)
    big = np.abs(x) >= np.repeat(sc, 128)[:300, None] * 2.0 ** -6   # normal range of the format
    assert np.all(np.abs(deq - x)[big] <= np.abs(x)[big] * 2.0 ** -4 + 1e-300)


def test_values_on_the_grid_and_identical_keys_give_mean_of_values():
    """Without rotation, Q, K, V already on the FP8 grid quantise exactly; with
    every key equal, every probability is the same and O is the mean of V."""
    rng = np.random.default_rng(4)
    B, H, N, d = 1, 2, 200, 16
    grid = lambda shape: F8.e4m3_round(rng.standard_normal(shape))
    q, v = grid((B, H, N, d)), grid((B, H, N, d))
    k = np.broadcast_to(grid((B, H, 1, d)), (B, H, N, d)).copy()
    O, L = F8.fp8_forward(q, k, v, 0.3, np.ones(d), causal=True, rotate=False)
    for h in range(H):
        csum = np.cumsum(v[0, h], axis=0) / np.arange(1, N + 1)[:, None]
        np.testing.assert_allclose(O[0, h], csum, atol=1e-12)
        s = 0.3 * q[0, h] @ k[0, h, 0]
        np.testing.assert_allclose(L[0, h], s + np.log(np.arange(1, N + 1)), atol=1e-12)


def test_close_to_exact_attention():
    rng = np.random.default_rng(5)
    B, H, N, d = 1, 2, 256, 64
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    O8, L8 = F8.fp8_forward(q, k, v, 1 / np.sqrt(d), signs, causal=True)
    O, L = A.forward(q, k, v, 1 / np.sqrt(d), causal=True)
    assert np.abs(O8 - O).max() < 0.15
    assert np.linalg.norm(O8 - O) / np.linalg.norm(O) < 0.05
    assert np.abs(L8 - L).max() < 0.1


def test_rotation_lowers_error_with_outlier_channels():
    """Q and K with a few channels 30x larger than the rest: block scales are
    set by the outliers, the rest lose precision unless the rotation spreads
    the outliers over all channels."""
    ratios = []
    for seed in range(4):
        rng = np.random.default_rng(10 + seed)
        B, H, N, d = 1, 1, 256, 64
        q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
        out = rng.choice(d, 3, replace=False)
        q[..., out] *= 30.0
        k[..., out] *= 30.0
        scale = 1 / np.sqrt(d) / 10.0
        O, _ = A.forward(q, k, v, scale)
        signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
        e_rot = np.linalg.norm(F8.fp8_forward(q, k, v, scale, signs)[0] - O)
        e_plain = np.linalg.norm(F8.fp8_forward(q, k, v, scale, signs, rotate=False)[0] - O)
        ratios.append(e_plain / e_rot)
    assert np.median(ratios) > 1.5, ratios


def test_key_padding_rows_and_empty_rows():
    rng = np.random.default_rng(6)
    B, H, N, d = 2, 1, 130, 16
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    signs = np.ones(d)
    O, L = F8.fp8_forward(q, k, v, 0.25, signs, kv_len=np.array([1, 0]))
    # one valid key: every row is that key's (quantised) value row
    _, _, _, _, v8, sv = F8.quantized_inputs(q[0, 0], k[0, 0], v[0, 0], signs)
    np.testing.assert_allclose(O[0, 0], np.broadcast_to(v8[0] * sv, O[0, 0].shape), atol=1e-14)
    assert np.all(O[1] == 0) and np.all(np.isneginf(L[1]))


def test_definition_weights_match_torch_float8_conversion():
    """Step 5 of the definition with the weights rounded by torch's
    float8_e4m3fn conversion (a library routine the oracle does not use):
    weights relative to floor(row max), O normalised by their sum."""
    rng = np.random.default_rng(8)
    B, H, N, d = 1, 2, 256, 32
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    k *= 2.0   # wide scores: many weights in the subnormal range
    scale = 1 / np.sqrt(d)
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    O, L = F8.fp8_forward(q, k, v, scale, signs, causal=True)
    T = np.diag(signs) @ F8.hadamard(d)
    vis = np.tril(np.ones((N, N), dtype=bool))
    for h in range(H):
        q8, sq = F8.quantize_rows(q[0, h] @ T)
        k8, sk = F8.quantize_rows(k[0, h] @ T)
        sv = F8.pow2_scale(float(np.abs(v[0, h]).max()))
        vd = F8.e4m3_round(v[0, h] / sv) * sv
        x = np.where(vis, scale / d * (F8.dequantize_rows(q8, sq) @ F8.dequantize_rows(k8, sk).T), -np.inf)
        x = x * np.log2(np.e)
        w = np.exp2(x - np.floor(x.max(axis=1, keepdims=True)))
        p8 = torch.from_numpy(w).to(torch.float8_e4m3fn).to(torch.float64).numpy()
        assert (p8[vis] < 2.0 ** -6).sum() > 1000   # the subnormal range is exercised
        np.testing.assert_allclose(O[0, h], (p8 @ vd) / p8.sum(axis=1, keepdims=True), atol=1e-13)


def test_online_model_equals_definition_away_from_subnormals():
    """With every weight far from E4M3's subnormal range (scores spread by
    less than 5 in log2 units, so no tile raises the reference past the
    threshold either) the single-pass model equals the definition."""
    rng = np.random.default_rng(7)
    B, H, N, d = 1, 1, 384, 16
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    scale = 0.05
    O, L = F8.fp8_forward(q, k, v, scale, np.ones(d), rotate=False)
    O1, L1 = F8.fp8_forward_online(q, k, v, scale, np.ones(d), rotate=False)
    x = scale * (q[0, 0] @ k[0, 0].T) * np.log2(np.e)
    assert (x.max(axis=1) - x.min(axis=1)).max() < 5.0
    assert np.all(F8.fp8_shift_bound(q, k, v, scale, np.ones(d), rotate=False) == 0.0)
    np.testing.assert_allclose(O1, O, atol=1e-13)
    np.testing.assert_allclose(L1, L, atol=1e-12)


def test_online_model_within_the_shift_bound_on_wide_scores():
    """Wide scores (K x 2, causal, N = 512): the model's references trail the
    final maxima, so weights in the subnormal range round differently; every
    element stays within the derived bound, and the bound is not vacuous."""
    rng = np.random.default_rng(12)
    B, H, N, d = 1, 2, 512, 64
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    k *= 2.0
    scale = 1 / np.sqrt(d)
    signs = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    O, _ = F8.fp8_forward(q, k, v, scale, signs, causal=True)
    O1, _ = F8.fp8_forward_online(q, k, v, scale, signs, causal=True)
    bound = F8.fp8_shift_bound(q, k, v, scale, signs, causal=True)
    diff = np.abs(O1 - O)
    assert diff.max() > 1e-3                      # the two roundings do differ
    assert np.all(diff <= bound + 1e-12)
    assert np.median(bound[diff > 0]) < 0.2       # and the bound is informative


def test_online_model_rescales_within_the_shift_bound():
    """Keys whose scores grow tile by tile (K x 1, 4, 8 over three 128-key
    tiles): most rows see a later tile exceed the reference by more than 7,
    so the model moves its reference and rescales its sums. O stays within
    the derived bound of the definition, and L (from the unrounded weights)
    equals the definition's."""
    rng = np.random.default_rng(13)
    B, H, N, d = 1, 1, 384, 16
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    k *= np.repeat([1.0, 4.0, 8.0], 128)[None, None, :, None]
    scale = 0.17
    x = scale * (q[0, 0] @ k[0, 0].T) * np.log2(np.e)
    tmax = x.reshape(N, 3, 128).max(axis=2)
    moved = (tmax[:, 1] - np.floor(tmax[:, 0]) > 7) | (tmax[:, 2] - np.floor(tmax[:, :2].max(axis=1)) > 7)
    assert moved.mean() > 0.5
    O, L = F8.fp8_forward(q, k, v, scale, None, rotate=False)
    O1, L1 = F8.fp8_forward_online(q, k, v, scale, None, rotate=False)
    bound = F8.fp8_shift_bound(q, k, v, scale, None, rotate=False)
    assert np.all(np.abs(O1 - O) <= bound + 1e-12)
    np.testing.assert_allclose(L1, L, atol=1e-12)
