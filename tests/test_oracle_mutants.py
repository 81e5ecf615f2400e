"""Planted mistakes in the oracle must be caught by its pins (CPU).

Each mutant changes one thing in an in-memory copy of one oracle module (a
dropped term, a wrong sign, an off-by-one mask, a transposed or wrong
operand, a missing rescale, a wrong constant), is installed in place of that
module's functions, and the module's pins (``tests/test_oracle*.py``) are run
against it: at least one must fail. The unmutated copy of every module must
pass all of them. The mistakes live only in these copies; no oracle file is
ever changed.
"""

import importlib
import types

import pytest

import oracle
from oracle import attention as A
from oracle import decode as DEC
from oracle import dropout as DR
from oracle import fp8 as F8
from oracle import varlen as VL

COPY = "oracle_mutant_copy"


def load_copy(module, replace=None):
    src = open(module.__file__).read()
    if replace is not None:
        old, new = replace
        assert src.count(old) == 1, old
        src = src.replace(old, new)
    mod = types.ModuleType(COPY)
    mod.__file__ = module.__file__
    mod.__package__ = "oracle"            # the copy's relative imports reach the real package
    exec(compile(src, module.__file__, "exec"), mod.__dict__)
    return mod


def install(monkeypatch, module, copy):
    for name, obj in vars(copy).items():
        if isinstance(obj, types.FunctionType) and obj.__module__ == COPY:
            if getattr(oracle, name, None) is getattr(module, name, None):
                monkeypatch.setattr(oracle, name, obj)
            monkeypatch.setattr(module, name, obj)


def pins(test_module, calls):
    t = importlib.import_module(test_module)
    return [(f"{fn}{args}", (lambda fn=fn, args=args: getattr(t, fn)(*args))) for fn, args in calls]


BATTERY = {
    "attention": ("test_oracle", [
        ("test_golden_two_keys", ()), ("test_scale_applied_before_max", ()), ("test_visible_definition", ()),
        ("test_causal_row0_is_v0", ()), ("test_fully_masked_rows", ()),
        ("test_rows_sum_to_one_and_masks_exact", (37, 8)),
        ("test_identical_keys_give_mean_of_visible_values", (False, None, False)),
        ("test_identical_keys_give_mean_of_visible_values", (True, None, False)),
        ("test_identical_keys_give_mean_of_visible_values", (False, 9, False)),
        ("test_identical_keys_give_mean_of_visible_values", (False, None, True)),
        ("test_tiled_online_softmax_equals_direct", (64, 16)), ("test_D_equals_rowsum_P_dP", ()),
        ("test_against_torch_sdpa_fp64", (33, 8)), ("test_finite_difference_gradients", (8, 4))]),
    "decode": ("test_oracle_decode", [
        ("test_identical_keys_give_mean_of_valid_values", ()), ("test_single_key_and_empty_cache", ()),
        ("test_against_torch_sdpa_with_mask", ()), ("test_square_case_equals_dense_oracle_with_key_padding", ()),
        ("test_split_and_merge_equals_direct", (7,)), ("test_merge_ignores_empty_splits_and_is_order_free", ())]),
    "varlen": ("test_oracle_varlen", [
        ("test_identical_keys_give_mean_of_visible_values", (True,)), ("test_sequences_do_not_see_each_other", ()),
        ("test_matches_padded_batch_with_key_padding", (True,)), ("test_against_torch_sdpa_per_sequence", ()),
        ("test_finite_difference_gradients", (True,))]),
    "dropout": ("test_oracle_dropout", [
        *[("test_philox_known_answers", kat) for kat in importlib.import_module("test_oracle_dropout").KAT],
        ("test_mask_layout_matches_scalar_restatement", ()), ("test_threshold_is_the_nearest_byte_rate", ()),
        ("test_keep_rate_is_binomial", ()), ("test_zero_rate_is_the_dense_definition", ()),
        ("test_finite_differences", (True,)), ("test_D_identity_with_dropout", ())]),
    "fp8": ("test_oracle_fp8", [
        ("test_e4m3_round_matches_torch_float8", ()), ("test_e4m3_grid_points_and_ties", ()),
        ("test_power_of_two_invariance_of_rounding", ()), ("test_hadamard_and_rotation", (8,)),
        ("test_hadamard_is_the_sylvester_matrix", (8,)), ("test_block_scales_are_tight_powers_of_two", ()),
        ("test_values_on_the_grid_and_identical_keys_give_mean_of_values", ()),
        ("test_close_to_exact_attention", ()), ("test_rotation_lowers_error_with_outlier_channels", ()),
        ("test_key_padding_rows_and_empty_rows", ()), ("test_definition_weights_match_torch_float8_conversion", ()),
        ("test_online_model_equals_definition_away_from_subnormals", ()),
        ("test_online_model_within_the_shift_bound_on_wide_scores", ()),
        ("test_online_model_rescales_within_the_shift_bound", ())]),
}

MODULES = {"attention": A, "decode": DEC, "varlen": VL, "dropout": DR, "fp8": F8}

# (module, what the mistake is, text in the module's file, replacement); each text occurs once
MUTANTS = [
    ("attention", "scale dropped from S", "s = scale * (q @ k.T)", "s = (q @ k.T)"),
    ("attention", "Q K^T transposed", "s = scale * (q @ k.T)", "s = scale * (k @ q.T)"),
    ("attention", "causal mask off by one", "vis &= j[None, :] <= i[:, None]", "vis &= j[None, :] < i[:, None]"),
    ("attention", "causal mask reversed", "vis &= j[None, :] <= i[:, None]", "vis &= j[None, :] >= i[:, None]"),
    ("attention", "key padding off by one", "vis &= j[None, :] < int(kv_len_b)", "vis &= j[None, :] <= int(kv_len_b)"),
    ("attention", "tile mask transposed", "bm[(i // tile)[:, None], (j // tile)[None, :]]",
     "bm[(j // tile)[None, :], (i // tile)[:, None]]"),
    ("attention", "row maximum not subtracted in the sum", "lsum = e.sum(axis=1)", "lsum = np.exp(s).sum(axis=1)"),
    ("attention", "max dropped from L", "L[b, h, rr] = np.where(lsum > 0, m + np.log(",
     "L[b, h, rr] = np.where(lsum > 0, 0.0 + np.log("),
    ("attention", "log2 instead of natural log in L", "m + np.log(np.where(lsum > 0, lsum, 1.0))",
     "m + np.log2(np.where(lsum > 0, lsum, 1.0))"),
    ("attention", "empty row L = 0", "lsum, 1.0)), -np.inf)\n    return O, L\n\n\ndef row_stat_D",
     "lsum, 1.0)), 0.0)\n    return O, L\n\n\ndef row_stat_D"),
    ("attention", "D subtracted with the wrong sign", "ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))",
     "ds = p * (dp + (p * dp).sum(axis=1, keepdims=True))"),
    ("attention", "D term dropped", "ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))", "ds = p * dp"),
    ("attention", "dP from K instead of V", "dp = do_c @ v[b, h].T", "dp = do_c @ k[b, h].T"),
    ("attention", "scale dropped from dQ", "dq[b, h, rr] = scale * (ds @ k[b, h])", "dq[b, h, rr] = (ds @ k[b, h])"),
    ("attention", "dK from V instead of Q", "dk_bh += scale * (ds.T @ q[b, h, rr])",
     "dk_bh += scale * (ds.T @ v[b, h, rr])"),
    ("attention", "scale applied to dV", "dv_bh += p.T @ do_c", "dv_bh += scale * (p.T @ do_c)"),
    ("attention", "D summed over the wrong axis", "(_f64(do) * _f64(o)).sum(axis=-1)",
     "(_f64(do) * _f64(o)).sum(axis=-2)[..., None]"),
    ("attention", "online rescale inverted", "corr = np.exp(m - shift)", "corr = np.exp(shift - m)"),
    ("attention", "running sum not rescaled", "lsum = corr * lsum + pt.sum(axis=1)", "lsum = lsum + pt.sum(axis=1)"),
    ("attention", "running output not rescaled", "o = corr[:, None] * o + pt @ v[cols]", "o = o + pt @ v[cols]"),

    ("decode", "max dropped from L", "L[b] = (m + np.log(lsum))[..., 0]", "L[b] = np.log(lsum)[..., 0]"),
    ("decode", "one cached key too many", "n = int(cl[b])", "n = min(Nk, int(cl[b]) + 1)"),
    ("decode", "scale dropped in the splits", "s = scale * (q[b] @ k[b, :, j0:j1].transpose(0, 2, 1))",
     "s = (q[b] @ k[b, :, j0:j1].transpose(0, 2, 1))"),
    ("decode", "split ignores the cache length", "min(Nk, (c + 1) * split, int(cl[b]))", "min(Nk, (c + 1) * split)"),
    ("decode", "ragged last split dropped", "S = -(-Nk // split)", "S = Nk // split"),
    ("decode", "merge weights inverted", "w = np.exp(m - shift[..., None])", "w = np.exp(shift[..., None] - m)"),
    ("decode", "partial sums merged unweighted", "lt = (w * lsum).sum(axis=-1)", "lt = lsum.sum(axis=-1)"),
    ("decode", "merged L without the maximum", "L = np.where(ok, shift + np.log(", "L = np.where(ok, 0.0 + np.log("),

    ("varlen", "causal flag not passed on", "scale, causal=causal)\n        O[s:e]", "scale, causal=False)\n        O[s:e]"),
    ("varlen", "keys taken from the batch start", "_seq(k, s, e), _seq(v, s, e), scale, causal=causal)\n        O",
     "_seq(k, 0, e - s), _seq(v, 0, e - s), scale, causal=causal)\n        O"),
    ("varlen", "output rows reversed", "O[s:e] = o[0].transpose(1, 0, 2)", "O[s:e] = o[0].transpose(1, 0, 2)[::-1]"),
    ("varlen", "dK and dV swapped", "zip((dq, dk, dv), g)", "zip((dq, dv, dk), g)"),
    ("varlen", "L of the next sequence's slot", "L[:, s:e] = lse[0]", "L[:, s:e] = np.roll(lse[0], 1, axis=-1)"),

    ("dropout", "Philox multipliers swapped", "p0 = np.uint64(PHILOX_M0) * c0", "p0 = np.uint64(PHILOX_M1) * c0"),
    ("dropout", "nine Philox rounds", "for _ in range(10):", "for _ in range(9):"),
    ("dropout", "second key word not bumped", "k1 = (k1 + np.uint64(PHILOX_W1)) & M", "k1 = k1 & M"),
    ("dropout", "Philox output words swapped", "(hi1 ^ c1 ^ k0) & M, lo1, (hi0 ^ c3 ^ k1) & M, lo0",
     "(hi1 ^ c1 ^ k0) & M, lo0, (hi0 ^ c3 ^ k1) & M, lo1"),
    ("dropout", "head and batch counters swapped", "np.uint64(h), np.uint64(b),", "np.uint64(b), np.uint64(h),"),
    ("dropout", "key byte chosen by the row", "byte = (w >> ((j & np.uint64(3))", "byte = (w >> ((i & np.uint64(3))"),
    ("dropout", "keep test off by one", "return byte >= np.uint64(t)", "return byte > np.uint64(t)"),
    ("dropout", "threshold rounded down", "round(256.0 * float(p))", "int(256.0 * float(p))"),
    ("dropout", "kept probabilities not rescaled", "O[b, h, rr] = (P * Z / keep) @ v[b, h]", "O[b, h, rr] = (P * Z) @ v[b, h]"),
    ("dropout", "dP without the mask", "dP = (do[b, h, rr] @ v[b, h].T) * Zs", "dP = (do[b, h, rr] @ v[b, h].T)"),
    ("dropout", "dV without the mask", "dv_bh += (P * Zs).T @ do[b, h, rr]", "dv_bh += P.T @ do[b, h, rr]"),

    ("fp8", "subnormal floor one binade low", "e = np.maximum(e, -6.0)", "e = np.maximum(e, -7.0)"),
    ("fp8", "two mantissa bits", "step = np.exp2(e - 3.0)", "step = np.exp2(e - 2.0)"),
    ("fp8", "ties rounded away from zero", "r = np.round(a / step) * step", "r = np.floor(a / step + 0.5) * step"),
    ("fp8", "no saturation", "r = np.minimum(r, E4M3_MAX)", "r = r"),
    ("fp8", "Hadamard blocks in another order", "h = np.block([[h, h], [h, -h]])", "h = np.block([[h, h], [-h, h]])"),
    ("fp8", "signs applied to columns", "(s[:, None] * hadamard(d))", "(hadamard(d) * s[None, :])"),
    ("fp8", "block scale rounded down", "np.exp2(np.ceil(np.log2(amax / E4M3_MAX)))",
     "np.exp2(np.floor(np.log2(amax / E4M3_MAX)))"),
    ("fp8", "block maximum without the absolute value", "sc[b] = pow2_scale(float(np.abs(blk).max())",
     "sc[b] = pow2_scale(float(blk.max())"),
    ("fp8", "rotation folded as 1/sqrt(d)", "s_fold = scale / d if rotate else scale",
     "s_fold = scale / np.sqrt(d) if rotate else scale"),
    ("fp8", "V not scaled per head", "sv = pow2_scale(float(np.abs(v[b, h]).max()))\n            v8",
     "sv = 1.0\n            v8"),
    ("fp8", "weights relative to the ceiling", "M = np.floor(np.where(np.isfinite(xm), xm, 0.0))",
     "M = np.ceil(np.where(np.isfinite(xm), xm, 0.0))"),
    ("fp8", "L left in log2 units", "(M + np.log2(np.where(lx > 0, lx, 1.0))) * np.log(2.0)",
     "(M + np.log2(np.where(lx > 0, lx, 1.0)))"),
    ("fp8", "online sums not rescaled", "l8 *= alpha\n", "l8 *= 1.0\n"),
    ("fp8", "online output not rescaled", "o *= alpha[:, None]", "o *= 1.0"),
    ("fp8", "online unrounded sum not rescaled", "lx *= alpha\n", "lx *= 1.0\n"),
    ("fp8", "shift bound over the normal weights", "sub = np.isfinite(x) & (w < 2.0 ** -6)",
     "sub = np.isfinite(x) & (w >= 2.0 ** -6)"),
]


def failing_pins(monkeypatch, module_name, copy):
    install(monkeypatch, MODULES[module_name], copy)
    failed = []
    for name, pin in pins(*BATTERY[module_name]):
        try:
            pin()
        except Exception:  # an assertion, or an error the mistake causes
            failed.append(name)
    monkeypatch.undo()
    return failed


@pytest.mark.parametrize("module_name", sorted(MODULES))
def test_unmutated_copy_passes_every_pin(monkeypatch, module_name):
    assert failing_pins(monkeypatch, module_name, load_copy(MODULES[module_name])) == []


@pytest.mark.parametrize("module_name,name,old,new", MUTANTS, ids=[f"{m[0]}: {m[1]}" for m in MUTANTS])
def test_pins_catch_planted_mistake(monkeypatch, module_name, name, old, new):
    failed = failing_pins(monkeypatch, module_name, load_copy(MODULES[module_name], (old, new)))
    assert failed, f"no pin of the {module_name} oracle caught: {name}"
