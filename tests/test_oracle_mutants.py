"""Planted mistakes in the attention oracle must be caught by its pins (CPU).

Each mutant changes one thing in a copy of ``oracle/attention.py`` (a dropped
term, a wrong sign, an off-by-one mask, a transposed or wrong operand, a
missing rescale), is installed in place of the oracle's functions, and the
pins of ``tests/test_oracle.py`` are run against it: at least one must fail.
The unmutated copy must pass all of them. The mistakes live only in these
in-memory copies; the oracle's file is never changed.
"""

import importlib
import types

import pytest

import oracle
from oracle import attention as A

PUBLIC = ("visible", "scores", "probabilities", "forward", "backward", "tiled_forward", "row_stat_D")

# (name, text in oracle/attention.py, replacement): each text occurs exactly once
MUTANTS = [
    ("scale dropped from S", "s = scale * (q @ k.T)", "s = (q @ k.T)"),
    ("Q K^T transposed", "s = scale * (q @ k.T)", "s = scale * (k @ q.T)"),
    ("causal mask off by one", "vis &= j[None, :] <= i[:, None]", "vis &= j[None, :] < i[:, None]"),
    ("causal mask reversed", "vis &= j[None, :] <= i[:, None]", "vis &= j[None, :] >= i[:, None]"),
    ("key padding off by one", "vis &= j[None, :] < int(kv_len_b)", "vis &= j[None, :] <= int(kv_len_b)"),
    ("tile mask transposed", "bm[(i // tile)[:, None], (j // tile)[None, :]]",
     "bm[(j // tile)[None, :], (i // tile)[:, None]]"),
    ("row maximum not subtracted in the sum", "lsum = e.sum(axis=1)", "lsum = np.exp(s).sum(axis=1)"),
    ("max dropped from L", "L[b, h, rr] = np.where(lsum > 0, m + np.log(",
     "L[b, h, rr] = np.where(lsum > 0, 0.0 + np.log("),
    ("log2 instead of natural log in L", "m + np.log(np.where(lsum > 0, lsum, 1.0))",
     "m + np.log2(np.where(lsum > 0, lsum, 1.0))"),
    ("empty row L = 0", "lsum, 1.0)), -np.inf)\n    return O, L\n\n\ndef row_stat_D",
     "lsum, 1.0)), 0.0)\n    return O, L\n\n\ndef row_stat_D"),
    ("D subtracted with the wrong sign", "ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))",
     "ds = p * (dp + (p * dp).sum(axis=1, keepdims=True))"),
    ("D term dropped", "ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))", "ds = p * dp"),
    ("dP from V instead of V^T", "dp = do_c @ v[b, h].T", "dp = do_c @ k[b, h].T"),
    ("scale dropped from dQ", "dq[b, h, rr] = scale * (ds @ k[b, h])", "dq[b, h, rr] = (ds @ k[b, h])"),
    ("dK from V instead of Q", "dk_bh += scale * (ds.T @ q[b, h, rr])", "dk_bh += scale * (ds.T @ v[b, h, rr])"),
    ("scale applied to dV", "dv_bh += p.T @ do_c", "dv_bh += scale * (p.T @ do_c)"),
    ("D summed over the wrong axis", "(_f64(do) * _f64(o)).sum(axis=-1)", "(_f64(do) * _f64(o)).sum(axis=-2)[..., None]"),
    ("online rescale inverted", "corr = np.exp(m - shift)", "corr = np.exp(shift - m)"),
    ("running sum not rescaled", "lsum = corr * lsum + pt.sum(axis=1)", "lsum = lsum + pt.sum(axis=1)"),
    ("running output not rescaled", "o = corr[:, None] * o + pt @ v[cols]", "o = o + pt @ v[cols]"),
]


def load_copy(replace=None):
    src = open(A.__file__).read()
    if replace is not None:
        old, new = replace
        assert src.count(old) == 1, old
        src = src.replace(old, new)
    mod = types.ModuleType("oracle_attention_copy")
    mod.__file__ = A.__file__
    exec(compile(src, A.__file__, "exec"), mod.__dict__)
    return mod


def install(monkeypatch, mod):
    for name in PUBLIC:
        monkeypatch.setattr(A, name, getattr(mod, name))
        monkeypatch.setattr(oracle, name, getattr(mod, name))


def battery():
    """The pins, each with one representative parameter set."""
    t = importlib.import_module("test_oracle")
    return [
        ("golden two keys", t.test_golden_two_keys),
        ("scale before max", t.test_scale_applied_before_max),
        ("visible definition", t.test_visible_definition),
        ("causal row 0", t.test_causal_row0_is_v0),
        ("fully masked rows", t.test_fully_masked_rows),
        ("rows sum to one", lambda: t.test_rows_sum_to_one_and_masks_exact(37, 8)),
        *[(f"identical keys {c}", (lambda c=c: t.test_identical_keys_give_mean_of_visible_values(*c)))
          for c in [(False, None, False), (True, None, False), (False, 9, False), (False, None, True)]],
        ("tiled = direct", lambda: t.test_tiled_online_softmax_equals_direct(64, 16)),
        ("D identity", t.test_D_equals_rowsum_P_dP),
        ("torch SDPA fp64", lambda: t.test_against_torch_sdpa_fp64(33, 8)),
        ("finite differences", lambda: t.test_finite_difference_gradients(8, 4)),
    ]


def caught_by(monkeypatch, mod):
    install(monkeypatch, mod)
    failed = []
    for name, pin in battery():
        try:
            pin()
        except Exception:  # an assertion, or a shape error the mistake causes
            failed.append(name)
    monkeypatch.undo()
    return failed


def test_unmutated_copy_passes_every_pin(monkeypatch):
    assert caught_by(monkeypatch, load_copy()) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(monkeypatch, name, old, new):
    failed = caught_by(monkeypatch, load_copy((old, new)))
    assert failed, f"no pin caught: {name}"
