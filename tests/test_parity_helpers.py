"""The GPU parity tests' comparison helper, checked on the CPU: it reports
near-zero errors for the oracle's own results, and it sees a mistake of the
size the tolerances are meant to catch in every output and on exactly the
heads it is asked to check."""

import numpy as np
import torch

import oracle
import parity as P
from io_aware_exact_tiled_gb300 import workloads as W


def case():
    w = W.Workload("helper", 2, 2, 256, 64)
    x = W.make_inputs(w, seed=3)
    x.blockmask = torch.tensor([[0, 0], [1, 1]], dtype=torch.uint8)  # query block 0 sees no key
    O, L = oracle.forward(x.q, x.k, x.v, x.scale, blockmask=x.blockmask)
    dq, dk, dv = oracle.backward(x.q, x.k, x.v, x.do, x.scale, blockmask=x.blockmask)
    g = {"o": O.astype(np.float32), "lse": L.astype(np.float32), "dq": dq, "dk": dk, "dv": dv}
    return x, g


def test_oracle_results_pass():
    x, g = case()
    e = P.errors(x, g)
    assert e["o"] < 1e-6 and e["lse"] < 1e-5 and max(e["dq"], e["dk"], e["dv"]) < 1e-6


def test_each_output_mistake_is_seen():
    x, g0 = case()
    for name, change, tol in [("o", lambda a: a.__setitem__((1, 0, 200, 5), a[1, 0, 200, 5] + 0.05), P.TOL_O),
                              ("lse", lambda a: a.__setitem__((0, 1, 131), a[0, 1, 131] + 0.01), P.TOL_L),
                              ("dq", lambda a: a.__imul__(1.05), P.TOL_G),
                              ("dk", lambda a: a.__setitem__(slice(None), a[..., ::-1, :]), P.TOL_G),
                              ("dv", lambda a: a.__imul__(-1.0), P.TOL_G)]:
        g = {n: a.copy() for n, a in g0.items()}
        change(g[name])
        assert P.errors(x, g)[name] > tol, name
    # swapped gradients
    g = dict(g0, dk=g0["dv"], dv=g0["dk"])
    e = P.errors(x, g)
    assert e["dk"] > P.TOL_G and e["dv"] > P.TOL_G


def test_only_the_listed_heads_are_compared():
    x, g0 = case()
    g = {n: a.copy() for n, a in g0.items()}
    g["o"][0, 1] += 1.0                                  # head (0, 1) wrong
    assert P.errors(x, g, heads=[(0, 0), (1, 1)], backward=False)["o"] < 1e-6
    assert P.errors(x, g, heads=[(1, 1), (0, 1)], backward=False)["o"] > 0.5


def test_rows_that_see_no_key_must_agree_on_minus_infinity():
    x, g0 = case()
    g = {n: a.copy() for n, a in g0.items()}
    assert np.isneginf(g["lse"][:, :, :128]).all()
    g["lse"][1, 1, 7] = 0.0                              # a finite L where the oracle has -inf
    assert not P.errors(x, g, backward=False)["lse"] <= P.TOL_L
