"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded inputs and measure the errors with the
tolerances of the method (bf16 inputs from N(0, 1)):

  O max-abs error <= 1e-2, L max-abs error <= 1e-3,
  dQ, dK, dV relative Frobenius error <= 2e-2.
"""

import numpy as np
import torch

import io_aware_exact_tiled_gb300 as fa
import oracle

TOL_O = 1e-2
TOL_L = 1e-3
TOL_G = 2e-2


def to_dev(x, dev):
    return None if x is None else x.to(dev)


def run_gpu(x, dev, backward=True):
    q, k, v, do = (t.to(dev) for t in (x.q, x.k, x.v, x.do))
    bm, kl = to_dev(x.blockmask, dev), to_dev(x.kv_len, dev)
    o, lse = fa.forward(q, k, v, scale=x.scale, causal=x.causal, blockmask=bm, kv_len=kl)
    out = {"o": o, "lse": lse}
    if backward:
        dq, dk, dv = fa.backward(q, k, v, o, lse, do, scale=x.scale, causal=x.causal, blockmask=bm, kv_len=kl)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    return {n: t.float().cpu().numpy() for n, t in out.items()}


def rel(a, b):
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def errors(x, g, heads=None, backward=True):
    """Errors of GPU results `g` against the oracle, on all heads or on the
    listed (b, h) heads (heads are independent, so a head is checked whole)."""
    kw = dict(causal=x.causal, kv_len=x.kv_len, blockmask=x.blockmask, heads=heads)
    O, L = oracle.forward(x.q, x.k, x.v, x.scale, **kw)
    sel = (slice(None),) if heads is None else tuple(np.array(ix) for ix in zip(*heads))
    e = {}
    o_ref, l_ref = O[sel], L[sel]
    e["o"] = float(np.abs(g["o"][sel] - o_ref).max())
    lg = g["lse"][sel]
    both_inf = np.isneginf(lg) & np.isneginf(l_ref)
    with np.errstate(invalid="ignore"):  # -inf - -inf on rows that see no key, replaced by 0
        e["lse"] = float(np.where(both_inf, 0.0, np.abs(lg - l_ref)).max())
    if backward:
        dq, dk, dv = oracle.backward(x.q, x.k, x.v, x.do, x.scale, **kw)
        e["dq"] = rel(g["dq"][sel], dq[sel])
        e["dk"] = rel(g["dk"][sel], dk[sel])
        e["dv"] = rel(g["dv"][sel], dv[sel])
    return e


def check(e):
    assert e["o"] <= TOL_O, e
    assert e["lse"] <= TOL_L, e
    for n in ("dq", "dk", "dv"):
        if n in e:
            assert e[n] <= TOL_G, e
