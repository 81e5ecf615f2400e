"""GPU parity of fused dropout (fa_fwd_dropout / fa_bwd_dropout) against the
dropout oracle.

The keep mask is regenerated on both sides from Philox-4x32-10 (the oracle's
implementation is pinned to the published known-answer vectors), so the
outputs are compared element by element with the tolerances of the dense
path adapted to dropout (O within 1e-2 / keep + 2^-8 |O| elementwise, see
check_o), L <= 1e-3, gradients relative Frobenius <= 2e-2. A wrong mask
(a different bit layout, a swapped query and key) changes O by far more.
"""

import numpy as np
import pytest
import torch

from io_aware_exact_tiled_gb300 import binding as fb
from io_aware_exact_tiled_gb300 import workloads as W
import oracle
from oracle import dropout as DR

from parity import TOL_G, TOL_L, TOL_O, rel

SEED = 0x1234_5678_9ABC_DEF0


def check_o(o, O, p):
    """O within 1e-2 / keep + 2^-8 |O| elementwise. With dropout a row of O
    is no longer a convex combination of V (kept weights are divided by the
    keep rate and do not sum to one), so |O| can pass 4, where one rounding
    step of the bf16 output is already 2^-6: the bound adds the output's own
    bf16 quantum (2^-8 relative) to the dense path's 1e-2, scaled by 1 / keep."""
    keep = 1.0 - DR.threshold(p) / 256.0
    err = np.abs(o - O)
    bound = TOL_O / keep + np.abs(O) * 2.0 ** -8
    assert np.all(err <= bound), (float(err.max()), float((err / bound).max()))


def run(x, dev, p, seed, causal, kv_len=None, backward=True):
    q, k, v, do = (t.to(dev) for t in (x.q, x.k, x.v, x.do))
    kl = None if kv_len is None else kv_len.to(dev)
    o, lse = fb.forward_dropout(q, k, v, p, seed, scale=x.scale, causal=causal, kv_len=kl)
    out = [o, lse]
    if backward:
        out += list(fb.backward_dropout(q, k, v, o, lse, do, p, seed, scale=x.scale, causal=causal, kv_len=kl))
    torch.cuda.synchronize()
    return [t.float().cpu().numpy() for t in out]


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("p", [0.0, 0.1, 0.5])
def test_dropout_parity(cuda_device, d, causal, p):
    w = W.Workload("drop", 2, 2, 384, d, causal=causal)
    x = W.make_inputs(w, seed=d + int(10 * p))
    o, lse, dq, dk, dv = run(x, cuda_device, p, SEED, causal)
    O, L = DR.forward(x.q, x.k, x.v, x.scale, p, SEED, causal=causal)
    check_o(o, O, p)
    assert float(np.abs(lse - L).max()) <= TOL_L
    gq, gk, gv = DR.backward(x.q, x.k, x.v, x.do, x.scale, p, SEED, causal=causal)
    e = {"dq": rel(dq, gq), "dk": rel(dk, gk), "dv": rel(dv, gv)}
    assert max(e.values()) <= TOL_G, e


@pytest.mark.gpu
def test_dropout_key_padding_and_seeds(cuda_device):
    w = W.Workload("droppad", 2, 3, 256, 64, kv_len_range=(1, 256))
    x = W.make_inputs(w, seed=4)
    x.kv_len[:] = torch.tensor([200, 3], dtype=torch.int32)
    for seed in (0, 7, 2 ** 63 + 5):
        o, lse, dq, dk, dv = run(x, cuda_device, 0.25, seed, False, kv_len=x.kv_len)
        O, L = DR.forward(x.q, x.k, x.v, x.scale, 0.25, seed, kv_len=x.kv_len)
        check_o(o, O, 0.25)
        gq, gk, gv = DR.backward(x.q, x.k, x.v, x.do, x.scale, 0.25, seed, kv_len=x.kv_len)
        assert max(rel(dq, gq), rel(dk, gk), rel(dv, gv)) <= TOL_G


@pytest.mark.gpu
def test_dropout_zero_rate_matches_plain_kernel(cuda_device):
    w = W.Workload("drop0", 1, 2, 256, 128, causal=True)
    x = W.make_inputs(w, seed=5)
    o, lse = run(x, cuda_device, 0.0, 9, True, backward=False)
    q, k, v = (t.to(cuda_device) for t in (x.q, x.k, x.v))
    o2, lse2 = fb.forward(q, k, v, scale=x.scale, causal=True)
    np.testing.assert_array_equal(o, o2.float().cpu().numpy())
    np.testing.assert_array_equal(lse, lse2.cpu().numpy())


@pytest.mark.gpu
def test_dropout_rejects(cuda_device):
    w = W.Workload("dropbad", 1, 1, 128, 64)
    x = W.make_inputs(w, seed=1)
    with pytest.raises(fb.FAError):
        run(x, cuda_device, 1.0, 1, False, backward=False)
    with pytest.raises(fb.FAError):
        run(x, cuda_device, -0.1, 1, False, backward=False)


@pytest.mark.gpu
def test_dropout_long8k_sampled_heads(cuda_device):
    """The benchmarked shape (B 1, H 32, N 8192, d 128, causal, K x 2,
    p = 0.1): the Philox counters reach query index 8191 and head 31. Whole
    heads (0, 0) and (0, 31) are compared with the oracle (heads are
    independent, so the check is exact for them)."""
    w = W.WORKLOADS["long8k"]
    x = W.make_inputs(w, seed=0)
    p, seed = 0.1, 1234
    o, lse, dq, dk, dv = run(x, cuda_device, p, seed, True)
    heads = [(0, 0), (0, 31)]
    O, L = DR.forward(x.q, x.k, x.v, x.scale, p, seed, causal=True, heads=heads)
    G = DR.backward(x.q, x.k, x.v, x.do, x.scale, p, seed, causal=True, heads=heads)
    for (b, h) in heads:
        check_o(o[b, h], O[b, h], p)
        assert float(np.abs(lse[b, h] - L[b, h]).max()) <= TOL_L
        e = {n: rel(g[b, h], ref[b, h]) for n, g, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), G)}
        assert max(e.values()) <= TOL_G, ((b, h), e)
