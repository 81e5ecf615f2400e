"""GPU parity of split-key decoding (fa_decode) against the fp64 oracle.

Cases cover one and several query rows, cache lengths that are not
multiples of the 64-key tile, empty caches, explicit and automatic split
counts (one split per head up to one per 64 keys), both head sizes, and the
full decode16k shape on sampled heads.
"""

import numpy as np
import pytest
import torch

from io_aware_exact_tiled_gb300 import binding as fb
from io_aware_exact_tiled_gb300 import workloads as W
from oracle import decode as DEC

from parity import TOL_L, TOL_O


def run(x, dev, num_splits=0, cache_len=True):
    q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
    cl = x.cache_len.to(dev) if cache_len else None
    o, lse = fb.decode(q, k, v, cache_len=cl, scale=x.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def errors(x, o, lse, cache_len=True):
    O, L = DEC.decode_forward(x.q, x.k, x.v, x.scale, x.cache_len if cache_len else None)
    both = np.isneginf(L) & np.isneginf(lse)
    with np.errstate(invalid="ignore"):
        el = float(np.where(both, 0.0, np.abs(lse - L)).max())
    return float(np.abs(o - O).max()), el


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq", [1, 2, 3, 8])
@pytest.mark.parametrize("splits", [0, 1, 5, 1000])
def test_decode_parity(cuda_device, d, Nq, splits):
    x = W.make_decode(3, 2, Nq, 1000, d, (1, 1000), seed=Nq + d)
    x.cache_len[:] = torch.tensor([1000, 63, 129], dtype=torch.int32)
    eo, el = errors(x, *run(x, cuda_device, splits))
    assert eo <= TOL_O and el <= TOL_L, (eo, el)


@pytest.mark.gpu
def test_decode_full_cache_and_empty_cache(cuda_device):
    x = W.make_decode(2, 3, 1, 300, 128, (0, 0), seed=9)
    eo, el = errors(x, *run(x, cuda_device, cache_len=False), cache_len=False)
    assert eo <= TOL_O and el <= TOL_L, (eo, el)
    o, lse = run(x, cuda_device)  # cache_len = 0 everywhere
    assert np.all(o == 0) and np.all(np.isneginf(lse))


@pytest.mark.gpu
def test_decode16k_sampled(cuda_device):
    w = W.DECODE_WORKLOADS["decode16k"]
    x = W.make_decode_workload(w, seed=0)
    o, lse = run(x, cuda_device)
    # the oracle on a few batch elements (heads are independent)
    for b in (0, 7, 15):
        sub = W.DecodeInputs(x.q[b:b + 1], x.k[b:b + 1], x.v[b:b + 1], x.cache_len[b:b + 1], x.scale)
        O, L = DEC.decode_forward(sub.q, sub.k, sub.v, sub.scale, sub.cache_len)
        assert float(np.abs(o[b:b + 1] - O).max()) <= TOL_O
        assert float(np.abs(lse[b:b + 1] - L).max()) <= TOL_L


@pytest.mark.gpu
def test_decode_rejects(cuda_device):
    x = W.make_decode(1, 1, 9, 64, 64, (64, 64), seed=1)
    with pytest.raises(fb.FAError):
        run(x, cuda_device)  # Nq > 8
    with pytest.raises(ValueError):
        fb.decode(x.q.float().to(cuda_device), x.k.to(cuda_device), x.v.to(cuda_device))
