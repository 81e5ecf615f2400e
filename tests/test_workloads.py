"""Seeded input recipe (no GPU)."""

import math

import torch

from io_aware_exact_tiled_gb300 import workloads as W


def test_shapes_and_dtypes():
    for name, w in W.WORKLOADS.items():
        assert w.N % 128 == 0 and w.d in (64, 128)
        assert w.scale == 1.0 / math.sqrt(w.d)
    small = W.WORKLOADS["bert"].with_(B=2, H=2)
    x = W.make_inputs(small)
    assert x.q.shape == (2, 2, 512, 64) and x.q.dtype == torch.bfloat16
    assert x.kv_len.dtype == torch.int32 and x.kv_len.shape == (2,)
    t = W.make_inputs(W.WORKLOADS["tiny"])
    assert t.q.dtype == torch.float32 and t.kv_len is None and t.blockmask is None


def test_seeded_and_reproducible():
    w = W.WORKLOADS["gpt2"].with_(B=1, H=2, N=256)
    a, b = W.make_inputs(w, seed=0), W.make_inputs(w, seed=0)
    c = W.make_inputs(w, seed=1)
    assert torch.equal(a.q, b.q) and torch.equal(a.do, b.do)
    assert not torch.equal(a.q, c.q)
    # recipe: Q, K, V, dO drawn in that order from one generator, then rounded
    g = torch.Generator().manual_seed(0)
    q = torch.randn(w.B, w.H, w.N, w.d, generator=g)
    k = torch.randn(w.B, w.H, w.N, w.d, generator=g)
    assert torch.equal(a.q, q.to(torch.bfloat16)) and torch.equal(a.k, k.to(torch.bfloat16))


def test_key_scale_exact():
    w = W.WORKLOADS["long4k"].with_(H=1, N=256)
    x = W.make_inputs(w)
    g = torch.Generator().manual_seed(0)
    torch.randn(1, 1, 256, 128, generator=g)
    k = torch.randn(1, 1, 256, 128, generator=g)
    assert torch.equal(x.k, (2.0 * k).to(torch.bfloat16))
    assert torch.equal(x.k.float() / 2, k.to(torch.bfloat16).float())


def test_kv_len_range_inclusive():
    g = torch.Generator().manual_seed(0)
    lens = torch.randint(256, 513, (20000,), generator=g)
    assert lens.min() == 256 and lens.max() == 512


def test_blockmask_recipe():
    g = torch.Generator().manual_seed(0)
    T = 128
    bm = W.make_blockmask(T, 0.125, g)
    assert bm.dtype == torch.uint8 and bm.shape == (T, T)
    assert bm.diagonal().all()
    off = int(bm.sum()) - T
    assert off == math.floor(0.125 * (T * T - T)) == 2032
    assert not torch.equal(bm, bm.t())
