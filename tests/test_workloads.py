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


def test_packed_recipe():
    w = W.PACKED_WORKLOADS["bert_packed"]
    x = W.make_packed_workload(w, seed=3)
    g = torch.Generator().manual_seed(3)
    lens = torch.randint(256, 513, (w.B,), generator=g).tolist()
    assert x.lens == lens and all(256 <= n <= 512 for n in lens)
    total = sum(lens)
    assert x.q.shape == (total, w.H, w.d) and x.q.dtype == torch.bfloat16
    assert x.cu_seqlens.dtype == torch.int32 and x.cu_seqlens.shape == (w.B + 1,)
    assert int(x.cu_seqlens[0]) == 0 and int(x.cu_seqlens[-1]) == total
    assert torch.equal(x.cu_seqlens[1:] - x.cu_seqlens[:-1], torch.tensor(lens, dtype=torch.int32))
    assert x.max_seqlen == max(lens) and x.scale == 1.0 / math.sqrt(w.d) and not x.causal
    # Q, K, V, dO drawn in that order from one generator seeded with the same seed
    g = torch.Generator().manual_seed(3)
    q = torch.randn(total, w.H, w.d, generator=g)
    k = torch.randn(total, w.H, w.d, generator=g)
    v = torch.randn(total, w.H, w.d, generator=g)
    assert torch.equal(x.q, q.to(torch.bfloat16)) and torch.equal(x.k, k.to(torch.bfloat16))
    assert torch.equal(x.v, v.to(torch.bfloat16))
    y = W.make_packed_workload(w, seed=3)
    assert torch.equal(x.do, y.do) and y.lens == x.lens
    assert W.make_packed_workload(w, seed=4).lens != x.lens
    assert W.PACKED_WORKLOADS["mix8k_packed"].causal


def test_packed_empty_and_zero_length_sequences():
    x = W.make_packed([0, 5, 0, 3], H=2, d=64)
    assert x.cu_seqlens.tolist() == [0, 0, 5, 5, 8] and x.q.shape == (8, 2, 64)
    assert x.max_seqlen == 5
    e = W.make_packed([], H=2, d=64)
    assert e.q.shape == (0, 2, 64) and e.cu_seqlens.tolist() == [0] and e.max_seqlen == 0


def test_decode_recipe():
    x = W.make_decode(B=3, H=2, Nq=1, Nk=256, d=128, len_range=(100, 256), seed=5)
    assert x.q.shape == (3, 2, 1, 128) and x.k.shape == (3, 2, 256, 128) == x.v.shape
    assert x.q.dtype == x.k.dtype == torch.bfloat16
    expect = torch.randint(100, 257, (3,), generator=torch.Generator().manual_seed(6)).to(torch.int32)
    assert torch.equal(x.cache_len, expect) and x.cache_len.dtype == torch.int32
    g = torch.Generator().manual_seed(5)
    q = torch.randn(3, 2, 1, 128, generator=g)
    k = torch.randn(3, 2, 256, 128, generator=g)
    assert torch.equal(x.q, q.to(torch.bfloat16)) and torch.equal(x.k, k.to(torch.bfloat16))
    w = W.DECODE_WORKLOADS["decode16k"]
    assert (w.Nq, w.Nk, w.d) == (1, 16384, 128) and w.len_range[1] <= w.Nk
