"""Run-to-run determinism of every entry point on inputs large enough that
every kernel refills its shared-memory buffers many times: repeated calls on
the same inputs give bitwise-identical results (dQ excepted: its fp32
reduce-adds from different key blocks may arrive in another order, so it is
compared at a relative 1e-3). A buffer refilled by a bulk copy before every
thread's reads of it were performed would show here as a few changed rows."""

import pytest
import torch

import io_aware_exact_tiled_gb300 as fa
from io_aware_exact_tiled_gb300 import binding as fb
from io_aware_exact_tiled_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CALLS = 6


def _rel(a, b):
    return ((a.double() - b.double()).norm() / b.double().norm()).item()


def _repeat(fn, flush):
    """Results of CALLS calls, an L2-flush write before each."""
    out = []
    for i in range(CALLS):
        flush.fill_(i)
        r = fn()
        torch.cuda.synchronize()
        out.append(tuple(t.clone() for t in r))
    return out


@pytest.fixture(scope="module")
def flush(cuda_device):
    return torch.empty(256 << 20, dtype=torch.uint8, device=cuda_device)


@pytest.mark.parametrize("mask", ["causal", "tile-mask", "padding"])
def test_forward_backward_repeat(cuda_device, flush, mask):
    w = W.Workload("det", 2, 8, 4096, 128, causal=mask == "causal",
                   block_density=0.3 if mask == "tile-mask" else None,
                   kv_len_range=(1000, 4096) if mask == "padding" else None)
    x = W.make_inputs(w, seed=9, device="cuda")
    bm = None if x.blockmask is None else x.blockmask.to(cuda_device)
    kl = None if x.kv_len is None else x.kv_len.to(cuda_device)
    kw = dict(causal=x.causal, blockmask=bm, kv_len=kl)
    o, lse = fa.forward(x.q, x.k, x.v, **kw)
    res = _repeat(lambda: fa.forward(x.q, x.k, x.v, **kw) + fa.backward(x.q, x.k, x.v, o, lse, x.do, **kw), flush)
    o0, l0, dq0, dk0, dv0 = res[0]
    for o1, l1, dq1, dk1, dv1 in res[1:]:
        assert torch.equal(o1, o0) and torch.equal(l1, l0)
        assert torch.equal(dk1, dk0) and torch.equal(dv1, dv0)
        assert _rel(dq1, dq0) < 1e-3


def test_varlen_repeat(cuda_device, flush):
    pw = W.PackedWorkload("detpk", 6, 8, 128, (500, 3000), causal=True)
    x = W.make_packed_workload(pw, seed=4, device="cuda")
    cu = x.cu_seqlens.to(cuda_device)
    mx = max(x.lens)
    o, lse = fb.forward_varlen(x.q, x.k, x.v, cu, mx, scale=x.scale, causal=True)
    res = _repeat(lambda: fb.forward_varlen(x.q, x.k, x.v, cu, mx, scale=x.scale, causal=True)
                  + fb.backward_varlen(x.q, x.k, x.v, o, lse, x.do, cu, mx, scale=x.scale, causal=True), flush)
    for r in res[1:]:
        assert torch.equal(r[0], res[0][0]) and torch.equal(r[1], res[0][1])
        assert torch.equal(r[3], res[0][3]) and torch.equal(r[4], res[0][4])
        assert _rel(r[2], res[0][2]) < 1e-3


def test_dropout_repeat(cuda_device, flush):
    w = W.Workload("detdrop", 1, 8, 4096, 128, causal=True)
    x = W.make_inputs(w, seed=6, device="cuda")
    o, lse = fb.forward_dropout(x.q, x.k, x.v, 0.1, 77, scale=x.scale, causal=True)
    res = _repeat(lambda: fb.forward_dropout(x.q, x.k, x.v, 0.1, 77, scale=x.scale, causal=True)
                  + fb.backward_dropout(x.q, x.k, x.v, o, lse, x.do, 0.1, 77, scale=x.scale, causal=True), flush)
    for r in res[1:]:
        assert torch.equal(r[0], res[0][0]) and torch.equal(r[1], res[0][1])
        assert torch.equal(r[3], res[0][3]) and torch.equal(r[4], res[0][4])
        assert _rel(r[2], res[0][2]) < 1e-3


def test_decode_repeat(cuda_device, flush):
    dw = W.DecodeWorkload("detdec", 8, 16, 4, 8192, 128, (3000, 8192))
    x = W.make_decode_workload(dw, seed=2, device="cuda")
    cl = x.cache_len.to(cuda_device)
    res = _repeat(lambda: fb.decode(x.q, x.k, x.v, cache_len=cl, scale=x.scale), flush)
    for r in res[1:]:
        assert torch.equal(r[0], res[0][0]) and torch.equal(r[1], res[0][1])
