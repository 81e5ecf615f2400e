"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (it uses a fixed scratch array inside the library instead of a
caller-supplied workspace). Its results must match fa_bwd's, call after call,
since every call reuses the same scratch. This file is collected last so that
a run stopping at its first failure has already run every other test."""

import ctypes

import numpy as np
import pytest
import torch

import io_aware_exact_tiled_gb300 as fa
from io_aware_exact_tiled_gb300 import binding as fb
from io_aware_exact_tiled_gb300 import build as fbuild
from io_aware_exact_tiled_gb300 import workloads as W

TOL_G = 2e-2  # relative Frobenius error bound used for dQ, dK, dV everywhere


def rel(a, b):
    a, b = a.float().cpu().numpy(), b.float().cpu().numpy()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return fb.load()


def test_noalloc_symbol_declared(lib):
    assert "fa_bwd_noalloc" in fb.declared_functions()
    assert hasattr(lib, "fa_bwd_noalloc")


def test_noalloc_rejects_oversized_request(lib):
    # 1 x 32 x 8192 x 128 needs ~129 MiB of scratch > 32 MiB: refused on the host
    lib.fa_bwd_noalloc.restype = ctypes.c_int
    vp = ctypes.c_void_p
    big = 1 << 20
    rc = lib.fa_bwd_noalloc(vp(big), vp(big), vp(big), vp(big), vp(big), vp(big), vp(big), vp(big), vp(big),
                            1, 32, 8192, 128, ctypes.c_float(0.088), 1, None, None, fb.FA_BF16, None)
    assert rc == fb.FA_ERR_UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.parametrize("w", [
    W.Workload("nalloc-causal", 2, 3, 512, 64, causal=True),
    W.Workload("nalloc-kvlen", 2, 2, 384, 128, kv_len_range=(100, 384)),
    W.Workload("nalloc-sparse", 1, 2, 768, 128, block_density=0.4),
], ids=lambda w: w.name)
def test_noalloc_matches_fa_bwd_two_calls(lib, cuda_device, w):
    x = W.make_inputs(w, seed=11)
    q, k, v, do = (t.to(cuda_device) for t in (x.q, x.k, x.v, x.do))
    bm = None if x.blockmask is None else x.blockmask.to(cuda_device)
    kl = None if x.kv_len is None else x.kv_len.to(cuda_device)
    kw = dict(scale=x.scale, causal=x.causal, blockmask=bm, kv_len=kl)
    o, lse = fa.forward(q, k, v, **kw)
    ref = fa.backward(q, k, v, o, lse, do, **kw)
    for call in range(2):
        got = fb.backward_noalloc(q, k, v, o, lse, do, **kw)
        torch.cuda.synchronize()
        assert fb.noalloc_status() == fb.FA_OK
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            e = rel(a, b)
            assert e <= TOL_G, (call, name, e)
            assert torch.isfinite(a.float()).all()
