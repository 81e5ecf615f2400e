"""Device-side give-up: every wait in the kernels is bounded. A debug build
(FA_DEBUG_DROP_ARRIVE, 0.2 s limit) withholds one "P ready" arrival so that
the MMA thread's wait runs out; the kernel must then stop, release its TMEM
and report FA_ERR_TIMEOUT through the status word, and the CUDA context must
stay usable. Nothing faults, traps or hangs."""

import ctypes
import math

import numpy as np
import pytest
import torch

import io_aware_exact_tiled_gb300 as fa
from io_aware_exact_tiled_gb300 import binding as fb
from io_aware_exact_tiled_gb300 import build as fbuild

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    path = fbuild.build_debug()
    lib = ctypes.CDLL(path)
    vp, sz, i, f = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, i, vp, sz, vp]
    lib.fa_fwd.restype = i
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, i, vp, sz, vp]
    lib.fa_bwd.restype = i
    lib.fa_get_status.argtypes = [vp, vp]
    lib.fa_get_status.restype = i
    lib.fa_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.fa_bwd_workspace_size.restype = sz
    lib.fa_fwd_dropout.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, f, ctypes.c_ulonglong, vp, sz, vp]
    lib.fa_fwd_dropout.restype = i
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, i, vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_bwd_noalloc_get_status.argtypes = [vp]
    lib.fa_bwd_noalloc_get_status.restype = i
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, vp, sz, vp]
    lib.fa_fwd_fp8.restype = i
    lib.fa_fwd_fp8_workspace_size.argtypes = [i, i, i, i]
    lib.fa_fwd_fp8_workspace_size.restype = sz
    return lib


def ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_bounded_waits_report_timeout(dbg, cuda_device):
    B, H, N, d = 1, 1, 256, 64
    g = torch.Generator(device="cpu").manual_seed(0)
    q, k, v, do = (torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).to(cuda_device) for _ in range(4))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=cuda_device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    scale = 1.0 / math.sqrt(d)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ws = torch.empty(dbg.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=cuda_device)

    rc = dbg.fa_fwd(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), B, H, N, d, scale, 1, None, None, fb.FA_BF16,
                    ptr(ws), ws.numel(), s)
    assert rc == fb.FA_OK
    assert dbg.fa_get_status(ptr(ws), s) == fb.FA_ERR_TIMEOUT
    assert dbg.fa_get_status(ptr(ws), s) == fb.FA_OK  # reading clears the word

    # the pair-tile forward kernel (it serves dropout, packed batches and fp32)
    rc = dbg.fa_fwd_dropout(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), B, H, N, d, scale, 1, None, 0.1, 1234,
                            ptr(ws), ws.numel(), s)
    assert rc == fb.FA_OK
    assert dbg.fa_get_status(ptr(ws), s) == fb.FA_ERR_TIMEOUT

    # a tile-masked forward
    bm = torch.ones(N // 128, N // 128, dtype=torch.uint8, device=cuda_device)
    rc = dbg.fa_fwd(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), B, H, N, d, scale, 0, ptr(bm), None, fb.FA_BF16,
                    ptr(ws), ws.numel(), s)
    assert rc == fb.FA_OK
    assert dbg.fa_get_status(ptr(ws), s) == fb.FA_ERR_TIMEOUT

    rc = dbg.fa_bwd(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), ptr(do), ptr(dq), ptr(dk), ptr(dv), B, H, N, d,
                    scale, 1, None, None, fb.FA_BF16, ptr(ws), ws.numel(), s)
    assert rc == fb.FA_OK
    assert dbg.fa_get_status(ptr(ws), s) == fb.FA_ERR_TIMEOUT

    # the workspace-free backward reports its give-up through its own reader
    rc = dbg.fa_bwd_noalloc(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), ptr(do), ptr(dq), ptr(dk), ptr(dv), B, H, N,
                            d, scale, 1, None, None, fb.FA_BF16, s)
    assert rc == fb.FA_OK
    assert dbg.fa_bwd_noalloc_get_status(s) == fb.FA_ERR_TIMEOUT
    assert dbg.fa_bwd_noalloc_get_status(s) == fb.FA_OK  # reading clears the word

    # the context is still usable: the regular library computes correct results
    o2, lse2 = fa.forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    x = q.double().cpu()[0, 0] @ k.double().cpu()[0, 0].T * scale
    x = x.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
    ref = torch.softmax(x, -1) @ v.double().cpu()[0, 0]
    assert (o2.double().cpu()[0, 0] - ref).abs().max().item() < 1e-2
    assert np.isfinite(lse2.cpu().numpy()).all()


def test_fp8_forward_reports_timeout(dbg, cuda_device):
    """The FP8 path (quantisation kernel, then the FP8 attention kernel,
    whose MMA thread's wait the debug build makes run out): the call reports
    FA_ERR_TIMEOUT and the regular library's FP8 call works afterwards."""
    B, H, N, d = 1, 3, 512, 128
    g = torch.Generator(device="cpu").manual_seed(1)
    q, k, v = (torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).to(cuda_device) for _ in range(3))
    signs = (torch.randint(0, 2, (d,), generator=g) * 2 - 1).float().to(cuda_device)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=cuda_device)
    ws = torch.empty(dbg.fa_fwd_fp8_workspace_size(B, H, N, d), dtype=torch.uint8, device=cuda_device)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = dbg.fa_fwd_fp8(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), B, H, N, d, 1.0 / math.sqrt(d), 1, None,
                        ptr(signs), ptr(ws), ws.numel(), s)
    assert rc == fb.FA_OK
    assert dbg.fa_get_status(ptr(ws), s) == fb.FA_ERR_TIMEOUT
    assert dbg.fa_get_status(ptr(ws), s) == fb.FA_OK
    o2, lse2 = fb.forward_fp8(q, k, v, signs, scale=1.0 / math.sqrt(d), causal=True)
    torch.cuda.synchronize()
    assert torch.isfinite(o2.float()).all() and torch.isfinite(lse2).all()
