"""GPU parity of packed variable-length attention against the fp64 oracle.

Forward and backward go through the C ABI (fa_fwd_varlen / fa_bwd_varlen)
on seeded packed batches whose lengths straddle the 128-row tile edges
(1, 127, 128, 129, ...), include empty sequences and run to a few thousand
tokens; every output row is compared with the per-sequence oracle.
"""

import numpy as np
import pytest
import torch

import io_aware_exact_tiled_gb300 as fa
from io_aware_exact_tiled_gb300 import binding as fb
from io_aware_exact_tiled_gb300 import workloads as W
from oracle import varlen as VL

from parity import TOL_G, TOL_L, TOL_O, rel

LENS = {
    "ragged": [1, 127, 128, 129, 300, 0, 513, 64],
    "single_long": [2000],
    "many_short": [5, 17, 33, 2, 90, 128, 7, 64, 1, 250, 3, 129],
}


def run_fwd(x, dev):
    q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
    cu = x.cu_seqlens.to(dev)
    o, lse = fb.forward_varlen(q, k, v, cu, x.max_seqlen, scale=x.scale, causal=x.causal)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def fwd_errors(x, o, lse):
    O, L = VL.forward_varlen(x.q, x.k, x.v, x.cu_seqlens, x.scale, causal=x.causal)
    return float(np.abs(o - O).max()), float(np.abs(lse - L).max())


@pytest.mark.gpu
@pytest.mark.parametrize("case", sorted(LENS))
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_parity(cuda_device, case, d, causal):
    x = W.make_packed(LENS[case], 3, d, causal=causal, seed=11)
    o, lse = run_fwd(x, cuda_device)
    eo, el = fwd_errors(x, o, lse)
    assert eo <= TOL_O and el <= TOL_L, (eo, el)


@pytest.mark.gpu
def test_forward_bert_packed_full(cuda_device):
    x = W.make_packed_workload(W.PACKED_WORKLOADS["bert_packed"], seed=0)
    o, lse = run_fwd(x, cuda_device)
    eo, el = fwd_errors(x, o, lse)
    assert eo <= TOL_O and el <= TOL_L, (eo, el)


@pytest.mark.gpu
def test_forward_matches_padded_call(cuda_device):
    """One sequence padded to a multiple of 128 with the key-padding mask
    gives the same rows as the packed call (both on the GPU, same kernel
    arithmetic, so the agreement is close to bit level)."""
    lens = [200, 77, 384]
    x = W.make_packed(lens, 2, 64, seed=5)
    o, lse = run_fwd(x, cuda_device)
    for b, n in enumerate(lens):
        s = int(x.cu_seqlens[b])
        Np = -(-n // 128) * 128
        pad = lambda t: torch.nn.functional.pad(t[s:s + n].permute(1, 0, 2), (0, 0, 0, Np - n))[None]
        qp, kp, vp = (pad(t).contiguous().to(cuda_device) for t in (x.q, x.k, x.v))
        kl = torch.tensor([n], dtype=torch.int32, device=cuda_device)
        od, ld = fa.forward(qp, kp, vp, scale=x.scale, kv_len=kl)
        od = od[0, :, :n].permute(1, 0, 2).float().cpu().numpy()
        np.testing.assert_allclose(o[s:s + n], od, atol=1e-2)
        np.testing.assert_allclose(lse[:, s:s + n], ld[0, :, :n].cpu().numpy(), atol=1e-5)


@pytest.mark.gpu
def test_forward_leaves_rows_of_other_buffers_alone(cuda_device):
    """Output rows are written only inside [0, total): a guard region after
    the output and lse buffers keeps its sentinel values."""
    x = W.make_packed([129, 3, 250], 2, 128, causal=True, seed=2)
    total, H, d = x.q.shape
    q, k, v = (t.to(cuda_device) for t in (x.q, x.k, x.v))
    o_big = torch.full((total + 128, H, d), 7.0, dtype=torch.bfloat16, device=cuda_device)
    l_big = torch.full((H, total + 128), 7.0, dtype=torch.float32, device=cuda_device)
    o = o_big[:total]
    fb.forward_varlen(q, k, v, x.cu_seqlens.to(cuda_device), x.max_seqlen, scale=x.scale, causal=True, out=o,
                      lse=torch.empty((H, total), dtype=torch.float32, device=cuda_device))
    torch.cuda.synchronize()
    assert bool((o_big[total:] == 7.0).all())


@pytest.mark.gpu
def test_too_short_max_seqlen_is_reported(cuda_device):
    """A sequence longer than max_seqlen is cut and reported through the
    status word as FA_ERR_INVALID_ARG (no fault, no hang)."""
    x = W.make_packed([300, 40], 1, 64, seed=3)
    q, k, v = (t.to(cuda_device) for t in (x.q, x.k, x.v))
    ws = fb.workspace(256, cuda_device)
    fb.forward_varlen(q, k, v, x.cu_seqlens.to(cuda_device), 200, scale=x.scale, ws=ws)
    assert fb.get_status(ws) == fb.FA_ERR_INVALID_ARG
    fb.forward_varlen(q, k, v, x.cu_seqlens.to(cuda_device), 300, scale=x.scale, ws=ws)
    assert fb.get_status(ws) == fb.FA_OK


@pytest.mark.gpu
def test_rejects_fp32_and_bad_arguments(cuda_device):
    x = W.make_packed([10, 20], 1, 64, seed=4)
    q, k, v = (t.to(cuda_device) for t in (x.q, x.k, x.v))
    cu = x.cu_seqlens.to(cuda_device)
    with pytest.raises(ValueError):
        fb.forward_varlen(q.float(), k.float(), v.float(), cu, 20)
    with pytest.raises(fb.FAError):
        fb.forward_varlen(q, k, v, cu, 0)
    with pytest.raises(fb.FAError):
        fb.forward_varlen(q, k, v, cu, 31)  # max_seqlen > total


def bwd_errors(x, g):
    dq, dk, dv = VL.backward_varlen(x.q, x.k, x.v, x.do, x.cu_seqlens, x.scale, causal=x.causal)
    return {"dq": rel(g[0], dq), "dk": rel(g[1], dk), "dv": rel(g[2], dv)}


def run_bwd(x, dev):
    q, k, v, do = (t.to(dev) for t in (x.q, x.k, x.v, x.do))
    cu = x.cu_seqlens.to(dev)
    o, lse = fb.forward_varlen(q, k, v, cu, x.max_seqlen, scale=x.scale, causal=x.causal)
    g = fb.backward_varlen(q, k, v, o, lse, do, cu, x.max_seqlen, scale=x.scale, causal=x.causal)
    torch.cuda.synchronize()
    return [t.float().cpu().numpy() for t in g]


@pytest.mark.gpu
@pytest.mark.parametrize("case", sorted(LENS))
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_parity(cuda_device, case, d, causal):
    x = W.make_packed(LENS[case], 3, d, causal=causal, seed=12)
    e = bwd_errors(x, run_bwd(x, cuda_device))
    assert max(e.values()) <= TOL_G, e


@pytest.mark.gpu
def test_backward_bert_packed_full(cuda_device):
    x = W.make_packed_workload(W.PACKED_WORKLOADS["bert_packed"], seed=0)
    e = bwd_errors(x, run_bwd(x, cuda_device))
    assert max(e.values()) <= TOL_G, e


@pytest.mark.gpu
def test_backward_status_clear(cuda_device):
    x = W.make_packed([130, 0, 257], 2, 64, causal=True, seed=6)
    q, k, v, do = (t.to(cuda_device) for t in (x.q, x.k, x.v, x.do))
    cu = x.cu_seqlens.to(cuda_device)
    total, H, d = q.shape
    o, lse = fb.forward_varlen(q, k, v, cu, x.max_seqlen, causal=True)
    ws = fb.workspace(fb.load().fa_bwd_varlen_workspace_size(3, H, total, d), cuda_device)
    fb.backward_varlen(q, k, v, o, lse, do, cu, x.max_seqlen, causal=True, ws=ws)
    assert fb.get_status(ws) == fb.FA_OK


@pytest.mark.gpu
def test_mix8k_packed_sampled_sequences(cuda_device):
    """The benchmarked packed batch (16 causal sequences, lengths
    U{512..8192}, H 32, d 128), run whole on the GPU; the two longest
    sequences (several thousand tokens each) are compared with the oracle on
    heads 0 and 31 (sequences and heads are independent, so the oracle runs
    on each as a packed batch of one)."""
    w = W.PACKED_WORKLOADS["mix8k_packed"]
    x = W.make_packed_workload(w, seed=0)
    dev = cuda_device
    q, k, v, do = (t.to(dev) for t in (x.q, x.k, x.v, x.do))
    cu = x.cu_seqlens.to(dev)
    o, lse = fb.forward_varlen(q, k, v, cu, x.max_seqlen, scale=x.scale, causal=True)
    dq, dk, dv = fb.backward_varlen(q, k, v, o, lse, do, cu, x.max_seqlen, scale=x.scale, causal=True)
    torch.cuda.synchronize()
    o, lse, dq, dk, dv = (t.float().cpu().numpy() for t in (o, lse, dq, dk, dv))
    cuh = x.cu_seqlens.tolist()
    order = sorted(range(len(x.lens)), key=lambda b: -x.lens[b])[:2]
    assert min(x.lens[b] for b in order) >= 4096
    hs = [0, 31]
    for b in order:
        s, e = cuh[b], cuh[b + 1]
        one = torch.tensor([0, e - s], dtype=torch.int32)
        sub = lambda t: t[s:e][:, hs]
        O, L = VL.forward_varlen(sub(x.q), sub(x.k), sub(x.v), one, x.scale, causal=True)
        G = VL.backward_varlen(sub(x.q), sub(x.k), sub(x.v), sub(x.do), one, x.scale, causal=True)
        assert float(np.abs(o[s:e][:, hs] - O).max()) <= TOL_O
        assert float(np.abs(lse[hs][:, s:e] - L).max()) <= TOL_L
        e_g = {n: rel(g[s:e][:, hs], ref) for n, g, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), G)}
        assert max(e_g.values()) <= TOL_G, (b, x.lens[b], e_g)
