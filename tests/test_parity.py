"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs. Small shapes span several tiles and the edge cases; the
full workload shapes are checked on whole sampled heads."""

import numpy as np
import pytest
import torch

import io_aware_exact_tiled_gb300 as fa
from io_aware_exact_tiled_gb300 import workloads as W

import oracle
from parity import TOL_G, TOL_L, TOL_O, check, errors, run_gpu

pytestmark = pytest.mark.gpu


def small(name, **kw):
    return W.WORKLOADS[name].with_(**kw)


SWEEP = []
for d in (64, 128):
    for N in (128, 384, 1024):
        SWEEP.append(W.Workload(f"dense-{N}-{d}", 2, 2, N, d))
        SWEEP.append(W.Workload(f"causal-{N}-{d}", 2, 2, N, d, causal=True))
        SWEEP.append(W.Workload(f"kvlen-{N}-{d}", 3, 2, N, d, kv_len_range=(1, N)))
        SWEEP.append(W.Workload(f"sparse-{N}-{d}", 1, 2, N, d, block_density=0.3))
for d in (64, 128):
    SWEEP.append(W.Workload(f"causal-kvlen-sparse-768-{d}", 2, 2, 768, d, causal=True, kv_len_range=(200, 700),
                            block_density=0.5))
SWEEP.append(W.Workload("wide-scores-512-128", 1, 2, 512, 128, causal=True, k_scale=4.0))
# tile masks: ragged key padding inside visible tiles, rows that see most
# tiles (the K and V rings wrap several times), and a rescale of O (K x 4
# widens the scores)
for d in (64, 128):
    SWEEP.append(W.Workload(f"sparse-kvlen-640-{d}", 3, 2, 640, d, kv_len_range=(100, 600), block_density=0.5))
    SWEEP.append(W.Workload(f"sparse-dense-1024-{d}", 1, 2, 1024, d, block_density=0.9))
SWEEP.append(W.Workload("wide-scores-sparse-1024-128", 1, 2, 1024, 128, k_scale=4.0, block_density=0.6))


@pytest.mark.parametrize("w", SWEEP, ids=lambda w: w.name)
def test_sweep(cuda_device, w):
    x = W.make_inputs(w, seed=3)
    g = run_gpu(x, cuda_device)
    check(errors(x, g))


def test_tiny_fp32_forward(cuda_device):
    w = W.WORKLOADS["tiny"]
    x = W.make_inputs(w, seed=0)
    g = run_gpu(x, cuda_device, backward=False)
    e = errors(x, g, backward=False)
    check(e)
    assert e["lse"] <= 1e-3


def test_bert_full(cuda_device):
    x = W.make_inputs(W.WORKLOADS["bert"], seed=0)
    check(errors(x, run_gpu(x, cuda_device)))


def test_gpt2_full(cuda_device):
    x = W.make_inputs(W.WORKLOADS["gpt2"], seed=0)
    check(errors(x, run_gpu(x, cuda_device)))


@pytest.mark.parametrize("name", ["long4k", "long8k"])
def test_long_context_sampled_heads(cuda_device, name):
    w = W.WORKLOADS[name]
    x = W.make_inputs(w, seed=0)
    g = run_gpu(x, cuda_device)
    heads = [(0, 0), (0, 17), (0, w.H - 1)]
    check(errors(x, g, heads=heads))


def test_block_sparse_sampled_heads(cuda_device):
    w = W.WORKLOADS["sparse16k"]
    x = W.make_inputs(w, seed=0)
    g = run_gpu(x, cuda_device)
    check(errors(x, g, heads=[(0, 0), (w.B - 1, w.H - 1)]))


def test_fully_masked_rows_and_empty_key_blocks(cuda_device):
    # kv_len = 0 for one batch element: every row sees no key (O = 0,
    # L = -inf, zero gradients); a tile mask with an empty query row and an
    # empty key column.
    w = W.Workload("edge", 2, 2, 384, 64)
    x = W.make_inputs(w, seed=5)
    x.kv_len = torch.tensor([0, 300], dtype=torch.int32)
    bm = torch.ones(3, 3, dtype=torch.uint8)
    bm[1, :] = 0
    bm[:, 2] = 0
    x.blockmask = bm
    g = run_gpu(x, cuda_device)
    check(errors(x, g))
    assert (g["o"][0] == 0).all() and np.isneginf(g["lse"][0]).all()
    assert (g["dk"][0] == 0).all() and (g["dv"][0] == 0).all() and (g["dq"][0] == 0).all()
    assert (g["o"][1, :, 128:256] == 0).all()
    assert (g["dk"][:, :, 256:] == 0).all() and (g["dv"][:, :, 256:] == 0).all()


def test_forward_deterministic(cuda_device):
    w = W.Workload("det", 1, 4, 1024, 128, causal=True)
    x = W.make_inputs(w, seed=1)
    a = run_gpu(x, cuda_device, backward=False)
    b = run_gpu(x, cuda_device, backward=False)
    assert np.array_equal(a["o"], b["o"]) and np.array_equal(a["lse"], b["lse"])


def test_status_word_clear_after_calls(cuda_device):
    w = W.Workload("st", 1, 2, 256, 128, causal=True)
    x = W.make_inputs(w, seed=2)
    q, k, v, do = (t.to(cuda_device) for t in (x.q, x.k, x.v, x.do))
    ws = fa.workspace(fa.bwd_workspace_size(1, 2, 256, 128), cuda_device)
    o, lse = fa.forward(q, k, v, causal=True, ws=ws)
    assert fa.get_status(ws) == 0
    fa.backward(q, k, v, o, lse, do, causal=True, ws=ws)
    assert fa.get_status(ws) == 0
    assert fa.last_launch_count() == 3


def test_tile_mask_longer_than_the_forward_bitmaps(cuda_device):
    """4,097 key tiles, one more than the tile-masked forward keeps as
    shared-memory bitmaps: it then reads the tile mask in global memory tile
    by tile. Sampled query tiles (first, middle, last) against the oracle."""
    T = 4097
    N = T * 128
    w = W.Workload("sparse-long", 1, 1, N, 64, backward=False)
    x = W.make_inputs(w, seed=7)
    g = torch.Generator().manual_seed(8)
    bm = (torch.rand(T, T, generator=g) < 0.002).to(torch.uint8)
    bm.fill_diagonal_(1)
    x.blockmask = bm
    out = run_gpu(x, cuda_device, backward=False)
    for r0 in (0, 2048 * 128, N - 128):
        O, L = oracle.forward(x.q, x.k, x.v, x.scale, blockmask=bm, rows=(r0, r0 + 128))
        assert np.abs(out["o"][0, 0, r0:r0 + 128] - O[0, 0, r0:r0 + 128]).max() <= TOL_O
        assert np.abs(out["lse"][0, 0, r0:r0 + 128] - L[0, 0, r0:r0 + 128]).max() <= TOL_L


def test_tile_mask_longer_than_the_backward_bitmaps(cuda_device):
    """2,049 query tiles, one more than the tile-masked backward keeps as a
    shared-memory bitmap. Sampled query tiles r whose key-tile column holds
    only the diagonal: dQ of their rows and dK, dV of key tile r then depend
    on those 128 rows alone, which the oracle computes one by one."""
    T = 2049
    N = T * 128
    w = W.Workload("sparse-long-bwd", 1, 1, N, 64)
    x = W.make_inputs(w, seed=9)
    g = torch.Generator().manual_seed(10)
    bm = (torch.rand(T, T, generator=g) < 0.002).to(torch.uint8)
    sampled = (0, 1024, T - 1)
    for r in sampled:
        bm[:, r] = 0
    bm.fill_diagonal_(1)
    x.blockmask = bm
    out = run_gpu(x, cuda_device)
    for r in sampled:
        rows = (r * 128, r * 128 + 128)
        sl = slice(*rows)
        O, L = oracle.forward(x.q, x.k, x.v, x.scale, blockmask=bm, rows=rows)
        assert np.abs(out["o"][0, 0, sl] - O[0, 0, sl]).max() <= TOL_O
        dq, dk, dv = oracle.backward(x.q, x.k, x.v, x.do, x.scale, blockmask=bm, rows=rows)
        for name, ref in (("dq", dq), ("dk", dk), ("dv", dv)):
            a, b = out[name][0, 0, sl], ref[0, 0, sl]
            assert np.linalg.norm(a - b) / np.linalg.norm(b) <= TOL_G, name


def test_causal_head_groups_with_a_partial_last_group(cuda_device):
    """Causal calls run head groups on a 1D grid: at N = 8192, d = 128 the
    forward takes 16 heads per group and the backward 8, so 36 heads end on
    a partial group in both. Whole heads from the first, a middle and the
    last (partial) group against the oracle."""
    w = W.Workload("groups", 1, 36, 8192, 128, causal=True)
    x = W.make_inputs(w, seed=11, device="cuda")
    x = W.Inputs(*(t.cpu() if torch.is_tensor(t) else t for t in (x.q, x.k, x.v, x.do)), x.kv_len, x.blockmask,
                 x.scale, x.causal)
    g = run_gpu(x, cuda_device)
    check(errors(x, g, heads=[(0, 0), (0, 20), (0, 35)]))


def test_causal_tile_mask_long_rows(cuda_device):
    """A causal tile mask over 1,025 key tiles: long bitmap rows cut at the
    diagonal, and causal calls run their query tiles longest first in head
    groups. Sampled query tiles against the oracle."""
    T = 1025
    N = T * 128
    w = W.Workload("causal-sparse-long", 1, 1, N, 128, causal=True, backward=False)
    x = W.make_inputs(w, seed=12)
    g = torch.Generator().manual_seed(13)
    bm = (torch.rand(T, T, generator=g) < 0.01).to(torch.uint8)
    bm.fill_diagonal_(1)
    x.blockmask = bm
    out = run_gpu(x, cuda_device, backward=False)
    for r0 in (0, 512 * 128, N - 128):
        O, L = oracle.forward(x.q, x.k, x.v, x.scale, causal=True, blockmask=bm, rows=(r0, r0 + 128))
        assert np.abs(out["o"][0, 0, r0:r0 + 128] - O[0, 0, r0:r0 + 128]).max() <= TOL_O
        assert np.abs(out["lse"][0, 0, r0:r0 + 128] - L[0, 0, r0:r0 + 128]).max() <= TOL_L
