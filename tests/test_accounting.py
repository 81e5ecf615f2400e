"""FLOP / byte accounting used by the benchmark (no GPU)."""

import json
import os

import numpy as np

from io_aware_exact_tiled_gb300 import accounting as acc
from io_aware_exact_tiled_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_4k_token_traffic_example():
    g = json.load(open(os.path.join(GOLDEN, "traffic_4k.json")))
    N, d, e, H = g["N"], g["d"], g["elem_bytes"], g["heads"]
    x = g["expect"]
    assert acc.tensor_bytes(1, 1, N, d, e) == x["qkv_tensor_bytes_one_head"]
    assert acc.standard_square_bytes(N, e) == x["square_matrix_bytes"]
    assert acc.standard_intermediate_traffic(N, e) == x["intermediate_traffic_one_head"]
    assert acc.standard_intermediate_traffic(N, e, H) == x["intermediate_traffic_all_heads"]


def test_flop_conventions():
    f, b = acc.flops(1, 1, 1024, 64)
    assert f == 4 * 64 * 1024 ** 2 and b == 10 * 64 * 1024 ** 2
    fc, bc = acc.flops(8, 12, 1024, 64, causal=True)
    assert fc == 4 * 64 * 1024 ** 2 / 2 * 96
    fk, _ = acc.flops(2, 1, 512, 64, kv_len=[256, 512])
    assert fk == 4 * 64 * 512 * (256 + 512)
    bm = np.eye(4, dtype=np.uint8)
    bm[0, 3] = 1
    fb, _ = acc.flops(1, 2, 512, 128, blockmask=bm)
    assert fb == 4 * 128 * 5 * 128 * 128 * 2


def test_long_context_flops_in_gflop():
    # causal N = 4096 and 8192, d = 128, 32 heads
    f4, b4 = acc.flops(1, 32, 4096, 128, causal=True)
    assert abs(f4 / 1e9 - 137.4) < 0.1 and abs(b4 / 1e9 - 343.6) < 0.1
    f8, b8 = acc.flops(1, 32, 8192, 128, causal=True)
    assert abs(f8 / 1e9 - 549.8) < 0.1 and abs(b8 / 1e9 - 1374.4) < 0.1


def test_block_sparse_workload_flops():
    w = W.WORKLOADS["sparse16k"]
    import torch
    bm = W.make_blockmask(128, 0.125, torch.Generator().manual_seed(1))
    f, _ = acc.flops(w.B, w.H, w.N, w.d, blockmask=bm.numpy())
    assert f == 4 * 128 * 2160 * 128 * 128 * 32
