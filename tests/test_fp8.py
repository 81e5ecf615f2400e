"""GPU parity of the FP8 forward pass (fa_fwd_fp8) against the FP8 oracle.

The quantised operands are compared bit for bit with the oracle's (the
Hadamard transform of these bf16 inputs needs no rounding in fp32), the
outputs element by element, with the tolerances derived in the design notes
for FP8 weights: O max-abs <= 2e-2 and relative Frobenius <= 5e-3, L max-abs
<= 1e-3. A last test checks the FP8 result against exact attention.
"""

import numpy as np
import pytest
import torch

from io_aware_exact_tiled_gb300 import binding as fb
from io_aware_exact_tiled_gb300 import workloads as W
import oracle
from oracle import fp8 as F8

TOL_O8, TOL_F8, TOL_L8 = 2e-2, 5e-3, 1e-3


def run(x, signs, dev, causal, kv_len=None, ws=None):
    q, k, v = (t.to(dev) for t in (x.q, x.k, x.v))
    o, lse = fb.forward_fp8(q, k, v, signs.to(dev), scale=x.scale, causal=causal,
                            kv_len=None if kv_len is None else kv_len.to(dev), ws=ws)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check(o, lse, O, L):
    eo = float(np.abs(o - O).max())
    ef = float(np.linalg.norm(o - O) / np.linalg.norm(O))
    both = np.isneginf(L) & np.isneginf(lse)
    with np.errstate(invalid="ignore"):
        el = float(np.where(both, 0.0, np.abs(lse - L)).max())
    assert eo <= TOL_O8 and ef <= TOL_F8 and el <= TOL_L8, (eo, ef, el)


@pytest.mark.gpu
@pytest.mark.parametrize("N", [128, 384, 1024])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_parity(cuda_device, N, causal):
    w = W.Workload("fp8case", 2, 2, N, 128, causal=causal)
    x = W.make_inputs(w, seed=N)
    signs = W.make_signs(128, seed=N)
    o, lse = run(x, signs, cuda_device, causal)
    O, L = F8.fp8_forward(x.q, x.k, x.v, x.scale, signs.numpy(), causal=causal)
    check(o, lse, O, L)


@pytest.mark.gpu
def test_fp8_key_padding_and_scaled_keys(cuda_device):
    w = W.Workload("fp8pad", 3, 2, 512, 128, kv_len_range=(1, 512), k_scale=2.0)
    x = W.make_inputs(w, seed=3)
    x.kv_len[:] = torch.tensor([512, 129, 1], dtype=torch.int32)
    signs = W.make_signs(128, seed=3)
    o, lse = run(x, signs, cuda_device, False, kv_len=x.kv_len)
    O, L = F8.fp8_forward(x.q, x.k, x.v, x.scale, signs.numpy(), kv_len=x.kv_len)
    check(o, lse, O, L)


@pytest.mark.gpu
def test_fp8_quantised_operands_bit_exact(cuda_device):
    """The workspace holds the E4M3 Q, K, V^T and the block exponents
    (layout: 256-byte status, then Q8, K8, V8^T, Q and K exponents, V
    exponents, each 256-byte aligned); they equal the oracle's steps 1-3."""
    B, H, N, d = 1, 2, 256, 128
    w = W.Workload("fp8q", B, H, N, d)
    x = W.make_inputs(w, seed=5)
    signs = W.make_signs(d, seed=5)
    ws = fb.workspace(fb.load().fa_fwd_fp8_workspace_size(B, H, N, d), cuda_device)
    run(x, signs, cuda_device, False, ws=ws)
    raw = ws.cpu().numpy()
    a256 = lambda n: (n + 255) // 256 * 256
    bhn, T = B * H * N, N // 128
    off = 256
    q8 = raw[off:off + bhn * d]; off += a256(bhn * d)
    k8 = raw[off:off + bhn * d]; off += a256(bhn * d)
    vt8 = raw[off:off + bhn * d]; off += a256(bhn * d)
    qe = raw[off:off + B * H * T * 4].view(np.int32); off += a256(B * H * T * 4)
    ke = raw[off:off + B * H * T * 4].view(np.int32); off += a256(B * H * T * 4)
    ve = raw[off:off + B * H * 4].view(np.int32)
    dec = lambda u8: torch.from_numpy(u8.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for h in range(H):
        q8r, sq, k8r, sk, v8r, sv = F8.quantized_inputs(x.q[0, h], x.k[0, h], x.v[0, h], signs.numpy())
        np.testing.assert_array_equal(dec(q8[h * N * d:(h + 1) * N * d]).reshape(N, d), q8r)
        np.testing.assert_array_equal(dec(k8[h * N * d:(h + 1) * N * d]).reshape(N, d), k8r)
        np.testing.assert_array_equal(dec(vt8[h * N * d:(h + 1) * N * d]).reshape(d, N), v8r.T)
        np.testing.assert_array_equal(np.exp2(qe[h * T:(h + 1) * T].astype(np.float64)), sq)
        np.testing.assert_array_equal(np.exp2(ke[h * T:(h + 1) * T].astype(np.float64)), sk)
        assert 2.0 ** int(ve[h]) == sv


@pytest.mark.gpu
def test_fp8_close_to_exact_attention(cuda_device):
    w = W.Workload("fp8exact", 1, 4, 1024, 128, causal=True)
    x = W.make_inputs(w, seed=9)
    signs = W.make_signs(128, seed=9)
    o, lse = run(x, signs, cuda_device, True)
    O, L = oracle.forward(x.q, x.k, x.v, x.scale, causal=True)
    assert float(np.abs(o - O).max()) < 0.15
    assert float(np.linalg.norm(o - O) / np.linalg.norm(O)) < 0.05
    assert float(np.abs(lse - L).max()) < 0.1


@pytest.mark.gpu
def test_fp8_rejects_other_head_sizes(cuda_device):
    w = W.Workload("fp8d64", 1, 1, 128, 64)
    x = W.make_inputs(w, seed=1)
    with pytest.raises(fb.FAError):
        run(x, W.make_signs(64), cuda_device, False)
