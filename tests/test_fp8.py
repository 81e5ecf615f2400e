"""GPU parity of the FP8 forward pass (fa_fwd_fp8).

The reference is the FP8 oracle's definition (`oracle.fp8.fp8_forward`:
steps 1-6 of "FlashAttention-3"'s FP8 bullet, with every weight rounded to
E4M3 relative to the floor of its row's final maximum). The kernel rounds
relative to a running integer exponent instead, which changes only weights
in E4M3's subnormal range; the oracle's `fp8_shift_bound` bounds the effect
per element. So O must satisfy |o - O| <= 2e-2 + bound element by element
(2e-2: fp32 accumulation order and ex2.approx can move a weight across an
E4M3 rounding boundary, one step being 2^-4 of the weight), and L <= 1e-3
(L comes from the unrounded weights). A second, tighter comparison is made
with `fp8_forward_online`, a model of the running-exponent procedure:
O max-abs <= 2e-2, relative Frobenius <= 5e-3. The quantised operands are
compared bit for bit (the Hadamard transform of these bf16 inputs needs no
rounding in fp32), and the rotation's purpose is checked on the GPU: on
inputs with outlier channels the kernel's error against exact attention is
lower with the rotation than without.
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
    o, lse = fb.forward_fp8(q, k, v, None if signs is None else signs.to(dev), scale=x.scale, causal=causal,
                            kv_len=None if kv_len is None else kv_len.to(dev), ws=ws)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def lse_err(lse, L):
    both = np.isneginf(L) & np.isneginf(lse)
    with np.errstate(invalid="ignore"):
        return float(np.where(both, 0.0, np.abs(lse - L)).max())


def check(o, lse, x, signs, causal, kv_len=None):
    kw = dict(causal=causal, kv_len=kv_len)
    s = signs.numpy()
    # the definition, within the derived bound
    O, L = F8.fp8_forward(x.q, x.k, x.v, x.scale, s, **kw)
    bound = F8.fp8_shift_bound(x.q, x.k, x.v, x.scale, s, **kw)
    excess = float((np.abs(o - O) - bound).max())
    assert excess <= TOL_O8, ("O beyond 2e-2 + derived bound", excess)
    assert lse_err(lse, L) <= TOL_L8, lse_err(lse, L)
    # the running-exponent model, tightly
    O1, _ = F8.fp8_forward_online(x.q, x.k, x.v, x.scale, s, **kw)
    eo = float(np.abs(o - O1).max())
    ef = float(np.linalg.norm(o - O1) / np.linalg.norm(O1))
    assert eo <= TOL_O8 and ef <= TOL_F8, (eo, ef)


@pytest.mark.gpu
@pytest.mark.parametrize("N", [128, 384, 1024])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_parity(cuda_device, N, causal):
    w = W.Workload("fp8case", 2, 2, N, 128, causal=causal)
    x = W.make_inputs(w, seed=N)
    signs = W.make_signs(128, seed=N)
    o, lse = run(x, signs, cuda_device, causal)
    check(o, lse, x, signs, causal)


@pytest.mark.gpu
def test_fp8_parity_wide_scores_long_rows(cuda_device):
    """K x 2 (the long-context workloads' score range), causal, N = 2048:
    many weights fall in E4M3's subnormal range relative to the final
    maxima, so the derived bound is exercised."""
    w = W.Workload("fp8wide", 1, 2, 2048, 128, causal=True, k_scale=2.0)
    x = W.make_inputs(w, seed=21)
    signs = W.make_signs(128, seed=21)
    o, lse = run(x, signs, cuda_device, True)
    check(o, lse, x, signs, True)


@pytest.mark.gpu
def test_fp8_key_padding_and_scaled_keys(cuda_device):
    w = W.Workload("fp8pad", 3, 2, 512, 128, kv_len_range=(1, 512), k_scale=2.0)
    x = W.make_inputs(w, seed=3)
    x.kv_len[:] = torch.tensor([512, 129, 1], dtype=torch.int32)
    signs = W.make_signs(128, seed=3)
    o, lse = run(x, signs, cuda_device, False, kv_len=x.kv_len)
    check(o, lse, x, signs, False, kv_len=x.kv_len)


@pytest.mark.gpu
@pytest.mark.parametrize("rotate", [True, False], ids=["rotated", "unrotated"])
def test_fp8_quantised_operands_bit_exact(cuda_device, rotate):
    """The workspace holds the E4M3 Q, K, V^T and the block exponents
    (layout: 256-byte status, then Q8, K8, V8^T, Q and K exponents, V
    exponents, each 256-byte aligned); they equal the oracle's steps 1-3."""
    B, H, N, d = 1, 2, 256, 128
    w = W.Workload("fp8q", B, H, N, d)
    x = W.make_inputs(w, seed=5)
    signs = W.make_signs(d, seed=5)
    ws = fb.workspace(fb.load().fa_fwd_fp8_workspace_size(B, H, N, d), cuda_device)
    run(x, signs if rotate else None, cuda_device, False, ws=ws)
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
        q8r, sq, k8r, sk, v8r, sv = F8.quantized_inputs(x.q[0, h], x.k[0, h], x.v[0, h], signs.numpy(),
                                                        rotate=rotate)
        np.testing.assert_array_equal(dec(q8[h * N * d:(h + 1) * N * d]).reshape(N, d), q8r)
        np.testing.assert_array_equal(dec(k8[h * N * d:(h + 1) * N * d]).reshape(N, d), k8r)
        np.testing.assert_array_equal(dec(vt8[h * N * d:(h + 1) * N * d]).reshape(d, N), v8r.T)
        np.testing.assert_array_equal(np.exp2(qe[h * T:(h + 1) * T].astype(np.float64)), sq)
        np.testing.assert_array_equal(np.exp2(ke[h * T:(h + 1) * T].astype(np.float64)), sk)
        assert 2.0 ** int(ve[h]) == sv


@pytest.mark.gpu
def test_fp8_unrotated_parity(cuda_device):
    w = W.Workload("fp8plain", 1, 2, 512, 128, causal=True)
    x = W.make_inputs(w, seed=17)
    o, lse = run(x, None, cuda_device, True)
    ones = np.ones(128)
    O, L = F8.fp8_forward(x.q, x.k, x.v, x.scale, ones, causal=True, rotate=False)
    bound = F8.fp8_shift_bound(x.q, x.k, x.v, x.scale, ones, causal=True, rotate=False)
    assert float((np.abs(o - O) - bound).max()) <= TOL_O8
    assert lse_err(lse, L) <= TOL_L8


@pytest.mark.gpu
def test_fp8_rotation_lowers_error_with_outlier_channels(cuda_device):
    """FlashAttention-3's reason for the rotation, on the GPU: Q and K with a
    few channels 30x larger than the rest set the block scales, so the other
    channels lose precision; spreading the outliers over all channels with
    the Hadamard rotation lowers the kernel's error against exact fp64
    attention."""
    ratios = []
    for seed in range(4):
        g = torch.Generator().manual_seed(100 + seed)
        B, H, N, d = 1, 2, 256, 128
        q, k, v = (torch.randn(B, H, N, d, generator=g) for _ in range(3))
        out = torch.randperm(d, generator=g)[:3]
        q[..., out] *= 30.0
        k[..., out] *= 30.0
        q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
        scale = 1 / np.sqrt(d) / 10.0
        x = W.Inputs(q=q, k=k, v=v, do=None, scale=scale, causal=False, kv_len=None, blockmask=None)
        signs = W.make_signs(d, seed=100 + seed)
        O, _ = oracle.forward(q, k, v, scale)
        o_rot, _ = run(x, signs, cuda_device, False)
        o_plain, _ = run(x, None, cuda_device, False)
        e_rot = np.linalg.norm(o_rot - O) / np.linalg.norm(O)
        e_plain = np.linalg.norm(o_plain - O) / np.linalg.norm(O)
        ratios.append(e_plain / e_rot)
    assert np.median(ratios) > 1.5, ratios


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


@pytest.mark.gpu
def test_fp8_long8k_sampled_heads(cuda_device):
    """The benchmarked shape (B 1, H 32, N 8192, d 128, causal, K x 2), run
    whole on the GPU; whole heads 0 and 31 are compared with the definition
    within the derived bound, and head 31 also with the single-pass model at
    the tight tolerances (quantisation is per head, so a head taken on its
    own is exact). With 8K keys per row the bound is wide, which is why the
    model comparison is kept here as well."""
    w = W.WORKLOADS["long8k"]
    x = W.make_inputs(w, seed=0)
    signs = W.make_signs(128, seed=0)
    o, lse = run(x, signs, cuda_device, True)
    s = signs.numpy()
    for h in (0, 31):
        sub = lambda t: t[:, h:h + 1]
        O, L = F8.fp8_forward(sub(x.q), sub(x.k), sub(x.v), x.scale, s, causal=True)
        bound = F8.fp8_shift_bound(sub(x.q), sub(x.k), sub(x.v), x.scale, s, causal=True)
        excess = float((np.abs(o[:, h:h + 1] - O) - bound).max())
        assert excess <= TOL_O8, (h, excess)
        assert lse_err(lse[:, h:h + 1], L) <= TOL_L8, (h, lse_err(lse[:, h:h + 1], L))
        if h == 31:
            O1, _ = F8.fp8_forward_online(sub(x.q), sub(x.k), sub(x.v), x.scale, s, causal=True)
            oh = o[:, h:h + 1]
            eo = float(np.abs(oh - O1).max())
            ef = float(np.linalg.norm(oh - O1) / np.linalg.norm(O1))
            assert eo <= TOL_O8 and ef <= TOL_F8, (eo, ef)
