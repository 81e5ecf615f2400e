"""Seeded synthetic inputs for exact tiled attention.

This module only draws random tensors and structure (key lengths, tile masks).
It holds none of the attention arithmetic, so both the CUDA path and the CPU
oracle can take their inputs from here without sharing any of the method.

Workloads (shapes follow the BERT-large / GPT-2 / long-context / block-sparse
settings used to evaluate fused exact attention; weights and datasets are not
needed because attention inputs are drawn directly):

  tiny      [1, 1, 128, 64]    fp32, no mask
  bert      [8, 16, 512, 64]   bf16, key padding, valid length ~ U{256..512}
  gpt2      [8, 12, 1024, 64]  bf16, causal
  long4k    [1, 32, 4096, 128] bf16, causal, K rows scaled by 2
  long8k    [1, 32, 8192, 128] bf16, causal, K rows scaled by 2
  sparse16k [2, 16, 16384, 128] bf16, 128x128 tile mask: the diagonal plus
            floor(0.125 * (T*T - T)) other tiles, T = N / 128

Recipe: one CPU ``torch.Generator`` seeded with ``seed`` draws standard normal
fp32 tensors in the order Q, K, V, dO; then the key lengths; then the tile
mask. K is multiplied by ``k_scale`` (exact in bf16) and all four tensors are
rounded to the working dtype with round-to-nearest-even.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

TILE = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str = "bf16"          # "bf16" or "fp32"
    causal: bool = False
    kv_len_range: Optional[tuple] = None   # inclusive (lo, hi) for key padding
    block_density: Optional[float] = None  # fraction of off-diagonal tiles kept
    k_scale: float = 1.0
    backward: bool = True

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 128, 64, dtype="fp32", backward=False),
    "bert": Workload("bert", 8, 16, 512, 64, kv_len_range=(256, 512)),
    "gpt2": Workload("gpt2", 8, 12, 1024, 64, causal=True),
    "long4k": Workload("long4k", 1, 32, 4096, 128, causal=True, k_scale=2.0),
    "long8k": Workload("long8k", 1, 32, 8192, 128, causal=True, k_scale=2.0),
    "sparse16k": Workload("sparse16k", 2, 16, 16384, 128, block_density=0.125),
}


def make_blockmask(T: int, density: float, gen: torch.Generator) -> torch.Tensor:
    """uint8 [T, T] tile mask: every diagonal tile kept plus exactly
    floor(density * (T*T - T)) off-diagonal tiles chosen uniformly without
    replacement (one seeded permutation of the off-diagonal positions)."""
    keep = torch.eye(T, dtype=torch.uint8)
    off = [(i, j) for i in range(T) for j in range(T) if i != j]
    n_keep = int(math.floor(density * len(off)))
    perm = torch.randperm(len(off), generator=gen)[:n_keep]
    for p in perm.tolist():
        i, j = off[p]
        keep[i, j] = 1
    return keep


@dataclasses.dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    do: torch.Tensor
    kv_len: Optional[torch.Tensor]    # int32 [B] or None
    blockmask: Optional[torch.Tensor]  # uint8 [T, T] or None
    scale: float
    causal: bool


def make_inputs(w: Workload, seed: int = 0, device: str = "cpu") -> Inputs:
    """Draw the seeded inputs of workload ``w``.

    ``device="cpu"`` follows the recipe above exactly. ``device="cuda"`` draws
    the same distributions with a CUDA generator (different numbers, same
    recipe), which is much faster for the largest shapes; whichever device
    draws, both sides of a comparison receive the same tensors.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    shape = (w.B, w.H, w.N, w.d)
    q = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    k = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    do = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if w.k_scale != 1.0:
        k.mul_(w.k_scale)
    kv_len = None
    blockmask = None
    cpu_gen = gen if device == "cpu" else torch.Generator().manual_seed(seed + 1)
    if w.kv_len_range is not None:
        lo, hi = w.kv_len_range
        kv_len = torch.randint(lo, hi + 1, (w.B,), generator=cpu_gen, dtype=torch.int64).to(torch.int32)
    if w.block_density is not None:
        blockmask = make_blockmask(w.N // TILE, w.block_density, cpu_gen)
    dt = w.torch_dtype
    return Inputs(q.to(dt), k.to(dt), v.to(dt), do.to(dt), kv_len, blockmask, w.scale, w.causal)


# --------------------------------------------------------------------------
# Packed variable-length batches (sequences concatenated along one token axis)
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class PackedWorkload:
    """A packed batch: B sequences with lengths drawn uniformly from the
    inclusive range ``len_range``, H heads of size d, bf16."""
    name: str
    B: int
    H: int
    d: int
    len_range: tuple
    causal: bool = False

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# bert_packed: the key-padding batch of the "bert" workload without its
#   padding: 8 sequences, lengths ~ U{256..512}, 16 heads, d = 64.
# mix8k_packed: a long-context mix, 16 sequences, lengths ~ U{512..8192},
#   32 heads, d = 128, causal.
PACKED_WORKLOADS = {
    "bert_packed": PackedWorkload("bert_packed", 8, 16, 64, (256, 512)),
    "mix8k_packed": PackedWorkload("mix8k_packed", 16, 32, 128, (512, 8192), causal=True),
}


@dataclasses.dataclass
class PackedInputs:
    q: torch.Tensor           # [total, H, d]
    k: torch.Tensor
    v: torch.Tensor
    do: torch.Tensor
    cu_seqlens: torch.Tensor  # int32 [B + 1], on the CPU
    lens: list
    scale: float
    causal: bool

    @property
    def max_seqlen(self) -> int:
        return max(self.lens) if self.lens else 0


def make_packed(lens, H: int, d: int, causal: bool = False, seed: int = 0, device: str = "cpu",
                k_scale: float = 1.0) -> PackedInputs:
    """Seeded packed inputs for the given sequence lengths: standard normal
    fp32 Q, K, V, dO of shape [sum(lens), H, d] drawn in that order, K times
    ``k_scale``, rounded to bf16."""
    lens = [int(x) for x in lens]
    total = sum(lens)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    shape = (total, H, d)
    q, k, v, do = (torch.randn(shape, generator=gen, device=device, dtype=torch.float32) for _ in range(4))
    if k_scale != 1.0:
        k.mul_(k_scale)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    bf = torch.bfloat16
    return PackedInputs(q.to(bf), k.to(bf), v.to(bf), do.to(bf), cu, lens, 1.0 / math.sqrt(d), causal)


def make_packed_workload(w: PackedWorkload, seed: int = 0, device: str = "cpu") -> PackedInputs:
    """Lengths ~ U{len_range} from a CPU generator seeded with ``seed``, then
    the tensors as in make_packed."""
    g = torch.Generator().manual_seed(seed)
    lo, hi = w.len_range
    lens = torch.randint(lo, hi + 1, (w.B,), generator=g).tolist()
    return make_packed(lens, w.H, w.d, w.causal, seed, device)


# --------------------------------------------------------------------------
# Decoding: a few query rows against a key/value cache
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """Nq new query rows per (b, h) against a [B, H, Nk, d] bf16 cache whose
    valid length per batch element is drawn uniformly from the inclusive
    range ``len_range``."""
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    len_range: tuple

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# decode16k: one new token for 16 requests of 32 heads, d = 128, caches of
#   8K..16K valid entries in a 16K-entry allocation.
DECODE_WORKLOADS = {
    "decode16k": DecodeWorkload("decode16k", 16, 32, 1, 16384, 128, (8192, 16384)),
}


@dataclasses.dataclass
class DecodeInputs:
    q: torch.Tensor          # [B, H, Nq, d]
    k: torch.Tensor          # [B, H, Nk, d]
    v: torch.Tensor
    cache_len: torch.Tensor  # int32 [B], on the CPU
    scale: float


def make_decode(B: int, H: int, Nq: int, Nk: int, d: int, len_range, seed: int = 0,
                device: str = "cpu") -> DecodeInputs:
    """Seeded decode inputs: standard normal fp32 q, then the K and V caches,
    rounded to bf16; cache lengths ~ U{len_range} from a CPU generator seeded
    with ``seed + 1``."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = torch.randn((B, H, Nq, d), generator=gen, device=device, dtype=torch.float32)
    k = torch.randn((B, H, Nk, d), generator=gen, device=device, dtype=torch.float32)
    v = torch.randn((B, H, Nk, d), generator=gen, device=device, dtype=torch.float32)
    lo, hi = len_range
    cl = torch.randint(lo, hi + 1, (B,), generator=torch.Generator().manual_seed(seed + 1)).to(torch.int32)
    bf = torch.bfloat16
    return DecodeInputs(q.to(bf), k.to(bf), v.to(bf), cl, 1.0 / math.sqrt(d))


def make_decode_workload(w: DecodeWorkload, seed: int = 0, device: str = "cpu") -> DecodeInputs:
    return make_decode(w.B, w.H, w.Nq, w.Nk, w.d, w.len_range, seed, device)


def make_signs(d: int, seed: int = 0) -> torch.Tensor:
    """Random signs (float32 +-1, [d]) for the FP8 path's Hadamard rotation,
    from a CPU generator seeded with ``seed + 7``."""
    g = torch.Generator().manual_seed(seed + 7)
    return torch.where(torch.rand(d, generator=g) < 0.5, -1.0, 1.0).to(torch.float32)
