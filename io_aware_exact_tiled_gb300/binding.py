"""ctypes binding of libfa.so (include/fa.h), argument marshalling only.

Every step of the attention path runs in the CUDA kernels behind the C ABI;
this module checks tensor properties, allocates outputs and workspace with
PyTorch when the caller does not pass them, and forwards raw device pointers
and the current CUDA stream. There is no fallback: if the library is missing
or a call fails, an exception is raised.
"""

from __future__ import annotations

import ctypes
import math
import os
import re
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "fa.h")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
FA_BF16, FA_FP32 = 0, 1


class FAError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})")


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libfa.so and declare the C signatures. Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, sz, i, f = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
    lib.fa_fwd_workspace_size.argtypes = [i, i, i, i]
    lib.fa_fwd_workspace_size.restype = sz
    lib.fa_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.fa_bwd_workspace_size.restype = sz
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, i, vp, sz, vp]
    lib.fa_fwd.restype = i
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, i, vp, sz, vp]
    lib.fa_bwd.restype = i
    lib.fa_fwd_varlen_workspace_size.argtypes = [i, i, i]
    lib.fa_fwd_varlen_workspace_size.restype = sz
    lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz, vp]
    lib.fa_fwd_varlen.restype = i
    lib.fa_bwd_varlen_workspace_size.argtypes = [i, i, i, i]
    lib.fa_bwd_varlen_workspace_size.restype = sz
    lib.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz, vp]
    lib.fa_bwd_varlen.restype = i
    lib.fa_decode_workspace_size.argtypes = [i, i, i, i, i, i]
    lib.fa_decode_workspace_size.restype = sz
    lib.fa_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, i, i, vp, sz, vp]
    lib.fa_decode.restype = i
    lib.fa_fwd_fp8_workspace_size.argtypes = [i, i, i, i]
    lib.fa_fwd_fp8_workspace_size.restype = sz
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, vp, sz, vp]
    lib.fa_fwd_fp8.restype = i
    u64 = ctypes.c_ulonglong
    lib.fa_fwd_dropout.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, f, u64, vp, sz, vp]
    lib.fa_fwd_dropout.restype = i
    lib.fa_bwd_dropout.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, f, u64, vp, sz, vp]
    lib.fa_bwd_dropout.restype = i
    lib.fa_get_status.argtypes = [vp, vp]
    lib.fa_get_status.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_last_launch_count.argtypes = []
    lib.fa_last_launch_count.restype = i
    lib.fa_set_timing_events.argtypes = [vp, vp]
    lib.fa_set_timing_events.restype = i
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, i, vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_bwd_noalloc_get_status.argtypes = [vp]
    lib.fa_bwd_noalloc_get_status.restype = i
    _lib = lib
    return lib


def declared_functions(header: str = HEADER_PATH):
    """Names of the functions include/fa.h declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def status_string(code: int) -> str:
    return load().fa_status_string(code).decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check_device(q: torch.Tensor):
    """The kernels run on the current CUDA device: q must live there."""
    if q.device.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    if q.device.index != torch.cuda.current_device():
        raise ValueError(f"tensors are on {q.device} but the current device is cuda:{torch.cuda.current_device()}:"
                         " call under torch.cuda.device(q.device)")


def _in(t: torch.Tensor, shape, dtype, device, name: str) -> torch.Tensor:
    """Check a buffer the kernels read or write as exactly `shape` contiguous
    elements of `dtype` on `device` (the library cannot see its size)."""
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or t.device != device or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} {list(shape)} tensor on {device}")
    return t


def _out(t: Optional[torch.Tensor], shape, dtype, device, name: str) -> torch.Tensor:
    """A caller-supplied output, checked as in _in, or a new one."""
    if t is None:
        return torch.empty(tuple(shape), dtype=dtype, device=device)
    return _in(t, shape, dtype, device, name)


def _ws(ws: Optional[torch.Tensor], nbytes, device) -> torch.Tensor:
    """A caller-supplied workspace (on the device, contiguous; its size is
    checked by the library) or a new one of `nbytes`."""
    if ws is None:
        return workspace(nbytes() if callable(nbytes) else nbytes, device)
    if ws.device != device or not ws.is_contiguous():
        raise ValueError(f"the workspace must be a contiguous tensor on {device}")
    return ws


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def _check_qkv(*ts: torch.Tensor):
    q = ts[0]
    _check_device(q)
    for t in ts:
        if t.device != q.device:
            raise ValueError("tensors must be on the same CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous [B, H, N, d]")
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError("q, k, v (and o, dO) must share shape and dtype")
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    if q.dtype == torch.bfloat16:
        return FA_BF16
    if q.dtype == torch.float32:
        return FA_FP32
    raise ValueError("dtype must be bfloat16 or float32")


def _mask_ptrs(blockmask, kv_len, q):
    if blockmask is not None:
        T = q.shape[2] // 128
        if blockmask.dtype != torch.uint8 or blockmask.shape != (T, T) or not blockmask.is_contiguous():
            raise ValueError(f"blockmask must be a contiguous uint8 [{T}, {T}] tensor")
        if blockmask.device != q.device:
            raise ValueError("blockmask must be on the same device")
    if kv_len is not None:
        if kv_len.dtype != torch.int32 or kv_len.shape != (q.shape[0],) or kv_len.device != q.device:
            raise ValueError("kv_len must be an int32 [B] tensor on the same device")
    return _ptr(blockmask), _ptr(kv_len)


def fwd_workspace_size(B, H, N, d) -> int:
    return load().fa_fwd_workspace_size(B, H, N, d)


def bwd_workspace_size(B, H, N, d) -> int:
    return load().fa_bwd_workspace_size(B, H, N, d)


def fwd_varlen_workspace_size(H, total, d) -> int:
    return load().fa_fwd_varlen_workspace_size(H, total, d)


def bwd_varlen_workspace_size(B, H, total, d) -> int:
    return load().fa_bwd_varlen_workspace_size(B, H, total, d)


def decode_workspace_size(B, H, Nq, Nk, d, num_splits: int = 0) -> int:
    return load().fa_decode_workspace_size(B, H, Nq, Nk, d, num_splits)


def fwd_fp8_workspace_size(B, H, N, d) -> int:
    return load().fa_fwd_fp8_workspace_size(B, H, N, d)


def workspace(nbytes: int, device) -> torch.Tensor:
    """A device buffer usable as workspace (256-byte aligned by the allocator)."""
    return torch.empty(max(256, nbytes), dtype=torch.uint8, device=device)


def forward(q, k, v, scale: Optional[float] = None, causal: bool = False, blockmask=None, kv_len=None,
            out=None, lse=None, ws=None, stream=None):
    """O, L = fa_fwd(...). Returns (o [B,H,N,d], lse fp32 [B,H,N])."""
    lib = load()
    dtype = _check_qkv(q, k, v)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = _out(out, q.shape, q.dtype, q.device, "out")
    L = _out(lse, (B, H, N), torch.float32, q.device, "lse")
    ws = _ws(ws, lambda: lib.fa_fwd_workspace_size(B, H, N, d) if dtype == FA_FP32 else 256, q.device)
    bm, kl = _mask_ptrs(blockmask, kv_len, q)
    rc = lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(L), B, H, N, d, scale, int(bool(causal)), bm, kl,
                    dtype, _ptr(ws), _nbytes(ws), _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd")
    return o, L


def _check_packed(cu_seqlens, *ts: torch.Tensor):
    q = ts[0]
    _check_device(q)
    for t in ts:
        if t.device != q.device:
            raise ValueError("tensors must be on the same CUDA device")
        if not t.is_contiguous() or t.dim() != 3:
            raise ValueError("packed tensors must be contiguous [total, H, d]")
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError("packed q, k, v (and o, dO) must share shape and dtype")
    if q.dtype != torch.bfloat16:
        raise ValueError("packed variable-length batches are bfloat16 only")
    if (cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2
            or cu_seqlens.device != q.device or not cu_seqlens.is_contiguous()):
        raise ValueError("cu_seqlens must be a contiguous int32 [B + 1] tensor on the same device")
    return FA_BF16


def forward_varlen(q, k, v, cu_seqlens, max_seqlen: int, scale: Optional[float] = None, causal: bool = False,
                   out=None, lse=None, ws=None, stream=None):
    """O, L = fa_fwd_varlen(...) on a packed batch. q, k, v: [total, H, d]
    bf16; cu_seqlens: int32 [B + 1] offsets on the device; max_seqlen: the
    longest sequence. Returns (o [total, H, d], lse fp32 [H, total])."""
    lib = load()
    dtype = _check_packed(cu_seqlens, q, k, v)
    total, H, d = q.shape
    B = cu_seqlens.numel() - 1
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = _out(out, q.shape, q.dtype, q.device, "out")
    L = _out(lse, (H, total), torch.float32, q.device, "lse")
    ws = _ws(ws, lambda: lib.fa_fwd_varlen_workspace_size(H, total, d), q.device)
    rc = lib.fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(L), _ptr(cu_seqlens), B, H, total,
                           int(max_seqlen), d, scale, int(bool(causal)), dtype, _ptr(ws), _nbytes(ws),
                           _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_varlen")
    return o, L


def backward_varlen(q, k, v, o, lse, do, cu_seqlens, max_seqlen: int, scale: Optional[float] = None,
                    causal: bool = False, dq=None, dk=None, dv=None, ws=None, stream=None):
    """dQ, dK, dV = fa_bwd_varlen(...) on a packed batch ([total, H, d] bf16;
    lse fp32 [H, total] from forward_varlen). Returns (dq, dk, dv)."""
    lib = load()
    dtype = _check_packed(cu_seqlens, q, k, v, o, do)
    total, H, d = q.shape
    B = cu_seqlens.numel() - 1
    _in(lse, (H, total), torch.float32, q.device, "lse")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = _out(dq, q.shape, q.dtype, q.device, "dq")
    dk = _out(dk, q.shape, q.dtype, q.device, "dk")
    dv = _out(dv, q.shape, q.dtype, q.device, "dv")
    ws = _ws(ws, lambda: lib.fa_bwd_varlen_workspace_size(B, H, total, d), q.device)
    rc = lib.fa_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                           _ptr(cu_seqlens), B, H, total, int(max_seqlen), d, scale, int(bool(causal)), dtype,
                           _ptr(ws), _nbytes(ws), _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc, "fa_bwd_varlen")
    return dq, dk, dv


def forward_fp8(q, k, v, signs, scale: Optional[float] = None, causal: bool = False, kv_len=None, out=None,
                lse=None, ws=None, stream=None):
    """O, L = fa_fwd_fp8(...): the FP8 forward pass with a Hadamard rotation
    (signs: float32 [128] of +-1 on the device; None skips the rotation) and
    per-block scales. q, k, v: [B, H, N, 128] bf16. Returns (o bf16, lse fp32
    [B, H, N])."""
    lib = load()
    dtype = _check_qkv(q, k, v)
    if dtype != FA_BF16:
        raise ValueError("the FP8 path takes bfloat16 inputs")
    B, H, N, d = q.shape
    if signs is not None and (signs.dtype != torch.float32 or signs.shape != (d,) or signs.device != q.device):
        raise ValueError("signs must be None or a float32 [d] tensor on the same device")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = _out(out, q.shape, q.dtype, q.device, "out")
    L = _out(lse, (B, H, N), torch.float32, q.device, "lse")
    ws = _ws(ws, lambda: lib.fa_fwd_fp8_workspace_size(B, H, N, d), q.device)
    _, kl = _mask_ptrs(None, kv_len, q)
    rc = lib.fa_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(L), B, H, N, d, scale, int(bool(causal)), kl,
                        _ptr(signs), _ptr(ws), _nbytes(ws), _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_fp8")
    return o, L


def forward_dropout(q, k, v, dropout_p: float, seed: int, scale: Optional[float] = None, causal: bool = False,
                    kv_len=None, out=None, lse=None, ws=None, stream=None):
    """O, L = fa_fwd_dropout(...): attention with dropout on the
    probabilities (bf16 [B, H, N, d]). Returns (o, lse)."""
    lib = load()
    if _check_qkv(q, k, v) != FA_BF16:
        raise ValueError("dropout takes bfloat16 inputs")
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = _out(out, q.shape, q.dtype, q.device, "out")
    L = _out(lse, (B, H, N), torch.float32, q.device, "lse")
    ws = _ws(ws, 256, q.device)
    _, kl = _mask_ptrs(None, kv_len, q)
    rc = lib.fa_fwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(L), B, H, N, d, scale, int(bool(causal)), kl,
                            float(dropout_p), int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(ws), _nbytes(ws),
                            _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_dropout")
    return o, L


def backward_dropout(q, k, v, o, lse, do, dropout_p: float, seed: int, scale: Optional[float] = None,
                     causal: bool = False, kv_len=None, dq=None, dk=None, dv=None, ws=None, stream=None):
    """dQ, dK, dV = fa_bwd_dropout(...) for forward_dropout's outputs."""
    lib = load()
    if _check_qkv(q, k, v, o, do) != FA_BF16:
        raise ValueError("dropout takes bfloat16 inputs")
    B, H, N, d = q.shape
    _in(lse, (B, H, N), torch.float32, q.device, "lse")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = _out(dq, q.shape, q.dtype, q.device, "dq")
    dk = _out(dk, q.shape, q.dtype, q.device, "dk")
    dv = _out(dv, q.shape, q.dtype, q.device, "dv")
    ws = _ws(ws, lambda: lib.fa_bwd_workspace_size(B, H, N, d), q.device)
    _, kl = _mask_ptrs(None, kv_len, q)
    rc = lib.fa_bwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                            B, H, N, d, scale, int(bool(causal)), kl, float(dropout_p),
                            int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(ws), _nbytes(ws), _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc, "fa_bwd_dropout")
    return dq, dk, dv


def decode(q, k_cache, v_cache, cache_len=None, scale: Optional[float] = None, num_splits: int = 0, out=None,
           lse=None, ws=None, stream=None):
    """O, L = fa_decode(...): Nq (1..8) query rows per (b, h) against a
    [B, H, Nk, d] bf16 cache, keys split across CTAs and merged. Returns
    (o [B, H, Nq, d], lse fp32 [B, H, Nq])."""
    lib = load()
    _check_device(q)
    for t in (q, k_cache, v_cache):
        if t.device != q.device or not t.is_contiguous() or t.dim() != 4 or t.dtype != torch.bfloat16:
            raise ValueError("q and the cache must be contiguous bf16 [B, H, N, d] tensors on one CUDA device")
    B, H, Nq, d = q.shape
    if k_cache.shape != v_cache.shape or k_cache.shape[:2] != (B, H) or k_cache.shape[3] != d:
        raise ValueError("the cache must be [B, H, Nk, d] with q's B, H and d")
    Nk = k_cache.shape[2]
    if cache_len is not None and (cache_len.dtype != torch.int32 or cache_len.shape != (B,)
                                  or cache_len.device != q.device):
        raise ValueError("cache_len must be an int32 [B] tensor on the same device")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = _out(out, q.shape, q.dtype, q.device, "out")
    L = _out(lse, (B, H, Nq), torch.float32, q.device, "lse")
    ws = _ws(ws, lambda: lib.fa_decode_workspace_size(B, H, Nq, Nk, d, num_splits), q.device)
    rc = lib.fa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(L), B, H, Nq, Nk, d, scale,
                       _ptr(cache_len), int(num_splits), FA_BF16, _ptr(ws), _nbytes(ws), _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc, "fa_decode")
    return o, L


def backward(q, k, v, o, lse, do, scale: Optional[float] = None, causal: bool = False, blockmask=None,
             kv_len=None, dq=None, dk=None, dv=None, ws=None, stream=None):
    """dQ, dK, dV = fa_bwd(...). Returns (dq, dk, dv)."""
    lib = load()
    dtype = _check_qkv(q, k, v, o, do)
    B, H, N, d = q.shape
    _in(lse, (B, H, N), torch.float32, q.device, "lse")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = _out(dq, q.shape, q.dtype, q.device, "dq")
    dk = _out(dk, q.shape, q.dtype, q.device, "dk")
    dv = _out(dv, q.shape, q.dtype, q.device, "dv")
    ws = _ws(ws, lambda: lib.fa_bwd_workspace_size(B, H, N, d), q.device)
    bm, kl = _mask_ptrs(blockmask, kv_len, q)
    rc = lib.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                    B, H, N, d, scale, int(bool(causal)), bm, kl, dtype, _ptr(ws), _nbytes(ws),
                    _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc, "fa_bwd")
    return dq, dk, dv


def get_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronise and read (then clear) the device status word of a workspace."""
    return load().fa_get_status(_ptr(ws), _stream_handle(stream))


def last_launch_count() -> int:
    return load().fa_last_launch_count()


def set_timing_events(begin=None, end=None):
    """Record torch.cuda.Event `begin`/`end` around the main attention kernel
    of the following calls on this thread (None, None turns it off)."""
    b = None if begin is None else ctypes.c_void_p(begin.cuda_event)
    e = None if end is None else ctypes.c_void_p(end.cuda_event)
    rc = load().fa_set_timing_events(b, e)
    if rc != FA_OK:
        raise FAError(rc, "fa_set_timing_events")


def backward_noalloc(q, k, v, o, lse, do, scale: Optional[float] = None, causal: bool = False, blockmask=None,
                     kv_len=None, dq=None, dk=None, dv=None, stream=None):
    """dQ, dK, dV = fa_bwd_noalloc(...): the backward pass with the library's
    own fixed scratch instead of a workspace (for callers that cannot allocate
    device memory). Outputs are allocated here only if not passed in."""
    fn = load().fa_bwd_noalloc
    dtype = _check_qkv(q, k, v, o, do)
    B, H, N, d = q.shape
    _in(lse, (B, H, N), torch.float32, q.device, "lse")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = _out(dq, q.shape, q.dtype, q.device, "dq")
    dk = _out(dk, q.shape, q.dtype, q.device, "dk")
    dv = _out(dv, q.shape, q.dtype, q.device, "dv")
    bm, kl = _mask_ptrs(blockmask, kv_len, q)
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d,
            scale, int(bool(causal)), bm, kl, dtype, _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc, "fa_bwd_noalloc")
    return dq, dk, dv


def noalloc_status(stream=None) -> int:
    """Synchronise and read (then clear) the status word of the last
    fa_bwd_noalloc call on the current device (fa_bwd_noalloc_get_status)."""
    return load().fa_bwd_noalloc_get_status(_stream_handle(stream))


# The names of include/fa.h, bound to the wrappers above (same arguments in
# tensor form; outputs returned rather than passed as pointers).
C_NAMES = {
    "fa_fwd": forward,
    "fa_bwd": backward,
    "fa_fwd_workspace_size": fwd_workspace_size,
    "fa_bwd_workspace_size": bwd_workspace_size,
    "fa_fwd_varlen": forward_varlen,
    "fa_bwd_varlen": backward_varlen,
    "fa_fwd_varlen_workspace_size": fwd_varlen_workspace_size,
    "fa_bwd_varlen_workspace_size": bwd_varlen_workspace_size,
    "fa_decode": decode,
    "fa_decode_workspace_size": decode_workspace_size,
    "fa_fwd_fp8": forward_fp8,
    "fa_fwd_fp8_workspace_size": fwd_fp8_workspace_size,
    "fa_fwd_dropout": forward_dropout,
    "fa_bwd_dropout": backward_dropout,
    "fa_bwd_noalloc": backward_noalloc,
    "fa_bwd_noalloc_get_status": noalloc_status,
    "fa_get_status": get_status,
    "fa_status_string": status_string,
    "fa_last_launch_count": last_launch_count,
    "fa_set_timing_events": set_timing_events,
}
globals().update(C_NAMES)
