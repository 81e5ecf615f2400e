"""The Python binding's marshalling, on the CPU: a stand-in for libfa.so
records every call, so each wrapper is checked for the argument order of
include/fa.h, for the byte size of the workspace it passes, and for refusing
caller-supplied buffers of the wrong shape, type or layout before any call
is made (the library cannot see a device buffer's size)."""

import ctypes
import math

import re

import pytest
import torch

from io_aware_exact_tiled_gb300 import binding as fb
from io_aware_exact_tiled_gb300 import build as fbuild


class FakeLib:
    """Records (name, args); entry points return FA_OK, size queries 4096."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if not name.startswith("fa_"):
            raise AttributeError(name)

        def call(*args):
            self.calls.append((name, args))
            return 4096 if name.endswith("_workspace_size") else fb.FA_OK
        return call


def addr(t):
    return t.data_ptr()


def val(a):
    return a.value if isinstance(a, ctypes.c_void_p) else a


@pytest.fixture
def lib(monkeypatch):
    fake = FakeLib()
    monkeypatch.setattr(fb, "_lib", fake)
    monkeypatch.setattr(fb, "_check_device", lambda q: None)
    monkeypatch.setattr(fb, "_stream_handle", lambda stream=None: None)
    return fake


def qkv(B=1, H=2, N=128, d=64, dtype=torch.bfloat16):
    return [torch.zeros(B, H, N, d, dtype=dtype) for _ in range(4)]


def last(lib, name):
    names = [c[0] for c in lib.calls]
    assert name in names, names
    return [val(a) for a in [c for c in lib.calls if c[0] == name][-1][1]]


def test_forward_and_backward_argument_order(lib):
    q, k, v, do = qkv()
    o, L = torch.empty_like(q), torch.empty(1, 2, 128)
    ws = torch.empty(100, dtype=torch.float32)
    kl = torch.tensor([77], dtype=torch.int32)
    bm = torch.ones(1, 1, dtype=torch.uint8)
    fb.forward(q, k, v, scale=0.5, causal=True, blockmask=bm, kv_len=kl, out=o, lse=L, ws=ws)
    a = last(lib, "fa_fwd")
    assert a[:5] == [addr(q), addr(k), addr(v), addr(o), addr(L)]
    assert a[5:11] == [1, 2, 128, 64, 0.5, 1] and a[11:14] == [addr(bm), addr(kl), fb.FA_BF16]
    assert a[14] == addr(ws) and a[15] == 400          # bytes, not elements
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    fb.backward(q, k, v, o, L, do, scale=0.5, causal=False, dq=dq, dk=dk, dv=dv, ws=ws)
    a = last(lib, "fa_bwd")
    assert a[:9] == [addr(t) for t in (q, k, v, o, L, do, dq, dk, dv)]
    assert a[9:15] == [1, 2, 128, 64, 0.5, 0] and a[15:17] == [None, None]
    assert a[17:19] == [fb.FA_BF16, addr(ws)] and a[19] == 400
    fb.backward_noalloc(q, k, v, o, L, do, dq=dq, dk=dk, dv=dv)
    a = last(lib, "fa_bwd_noalloc")
    assert a[:9] == [addr(t) for t in (q, k, v, o, L, do, dq, dk, dv)] and len(a) == 19


def test_workspace_allocated_from_the_size_query(lib):
    q, k, v, do = qkv()
    o, L = fb.forward(q, k, v)
    a = last(lib, "fa_fwd")
    assert a[15] == 256 and o.shape == q.shape and L.shape == (1, 2, 128) and L.dtype == torch.float32
    fb.backward(q, k, v, o, L, do)
    assert last(lib, "fa_bwd_workspace_size") == [1, 2, 128, 64] and last(lib, "fa_bwd")[19] == 4096
    q32 = [t.float() for t in qkv()]
    fb.forward(*q32[:3])
    assert last(lib, "fa_fwd")[13] == fb.FA_FP32 and last(lib, "fa_fwd")[15] == 4096


def test_wrong_outputs_are_refused_before_the_call(lib):
    q, k, v, do = qkv()
    o, L = torch.empty_like(q), torch.empty(1, 2, 128)
    bad_o = [torch.empty(1, 2, 128, 32, dtype=torch.bfloat16), torch.empty_like(q, dtype=torch.float16),
             torch.empty(1, 2, 64, 128, dtype=torch.bfloat16).transpose(2, 3)]
    for b in bad_o:
        with pytest.raises(ValueError, match="out"):
            fb.forward(q, k, v, out=b, lse=L)
        with pytest.raises(ValueError, match="dq"):
            fb.backward(q, k, v, o, L, do, dq=b)
        with pytest.raises(ValueError, match="dv"):
            fb.backward_dropout(q, k, v, o, L, do, 0.1, 1, dv=b)
        with pytest.raises(ValueError, match="dk"):
            fb.backward_noalloc(q, k, v, o, L, do, dk=b)
    for b in (torch.empty(1, 2, 127), torch.empty(1, 2, 128, dtype=torch.float64), torch.empty(2, 128).t()):
        with pytest.raises(ValueError, match="lse"):
            fb.forward(q, k, v, lse=b)
        with pytest.raises(ValueError, match="lse"):
            fb.backward(q, k, v, o, b, do)
        with pytest.raises(ValueError, match="lse"):
            fb.forward_dropout(q, k, v, 0.1, 1, lse=b)
    with pytest.raises(ValueError, match="workspace"):
        fb.forward(q, k, v, ws=torch.empty(8, 64, dtype=torch.uint8)[:, ::2])
    assert lib.calls == []


def test_packed_decode_fp8_dropout_argument_order(lib):
    total, H, d = 300, 2, 128
    q, k, v, do = (torch.zeros(total, H, d, dtype=torch.bfloat16) for _ in range(4))
    cu = torch.tensor([0, 100, 300], dtype=torch.int32)
    o, L = fb.forward_varlen(q, k, v, cu, 200, causal=True)
    a = last(lib, "fa_fwd_varlen")
    assert a[:6] == [addr(q), addr(k), addr(v), addr(o), addr(L), addr(cu)]
    assert a[6:11] == [2, H, total, 200, d] and L.shape == (H, total)
    fb.backward_varlen(q, k, v, o, L, do, cu, 200)
    a = last(lib, "fa_bwd_varlen")
    assert a[9] == addr(cu) and a[10:15] == [2, H, total, 200, d] and a[19] == 4096
    with pytest.raises(ValueError, match="lse"):
        fb.backward_varlen(q, k, v, o, torch.empty(total, H), do, cu, 200)
    with pytest.raises(ValueError, match="out"):
        fb.forward_varlen(q, k, v, cu, 200, out=torch.empty(total, H, 64, dtype=torch.bfloat16))

    qd = torch.zeros(2, 4, 3, 128, dtype=torch.bfloat16)
    kc, vc = torch.zeros(2, 4, 1000, 128, dtype=torch.bfloat16), torch.zeros(2, 4, 1000, 128, dtype=torch.bfloat16)
    cl = torch.tensor([5, 1000], dtype=torch.int32)
    o, L = fb.decode(qd, kc, vc, cache_len=cl, num_splits=7)
    a = last(lib, "fa_decode")
    assert a[:5] == [addr(qd), addr(kc), addr(vc), addr(o), addr(L)] and a[5:10] == [2, 4, 3, 1000, 128]
    assert a[11:14] == [addr(cl), 7, fb.FA_BF16] and L.shape == (2, 4, 3)
    assert last(lib, "fa_decode_workspace_size") == [2, 4, 3, 1000, 128, 7]
    with pytest.raises(ValueError, match="lse"):
        fb.decode(qd, kc, vc, lse=torch.empty(2, 4, 1))

    q4, k4, v4, do4 = qkv(d=128)
    signs = torch.ones(128)
    o, L = fb.forward_fp8(q4, k4, v4, signs, causal=True)
    a = last(lib, "fa_fwd_fp8")
    assert a[:5] == [addr(q4), addr(k4), addr(v4), addr(o), addr(L)]
    assert a[9:13] == [1 / math.sqrt(128), 1, None, addr(signs)]
    fb.forward_fp8(q4, k4, v4, None)
    assert last(lib, "fa_fwd_fp8")[12] is None
    o, L = fb.forward_dropout(q4, k4, v4, 0.25, -1)
    a = last(lib, "fa_fwd_dropout")
    assert a[12:14] == [0.25, 2 ** 64 - 1]
    fb.backward_dropout(q4, k4, v4, o, L, do4, 0.25, 3)
    a = last(lib, "fa_bwd_dropout")
    assert a[:9][3:6] == [addr(o), addr(L), addr(do4)] and a[16:18] == [0.25, 3]


def test_inputs_must_share_a_device_and_be_cuda():
    q, k, v, _ = qkv()
    with pytest.raises(ValueError, match="CUDA"):
        fb._check_qkv(q, k, v)
    with pytest.raises(ValueError, match="CUDA"):
        fb._check_device(q)


C_TO_CTYPES = {"int": ctypes.c_int, "float": ctypes.c_float, "size_t": ctypes.c_size_t,
               "unsigned long long": ctypes.c_ulonglong, "fa_dtype": ctypes.c_int, "fa_status": ctypes.c_int,
               "const char*": ctypes.c_char_p}


def header_signatures():
    """{name: (return type, [parameter types])} from include/fa.h."""
    text = re.sub(r"/\*.*?\*/", "", open(fb.HEADER_PATH).read(), flags=re.S)
    sigs = {}
    for m in re.finditer(r"(\w[\w\s*]*?)\b(fa_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        params = [] if m.group(3).strip() == "void" else [" ".join(p.split()) for p in m.group(3).split(",")]
        types = []
        for p in params:
            t = p.rsplit(" ", 1)[0] if "*" not in p else p[: p.rindex("*") + 1]
            types.append("ptr" if t.endswith("*") else t)
        sigs[m.group(2)] = (" ".join(m.group(1).split()), types)
    return sigs


def test_ctypes_signatures_match_the_header(monkeypatch):
    fbuild.build()
    monkeypatch.setattr(fb, "_lib", None)
    lib = fb.load()
    sigs = header_signatures()
    assert set(sigs) == set(fb.declared_functions())
    for name, (ret, params) in sigs.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, f"{name}: argtypes not declared"
        expect = [ctypes.c_void_p if t == "ptr" else C_TO_CTYPES[t.replace("const ", "")] for t in params]
        assert list(fn.argtypes) == expect, name
        assert fn.restype == C_TO_CTYPES[ret], name


def test_python_names_follow_the_header():
    import io_aware_exact_tiled_gb300 as pkg
    declared = fb.declared_functions()
    assert set(fb.C_NAMES) == set(declared)
    for name in declared:
        assert getattr(pkg, name) is fb.C_NAMES[name] and getattr(fb, name) is fb.C_NAMES[name]


def test_workspace_size_wrappers(lib):
    assert fb.fa_decode_workspace_size(2, 4, 1, 1000, 128) == 4096
    assert last(lib, "fa_decode_workspace_size") == [2, 4, 1, 1000, 128, 0]
    fb.fa_fwd_varlen_workspace_size(2, 300, 64)
    assert last(lib, "fa_fwd_varlen_workspace_size") == [2, 300, 64]
    fb.fa_bwd_varlen_workspace_size(3, 2, 300, 64)
    assert last(lib, "fa_bwd_varlen_workspace_size") == [3, 2, 300, 64]
    fb.fa_fwd_fp8_workspace_size(1, 2, 256, 128)
    assert last(lib, "fa_fwd_fp8_workspace_size") == [1, 2, 256, 128]
