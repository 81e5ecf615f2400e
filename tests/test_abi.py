"""C-ABI library: loads, exports what include/fa.h declares, and rejects bad
arguments on the host before launching anything (no GPU needed)."""

import ctypes
import os
import subprocess

import pytest

from io_aware_exact_tiled_gb300 import binding as fb
from io_aware_exact_tiled_gb300 import build as fbuild


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return fb.load()


def test_exports_every_declared_symbol(lib):
    declared = fb.declared_functions()
    assert {"fa_fwd", "fa_bwd", "fa_fwd_workspace_size", "fa_bwd_workspace_size", "fa_get_status",
            "fa_status_string"} <= set(declared)
    out = subprocess.run(["nm", "-D", "--defined-only", fb.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in declared:
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings(lib):
    for code in range(5):
        s = fb.status_string(code)
        assert s.startswith("FA_")
    assert "unknown" in fb.status_string(77)


def test_workspace_sizes(lib):
    B, H, N, d = 2, 3, 256, 64
    rows = B * H * N
    a256 = lambda x: (x + 255) // 256 * 256
    assert lib.fa_bwd_workspace_size(B, H, N, d) == 256 + 2 * a256(rows * 4) + a256(rows * d * 4)
    assert lib.fa_fwd_workspace_size(B, H, N, d) == 256 + 5 * a256(rows * d * 4)
    assert lib.fa_fwd_workspace_size(0, 1, 128, 64) == 0


FAKE = 1 << 20          # a 16-byte aligned non-null value; never dereferenced
MIS = (1 << 20) + 2     # misaligned


def fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=128, d=64, scale=0.125, causal=0,
        bm=None, kl=None, dtype=fb.FA_BF16, ws=FAKE, wsb=1 << 30):
    vp = ctypes.c_void_p
    return lib.fa_fwd(vp(q), vp(k), vp(v), vp(o), vp(lse), B, H, N, d, scale, causal, bm, kl, dtype, vp(ws),
                      wsb, None)


def bwd(lib, dtype=fb.FA_BF16, d=64, N=128, wsb=1 << 30, do=FAKE, scale=0.125, lse=FAKE):
    vp = ctypes.c_void_p
    return lib.fa_bwd(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(lse), vp(do), vp(FAKE), vp(FAKE), vp(FAKE),
                      1, 1, N, d, scale, 0, None, None, dtype, vp(FAKE), wsb, None)


def test_fwd_rejects_bad_arguments(lib):
    assert fwd(lib, q=0) == fb.FA_ERR_INVALID_ARG
    assert fwd(lib, lse=0) == fb.FA_ERR_INVALID_ARG
    assert fwd(lib, ws=0) == fb.FA_ERR_INVALID_ARG
    assert fwd(lib, B=0) == fb.FA_ERR_INVALID_ARG
    assert fwd(lib, N=-128) == fb.FA_ERR_INVALID_ARG
    assert fwd(lib, scale=0.0) == fb.FA_ERR_INVALID_ARG
    assert fwd(lib, scale=float("nan")) == fb.FA_ERR_INVALID_ARG
    assert fwd(lib, causal=2) == fb.FA_ERR_INVALID_ARG
    assert fwd(lib, dtype=7) == fb.FA_ERR_INVALID_ARG
    assert fwd(lib, q=MIS) == fb.FA_ERR_INVALID_ARG
    assert fwd(lib, ws=FAKE + 16) == fb.FA_ERR_INVALID_ARG
    assert fwd(lib, d=96) == fb.FA_ERR_UNSUPPORTED
    assert fwd(lib, d=256) == fb.FA_ERR_UNSUPPORTED
    assert fwd(lib, N=100) == fb.FA_ERR_UNSUPPORTED
    assert fwd(lib, B=1 << 16) == fb.FA_ERR_UNSUPPORTED
    assert fwd(lib, H=1 << 16) == fb.FA_ERR_UNSUPPORTED
    assert fwd(lib, B=4096, H=4096, N=256) == fb.FA_ERR_UNSUPPORTED
    assert fwd(lib, dtype=fb.FA_FP32, d=128) == fb.FA_ERR_UNSUPPORTED
    assert fwd(lib, dtype=fb.FA_FP32, wsb=1000) == fb.FA_ERR_INVALID_ARG
    assert fwd(lib, wsb=100) == fb.FA_ERR_INVALID_ARG


def test_bwd_rejects_bad_arguments(lib):
    assert bwd(lib, do=0) == fb.FA_ERR_INVALID_ARG
    assert bwd(lib, lse=FAKE + 4) == fb.FA_ERR_INVALID_ARG
    assert bwd(lib, dtype=fb.FA_FP32) == fb.FA_ERR_UNSUPPORTED
    assert bwd(lib, d=80) == fb.FA_ERR_UNSUPPORTED
    assert bwd(lib, N=130) == fb.FA_ERR_UNSUPPORTED
    assert bwd(lib, scale=-1.0) == fb.FA_ERR_INVALID_ARG
    assert bwd(lib, wsb=4096) == fb.FA_ERR_INVALID_ARG


def test_get_status_null(lib):
    assert lib.fa_get_status(None, None) == fb.FA_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(fb, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        fb.load(str(tmp_path / "nope.so"))


def test_other_entry_points_reject_bad_arguments_on_the_host(lib):
    """Every entry point's argument checks run before anything touches the
    GPU, so they answer here without one."""
    vp = ctypes.c_void_p
    P = vp(FAKE)
    big = 1 << 30

    def fp8(d=128, N=256, signs=FAKE, q=FAKE, wsb=big, causal=0):
        return lib.fa_fwd_fp8(vp(q), P, P, P, P, 1, 2, N, d, 0.1, causal, None,
                              None if signs is None else vp(signs), P, wsb, None)
    assert fp8(q=0) == fb.FA_ERR_INVALID_ARG
    assert fp8(d=64) == fb.FA_ERR_UNSUPPORTED
    assert fp8(N=200) == fb.FA_ERR_UNSUPPORTED
    assert fp8(causal=3) == fb.FA_ERR_INVALID_ARG
    assert fp8(signs=FAKE + 2) == fb.FA_ERR_INVALID_ARG
    assert fp8(wsb=1024) == fb.FA_ERR_INVALID_ARG

    def dec(Nq=1, d=128, splits=0, dtype=fb.FA_BF16, wsb=big, scale=0.1):
        return lib.fa_decode(P, P, P, P, P, 2, 2, Nq, 4096, d, scale, None, splits, dtype, P, wsb, None)
    assert dec(Nq=9) == fb.FA_ERR_UNSUPPORTED
    assert dec(d=32) == fb.FA_ERR_UNSUPPORTED
    assert dec(dtype=fb.FA_FP32) == fb.FA_ERR_UNSUPPORTED
    assert dec(splits=-1) == fb.FA_ERR_INVALID_ARG
    assert dec(scale=float("inf")) == fb.FA_ERR_INVALID_ARG
    assert dec(wsb=64) == fb.FA_ERR_INVALID_ARG

    def vfwd(cu=FAKE, total=1000, max_seqlen=600, d=64, dtype=fb.FA_BF16, wsb=big):
        return lib.fa_fwd_varlen(P, P, P, P, P, None if cu is None else vp(cu), 3, 2, total, max_seqlen, d, 0.1, 0,
                                 dtype, P, wsb, None)
    assert vfwd(cu=None) == fb.FA_ERR_INVALID_ARG
    assert vfwd(max_seqlen=1001) == fb.FA_ERR_INVALID_ARG
    assert vfwd(d=96) == fb.FA_ERR_UNSUPPORTED
    assert vfwd(dtype=fb.FA_FP32) == fb.FA_ERR_UNSUPPORTED
    assert vfwd(cu=FAKE + 2) == fb.FA_ERR_INVALID_ARG
    assert vfwd(wsb=16) == fb.FA_ERR_INVALID_ARG

    def dfwd(p=0.1, d=64, N=256):
        return lib.fa_fwd_dropout(P, P, P, P, P, 1, 1, N, d, 0.1, 0, None, p, 7, P, big, None)
    assert dfwd(p=1.0) == fb.FA_ERR_INVALID_ARG
    assert dfwd(p=-0.1) == fb.FA_ERR_INVALID_ARG
    assert dfwd(p=float("nan")) == fb.FA_ERR_INVALID_ARG
    assert dfwd(d=80) == fb.FA_ERR_UNSUPPORTED
    assert dfwd(N=300) == fb.FA_ERR_UNSUPPORTED


def test_timing_hook_and_launch_counter_on_the_host(lib):
    vp = ctypes.c_void_p
    assert lib.fa_set_timing_events(vp(FAKE), None) == fb.FA_ERR_INVALID_ARG
    assert lib.fa_set_timing_events(None, vp(FAKE)) == fb.FA_ERR_INVALID_ARG
    assert lib.fa_set_timing_events(None, None) == fb.FA_OK
    before = lib.fa_last_launch_count()
    assert fwd(lib, q=0) == fb.FA_ERR_INVALID_ARG    # a refused call launches nothing and keeps the count
    assert lib.fa_last_launch_count() == before
