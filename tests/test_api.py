"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every symbol the
header declares, and rejects every invalid argument before any CUDA call."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flashattn.h")

A = 0x10000        # a 16-byte aligned fake device address (never dereferenced: checks fail first)
MIS = 0x10008      # 8-byte aligned only


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_names(built_lib):
    assert declared_functions() == sorted(built_lib.EXPORTED)


def test_library_exports_every_declared_symbol(built_lib):
    L = built_lib.lib()
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings(built_lib):
    names = ["FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_MISALIGNED",
             "FA_ERR_WORKSPACE", "FA_ERR_CUDA", "FA_ERR_DEVICE_TIMEOUT", "FA_ERR_DEVICE_BOUNDS"]
    for code, name in enumerate(names):
        assert built_lib.fa_status_string(code) == name
    assert built_lib.fa_status_string(99) == "FA_ERR_UNKNOWN"


def test_workspace_bytes(built_lib):
    f = built_lib.fa_bwd_workspace_bytes
    rows = 2 * 32 * 4096
    assert f(2, 32, 4096, 128) == ((rows * 4 + 255) // 256) * 256 + rows * 128 * 4
    assert f(1, 1, 1, 1) == 256 + 4
    assert f(0, 1, 1, 1) == 0 and f(1, 1, -1, 64) == 0
    # sizes whose byte count does not fit in size_t give SIZE_MAX, never a wrapped small value
    big = 2 ** 31 - 1
    assert f(big, big, big, 128) == 2 ** 64 - 1
    assert f(big, big, big, big) == 2 ** 64 - 1
    assert f(big, big, 1, 1) == 2 ** 64 - 1          # 8 * (2^31 - 1)^2 bytes > 2^64
    assert f(big, 4, 1, 1) == ((big * 4 * 4 + 255) // 256) * 256 + big * 4 * 4
    L = built_lib.lib()
    # ... so the backward's workspace check rejects every buffer for them
    st = L.fa_bwd_noalloc(*([A] * 9), big, 2, 2, big, 128, 1, 0.088, None)
    assert st == built_lib.FA_ERR_WORKSPACE


def test_deterministic_workspace_bytes(built_lib):
    f, g = built_lib.fa_bwd_deterministic_workspace_bytes, built_lib.fa_bwd_workspace_bytes
    # the fa_bwd workspace, then 16 bytes of turn counters per 64-row query tile, then the abort
    # word padded to 16 bytes
    for B, Hq, N, d in [(2, 32, 4096, 128), (1, 1, 1, 64), (3, 5, 1000, 64), (1, 16, 32768, 128)]:
        assert f(B, Hq, N, d) == g(B, Hq, N, d) + B * Hq * ((N + 63) // 64) * 16 + 16
    assert f(0, 1, 1, 1) == 0 and f(1, 1, -1, 64) == 0
    big = 2 ** 31 - 1
    assert f(big, big, big, 128) == 2 ** 64 - 1
    assert f(big, big, 1, 1) == 2 ** 64 - 1


def fwd(L, Q=A, K=A, V=A, O=A, LSE=A, B=1, Hq=2, Hkv=1, N=64, d=128, causal=1, scale=0.1, fp32=False):
    fn = L.fa_fwd_fp32 if fp32 else L.fa_fwd
    return fn(Q, K, V, O, LSE, B, Hq, Hkv, N, d, causal, scale, None)


def bwd(L, ptrs=None, B=1, Hq=2, Hkv=1, N=64, d=128, causal=1, scale=0.1, ws=A, wbytes=None,
        fp32=False, det=False):
    ptrs = ptrs or [A] * 9
    if wbytes is None:
        wbytes = (L.fa_bwd_deterministic_workspace_bytes if det else
                  L.fa_bwd_workspace_bytes)(B, Hq, N, d)
    fn = L.fa_bwd_fp32 if fp32 else L.fa_bwd_deterministic if det else L.fa_bwd
    return fn(*ptrs, B, Hq, Hkv, N, d, causal, scale, ws, wbytes, None)


@pytest.mark.parametrize("fp32", [False, True])
def test_forward_rejects_invalid_arguments(built_lib, fp32):
    L = built_lib.lib()
    E = built_lib
    assert fwd(L, B=0, fp32=fp32) == E.FA_ERR_INVALID_ARG
    assert fwd(L, Hq=0, fp32=fp32) == E.FA_ERR_INVALID_ARG
    assert fwd(L, Hkv=0, fp32=fp32) == E.FA_ERR_INVALID_ARG
    assert fwd(L, N=0, fp32=fp32) == E.FA_ERR_INVALID_ARG
    assert fwd(L, N=-5, fp32=fp32) == E.FA_ERR_INVALID_ARG
    assert fwd(L, Hq=3, Hkv=2, fp32=fp32) == E.FA_ERR_INVALID_ARG
    for s in (0.0, -0.5, math.nan, math.inf):
        assert fwd(L, scale=s, fp32=fp32) == E.FA_ERR_INVALID_ARG
    assert fwd(L, d=0, fp32=fp32) == E.FA_ERR_INVALID_ARG
    assert fwd(L, d=129 if fp32 else 96, fp32=fp32) == E.FA_ERR_UNSUPPORTED
    for k in ("Q", "K", "V", "O", "LSE"):
        assert fwd(L, **{k: None}, fp32=fp32) == E.FA_ERR_MISALIGNED
        assert fwd(L, **{k: MIS}, fp32=fp32) == E.FA_ERR_MISALIGNED


@pytest.mark.parametrize("fp32", [False, True])
def test_backward_rejects_invalid_arguments(built_lib, fp32):
    L = built_lib.lib()
    E = built_lib
    assert bwd(L, B=0, fp32=fp32) == E.FA_ERR_INVALID_ARG
    assert bwd(L, Hq=4, Hkv=3, fp32=fp32) == E.FA_ERR_INVALID_ARG
    assert bwd(L, scale=math.nan, fp32=fp32) == E.FA_ERR_INVALID_ARG
    if not fp32:
        assert bwd(L, d=96, fp32=fp32) == E.FA_ERR_UNSUPPORTED
    assert bwd(L, d=200, fp32=fp32) == E.FA_ERR_UNSUPPORTED
    for k in range(9):
        ptrs = [A] * 9
        ptrs[k] = None
        assert bwd(L, ptrs, fp32=fp32) == E.FA_ERR_MISALIGNED
        ptrs[k] = MIS
        assert bwd(L, ptrs, fp32=fp32) == E.FA_ERR_MISALIGNED
    need = L.fa_bwd_workspace_bytes(1, 2, 64, 128)
    assert bwd(L, wbytes=need - 1, fp32=fp32) == E.FA_ERR_WORKSPACE
    assert bwd(L, ws=None, fp32=fp32) == E.FA_ERR_WORKSPACE
    assert bwd(L, ws=MIS, fp32=fp32) == E.FA_ERR_WORKSPACE


def test_deterministic_backward_rejects_invalid_arguments(built_lib):
    L = built_lib.lib()
    E = built_lib
    assert bwd(L, B=0, det=True) == E.FA_ERR_INVALID_ARG
    assert bwd(L, Hq=4, Hkv=3, det=True) == E.FA_ERR_INVALID_ARG
    assert bwd(L, scale=math.nan, det=True) == E.FA_ERR_INVALID_ARG
    assert bwd(L, d=96, det=True) == E.FA_ERR_UNSUPPORTED
    for k in range(9):
        ptrs = [A] * 9
        ptrs[k] = MIS
        assert bwd(L, ptrs, det=True) == E.FA_ERR_MISALIGNED
    need = L.fa_bwd_deterministic_workspace_bytes(1, 2, 64, 128)
    # fa_bwd's workspace size is not enough: the counters need their own bytes
    assert bwd(L, wbytes=L.fa_bwd_workspace_bytes(1, 2, 64, 128), det=True) == E.FA_ERR_WORKSPACE
    assert bwd(L, wbytes=need - 1, det=True) == E.FA_ERR_WORKSPACE
    assert bwd(L, ws=None, det=True) == E.FA_ERR_WORKSPACE
    assert bwd(L, ws=MIS, det=True) == E.FA_ERR_WORKSPACE


def test_split_forward_rejects_invalid_arguments(built_lib):
    L = built_lib.lib()
    E = built_lib

    def split(Q=A, K=A, V=A, Op=A, Lp=A, B=1, Hq=2, Hkv=1, N=300, d=128, S=3, scale=0.1):
        return L.fa_fwd_split(Q, K, V, Op, Lp, B, Hq, Hkv, N, d, 1, scale, S, None)

    assert split(B=0) == E.FA_ERR_INVALID_ARG
    assert split(Hq=3, Hkv=2) == E.FA_ERR_INVALID_ARG
    assert split(scale=math.nan) == E.FA_ERR_INVALID_ARG
    assert split(S=0) == E.FA_ERR_INVALID_ARG
    assert split(S=E.MAX_SPLITS + 1) == E.FA_ERR_INVALID_ARG
    assert split(d=96) == E.FA_ERR_UNSUPPORTED
    for k in ("Q", "K", "V", "Op", "Lp"):
        assert split(**{k: None}) == E.FA_ERR_MISALIGNED
        assert split(**{k: MIS}) == E.FA_ERR_MISALIGNED


def test_merge_rejects_invalid_arguments(built_lib):
    L = built_lib.lib()
    E = built_lib

    def merge(Op=A, Lp=A, S=2, rows=4, d=8, O=A, bf16=1, Lo=A):
        return L.fa_merge(Op, Lp, S, rows, d, O, bf16, Lo, None)

    for kw in ({"S": 0}, {"S": E.MAX_SPLITS + 1}, {"rows": 0}, {"d": 0}, {"d": 6},
               {"d": 1028}):
        assert merge(**kw) == E.FA_ERR_INVALID_ARG, kw
    for k in ("Op", "Lp", "O", "Lo"):
        assert merge(**{k: None}) == E.FA_ERR_MISALIGNED
        assert merge(**{k: MIS}) == E.FA_ERR_MISALIGNED


def test_masked_forward_rejects_invalid_arguments(built_lib):
    L = built_lib.lib()
    E = built_lib

    def masked(Q=A, ql=None, kl=None, bm=None, mh=0, B=2, Hq=4, Hkv=2, N=300, d=128):
        return L.fa_fwd_masked(Q, A, A, A, A, B, Hq, Hkv, N, d, 1, 0.1, ql, kl, bm, mh, None)

    assert masked(B=0) == E.FA_ERR_INVALID_ARG
    assert masked(d=96) == E.FA_ERR_UNSUPPORTED
    assert masked(Q=MIS) == E.FA_ERR_MISALIGNED
    assert masked(ql=A + 2) == E.FA_ERR_MISALIGNED
    assert masked(kl=A + 1) == E.FA_ERR_MISALIGNED
    for mh in (0, 2, 3, 9):
        assert masked(bm=A + 1, mh=mh) == E.FA_ERR_INVALID_ARG, mh


def test_masked_backward_rejects_invalid_arguments(built_lib):
    L = built_lib.lib()
    E = built_lib

    def masked(ptrs=None, ql=None, bm=None, mh=0, B=2, Hq=4, Hkv=2, N=300, d=128, ws=A,
               wbytes=None):
        ptrs = ptrs or [A] * 9
        if wbytes is None:
            wbytes = L.fa_bwd_workspace_bytes(B, Hq, N, d)
        return L.fa_bwd_masked(*ptrs, B, Hq, Hkv, N, d, 1, 0.1, ql, None, bm, mh, ws, wbytes, None)

    assert masked(B=0) == E.FA_ERR_INVALID_ARG
    assert masked(d=96) == E.FA_ERR_UNSUPPORTED
    assert masked(Hq=64, Hkv=1, N=32768) == E.FA_ERR_UNSUPPORTED      # step list too long
    for k in range(9):
        ptrs = [A] * 9
        ptrs[k] = MIS
        assert masked(ptrs) == E.FA_ERR_MISALIGNED
    assert masked(ql=A + 2) == E.FA_ERR_MISALIGNED
    assert masked(bm=A, mh=3) == E.FA_ERR_INVALID_ARG
    assert masked(wbytes=16) == E.FA_ERR_WORKSPACE


def test_dropout_entry_points_reject_invalid_arguments(built_lib):
    L = built_lib.lib()
    E = built_lib
    for pd in (-0.1, 1.0, 1.5, math.nan):
        assert L.fa_fwd_dropout(A, A, A, A, A, 1, 2, 1, 64, 128, 1, 0.1, pd, 1, 0, None) == E.FA_ERR_INVALID_ARG
        assert L.fa_bwd_dropout(*([A] * 9), 1, 2, 1, 64, 128, 1, 0.1, pd, 1, 0, A,
                                L.fa_bwd_workspace_bytes(1, 2, 64, 128), None) == E.FA_ERR_INVALID_ARG
        assert L.fa_dropout_mask(2, 64, pd, 1, 0, A, None) == E.FA_ERR_INVALID_ARG
    assert L.fa_fwd_dropout(A, A, A, A, A, 0, 2, 1, 64, 128, 1, 0.1, 0.1, 1, 0, None) == E.FA_ERR_INVALID_ARG
    assert L.fa_fwd_dropout(A, A, A, A, A, 1, 2, 1, 64, 96, 1, 0.1, 0.1, 1, 0, None) == E.FA_ERR_UNSUPPORTED
    assert L.fa_fwd_dropout(MIS, A, A, A, A, 1, 2, 1, 64, 128, 1, 0.1, 0.1, 1, 0, None) == E.FA_ERR_MISALIGNED
    assert L.fa_bwd_dropout(*([A] * 9), 1, 2, 1, 64, 128, 1, 0.1, 0.1, 1, 0, A, 16, None) == E.FA_ERR_WORKSPACE
    assert L.fa_dropout_mask(0, 64, 0.1, 1, 0, A, None) == E.FA_ERR_INVALID_ARG
    assert L.fa_dropout_mask(2, 64, 0.1, 1, 0, None, None) == E.FA_ERR_MISALIGNED


def test_kvouter_forward_rejects_invalid_arguments(built_lib):
    L = built_lib.lib()
    E = built_lib
    need = L.fa_fwd_kvouter_workspace_bytes(1, 2, 64, 128)
    assert need == 2 * 64 * 128 * 4 + 3 * 2 * 64 * 4
    assert L.fa_fwd_kvouter_workspace_bytes(0, 2, 64, 128) == 0

    def kvo(Q=A, B=1, d=128, ws=A, wbytes=need):
        return L.fa_fwd_kvouter(Q, A, A, A, A, B, 2, 1, 64, d, 1, 0.1, ws, wbytes, None)
    assert kvo(B=0) == E.FA_ERR_INVALID_ARG
    assert kvo(d=64) == E.FA_ERR_UNSUPPORTED
    assert kvo(Q=MIS) == E.FA_ERR_MISALIGNED
    assert kvo(wbytes=need - 1) == E.FA_ERR_WORKSPACE
    assert kvo(ws=MIS) == E.FA_ERR_WORKSPACE


def test_fp32_tensor_core_forward_rejects_invalid_arguments(built_lib):
    L = built_lib.lib()
    E = built_lib
    need = L.fa_fwd_fp32_tc_workspace_bytes(1, 2, 1, 100, 64)
    assert need == 4 * (2 * 2 * 100 * 64 + 2 * 1 * 100 * 64 + 2 * 1 * 64 * 128)
    assert L.fa_fwd_fp32_tc_workspace_bytes(1, 2, 1, 0, 64) == 0

    def tc(Q=A, d=64, ws=A, wbytes=need, Hq=2, Hkv=1):
        return L.fa_fwd_fp32_tc(Q, A, A, A, A, 1, Hq, Hkv, 100, d, 1, 0.1, ws, wbytes, None)
    assert tc(Hq=3, Hkv=2) == E.FA_ERR_INVALID_ARG
    assert tc(d=128) == E.FA_ERR_UNSUPPORTED
    assert tc(Q=MIS) == E.FA_ERR_MISALIGNED
    assert tc(wbytes=need - 1) == E.FA_ERR_WORKSPACE


def test_fp32_tensor_core_backward_rejects_invalid_arguments(built_lib):
    L = built_lib.lib()
    E = built_lib
    need = L.fa_bwd_fp32_tc_workspace_bytes(1, 2, 1, 100, 64)
    # hi / lo of Q, dO (2 heads) and K, V (1 head), transposed hi / lo of Q, dO and K over
    # 128 padded columns, and D
    assert need == 4 * (4 * 2 * 100 * 64 + 4 * 1 * 100 * 64 + 4 * 2 * 64 * 128
                        + 2 * 1 * 64 * 128 + 2 * 100)
    assert L.fa_bwd_fp32_tc_workspace_bytes(1, 2, 1, 0, 64) == 0

    def tc(Q=A, dQ=A, d=64, ws=A, wbytes=need, Hq=2, Hkv=1):
        return L.fa_bwd_fp32_tc(Q, A, A, A, A, A, dQ, A, A, 1, Hq, Hkv, 100, d, 1, 0.1, ws, wbytes,
                                None)
    assert tc(Hq=3, Hkv=2) == E.FA_ERR_INVALID_ARG
    assert tc(d=128) == E.FA_ERR_UNSUPPORTED
    assert tc(Q=MIS) == E.FA_ERR_MISALIGNED
    assert tc(dQ=MIS) == E.FA_ERR_MISALIGNED
    assert tc(wbytes=need - 1) == E.FA_ERR_WORKSPACE
    assert tc(ws=MIS) == E.FA_ERR_WORKSPACE


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    """The binding never falls back: a missing library is an error, not a CPU path."""
    from exact_attention_89_gb300 import flashattn
    monkeypatch.setattr(flashattn, "_lib", None)
    monkeypatch.setattr(flashattn, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        flashattn.lib()


def test_product_path_does_not_reference_the_oracle():
    """Nothing in the package or the CUDA sources imports, loads or names the oracle module."""
    pkg = os.path.join(ROOT, "exact_attention_89_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"\bimport\s+oracle\b|\bfrom\s+oracle\b|liboracle", text), fn
