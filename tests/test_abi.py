"""The C-ABI library loads, exports every function include/fa.h declares,
and rejects bad arguments before touching the GPU (no launch, no device
call: runs on a machine without a GPU)."""
import ctypes
import os
import re

import pytest

import exact_attention_forward_07_gb300 as fa
from exact_attention_forward_07_gb300 import build as fa_build

HEADER = os.path.join(fa_build.INCLUDE, "fa.h")


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("fa_fwd", "fa_fwd_fp16", "fa_fwd_ex", "fa_get_status", "fa_strerror",
              "fa_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in fa.h but not exported"


def test_version_and_strerror(lib):
    assert lib.fa_version() == 100
    for code in range(0, -15, -1):
        msg = fa.fa_strerror(code)
        assert msg and msg != "unknown error code"
    assert fa.fa_strerror(-999) == "unknown error code"


# Fake, 16-byte aligned, distinct "device" addresses: argument checks run
# before any CUDA call, so nothing dereferences them.
Q, K, V, O, L = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000


def call(lib, q=Q, k=K, v=V, o=O, lse=L, B=1, H=1, N=128, d=64, causal=0, scale=0.125,
         fp16=False):
    fn = lib.fa_fwd_fp16 if fp16 else lib.fa_fwd
    return fn(q, k, v, o, lse, B, H, N, d, causal, scale, None)


@pytest.mark.parametrize("fp16", [False, True])
def test_argument_errors(lib, fp16):
    c = lambda **kw: call(lib, fp16=fp16, **kw)
    assert c(q=None) == fa.FA_ERR_NULL
    assert c(lse=None) == fa.FA_ERR_NULL
    assert c(B=0) == fa.FA_ERR_SHAPE
    assert c(H=-1) == fa.FA_ERR_SHAPE
    assert c(N=0) == fa.FA_ERR_SHAPE
    assert c(d=96) == fa.FA_ERR_HEADDIM
    assert c(d=256) == fa.FA_ERR_HEADDIM
    assert c(N=fa.FA_MAX_N + 1) == fa.FA_ERR_UNSUPPORTED_N
    assert c(B=1 << 30, H=1 << 30) == fa.FA_ERR_SHAPE
    assert c(q=Q + 8) == fa.FA_ERR_ALIGN
    assert c(o=O + 2) == fa.FA_ERR_ALIGN
    assert c(lse=L + 2) == fa.FA_ERR_ALIGN
    assert c(scale=0.0) == fa.FA_ERR_SCALE
    assert c(scale=-0.5) == fa.FA_ERR_SCALE
    assert c(scale=float("inf")) == fa.FA_ERR_SCALE
    assert c(scale=float("nan")) == fa.FA_ERR_SCALE
    assert c(o=Q) == fa.FA_ERR_ALIAS
    assert c(o=K + 64) == fa.FA_ERR_ALIAS
    assert c(lse=V) == fa.FA_ERR_ALIAS
    assert c(lse=O + 128) == fa.FA_ERR_ALIAS


def test_python_binding_rejects_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q, q, q.clone(), torch.zeros(1, 1, 128))


def test_fa_fwd_ex_option_errors(lib):
    def ex(thr, **kw):
        a = dict(q=Q, k=K, v=V, o=O, lse=L, B=1, H=1, N=128, d=64, causal=0, scale=0.125,
                 fp16=0)
        a.update(kw)
        return lib.fa_fwd_ex(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"],
                             a["d"], a["causal"], a["scale"], a["fp16"], thr, None)
    assert ex(-0.5) == fa.FA_ERR_OPTION
    assert ex(12.5) == fa.FA_ERR_OPTION
    assert ex(float("nan")) == fa.FA_ERR_OPTION
    assert ex(float("inf")) == fa.FA_ERR_OPTION
    assert ex(8.0, q=None) == fa.FA_ERR_NULL
    assert ex(8.0, d=32, fp16=1) == fa.FA_ERR_HEADDIM


def test_fa_fwd_noalloc_argument_errors(lib):
    """The no-alloc entry point checks its arguments like fa_fwd_ex, before
    touching the device."""
    def na(thr=8.0, **kw):
        a = dict(q=Q, k=K, v=V, o=O, lse=L, B=1, H=1, N=128, d=128, causal=0, scale=0.125,
                 fp16=0)
        a.update(kw)
        return lib.fa_fwd_noalloc(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"],
                                  a["N"], a["d"], a["causal"], a["scale"], a["fp16"], thr, None)
    assert na(q=None) == fa.FA_ERR_NULL
    assert na(N=0) == fa.FA_ERR_SHAPE
    assert na(d=96) == fa.FA_ERR_HEADDIM
    assert na(scale=0.0) == fa.FA_ERR_SCALE
    assert na(thr=-1.0) == fa.FA_ERR_OPTION
    assert na(o=Q) == fa.FA_ERR_ALIAS
    assert fa.FA_ERR_SCRATCH == -12 and fa.FA_NOALLOC_SCRATCH_BYTES == 16 << 20
    assert "FA_NOALLOC_SCRATCH_BYTES" in lib.fa_strerror(fa.FA_ERR_SCRATCH).decode()


def test_fa_fwd_host_argument_errors(lib):
    """The host-buffer entry point checks its arguments before touching the
    device (host pointers need no alignment)."""
    def h(chunks=0, **kw):
        a = dict(q=Q, k=K, v=V, o=O, lse=L, B=1, H=1, N=128, d=128, causal=0, scale=0.125,
                 fp16=0)
        a.update(kw)
        return lib.fa_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"],
                               a["d"], a["causal"], a["scale"], a["fp16"], chunks)
    assert h(q=None) == fa.FA_ERR_NULL
    assert h(B=0) == fa.FA_ERR_SHAPE
    assert h(d=32) == fa.FA_ERR_HEADDIM
    assert h(N=fa.FA_MAX_N + 1) == fa.FA_ERR_UNSUPPORTED_N
    assert h(scale=float("nan")) == fa.FA_ERR_SCALE
    assert h(chunks=-1) == fa.FA_ERR_OPTION
    assert h(chunks=fa.FA_HOST_MAX_CHUNKS + 1) == fa.FA_ERR_OPTION
    assert h(o=Q) == fa.FA_ERR_ALIAS


def test_selftest_argument_errors(lib):
    assert lib.fa_selftest_wait_timeout(1000, None, None) == fa.FA_ERR_NULL
    assert lib.fa_selftest_wait_timeout(0, 0x10000000, None) == fa.FA_ERR_OPTION
    assert lib.fa_selftest_wait_timeout(2000000, 0x10000000, None) == fa.FA_ERR_OPTION


def test_fa_fwd_variant_argument_errors(lib):
    """Variants that are not built, and bad arguments, are refused before
    any device call; every built variant is listed with a valid shape."""
    def var(stages=0, exp_split=0, stats=None, order=fa.FA_ORDER_AUTO, **kw):
        a = dict(q=Q, k=K, v=V, o=O, lse=L, B=1, H=1, N=128, d=128, causal=0, scale=0.125,
                 fp16=0, thr=8.0)
        a.update(kw)
        return lib.fa_fwd_variant(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"],
                                  a["N"], a["d"], a["causal"], a["scale"], a["fp16"], a["thr"],
                                  stages, exp_split, order, stats, None)
    assert var(stages=5) == fa.FA_ERR_OPTION        # no room for five 32 KiB slots
    assert var(stages=7, d=64) == fa.FA_ERR_OPTION  # not built
    assert var(exp_split=3) == fa.FA_ERR_OPTION
    assert var(exp_split=4, fp16=1) == fa.FA_ERR_OPTION
    assert var(stages=3, stats=0x10000000) == fa.FA_ERR_OPTION  # no counting build there
    assert var(stats=0x10000004) == fa.FA_ERR_ALIGN
    assert var(d=96) == fa.FA_ERR_HEADDIM
    assert var(stages=3, q=None) == fa.FA_ERR_NULL
    assert var(stages=3, thr=13.0) == fa.FA_ERR_OPTION
    assert var(stages=3, o=Q) == fa.FA_ERR_ALIAS
    assert var(order=-3) == fa.FA_ERR_OPTION
    assert var(order=2, B=1, H=1) == fa.FA_ERR_OPTION  # more tail heads than heads
    vs = fa.variants()
    assert len(vs) == lib.fa_variant_count()
    assert vs[:4] == [dict(d=64, fp16=0, stages=8, exp_split=0, stats=0),
                      dict(d=64, fp16=1, stages=8, exp_split=0, stats=0),
                      dict(d=128, fp16=0, stages=4, exp_split=0, stats=0),
                      dict(d=128, fp16=1, stages=4, exp_split=0, stats=0)]
    for x in vs:
        assert x["d"] in (64, 128) and x["stages"] >= 2 and x["exp_split"] in (0, 2, 4)
        # shared memory: Q tiles + ring within the 227 KiB a CTA may use
        tile = 128 * x["d"] * 2
        assert (2 + x["stages"]) * tile + 9 * 1024 <= 227 * 1024
    i = ctypes.c_int()
    assert lib.fa_variant_info(len(vs), *[ctypes.byref(i)] * 5) == fa.FA_ERR_OPTION


def test_fa_bwd_argument_errors(lib):
    """The backward checks its arguments and workspace before any device
    call; the workspace size follows its documented formula."""
    DO, DQ, DK, DV, WS = 0x60000000, 0x70000000, 0x80000000, 0x90000000, 0xA0000000
    need = fa.fa_bwd_workspace_size(2, 3, 1000, 128)
    assert need == 2 * 3 * 1024 * (4 * 128 + 8)
    assert fa.fa_bwd_workspace_size(1, 1, 1, 64) == 128 * (4 * 64 + 8)

    def bwd(ws_bytes=None, **kw):
        a = dict(q=Q, k=K, v=V, o=O, lse=L, do=DO, dq=DQ, dk=DK, dv=DV, ws=WS, B=2, H=3,
                 N=1000, d=128, causal=0, scale=0.125, fp16=0)
        a.update(kw)
        nb = need if ws_bytes is None else ws_bytes
        return lib.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"],
                          a["dv"], a["ws"], nb, a["B"], a["H"], a["N"], a["d"], a["causal"],
                          a["scale"], a["fp16"], None)
    assert bwd(do=None) == fa.FA_ERR_NULL
    assert bwd(ws=None) == fa.FA_ERR_NULL
    assert bwd(N=0) == fa.FA_ERR_SHAPE
    assert bwd(d=96) == fa.FA_ERR_HEADDIM
    assert bwd(N=fa.FA_MAX_N + 1) == fa.FA_ERR_UNSUPPORTED_N
    assert bwd(B=256, H=256, N=128) == fa.FA_ERR_SHAPE  # more than 65535 heads
    assert bwd(dq=DQ + 8) == fa.FA_ERR_ALIGN
    assert bwd(ws=WS + 128) == fa.FA_ERR_ALIGN
    assert bwd(scale=0.0) == fa.FA_ERR_SCALE
    assert bwd(ws_bytes=need - 1) == fa.FA_ERR_WORKSPACE
    assert bwd(dq=Q) == fa.FA_ERR_ALIAS
    assert bwd(dv=DK) == fa.FA_ERR_ALIAS
    assert bwd(ws=DO) == fa.FA_ERR_ALIAS
    assert bwd(dk=WS + 4096) == fa.FA_ERR_ALIAS
    assert bwd(lse=DV + 64) == fa.FA_ERR_ALIAS
    # fa_bwd_variant: the same checks, and only cta_pairs 0 or 1

    def bwdv(pairs, **kw):
        a = dict(q=Q, k=K, v=V, o=O, lse=L, do=DO, dq=DQ, dk=DK, dv=DV, ws=WS, B=2, H=3,
                 N=1000, d=128, causal=0, scale=0.125, fp16=0)
        a.update(kw)
        return lib.fa_bwd_variant(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"],
                                  a["dk"], a["dv"], a["ws"], need, a["B"], a["H"], a["N"], a["d"],
                                  a["causal"], a["scale"], a["fp16"], pairs, None)
    for bad in (-1, 2, 7):
        assert bwdv(bad) == fa.FA_ERR_OPTION
    for pairs in (0, 1):
        assert bwdv(pairs, do=None) == fa.FA_ERR_NULL
        assert bwdv(pairs, d=96) == fa.FA_ERR_HEADDIM
        assert bwdv(pairs, dq=DQ + 8) == fa.FA_ERR_ALIGN
        assert bwdv(pairs, dv=DK) == fa.FA_ERR_ALIAS
    n = ctypes.c_size_t()
    assert lib.fa_bwd_workspace_size(1, 1, 128, 64, None) == fa.FA_ERR_NULL
    assert lib.fa_bwd_workspace_size(1, 1, 128, 32, ctypes.byref(n)) == fa.FA_ERR_HEADDIM
