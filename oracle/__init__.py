"""CPU oracle for the exact attention forward and its gradients (fp64).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers; the product library
never imports, links or runs anything here, and nothing here imports the
product package.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, three-pass safe
softmax written out from the definition of attention) and
``attn_bwd_oracle.c`` (the chain rule of that definition: the gradients of
sum(dO * O) with respect to Q, K and V).  This module only builds those
files with gcc, marshals numpy arrays into them and back, and offers the
probability matrix for small shapes.

Definition followed (see the C file for the passage each step comes from):
    s_ij = scale * <q_i, k_j>,  j in A(i)   (A(i) = all keys, or j <= i if causal)
    o_i  = sum_j softmax_j(s_i.) v_j,       lse_i = ln sum_{j in A(i)} exp(s_ij)

Every part of it is pinned against closed forms, invariants, a
brute-force decimal-arithmetic recompute, a library softmax
(tests/test_oracle.py) and, for the gradients, central finite differences
of the forward oracle and library autograd (tests/test_oracle_bwd.py); no
function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_SRC_BWD = os.path.join(_HERE, "attn_bwd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so (gcc, IEEE fp64, no fast-math)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                                  os.path.getmtime(_SRC_BWD)))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c99", "-fno-fast-math",
               "-ffp-contract=off", "-o", tmp, _SRC, _SRC_BWD, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    """Bind the oracle functions a build exports (a build of one source
    file, as the mutation tests make, exports only its own)."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    if hasattr(lib, "oracle_attn_fwd_rows"):
        lib.oracle_attn_fwd_rows.argtypes = [P, P, P, I64, I64, I64, I64, ctypes.c_int,
                                             ctypes.c_double, P, I64, P, P, ctypes.c_int]
        lib.oracle_attn_fwd_rows.restype = ctypes.c_int
        lib.oracle_attn_probs.argtypes = [P, P, I64, I64, I64, I64, ctypes.c_int,
                                          ctypes.c_double, P]
        lib.oracle_attn_probs.restype = ctypes.c_int
    if hasattr(lib, "oracle_attn_bwd"):
        lib.oracle_attn_bwd.argtypes = [P, P, P, P, I64, I64, I64, I64, ctypes.c_int,
                                        ctypes.c_double, P, P, P, ctypes.c_int]
        lib.oracle_attn_bwd.restype = ctypes.c_int
        lib.oracle_attn_bwd_dq_rows.argtypes = [P, P, P, P, I64, I64, I64, I64, ctypes.c_int,
                                                ctypes.c_double, P, I64, P, ctypes.c_int]
        lib.oracle_attn_bwd_dq_rows.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _as_f64(x) -> np.ndarray:
    """Accept numpy arrays or CPU torch tensors (any float dtype); the
    upcast of bf16/fp16 values to fp64 is exact."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def attn_fwd(q, k, v, causal: bool, scale: float, rows=None, nthreads: int | None = None,
             lib=None):
    """O and LSE of attention on [B, H, N, d] inputs.

    rows: optional 1-D array of flat row ids (b*H + h)*N + i.  When given,
    returns (o [len(rows), d], lse [len(rows)]); otherwise the full
    (o [B,H,N,d], lse [B,H,N]).  `lib` selects another build of the same C
    source (the mutation tests use it); default is liboracle.so.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    if rows is None:
        nrows = B * H * N
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
        nrows = rows_arr.size
    o = np.empty((nrows, d), dtype=np.float64)
    lse = np.empty((nrows,), dtype=np.float64)
    lib = lib or _load()
    rc = lib.oracle_attn_fwd_rows(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, B, H, N, d, int(bool(causal)),
        float(scale), None if rows_arr is None else rows_arr.ctypes.data, nrows,
        o.ctypes.data, lse.ctypes.data, int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd_rows failed with code {rc}")
    if rows is None:
        return o.reshape(B, H, N, d), lse.reshape(B, H, N)
    return o, lse


def attn_bwd(q, k, v, dout, causal: bool, scale: float, nthreads: int | None = None,
             lib=None):
    """Gradients (dq, dk, dv), each [B, H, N, d] fp64, of sum(dout * O) for
    the attention forward O(q, k, v) on [B, H, N, d] inputs."""
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    if q.ndim != 4 or any(x.shape != q.shape for x in (k, v, dout)):
        raise ValueError("q, k, v, dout must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    dq, dk, dv = (np.empty_like(q) for _ in range(3))
    rc = (lib or _load()).oracle_attn_bwd(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, B, H, N, d,
        int(bool(causal)), float(scale), dq.ctypes.data, dk.ctypes.data, dv.ctypes.data,
        int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd failed with code {rc}")
    return dq, dk, dv


def attn_bwd_dq_rows(q, k, v, dout, causal: bool, scale: float, rows,
                     nthreads: int | None = None, lib=None):
    """dQ [len(rows), d] fp64 of sum(dout * O) for the listed flat query rows
    (b*H + h)*N + i: each needs only its own row of probabilities."""
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    if q.ndim != 4 or any(x.shape != q.shape for x in (k, v, dout)):
        raise ValueError("q, k, v, dout must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    rows_arr = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
    dq = np.empty((rows_arr.size, d), dtype=np.float64)
    rc = (lib or _load()).oracle_attn_bwd_dq_rows(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, B, H, N, d,
        int(bool(causal)), float(scale), rows_arr.ctypes.data, rows_arr.size, dq.ctypes.data,
        int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd_dq_rows failed with code {rc}")
    return dq


def attn_probs(q, k, causal: bool, scale: float, lib=None) -> np.ndarray:
    """The probability matrix P [B, H, N, N] for small shapes."""
    q, k = _as_f64(q), _as_f64(k)
    B, H, N, d = q.shape
    if B * H * N * N > 1 << 24:
        raise ValueError("attn_probs is meant for small shapes only")
    p = np.empty((B, H, N, N), dtype=np.float64)
    rc = (lib or _load()).oracle_attn_probs(q.ctypes.data, k.ctypes.data, B, H, N, d,
                                   int(bool(causal)), float(scale), p.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle_attn_probs failed with code {rc}")
    return p


def load_library(path: str):
    """Bind another build of attn_oracle.c (used by the mutation tests)."""
    return _bind(path)
