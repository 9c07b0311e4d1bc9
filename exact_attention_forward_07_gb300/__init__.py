"""Exact attention forward for NVIDIA GB300 (sm_103a).

A thin ctypes binding over the C ABI in include/fa.h (libfa_gb300.so, built
in-tree by ``build.py``).  Every step of the computation runs in the CUDA
kernels of that library; this module only checks tensor properties and
passes pointers, sizes and the current CUDA stream.  There is no CPU or
PyTorch fallback: if the library is missing the import of the binding
fails loudly.

    from exact_attention_forward_07_gb300 import forward
    o, lse = forward(q, k, v, causal=True)          # q, k, v: [B,H,N,d] cuda
"""
from __future__ import annotations

import ctypes
import math
import os

__all__ = ["FaError", "fa_fwd_host", "fa_fwd_noalloc", "fa_fwd", "fa_fwd_fp16", "fa_fwd_ex",
           "fa_fwd_variant", "fa_bwd", "fa_bwd_variant", "fa_bwd_workspace_size", "fa_get_status", "fa_strerror",
           "fa_version", "forward", "backward", "library_path", "lib", "variants"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libfa_gb300.so")

FA_OK = 0
FA_ERR_NULL = -1
FA_ERR_SHAPE = -2
FA_ERR_HEADDIM = -3
FA_ERR_UNSUPPORTED_N = -4
FA_ERR_ALIGN = -5
FA_ERR_SCALE = -6
FA_ERR_DEVICE = -7
FA_ERR_CUDA = -8
FA_ERR_TIMEOUT = -9
FA_ERR_ALIAS = -10
FA_ERR_OPTION = -11
FA_ERR_SCRATCH = -12
FA_ERR_WORKSPACE = -13
FA_ERR_INTERNAL = -14
FA_MAX_N = 1 << 20
FA_NOALLOC_SCRATCH_BYTES = 16 << 20
FA_HOST_DEFAULT_CHUNKS = 8
FA_HOST_MAX_CHUNKS = 1024
FA_DEFAULT_RESCALE_THRESHOLD = 8.0
FA_MAX_RESCALE_THRESHOLD = 12.0
FA_ORDER_AUTO = -2

_lib = None


class FaError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = code
        msg = fa_strerror(code)
        if code == FA_ERR_CUDA:
            msg += f" (cudaError {lib().fa_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [{code}]" if where else f"{msg} [{code}]")


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded libfa_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                f"{_LIB_PATH} is missing: build it with "
                "`python -m exact_attention_forward_07_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(_LIB_PATH)
        P, I64 = ctypes.c_void_p, ctypes.c_int64
        for name in ("fa_fwd", "fa_fwd_fp16"):
            fn = getattr(L, name)
            fn.argtypes = [P, P, P, P, P, I64, I64, I64, I64, ctypes.c_int, ctypes.c_float, P]
            fn.restype = ctypes.c_int
        L.fa_fwd_ex.argtypes = [P, P, P, P, P, I64, I64, I64, I64, ctypes.c_int, ctypes.c_float,
                                ctypes.c_int, ctypes.c_float, P]
        L.fa_fwd_ex.restype = ctypes.c_int
        L.fa_fwd_noalloc.argtypes = L.fa_fwd_ex.argtypes
        L.fa_fwd_noalloc.restype = ctypes.c_int
        L.fa_fwd_variant.argtypes = [P, P, P, P, P, I64, I64, I64, I64, ctypes.c_int,
                                     ctypes.c_float, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, P, P]
        L.fa_fwd_variant.restype = ctypes.c_int
        L.fa_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, I64, I64, I64, I64,
                             ctypes.c_int, ctypes.c_float, ctypes.c_int, P]
        L.fa_bwd.restype = ctypes.c_int
        L.fa_bwd_variant.argtypes = [P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, I64, I64, I64,
                                     I64, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                     P]
        L.fa_bwd_variant.restype = ctypes.c_int
        L.fa_bwd_workspace_size.argtypes = [I64, I64, I64, I64, ctypes.POINTER(ctypes.c_size_t)]
        L.fa_bwd_workspace_size.restype = ctypes.c_int
        L.fa_variant_count.argtypes = []
        L.fa_variant_count.restype = ctypes.c_int
        IP = ctypes.POINTER(ctypes.c_int)
        L.fa_variant_info.argtypes = [ctypes.c_int, IP, IP, IP, IP, IP]
        L.fa_variant_info.restype = ctypes.c_int
        L.fa_fwd_host.argtypes = [P, P, P, P, P, I64, I64, I64, I64, ctypes.c_int, ctypes.c_float,
                                  ctypes.c_int, ctypes.c_int]
        L.fa_fwd_host.restype = ctypes.c_int
        L.fa_selftest_wait_timeout.argtypes = [I64, P, P]
        L.fa_selftest_wait_timeout.restype = ctypes.c_int
        L.fa_get_status.argtypes = [P]
        L.fa_get_status.restype = ctypes.c_int
        L.fa_strerror.argtypes = [ctypes.c_int]
        L.fa_strerror.restype = ctypes.c_char_p
        L.fa_last_cuda_error.argtypes = []
        L.fa_last_cuda_error.restype = ctypes.c_int
        L.fa_version.argtypes = []
        L.fa_version.restype = ctypes.c_int
        _lib = L
    return _lib


def fa_strerror(code: int) -> str:
    return lib().fa_strerror(int(code)).decode()


def fa_version() -> int:
    return lib().fa_version()


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(t, name, dtype, shape):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _call(fn_name, q, k, v, o, lse, causal, scale, stream, dtype, extra=()):
    import torch
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _check(t, name, dtype, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rc = getattr(lib(), fn_name)(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), B, H, N, d, int(bool(causal)), float(scale),
                                 *extra, _stream_handle(stream, q.device))
    if rc != FA_OK:
        raise FaError(rc, fn_name)


def fa_fwd(q, k, v, o, lse, causal=False, scale=None, stream=None) -> None:
    """bf16 attention forward into caller-provided o [B,H,N,d] and lse [B,H,N] fp32."""
    import torch
    _call("fa_fwd", q, k, v, o, lse, causal, scale, stream, torch.bfloat16)


def fa_fwd_fp16(q, k, v, o, lse, causal=False, scale=None, stream=None) -> None:
    """fp16 attention forward into caller-provided o and lse."""
    import torch
    _call("fa_fwd_fp16", q, k, v, o, lse, causal, scale, stream, torch.float16)


def fa_fwd_ex(q, k, v, o, lse, causal=False, scale=None, rescale_threshold=None,
              stream=None) -> None:
    """Forward with an explicit online-softmax rescale threshold (log2 units;
    0 = rescale whenever the running max grows).  dtype from q (bf16/fp16)."""
    import torch
    if rescale_threshold is None:
        rescale_threshold = FA_DEFAULT_RESCALE_THRESHOLD
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"unsupported dtype {q.dtype}: use bfloat16 or float16")
    fp16 = int(q.dtype == torch.float16)
    _call("fa_fwd_ex", q, k, v, o, lse, causal, scale, stream, q.dtype,
          extra=(fp16, float(rescale_threshold)))


def fa_fwd_noalloc(q, k, v, o, lse, causal=False, scale=None, rescale_threshold=None,
                   stream=None) -> None:
    """fa_fwd_ex that never allocates device memory (its split scratch is a
    fixed array; FaError FA_ERR_SCRATCH when a call needs more).  Calls must
    not overlap in time."""
    import torch
    if rescale_threshold is None:
        rescale_threshold = FA_DEFAULT_RESCALE_THRESHOLD
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"unsupported dtype {q.dtype}: use bfloat16 or float16")
    fp16 = int(q.dtype == torch.float16)
    _call("fa_fwd_noalloc", q, k, v, o, lse, causal, scale, stream, q.dtype,
          extra=(fp16, float(rescale_threshold)))


def fa_fwd_variant(q, k, v, o, lse, causal=False, scale=None, rescale_threshold=None,
                   stages=0, exp_split=0, causal_order=FA_ORDER_AUTO, stats=None,
                   stream=None) -> None:
    """Forward through one of the library's kernel variants (tuning and
    measurement): `stages` K/V ring slots (0 = default), every
    `exp_split`-th pair of exponentials on the FMA pipes (0 = none), a
    forced causal item order (-1, or g >= 0 tail heads; default: the
    library's choice), and optional rescale counters `stats` (a CUDA int64
    tensor of 4, added to).  dtype from q (bf16/fp16)."""
    import torch
    if rescale_threshold is None:
        rescale_threshold = FA_DEFAULT_RESCALE_THRESHOLD
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"unsupported dtype {q.dtype}: use bfloat16 or float16")
    sp = None
    if stats is not None:
        if not (stats.is_cuda and stats.dtype == torch.int64 and stats.numel() == 4
                and stats.is_contiguous()):
            raise ValueError("stats must be a contiguous CUDA int64 tensor of 4 counters")
        sp = stats.data_ptr()
    fp16 = int(q.dtype == torch.float16)
    _call("fa_fwd_variant", q, k, v, o, lse, causal, scale, stream, q.dtype,
          extra=(fp16, float(rescale_threshold), int(stages), int(exp_split),
                 int(causal_order), sp))


def fa_bwd_workspace_size(B, H, N, d) -> int:
    """Bytes of device workspace fa_bwd needs for [B, H, N, d]."""
    n = ctypes.c_size_t(0)
    rc = lib().fa_bwd_workspace_size(int(B), int(H), int(N), int(d), ctypes.byref(n))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_workspace_size")
    return n.value


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, causal=False, scale=None,
           stream=None, cta_pairs=None) -> None:
    """Attention backward into caller-provided dq, dk, dv [B,H,N,d] (dtype of
    q) from the forward's q, k, v, o, lse and the output gradient dout;
    `workspace` is a CUDA uint8 tensor of at least fa_bwd_workspace_size
    bytes (256-byte aligned, as torch allocates).  cta_pairs = None calls
    fa_bwd (the library's default kernel); 0 or 1 calls fa_bwd_variant with
    that kernel: one CTA per key block, or clusters of two CTAs that halve
    the dQ additions."""
    import torch
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"unsupported dtype {q.dtype}: use bfloat16 or float16")
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout), ("dq", dq),
                    ("dk", dk), ("dv", dv)):
        _check(t, name, q.dtype, (B, H, N, d))
    _check(lse, "lse", torch.float32, (B, H, N))
    if not (isinstance(workspace, torch.Tensor) and workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
            dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
            B, H, N, d, int(bool(causal)), float(scale), int(q.dtype == torch.float16))
    if cta_pairs is None:
        rc = lib().fa_bwd(*args, _stream_handle(stream, q.device))
    else:
        rc = lib().fa_bwd_variant(*args, int(cta_pairs), _stream_handle(stream, q.device))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd" if cta_pairs is None else "fa_bwd_variant")


def backward(q, k, v, o, lse, dout, causal=False, scale=None, stream=None, cta_pairs=None):
    """Allocate dq, dk, dv and the workspace with torch and run the backward;
    returns (dq, dk, dv)."""
    import torch
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa_bwd_workspace_size(*q.shape), dtype=torch.uint8, device=q.device)
    fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, ws, causal, scale, stream, cta_pairs)
    return dq, dk, dv


def variants():
    """The kernel variants built into the library: a list of dicts with d,
    fp16, stages, exp_split and stats."""
    out = []
    L = lib()
    vals = [ctypes.c_int() for _ in range(5)]
    for i in range(L.fa_variant_count()):
        rc = L.fa_variant_info(i, *[ctypes.byref(x) for x in vals])
        if rc != FA_OK:
            raise FaError(rc, "fa_variant_info")
        out.append(dict(zip(("d", "fp16", "stages", "exp_split", "stats"),
                            (x.value for x in vals))))
    return out


def fa_get_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    import torch
    return lib().fa_get_status(_stream_handle(stream, torch.cuda.current_device()))


def forward(q, k, v, causal=False, scale=None, stream=None, rescale_threshold=None):
    """Allocate o and lse with torch and run the forward; returns (o, lse)."""
    import torch
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    if rescale_threshold is not None:
        fa_fwd_ex(q, k, v, o, lse, causal, scale, rescale_threshold, stream)
    elif q.dtype == torch.bfloat16:
        fa_fwd(q, k, v, o, lse, causal, scale, stream)
    elif q.dtype == torch.float16:
        fa_fwd_fp16(q, k, v, o, lse, causal, scale, stream)
    else:
        raise TypeError(f"unsupported dtype {q.dtype}: use bfloat16 or float16")
    return o, lse


def fa_fwd_host(q, k, v, o, lse, causal=False, scale=None, chunks=0) -> None:
    """Forward on HOST tensors through the C ABI (fa_fwd_host): q, k, v, o
    [B,H,N,d] bf16/fp16 and lse [B,H,N] fp32, contiguous CPU tensors
    (pinned for full copy speed).  The library pipelines the copies and the
    kernels over `chunks` groups of heads (0 = its default) and returns when
    o and lse are written."""
    import torch
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"unsupported dtype {q.dtype}: use bfloat16 or float16")
    B, H, N, d = q.shape
    for name, t, dt, shape in (("q", q, q.dtype, (B, H, N, d)), ("k", k, q.dtype, (B, H, N, d)),
                               ("v", v, q.dtype, (B, H, N, d)), ("o", o, q.dtype, (B, H, N, d)),
                               ("lse", lse, torch.float32, (B, H, N))):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.is_cuda:
            raise ValueError(f"{name} must be a host (CPU) tensor")
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}, got {t.dtype}")
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rc = lib().fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           B, H, N, d, int(bool(causal)), float(scale),
                           int(q.dtype == torch.float16), int(chunks))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_host")
