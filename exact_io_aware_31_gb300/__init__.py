"""Exact fused attention for NVIDIA GB300 (sm_103a): Python binding of ``libfa.so``.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/fa.h``.  PyTorch supplies
device memory and streams.  There is no fallback: if the library is missing
or the device is not sm_103, calls raise.

Raw entry points (same names and argument order as the C ABI, pointers as
ints):  ``fa_fwd``, ``fa_fwd_fp8``, ``fa_bwd``, ``fa_bwd_workspace_size``, the three phases
of ``fa_bwd`` (``fa_bwd_preprocess``, ``fa_bwd_dkdv``, ``fa_bwd_dq_convert``),
the split-KV decode forward (``fa_fwd_splitkv``,
``fa_fwd_splitkv_workspace_size``), ``fa_get_device_status``,
``fa_status_string``.
Tensor helpers: :func:`forward`, :func:`forward_fp8`, :func:`backward`, :func:`decode_forward`.
"""

from __future__ import annotations

import ctypes
import os

__all__ = [
    "LIB_PATH", "FaError", "load_library", "fa_fwd", "fa_fwd_fp8", "forward_fp8", "fa_bwd", "fa_bwd_workspace_size", "fa_bwd_deterministic",
    "fa_fwd_dropout", "fa_bwd_dropout",
    "fa_bwd_preprocess", "fa_bwd_dkdv", "fa_bwd_dq_convert", "fa_bwd_noalloc", "NOALLOC_SCRATCH_BYTES",
    "fa_fwd_splitkv", "fa_fwd_splitkv_workspace_size", "decode_forward",
    "fa_get_device_status", "fa_status_string", "forward", "backward", "EXPORTED_SYMBOLS",
    "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_WORKSPACE", "FA_ERR_CUDA",
    "FA_ERR_DEVICE_TIMEOUT", "FA_ERR_INTERNAL",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_WORKSPACE = 3
FA_ERR_CUDA = 4
FA_ERR_DEVICE_TIMEOUT = 5
FA_ERR_INTERNAL = 6

EXPORTED_SYMBOLS = ("fa_fwd", "fa_fwd_fp8", "fa_bwd", "fa_bwd_workspace_size", "fa_bwd_deterministic", "fa_fwd_dropout",
                    "fa_bwd_dropout", "fa_bwd_preprocess",
                    "fa_bwd_dkdv",
                    "fa_bwd_dq_convert", "fa_bwd_noalloc", "fa_fwd_splitkv", "fa_fwd_splitkv_workspace_size",
                    "fa_get_device_status", "fa_status_string")

# Size of the library-owned scratch behind fa_bwd_noalloc (FA_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 64 << 20

_lib = None


class FaError(RuntimeError):
    """A non-zero status from the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fa_status_string(status)} (status {status})")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libfa.so (once) and declare its signatures.  Raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m exact_io_aware_31_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.restype = i
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.fa_fwd_fp8.restype = i
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, f, f, i, vp]
    lib.fa_bwd_workspace_size.restype = sz
    lib.fa_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.fa_bwd.restype = i
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, sz, vp]
    u64, u32 = ctypes.c_ulonglong, ctypes.c_uint
    lib.fa_fwd_dropout.restype = i
    lib.fa_fwd_dropout.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, f, u64, u32, vp]
    lib.fa_bwd_dropout.restype = i
    lib.fa_bwd_dropout.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, f, u64, u32, vp, sz, vp]
    lib.fa_bwd_deterministic.restype = i
    lib.fa_bwd_deterministic.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, sz, vp]
    lib.fa_bwd_preprocess.restype = i
    lib.fa_bwd_preprocess.argtypes = [vp, vp, vp, i, i, i, i, vp, sz, vp]
    lib.fa_bwd_dkdv.restype = i
    lib.fa_bwd_dkdv.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, sz, vp]
    lib.fa_bwd_dq_convert.restype = i
    lib.fa_bwd_dq_convert.argtypes = [vp, i, i, i, i, f, vp, sz, vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.fa_fwd_splitkv.restype = i
    lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz, vp]
    lib.fa_fwd_splitkv_workspace_size.restype = sz
    lib.fa_fwd_splitkv_workspace_size.argtypes = [i, i, i, i, i, i]
    lib.fa_get_device_status.restype = i
    lib.fa_get_device_status.argtypes = [vp]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_status_string.argtypes = [i]
    _lib = lib
    return lib


# ------------------------------------------------------------- raw C ABI ----
def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream) -> int:
    return load_library().fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream)


def fa_fwd_fp8(q8, k8, v, o, lse, B, H, N, d, scale, q_descale, k_descale, causal, stream) -> int:
    return load_library().fa_fwd_fp8(q8, k8, v, o, lse, B, H, N, d, scale, q_descale, k_descale, causal, stream)


def fa_bwd_workspace_size(B, H, N, d) -> int:
    return load_library().fa_bwd_workspace_size(B, H, N, d)


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, workspace, workspace_bytes,
           stream) -> int:
    return load_library().fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, workspace,
                                 workspace_bytes, stream)


def fa_fwd_dropout(q, k, v, o, lse, B, H, N, d, scale, causal, p_drop, seed, offset, stream) -> int:
    return load_library().fa_fwd_dropout(q, k, v, o, lse, B, H, N, d, scale, causal, p_drop, seed, offset, stream)


def fa_bwd_dropout(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, p_drop, seed, offset, workspace,
                   workspace_bytes, stream) -> int:
    return load_library().fa_bwd_dropout(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, p_drop, seed,
                                         offset, workspace, workspace_bytes, stream)


def fa_bwd_deterministic(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, workspace, workspace_bytes,
                         stream) -> int:
    return load_library().fa_bwd_deterministic(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal,
                                               workspace, workspace_bytes, stream)


def fa_bwd_preprocess(o, dout, lse, B, H, N, d, workspace, workspace_bytes, stream) -> int:
    return load_library().fa_bwd_preprocess(o, dout, lse, B, H, N, d, workspace, workspace_bytes, stream)


def fa_bwd_dkdv(q, k, v, dout, dk, dv, B, H, N, d, scale, causal, workspace, workspace_bytes, stream) -> int:
    return load_library().fa_bwd_dkdv(q, k, v, dout, dk, dv, B, H, N, d, scale, causal, workspace,
                                      workspace_bytes, stream)


def fa_bwd_dq_convert(dq, B, H, N, d, scale, workspace, workspace_bytes, stream) -> int:
    return load_library().fa_bwd_dq_convert(dq, B, H, N, d, scale, workspace, workspace_bytes, stream)


def fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, stream) -> int:
    """fa_bwd with the library's own scratch instead of a workspace (for callers that cannot allocate)."""
    return load_library().fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, stream)


def fa_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, num_splits, workspace, workspace_bytes,
                   stream) -> int:
    return load_library().fa_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, num_splits, workspace,
                                         workspace_bytes, stream)


def fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, num_splits) -> int:
    return load_library().fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, num_splits)


def fa_get_device_status(stream) -> int:
    return load_library().fa_get_device_status(stream)


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(status).decode()


# --------------------------------------------------------- tensor helpers ----
def _check(t, name, shape, dtype):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous {dtype} of shape {tuple(shape)}, got "
                         f"{t.dtype} {tuple(t.shape)} contiguous={t.is_contiguous()}")


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def forward(q, k, v, scale=None, causal=False, out=None, lse=None, stream=None):
    """Exact attention forward on [B, H, N, d] bf16 CUDA tensors; returns ``(o, lse)``."""
    import torch
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, (B, H, N, d), torch.bfloat16)
    if scale is None:
        scale = d ** -0.5
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(o, "out", (B, H, N, d), torch.bfloat16)
    _check(l, "lse", (B, H, N), torch.float32)
    st = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), B, H, N, d,
                float(scale), int(bool(causal)), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd")
    return o, l


def forward_fp8(q8, k8, v, q_descale=1.0, k_descale=1.0, scale=None, causal=False, out=None, lse=None,
                stream=None):
    """Forward with E4M3 queries and keys (``torch.float8_e4m3fn`` or their ``uint8`` codes,
    [B, H, N, 128]) and bf16 values; returns ``(o, lse)``."""
    import torch
    B, H, N, d = q8.shape
    for name, t in (("q8", q8), ("k8", k8)):
        want = t.dtype if t.dtype in (torch.uint8, torch.float8_e4m3fn) else torch.float8_e4m3fn
        _check(t, name, (B, H, N, d), want)
    _check(v, "v", (B, H, N, d), torch.bfloat16)
    if scale is None:
        scale = d ** -0.5
    o = torch.empty_like(v) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=v.device) if lse is None else lse
    _check(o, "out", (B, H, N, d), torch.bfloat16)
    _check(l, "lse", (B, H, N), torch.float32)
    st = fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), B, H, N, d,
                    float(scale), float(q_descale), float(k_descale), int(bool(causal)), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_fp8")
    return o, l


def backward(q, k, v, o, lse, dout, scale=None, causal=False, workspace=None, grads=None, stream=None,
             deterministic=False):
    """Gradients ``(dq, dk, dv)`` of ``sum(O * dout)``; ``o`` and ``lse`` from :func:`forward`.

    ``deterministic=True`` uses ``fa_bwd_deterministic`` (bitwise reproducible, slower)."""
    import torch
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check(t, name, (B, H, N, d), torch.bfloat16)
    _check(lse, "lse", (B, H, N), torch.float32)
    if scale is None:
        scale = d ** -0.5
    need = fa_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if grads is None:
        grads = tuple(torch.empty_like(q) for _ in range(3))
    dq, dk, dv = grads
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check(t, name, (B, H, N, d), torch.bfloat16)
    fn = fa_bwd_deterministic if deterministic else fa_bwd
    st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, float(scale), int(bool(causal)),
            workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_bwd_deterministic" if deterministic else "fa_bwd")
    return dq, dk, dv


def decode_forward(q, k, v, scale=None, causal=True, num_splits=0, out=None, lse=None, workspace=None,
                   stream=None):
    """Split-KV attention of ``q [B, H, Nq, d]`` (Nq <= 8, the last Nq positions) against the cache
    ``k, v [B, H, Nk, d]`` (bf16 CUDA tensors); returns ``(o, lse)``."""
    import torch
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    _check(q, "q", (B, H, Nq, d), torch.bfloat16)
    for name, t in (("k", k), ("v", v)):
        _check(t, name, (B, H, Nk, d), torch.bfloat16)
    if scale is None:
        scale = d ** -0.5
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(o, "out", (B, H, Nq, d), torch.bfloat16)
    _check(l, "lse", (B, H, Nq), torch.float32)
    need = fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wptr = workspace.data_ptr() if workspace is not None else None
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), B, H, Nq, Nk, d,
                        float(scale), int(bool(causal)), int(num_splits), wptr, wbytes, _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_splitkv")
    return o, l
