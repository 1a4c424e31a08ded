"""GB300 (sm_103a) tiled exact attention, forward and backward.

Thin Python binding of the C ABI in ``include/fa.h``: every function here
only marshals arguments (tensors become device pointers, the current torch
stream becomes the CUDA stream) and calls the shared library built by
``build.py``; all computation runs in the library's CUDA kernels.  PyTorch is
used for device memory and streams only.  There is no CPU fallback: if the
library is missing, or no CUDA device is present, the calls raise.

Layouts (see ``include/fa.h``): q, o, dout, dq ``[T, Hq, d]``; k, v, dk, dv
``[T, Hkv, d]``; lse, D ``[Hq, T]`` fp32.  A dense batch of B sequences of
length N is ``T = B*N`` (pass ``cu_seqlens=None``); a packed variable-length
batch passes ``cu_seqlens`` (int32 ``[B+1]`` on the device) and the maximum
length N.  Queries and keys may differ in length (``k.shape[0] != q.shape[0]``
for a dense batch, or ``cu_seqlens_k`` / ``max_seqlen_k`` for a packed one):
the calls then go to the ``*_kv`` entry points, whose causal mask takes the
queries to be the last positions of the key sequence.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

__all__ = [
    "FAError", "lib", "fa_fwd", "fa_bwd_preprocess", "fa_bwd", "fa_fwd_workspace_size",
    "fa_bwd_workspace_size", "fa_bwd_workspace_semaphore_offset", "fa_check_device_status",
    "fa_bwd_noalloc", "fa_noalloc_check_device_status", "fa_fwd_kv", "fa_bwd_kv_workspace_size", "fa_bwd_kv_preprocess", "fa_bwd_kv",
    "fa_status_string", "forward", "backward", "attention", "FA_OK", "FA_ERR_INVALID_ARG",
    "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA", "FA_ERR_TIMEOUT", "FA_BF16", "FA_FP32",
]

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = 0, 1, 2, 3, 4
FA_BF16, FA_FP32 = 0, 1

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t
_f = ctypes.c_float

_SIGS = {
    "fa_status_string": (ctypes.c_char_p, [_i]),
    "fa_version": (ctypes.c_char_p, []),
    "fa_fwd_workspace_size": (_sz, [_i, _i, _i, _i]),
    "fa_fwd": (_i, [_vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _vp, _sz,
                    _vp]),
    "fa_bwd_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i]),
    "fa_bwd_workspace_semaphore_offset": (_sz, [_i, _i, _i, _i, _i, _i]),
    "fa_bwd_preprocess": (_i, [_vp, _i, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _i, _i, _i, _vp, _i,
                               _vp]),
    "fa_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _sz, _i, _i, _i, _i, _i,
                    _i, _f, _i, _vp, _i, _vp]),
    "fa_check_device_status": (_i, [_vp, _vp]),
    "fa_noalloc_check_device_status": (_i, [_vp]),
    "fa_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                            _i, _i, _f, _i, _vp, _i, _vp]),
    "fa_fwd_kv": (_i, [_vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp,
                       _vp, _vp, _sz, _vp]),
    "fa_bwd_kv_workspace_size": (_sz, [_i] * 8),
    "fa_bwd_kv_preprocess": (_i, [_vp, _i, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _i, _i, _i, _i,
                                  _i, _vp, _vp, _i, _vp]),
    "fa_bwd_kv": (_i, [_vp] * 9 + [_i, _vp, _sz, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp,
                                   _vp, _i, _vp]),
}

EXPORTED = tuple(_SIGS)


class FAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = int(status)
        super().__init__(f"{what}: {fa_status_string(status)}")


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is missing; build it with "
                    "`python -m bwd_tiled_attention_gb300.build`")
            L = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr() if x.numel() > 0 else None
    return int(x)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dt(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    if dtype == torch.float32:
        return FA_FP32
    if dtype == torch.bfloat16:
        return FA_BF16
    raise ValueError(f"unsupported dtype {dtype}")


# ----------------------------------------------------------------------------- raw C ABI


def fa_status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


def fa_fwd_workspace_size(B, Hq, N, total_tokens) -> int:
    return int(lib().fa_fwd_workspace_size(B, Hq, N, total_tokens))


def fa_bwd_workspace_size(B, Hq, Hkv, N, total_tokens, d) -> int:
    return int(lib().fa_bwd_workspace_size(B, Hq, Hkv, N, total_tokens, d))


def fa_bwd_workspace_semaphore_offset(B, Hq, Hkv, N, total_tokens, d) -> int:
    return int(lib().fa_bwd_workspace_semaphore_offset(B, Hq, Hkv, N, total_tokens, d))


def fa_fwd(q, k, v, o, o_dtype, lse, B, Hq, Hkv, N, total_tokens, d, scale, causal, cu_seqlens,
           workspace, workspace_bytes, stream=None) -> int:
    return int(lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _dt(o_dtype), _ptr(lse), B, Hq,
                            Hkv, N, total_tokens, d, float(scale), int(bool(causal)),
                            _ptr(cu_seqlens), _ptr(workspace), int(workspace_bytes),
                            _stream(stream)))


def fa_bwd_preprocess(o, o_dtype, dout, D, workspace, workspace_bytes, B, Hq, Hkv, N,
                      total_tokens, d, causal, cu_seqlens, deterministic, stream=None) -> int:
    return int(lib().fa_bwd_preprocess(_ptr(o), _dt(o_dtype), _ptr(dout), _ptr(D),
                                       _ptr(workspace), int(workspace_bytes), B, Hq, Hkv, N,
                                       total_tokens, d, int(bool(causal)), _ptr(cu_seqlens),
                                       int(bool(deterministic)), _stream(stream)))


def fa_bwd(q, k, v, dout, lse, D, dq, dk, dv, grad_dtype, workspace, workspace_bytes, B, Hq, Hkv,
           N, total_tokens, d, scale, causal, cu_seqlens, deterministic, stream=None) -> int:
    return int(lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse), _ptr(D), _ptr(dq),
                            _ptr(dk), _ptr(dv), _dt(grad_dtype), _ptr(workspace),
                            int(workspace_bytes), B, Hq, Hkv, N, total_tokens, d, float(scale),
                            int(bool(causal)), _ptr(cu_seqlens), int(bool(deterministic)),
                            _stream(stream)))


def fa_bwd_noalloc(q, k, v, o, o_dtype, dout, lse, dq, dk, dv, grad_dtype, B, Hq, Hkv, N,
                   total_tokens, d, scale, causal, cu_seqlens, deterministic, stream=None) -> int:
    """Backward without a caller workspace (library-owned 64 MiB scratch); see include/fa.h."""
    return int(lib().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _dt(o_dtype), _ptr(dout),
                                    _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _dt(grad_dtype), B,
                                    Hq, Hkv, N, total_tokens, d, float(scale), int(bool(causal)),
                                    _ptr(cu_seqlens), int(bool(deterministic)), _stream(stream)))


def fa_fwd_kv(q, k, v, o, o_dtype, lse, B, Hq, Hkv, Nq, total_q, Nk, total_k, d, scale, causal,
              cu_seqlens_q, cu_seqlens_k, workspace, workspace_bytes, stream=None) -> int:
    return int(lib().fa_fwd_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _dt(o_dtype), _ptr(lse), B,
                               Hq, Hkv, Nq, total_q, Nk, total_k, d, float(scale),
                               int(bool(causal)), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                               _ptr(workspace), int(workspace_bytes), _stream(stream)))


def fa_bwd_kv_workspace_size(B, Hq, Hkv, Nq, total_q, Nk, total_k, d) -> int:
    return int(lib().fa_bwd_kv_workspace_size(B, Hq, Hkv, Nq, total_q, Nk, total_k, d))


def fa_bwd_kv_preprocess(o, o_dtype, dout, D, workspace, workspace_bytes, B, Hq, Hkv, Nq,
                         total_q, Nk, total_k, d, causal, cu_seqlens_q, cu_seqlens_k,
                         deterministic, stream=None) -> int:
    return int(lib().fa_bwd_kv_preprocess(_ptr(o), _dt(o_dtype), _ptr(dout), _ptr(D),
                                          _ptr(workspace), int(workspace_bytes), B, Hq, Hkv, Nq,
                                          total_q, Nk, total_k, d, int(bool(causal)),
                                          _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                          int(bool(deterministic)), _stream(stream)))


def fa_bwd_kv(q, k, v, dout, lse, D, dq, dk, dv, grad_dtype, workspace, workspace_bytes, B, Hq,
              Hkv, Nq, total_q, Nk, total_k, d, scale, causal, cu_seqlens_q, cu_seqlens_k,
              deterministic, stream=None) -> int:
    return int(lib().fa_bwd_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse), _ptr(D),
                               _ptr(dq), _ptr(dk), _ptr(dv), _dt(grad_dtype), _ptr(workspace),
                               int(workspace_bytes), B, Hq, Hkv, Nq, total_q, Nk, total_k, d,
                               float(scale), int(bool(causal)), _ptr(cu_seqlens_q),
                               _ptr(cu_seqlens_k), int(bool(deterministic)), _stream(stream)))


def fa_check_device_status(workspace, stream=None) -> int:
    return int(lib().fa_check_device_status(_ptr(workspace), _stream(stream)))


def fa_noalloc_check_device_status(stream=None) -> int:
    """Device status of the last fa_bwd_noalloc call on the current device (synchronises)."""
    return int(lib().fa_noalloc_check_device_status(_stream(stream)))


# ----------------------------------------------------------------------------- tensor API


def _check(status, what):
    if status != FA_OK:
        raise FAError(status, what)


def _geometry(q, k, cu_seqlens, max_seqlen, batch):
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if cu_seqlens is None:
        if batch is None:
            raise ValueError("dense inputs need batch (B); T = B * N")
        B = int(batch)
        N = T // B if B > 0 else 0
        if B * N != T:
            raise ValueError("T must equal B * N for a dense batch")
    else:
        B = cu_seqlens.numel() - 1
        if max_seqlen is None:
            raise ValueError("variable-length inputs need max_seqlen")
        N = int(max_seqlen)
    return B, Hq, Hkv, N, T, d


def _check_tensor(name, t, dtypes, ndim):
    """The tensor API passes raw device pointers: every tensor must be a
    contiguous tensor of the expected dtype and rank (and, checked last by
    _check_inputs, on a CUDA device)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must be {' or '.join(str(x) for x in dtypes)}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_inputs(q, k, v, cu_seqlens, cu_seqlens_k, dout=None, o=None, lse=None):
    bf16 = (torch.bfloat16,)
    _check_tensor("q", q, bf16, 3)
    _check_tensor("k", k, bf16, 3)
    _check_tensor("v", v, bf16, 3)
    if k.shape != v.shape:
        raise ValueError(f"k {tuple(k.shape)} and v {tuple(v.shape)} differ in shape")
    if k.shape[2] != q.shape[2]:
        raise ValueError("q and k differ in head dimension")
    if q.shape[1] % k.shape[1] != 0:
        raise ValueError("the query heads must be a multiple of the key/value heads")
    for name, t in (("cu_seqlens", cu_seqlens), ("cu_seqlens_k", cu_seqlens_k)):
        if t is not None:
            _check_tensor(name, t, (torch.int32,), 1)
    if dout is not None:
        _check_tensor("dout", dout, bf16, 3)
        if dout.shape != q.shape:
            raise ValueError("dout must have the shape of q")
    if o is not None:
        _check_tensor("o", o, (torch.bfloat16, torch.float32), 3)
        if o.shape != q.shape:
            raise ValueError("o must have the shape of q")
    if lse is not None:
        _check_tensor("lse", lse, (torch.float32,), 2)
        if tuple(lse.shape) != (q.shape[1], q.shape[0]):
            raise ValueError("lse must be [Hq, Tq]")
    for name, t in (("q", q), ("k", k), ("v", v), ("cu_seqlens", cu_seqlens),
                    ("cu_seqlens_k", cu_seqlens_k), ("dout", dout), ("o", o), ("lse", lse)):
        if t is not None and not t.is_cuda:
            raise ValueError(f"{name} must be on a CUDA device")


def _geometry_kv(q, k, cu_seqlens, max_seqlen, cu_seqlens_k, max_seqlen_k, batch):
    """(B, Hq, Hkv, Nq, Tq, Nk, Tk, d, kv): kv is True when queries and keys
    have separate lengths (the *_kv entry points)."""
    B, Hq, Hkv, Nq, Tq, d = _geometry(q, k, cu_seqlens, max_seqlen, batch)
    Tk = k.shape[0]
    if cu_seqlens is None:
        if cu_seqlens_k is not None:
            raise ValueError("cu_seqlens_k needs cu_seqlens")
        Nk = Tk // B if B > 0 else 0
        if B * Nk != Tk:
            raise ValueError("Tk must equal B * Nk for a dense batch")
        return B, Hq, Hkv, Nq, Tq, Nk, Tk, d, Tk != Tq
    if cu_seqlens_k is None:
        if Tk != Tq:
            raise ValueError("keys of another length need cu_seqlens_k")
        return B, Hq, Hkv, Nq, Tq, Nq, Tk, d, False
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens and cu_seqlens_k name different batch sizes")
    if max_seqlen_k is None:
        raise ValueError("cu_seqlens_k needs max_seqlen_k")
    return B, Hq, Hkv, Nq, Tq, int(max_seqlen_k), Tk, d, True


def forward(q, k, v, causal=False, scale=None, cu_seqlens=None, max_seqlen=None, batch=None,
            out_dtype=torch.bfloat16, stream=None, workspace=None, cu_seqlens_k=None,
            max_seqlen_k=None):
    """Attention forward through the C ABI; returns (o, lse)."""
    _check_inputs(q, k, v, cu_seqlens, cu_seqlens_k)
    B, Hq, Hkv, Nq, Tq, Nk, Tk, d, kv = _geometry_kv(q, k, cu_seqlens, max_seqlen, cu_seqlens_k,
                                                     max_seqlen_k, batch)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty((Tq, Hq, d), dtype=out_dtype, device=q.device)
    lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
    ws_bytes = fa_fwd_workspace_size(B, Hq, Nq, Tq)
    ws = workspace if workspace is not None else torch.empty(
        max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    if kv:
        _check(fa_fwd_kv(q, k, v, o, out_dtype, lse, B, Hq, Hkv, Nq, Tq, Nk, Tk, d, scale, causal,
                         cu_seqlens, cu_seqlens_k, ws, ws_bytes, stream), "fa_fwd_kv")
    else:
        _check(fa_fwd(q, k, v, o, out_dtype, lse, B, Hq, Hkv, Nq, Tq, d, scale, causal,
                      cu_seqlens, ws, ws_bytes, stream), "fa_fwd")
    return o, lse


def backward(q, k, v, o, dout, lse, causal=False, scale=None, cu_seqlens=None, max_seqlen=None,
             batch=None, deterministic=False, grad_dtype=torch.bfloat16, stream=None,
             workspace=None, check_status=False, cu_seqlens_k=None, max_seqlen_k=None):
    """Attention backward (preprocess + backward) through the C ABI; returns (dq, dk, dv)."""
    _check_inputs(q, k, v, cu_seqlens, cu_seqlens_k, dout=dout, o=o, lse=lse)
    B, Hq, Hkv, Nq, Tq, Nk, Tk, d, kv = _geometry_kv(q, k, cu_seqlens, max_seqlen, cu_seqlens_k,
                                                     max_seqlen_k, batch)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty((Tq, Hq, d), dtype=grad_dtype, device=q.device)
    dk = torch.empty((Tk, Hkv, d), dtype=grad_dtype, device=q.device)
    dv = torch.empty((Tk, Hkv, d), dtype=grad_dtype, device=q.device)
    D = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
    if kv:
        ws_bytes = fa_bwd_kv_workspace_size(B, Hq, Hkv, Nq, Tq, Nk, Tk, d)
    else:
        ws_bytes = fa_bwd_workspace_size(B, Hq, Hkv, Nq, Tq, d)
    ws = workspace if workspace is not None else torch.empty(
        max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    if kv:
        _check(fa_bwd_kv_preprocess(o, o.dtype, dout, D, ws, ws_bytes, B, Hq, Hkv, Nq, Tq, Nk, Tk,
                                    d, causal, cu_seqlens, cu_seqlens_k, deterministic, stream),
               "fa_bwd_kv_preprocess")
        _check(fa_bwd_kv(q, k, v, dout, lse, D, dq, dk, dv, grad_dtype, ws, ws_bytes, B, Hq, Hkv,
                         Nq, Tq, Nk, Tk, d, scale, causal, cu_seqlens, cu_seqlens_k,
                         deterministic, stream), "fa_bwd_kv")
    else:
        _check(fa_bwd_preprocess(o, o.dtype, dout, D, ws, ws_bytes, B, Hq, Hkv, Nq, Tq, d, causal,
                                 cu_seqlens, deterministic, stream), "fa_bwd_preprocess")
        _check(fa_bwd(q, k, v, dout, lse, D, dq, dk, dv, grad_dtype, ws, ws_bytes, B, Hq, Hkv, Nq,
                      Tq, d, scale, causal, cu_seqlens, deterministic, stream), "fa_bwd")
    if check_status and Tq > 0 and Tk > 0 and B > 0:
        _check(fa_check_device_status(ws, stream), "fa_bwd (device)")
    return dq, dk, dv


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, scale, cu_seqlens, max_seqlen, batch, deterministic,
                cu_seqlens_k, max_seqlen_k):
        o, lse = forward(q, k, v, causal, scale, cu_seqlens, max_seqlen, batch,
                         cu_seqlens_k=cu_seqlens_k, max_seqlen_k=max_seqlen_k)
        ctx.save_for_backward(q, k, v, o, lse, cu_seqlens, cu_seqlens_k)
        ctx.args = (causal, scale, max_seqlen, batch, deterministic, max_seqlen_k)
        return o

    @staticmethod
    def backward(ctx, dout):
        q, k, v, o, lse, cu_seqlens, cu_seqlens_k = ctx.saved_tensors
        causal, scale, max_seqlen, batch, deterministic, max_seqlen_k = ctx.args
        dq, dk, dv = backward(q, k, v, o, dout.contiguous(), lse, causal, scale, cu_seqlens,
                              max_seqlen, batch, deterministic, cu_seqlens_k=cu_seqlens_k,
                              max_seqlen_k=max_seqlen_k)
        return dq, dk, dv, None, None, None, None, None, None, None, None


def attention(q, k, v, causal=False, scale=None, cu_seqlens=None, max_seqlen=None, batch=None,
              deterministic=False, cu_seqlens_k=None, max_seqlen_k=None):
    """Differentiable attention (autograd wrapper around forward/backward)."""
    return _Attention.apply(q, k, v, causal, scale, cu_seqlens, max_seqlen, batch, deterministic,
                            cu_seqlens_k, max_seqlen_k)
