"""fp64 CPU oracle for exact softmax attention, forward and backward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The CUDA
library never calls it and shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over rows and
key columns).  This module compiles it with gcc on first use and wraps it with
ctypes and numpy.  Inputs are the bf16-rounded tensors converted exactly to
float64; layouts are packed ``[T, H, d]`` with ``cu_seqlens`` giving sequence
boundaries, and ``lse``/``D`` are ``[Hq, T]``.

Definitions followed (see the C file's header for the full statement):
"FlashAttention-2-ICLR24" sections 问题与动机 (exact attention: S = QK^T,
P = softmax(S)), 核心方法 1 (LSE = m + log l is the only softmax statistic kept),
核心方法 4 (GQA/MQA head map and dK/dV summation); "FlashAttention-4反向传播优化"
section 1.1 (the backward is the five products S, dP, dV, dK, dQ).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, -O2, OpenMP); return its path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c99", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_attention.argtypes = [_dp] * 10 + [
                ctypes.c_int, _ip, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                ctypes.c_int, ctypes.c_int, ctypes.c_int]
            lib.oracle_rows.restype = ctypes.c_int
            lib.oracle_rows.argtypes = [_dp] * 4 + [
                ctypes.c_int, _ip, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, _ip, ctypes.c_int, _dp, _dp, _dp, _dp]
            lib.oracle_key_grads.restype = ctypes.c_int
            lib.oracle_key_grads.argtypes = [_dp] * 4 + [
                ctypes.c_int, _ip, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, _ip, ctypes.c_int, _dp, _dp]
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle uses (set OMP_NUM_THREADS to change)."""
    return int(_load().oracle_num_threads())


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a):
    return a.ctypes.data_as(_dp) if a is not None else None


def _cu(cu_seqlens, T):
    if cu_seqlens is None:
        raise ValueError("cu_seqlens is required (dense batch: [0, N, 2N, ...])")
    cu = _i32(cu_seqlens)
    if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
        raise ValueError("bad cu_seqlens")
    return cu


def attention(q, k, v, cu_seqlens, scale, causal, dout=None, heads=None):
    """Forward (and backward when ``dout`` is given) over query heads ``heads``.

    q: [T, Hq, d]; k, v: [T, Hkv, d]; dout: [T, Hq, d] or None.
    heads: (h_lo, h_hi) half-open range of query heads, default all.
    Returns a dict with o [T,Hq,d], lse [Hq,T] and, for the backward,
    D [Hq,T], dq [T,Hq,d], dk, dv [T,Hkv,d].  Entries for heads outside the
    range (and kv heads they do not reach) are left at zero.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    assert k.shape == (T, Hkv, d) and v.shape == (T, Hkv, d)
    cu = _cu(cu_seqlens, T)
    h_lo, h_hi = heads if heads is not None else (0, Hq)
    o = np.zeros((T, Hq, d))
    lse = np.zeros((Hq, T))
    out = {"o": o, "lse": lse}
    D = dq = dk = dv = None
    if dout is not None:
        dout = _f64(dout)
        assert dout.shape == q.shape
        D = np.zeros((Hq, T))
        dq = np.zeros((T, Hq, d))
        dk = np.zeros((T, Hkv, d))
        dv = np.zeros((T, Hkv, d))
        out.update(D=D, dq=dq, dk=dk, dv=dv)
    rc = _load().oracle_attention(
        _p(q), _p(k), _p(v), _p(dout), _p(o), _p(lse), _p(D), _p(dq), _p(dk), _p(dv),
        len(cu) - 1, cu.ctypes.data_as(_ip), Hq, Hkv, d, float(scale), int(bool(causal)),
        int(h_lo), int(h_hi))
    if rc != 0:
        raise ValueError(f"oracle_attention rejected its arguments (rc={rc})")
    return out


def rows(q, k, v, cu_seqlens, scale, causal, b, h, row_idx, dout=None):
    """O, LSE (and D, dQ when ``dout`` is given) for selected rows of (sequence b, head h).

    row_idx are positions within the sequence.  Returns compact arrays
    o [n,d], lse [n] and, for the backward, D [n], dq [n,d].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    cu = _cu(cu_seqlens, T)
    r = _i32(row_idx)
    n = len(r)
    o = np.zeros((n, d))
    lse = np.zeros(n)
    D = dq = None
    if dout is not None:
        dout = _f64(dout)
        D = np.zeros(n)
        dq = np.zeros((n, d))
    rc = _load().oracle_rows(
        _p(q), _p(k), _p(v), _p(dout), len(cu) - 1, cu.ctypes.data_as(_ip), Hq, Hkv, d,
        float(scale), int(bool(causal)), int(b), int(h), r.ctypes.data_as(_ip), n,
        _p(o), _p(lse), _p(D), _p(dq))
    if rc != 0:
        raise ValueError(f"oracle_rows rejected its arguments (rc={rc})")
    res = {"o": o, "lse": lse}
    if dout is not None:
        res.update(D=D, dq=dq)
    return res


def key_grads(q, k, v, dout, cu_seqlens, scale, causal, b, g, key_idx):
    """dK, dV for selected keys (positions within sequence b) of kv head g,
    summed over all query heads of the group.  Returns dk [n,d], dv [n,d]."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    cu = _cu(cu_seqlens, T)
    kk = _i32(key_idx)
    n = len(kk)
    dk = np.zeros((n, d))
    dv = np.zeros((n, d))
    rc = _load().oracle_key_grads(
        _p(q), _p(k), _p(v), _p(dout), len(cu) - 1, cu.ctypes.data_as(_ip), Hq, Hkv, d,
        float(scale), int(bool(causal)), int(b), int(g), kk.ctypes.data_as(_ip), n,
        _p(dk), _p(dv))
    if rc != 0:
        raise ValueError(f"oracle_key_grads failed (rc={rc})")
    return {"dk": dk, "dv": dv}
