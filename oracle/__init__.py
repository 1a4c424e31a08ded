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
            for name in ("oracle_attention", "oracle_attention_kv"):
                f = getattr(lib, name)
                f.restype = ctypes.c_int
                f.argtypes = [_dp] * 10 + [ctypes.c_int, _ip] + (
                    [_ip] if name.endswith("_kv") else []) + [
                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                    ctypes.c_int, ctypes.c_int, ctypes.c_int]
            for name in ("oracle_rows", "oracle_rows_kv"):
                f = getattr(lib, name)
                f.restype = ctypes.c_int
                f.argtypes = [_dp] * 4 + [ctypes.c_int, _ip] + (
                    [_ip] if name.endswith("_kv") else []) + [
                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                    ctypes.c_int, ctypes.c_int, ctypes.c_int, _ip, ctypes.c_int, _dp, _dp, _dp,
                    _dp]
            for name in ("oracle_key_grads", "oracle_key_grads_kv"):
                f = getattr(lib, name)
                f.restype = ctypes.c_int
                f.argtypes = [_dp] * 4 + [ctypes.c_int, _ip] + (
                    [_ip] if name.endswith("_kv") else []) + [
                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
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


def _cu_pair(cu_seqlens, cu_seqlens_k, Tq, Tk):
    cu_q = _cu(cu_seqlens, Tq)
    cu_k = cu_q if cu_seqlens_k is None else _cu(cu_seqlens_k, Tk)
    if len(cu_k) != len(cu_q):
        raise ValueError("cu_seqlens and cu_seqlens_k name different batch sizes")
    return cu_q, cu_k


def attention(q, k, v, cu_seqlens, scale, causal, dout=None, heads=None, cu_seqlens_k=None):
    """Forward (and backward when ``dout`` is given) over query heads ``heads``.

    q: [Tq, Hq, d]; k, v: [Tk, Hkv, d]; dout: [Tq, Hq, d] or None.
    cu_seqlens bounds the query sequences; cu_seqlens_k the key/value
    sequences (default: the same as cu_seqlens).  With different lengths the
    causal mask is aligned at the end: query i of Lq sees key j iff
    j <= i + Lk - Lq.
    heads: (h_lo, h_hi) half-open range of query heads, default all.
    Returns a dict with o [Tq,Hq,d], lse [Hq,Tq] and, for the backward,
    D [Hq,Tq], dq [Tq,Hq,d], dk, dv [Tk,Hkv,d].  Entries for heads outside the
    range (and kv heads they do not reach) are left at zero.  A row that sees
    no key has O = 0 and LSE = -inf.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, Hq, d = q.shape
    Tk, Hkv = k.shape[0], k.shape[1]
    assert k.shape == (Tk, Hkv, d) and v.shape == (Tk, Hkv, d)
    cu_q, cu_k = _cu_pair(cu_seqlens, cu_seqlens_k, Tq, Tk)
    h_lo, h_hi = heads if heads is not None else (0, Hq)
    o = np.zeros((Tq, Hq, d))
    lse = np.zeros((Hq, Tq))
    out = {"o": o, "lse": lse}
    D = dq = dk = dv = None
    if dout is not None:
        dout = _f64(dout)
        assert dout.shape == q.shape
        D = np.zeros((Hq, Tq))
        dq = np.zeros((Tq, Hq, d))
        dk = np.zeros((Tk, Hkv, d))
        dv = np.zeros((Tk, Hkv, d))
        out.update(D=D, dq=dq, dk=dk, dv=dv)
    rc = _load().oracle_attention_kv(
        _p(q), _p(k), _p(v), _p(dout), _p(o), _p(lse), _p(D), _p(dq), _p(dk), _p(dv),
        len(cu_q) - 1, cu_q.ctypes.data_as(_ip), cu_k.ctypes.data_as(_ip), Hq, Hkv, d,
        float(scale), int(bool(causal)), int(h_lo), int(h_hi))
    if rc != 0:
        raise ValueError(f"oracle_attention rejected its arguments (rc={rc})")
    return out


def rows(q, k, v, cu_seqlens, scale, causal, b, h, row_idx, dout=None, cu_seqlens_k=None):
    """O, LSE (and D, dQ when ``dout`` is given) for selected rows of (sequence b, head h).

    row_idx are positions within the query sequence; cu_seqlens_k as in
    ``attention``.  Returns compact arrays o [n,d], lse [n] and, for the
    backward, D [n], dq [n,d].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, Hq, d = q.shape
    Hkv = k.shape[1]
    cu_q, cu_k = _cu_pair(cu_seqlens, cu_seqlens_k, Tq, k.shape[0])
    r = _i32(row_idx)
    n = len(r)
    o = np.zeros((n, d))
    lse = np.zeros(n)
    D = dq = None
    if dout is not None:
        dout = _f64(dout)
        D = np.zeros(n)
        dq = np.zeros((n, d))
    rc = _load().oracle_rows_kv(
        _p(q), _p(k), _p(v), _p(dout), len(cu_q) - 1, cu_q.ctypes.data_as(_ip),
        cu_k.ctypes.data_as(_ip), Hq, Hkv, d, float(scale), int(bool(causal)), int(b), int(h),
        r.ctypes.data_as(_ip), n, _p(o), _p(lse), _p(D), _p(dq))
    if rc != 0:
        raise ValueError(f"oracle_rows rejected its arguments (rc={rc})")
    res = {"o": o, "lse": lse}
    if dout is not None:
        res.update(D=D, dq=dq)
    return res


def key_grads(q, k, v, dout, cu_seqlens, scale, causal, b, g, key_idx, cu_seqlens_k=None):
    """dK, dV for selected keys (positions within key sequence b) of kv head g,
    summed over all query heads of the group; cu_seqlens_k as in
    ``attention``.  Returns dk [n,d], dv [n,d]."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    Tq, Hq, d = q.shape
    Hkv = k.shape[1]
    cu_q, cu_k = _cu_pair(cu_seqlens, cu_seqlens_k, Tq, k.shape[0])
    kk = _i32(key_idx)
    n = len(kk)
    dk = np.zeros((n, d))
    dv = np.zeros((n, d))
    rc = _load().oracle_key_grads_kv(
        _p(q), _p(k), _p(v), _p(dout), len(cu_q) - 1, cu_q.ctypes.data_as(_ip),
        cu_k.ctypes.data_as(_ip), Hq, Hkv, d, float(scale), int(bool(causal)), int(b), int(g),
        kk.ctypes.data_as(_ip), n, _p(dk), _p(dv))
    if rc != 0:
        raise ValueError(f"oracle_key_grads failed (rc={rc})")
    return {"dk": dk, "dv": dv}
