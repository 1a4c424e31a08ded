"""Seeded synthetic inputs for attention, shared by the oracle and the CUDA path.

This module holds no attention arithmetic: it only draws random tensors with
torch's CPU generator and rounds them to bfloat16 (round to nearest even), so
that the oracle (which converts the bf16 values exactly to float64) and the
CUDA library see the same bytes.

Draw order for one workload: sequence lengths first (variable-length batches
only), then Q, K, V, dO with ``randn`` in float32 at the packed shape
``[T, H, d]``, then the per-tensor scale, then the bf16 rounding.

The named workloads are the shapes the tiled-attention pages discuss (dense
mid-size batches, one long causal sequence, grouped/multi-query heads, and a
packed variable-length batch) at head dimension 64 or 128.  ``make_inputs_kv``
draws queries and keys of different lengths (new tokens against a longer key
sequence): Q and dO over the query tokens, K and V over the key tokens.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    causal: bool
    seed: int
    N: int = 0                      # sequence length (dense) or max length (varlen)
    lengths: list | None = None     # per-sequence lengths (varlen), drawn from the seed
    len_range: tuple | None = None  # (lo, hi) inclusive range for drawn lengths
    qk_scale: float = 1.0           # Q and K multiplied by this before rounding
    o_fp32: bool = False            # forward writes an fp32 O
    deterministic: bool = False     # backward in deterministic mode
    lengths_k: list | None = None   # key/value lengths, when they differ from the query lengths
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


def workloads() -> dict:
    """The named workloads, keyed by name."""
    return {
        "tiny": Workload("tiny", B=1, Hq=2, Hkv=2, d=64, causal=False, seed=0, N=128,
                         o_fp32=True),
        "mid_dense": Workload("mid_dense", B=4, Hq=16, Hkv=16, d=128, causal=False, seed=1,
                              N=2048),
        "mid_causal": Workload("mid_causal", B=4, Hq=16, Hkv=16, d=128, causal=True, seed=1,
                               N=2048),
        "long_causal": Workload("long_causal", B=1, Hq=16, Hkv=16, d=128, causal=True, seed=2,
                                N=32768, qk_scale=0.5),
        "gqa8_causal": Workload("gqa8_causal", B=2, Hq=32, Hkv=8, d=128, causal=True, seed=3,
                                N=8192),
        "mqa_causal": Workload("mqa_causal", B=2, Hq=32, Hkv=1, d=128, causal=True, seed=3,
                               N=8192),
        "varlen_det": Workload("varlen_det", B=16, Hq=16, Hkv=16, d=128, causal=True, seed=4,
                               len_range=(256, 8192), deterministic=True),
        "mid_causal_d64": Workload("mid_causal_d64", B=4, Hq=16, Hkv=16, d=64, causal=True,
                                   seed=7, N=2048),
        "mid_causal_d96": Workload("mid_causal_d96", B=4, Hq=16, Hkv=16, d=96, causal=True,
                                   seed=7, N=2048),
        # forward only (bench.py --forward-only): the backward stops at d = 128
        "mid_causal_d192": Workload("mid_causal_d192", B=4, Hq=16, Hkv=16, d=192, causal=True,
                                    seed=8, N=2048),
        "mid_causal_d256": Workload("mid_causal_d256", B=4, Hq=16, Hkv=16, d=256, causal=True,
                                    seed=8, N=2048),
        **kv_workloads(),
    }


def draw_lengths(gen: torch.Generator, B: int, lo: int, hi: int) -> list:
    return [int(x) for x in torch.randint(lo, hi + 1, (B,), generator=gen)]


def cu_from_lengths(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def make_inputs(B, Hq, Hkv, d, seed, N=None, lengths=None, len_range=None, qk_scale=1.0):
    """Draw (q, k, v, dout, cu_seqlens, lengths) as bf16 CPU tensors.

    Exactly one of N (dense batch of B sequences of length N), lengths
    (explicit) or len_range (lengths drawn uniformly from [lo, hi]) is used.
    q, dout: [T, Hq, d]; k, v: [T, Hkv, d]; cu_seqlens: int32 [B+1].
    """
    gen = torch.Generator().manual_seed(int(seed))
    if len_range is not None:
        lengths = draw_lengths(gen, B, *len_range)
    elif lengths is None:
        lengths = [int(N)] * B
    lengths = [int(x) for x in lengths]
    T = sum(lengths)
    q = torch.randn((T, Hq, d), generator=gen, dtype=torch.float32)
    k = torch.randn((T, Hkv, d), generator=gen, dtype=torch.float32)
    v = torch.randn((T, Hkv, d), generator=gen, dtype=torch.float32)
    dout = torch.randn((T, Hq, d), generator=gen, dtype=torch.float32)
    if qk_scale != 1.0:
        q = q * qk_scale
        k = k * qk_scale
    return dict(
        q=q.to(torch.bfloat16), k=k.to(torch.bfloat16), v=v.to(torch.bfloat16),
        dout=dout.to(torch.bfloat16), cu_seqlens=cu_from_lengths(lengths), lengths=lengths)


def make_workload(w: Workload, **override):
    """Inputs for a named workload (fields may be overridden, e.g. N=256)."""
    if w.lengths_k is not None:
        kw = dict(Hq=w.Hq, Hkv=w.Hkv, d=w.d, seed=w.seed, lengths_q=w.lengths,
                  lengths_k=w.lengths_k, qk_scale=w.qk_scale)
        kw.update(override)
        return make_inputs_kv(**kw)
    kw = dict(B=w.B, Hq=w.Hq, Hkv=w.Hkv, d=w.d, seed=w.seed, qk_scale=w.qk_scale)
    if w.len_range is not None:
        kw["len_range"] = w.len_range
    elif w.lengths is not None:
        kw["lengths"] = w.lengths
    else:
        kw["N"] = w.N
    kw.update(override)
    if "N" in override:
        kw.pop("len_range", None)
        kw.pop("lengths", None)
    return make_inputs(**kw)


def make_inputs_kv(Hq, Hkv, d, seed, lengths_q, lengths_k, qk_scale=1.0):
    """Draw (q, k, v, dout, cu_seqlens, cu_seqlens_k, lengths, lengths_k) as bf16
    CPU tensors with separate query and key/value lengths per sequence.
    q, dout: [Tq, Hq, d]; k, v: [Tk, Hkv, d]; draw order Q, K, V, dO."""
    gen = torch.Generator().manual_seed(int(seed))
    lengths_q = [int(x) for x in lengths_q]
    lengths_k = [int(x) for x in lengths_k]
    assert len(lengths_q) == len(lengths_k)
    Tq, Tk = sum(lengths_q), sum(lengths_k)
    q = torch.randn((Tq, Hq, d), generator=gen, dtype=torch.float32)
    k = torch.randn((Tk, Hkv, d), generator=gen, dtype=torch.float32)
    v = torch.randn((Tk, Hkv, d), generator=gen, dtype=torch.float32)
    dout = torch.randn((Tq, Hq, d), generator=gen, dtype=torch.float32)
    if qk_scale != 1.0:
        q = q * qk_scale
        k = k * qk_scale
    return dict(
        q=q.to(torch.bfloat16), k=k.to(torch.bfloat16), v=v.to(torch.bfloat16),
        dout=dout.to(torch.bfloat16), cu_seqlens=cu_from_lengths(lengths_q),
        cu_seqlens_k=cu_from_lengths(lengths_k), lengths=lengths_q, lengths_k=lengths_k)


def kv_workloads() -> dict:
    """Named workloads with different query and key lengths.  ``chunk_causal``:
    2048 new tokens per sequence against 8192 keys (6144 earlier positions plus
    the new ones); ``varlen_chunks``: packed sequences whose key length is the
    query length plus a drawn number of earlier positions."""
    gen = torch.Generator().manual_seed(9)
    lq = [int(x) for x in torch.randint(1, 2049, (8,), generator=gen)]
    extra = [int(x) for x in torch.randint(0, 6145, (8,), generator=gen)]
    return {
        "chunk_causal": Workload("chunk_causal", B=4, Hq=16, Hkv=16, d=128, causal=True, seed=5,
                                 lengths=[2048] * 4, lengths_k=[8192] * 4),
        "varlen_chunks": Workload("varlen_chunks", B=8, Hq=16, Hkv=4, d=128, causal=True, seed=6,
                                  lengths=lq, lengths_k=[a + b for a, b in zip(lq, extra)]),
    }


def make_inputs_device(Hq, Hkv, d, seed, lengths, device, lengths_k=None):
    """Like ``make_inputs`` / ``make_inputs_kv`` but drawn on ``device`` with
    torch's seeded generator for that device, for sizes whose host copies would
    not fit comfortably (tens of GB).  Same draw order (Q, K, V, dO in float32,
    then bf16 rounding).  Checks copy the slices they compare to the host."""
    gen = torch.Generator(device=device).manual_seed(int(seed))
    lengths = [int(x) for x in lengths]
    lengths_k = lengths if lengths_k is None else [int(x) for x in lengths_k]
    Tq, Tk = sum(lengths), sum(lengths_k)
    out = {}
    for name, T, H in (("q", Tq, Hq), ("k", Tk, Hkv), ("v", Tk, Hkv), ("dout", Tq, Hq)):
        t = torch.empty((T, H, d), dtype=torch.bfloat16, device=device)
        # draw in chunks of rows so the float32 temporary stays small
        step = max(1, (1 << 26) // (H * d))
        for r0 in range(0, T, step):
            r1 = min(T, r0 + step)
            t[r0:r1] = torch.randn((r1 - r0, H, d), generator=gen, device=device,
                                   dtype=torch.float32).to(torch.bfloat16)
        out[name] = t
    out["cu_seqlens"] = cu_from_lengths(lengths).to(device)
    out["cu_seqlens_k"] = cu_from_lengths(lengths_k).to(device)
    out["lengths"], out["lengths_k"] = lengths, lengths_k
    return out
