"""A model of where the kernels round, for explaining their errors.

Test infrastructure, not the oracle and not the product: plain numpy, in
float64 with explicit rounding to float32 and to bfloat16 (round to nearest
even) at the points where the CUDA kernels round.  With every rounding off it
computes exactly what the oracle computes, which a CPU test checks; with the
roundings on it reproduces the kernels' arithmetic closely enough to show how
large the error of a design that feeds bf16 operands to the tensor cores is
on a given input, independently of the kernels' code.

The rounding points (FlashAttention-2-ICLR24, 核心方法 1, and
"FlashAttention-4反向传播优化" section 1.1 describe the steps; the precisions
are this design's):

  forward, per 128-key tile of a row: S in fp32; the reference maximum m
  moves only when the tile's row maximum exceeds it by more than 8 (log2
  units); p = 2^(S*c - m) in fp32, summed into l in fp32; **p rounded to bf16**
  as the A operand of O~ += P V (fp32 accumulation); O = O~ / l, **stored in
  bf16** (or fp32); LSE = (m + log2 l) * ln 2 in fp32.
  backward: D = rowsum(dO * O as stored) in fp32; P = 2^(S*c - LSE*log2 e) in
  fp32, **rounded to bf16** (the A operand of dV += P^T dO, and the P in dS);
  dP in fp32; dS = P * (dP - D) in fp32, **rounded to bf16** (the A operand of
  dK += dS^T Q and dQ += dS K); dK, dV, dQ accumulated in fp32.

Shapes: one sequence and one key/value head: q, dout [L, H, d] (the H query
heads that share the key/value head), k, v [L, d].  Queries and keys have
equal length; causal hides key j from query i when j > i.
"""
from __future__ import annotations

import numpy as np

ROUNDINGS = ("fwd_p", "o_store", "bwd_p", "ds")


def bf16(x):
    """Round to the nearest bfloat16 (ties to even), returned as float64."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    out = u.astype(np.uint32).view(np.float32).astype(np.float64)
    return np.where(np.isfinite(f), out, f.astype(np.float64))


def f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def _ident(x):
    return np.asarray(x, dtype=np.float64)


def grads(q, k, v, dout, scale, causal, roundings=ROUNDINGS, fp32=True, tile=128,
          threshold=8.0):
    """O, LSE, dQ for every head and dK, dV summed over the heads, computed
    with the kernels' rounding points.  `roundings` names the bf16 roundings
    to apply (any subset of ROUNDINGS); fp32=False also drops the float32
    roundings, which makes the result the exact one."""
    r32 = f32 if fp32 else _ident
    rb = {n: (bf16 if n in roundings else r32) for n in ROUNDINGS}
    L, H, d = q.shape
    c = scale / np.log(2.0)           # scale * log2(e)
    vis = np.tril(np.ones((L, L), bool)) if causal else np.ones((L, L), bool)
    o = np.zeros((L, H, d))
    lse = np.zeros((H, L))
    dq = np.zeros((L, H, d))
    dk = np.zeros((L, d))
    dv = np.zeros((L, d))
    for h in range(H):
        Q, dO = q[:, h], dout[:, h]
        S = r32(Q @ k.T)
        # forward: online softmax over 128-key tiles with the conditional rescale
        m_ref = np.full(L, -np.inf)
        l = np.zeros(L)
        Ot = np.zeros((L, d))
        for j0 in range(0, L, tile):
            St = np.where(vis[:, j0:j0 + tile], S[:, j0:j0 + tile], -np.inf)
            mx = r32(St.max(1) * c)
            first = ~np.isfinite(m_ref)
            need = ~first & (mx > m_ref + threshold)
            alpha = np.where(need, r32(np.exp2(np.where(need, m_ref - mx, 0.0))), 1.0)
            Ot = r32(Ot * alpha[:, None])
            l = r32(l * alpha)
            m_ref = np.where(first | need, mx, m_ref)
            x = np.where(np.isfinite(St), r32(St * c - m_ref[:, None]), -np.inf)
            p = r32(np.exp2(x))
            l = r32(l + p.sum(1))
            Ot = r32(Ot + rb["fwd_p"](p) @ v[j0:j0 + tile])
        O = r32(Ot / l[:, None])
        o[:, h] = O
        lse[h] = r32((m_ref + np.log2(l)) * np.log(2.0))
        # backward
        Os = rb["o_store"](O)
        D = r32((dO * Os).sum(1))
        lse2 = r32(lse[h] / np.log(2.0))
        P = np.where(vis, r32(np.exp2(r32(S * c - lse2[:, None]))), 0.0)
        Pb = rb["bwd_p"](P)
        dP = r32(dO @ v.T)
        dS = rb["ds"](r32(Pb * (dP - D[:, None])))
        dv += r32(Pb.T @ dO)
        dk += r32(scale * (dS.T @ Q))
        dq[:, h] = r32(scale * (dS @ k))
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)
