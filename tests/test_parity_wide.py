"""Parity for head dimensions 192 and 256 against the fp64 oracle.

The forward runs one 128-row query tile per work unit on 192- or 256-column
tiles.  The backward walks each key/value tile's query tiles twice (dV, then
dK and dQ) with Q and dO streamed in 64-column chunks.  Cases: packed varlen
with ragged tails, GQA and MQA, causal and not, different query and key
lengths (including rows that see no key and keys no query sees), more units
than CTAs, fp32 outputs with the literal bound, atomic and deterministic dQ
(bit-identical repeats)."""
import numpy as np
import pytest
import torch

import bwd_tiled_attention_gb300 as fa
import oracle
import synth
from harness import assert_close, cuda_inputs, oracle_inputs, to_np

pytestmark = pytest.mark.gpu


def assert_lse_kv(got, ref, tol=1e-3):
    dead = np.isneginf(ref)
    assert np.all(np.isneginf(got[dead]))
    if np.any(~dead):
        assert float(np.max(np.abs(got[~dead] - ref[~dead]))) <= tol


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,Hq,Hkv,lq,lk", [
    (256, 4, 2, [129, 300, 1], None),
    (192, 6, 1, [257, 64, 500], None),
    (256, 2, 2, [100, 300], [400, 300]),
    (192, 4, 4, [300, 77], [129, 600]),
    # more units than CTAs, so CTAs walk several units: with Lq > Lk the first
    # query tiles of a sequence see no key (dummy steps between real ones)
    (256, 24, 4, [600, 333, 900], [200, 333, 1000]),
    (192, 16, 2, [700, 1000, 520, 900], None),
])
def test_wide_head_forward(d, Hq, Hkv, lq, lk, causal):
    kv = lk is not None
    if kv:
        inp = synth.make_inputs_kv(Hq, Hkv, d, 41, lq, lk)
    else:
        inp = synth.make_inputs(B=len(lq), Hq=Hq, Hkv=Hkv, d=d, seed=41, lengths=lq)
    x = cuda_inputs(inp)
    kw = dict(cu_seqlens=x["cu_seqlens"], max_seqlen=max(lq))
    cu_k = None
    if kv:
        x["cu_seqlens_k"] = inp["cu_seqlens_k"].cuda()
        kw.update(cu_seqlens_k=x["cu_seqlens_k"], max_seqlen_k=max(lk))
        cu_k = inp["cu_seqlens_k"].numpy()
    scale = 1.0 / np.sqrt(d)
    oi = oracle_inputs(inp)
    ref = oracle.attention(oi["q"], oi["k"], oi["v"], inp["cu_seqlens"].numpy(), scale, causal,
                           cu_seqlens_k=cu_k)
    # repeated: a write into another unit's rows shows up as a race
    for out_dtype in (torch.bfloat16, torch.float32) * 3:
        o, lse = fa.forward(x["q"], x["k"], x["v"], causal=causal, scale=scale,
                            out_dtype=out_dtype, **kw)
        torch.cuda.synchronize()
        assert_close(f"o d{d} {out_dtype}", to_np(o), ref["o"],
                     stored_bf16=out_dtype == torch.bfloat16)
        assert_lse_kv(to_np(lse), ref["lse"])


def within_model(inp, oi, ref, got, name, scale, label):
    """dK or dV of a key/value head shared by many query heads under the
    causal mask: the first keys collect the gradient of every row of every
    head, and bf16 P and dS operands leave them up to a few hundredths from
    the exact values (tests/rounding_model.py).  Checked: the relative bound
    on the whole tensor, and every element either within the absolute bound
    or no further from the oracle than the rounding model (the kernels'
    rounding points in float64, with O in fp32 as here) plus 3e-3."""
    from rounding_model import grads
    assert_close(label + " (relative)", got, ref[name], stored_bf16=False, mabs=1.0)
    cu = inp["cu_seqlens"].numpy()
    Hkv = got.shape[1]
    grp = oi["q"].shape[1] // Hkv
    allowed = np.full(got.shape, 2e-2)
    for b in range(len(cu) - 1):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        if s1 == s0:
            continue
        for g in range(Hkv):
            hs = slice(g * grp, (g + 1) * grp)
            m = grads(oi["q"][s0:s1, hs], oi["k"][s0:s1, g], oi["v"][s0:s1, g],
                      oi["dout"][s0:s1, hs], scale, True, roundings=("fwd_p", "bwd_p", "ds"))
            dist = np.abs(m[name] - ref[name][s0:s1, g]) + 3e-3
            allowed[s0:s1, g] = np.maximum(allowed[s0:s1, g], dist)
    excess = float(np.max(np.abs(got - ref[name]) - allowed))
    assert excess <= 0.0, f"{label}: {excess:.3e} beyond max(2e-2, rounding model + 3e-3)"


WIDE_BWD_CASES = [
    # d, Hq, Hkv, lq, lk (None: equal lengths)
    (256, 4, 2, [129, 300, 1], None),
    (192, 6, 1, [257, 64, 500], None),
    (256, 2, 2, [100, 300], [400, 300]),
    (192, 4, 4, [300, 77, 0], [129, 600, 50]),
    # more units than CTAs
    (256, 16, 4, [600, 333, 900], None),
]


def _wide_inputs(d, Hq, Hkv, lq, lk, seed):
    kv = lk is not None
    if kv:
        inp = synth.make_inputs_kv(Hq, Hkv, d, seed, lq, lk)
    else:
        inp = synth.make_inputs(B=len(lq), Hq=Hq, Hkv=Hkv, d=d, seed=seed, lengths=lq)
    x = cuda_inputs(inp)
    kw = dict(cu_seqlens=x["cu_seqlens"], max_seqlen=max(max(lq), 1))
    cu_k = None
    if kv:
        x["cu_seqlens_k"] = inp["cu_seqlens_k"].cuda()
        kw.update(cu_seqlens_k=x["cu_seqlens_k"], max_seqlen_k=max(max(lk), 1))
        cu_k = inp["cu_seqlens_k"].numpy()
    return inp, x, kw, cu_k


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,Hq,Hkv,lq,lk", WIDE_BWD_CASES)
def test_wide_head_backward(d, Hq, Hkv, lq, lk, causal, deterministic):
    inp, x, kw, cu_k = _wide_inputs(d, Hq, Hkv, lq, lk, 43)
    scale = 1.0 / np.sqrt(d)
    oi = oracle_inputs(inp)
    ref = oracle.attention(oi["q"], oi["k"], oi["v"], inp["cu_seqlens"].numpy(), scale, causal,
                           dout=oi["dout"], cu_seqlens_k=cu_k)
    o, lse = fa.forward(x["q"], x["k"], x["v"], causal=causal, scale=scale, **kw)
    g = fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=causal, scale=scale,
                    deterministic=deterministic, check_status=True, **kw)
    torch.cuda.synchronize()
    for name, t in zip(("dq", "dk", "dv"), g):
        assert_close(f"{name} d{d}", to_np(t), ref[name])
    # fp32 gradients (O in fp32 too): the literal bound
    o32, lse32 = fa.forward(x["q"], x["k"], x["v"], causal=causal, scale=scale,
                            out_dtype=torch.float32, **kw)
    g32 = fa.backward(x["q"], x["k"], x["v"], o32, x["dout"], lse32, causal=causal, scale=scale,
                      deterministic=deterministic, grad_dtype=torch.float32, check_status=True,
                      **kw)
    torch.cuda.synchronize()
    for name, t in zip(("dq", "dk", "dv"), g32):
        if Hq // Hkv >= 6 and causal and lk is None and name != "dq":
            within_model(inp, oi, ref, to_np(t), name, scale, f"{name} d{d} (fp32 out)")
        else:
            assert_close(f"{name} d{d} (fp32 out)", to_np(t), ref[name], stored_bf16=False)
    if deterministic:
        for _ in range(3):
            again = fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=causal,
                                scale=scale, deterministic=True, check_status=True, **kw)
            for a, b in zip(g, again):
                assert torch.equal(a.view(torch.int16), b.view(torch.int16))
