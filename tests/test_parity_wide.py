"""Forward parity for head dimensions 192 and 256 (forward only: the backward
returns FA_ERR_UNSUPPORTED above 128), against the fp64 oracle.

These run one 128-row query tile per work unit on 192- or 256-column tiles.
Cases: packed varlen with ragged tails, GQA and MQA, causal and not,
different query and key lengths (including rows that see no key), more units
than CTAs, fp32 O."""
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


def test_wide_head_backward_is_unsupported():
    inp = synth.make_inputs(B=1, Hq=2, Hkv=2, d=256, seed=42, lengths=[128])
    x = cuda_inputs(inp)
    o, lse = fa.forward(x["q"], x["k"], x["v"], causal=True, batch=1)
    with pytest.raises(fa.FAError) as e:
        fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=True, batch=1)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
