"""GPU parity at the size limits, against the fp64 oracle on sampled outputs.

- Offsets past 2^31 elements: a packed batch of 2049 sequences x 8 heads x
  d = 128 (T*H*d > 2^31 in every token-major tensor) -- the first and the last
  sequences are checked whole.
- 4096 packed sequences (the scheduler's limit) of lengths 1..300, GQA,
  sampled sequences whole, atomic and deterministic.
- One 131072-token causal sequence (1024 tiles per sequence, MQA): rows near
  both ends and keys near the end, atomic and deterministic, and the
  deterministic backward bit-identical over a repeat.

Inputs are drawn on the device (synth.make_inputs_device); only the checked
slices go to the oracle."""
import numpy as np
import pytest
import torch

import bwd_tiled_attention_gb300 as fa
import oracle
import synth
from harness import assert_close, assert_lse, to_np

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def test_offsets_past_2_pow_31_elements():
    lengths = [1024] * 2049
    Hq = Hkv = 8
    d = 128
    x = synth.make_inputs_device(Hq, Hkv, d, 31, lengths, "cuda")
    T = sum(lengths)
    assert T * Hq * d > 2 ** 31
    scale = 1.0 / np.sqrt(d)
    kw = dict(cu_seqlens=x["cu_seqlens"], max_seqlen=1024)
    o, lse = fa.forward(x["q"], x["k"], x["v"], causal=True, scale=scale, **kw)
    dq, dk, dv = fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=True,
                             scale=scale, check_status=True, **kw)
    torch.cuda.synchronize()
    for b in (0, len(lengths) - 1):
        s0, s1 = b * 1024, (b + 1) * 1024
        for h in (0, Hq - 1):
            sl = lambda t: f64(t[s0:s1, h:h + 1])
            ref = oracle.attention(sl(x["q"]), sl(x["k"]), sl(x["v"]), [0, 1024], scale, True,
                                   dout=sl(x["dout"]))
            for name, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
                assert_close(f"{name} b{b} h{h}", f64(t[s0:s1, h]), ref[name][:, 0])
            assert_lse(f64(lse[h, s0:s1]), ref["lse"][0])


def test_longest_sequence_mqa():
    N, Hq, Hkv, d = 131072, 2, 1, 128
    x = synth.make_inputs_device(Hq, Hkv, d, 32, [N], "cuda")
    scale = 1.0 / np.sqrt(d)
    kw = dict(cu_seqlens=x["cu_seqlens"], max_seqlen=N)
    o, lse = fa.forward(x["q"], x["k"], x["v"], causal=True, scale=scale, **kw)
    grads = {}
    for det in (False, True):
        grads[det] = fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=True,
                                 scale=scale, deterministic=det, check_status=True, **kw)
    again = fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=True, scale=scale,
                        deterministic=True, check_status=True, **kw)
    torch.cuda.synchronize()
    for a, b in zip(grads[True], again):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    q, k, v, do = (f64(x[n]) for n in ("q", "k", "v", "dout"))
    cu = np.array([0, N], dtype=np.int32)
    rng = np.random.default_rng(33)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, N - 1], rng.integers(0, 512, 6),
                                     rng.integers(N - 4096, N, 6)]))
    keys = np.unique(np.concatenate([[N - 1, N - 128, N - 129], rng.integers(N - 512, N, 8)]))
    for h in range(Hq):
        ref = oracle.rows(q, k, v, cu, scale, True, 0, h, rows, dout=do)
        assert_close(f"o h{h}", f64(o[rows, h]), ref["o"])
        assert_lse(f64(lse[h, rows]), ref["lse"])
        for det in (False, True):
            assert_close(f"dq h{h} det={det}", f64(grads[det][0][rows, h]), ref["dq"])
    kg = oracle.key_grads(q, k, v, do, cu, scale, True, 0, 0, keys)
    for det in (False, True):
        assert_close(f"dk det={det}", f64(grads[det][1][keys, 0]), kg["dk"])
        assert_close(f"dv det={det}", f64(grads[det][2][keys, 0]), kg["dv"])


@pytest.mark.parametrize("deterministic", [False, True])
def test_largest_packed_batch(deterministic):
    """4096 sequences (the scheduler's limit), lengths 1..300, GQA: the
    one-CTA ranking of the scheduler at full size and thousands of ragged
    tiles; sampled sequences against the oracle."""
    gen = np.random.default_rng(34)
    lengths = [int(x) for x in gen.integers(1, 301, 4096)]
    Hq, Hkv, d = 4, 2, 64
    x = synth.make_inputs_device(Hq, Hkv, d, 35, lengths, "cuda")
    scale = 1.0 / np.sqrt(d)
    kw = dict(cu_seqlens=x["cu_seqlens"], max_seqlen=max(lengths))
    o, lse = fa.forward(x["q"], x["k"], x["v"], causal=True, scale=scale, **kw)
    dq, dk, dv = fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=True,
                             scale=scale, deterministic=deterministic, check_status=True, **kw)
    torch.cuda.synchronize()
    cu = np.concatenate([[0], np.cumsum(lengths)])
    for b in sorted({0, 1, 4095, int(np.argmax(lengths)), int(np.argmin(lengths)),
                     *gen.integers(0, 4096, 5).tolist()}):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        sl = lambda t: f64(t[s0:s1])
        ref = oracle.attention(sl(x["q"]), sl(x["k"]), sl(x["v"]), [0, s1 - s0], scale, True,
                               dout=sl(x["dout"]))
        for name, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
            assert_close(f"{name} b{b}", f64(t[s0:s1]), ref[name])
        assert_lse(f64(lse[:, s0:s1]), ref["lse"])
