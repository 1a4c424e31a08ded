"""GPU parity with different query and key lengths (the *_kv entry points),
against the fp64 oracle.  Under the causal mask the queries are the last
positions of the key sequence: query i sees key j iff j <= i + Lk - Lq.

Small packed batches are compared element by element: shorter and longer key
sequences, ragged tails, a single query, more queries than keys (rows that
see no key: O = 0, LSE = -inf, dQ = 0), empty query or key sequences (dK =
dV = 0 for keys no query sees, also in long runs of such units per CTA),
GQA/MQA and three head dims, atomic and deterministic.  The full-size chunk workload (2048 new tokens against 8192
keys) is checked on sampled rows and keys, and must be bit-identical over
repeats in deterministic mode."""
import numpy as np
import pytest
import torch

import bwd_tiled_attention_gb300 as fa
import oracle
import synth
from harness import assert_close, cuda_inputs, oracle_inputs, to_np

pytestmark = pytest.mark.gpu

CASES = [
    # name, lengths_q, lengths_k, Hq, Hkv, d
    ("longer_keys", [129, 1, 300, 77], [400, 513, 300, 1000], 4, 2, 128),
    ("more_queries", [300, 200, 129], [129, 64, 1], 4, 4, 128),
    ("d64_mqa", [256, 100, 5], [700, 100, 383], 6, 1, 64),
    ("empty_sides", [0, 50, 128, 0], [200, 0, 128, 0], 2, 2, 128),
    ("d96", [129, 300], [700, 300], 4, 2, 96),
    # ~1500 key/value units that no query sees, about ten in a row per CTA,
    # between ordinary ones: their dK/dV hand-offs must keep in step
    ("many_keyless_units", [0, 300, 0, 129], [8192, 400, 4096, 129], 16, 4, 128),
]


def assert_lse_kv(got, ref, tol=1e-3):
    dead = np.isneginf(ref)
    assert np.all(np.isneginf(got[dead])), "rows that see no key must have LSE = -inf"
    if np.any(~dead):
        m = float(np.max(np.abs(got[~dead] - ref[~dead])))
        assert m <= tol, f"lse: max_abs={m:.3e}"


def kv_inputs(lq, lk, Hq, Hkv, d, seed):
    inp = synth.make_inputs_kv(Hq, Hkv, d, seed, lq, lk)
    x = cuda_inputs(inp)
    x["cu_seqlens_k"] = inp["cu_seqlens_k"].cuda()
    return inp, x


def run_kv(x, lq, lk, causal, scale, deterministic=False, grad_dtype=torch.bfloat16,
           out_dtype=None):
    """Forward + backward; O is stored in out_dtype, by default the gradients'
    dtype (a bf16 O feeds its rounding into D = rowsum(dO * O) and from there
    into dK)."""
    kw = dict(cu_seqlens=x["cu_seqlens"], max_seqlen=max(max(lq), 1),
              cu_seqlens_k=x["cu_seqlens_k"], max_seqlen_k=max(max(lk), 1))
    o, lse = fa.forward(x["q"], x["k"], x["v"], causal=causal, scale=scale,
                        out_dtype=grad_dtype if out_dtype is None else out_dtype, **kw)
    dq, dk, dv = fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=causal,
                             scale=scale, deterministic=deterministic, grad_dtype=grad_dtype,
                             check_status=True, **kw)
    torch.cuda.synchronize()
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("name,lq,lk,Hq,Hkv,d", CASES)
def test_kv_parity(name, lq, lk, Hq, Hkv, d, causal, deterministic):
    inp, x = kv_inputs(lq, lk, Hq, Hkv, d, seed=21)
    scale = 1.0 / np.sqrt(d)
    oi = oracle_inputs(inp)
    ref = oracle.attention(oi["q"], oi["k"], oi["v"], inp["cu_seqlens"].numpy(), scale, causal,
                           dout=oi["dout"], cu_seqlens_k=inp["cu_seqlens_k"].numpy())
    got = run_kv(x, lq, lk, causal, scale, deterministic)
    assert_close("o", to_np(got["o"]), ref["o"])
    assert_lse_kv(to_np(got["lse"]), ref["lse"])
    for g in ("dq", "dk", "dv"):
        assert_close(g, to_np(got[g]), ref[g])
    # the literal bound on fp32 gradients, with the default bf16 O and with O in fp32
    for o_dt in (torch.bfloat16, torch.float32):
        g32 = run_kv(x, lq, lk, causal, scale, deterministic, grad_dtype=torch.float32,
                     out_dtype=o_dt)
        for g in ("dq", "dk", "dv"):
            got32 = to_np(g32[g])
            label = f"{g} (fp32 out, {str(o_dt)[6:]} O)"
            if (name, causal, g, o_dt) == ("d64_mqa", True, "dk", torch.bfloat16):
                keys_beyond_bound(inp, oi, ref, got32, scale, label)
            else:
                assert_close(label, got32, ref[g], stored_bf16=False)


def keys_beyond_bound(inp, oi, ref, dk, scale, label):
    """The one output of these cases that passes the absolute bound of 2e-2:
    dK of key 0 of sequence 1 (100 queries and 100 keys, 6 query heads on one
    key/value head, d = 64) with the default bf16 O, off by 0.0216 at a
    relative Frobenius error of 2.4e-3.  The rounding model
    (tests/rounding_model.py: the kernels' bf16 rounding points in float64
    numpy) lands exactly as far from the oracle there -- and 0.0184 with O in
    fp32, under the bound, as the kernel does -- so the excess is the bf16
    precision of P, dS and the stored O, not a defect.  Checked here: the
    relative bound on the whole tensor, the literal bound on every other
    sequence's keys, and the kernel within 3e-3 of the model on sequence 1."""
    from rounding_model import grads
    assert_close(label + " (relative)", dk, ref["dk"], stored_bf16=False, mabs=1.0)
    cq, ck = inp["cu_seqlens"].numpy(), inp["cu_seqlens_k"].numpy()
    b = 1
    q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
    assert q1 - q0 == k1 - k0, "the model covers equal query and key lengths"
    others = np.r_[0:k0, k1:dk.shape[0]]
    assert_close(label + " other sequences", dk[others], ref["dk"][others], stored_bf16=False)
    model = grads(oi["q"][q0:q1], oi["k"][k0:k1, 0], oi["v"][k0:k1, 0], oi["dout"][q0:q1],
                  scale, True)
    err_kernel = float(np.max(np.abs(dk[k0:k1] - ref["dk"][k0:k1])))
    err_model = float(np.max(np.abs(model["dk"] - ref["dk"][k0:k1, 0])))
    assert err_model > 2e-2 and err_kernel <= err_model + 3e-3, (err_kernel, err_model)
    assert_close(label + " vs the rounding model", dk[k0:k1, 0], model["dk"], stored_bf16=False,
                 mabs=3e-3)


@pytest.mark.parametrize("causal", [False, True])
def test_kv_dense_batch(causal):
    """Dense batch (no boundaries): Tq = B*Nq queries against Tk = B*Nk keys."""
    B, Nq, Nk, H, d = 2, 200, 520, 4, 128
    inp = synth.make_inputs_kv(H, H, d, 23, [Nq] * B, [Nk] * B)
    x = cuda_inputs(inp)
    scale = 1.0 / np.sqrt(d)
    oi = oracle_inputs(inp)
    ref = oracle.attention(oi["q"], oi["k"], oi["v"], inp["cu_seqlens"].numpy(), scale, causal,
                           dout=oi["dout"], cu_seqlens_k=inp["cu_seqlens_k"].numpy())
    o, lse = fa.forward(x["q"], x["k"], x["v"], causal=causal, scale=scale, batch=B)
    dq, dk, dv = fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=causal,
                             scale=scale, batch=B, check_status=True)
    assert_close("o", to_np(o), ref["o"])
    assert_lse_kv(to_np(lse), ref["lse"])
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close(name, to_np(t), ref[name])


def test_kv_entry_with_equal_lengths_matches_equal_length_entry():
    """Equal lengths through the *_kv calls: the same kernels, the same bits as
    fa_fwd / fa_bwd (O, LSE, and the dQ-free dK/dV of atomic mode)."""
    lengths = [300, 129, 512]
    inp = synth.make_inputs(B=3, Hq=4, Hkv=2, d=128, seed=25, lengths=lengths)
    x = cuda_inputs(inp)
    kw = dict(cu_seqlens=x["cu_seqlens"], max_seqlen=512)
    o, lse = fa.forward(x["q"], x["k"], x["v"], causal=True, **kw)
    dq, dk, dv = fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=True,
                             deterministic=True, **kw)
    kw_kv = dict(kw, cu_seqlens_k=x["cu_seqlens"].clone(), max_seqlen_k=512)
    o2, lse2 = fa.forward(x["q"], x["k"], x["v"], causal=True, **kw_kv)
    dq2, dk2, dv2 = fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=True,
                                deterministic=True, **kw_kv)
    torch.cuda.synchronize()
    for a, b in ((o, o2), (lse, lse2), (dq, dq2), (dk, dk2), (dv, dv2)):
        assert torch.equal(a, b)


def _sampled_check(w, inp, got, rng):
    oi = oracle_inputs(inp)
    cu_q, cu_k = inp["cu_seqlens"].numpy(), inp["cu_seqlens_k"].numpy()
    B = len(w.lengths)
    for b in sorted({0, B - 1, int(rng.integers(0, B))}):
        Lq, Lk = int(cu_q[b + 1] - cu_q[b]), int(cu_k[b + 1] - cu_k[b])
        h = int(rng.integers(0, w.Hq))
        rows = np.unique(np.concatenate([[0, Lq - 1], rng.integers(0, Lq, 16)]))
        ref = oracle.rows(oi["q"], oi["k"], oi["v"], cu_q, w.scale, w.causal, b, h, rows,
                          dout=oi["dout"], cu_seqlens_k=cu_k)
        t = cu_q[b] + rows
        assert_close(f"o b{b} h{h}", to_np(got["o"][t, h]), ref["o"])
        assert_lse_kv(to_np(got["lse"][h, t]), ref["lse"])
        assert_close(f"dq b{b} h{h}", to_np(got["dq"][t, h]), ref["dq"])
        g = int(rng.integers(0, w.Hkv))
        lo = int(Lk * 0.8)
        keys = np.unique(np.concatenate([[lo, Lk - 1], rng.integers(lo, Lk, 8)]))
        kg = oracle.key_grads(oi["q"], oi["k"], oi["v"], oi["dout"], cu_q, w.scale, w.causal, b,
                              g, keys, cu_seqlens_k=cu_k)
        t = cu_k[b] + keys
        assert_close(f"dk b{b} g{g}", to_np(got["dk"][t, g]), kg["dk"])
        assert_close(f"dv b{b} g{g}", to_np(got["dv"][t, g]), kg["dv"])


@pytest.mark.slow
@pytest.mark.parametrize("name", ["chunk_causal", "varlen_chunks"])
def test_kv_workloads_sampled(name):
    w = synth.workloads()[name]
    inp, x = kv_inputs(w.lengths, w.lengths_k, w.Hq, w.Hkv, w.d, w.seed)
    got = run_kv(x, w.lengths, w.lengths_k, w.causal, w.scale)
    _sampled_check(w, inp, got, np.random.default_rng(8))
    det = run_kv(x, w.lengths, w.lengths_k, w.causal, w.scale, deterministic=True)
    _sampled_check(w, inp, det, np.random.default_rng(9))
    for _ in range(3):
        again = run_kv(x, w.lengths, w.lengths_k, w.causal, w.scale, deterministic=True)
        for k in ("dq", "dk", "dv"):
            assert torch.equal(det[k].view(torch.int16), again[k].view(torch.int16))
