"""Pins for the oracle with different query and key lengths.

The pages state the causal mask for equal lengths only.  The reading taken is
that the Lq queries are the last Lq positions of the Lk-long key sequence
(new tokens attending to a cache of earlier ones), so query i sees key j iff
j <= i + Lk - Lq.  These pins tie that case to facts fixed elsewhere:

- the suffix identity: for Lq <= Lk, the result equals the last Lq rows of the
  square (Lk x Lk) problem whose first Lk - Lq rows carry zero output
  gradient.  Those rows then add nothing to dK or dV, so every output is fixed
  by the square oracle, which the pins in test_oracle_pins.py tie to the hand
  example, finite differences and library autograd;
- for Lq > Lk, rows i < Lq - Lk see no key (O = 0, LSE = -inf, no gradient)
  and the remaining rows are the square Lk x Lk problem;
- autograd through torch.softmax / torch.matmul in float64 with the mask
  written as a boolean matrix;
- the row and key samplers agree with the full computation.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def kv_case(rng, lq, lk, Hq, Hkv, d):
    Tq, Tk = sum(lq), sum(lk)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    q = rng.standard_normal((Tq, Hq, d))
    k = rng.standard_normal((Tk, Hkv, d))
    v = rng.standard_normal((Tk, Hkv, d))
    do = rng.standard_normal((Tq, Hq, d))
    return q, k, v, do, cu_q, cu_k


LQ_LE_LK = ([5, 1, 12, 7, 3], [9, 6, 12, 20, 3])   # includes Lq = Lk and a single query


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv,d", [(2, 2, 6), (4, 2, 8)])
def test_suffix_of_square_problem(causal, Hq, Hkv, d):
    rng = np.random.default_rng(31 + Hq + int(causal))
    lq, lk = LQ_LE_LK
    q, k, v, do, cu_q, cu_k = kv_case(rng, lq, lk, Hq, Hkv, d)
    r = oracle.attention(q, k, v, cu_q, 0.4, causal, dout=do, cu_seqlens_k=cu_k)
    for b, (Lq, Lk) in enumerate(zip(lq, lk)):
        qs, ks = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
        # square problem: Lk query rows, the first Lk - Lq random, with zero dO
        q_full = np.concatenate([rng.standard_normal((Lk - Lq, Hq, d)), q[qs]])
        do_full = np.concatenate([np.zeros((Lk - Lq, Hq, d)), do[qs]])
        sq = oracle.attention(q_full, k[ks], v[ks], [0, Lk], 0.4, causal, dout=do_full)
        tail = slice(Lk - Lq, Lk)
        np.testing.assert_allclose(r["o"][qs], sq["o"][tail], atol=1e-13)
        np.testing.assert_allclose(r["lse"][:, qs], sq["lse"][:, tail], atol=1e-13)
        np.testing.assert_allclose(r["D"][:, qs], sq["D"][:, tail], atol=1e-12)
        np.testing.assert_allclose(r["dq"][qs], sq["dq"][tail], atol=1e-12)
        np.testing.assert_allclose(r["dk"][ks], sq["dk"], atol=1e-12)
        np.testing.assert_allclose(r["dv"][ks], sq["dv"], atol=1e-12)


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 1)])
def test_more_queries_than_keys_causal(Hq, Hkv):
    rng = np.random.default_rng(47 + Hq)
    lq, lk = [9, 4, 6], [4, 4, 1]
    d = 5
    q, k, v, do, cu_q, cu_k = kv_case(rng, lq, lk, Hq, Hkv, d)
    r = oracle.attention(q, k, v, cu_q, 0.7, True, dout=do, cu_seqlens_k=cu_k)
    for b, (Lq, Lk) in enumerate(zip(lq, lk)):
        dead = slice(cu_q[b], cu_q[b] + Lq - Lk)
        live = slice(cu_q[b] + Lq - Lk, cu_q[b + 1])
        ks = slice(cu_k[b], cu_k[b + 1])
        assert np.all(r["o"][dead] == 0) and np.all(r["dq"][dead] == 0)
        assert np.all(np.isneginf(r["lse"][:, dead])) and np.all(r["D"][:, dead] == 0)
        sq = oracle.attention(q[live], k[ks], v[ks], [0, Lk], 0.7, True, dout=do[live])
        for key in ("o", "dq"):
            np.testing.assert_allclose(r[key][live], sq[key], atol=1e-13)
        np.testing.assert_allclose(r["lse"][:, live], sq["lse"], atol=1e-13)
        for key in ("dk", "dv"):
            np.testing.assert_allclose(r[key][ks], sq[key], atol=1e-13)


def torch_reference_kv(q, k, v, do, lq, lk, Hq, Hkv, scale, causal):
    """Autograd through torch.softmax / torch.matmul in float64, per sequence,
    with the end-aligned causal mask as a boolean matrix."""
    qt = torch.tensor(q, requires_grad=True)
    kt = torch.tensor(k, requires_grad=True)
    vt = torch.tensor(v, requires_grad=True)
    grp = Hq // Hkv
    outs, lses = [], []
    tq = tk = 0
    for Lq, Lk in zip(lq, lk):
        qs = qt[tq:tq + Lq].transpose(0, 1)
        ks = kt[tk:tk + Lk].transpose(0, 1).repeat_interleave(grp, 0)
        vs = vt[tk:tk + Lk].transpose(0, 1).repeat_interleave(grp, 0)
        s = torch.matmul(qs, ks.transpose(1, 2)) * scale
        if causal:
            ii = torch.arange(Lq).view(-1, 1)
            jj = torch.arange(Lk).view(1, -1)
            s = s.masked_fill(jj > ii + (Lk - Lq), float("-inf"))
        lses.append(torch.logsumexp(s, dim=-1))
        outs.append(torch.matmul(torch.softmax(s, dim=-1), vs).transpose(0, 1))
        tq += Lq
        tk += Lk
    o = torch.cat(outs, 0)
    (o * torch.tensor(do)).sum().backward()
    return (o.detach().numpy(), torch.cat(lses, 1).detach().numpy(), qt.grad.numpy(),
            kt.grad.numpy(), vt.grad.numpy())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lq,lk", [([5, 1, 12, 7], [9, 6, 12, 20]), ([8, 3], [2, 3])])
def test_autograd_library_kv(causal, lq, lk):
    if causal and any(a > b for a, b in zip(lq, lk)):
        pytest.skip("rows without a visible key are NaN in library softmax; pinned above")
    rng = np.random.default_rng(61 + len(lq) + int(causal))
    Hq, Hkv, d = 4, 2, 7
    q, k, v, do, cu_q, cu_k = kv_case(rng, lq, lk, Hq, Hkv, d)
    scale = 1.0 / math.sqrt(d)
    r = oracle.attention(q, k, v, cu_q, scale, causal, dout=do, cu_seqlens_k=cu_k)
    want = torch_reference_kv(q, k, v, do, lq, lk, Hq, Hkv, scale, causal)
    for key, w in zip(("o", "lse", "dq", "dk", "dv"), want):
        np.testing.assert_allclose(r[key], w, atol=1e-12, rtol=1e-9, err_msg=key)


@pytest.mark.parametrize("causal", [False, True])
def test_rows_and_key_grads_match_full_kv(causal):
    rng = np.random.default_rng(77 + int(causal))
    lq, lk = [7, 13, 2], [19, 13, 9]
    Hq, Hkv, d = 4, 2, 6
    q, k, v, do, cu_q, cu_k = kv_case(rng, lq, lk, Hq, Hkv, d)
    full = oracle.attention(q, k, v, cu_q, 0.5, causal, dout=do, cu_seqlens_k=cu_k)
    for b in range(len(lq)):
        rows = np.arange(lq[b])
        for h in (0, Hq - 1):
            r = oracle.rows(q, k, v, cu_q, 0.5, causal, b, h, rows, dout=do, cu_seqlens_k=cu_k)
            t = cu_q[b] + rows
            np.testing.assert_allclose(r["o"], full["o"][t, h], atol=1e-14)
            np.testing.assert_allclose(r["lse"], full["lse"][h, t], atol=1e-14)
            np.testing.assert_allclose(r["dq"], full["dq"][t, h], atol=1e-14)
        keys = np.array([lk[b] - 1, lk[b] // 2, 0])
        for g in range(Hkv):
            kg = oracle.key_grads(q, k, v, do, cu_q, 0.5, causal, b, g, keys, cu_seqlens_k=cu_k)
            t = cu_k[b] + keys
            np.testing.assert_allclose(kg["dk"], full["dk"][t, g], atol=1e-13)
            np.testing.assert_allclose(kg["dv"], full["dv"][t, g], atol=1e-13)
