"""Pins for the fp64 CPU oracle: checks against facts the mathematics fixes.

None of these re-types the oracle's formula.  Each pin comes from somewhere
else: a hand-derived example, finite differences of the forward pass, autograd
through library softmax/matmul, closed forms (identical keys, the first causal
row, a single key), invariants (row sums, shift invariance, zero-sum dK), an
independently written tiled online softmax, and the GQA = repeated-heads
identity.  A plausible mistake in the oracle -- a dropped scale, a wrong sign,
a transposed operand, an off-by-one causal mask, a wrong kv-head map -- fails
at least one of them (the mutation test at the end checks that claim for a few
such mistakes).
"""
import math
import os
import re
import subprocess

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_n2_d1.txt")


def rand_case(rng, lengths, Hq, Hkv, d, scale_in=1.0):
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q = rng.standard_normal((T, Hq, d)) * scale_in
    k = rng.standard_normal((T, Hkv, d)) * scale_in
    v = rng.standard_normal((T, Hkv, d))
    do = rng.standard_normal((T, Hq, d))
    return q, k, v, do, cu


# --------------------------------------------------------------------------- golden


def _golden():
    env = {"ln2": math.log(2.0), "ln3": math.log(3.0)}
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        lhs, rhs = line.split("=")
        case, key, idx = lhs.split()
        out[(case, key, int(idx))] = float(eval(rhs, {"__builtins__": {}}, env))
    return out


def test_golden_hand_example():
    g = _golden()
    q = np.array([0.0, 1.0]).reshape(2, 1, 1)
    k = np.array([0.0, math.log(3.0)]).reshape(2, 1, 1)
    v = np.array([2.0, 6.0]).reshape(2, 1, 1)
    do = np.ones((2, 1, 1))
    for case, causal in (("noncausal", False), ("causal", True)):
        r = oracle.attention(q, k, v, [0, 2], 1.0, causal, dout=do)
        for i in range(2):
            assert r["o"][i, 0, 0] == pytest.approx(g[(case, "o", i)], abs=1e-14)
            assert r["lse"][0, i] == pytest.approx(g[(case, "lse", i)], abs=1e-14)
            assert r["D"][0, i] == pytest.approx(g[(case, "D", i)], abs=1e-14)
            assert r["dq"][i, 0, 0] == pytest.approx(g[(case, "dq", i)], abs=1e-14)
            assert r["dk"][i, 0, 0] == pytest.approx(g[(case, "dk", i)], abs=1e-14)
            assert r["dv"][i, 0, 0] == pytest.approx(g[(case, "dv", i)], abs=1e-14)
    # grouped heads: head 1 has q = [0, 0]
    q2 = np.zeros((2, 2, 1))
    q2[:, 0, 0] = [0.0, 1.0]
    do2 = np.ones((2, 2, 1))
    r = oracle.attention(q2, k, v, [0, 2], 1.0, False, dout=do2)
    for i in range(2):
        assert r["o"][i, 1, 0] == pytest.approx(g[("gqa", "o_h1", i)], abs=1e-14)
        assert r["lse"][1, i] == pytest.approx(g[("gqa", "lse_h1", i)], abs=1e-14)
        assert r["dq"][i, 1, 0] == pytest.approx(g[("gqa", "dq_h1", i)], abs=1e-14)
        assert r["dk"][i, 0, 0] == pytest.approx(g[("gqa", "dk", i)], abs=1e-14)
        assert r["dv"][i, 0, 0] == pytest.approx(g[("gqa", "dv", i)], abs=1e-14)


# --------------------------------------------------------------------------- finite differences


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2), (3, 1)])
def test_finite_differences(causal, Hq, Hkv):
    """Central differences of L = sum(dO * O) match dQ, dK, dV."""
    rng = np.random.default_rng(10 + Hq * 3 + Hkv + int(causal))
    lengths = [5, 3]
    d = 3
    scale = 0.7
    q, k, v, do, cu = rand_case(rng, lengths, Hq, Hkv, d)
    r = oracle.attention(q, k, v, cu, scale, causal, dout=do)

    def loss(qq, kk, vv):
        return float(np.sum(do * oracle.attention(qq, kk, vv, cu, scale, causal)["o"]))

    h = 1e-6
    for name, x, grad in (("q", q, r["dq"]), ("k", k, r["dk"]), ("v", v, r["dv"])):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp = x.copy()
            xm = x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name] = xp
            args_m[name] = xm
            num[idx] = (loss(**{"qq": args_p["q"], "kk": args_p["k"], "vv": args_p["v"]})
                        - loss(**{"qq": args_m["q"], "kk": args_m["k"], "vv": args_m["v"]})) / (2 * h)
        err = np.max(np.abs(num - grad)) / max(1.0, np.max(np.abs(grad)))
        assert err < 1e-7, (name, err)


# --------------------------------------------------------------------------- autograd


def _torch_reference(q, k, v, do, lengths, Hq, Hkv, scale, causal):
    """Autograd through torch.softmax / torch.matmul in float64, per sequence."""
    qt = torch.tensor(q, requires_grad=True)
    kt = torch.tensor(k, requires_grad=True)
    vt = torch.tensor(v, requires_grad=True)
    grp = Hq // Hkv
    outs, lses = [], []
    t0 = 0
    for L in lengths:
        qs = qt[t0:t0 + L].transpose(0, 1)                     # [Hq, L, d]
        ks = kt[t0:t0 + L].transpose(0, 1).repeat_interleave(grp, 0)
        vs = vt[t0:t0 + L].transpose(0, 1).repeat_interleave(grp, 0)
        s = torch.matmul(qs, ks.transpose(1, 2)) * scale
        if causal:
            mask = torch.ones(L, L, dtype=torch.bool).triu(1)
            s = s.masked_fill(mask, float("-inf"))
        lses.append(torch.logsumexp(s, dim=-1))               # [Hq, L]
        outs.append(torch.matmul(torch.softmax(s, dim=-1), vs).transpose(0, 1))
        t0 += L
    o = torch.cat(outs, 0)
    (o * torch.tensor(do)).sum().backward()
    return (o.detach().numpy(), torch.cat(lses, 1).detach().numpy(), qt.grad.numpy(),
            kt.grad.numpy(), vt.grad.numpy())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv,d", [(2, 2, 8), (4, 1, 16), (6, 2, 5)])
def test_autograd_library(causal, Hq, Hkv, d):
    rng = np.random.default_rng(100 + Hq + d + int(causal))
    lengths = [17, 1, 9, 32]
    scale = 1.0 / math.sqrt(d)
    q, k, v, do, cu = rand_case(rng, lengths, Hq, Hkv, d)
    r = oracle.attention(q, k, v, cu, scale, causal, dout=do)
    o, lse, dq, dk, dv = _torch_reference(q, k, v, do, lengths, Hq, Hkv, scale, causal)
    np.testing.assert_allclose(r["o"], o, atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(r["lse"], lse, atol=1e-12, rtol=1e-10)
    np.testing.assert_allclose(r["dq"], dq, atol=1e-12, rtol=1e-9)
    np.testing.assert_allclose(r["dk"], dk, atol=1e-12, rtol=1e-9)
    np.testing.assert_allclose(r["dv"], dv, atol=1e-12, rtol=1e-9)


# --------------------------------------------------------------------------- closed forms


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_rows_sum_to_one(causal):
    """With V == 1 every output row is sum_j P_ij, which must be exactly 1."""
    rng = np.random.default_rng(3)
    q, k, v, do, cu = rand_case(rng, [40, 7], 3, 3, 6, scale_in=3.0)
    v = np.ones_like(v)
    r = oracle.attention(q, k, v, cu, 0.9, causal)
    assert np.max(np.abs(r["o"] - 1.0)) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys(causal):
    """All keys equal: P is uniform over the visible keys, so O_i is the mean
    of the visible V rows and LSE_i = s q_i.k + ln(#visible)."""
    rng = np.random.default_rng(4)
    L, H, d, s = 24, 2, 8, 0.3
    q, k, v, do, cu = rand_case(rng, [L], H, H, d)
    k[:] = k[0:1]
    r = oracle.attention(q, k, v, cu, s, causal)
    for h in range(H):
        for i in range(L):
            n = i + 1 if causal else L
            np.testing.assert_allclose(r["o"][i, h], v[:n, h].mean(0), atol=1e-12)
            expect = s * q[i, h] @ k[0, h] + math.log(n)
            assert abs(r["lse"][h, i] - expect) < 1e-12


def test_causal_first_row():
    """Row 0 under the causal mask sees key 0 only: O_0 = V_0, LSE_0 = s q_0.k_0."""
    rng = np.random.default_rng(5)
    q, k, v, do, cu = rand_case(rng, [30, 12], 4, 2, 7)
    r = oracle.attention(q, k, v, cu, 0.5, True)
    for b0 in (0, 30):
        for h in range(4):
            g = h // 2
            np.testing.assert_allclose(r["o"][b0, h], v[b0, g], atol=1e-14)
            assert abs(r["lse"][h, b0] - 0.5 * q[b0, h] @ k[b0, g]) < 1e-13


def test_single_key():
    """N = 1: P = 1, so O = V, dS = 0 (dQ = dK = 0) and dV = dO."""
    rng = np.random.default_rng(6)
    q, k, v, do, cu = rand_case(rng, [1, 1, 1], 2, 1, 4)
    r = oracle.attention(q, k, v, cu, 0.8, False, dout=do)
    np.testing.assert_allclose(r["o"][:, 0], v[:, 0], atol=1e-15)
    np.testing.assert_allclose(r["o"][:, 1], v[:, 0], atol=1e-15)
    assert np.max(np.abs(r["dq"])) < 1e-15 and np.max(np.abs(r["dk"])) < 1e-15
    np.testing.assert_allclose(r["dv"][:, 0], do[:, 0] + do[:, 1], atol=1e-15)


# --------------------------------------------------------------------------- invariants


@pytest.mark.parametrize("causal", [False, True])
def test_invariants(causal):
    rng = np.random.default_rng(7)
    q, k, v, do, cu = rand_case(rng, [20, 11], 4, 2, 6)
    s = 0.6
    base = oracle.attention(q, k, v, cu, s, causal, dout=do)
    # sum_j dS_ij = 0 for every row, hence sum_j dK_j = 0 per (sequence, kv head)
    for b in range(2):
        sl = slice(cu[b], cu[b + 1])
        assert np.max(np.abs(base["dk"][sl].sum(0))) < 1e-12
    # K + c: O unchanged, LSE_i shifts by s q_i.c, dQ/dK unchanged
    c = rng.standard_normal(6)
    r = oracle.attention(q, k + c, v, cu, s, causal, dout=do)
    np.testing.assert_allclose(r["o"], base["o"], atol=1e-12)
    grp = np.repeat(np.arange(2), 2)
    shift = s * np.einsum("thd,d->ht", q, c)
    np.testing.assert_allclose(r["lse"], base["lse"] + shift, atol=1e-12)
    np.testing.assert_allclose(r["dq"], base["dq"], atol=1e-12)
    np.testing.assert_allclose(r["dk"], base["dk"], atol=1e-12)
    # V + c: O + c, dQ and dK unchanged
    r = oracle.attention(q, k, v + c, cu, s, causal, dout=do)
    np.testing.assert_allclose(r["o"], base["o"] + c, atol=1e-12)
    np.testing.assert_allclose(r["dq"], base["dq"], atol=1e-12)
    np.testing.assert_allclose(r["dk"], base["dk"], atol=1e-12)
    del grp


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (6, 1), (8, 4)])
def test_gqa_equals_repeated_heads(causal, Hq, Hkv):
    """GQA on (K, V) equals MHA on K, V with each kv head repeated for its query
    heads, with the repeated heads' dK/dV summed per group."""
    rng = np.random.default_rng(8 + Hq + Hkv)
    q, k, v, do, cu = rand_case(rng, [13, 6], Hq, Hkv, 5)
    grp = Hq // Hkv
    r = oracle.attention(q, k, v, cu, 0.4, causal, dout=do)
    kr = np.repeat(k, grp, axis=1)
    vr = np.repeat(v, grp, axis=1)
    m = oracle.attention(q, kr, vr, cu, 0.4, causal, dout=do)
    np.testing.assert_allclose(r["o"], m["o"], atol=1e-13)
    np.testing.assert_allclose(r["dq"], m["dq"], atol=1e-13)
    T = q.shape[0]
    np.testing.assert_allclose(r["dk"], m["dk"].reshape(T, Hkv, grp, 5).sum(2), atol=1e-13)
    np.testing.assert_allclose(r["dv"], m["dv"].reshape(T, Hkv, grp, 5).sum(2), atol=1e-13)


# --------------------------------------------------------------------------- tiled online softmax


def _tiled_online_forward(q, k, v, scale, causal, br, bc):
    """Forward for one sequence and one head, written from the tiled method:
    query row blocks outside, key/value blocks inside, a running row max m and
    running sum l, an unnormalised output rescaled by exp(m_old - m_new) when
    the max grows, and one division by l at the end; LSE = m + log l
    ("FlashAttention-2-ICLR24", 核心方法 1 and 2)."""
    L, d = q.shape
    o = np.zeros((L, d))
    lse = np.zeros(L)
    for r0 in range(0, L, br):
        r1 = min(L, r0 + br)
        m = np.full(r1 - r0, -np.inf)
        ell = np.zeros(r1 - r0)
        acc = np.zeros((r1 - r0, d))
        for c0 in range(0, L, bc):
            c1 = min(L, c0 + bc)
            if causal and c0 > r1 - 1:
                break                       # block entirely above the diagonal: skipped
            s = scale * q[r0:r1] @ k[c0:c1].T
            if causal:
                rows = np.arange(r0, r1)[:, None]
                cols = np.arange(c0, c1)[None, :]
                s = np.where(cols > rows, -np.inf, s)
            m_new = np.maximum(m, s.max(1))
            alpha = np.exp(m - m_new)
            p = np.exp(s - m_new[:, None])
            ell = alpha * ell + p.sum(1)
            acc = alpha[:, None] * acc + p @ v[c0:c1]
            m = m_new
        o[r0:r1] = acc / ell[:, None]
        lse[r0:r1] = m + np.log(ell)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("br,bc", [(4, 4), (3, 5), (8, 2)])
def test_dense_vs_tiled_online(causal, br, bc):
    rng = np.random.default_rng(9)
    L, d = 23, 6
    q, k, v, do, cu = rand_case(rng, [L], 1, 1, d, scale_in=2.0)
    r = oracle.attention(q, k, v, cu, 0.5, causal)
    o, lse = _tiled_online_forward(q[:, 0], k[:, 0], v[:, 0], 0.5, causal, br, bc)
    np.testing.assert_allclose(r["o"][:, 0], o, atol=1e-12)
    np.testing.assert_allclose(r["lse"][0], lse, atol=1e-12)


# --------------------------------------------------------------------------- sampled entry points


@pytest.mark.parametrize("causal", [False, True])
def test_rows_and_key_grads_match_full(causal):
    rng = np.random.default_rng(11)
    q, k, v, do, cu = rand_case(rng, [37, 50], 6, 2, 8)
    s = 0.35
    full = oracle.attention(q, k, v, cu, s, causal, dout=do)
    rows = [0, 5, 36, 49, 17]
    r = oracle.rows(q, k, v, cu, s, causal, 1, 4, rows, dout=do)
    t = cu[1] + np.array(rows)
    np.testing.assert_allclose(r["o"], full["o"][t, 4], atol=1e-13)
    np.testing.assert_allclose(r["lse"], full["lse"][4, t], atol=1e-13)
    np.testing.assert_allclose(r["D"], full["D"][4, t], atol=1e-13)
    np.testing.assert_allclose(r["dq"], full["dq"][t, 4], atol=1e-13)
    keys = [49, 45, 30]
    kg = oracle.key_grads(q, k, v, do, cu, s, causal, 1, 1, keys)
    t = cu[1] + np.array(keys)
    np.testing.assert_allclose(kg["dk"], full["dk"][t, 1], atol=1e-13)
    np.testing.assert_allclose(kg["dv"], full["dv"][t, 1], atol=1e-13)


def test_head_range_subset():
    rng = np.random.default_rng(12)
    q, k, v, do, cu = rand_case(rng, [19], 4, 4, 5)
    full = oracle.attention(q, k, v, cu, 0.5, True, dout=do)
    part = oracle.attention(q, k, v, cu, 0.5, True, dout=do, heads=(1, 3))
    for key in ("o", "dq"):
        np.testing.assert_allclose(part[key][:, 1:3], full[key][:, 1:3], atol=1e-14)
    for key in ("dk", "dv"):
        np.testing.assert_allclose(part[key][:, 1:3], full[key][:, 1:3], atol=1e-14)
    np.testing.assert_allclose(part["lse"][1:3], full["lse"][1:3], atol=1e-14)


# --------------------------------------------------------------------------- mutations


MUTATIONS = {
    # (pattern in the C source, replacement): each is a plausible slip
    "dropped_scale_dq": ("dqi[c] += scale * dS * kj[c];", "dqi[c] += dS * kj[c];"),
    "wrong_sign_dS": ("const double dS = P * (dP - D[", "const double dS = P * (D["),
    "causal_off_by_one": ("nv = i + off + 1;", "nv = i + off;"),
    # the end-aligned causal offset for different query and key lengths
    "kv_offset_sign_rows": ("Lk, Lk - Lq, i, g,", "Lk, Lq - Lk, i, g,"),
    "kv_offset_sign_cols": ("int i0 = causal ? j - off : 0;", "int i0 = causal ? j + off : 0;"),
    "kv_keys_from_query_base": ("row_s[j] = scale * dot(qi, k + IDX(tk0 + j,",
                                "row_s[j] = scale * dot(qi, k + IDX(j,"),
    "kv_head_map": ("return (int)(((long long)h * Hkv) / Hq);", "return h % Hkv;"),
    "transposed_dv": ("dvj[c] += P * doi[c];", "dvj[c] += P * qi[c];"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistakes(name, tmp_path):
    """Plant one mistake in a private copy of the oracle's C source (CPU only)
    and check that the pins above notice it."""
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()
    pat, rep = MUTATIONS[name]
    assert pat in src, name
    mutated = src.replace(pat, rep)
    c_path = tmp_path / "m.c"
    so_path = tmp_path / "libm.so"
    c_path.write_text(mutated)
    subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", "-fopenmp", "-std=c99", "-o",
                           str(so_path), str(c_path), "-lm"])
    import ctypes
    lib = ctypes.CDLL(str(so_path))
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int)
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_attention.argtypes = [dp] * 10 + [ctypes.c_int, ip, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int]
    lib.oracle_attention_kv.restype = ctypes.c_int
    lib.oracle_attention_kv.argtypes = [dp] * 10 + [ctypes.c_int, ip, ip, ctypes.c_int,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_int]
    rng = np.random.default_rng(13)
    lengths = [9, 4]
    Hq, Hkv, d = 4, 2, 5
    q, k, v, do, cu = rand_case(rng, lengths, Hq, Hkv, d)
    T = q.shape[0]
    caught = False
    for causal in (False, True):
        o = np.zeros((T, Hq, d)); lse = np.zeros((Hq, T)); D = np.zeros((Hq, T))
        dq = np.zeros((T, Hq, d)); dk = np.zeros((T, Hkv, d)); dv = np.zeros((T, Hkv, d))
        P = lambda a: a.ctypes.data_as(dp)
        lib.oracle_attention(P(q), P(k), P(v), P(do), P(o), P(lse), P(D), P(dq), P(dk), P(dv),
                             2, cu.ctypes.data_as(ip), Hq, Hkv, d, 0.5, int(causal), 0, Hq)
        ref = _torch_reference(q, k, v, do, lengths, Hq, Hkv, 0.5, causal)
        for got, want in zip((o, lse, dq, dk, dv), ref):
            if not np.allclose(got, want, atol=1e-9):
                caught = True
    # different query and key lengths (queries at the end of the key sequence)
    from test_oracle_kv_pins import kv_case, torch_reference_kv
    lq, lk = [3, 6], [8, 6]
    q, k, v, do, cu_q, cu_k = kv_case(rng, lq, lk, Hq, Hkv, d)
    Tq, Tk = q.shape[0], k.shape[0]
    for causal in (False, True):
        o = np.zeros((Tq, Hq, d)); lse = np.zeros((Hq, Tq)); D = np.zeros((Hq, Tq))
        dq = np.zeros((Tq, Hq, d)); dk = np.zeros((Tk, Hkv, d)); dv = np.zeros((Tk, Hkv, d))
        P = lambda a: a.ctypes.data_as(dp)
        lib.oracle_attention_kv(P(q), P(k), P(v), P(do), P(o), P(lse), P(D), P(dq), P(dk),
                                P(dv), 2, cu_q.ctypes.data_as(ip), cu_k.ctypes.data_as(ip), Hq,
                                Hkv, d, 0.5, int(causal), 0, Hq)
        ref = torch_reference_kv(q, k, v, do, lq, lk, Hq, Hkv, 0.5, causal)
        for got, want in zip((o, lse, dq, dk, dv), ref):
            if not np.allclose(got, want, atol=1e-9):
                caught = True
    assert caught, f"planted mistake {name} went unnoticed"
