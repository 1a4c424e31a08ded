"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory
where they run it (an engine plugin whose execute step must not allocate, a
process whose device memory is all reserved up front).  It keeps D and the
backward workspace in a scratch array owned by the library, so its results
must match fa_bwd_preprocess + fa_bwd with a caller workspace -- on two calls
in a row, since the second call reuses the array the first one left behind.
Errors found inside its kernels are read back with
fa_noalloc_check_device_status, since such a caller holds no workspace.

This file is collected last, so a run that stops at the first failure has run
every other test before it."""
import numpy as np
import pytest
import torch

import bwd_tiled_attention_gb300 as fa
import synth
from bwd_tiled_attention_gb300 import build as fabuild
from harness import assert_close, cuda_inputs, to_np

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20   # the library's fixed scratch array


@pytest.fixture(scope="module", autouse=True)
def _built():
    fabuild.build()


def _case(lengths, Hq, Hkv, d, seed):
    inp = synth.make_inputs(B=len(lengths), Hq=Hq, Hkv=Hkv, d=d, seed=seed, lengths=lengths)
    x = cuda_inputs(inp)
    N, T = max(lengths), sum(lengths)
    return x, N, T


def _noalloc_vs_workspace(lengths, Hq, Hkv, d, seed, causal, deterministic, calls=2,
                          packed=True):
    x, N, T = _case(lengths, Hq, Hkv, d, seed)
    B = len(lengths)
    scale = 1.0 / np.sqrt(d)
    kw = dict(cu_seqlens=x["cu_seqlens"], max_seqlen=N) if packed else dict(batch=B)
    cu = x["cu_seqlens"] if packed else None
    o, lse = fa.forward(x["q"], x["k"], x["v"], causal=causal, scale=scale, **kw)
    ref = fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=causal, scale=scale,
                      deterministic=deterministic, check_status=True, **kw)
    for call in range(calls):
        dq = torch.full_like(x["q"], float("nan"))
        dk = torch.full_like(x["k"], float("nan"))
        dv = torch.full_like(x["v"], float("nan"))
        st = fa.fa_bwd_noalloc(x["q"], x["k"], x["v"], o, fa.FA_BF16, x["dout"], lse, dq, dk, dv,
                               fa.FA_BF16, B, Hq, Hkv, N, T, d, scale, causal, cu,
                               deterministic)
        assert st == fa.FA_OK, fa.fa_status_string(st)
        assert fa.fa_noalloc_check_device_status() == fa.FA_OK
        for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            assert_close(f"{name} call {call}", to_np(got), to_np(want))
            if deterministic:   # same kernels, same order: identical bits
                assert torch.equal(got.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("causal,deterministic", [(True, False), (False, True), (True, True)])
def test_noalloc_matches_workspace_backward_twice(causal, deterministic):
    _noalloc_vs_workspace([300, 512, 77], 4, 2, 128, 31, causal, deterministic)


def test_noalloc_just_under_its_limit():
    """A request that fills the scratch array to within 1 MiB of its end: every
    byte the kernels touch must lie inside it (an off-by-one between the size
    check and the layout would write past the array).  Deterministic, so the
    result must equal the caller-workspace backward bit for bit."""
    B, Hq, d, N = 1, 16, 128, 8064
    ws = fa.fa_bwd_workspace_size(B, Hq, Hq, N, 0, d)
    need = ws + ((Hq * B * N * 4 + 255) // 256) * 256
    assert SCRATCH_BYTES - (1 << 20) < need <= SCRATCH_BYTES
    _noalloc_vs_workspace([N], Hq, Hq, d, 32, True, True, calls=1, packed=False)


def test_noalloc_rejects_requests_beyond_its_scratch():
    # one 128-token tile more than the case above: the dQ accumulator alone fills 64 MiB
    st = fa.fa_bwd_noalloc(16, 16, 16, 16, fa.FA_BF16, 16, 16, 16, 16, 16, fa.FA_BF16,
                           1, 16, 16, 8192, 0, 128, 0.088, 1, None, 0)
    assert st == fa.FA_ERR_UNSUPPORTED
    # 4 x 8192 tokens x 16 heads x 128 x 4 B of dQ accumulator alone is 256 MiB
    st = fa.fa_bwd_noalloc(16, 16, 16, 16, fa.FA_BF16, 16, 16, 16, 16, 16, fa.FA_BF16,
                           4, 16, 16, 8192, 0, 128, 0.088, 1, None, 0)
    assert st == fa.FA_ERR_UNSUPPORTED


def test_noalloc_reports_device_errors():
    """cu_seqlens that contradict N: the scheduler refuses to build a schedule,
    records the error in the scratch array's error word, and the status call
    reports it; the next valid call clears it."""
    inp = synth.make_inputs(B=2, Hq=2, Hkv=2, d=64, seed=8, lengths=[100, 300])
    x = cuda_inputs(inp)
    T, N = 400, 128            # the second sequence is longer than N
    o = torch.zeros((T, 2, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((2, T), dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.empty_like(x[k]) for k in ("q", "k", "v"))
    st = fa.fa_bwd_noalloc(x["q"], x["k"], x["v"], o, fa.FA_BF16, x["dout"], lse, dq, dk, dv,
                           fa.FA_BF16, 2, 2, 2, N, T, 64, 0.125, True, x["cu_seqlens"], False)
    assert st == fa.FA_OK
    assert fa.fa_noalloc_check_device_status() == fa.FA_ERR_INVALID_ARG
    _noalloc_vs_workspace([100, 300], 2, 2, 64, 8, True, False, calls=1)
