"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory
where they run it (an engine plugin whose execute step must not allocate, a
process whose device memory is all reserved up front).  It keeps D and the
backward workspace in a scratch array owned by the library, so its results
must match fa_bwd_preprocess + fa_bwd with a caller workspace -- on two calls
in a row, since the second call reuses the array the first one left behind.

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


@pytest.fixture(scope="module", autouse=True)
def _built():
    fabuild.build()


def _case(lengths, Hq, Hkv, d, seed):
    inp = synth.make_inputs(B=len(lengths), Hq=Hq, Hkv=Hkv, d=d, seed=seed, lengths=lengths)
    x = cuda_inputs(inp)
    N, T = max(lengths), sum(lengths)
    return x, N, T


@pytest.mark.parametrize("causal,deterministic", [(True, False), (False, True), (True, True)])
def test_noalloc_matches_workspace_backward_twice(causal, deterministic):
    lengths, Hq, Hkv, d = [300, 512, 77], 4, 2, 128
    x, N, T = _case(lengths, Hq, Hkv, d, seed=31)
    B = len(lengths)
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.forward(x["q"], x["k"], x["v"], causal=causal, scale=scale,
                        cu_seqlens=x["cu_seqlens"], max_seqlen=N)
    ref = fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=causal, scale=scale,
                      cu_seqlens=x["cu_seqlens"], max_seqlen=N, deterministic=deterministic,
                      check_status=True)
    for call in range(2):
        dq = torch.full_like(x["q"], float("nan"))
        dk = torch.full_like(x["k"], float("nan"))
        dv = torch.full_like(x["v"], float("nan"))
        st = fa.fa_bwd_noalloc(x["q"], x["k"], x["v"], o, fa.FA_BF16, x["dout"], lse, dq, dk, dv,
                               fa.FA_BF16, B, Hq, Hkv, N, T, d, scale, causal, x["cu_seqlens"],
                               deterministic)
        assert st == fa.FA_OK, fa.fa_status_string(st)
        torch.cuda.synchronize()
        for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            assert_close(f"{name} call {call}", to_np(got), to_np(want))
            if deterministic:   # same kernels, same order: identical bits
                assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_noalloc_rejects_requests_beyond_its_scratch():
    # 4 x 8192 tokens x 16 heads x 128 x 4 B of dQ accumulator alone is 256 MiB > 64 MiB
    st = fa.fa_bwd_noalloc(16, 16, 16, 16, fa.FA_BF16, 16, 16, 16, 16, 16, fa.FA_BF16,
                           4, 16, 16, 8192, 0, 128, 0.088, 1, None, 0)
    assert st == fa.FA_ERR_UNSUPPORTED
