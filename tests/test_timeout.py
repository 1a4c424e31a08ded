"""Failure detection without a GPU fault: a semaphore that nothing will ever
set makes the deterministic backward's bounded wait give up (about 1 s); the
kernel records FA_ERR_TIMEOUT in the workspace and returns normally, and the
same context then runs a correct backward."""
import numpy as np
import pytest
import torch

import bwd_tiled_attention_gb300 as fa
import synth
from harness import cuda_inputs

pytestmark = pytest.mark.gpu


def test_poisoned_semaphore_times_out_and_gpu_recovers():
    lengths = [256, 384]
    Hq = Hkv = 2
    d = 128
    inp = synth.make_inputs(B=2, Hq=Hq, Hkv=Hkv, d=d, seed=7, lengths=lengths)
    x = cuda_inputs(inp)
    N, T = max(lengths), sum(lengths)
    o, lse = fa.forward(x["q"], x["k"], x["v"], causal=True, cu_seqlens=x["cu_seqlens"],
                        max_seqlen=N)
    ws_b = fa.fa_bwd_workspace_size(2, Hq, Hkv, N, T, d)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    D = torch.empty((Hq, T), dtype=torch.float32, device="cuda")
    dq = torch.empty_like(x["q"]); dk = torch.empty_like(x["k"]); dv = torch.empty_like(x["v"])
    scale = 1.0 / np.sqrt(d)
    args = (2, Hq, Hkv, N, T, d)
    assert fa.fa_bwd_preprocess(o, fa.FA_BF16, x["dout"], D, ws, ws_b, *args, True,
                                x["cu_seqlens"], True) == fa.FA_OK
    # semaphore (head 0, tile 0) can never reach its first target (0)
    off = fa.fa_bwd_workspace_semaphore_offset(*args)
    ws[off:off + 4].view(torch.int32).fill_(1 << 30)
    assert fa.fa_bwd(x["q"], x["k"], x["v"], x["dout"], lse, D, dq, dk, dv, fa.FA_BF16, ws, ws_b,
                     *args[:5], d, scale, True, x["cu_seqlens"], True) == fa.FA_OK
    assert fa.fa_check_device_status(ws) == fa.FA_ERR_TIMEOUT
    # the context is healthy: a fresh preprocess + backward succeeds and is deterministic
    g1 = fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=True,
                     cu_seqlens=x["cu_seqlens"], max_seqlen=N, deterministic=True,
                     check_status=True)
    g2 = fa.backward(x["q"], x["k"], x["v"], o, x["dout"], lse, causal=True,
                     cu_seqlens=x["cu_seqlens"], max_seqlen=N, deterministic=True,
                     check_status=True)
    for a, b in zip(g1, g2):
        assert torch.isfinite(a.float()).all()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_sequence_longer_than_n_is_reported():
    """cu_seqlens that contradict N: the scheduler refuses to build a schedule and
    the device status says so; nothing is read out of bounds."""
    inp = synth.make_inputs(B=2, Hq=2, Hkv=2, d=64, seed=8, lengths=[100, 300])
    x = cuda_inputs(inp)
    T = 400
    ws_b = fa.fa_fwd_workspace_size(2, 2, 128, T)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    o = torch.empty((T, 2, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, T), dtype=torch.float32, device="cuda")
    st = fa.fa_fwd(x["q"], x["k"], x["v"], o, fa.FA_BF16, lse, 2, 2, 2, 128, T, 64, 0.125, 1,
                   x["cu_seqlens"], ws, ws_b)
    assert st == fa.FA_OK
    assert fa.fa_check_device_status(ws) == fa.FA_ERR_INVALID_ARG
