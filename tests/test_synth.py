"""The seeded input generator: reproducible, right shapes, bf16-rounded."""
import torch

import synth


def test_reproducible_and_shapes():
    a = synth.make_inputs(B=2, Hq=4, Hkv=2, d=64, seed=7, N=33)
    b = synth.make_inputs(B=2, Hq=4, Hkv=2, d=64, seed=7, N=33)
    for key in ("q", "k", "v", "dout"):
        assert torch.equal(a[key], b[key])
        assert a[key].dtype == torch.bfloat16
    assert a["q"].shape == (66, 4, 64) and a["k"].shape == (66, 2, 64)
    assert a["cu_seqlens"].tolist() == [0, 33, 66]


def test_varlen_lengths_in_range():
    w = synth.workloads()["varlen_det"]
    x = synth.make_workload(w, len_range=(256, 300))
    assert len(x["lengths"]) == 16
    assert all(256 <= L <= 300 for L in x["lengths"])
    assert x["cu_seqlens"][-1].item() == x["q"].shape[0] == sum(x["lengths"])


def test_qk_scale_applied_before_rounding():
    a = synth.make_inputs(B=1, Hq=1, Hkv=1, d=8, seed=3, N=16, qk_scale=0.5)
    b = synth.make_inputs(B=1, Hq=1, Hkv=1, d=8, seed=3, N=16)
    # scaling by a power of two commutes with rounding to bf16
    assert torch.equal(a["q"].float(), b["q"].float() * 0.5)
    assert torch.equal(a["v"], b["v"])
