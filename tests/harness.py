"""Shared helpers for the parity tests: run the oracle and the CUDA path on the
same seeded bf16 inputs and compare element by element.

Tolerances (fixed for this method): O, dQ, dK, dV must have relative
Frobenius error <= 1e-2 and max-abs error <= 2e-2 against the fp64 oracle;
LSE max-abs error <= 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

REL_FROB = 1e-2
MAX_ABS = 2e-2
LSE_ABS = 1e-3


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def errors(got: np.ndarray, ref: np.ndarray):
    diff = got - ref
    den = np.linalg.norm(ref)
    rel = np.linalg.norm(diff) / den if den > 0 else np.linalg.norm(diff)
    return float(rel), float(np.max(np.abs(diff))) if diff.size else 0.0


def assert_close(name, got, ref, rel=REL_FROB, mabs=MAX_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    r, m = errors(got, ref)
    assert r <= rel and m <= mabs, (
        f"{name}: rel_frob={r:.3e} max_abs={m:.3e} (max|ref|={np.max(np.abs(ref)):.3g})")
    return r, m


def assert_lse(got, ref, tol=LSE_ABS):
    m = float(np.max(np.abs(np.asarray(got) - np.asarray(ref)))) if np.size(ref) else 0.0
    assert m <= tol, f"lse: max_abs={m:.3e}"
    return m


def oracle_inputs(inp):
    """bf16 CPU tensors -> float64 numpy (exact)."""
    return {k: to_np(inp[k]) for k in ("q", "k", "v", "dout")}


def cuda_inputs(inp, device="cuda"):
    out = {k: inp[k].to(device).contiguous() for k in ("q", "k", "v", "dout")}
    out["cu_seqlens"] = inp["cu_seqlens"].to(device)
    return out
