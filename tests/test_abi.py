"""The C-ABI library: it builds, loads, exports every symbol include/fa.h
declares, and rejects bad arguments on the host (no GPU needed: validation
returns before any CUDA call)."""
import os
import re

import pytest

import bwd_tiled_attention_gb300 as fa
from bwd_tiled_attention_gb300 import build as fabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    fabuild.build()
    return fa.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", src)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert "fa_fwd" in names and "fa_bwd" in names and "fa_bwd_preprocess" in names
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(fa.EXPORTED)


def test_status_strings(L):
    assert fa.fa_status_string(0) == "FA_OK"
    assert fa.fa_status_string(4) == "FA_ERR_TIMEOUT"
    assert L.fa_version().decode().startswith("gb300")


def test_workspace_sizes(L):
    # forward: header + unit list, grows with heads and tokens
    a = fa.fa_fwd_workspace_size(4, 16, 2048, 0)
    b = fa.fa_fwd_workspace_size(4, 32, 2048, 0)
    assert 0 < a < b
    # backward: includes the fp32 dQ accumulator [T, Hq, d]
    T, Hq, d = 4 * 2048, 16, 128
    w = fa.fa_bwd_workspace_size(4, Hq, Hq, 2048, 0, d)
    assert w >= T * Hq * d * 4
    # A backward unit walks a run of up to 4 query heads of one key/value head
    # (the largest divisor of the group that leaves >= 512 units) and sums
    # dK/dV over them on chip; fp32 partials [T, Hkv * runs, d] exist only
    # when a group takes more than one run.
    # GQA-4 with one run per group (16/4 heads x 64 tiles = 256 units < 512
    # for runs of 4, so runs of 2): 2 runs per key/value head -> partials
    wg = fa.fa_bwd_workspace_size(4, Hq, 4, 2048, 0, d)
    # (its unit list is shorter than MHA's: 8 runs of heads per tile, not 16)
    assert abs((wg - w) - 2 * T * (4 * 2) * d * 4) < (1 << 16)
    # the GQA-8 workload (B2 Hq32 Hkv8 N8192): runs of 4 cover each group, no partials
    w8 = fa.fa_bwd_workspace_size(2, 32, 8, 8192, 0, d)
    w32 = fa.fa_bwd_workspace_size(2, 32, 32, 8192, 0, d)
    assert w8 <= w32 < w8 + (1 << 20)   # (a shorter unit list, nothing more)
    # the MQA workload: 32 heads in runs of 4 -> 8 runs, partials [T, 8, d] x 2
    w1 = fa.fa_bwd_workspace_size(2, 32, 1, 8192, 0, d)
    assert w1 - w8 >= 2 * 2 * 8192 * 8 * d * 4
    assert w1 - w8 < 2 * 2 * 8192 * 8 * d * 4 + (1 << 20)
    off = fa.fa_bwd_workspace_semaphore_offset(4, Hq, Hq, 2048, 0, d)
    assert 0 < off < w and off % 256 == 0
    assert fa.fa_bwd_workspace_size(1, 4, 4, 16, 0, 320) == 0  # unsupported head dim
    assert fa.fa_bwd_workspace_size(1, 4, 4, 16, 0, 256) > 0   # 192 and 256: the wide backward
    assert fa.fa_bwd_workspace_size(1, 4, 4, 16, 0, 96) > 0    # 96 runs on 128-column tiles


FAKE = 0x10000          # 16-byte aligned non-null fake device address (never dereferenced)


def fwd_call(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, o_dtype=fa.FA_BF16, lse=FAKE, B=2, Hq=4, Hkv=2,
                N=64, total_tokens=0, d=64, scale=0.125, causal=1, cu_seqlens=None,
                workspace=FAKE, workspace_bytes=1 << 20, stream=0)
    args.update(kw)
    return fa.fa_fwd(**args)


def test_fwd_rejects_bad_arguments(L):
    assert fwd_call(Hkv=3) == fa.FA_ERR_INVALID_ARG            # Hq % Hkv != 0
    assert fwd_call(d=512) == fa.FA_ERR_UNSUPPORTED             # head dim
    assert fwd_call(d=80) == fa.FA_ERR_UNSUPPORTED
    assert fwd_call(q=FAKE + 8) == fa.FA_ERR_INVALID_ARG        # TMA needs 16-byte alignment
    assert fwd_call(lse=None) == fa.FA_ERR_INVALID_ARG          # null output
    assert fwd_call(workspace_bytes=8) == fa.FA_ERR_INVALID_ARG
    assert fwd_call(scale=0.0) == fa.FA_ERR_UNSUPPORTED
    assert fwd_call(scale=float("nan")) == fa.FA_ERR_UNSUPPORTED
    assert fwd_call(total_tokens=100) == fa.FA_ERR_INVALID_ARG  # dense T must be B*N
    assert fwd_call(o_dtype=7) == fa.FA_ERR_INVALID_ARG
    assert fwd_call(B=-1) == fa.FA_ERR_INVALID_ARG
    assert fwd_call(B=5000, cu_seqlens=FAKE, total_tokens=10) == fa.FA_ERR_UNSUPPORTED
    assert fwd_call(cu_seqlens=FAKE + 2, total_tokens=10) == fa.FA_ERR_INVALID_ARG


def test_empty_inputs_are_a_no_op(L):
    # nothing to compute: success without touching the device
    assert fwd_call(B=0, N=0) == fa.FA_OK
    assert fwd_call(N=0) == fa.FA_OK
    assert fwd_call(cu_seqlens=FAKE, total_tokens=0) == fa.FA_OK


def bwd_call(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, dout=FAKE, lse=FAKE, D=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
                grad_dtype=fa.FA_BF16, workspace=FAKE, workspace_bytes=1 << 30, B=2, Hq=4, Hkv=2,
                N=64, total_tokens=0, d=128, scale=0.1, causal=0, cu_seqlens=None,
                deterministic=1, stream=0)
    args.update(kw)
    return fa.fa_bwd(**args)


def test_bwd_rejects_bad_arguments(L):
    assert bwd_call(Hkv=3) == fa.FA_ERR_INVALID_ARG
    assert bwd_call(d=32) == fa.FA_ERR_UNSUPPORTED
    assert bwd_call(d=320) == fa.FA_ERR_UNSUPPORTED
    assert bwd_call(d=160) == fa.FA_ERR_UNSUPPORTED
    assert bwd_call(d=256, workspace_bytes=1024) == fa.FA_ERR_INVALID_ARG  # 256 is supported
    assert bwd_call(dk=FAKE + 4) == fa.FA_ERR_INVALID_ARG
    assert bwd_call(D=None) == fa.FA_ERR_INVALID_ARG
    assert bwd_call(workspace_bytes=1024) == fa.FA_ERR_INVALID_ARG
    assert bwd_call(grad_dtype=3) == fa.FA_ERR_INVALID_ARG
    assert bwd_call(scale=-1.0) == fa.FA_ERR_UNSUPPORTED
    assert bwd_call(B=0) == fa.FA_OK
    pre = dict(o=FAKE, o_dtype=fa.FA_BF16, dout=FAKE, D=FAKE, workspace=FAKE,
               workspace_bytes=1 << 30, B=2, Hq=4, Hkv=2, N=64, total_tokens=0, d=128, causal=1,
               cu_seqlens=None, deterministic=0, stream=0)
    assert fa.fa_bwd_preprocess(**dict(pre, Hq=5)) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_preprocess(**dict(pre, dout=FAKE + 2)) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_preprocess(**dict(pre, workspace_bytes=64)) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_preprocess(**dict(pre, o_dtype=9)) == fa.FA_ERR_INVALID_ARG


def test_packed_sequence_bound_fits_the_scheduler(L):
    """A packed batch is ranked by one scheduler CTA with 8 bytes per tile level
    of its longest sequence: past 227 KB of shared memory the calls refuse,
    before launching anything, what they would otherwise fail to launch.  The
    level height is the work unit's: 256 rows for the forward up to d = 128,
    128 otherwise.  Inside the bound the arguments pass validation (on a
    machine without a GPU the first CUDA call then fails)."""
    packed = dict(cu_seqlens=FAKE, total_tokens=10)
    assert fwd_call(d=256, N=4_000_000, **packed) == fa.FA_ERR_UNSUPPORTED
    assert fwd_call(d=64, N=8_000_000, **packed) == fa.FA_ERR_UNSUPPORTED
    assert fwd_call(d=64, N=4_000_000, **packed) != fa.FA_ERR_UNSUPPORTED   # 256-row units
    assert fwd_call(d=256, N=3_600_000, **packed) != fa.FA_ERR_UNSUPPORTED
    assert bwd_call(N=4_000_000, **packed) == fa.FA_ERR_UNSUPPORTED
    assert bwd_call(N=3_600_000, **packed) != fa.FA_ERR_UNSUPPORTED
    pre = dict(o=FAKE, o_dtype=fa.FA_BF16, dout=FAKE, D=FAKE, workspace=FAKE,
               workspace_bytes=1 << 30, B=2, Hq=4, Hkv=2, N=4_000_000, total_tokens=10, d=128,
               causal=1, cu_seqlens=FAKE, deterministic=0, stream=0)
    assert fa.fa_bwd_preprocess(**pre) == fa.FA_ERR_UNSUPPORTED
    # dense batches have no such bound (their order is closed-form)
    assert fwd_call(d=256, B=1, N=4_000_000) != fa.FA_ERR_UNSUPPORTED


def fwd_kv_call(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, o_dtype=fa.FA_BF16, lse=FAKE, B=2, Hq=4, Hkv=2,
                Nq=64, total_q=0, Nk=200, total_k=0, d=128, scale=0.125, causal=1,
                cu_seqlens_q=None, cu_seqlens_k=None, workspace=FAKE, workspace_bytes=1 << 20,
                stream=0)
    args.update(kw)
    return fa.fa_fwd_kv(**args)


def test_kv_calls_reject_bad_arguments(L):
    # queries and keys are both dense or both packed
    assert fwd_kv_call(cu_seqlens_q=FAKE, total_q=10) == fa.FA_ERR_INVALID_ARG
    assert fwd_kv_call(cu_seqlens_k=FAKE, total_k=10) == fa.FA_ERR_INVALID_ARG
    assert fwd_kv_call(total_k=300) == fa.FA_ERR_INVALID_ARG    # dense Tk must be B*Nk
    assert fwd_kv_call(Nk=-1) == fa.FA_ERR_INVALID_ARG
    assert fwd_kv_call(d=320) == fa.FA_ERR_UNSUPPORTED
    assert fwd_kv_call(k=FAKE + 8) == fa.FA_ERR_INVALID_ARG
    assert fwd_kv_call(Nq=0) == fa.FA_OK                        # no queries: nothing to do
    pre = dict(o=FAKE, o_dtype=fa.FA_BF16, dout=FAKE, D=FAKE, workspace=FAKE,
               workspace_bytes=1 << 30, B=2, Hq=4, Hkv=2, Nq=64, total_q=0, Nk=200, total_k=0,
               d=128, causal=1, cu_seqlens_q=None, cu_seqlens_k=FAKE, deterministic=0, stream=0)
    assert fa.fa_bwd_kv_preprocess(**pre) == fa.FA_ERR_INVALID_ARG
    bwd = dict(q=FAKE, k=FAKE, v=FAKE, dout=FAKE, lse=FAKE, D=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
               grad_dtype=fa.FA_BF16, workspace=FAKE, workspace_bytes=64, B=2, Hq=4, Hkv=2,
               Nq=64, total_q=0, Nk=200, total_k=0, d=128, scale=0.1, causal=1,
               cu_seqlens_q=None, cu_seqlens_k=None, deterministic=0, stream=0)
    assert fa.fa_bwd_kv(**bwd) == fa.FA_ERR_INVALID_ARG          # workspace too small
    assert fa.fa_bwd_kv(**dict(bwd, Hkv=3)) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_kv(**dict(bwd, B=0)) == fa.FA_OK


def test_kv_workspace_sizes(L):
    Hq, d = 8, 128
    # equal lengths: the same bytes as the equal-length call
    assert fa.fa_bwd_kv_workspace_size(2, Hq, 2, 300, 0, 300, 0, d) == \
        fa.fa_bwd_workspace_size(2, Hq, 2, 300, 0, d)
    # the dQ accumulator covers the queries, the GQA dK/dV partials the keys
    small_k = fa.fa_bwd_kv_workspace_size(2, Hq, 2, 1024, 0, 128, 0, d)
    big_k = fa.fa_bwd_kv_workspace_size(2, Hq, 2, 1024, 0, 4096, 0, d)
    assert big_k - small_k >= 2 * 2 * (4096 - 128) * Hq * d * 4
    assert small_k >= 2 * 1024 * Hq * d * 4


def test_check_status_null(L):
    assert fa.fa_check_device_status(None, 0) == fa.FA_ERR_INVALID_ARG


def test_product_package_does_not_import_oracle():
    """The product path never reaches the oracle (no CPU fallback)."""
    pkg = os.path.join(ROOT, "bwd_tiled_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f


def test_tensor_api_rejects_bad_tensors():
    """The tensor API checks dtype, rank, contiguity and device before any
    library call (these run on CPU tensors: the checks come first)."""
    import torch
    q = torch.zeros(8, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="bfloat16"):
        fa.forward(q.float(), q, q, batch=1)
    with pytest.raises(ValueError, match="contiguous"):
        fa.forward(q, q.transpose(0, 1).contiguous().transpose(0, 1), q, batch=1)
    with pytest.raises(ValueError, match="dimensions"):
        fa.forward(q[0], q, q, batch=1)
    with pytest.raises(ValueError, match="CUDA"):
        fa.forward(q, q, q, batch=1)
    with pytest.raises(ValueError, match="multiple"):
        fa.forward(torch.zeros(8, 3, 64, dtype=torch.bfloat16), q, q, batch=1)
    with pytest.raises(ValueError, match="shape of q"):
        fa.backward(q, q, q, q, q[:4], torch.zeros(2, 8), batch=1)


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "fa.h"

int main(void) {
    /* status strings and workspace sizes need no GPU */
    if (strcmp(fa_status_string(FA_ERR_TIMEOUT), "FA_ERR_TIMEOUT") != 0) return 1;
    size_t f = fa_fwd_workspace_size(4, 16, 2048, 0);
    size_t b = fa_bwd_workspace_size(4, 16, 16, 2048, 0, 128);
    size_t bk = fa_bwd_kv_workspace_size(4, 16, 16, 2048, 0, 2048, 0, 128);
    if (f == 0 || b == 0 || b != bk) return 2;
    /* argument validation returns before any CUDA call */
    void* p = (void*)(size_t)0x10000;
    if (fa_fwd(p, p, p, p, FA_BF16, (float*)p, 2, 4, 3, 64, 0, 64, 0.125f, 1, NULL, p, 1 << 20,
               NULL) != FA_ERR_INVALID_ARG) return 3;
    if (fa_bwd(p, p, p, p, (const float*)p, (const float*)p, p, p, p, FA_BF16, p, 1 << 30, 2, 4,
               2, 64, 0, 320, 0.1f, 0, NULL, 0, NULL) != FA_ERR_UNSUPPORTED) return 4;
    printf("%s\n", fa_version());
    return 0;
}
"""


def test_header_is_plain_c(tmp_path):
    """include/fa.h compiles as C99 with warnings as errors, and a C program
    linked against the library runs the calls that need no GPU."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    fabuild.build()
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    lib = fa.lib_path()
    subprocess.check_call([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I",
                           os.path.join(ROOT, "include"), str(src), "-o", str(exe), lib,
                           "-Wl,-rpath," + os.path.dirname(lib)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, (out.returncode, out.stderr)
    assert out.stdout.startswith("gb300")
