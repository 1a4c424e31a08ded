"""Benchmark: tiled attention forward + backward on GB300.

One step = forward (fa_fwd) + backward (fa_bwd_preprocess + fa_bwd) of the
whole workload, with inputs resident in HBM and the L2 flushed before every
step (a 512 MB write outside the step's events).  Throughput counts the
algorithmic FLOPs 4*B*Hq*N^2*d (forward) and 2.5x that (backward), halved for
causal; a packed variable-length batch uses sum(L_b^2) for B*N^2.  Workloads
with different query and key lengths (fa_fwd_kv / fa_bwd_kv, the causal mask
aligned at the end of the keys) count Lq*Lk per sequence, minus the hidden
triangle Lq^2/2 under the causal mask (Lk^2/2 when Lq > Lk).

Default workload: B=4, Hq=Hkv=16, N=2048, d=128, causal, bf16, seeded N(0,1)
inputs (the mid-size dense configuration, causal).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores

Under torchrun (N > 1) every rank runs its own replica of the workload (the
work partitions by batch/head with no exchange); the job value is the sum of
the ranks' FLOPs over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402  (input generator: no attention arithmetic)

METRIC = "attention fwd+bwd BF16 TFLOPs/s (hd128, causal) and % of GB300 dense BF16 peak"
# --forward-only: the forward alone
METRIC_FWD = "attention fwd BF16 TFLOPs/s and % of GB300 dense BF16 peak"

# DRAM bytes (read + write) of one fa_bwd call -- the backward kernel and its
# dQ conversion -- from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum) of this bench's own command on the same workload,
# with the sha256 (first 16 hex digits) of the sources that build those
# kernels and their schedule at the time of the capture.  When the sources
# have changed since, the figure no longer describes the kernels and the
# bench reports null.
FA_BWD_DRAM = {"mid_causal": {"bytes": 774.9e6, "sources": "f933512058619cac"}}
TRAFFIC_SOURCES = ["bwd_tiled_attention_gb300/csrc/" + f
                   for f in ("bwd.cu", "sched.cu", "api.cu", "common.cuh", "sm100_ptx.cuh",
                             "internal.h")]
NOMINAL_PEAK_TFLOPS = 2250.0


def code_tokens(text):
    """C/C++/CUDA source with its comments removed and every run of whitespace
    made one space: a change to a comment or to the layout leaves it as is,
    a change to the code does not.  String and character literals are kept
    whole (a "//" inside one is not a comment)."""
    out, i, n = [], 0, len(text)
    while i < n:
        ch = text[i]
        if ch in "\"'":
            j = i + 1
            while j < n and text[j] != ch:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(ch)
            i += 1
    return " ".join("".join(out).split())


def sources_sha(files=TRAFFIC_SOURCES):
    """sha256 (first 16 hex digits) of the code of the backward's sources,
    comments and layout excluded."""
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(code_tokens(fh.read()).encode())
            h.update(b"\0")
    return h.hexdigest()[:16]


def bwd_traffic(name):
    """Recorded DRAM bytes of one fa_bwd call on workload `name`, or None when
    none was captured on the current sources."""
    rec = FA_BWD_DRAM.get(name)
    if rec is None or rec["sources"] != sources_sha():
        return None
    return rec["bytes"]


def workload_flops(w, lengths, lengths_k=None):
    if lengths_k is None:
        sq = sum(L * L for L in lengths)
        fwd = 4.0 * w.Hq * sq * w.d
        if w.causal:
            fwd /= 2.0
        return fwd, 2.5 * fwd
    pairs = 0.0
    for lq, lk in zip(lengths, lengths_k):
        if not w.causal:
            pairs += lq * lk
        else:
            pairs += lq * lk - lq * lq / 2.0 if lq <= lk else lk * lk / 2.0
    fwd = 4.0 * w.Hq * pairs * w.d
    return fwd, 2.5 * fwd


def job_throughput(flops_per_rank, elapsed_ms, dist=None, device=None):
    """Whole-job TFLOP/s: every rank's FLOPs over the slowest rank's time.

    With torch.distributed initialised the elapsed time is max-reduced over the
    ranks (the only cross-rank traffic of the benchmark; the attention work
    itself partitions with no exchange).  Returns (tflops, max_elapsed_ms)."""
    world = 1
    if dist is not None and dist.is_initialized():
        import torch
        world = dist.get_world_size()
        t = torch.tensor([float(elapsed_ms)], dtype=torch.float64,
                         device=device if device is not None else "cpu")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
        f = torch.tensor([float(flops_per_rank)], dtype=torch.float64,
                         device=device if device is not None else "cpu")
        dist.all_reduce(f, op=dist.ReduceOp.SUM)
        total = float(f.item())
    else:
        total = float(flops_per_rank) * world
    return total / (elapsed_ms * 1e-3) / 1e12, elapsed_ms


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"fa_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return None

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        sm = [v for v in (num(r[1]) for r in rows) if v is not None]
        mx = [v for v in (num(r[2]) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def cpu_baseline(w, inp, budget_s=12.0):
    """The fp64 oracle on the host cores over a bounded sample of the workload:
    whole (sequence, head) problems, forward + backward, until ~budget_s."""
    import numpy as np

    import oracle

    def f64(t):
        return t.float().numpy().astype(np.float64)

    q, k, v, do = (f64(inp[x]) for x in ("q", "k", "v", "dout"))
    cu = inp["cu_seqlens"].numpy()
    cu_k = inp["cu_seqlens_k"].numpy() if "cu_seqlens_k" in inp else cu
    lengths = inp["lengths"]
    done_flops, heads = 0.0, 0
    grp = w.Hq // w.Hkv
    t0 = time.perf_counter()
    for b in range(len(lengths)):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        k0, k1 = int(cu_k[b]), int(cu_k[b + 1])
        for h in range(w.Hq):
            g = h // grp
            oracle.attention(q[s0:s1, h:h + 1], k[k0:k1, g:g + 1], v[k0:k1, g:g + 1],
                             [0, s1 - s0], w.scale, w.causal, dout=do[s0:s1, h:h + 1],
                             cu_seqlens_k=[0, k1 - k0])
            f, bw = workload_flops(w, [s1 - s0], None if w.lengths_k is None else [k1 - k0])
            done_flops += (f + bw) / w.Hq
            heads += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": done_flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{heads} (sequence, head) problems of the workload, fwd+bwd in fp64, "
                      f"{dt:.1f} s"}


def config_of(w, inp, world):
    lengths = inp["lengths"]
    nk = f" Nk={max(inp['lengths_k'])} (queries end-aligned)" if "lengths_k" in inp else ""
    return {"workload": f"{w.name}: B={w.B} Hq={w.Hq} Hkv={w.Hkv} "
                        f"N={max(lengths)}{nk} d={w.d} {'causal' if w.causal else 'non-causal'}"
                        f"{' deterministic' if w.deterministic else ''}",
            "global_batch": w.B * world, "seq_len": max(lengths), "tokens": sum(lengths) * world,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "flushed before every step (512 MB write, outside the step events)"}


def run_reference(args, w, inp, rank, world):
    if rank != 0:
        return 0
    K, W = args.steps, args.warmup
    for _ in range(min(W, 1)):
        cpu_baseline(w, inp, budget_s=1.0)
    vals = []
    t0 = time.perf_counter()
    for _ in range(K):
        vals.append(cpu_baseline(w, inp, budget_s=args.ref_step_s))
    wall = time.perf_counter() - t0
    value = statistics.mean(v["value"] for v in vals)
    flops_step = sum(workload_flops(w, inp["lengths"], inp.get("lengths_k")))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": flops_step / (value * 1e12) * 1e3 if value > 0 else None,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), bf16-rounded)", "config": config_of(w, inp, world),
        "cpu_baseline": dict(vals[-1], value=value),
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "wall_s": wall,
    }
    print(json.dumps(line), flush=True)
    return 0


class Runner:
    """One workload resident on the device: inputs, outputs and workspaces
    allocated once; step() runs the forward (fa_fwd) and the backward
    (fa_bwd_preprocess, fa_bwd) through the C ABI on the current stream."""

    def __init__(self, fa, w, inp, dev, forward_only=False):
        import torch
        self.fa, self.w, self.inp, self.dev = fa, w, inp, dev
        self.forward_only = forward_only
        lengths = inp["lengths"]
        lengths_k = inp.get("lengths_k")          # None: keys as long as the queries
        self.kv = kv = lengths_k is not None
        self.B, self.Hq, self.Hkv, self.d = w.B, w.Hq, w.Hkv, w.d
        self.N, self.T = max(lengths), sum(lengths)
        self.Nk, self.Tk = (max(lengths_k), sum(lengths_k)) if kv else (self.N, self.T)
        varlen = (w.len_range is not None or len(set(lengths)) > 1
                  or (kv and len(set(lengths_k)) > 1))
        self.x = {k: inp[k].to(dev) for k in ("q", "k", "v", "dout")}
        self.cu = inp["cu_seqlens"].to(dev) if varlen else None
        self.cu_k = inp["cu_seqlens_k"].to(dev) if (varlen and kv) else None
        T, Hq, d = self.T, self.Hq, self.d
        self.o = torch.empty((T, Hq, d), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((Hq, T), dtype=torch.float32, device=dev)
        self.D = torch.empty((Hq, T), dtype=torch.float32, device=dev)
        self.grads = (torch.empty_like(self.x["q"]), torch.empty_like(self.x["k"]),
                      torch.empty_like(self.x["v"]))
        self.fws_b = fa.fa_fwd_workspace_size(self.B, Hq, self.N, T)
        self.bws_b = (fa.fa_bwd_kv_workspace_size(self.B, Hq, self.Hkv, self.N, T, self.Nk,
                                                  self.Tk, d) if kv
                      else fa.fa_bwd_workspace_size(self.B, Hq, self.Hkv, self.N, T, d))
        self.fws = torch.empty(self.fws_b, dtype=torch.uint8, device=dev)
        self.bws = torch.empty(self.bws_b, dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream()
        self.det = bool(w.deterministic)
        self.fl_f, self.fl_b = workload_flops(w, lengths, lengths_k)
        if forward_only:
            self.fl_b = 0.0
        # kernels per step: scheduler + forward, then scheduler + preprocess and
        # backward + dQ conversion
        self.launches_per_step = 2 if forward_only else 6
        self.status_ws = self.fws if forward_only else self.bws

    def check(self, st, what):
        if st != self.fa.FA_OK:
            raise self.fa.FAError(st, what)

    def step(self, events=None, xin=None, grads=None):
        fa, w, s = self.fa, self.w, self.stream
        xi = self.x if xin is None else xin
        gq, gk, gv = self.grads if grads is None else grads
        B, Hq, Hkv, N, T, Nk, Tk, d = (self.B, self.Hq, self.Hkv, self.N, self.T, self.Nk,
                                       self.Tk, self.d)
        o, lse, Dv, cu, cu_k = self.o, self.lse, self.D, self.cu, self.cu_k
        if events:
            events[0].record(s)
        if self.kv:
            self.check(fa.fa_fwd_kv(xi["q"], xi["k"], xi["v"], o, fa.FA_BF16, lse, B, Hq, Hkv, N,
                                    T, Nk, Tk, d, w.scale, w.causal, cu, cu_k, self.fws,
                                    self.fws_b, s), "fa_fwd_kv")
        else:
            self.check(fa.fa_fwd(xi["q"], xi["k"], xi["v"], o, fa.FA_BF16, lse, B, Hq, Hkv, N, T,
                                 d, w.scale, w.causal, cu, self.fws, self.fws_b, s), "fa_fwd")
        if events:
            events[1].record(s)
        if self.forward_only:
            if events:
                events[2].record(s)
                events[3].record(s)
            return
        if self.kv:
            self.check(fa.fa_bwd_kv_preprocess(o, fa.FA_BF16, xi["dout"], Dv, self.bws,
                                               self.bws_b, B, Hq, Hkv, N, T, Nk, Tk, d, w.causal,
                                               cu, cu_k, self.det, s), "fa_bwd_kv_preprocess")
        else:
            self.check(fa.fa_bwd_preprocess(o, fa.FA_BF16, xi["dout"], Dv, self.bws, self.bws_b,
                                            B, Hq, Hkv, N, T, d, w.causal, cu, self.det, s),
                       "fa_bwd_preprocess")
        if events:
            events[2].record(s)
        if self.kv:
            self.check(fa.fa_bwd_kv(xi["q"], xi["k"], xi["v"], xi["dout"], lse, Dv, gq, gk, gv,
                                    fa.FA_BF16, self.bws, self.bws_b, B, Hq, Hkv, N, T, Nk, Tk, d,
                                    w.scale, w.causal, cu, cu_k, self.det, s), "fa_bwd_kv")
        else:
            self.check(fa.fa_bwd(xi["q"], xi["k"], xi["v"], xi["dout"], lse, Dv, gq, gk, gv,
                                 fa.FA_BF16, self.bws, self.bws_b, B, Hq, Hkv, N, T, d, w.scale,
                                 w.causal, cu, self.det, s), "fa_bwd")
        if events:
            events[3].record(s)

    def warmup(self, W, flush):
        """W untimed steps (at least 3), each after an L2 flush; returns the
        mean device time of a step in ms (from the last ones)."""
        import torch
        W = max(W, 3)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(W)]
        for i in range(W):
            flush.zero_()
            self.step(evs[i])
        torch.cuda.synchronize()
        self.check(self.fa.fa_check_device_status(self.status_ws, self.stream), "device status")
        tail = evs[1:] if W > 1 else evs
        return statistics.mean(e[0].elapsed_time(e[3]) for e in tail)

    def timed(self, K, flush, dist=None, gpu_index=0):
        """Exactly K steps, each after an L2 flush outside its events, bracketed
        by a barrier and a device synchronisation, with the clocks sampled
        throughout.  Returns per-step times (ms) of the forward, the
        preprocess, the fa_bwd call and the whole step, and the clock record."""
        import torch
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
        sampler = ClockSampler(gpu_index)
        sampler.start()
        time.sleep(0.3)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(K):
            flush.zero_()
            self.step(evs[i])
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        clocks = sampler.stop()
        self.check(self.fa.fa_check_device_status(self.status_ws, self.stream), "device status")
        return dict(fwd=[e[0].elapsed_time(e[1]) for e in evs],
                    pre=[e[1].elapsed_time(e[2]) for e in evs],
                    bwd=[e[2].elapsed_time(e[3]) for e in evs],
                    step=[e[0].elapsed_time(e[3]) for e in evs], clocks=clocks)


def steps_for(step_ms, target_s, lo=20, hi=20000):
    """Steps whose device time (plus the L2 flush between them, ~0.1 ms) fills
    about target_s seconds, so the 50 ms clock sampler sees the load."""
    import math
    return int(min(hi, max(lo, math.ceil(target_s * 1e3 / (step_ms + 0.1)))))


def rates(r, t):
    """TFLOP/s and percentages of a Runner's timed steps."""
    peaks, _ = measured_peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))
    fwd_ms, pre_ms, bwd_ms = (statistics.mean(t[k]) for k in ("fwd", "pre", "bwd"))
    step_ms = statistics.mean(t["step"])
    out = {"fwd_ms": fwd_ms, "fwd_tflops": r.fl_f / (fwd_ms * 1e-3) / 1e12}
    out["fwd_pct_nominal"] = 100.0 * out["fwd_tflops"] / NOMINAL_PEAK_TFLOPS
    out["fwd_pct_measured"] = 100.0 * out["fwd_tflops"] / peak
    if r.fl_b > 0:
        out.update({
            "bwd_preprocess_ms": pre_ms, "bwd_ms": bwd_ms,
            "bwd_tflops": r.fl_b / (bwd_ms * 1e-3) / 1e12,
            "bwd_tflops_incl_preprocess": r.fl_b / ((pre_ms + bwd_ms) * 1e-3) / 1e12,
            "step_ms": step_ms, "step_tflops": (r.fl_f + r.fl_b) / (step_ms * 1e-3) / 1e12})
        out["bwd_pct_nominal"] = 100.0 * out["bwd_tflops"] / NOMINAL_PEAK_TFLOPS
        out["bwd_pct_measured"] = 100.0 * out["bwd_tflops"] / peak
        out["step_pct_nominal"] = 100.0 * out["step_tflops"] / NOMINAL_PEAK_TFLOPS
    return out


# The other configurations of the tiled-attention workloads, each timed the way
# the headline is (L2 flushed before every step, CUDA events, >= 1 s of steps):
# the small, dense, long, grouped and packed deterministic ones, then other
# head dimensions and queries shorter than keys.
PER_CONFIG = ["tiny", "mid_dense", "long_causal", "gqa8_causal", "mqa_causal", "varlen_det",
              "mid_causal_d64", "mid_causal_d96", "mid_causal_d192", "mid_causal_d256",
              "chunk_causal"]


def per_config(fa, dev, flush, local, names=PER_CONFIG, target_s=1.0):
    import torch
    out = {}
    for name in names:
        w = synth.workloads()[name]
        inp = synth.make_workload(w)
        r = Runner(fa, w, inp, dev)
        step_ms = r.warmup(3, flush)
        K = steps_for(step_ms, target_s, lo=10)
        t = r.timed(K, flush, gpu_index=local)
        rec = rates(r, t)
        rec.update(steps=K, config=config_of(w, inp, 1)["workload"], clocks=t["clocks"],
                   deterministic=r.det)
        out[name] = rec
        del r, inp
        torch.cuda.empty_cache()
    return out


def report_forward_only(args, r, world, rank, K, value, ms_per_step, t, dist):
    """JSON line of a --forward-only run: the forward's TFLOP/s and its roofline."""
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))
    achieved = r.fl_f / (statistics.mean(t["fwd"]) * 1e-3) / 1e12
    line = {
        "metric": METRIC_FWD, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), bf16-rounded)", "config": config_of(r.w, r.inp, world),
        "pct_of_nominal_peak": 100.0 * value / world / NOMINAL_PEAK_TFLOPS,
        "pct_of_measured_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "tensor", "kernel": "fa_fwd (scheduler + forward kernel)",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} bf16 burst",
                     "traffic": None},
        "e2e": None, "gpu_launches": r.launches_per_step * K, "clocks": t["clocks"],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def e2e_through_api(r, E, dist, dev):
    """End to end through the public API with host buffers: every step copies
    its inputs host -> device, runs fwd + bwd and copies the gradients back.
    The copies run on their own streams with two buffer sets, so step i+1's
    upload and step i-1's download overlap step i's compute; events keep each
    buffer's writer after its last reader.  Returns (TFLOP/s, h2d, d2h bytes)."""
    import torch
    inp, x, stream = r.inp, r.x, r.stream
    host_in = {k: inp[k].pin_memory() for k in ("q", "k", "v", "dout")}
    host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in r.grads]
                for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    xs = [x, {k: torch.empty_like(x[k]) for k in x}]
    gs = [r.grads, tuple(torch.empty_like(t) for t in r.grads)]
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_h2d = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_d2h = [torch.cuda.Event() for _ in range(2)]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for i in range(E + 2):
        sl = i & 1
        if i == 2:  # the first two steps fill the pipeline, untimed
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            e0.record(stream)
            s_h2d.wait_event(e0)
        with torch.cuda.stream(s_h2d):
            if i >= 2:
                s_h2d.wait_event(ev_comp[sl])  # step i-2 has read this input set
            for k_ in ("q", "k", "v", "dout"):
                xs[sl][k_].copy_(host_in[k_], non_blocking=True)
            ev_h2d[sl].record(s_h2d)
        stream.wait_event(ev_h2d[sl])
        if i >= 2:
            stream.wait_event(ev_d2h[sl])  # step i-2's gradients have been copied out
        r.step(xin=xs[sl], grads=gs[sl])
        ev_comp[sl].record(stream)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev_comp[sl])
            for src, dst in zip(gs[sl], host_out[sl]):
                dst.copy_(src, non_blocking=True)
            ev_d2h[sl].record(s_d2h)
    for sl in range(2):
        stream.wait_event(ev_d2h[sl])
    e1.record(stream)
    torch.cuda.synchronize()
    value, _ = job_throughput((r.fl_f + r.fl_b) * E, e0.elapsed_time(e1), dist, dev)
    return value, h2d, d2h


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for ~2 s of device time)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="mid_causal", choices=sorted(synth.workloads()))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--ref-step-s", type=float, default=4.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing the other configurations")
    ap.add_argument("--forward-only", action="store_true",
                    help="time the forward alone (no end-to-end leg, no CPU baseline)")
    ap.add_argument("--deterministic", action="store_true",
                    help="run the backward in deterministic mode whatever the workload's default")
    ap.add_argument("--atomic", action="store_true",
                    help="run the backward in atomic mode whatever the workload's default")
    args = ap.parse_args()
    if args.deterministic and args.atomic:
        ap.error("--deterministic and --atomic exclude each other")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = synth.workloads()[args.workload]
    if args.deterministic:
        w.deterministic = True
    if args.atomic:
        w.deterministic = False
    inp = synth.make_workload(w)

    if args.impl == "reference":
        if args.steps is None:
            args.steps = 3
        return run_reference(args, w, inp, rank, world)

    import torch

    import bwd_tiled_attention_gb300 as fa
    from bwd_tiled_attention_gb300 import build as fabuild
    fabuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    r = Runner(fa, w, inp, dev, forward_only=args.forward_only)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    step_ms = r.warmup(args.warmup, flush)
    K = args.steps
    if K is None:
        K = steps_for(step_ms, 2.0, lo=200)
        if dist:  # every rank times the same number of steps
            kt = torch.tensor([K], dtype=torch.int64, device=dev)
            dist.all_reduce(kt, op=dist.ReduceOp.MAX)
            K = int(kt.item())
    t = r.timed(K, flush, dist, local)
    value, total_ms = job_throughput((r.fl_f + r.fl_b) * K, sum(t["step"]), dist, dev)
    ms_per_step = total_ms / K
    if args.forward_only:
        return report_forward_only(args, r, world, rank, K, value, ms_per_step, t, dist)

    e2e_value, h2d, d2h = e2e_through_api(r, args.e2e_steps, dist, dev)

    peaks, peak_kind = measured_peaks()
    rt = rates(r, t)
    peak = float(peaks.get("bf16_tflops", 1900.0))
    achieved = rt["bwd_tflops"]
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), bf16-rounded)",
        "config": config_of(w, inp, world),
        "pct_of_nominal_peak": 100.0 * value / world / NOMINAL_PEAK_TFLOPS,
        "pct_of_measured_peak": 100.0 * value / world / peak,
        "breakdown": {k: rt[k] for k in ("fwd_ms", "bwd_preprocess_ms", "bwd_ms", "fwd_tflops",
                                          "bwd_tflops", "bwd_tflops_incl_preprocess")},
        "roofline": {"bound": "tensor", "kernel": "fa_bwd (backward kernel + dQ conversion)",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} bf16 burst",
                     "traffic": bwd_traffic(w.name), "sources": sources_sha()},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": r.launches_per_step * K,
        "clocks": t["clocks"],
    }
    if world == 1 and not args.no_per_config:
        del r
        torch.cuda.empty_cache()
        line["per_config"] = per_config(fa, dev, flush, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
