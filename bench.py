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
# --forward-only (head dimensions 192 and 256 have no backward)
METRIC_FWD = "attention fwd BF16 TFLOPs/s and % of GB300 dense BF16 peak"

# DRAM bytes (read + write) of one fa_bwd call -- the backward kernel and its
# dQ conversion -- from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum) of this bench's own command on the same workload,
# for the kernels as they are; a workload without a capture reports null.
FA_BWD_DRAM_BYTES = {"mid_causal": 775.6e6, "chunk_causal": 5188e6}
NOMINAL_PEAK_TFLOPS = 2250.0


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


def report_forward_only(args, w, inp, world, rank, K, value, ms_per_step, fl_f, fwd_ms,
                        launches_per_step, clocks, dist):
    """JSON line of a --forward-only run: the forward's TFLOP/s and its roofline."""
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))
    achieved = fl_f / (fwd_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC_FWD, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), bf16-rounded)", "config": config_of(w, inp, world),
        "pct_of_nominal_peak": 100.0 * value / world / NOMINAL_PEAK_TFLOPS,
        "pct_of_measured_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "tensor", "kernel": "fa_fwd (scheduler + forward kernel)",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} bf16 burst",
                     "traffic": None},
        "e2e": None, "gpu_launches": launches_per_step * K, "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="mid_causal", choices=sorted(synth.workloads()))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--ref-step-s", type=float, default=4.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--forward-only", action="store_true",
                    help="time the forward alone (no end-to-end leg, no CPU baseline)")
    ap.add_argument("--deterministic", action="store_true",
                    help="run the backward in deterministic mode whatever the workload's default")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = synth.workloads()[args.workload]
    if args.deterministic:
        w.deterministic = True
    inp = synth.make_workload(w)

    if args.impl == "reference":
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

    lengths = inp["lengths"]
    lengths_k = inp.get("lengths_k")          # None: keys as long as the queries
    kv = lengths_k is not None
    B, Hq, Hkv, d = w.B, w.Hq, w.Hkv, w.d
    N, T = max(lengths), sum(lengths)
    Nk, Tk = (max(lengths_k), sum(lengths_k)) if kv else (N, T)
    scale = w.scale
    varlen = w.len_range is not None or len(set(lengths)) > 1 or (kv and len(set(lengths_k)) > 1)
    x = {k: inp[k].to(dev) for k in ("q", "k", "v", "dout")}
    cu = inp["cu_seqlens"].to(dev) if varlen else None
    cu_k = inp["cu_seqlens_k"].to(dev) if (varlen and kv) else None
    o = torch.empty((T, Hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Hq, T), dtype=torch.float32, device=dev)
    Dv = torch.empty((Hq, T), dtype=torch.float32, device=dev)
    dq = torch.empty_like(x["q"])
    dk = torch.empty_like(x["k"])
    dv = torch.empty_like(x["v"])
    fws_b = fa.fa_fwd_workspace_size(B, Hq, N, T)
    bws_b = (fa.fa_bwd_kv_workspace_size(B, Hq, Hkv, N, T, Nk, Tk, d) if kv
             else fa.fa_bwd_workspace_size(B, Hq, Hkv, N, T, d))
    fws = torch.empty(fws_b, dtype=torch.uint8, device=dev)
    bws = torch.empty(bws_b, dtype=torch.uint8, device=dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    det = bool(w.deterministic)

    def check(st, what):
        if st != fa.FA_OK:
            raise fa.FAError(st, what)

    def step(events=None, xin=None, grads=None):
        xi = x if xin is None else xin
        gq, gk, gv = (dq, dk, dv) if grads is None else grads
        if events:
            events[0].record(stream)
        if kv:
            check(fa.fa_fwd_kv(xi["q"], xi["k"], xi["v"], o, fa.FA_BF16, lse, B, Hq, Hkv, N, T, Nk,
                               Tk, d, scale, w.causal, cu, cu_k, fws, fws_b, stream), "fa_fwd_kv")
        else:
            check(fa.fa_fwd(xi["q"], xi["k"], xi["v"], o, fa.FA_BF16, lse, B, Hq, Hkv, N, T, d,
                            scale, w.causal, cu, fws, fws_b, stream), "fa_fwd")
        if events:
            events[1].record(stream)
        if args.forward_only:
            if events:
                events[2].record(stream)
                events[3].record(stream)
            return
        if kv:
            check(fa.fa_bwd_kv_preprocess(o, fa.FA_BF16, xi["dout"], Dv, bws, bws_b, B, Hq, Hkv, N,
                                          T, Nk, Tk, d, w.causal, cu, cu_k, det, stream),
                  "fa_bwd_kv_preprocess")
        else:
            check(fa.fa_bwd_preprocess(o, fa.FA_BF16, xi["dout"], Dv, bws, bws_b, B, Hq, Hkv, N, T,
                                       d, w.causal, cu, det, stream), "fa_bwd_preprocess")
        if events:
            events[2].record(stream)
        if kv:
            check(fa.fa_bwd_kv(xi["q"], xi["k"], xi["v"], xi["dout"], lse, Dv, gq, gk, gv,
                               fa.FA_BF16, bws, bws_b, B, Hq, Hkv, N, T, Nk, Tk, d, scale,
                               w.causal, cu, cu_k, det, stream), "fa_bwd_kv")
        else:
            check(fa.fa_bwd(xi["q"], xi["k"], xi["v"], xi["dout"], lse, Dv, gq, gk, gv,
                            fa.FA_BF16, bws, bws_b, B, Hq, Hkv, N, T, d, scale, w.causal, cu, det,
                            stream), "fa_bwd")
        if events:
            events[3].record(stream)

    # scheduler + fwd, scheduler + preprocess, bwd + postprocess
    launches_per_step = 2 if args.forward_only else 6
    status_ws = fws if args.forward_only else bws
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    check(fa.fa_check_device_status(status_ws, stream), "device status")

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(K):
        flush.zero_()
        step(evs[i])
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    check(fa.fa_check_device_status(status_ws, stream), "device status")
    t_fwd = [e[0].elapsed_time(e[1]) for e in evs]
    t_pre = [e[1].elapsed_time(e[2]) for e in evs]
    t_bwd = [e[2].elapsed_time(e[3]) for e in evs]
    t_step = [e[0].elapsed_time(e[3]) for e in evs]
    fl_f, fl_b = workload_flops(w, lengths, lengths_k)
    if args.forward_only:
        fl_b = 0.0
    value, total_ms = job_throughput((fl_f + fl_b) * K, sum(t_step), dist, dev)
    ms_per_step = total_ms / K
    if args.forward_only:
        return report_forward_only(args, w, inp, world, rank, K, value, ms_per_step, fl_f,
                                   statistics.mean(t_fwd), launches_per_step, clocks, dist)

    # End to end through the public API with host buffers: every step copies
    # its inputs host -> device, runs fwd + bwd and copies the gradients back.
    # The copies run on their own streams with two buffer sets, so step i+1's
    # upload and step i-1's download overlap step i's compute; events keep
    # each buffer's writer after its last reader.
    host_in = {k: inp[k].pin_memory() for k in ("q", "k", "v", "dout")}
    host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv)]
                for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    xs = [x, {k: torch.empty_like(x[k]) for k in x}]
    gs = [(dq, dk, dv), tuple(torch.empty_like(t) for t in (dq, dk, dv))]
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_h2d = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_d2h = [torch.cuda.Event() for _ in range(2)]
    E = args.e2e_steps
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
        step(xin=xs[sl], grads=gs[sl])
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
    e2e_value, _ = job_throughput((fl_f + fl_b) * E, e0.elapsed_time(e1), dist, dev)

    peaks, peak_kind = measured_peaks()
    bwd_call_ms = statistics.mean(t_bwd)
    achieved = fl_b / (bwd_call_ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", 1900.0))
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), bf16-rounded)",
        "config": config_of(w, inp, world),
        "pct_of_nominal_peak": 100.0 * value / world / NOMINAL_PEAK_TFLOPS,
        "pct_of_measured_peak": 100.0 * value / world / peak,
        "breakdown": {
            "fwd_ms": statistics.mean(t_fwd), "bwd_preprocess_ms": statistics.mean(t_pre),
            "bwd_ms": bwd_call_ms,
            "fwd_tflops": fl_f / (statistics.mean(t_fwd) * 1e-3) / 1e12,
            "bwd_tflops_incl_preprocess": fl_b / ((statistics.mean(t_pre) + bwd_call_ms) * 1e-3)
            / 1e12,
        },
        "roofline": {"bound": "tensor", "kernel": "fa_bwd (backward kernel + dQ conversion)",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} bf16 burst",
                     "traffic": FA_BWD_DRAM_BYTES.get(w.name)},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
