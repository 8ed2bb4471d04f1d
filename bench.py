#!/usr/bin/env python
"""Throughput of one GMM EM step on a B300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload embed_10m]

A step is one EM iteration over the whole data set: parameter preparation,
the fused logit / log-sum-exp / statistics kernel, the fixed-order reduction
and the M-step.  The default workload is the 10M x 128 x 1024 diagonal model
on bf16 embedding-like data (inputs larger than L2, so no flush is needed).
With --gpus N > 1 (launched by torchrun) every rank runs an independent
replica; nothing is exchanged on the data path, only the timing maximum.

--impl reference times the float64 CPU oracle on a bounded prefix of the
same workload per step and scales it to the full N (EM cost is linear in N).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "EM iter/s and N·K·D/s at N=10M,D=128,K=1024 diag; % tensor-core peak"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# dram__bytes_read.sum + dram__bytes_write.sum of one fused-kernel launch on the
# full 10M x 128 workload: 303.5 MB (296.2 read + 7.3 written) measured on its
# first 1M rows, times 10 (traffic grows in proportion to the rows)
TRAFFIC_EMBED_10M = 3.035e9
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    def __init__(self, dev_index: int):
        self.dev = dev_index
        self.proc = None
        out = os.environ.get("GMM_BENCH_CLOCKS_DIR", os.path.join(ROOT, "bench_out"))
        self.path = os.path.join(out, f"clocks_rank{dev_index}.csv")

    def __enter__(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.dev)], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, x: float) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_em_step(X, init, cov):
    import oracle
    if cov == "tied":
        return oracle.tied.em_step(X.astype("float64"), *init)
    return oracle.em_step(X, *init, cov)


def oracle_rows_for(w, seconds: float, X_host_prefix, init, probe_rows=1000):
    """Rows of the workload the oracle handles in about `seconds`."""
    probe = min(probe_rows, X_host_prefix.shape[0])
    t0 = time.perf_counter()
    oracle_em_step(X_host_prefix[:probe], init, w.cov)
    dt = max(time.perf_counter() - t0, 1e-3)
    return int(max(probe, min(X_host_prefix.shape[0], probe * seconds / dt)))


def cpu_oracle_step(w, X_host, init, rows):
    t0 = time.perf_counter()
    oracle_em_step(X_host[:rows], init, w.cov)
    return time.perf_counter() - t0


def run_reference(args, w, ws, rank):
    """The float64 CPU oracle as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    cap = min(w.N, 400_000)
    X = W.make_data(w, cap, device=dev)
    init = W.make_init(w, X)
    Xh = X.float().cpu().numpy()
    rows = oracle_rows_for(w, args.ref_step_seconds, Xh, init)
    for _ in range(args.warmup if args.warmup < 1 else 1):
        cpu_oracle_step(w, Xh, init, min(rows, 1000))
    times = [cpu_oracle_step(w, Xh, init, rows) for _ in range(args.steps)]
    per_full = statistics.mean(times) * (w.N / rows)
    value = 1.0 / per_full
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "EM iter/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_full * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, "oracle"),
        "extrapolated": rows < w.N,
        "cpu_baseline": {"value": value, "unit": "EM iter/s", "cores": oracle.threads(),
                         "kind": "oracle", "extrapolated": rows < w.N,
                         "sample": f"1 EM step on the first {rows} rows per step, scaled by N/{rows}"},
        "e2e": {"value": value, "unit": "EM iter/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w, precision, plan="auto"):
    return {"workload": w.name, "N": w.N, "D": w.D, "K": w.K, "cov": w.cov, "x_dtype": w.x_dtype,
            "precision": precision, "plan": plan, "parallelism": "replicas",
            "l2": "inputs larger than L2 (no flush)" if w.N * w.D * (2 if w.x_dtype == "bf16" else 4) > 126e6
            else "L2 flushed between steps"}


def run_ours(args, w, ws, rank, local):
    import em_gmm_step_02_b300 as G
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    X = W.make_data(w, device=dev)
    lw0, mu0, var0 = W.make_init(w, X)
    p = [torch.tensor(a, device=dev) for a in (lw0, mu0, var0)]
    x_bytes = X.numel() * X.element_size()
    flush = None
    if x_bytes <= 126e6:
        flush = torch.empty(int(256e6) // 4, dtype=torch.float32, device=dev)
    opts = G.gmm_default_opts(precision=args.precision, plan=args.plan)
    G.gmm_reserve(w.N, w.D, w.K, w.cov, w.x_dtype, precision=args.precision, plan=args.plan)

    def step():
        if flush is not None:
            flush.add_(1.0)
        return G.gmm_em_step(X, *p, w.cov, out=p, opts=opts)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert G.gmm_stream_status() == 0, G.gmm_last_error()

    stream = torch.cuda.current_stream(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    launches = 0
    barrier(ws)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        G.gmm_profile_begin()
        e0.record(stream)
        for _ in range(args.steps):
            step()
            launches += G.gmm_last_launch_count()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        main_ms, main_launches = G.gmm_profile_end()
    barrier(ws)
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(ws, ms)
    status = G.gmm_stream_status()
    assert status == 0, G.gmm_last_error()

    # the workload's final top-m soft assignment, timed on its own
    topm = None
    if w.topm > 0 and not args.no_topm:
        def time_topm(o):
            G.gmm_predict_topm(X, *p, w.cov, w.topm, opts=o)
            torch.cuda.synchronize(dev)
            assert G.gmm_stream_status() == 0, G.gmm_last_error()
            reps = 3
            e0.record(stream)
            for _ in range(reps):
                G.gmm_predict_topm(X, *p, w.cov, w.topm, opts=o)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            return e0.elapsed_time(e1) / reps

        t_ms = time_topm(opts)
        topm = {"m": w.topm, "ms": t_ms, "points_per_s": w.N * 1e3 / t_ms,
                "logit_tflops": 4.0 * w.N * w.K * w.D / (t_ms * 1e-3) / 1e12,
                "job_ms": w.iters * ms + t_ms,
                "job": f"{w.iters} EM iterations + top-{w.topm}"}
        if w.cov != "tied":
            # the same pass with the direct-form refinement of the candidates
            # switched on (the default refines on PRECISE only)
            o_ref = G.gmm_default_opts(precision=args.precision, plan=args.plan, topm_refine="on")
            topm["refine_on_ms"] = time_topm(o_ref)

    # approximate top-k EM (k = the workload's m): one EM step whose E-step
    # keeps each point's k largest logits, from the same parameters
    topk = None
    if w.topm > 0 and not args.no_topm and w.cov != "tied":
        kout = [torch.empty_like(a) for a in p]
        opts_k = G.gmm_default_opts(precision=args.precision, plan=args.plan, approx_top_k=w.topm)
        G.gmm_em_step(X, *p, w.cov, out=kout, opts=opts_k)
        torch.cuda.synchronize(dev)
        assert G.gmm_stream_status() == 0, G.gmm_last_error()
        reps = 3
        e0.record(stream)
        for _ in range(reps):
            G.gmm_em_step(X, *p, w.cov, out=kout, opts=opts_k)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        k_ms = e0.elapsed_time(e1) / reps
        topk = {"k": w.topm, "ms_per_step": k_ms, "iter_per_s": 1e3 / k_ms,
                "api": "gmm_em_step with opts.approx_top_k = k"}
        del kout

    # threshold multi-assignment (compressed rows) of the same final pass:
    # pairs with r >= 1/(m+1), at most m per point, so nothing is cut by the cap
    thresh = None
    if w.topm > 0 and not args.no_topm:
        tau = 1.0 / (w.topm + 1) + 1e-6
        G.gmm_assign_threshold(X, *p, w.cov, tau=tau, max_per_point=w.topm, opts=opts)
        torch.cuda.synchronize(dev)
        assert G.gmm_stream_status() == 0, G.gmm_last_error()
        reps = 3
        e0.record(stream)
        for _ in range(reps):
            off, _, _ = G.gmm_assign_threshold(X, *p, w.cov, tau=tau, max_per_point=w.topm,
                                               capacity=w.N * w.topm, opts=opts)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        thresh = {"tau": tau, "max_per_point": w.topm, "ms": e0.elapsed_time(e1) / reps,
                  "entries": int(off[-1].item())}

    # end to end through the public API with host buffers: X streams from
    # pinned host memory in chunks whose copies overlap the fused kernel
    # (gmm_em_step_host); parameters go up and results come back every step
    e2e = None
    if not args.no_e2e and w.cov != "tied":      # the host-data entry point takes spherical / diagonal
        Xh = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
        Xh.copy_(X)
        amax = float(X.abs().max().item()) * 1.0001    # the caller's bound on |X|, found once
        opts_h = G.gmm_default_opts(precision=args.precision, plan=args.plan, x_absmax=amax)
        ph = [a.cpu().pin_memory() for a in p]
        outh = [torch.empty_like(a).pin_memory() for a in ph]
        llh = torch.empty(1, dtype=torch.float64).pin_memory()
        pd = [torch.empty_like(a) for a in p]
        h2d = Xh.numel() * Xh.element_size() + sum(a.numel() * a.element_size() for a in ph)
        d2h = sum(a.numel() * a.element_size() for a in outh) + 8

        def step_host():
            for d_, h_ in zip(pd, ph):
                d_.copy_(h_, non_blocking=True)
            *o, ll = G.gmm_em_step_host(Xh, *pd, w.cov, out=pd, opts=opts_h)
            for h_, d_ in zip(outh, o):
                h_.copy_(d_, non_blocking=True)
            llh.copy_(ll, non_blocking=True)

        step_host()
        torch.cuda.synchronize(dev)
        assert G.gmm_stream_status() == 0, G.gmm_last_error()
        barrier(ws)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            step_host()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(ws, e0.elapsed_time(e1) / args.steps)
        e2e = {"value": ws * 1e3 / e2e_ms, "unit": "EM iter/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h),
               "api": "gmm_em_step_host: X from pinned host memory in chunks of the default 1M rows, copies overlapped"}
        del Xh

    if rank != 0:
        return
    peaks, peaks_kind = load_peaks()
    flops = 8.0 * w.N * w.K * w.D
    per_launch_ms = main_ms / max(1, main_launches)
    launches_per_step = max(1, main_launches // args.steps)
    achieved = flops / launches_per_step / (per_launch_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    # DRAM bytes per launch of the fused kernel from the committed ncu capture
    # (1M rows of this workload, scaled by rows: traffic grows with N); only
    # for the configuration that capture was taken of
    traffic = None
    if (w.name == "embed_10m" and args.plan in ("auto", "cluster") and args.precision == "auto"
            and not args.rows):
        traffic = TRAFFIC_EMBED_10M
    line = {
        "metric": METRIC, "value": ws * 1e3 / ms_max, "unit": "EM iter/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic", "config": config_of(w, args.precision, args.plan),
        "nkd_per_s": ws * w.N * w.K * w.D * 1e3 / ms_max,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "traffic_source": "ncu dram__bytes_read+write, 1M-row capture x 10" if traffic else None,
                     "kernel": "fused_em_kernel", "launch_ms": per_launch_ms,
                     "peak_source": f"{peaks_kind} bf16 burst (fp16 has the same nominal rate)",
                     "work": "8*N*K*D MMA flops per step"},
        "hbm": {"x_bytes_per_step": x_bytes, "gbs": x_bytes / (ms_max * 1e-3) / 1e9,
                "peak_gbs": float(peaks["hbm_gbs"])},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "plan": G.gmm_plan_info(w.N, w.D, w.K, w.cov, w.x_dtype, precision=args.precision, plan=args.plan),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if thresh is not None:
        line["threshold"] = thresh
    if topm is not None:
        line["topm"] = topm
    if topk is not None:
        line["approx_top_k"] = topk
    if not args.no_cpu and ws == 1:
        import oracle
        cap = min(w.N, 400_000)
        Xh = X[:cap].float().cpu().numpy()
        init = (lw0, mu0, var0)
        rows = oracle_rows_for(w, args.cpu_seconds, Xh, init)
        t = cpu_oracle_step(w, Xh, init, rows)
        line["cpu_baseline"] = {"value": 1.0 / (t * w.N / rows), "unit": "EM iter/s",
                                "cores": oracle.threads(), "kind": "oracle", "extrapolated": rows < w.N,
                                "sample": f"1 EM step on the first {rows} rows, scaled by N/{rows}"}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="embed_10m", choices=sorted(W.WORKLOADS))
    ap.add_argument("--precision", default="auto", choices=["auto", "fast", "precise"])
    ap.add_argument("--plan", default="auto", choices=["auto", "cluster", "split"])
    ap.add_argument("--rows", type=int, default=0,
                    help="run on the first ROWS rows of the workload (profiling a smaller case)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-topm", action="store_true")
    ap.add_argument("--cov", default=None, choices=["spherical", "diag", "tied"],
                    help="run the workload's data with this covariance type instead")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-step-seconds", type=float, default=8.0)
    args = ap.parse_args()
    w = W.WORKLOADS[args.workload]
    if args.cov and args.cov != w.cov:
        w = dataclasses.replace(w, cov=args.cov, name=f"{w.name}_{args.cov}")
    if args.rows > 0:
        w = w.scaled(min(args.rows, w.N))
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, w, ws, rank)
    else:
        run_ours(args, w, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
