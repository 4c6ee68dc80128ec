#!/usr/bin/env python3
"""Benchmark of the MoE EP hot path (layout + dispatch + combine) on GB300.

One step = one pass of the whole path over one batch of the
DeepSeek-V3-shaped workload (W=8 logical ranks, 256 experts, top-8,
T=4096 tokens per rank, H=7168, bf16 payload, fp32-accumulate bf16
combine): routing layout, dispatch send (copy of every token row to each of
its destination ranks), dispatch receive (recv_count), combine (ordered fp32
gather-reduce of the expert rows back to source order, weights included).
The expert between dispatch and combine is outside the path: combine reads
the registered combine buffer, filled once before timing by the identity
expert of the correctness check.

Prints ONE JSON line (rank 0).  `value` = tokens/s over all ranks (tokens =
W*T per replica per step), device-timed with CUDA events around K replays
of a CUDA graph of the step (`--eager`: K host-launched steps); the
per-kernel times and the roofline come from eager steps; `e2e` = the same
metric with the inputs copied from pinned host memory and the combined
output copied back inside every step.  `workloads` (one GPU) holds the same
figures for every workload of the benchmark at full size (tiny, the
DeepSeek-V3 shape, its FP8 + Zipf variant, the low-latency decode case in
its split-phase form on two streams, the Mixtral shape), each with the
oracle's CPU baseline on the same batch and a bit-for-bit comparison of
the combined output with the oracle's.  `--impl reference` times the CPU
oracle (plain scalar C, on every host core) on a bounded sample of the same
workload instead.  With torchrun (N>1) every rank runs an independent
replica ("replicas only": the path has no exchange between GPUs on one
device's segments).
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dispatch+combine tokens/s and HBM GB/s (% of GB300 peak), 1 GPU"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = "dsv3"
SELF_LAYOUT_CHUNKS = 8     # the library launches no layout kernel up to this many chunks


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--tokens", type=int, default=0,
                    help="override T (tokens per rank), e.g. for a profiling case")
    ap.add_argument("--cap", type=int, default=0,
                    help="receive rows per rank (0: W*T)")
    ap.add_argument("--fp8-input", action="store_true",
                    help="FP8 workloads: dispatch a pre-quantised payload (codes + scales)")
    ap.add_argument("--combine-dtype", choices=["bf16", "fp32", "fp8_e4m3"], default="bf16",
                    help="element type of the expert rows combine reads")
    ap.add_argument("--split", action="store_true",
                    help="split phases on two streams: dispatch_send / combine_recv on "
                         "one, dispatch_recv / combine_send on the other")
    ap.add_argument("--eager", action="store_true",
                    help="launch every step from the host instead of replaying a CUDA "
                         "graph of it (per-kernel times always come from eager steps)")
    ap.add_argument("--combine-mode", choices=["gather", "scatter"], default="gather",
                    help="gather combine, or scatter combine through a staging area")
    ap.add_argument("--flush-l2", action="store_true",
                    help="write twice the L2 size before every timed step (cold L2; for "
                         "workloads whose working set fits in L2) and time the steps alone")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload figures (every benchmark workload at full "
                         "size, measured after the headline)")
    ap.add_argument("--workload-steps", type=int, default=100,
                    help="timed graph replays per workload in the per-workload figures")
    ap.add_argument("--moe-group", type=int, default=0, metavar="GCAP",
                    help="also time the standard-MoE grouping / un-grouping with "
                         "GCAP grouped rows per rank (reported beside the step)")
    return ap.parse_args()


# ------------------------------------------------------------- bookkeeping

def algorithmic_bytes(wl, P, N, fp8, with_weights=True, fp8_input=False,
                      y_bytes=2, scatter=False):
    """Bytes the method must move (each counted once).
    dispatch: read N*(H*b_in + s_in + 8k) [row once (+ its scales) + ids +
              weights]; write P*(H*b + s_b + 8k + 4) [row, scales, weights,
              ids, src_pos]
    combine:  read P*H*y_bytes (+ P*4k weights); write N*H*2 (+ N*4k)."""
    H, k = wl.hidden, wl.topk
    b_out = 1 if fp8 else 2
    s_b = 4 * (H // 128) if fp8 else 0
    d_read = N * ((H + s_b) if fp8_input else H * 2) + N * 8 * k
    d_write = P * (H * b_out + s_b + 8 * k + 4)
    c_read = P * H * y_bytes + (P * 4 * k if with_weights else 0)
    if scatter:   # rows pushed to the staging area, then read back
        c_read += P * H * 2
        c_write_extra = P * H * 2
    else:
        c_write_extra = 0
    c_write = N * H * 2 + (N * 4 * k if with_weights else 0) + c_write_extra
    return dict(dispatch=d_read + d_write, combine=c_read + c_write,
                dispatch_read=d_read, dispatch_write=d_write,
                combine_read=c_read, combine_write=c_write)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha():
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(ROOT, "combine_ep_layout_06_gb300",
                                          "csrc", "*")))
    for f in files:
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[workload][kernel]
        if e.get("src_sha") != kernel_source_sha():
            return None
        return float(e["bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons every 100 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-i", str(index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            return
        self.first = threading.Event()
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        self.first.wait(timeout=10)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))
                self.first.set()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        if not self.samples:
            return None
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = "during timed region"
        if len(inside) < 2:
            inside = [p for (_, p) in self.samples]
            note = "whole run (timed region shorter than the sampling period)"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for p in inside:
            for n, v in zip(names, p[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(inside),
                "window": note}


# ------------------------------------------------------------ replicas

def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's time: every rank times its own replica and the job
    is done when the last one is (all_reduce MAX; a no-op for one rank)."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_replica: int, world: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: all replicas' tokens over the slowest step time."""
    return world * tokens_per_replica / (ms_per_step / 1e3)


# ------------------------------------------------------------ our path

class Case:
    """One workload on the device: the op, its inputs, the step functions."""

    def __init__(self, wl, dev, fp8_input=False, combine_dtype="bf16", cap=0,
                 moe_group=0, combine_mode="gather", split=False):
        import torch
        from combine_ep_layout_06_gb300 import inputs as gen
        from combine_ep_layout_06_gb300.op import (EpDispatchCombineConfig,
                                                   EpDispatchCombineOp)
        self.wl, self.dev, self.split = wl, dev, split
        self.fp8_input, self.combine_dtype = fp8_input, combine_dtype
        self.combine_mode = combine_mode
        W, T, H, k = wl.world_size, wl.max_tokens_per_rank, wl.hidden, wl.topk
        self.inp = inp = gen.make_inputs(wl)
        self.N = W * T
        Er = wl.experts_per_rank
        self.P = int(sum(len(set((inp.indices[s, t] // Er).tolist()))
                         for s in range(W) for t in range(T)))
        if fp8_input and not wl.fp8:
            raise SystemExit("--fp8-input needs an FP8 workload")
        cfg = EpDispatchCombineConfig(W, wl.num_experts, k, H, T,
                                      max_recv_tokens_per_rank=cap,
                                      dispatch_dtype="fp8_e4m3" if wl.fp8 else "bf16",
                                      combine_dtype=combine_dtype,
                                      max_grouped_rows_per_rank=moe_group,
                                      combine_mode=combine_mode)
        self.op = op = EpDispatchCombineOp(cfg, device=dev)
        self.x = torch.from_numpy(inp.x_bits.view(np.int16)).to(dev).view(torch.bfloat16)
        self.xsc = None
        if fp8_input:        # pre-quantised payload: E4M3 codes + block scales
            x8, sc8 = gen.draw_fp8_payload(wl)
            self.x = torch.from_numpy(x8).to(dev)
            self.xsc = torch.from_numpy(sc8).to(dev)
        self.w = torch.from_numpy(inp.weights).to(dev)
        self.idx = torch.from_numpy(inp.indices).to(dev)
        self.out = torch.empty((W, T, H), dtype=torch.bfloat16, device=dev)
        self.out_w = torch.empty((W, T, k), dtype=torch.float32, device=dev)
        self.stream = torch.cuda.Stream(device=dev)
        self.stream2 = torch.cuda.Stream(device=dev)
        self.nt = [T] * W
        self.identity_check()

    def identity_check(self):
        """The identity expert fills the registered combine buffer (not timed)
        and the combined output must give back the input."""
        op, stream = self.op, self.stream
        with torch_stream(stream):
            op.dispatch(self.x, self.w, self.xsc, self.idx, num_tokens=self.nt, stream=stream)
            op.identity_expert(stream=stream)
            op.combine(weights=op.out_w, out=self.out, out_weights=self.out_w, stream=stream)
        stream.synchronize()
        x, xsc = self.x, self.xsc
        if xsc is not None:       # expected: the dequantised payload
            import torch
            xs = x.view(torch.float8_e4m3fn).float() * xsc.repeat_interleave(128, dim=2)
        else:
            xs = x.float()
        ys = self.out.float()
        # tolerance: bf16 rounding of the expert product and of the sum; an
        # E4M3 step (2^-4 relative) where a payload is quantised on the way
        quantised = (self.wl.fp8 and xsc is None) or self.combine_dtype == "fp8_e4m3"
        if quantised:
            ok = bool(((ys - xs).abs() <= xs.abs() * 0.15 + xs.abs().amax() * 2.0 ** -8).all())
        else:
            ok = bool(((ys - xs).abs() <= xs.abs() * (2.0 ** -8 * 10) + 1e-30).all())
        st, mask = self.op.get_error(stream)
        self.ident_ok = ok and st == 0
        self.ident_mask = mask

    # one step = the whole path over one batch
    def step_onecall(self):
        # what a user calls: one-call dispatch (layout, then the copy launched
        # programmatically after it) and combine
        op, s = self.op, self.stream
        op.dispatch(self.x, self.w, self.xsc, self.idx, num_tokens=self.nt, stream=s)
        op.combine(weights=op.out_w, out=self.out, out_weights=self.out_w, stream=s)

    def step_split(self, ev=None):
        # sender side on `stream`, receiver / expert side on `stream2`
        op, s, s2 = self.op, self.stream, self.stream2
        if ev is not None:
            ev[0].record(s)
            ev[1].record(s)
        s2.wait_stream(s)
        op.dispatch_send(self.x, self.w, self.xsc, self.idx, num_tokens=self.nt, stream=s)
        op.dispatch_recv(stream=s2)
        op.combine_send(stream=s2)
        if ev is not None:
            ev[2].record(s)
        op.combine_recv(weights=op.out_w, out=self.out, out_weights=self.out_w, stream=s)
        s.wait_stream(s2)
        if ev is not None:
            ev[3].record(s)

    def step_events(self, ev):
        """The same work as separate calls, with CUDA events between them, so
        that the layout, copy and combine times can be read apart."""
        if self.split:
            return self.step_split(ev)
        op, s = self.op, self.stream
        ev[0].record(s)
        op.layout(self.idx, num_tokens=self.nt, stream=s)
        ev[1].record(s)
        op.dispatch_send_replay(self.x, self.w, self.idx, num_tokens=self.nt, stream=s,
                                scales=self.xsc)
        op.dispatch_recv(stream=s)
        ev[2].record(s)
        op.combine(weights=op.out_w, out=self.out, out_weights=self.out_w, stream=s)
        ev[3].record(s)

    def timed_step(self):
        return self.step_split() if self.split else self.step_onecall()

    def capture(self):
        import torch
        with torch_stream(self.stream):
            for _ in range(3):
                self.timed_step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            self.timed_step()
        torch.cuda.synchronize()
        return g

    def time_steps(self, steps, warmup, graph=None, flush_l2=False):
        """ms over `steps` steps (graph replays, or host launches without a
        graph), CUDA events on the launching stream.  flush_l2: a write of
        twice the L2 size before every step, outside the step's own events,
        and the step times summed."""
        import torch
        s = self.stream
        with torch_stream(s):
            for _ in range(warmup):
                graph.replay() if graph is not None else self.timed_step()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        if flush_l2:
            flush = torch.empty(2 * torch.cuda.get_device_properties(self.dev).L2_cache_size,
                                dtype=torch.uint8, device=self.dev)
            fev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
                   for _ in range(steps)]
        with torch_stream(s):
            start.record(s)
            for i in range(steps):
                if flush_l2:
                    flush.fill_(i & 0xFF)
                    fev[i][0].record(s)
                graph.replay() if graph is not None else self.timed_step()
                if flush_l2:
                    fev[i][1].record(s)
            stop.record(s)
        stop.synchronize()
        torch.cuda.synchronize()
        if flush_l2:
            return float(sum(e[0].elapsed_time(e[1]) for e in fev))
        return start.elapsed_time(stop)

    def kernel_times(self, steps):
        """Mean ms of layout, copy (+ receive) and combine, from eager steps."""
        import torch
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        with torch_stream(self.stream):
            for i in range(steps):
                self.step_events(evs[i])
        torch.cuda.synchronize()
        lay = np.array([e[0].elapsed_time(e[1]) for e in evs])
        dis = np.array([e[1].elapsed_time(e[2]) for e in evs])
        com = np.array([e[2].elapsed_time(e[3]) for e in evs])
        return float(lay.mean()), float(dis.mean()), float(com.mean())

    def bytes(self):
        return algorithmic_bytes(
            self.wl, self.P, self.N, self.wl.fp8, fp8_input=self.fp8_input,
            y_bytes={"fp32": 4, "bf16": 2, "fp8_e4m3": 1 + 4 / 128}[self.combine_dtype],
            scatter=self.combine_mode == "scatter")

    def kernel_name(self, dominant):
        if dominant == "combine":
            return "combine_kernel"
        return ("dispatch_kernel" if self.wl.fp8 and not self.fp8_input
                else "dispatch_bulk_kernel")

    def launches_per_step(self):
        # this library's kernels per timed step: layout (none when the routing
        # spans at most SELF_LAYOUT_CHUNKS 32-token chunks: the copy computes
        # it), copy, combine (the receive phase launches none without early
        # notification), plus the scatter send in scatter mode
        wl = self.wl
        chunks = wl.world_size * -(-wl.max_tokens_per_rank // 32)
        return (2 + (1 if chunks > SELF_LAYOUT_CHUNKS else 0) +
                (1 if self.combine_mode == "scatter" else 0))

    def close(self):
        import torch
        self.op.close()
        for a in ("op", "x", "xsc", "w", "idx", "out", "out_w"):
            setattr(self, a, None)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


class torch_stream:
    """torch.cuda.stream(s) as a context manager (imported lazily)."""

    def __init__(self, s):
        import torch
        self.cm = torch.cuda.stream(s)

    def __enter__(self):
        return self.cm.__enter__()

    def __exit__(self, *a):
        return self.cm.__exit__(*a)


def roofline_of(case, d_ms, c_ms, peak, peak_kind):
    ab = case.bytes()
    dominant = "combine" if c_ms >= d_ms else "dispatch"
    dom_ms = c_ms if dominant == "combine" else d_ms
    achieved = ab[dominant] / (dom_ms / 1e3) / 1e9
    kname = case.kernel_name(dominant)
    return {
        "bound": "hbm",
        "kernel": kname,
        "achieved": achieved,
        "peak": peak,
        "peak_kind": f"of {peak_kind} (hbm_gbs copy bandwidth)",
        "unit": "GB/s",
        "frac": achieved / peak,
        "traffic": recorded_traffic(kname, case.wl.name),
        "algorithmic_bytes_per_launch": int(ab[dominant]),
    }


def run_ours(args, rank, world, local_rank):
    import torch
    from combine_ep_layout_06_gb300 import inputs as gen

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = gen.WORKLOADS[args.workload]
    if args.tokens:
        wl = wl.scaled(args.tokens)
    W, T, H, k = wl.world_size, wl.max_tokens_per_rank, wl.hidden, wl.topk
    case = Case(wl, dev, fp8_input=args.fp8_input, combine_dtype=args.combine_dtype,
                cap=args.cap, moe_group=args.moe_group, combine_mode=args.combine_mode,
                split=args.split)
    op, stream, N, P = case.op, case.stream, case.N, case.P
    ident_ok = case.ident_ok

    graph = None if args.eager else case.capture()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_host0 = time.time()
    total_ms = case.time_steps(args.steps, args.warmup, graph=graph, flush_l2=args.flush_l2)
    if world > 1:
        torch.distributed.barrier()
    t_host1 = time.time()
    lay_ms, d_ms, c_ms = case.kernel_times(args.steps)   # per-kernel split, eagerly
    clocks = sampler.summary(t_host0, t_host1) if sampler else None
    if sampler:
        sampler.stop()
    st, mask = op.get_error(stream)

    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(N, world, ms_per_step)

    ab = case.bytes()
    step_bytes = ab["dispatch"] + ab["combine"]
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    peak, peak_kind = measured_peak()
    roof = roofline_of(case, d_ms, c_ms, peak, peak_kind)

    e2e = run_e2e(case, args, world, dev) if args.e2e_steps > 0 else None
    moe = run_moe(case, args) if args.moe_group else None

    cpu = None
    oracle_parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, oracle_parity = cpu_baseline(case)

    res = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8" if wl.fp8 else "bf16",
        "data": "synthetic (seeded; shapes and routing of the workload, no dataset)",
        "config": {
            "workload": workload_text(wl, args),
            "tokens_per_step": N,
            "routed_pairs": P,
            "l2": l2_text(step_bytes, l2_bytes, args.flush_l2),
            "parallelism": f"replicas x{world}",
            "step": step_text(args.split, graph is not None),
        },
        "gb_per_s": step_bytes / (ms_per_step / 1e3) / 1e9,
        "frac_of_nominal_8tbs": step_bytes / (ms_per_step / 1e3) / 1e9 / NOMINAL_HBM_GBS,
        "frac_of_measured_hbm": step_bytes / (ms_per_step / 1e3) / 1e9 / peak,
        "algorithmic_bytes_per_step": int(step_bytes),
        "layout_ms": lay_ms,
        "dispatch_ms": d_ms,
        "combine_ms": c_ms,
        "dispatch_gb_per_s": ab["dispatch"] / (d_ms / 1e3) / 1e9,
        "combine_gb_per_s": ab["combine"] / (c_ms / 1e3) / 1e9,
        "roofline": roof,
        "identity_check": "pass" if ident_ok else "FAIL",
        "oracle_parity": oracle_parity,
        "device_errors": int(mask),
        "gpu_launches": case.launches_per_step() * args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if moe is not None:
        res["standard_moe"] = moe
    headline_entry = None
    if not args.fp8_input and args.combine_dtype == "bf16" and args.combine_mode == "gather" \
            and not args.cap and not args.tokens and not args.flush_l2:
        headline_entry = workload_entry_from(case, ms_per_step, (lay_ms, d_ms, c_ms), roof,
                                             peak, cpu, oracle_parity, graph is not None,
                                             args.steps)
        if wl.name in COLD_L2 and graph is not None and not args.no_workloads:
            add_cold_l2(headline_entry, case, graph, args.workload_steps)
        headline_entry["device_errors"] = int(mask)
    case.close()
    del case, graph

    if rank == 0 and world == 1 and not args.no_workloads:
        res["workloads"] = run_workloads(args, dev, peak, peak_kind,
                                         reuse={args.workload: headline_entry}
                                         if headline_entry else {})
    return res


def l2_text(step_bytes, l2_bytes, flush):
    if flush:
        return ("L2 flushed before every timed step (a write of twice its size), "
                "the flush outside the step's events")
    if step_bytes >= 2 * l2_bytes:
        return (f"no flush: each step moves {step_bytes / 1e6:.0f} MB "
                f"({step_bytes / l2_bytes:.1f}x the {l2_bytes / 1e6:.0f} MB L2) between "
                "two reads of any input (every input and output is read or written once "
                "per step)")
    return (f"warm L2: the step's {step_bytes / 1e6:.1f} MB fit in the "
            f"{l2_bytes / 1e6:.0f} MB L2 (--flush-l2 gives the cold figure)")


def step_text(split, graph):
    return (("dispatch_send (layout + copy) on stream A, dispatch_recv + "
             "combine_send on stream B, combine_recv on A" if split else
             "dispatch (layout kernel, then the copy launched programmatically "
             "after it) + combine, one stream; per-kernel times from the same "
             "work as layout + dispatch_send (routing replay) + dispatch_recv + "
             "combine")
            + ("; timed as a CUDA-graph replay of the step (per-kernel times eager)"
               if graph else ""))


# the benchmark's workloads, each measured the same way in one run (the
# low-latency decode one in its split-phase form on two streams)
WORKLOAD_ORDER = ["tiny", "dsv3", "dsv3_fp8_zipf", "ll_decode", "mixtral"]
COLD_L2 = ("tiny", "ll_decode")     # working sets that fit in L2


def workload_entry_from(case, ms, kern, roof, peak, cpu, parity, graph, steps):
    ab = case.bytes()
    step_bytes = ab["dispatch"] + ab["combine"]
    gbs = step_bytes / (ms / 1e3) / 1e9
    lay, d_ms, c_ms = kern
    return {
        "workload": case.wl.name,
        "mode": ("split phases on two streams" if case.split else "one stream")
                + (", CUDA-graph replay" if graph else ", host launches"),
        "steps": steps,
        "ms_per_step": ms,
        "tokens_per_s": case.N / (ms / 1e3),
        "tokens_per_step": case.N,
        "routed_pairs": case.P,
        "algorithmic_bytes_per_step": int(step_bytes),
        "gb_per_s": gbs,
        "frac_of_measured_hbm": gbs / peak,
        "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS,
        "layout_ms": lay,
        "dispatch_ms": d_ms,
        "combine_ms": c_ms,
        "dominant_kernel": roof["kernel"],
        "dominant_frac_of_measured_hbm": roof["frac"],
        "identity_check": "pass" if case.ident_ok else "FAIL",
        "oracle_parity": parity,
        "cpu_baseline": cpu,
    }


def run_workloads(args, dev, peak, peak_kind, reuse):
    """Every workload of the benchmark at full size, each a few seconds: graph
    replays of the step, the per-kernel split, the identity check, the oracle
    baseline and its comparison; cold-L2 figures where the working set fits
    in L2."""
    from combine_ep_layout_06_gb300 import inputs as gen
    out = {}
    steps = args.workload_steps
    for name in WORKLOAD_ORDER:
        if name in reuse:
            out[name] = reuse[name]
            continue
        wl = gen.WORKLOADS[name]
        case = Case(wl, dev, split=wl.split)
        graph = case.capture()
        ms = case.time_steps(steps, max(3, args.warmup), graph=graph) / steps
        kern = case.kernel_times(min(steps, 50))
        roof = roofline_of(case, kern[1], kern[2], peak, peak_kind)
        cpu = parity = None
        if not args.no_cpu_baseline:
            cpu, parity = cpu_baseline(case)
        e = workload_entry_from(case, ms, kern, roof, peak, cpu, parity, True, steps)
        if name in COLD_L2:
            add_cold_l2(e, case, graph, steps)
        st, mask = case.op.get_error(case.stream)
        e["device_errors"] = int(mask)
        out[name] = e
        case.close()
        del case, graph
    return out


def add_cold_l2(entry, case, graph, steps):
    cold = case.time_steps(steps, 3, graph=graph, flush_l2=True) / steps
    entry["cold_l2_ms_per_step"] = cold
    entry["cold_l2_tokens_per_s"] = case.N / (cold / 1e3)


def run_e2e(case, args, world, dev):
    """End to end: pinned host inputs -> device, path, combined output ->
    host.  Every step copies its own inputs in and its combined output out;
    the copies of neighbouring steps overlap the compute through three
    streams (H2D of step i+1 | dispatch + combine of step i | D2H of step
    i-1) and double-buffered device inputs and outputs."""
    import torch
    op, stream, nt = case.op, case.stream, case.nt
    x, xsc, w, idx, out, out_w = case.x, case.xsc, case.w, case.idx, case.out, case.out_w
    W, T, H = case.wl.world_size, case.wl.max_tokens_per_rank, case.wl.hidden
    hx = x.cpu().pin_memory()
    hsc = None if xsc is None else xsc.cpu().pin_memory()
    hw = torch.from_numpy(case.inp.weights).pin_memory()
    hi = torch.from_numpy(case.inp.indices).pin_memory()
    hout = [torch.empty((W, T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dx = [torch.empty_like(x) for _ in range(2)]
    dw = [torch.empty_like(w) for _ in range(2)]
    di = [torch.empty_like(idx) for _ in range(2)]
    dsc = [None if xsc is None else torch.empty_like(xsc) for _ in range(2)]
    dout = [torch.empty_like(out) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):      # all buffers free at the start
        ev_comp[b].record(stream)
        ev_out[b].record(s_out)

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_comp[b])            # step i-2 has consumed slot b
            dx[b].copy_(hx, non_blocking=True)
            if dsc[b] is not None:
                dsc[b].copy_(hsc, non_blocking=True)
            dw[b].copy_(hw, non_blocking=True)
            di[b].copy_(hi, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])               # D2H of step i-2 has read dout[b]
        op.dispatch(dx[b], dw[b], dsc[b], di[b], num_tokens=nt, stream=stream)
        op.combine(weights=op.out_w, out=dout[b], out_weights=out_w, stream=stream)
        ev_comp[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            hout[b].copy_(dout[b], non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    stream.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(args.e2e_steps):
        e2e_step(i)
    s_out.wait_stream(stream)
    s_out.wait_stream(s_in)
    e1.record(s_out)
    e1.synchronize()
    e_ms = e0.elapsed_time(e1) / args.e2e_steps
    e_ms = max_over_ranks(e_ms, world, dev)
    h2d = hx.numel() * hx.element_size() + hw.numel() * 4 + hi.numel() * 4 + \
        (0 if hsc is None else hsc.numel() * 4)
    d2h = hout[0].numel() * 2
    # the copied-back output equals the device result of the same inputs
    e2e_ok = bool(torch.equal(hout[(args.e2e_steps - 1) % 2].to(dev), out))
    # The bound of a pipelined step: the same H2D and D2H bytes copied at
    # once on the two copy streams with nothing else running.
    lk = []
    for _ in range(4):
        torch.cuda.synchronize()
        l0 = torch.cuda.Event(enable_timing=True)
        l1 = torch.cuda.Event(enable_timing=True)
        l0.record(s_in)
        s_out.wait_event(l0)
        with torch.cuda.stream(s_in):
            dx[0].copy_(hx, non_blocking=True)
            if dsc[0] is not None:
                dsc[0].copy_(hsc, non_blocking=True)
            dw[0].copy_(hw, non_blocking=True)
            di[0].copy_(hi, non_blocking=True)
        with torch.cuda.stream(s_out):
            hout[0].copy_(dout[0], non_blocking=True)
        s_in.wait_stream(s_out)
        l1.record(s_in)
        l1.synchronize()
        lk.append(l0.elapsed_time(l1))
    link_ms = max_over_ranks(float(min(lk[1:])), world, dev)
    N = case.N
    return {"value": job_throughput(N, world, e_ms), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": e_ms, "pipelined": "H2D / compute / D2H on three streams",
            "output_check": "pass" if e2e_ok else "FAIL",
            "host_link": {"copy_ms": link_ms,
                          "h2d_gb_per_s": h2d / (link_ms / 1e3) / 1e9,
                          "d2h_gb_per_s": d2h / (link_ms / 1e3) / 1e9,
                          "frac": link_ms / e_ms,
                          "what": "the step's H2D and D2H bytes copied concurrently, "
                                  "alone: the bound of the pipelined step"}}


def run_moe(case, args):
    """Standard-MoE conversion after the step's dispatch: grouping, identity
    experts (a copy, untimed), un-grouping into the combine buffer."""
    import torch
    op, stream, wl, P = case.op, case.stream, case.wl, case.P
    H = wl.hidden
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    gms, ums = [], []
    with torch.cuda.stream(stream):
        for i in range(13):
            ev[0].record(stream)
            op.moe_group(stream=stream)
            ev[1].record(stream)
            op.moe_y.copy_(op.moe_x)
            ev[2].record(stream)
            op.moe_ungroup(stream=stream)
            ev[3].record(stream)
            stream.synchronize()
            if i >= 3:
                gms.append(ev[0].elapsed_time(ev[1]))
                ums.append(ev[2].elapsed_time(ev[3]))
    st_m, mask_m = op.get_error(stream)
    n_ent = int(op.moe_count.sum().item())
    rowb = H * (1 if wl.fp8 else 2)
    g_bytes = P * rowb + n_ent * (rowb + 8)
    u_bytes = n_ent * (2 * H + 8) + P * 2 * H
    g_ms, u_ms = float(np.median(gms)), float(np.median(ums))
    return {"entries": n_ent, "gcap": args.moe_group, "errors": int(mask_m),
            "group_ms": g_ms, "ungroup_ms": u_ms,
            "group_gb_per_s": g_bytes / (g_ms / 1e3) / 1e9,
            "ungroup_gb_per_s": u_bytes / (u_ms / 1e3) / 1e9,
            "group_algorithmic_bytes": int(g_bytes),
            "ungroup_algorithmic_bytes": int(u_bytes)}


# ------------------------------------------------------------ CPU oracle

def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_step_seconds(wl, inp, threads, cap, bufs, y, out, out_w):
    """One pass of the oracle over the batch on `threads` host threads:
    layout, then dispatch and combine over disjoint token ranges (timed);
    the identity expert between them fills y (untimed, the expert is not on
    the path).  Output buffers are allocated and touched beforehand."""
    import oracle
    W, T = wl.world_size, wl.max_tokens_per_rank
    nt = np.ascontiguousarray(inp.num_tokens, np.int32)
    t0 = time.perf_counter()
    pos, C, rc = oracle.layout(wl, inp.indices, nt)
    oracle.run_ranges(lambda a, b: oracle.dispatch_into(
        wl, inp.x_bits, inp.weights, inp.indices, nt, pos, cap, bufs, a, b), W * T, threads)
    t1 = time.perf_counter()
    oracle.run_ranges(lambda a, b: oracle.identity_expert_into(
        wl, rc, bufs, cap, y, a, b), W * cap, max(threads, 1))
    t2 = time.perf_counter()
    oracle.run_ranges(lambda a, b: oracle.combine_into(
        wl, nt, pos, y, bufs["out_w"], cap, out, out_w, a, b), W * T, threads)
    t3 = time.perf_counter()
    return (t1 - t0) + (t3 - t2)


def cpu_baseline(case):
    """The oracle as it stands (plain scalar C) on the benchmark's own batch:
    layout + dispatch + combine, the combine reading the identity expert's
    rows (as the device step does), single-threaded and on every host core
    (dispatch and combine split over disjoint token ranges; the layout's
    scan stays on one thread).  Median of 3 runs for the latency-sized
    workloads, one run otherwise.  Also returns whether the device's
    combined output of the same batch equals the oracle's bit for bit."""
    import oracle
    import torch
    wl, inp = case.wl, case.inp
    W, T, H, k = wl.world_size, wl.max_tokens_per_rank, wl.hidden, wl.topk
    rc = oracle.layout(wl, inp.indices, inp.num_tokens)[2]      # sizing pass
    cap = max(1, int(rc.max()))
    bufs = oracle.dispatch_buffers(wl, cap)
    y = np.empty((W, cap, H), np.uint16)
    out = np.empty((W, T, H), np.uint16)
    out_w = np.empty((W, T, k), np.float32)
    for a in (*bufs.values(), y, out, out_w):
        a.fill(0)                                   # touch every page now
    repeats = 3 if wl.name in COLD_L2 else 1
    cores = host_cores()
    single = float(np.median([oracle_step_seconds(wl, inp, 1, cap, bufs, y, out, out_w)
                              for _ in range(repeats)]))
    multi = float(np.median([oracle_step_seconds(wl, inp, cores, cap, bufs, y, out, out_w)
                             for _ in range(repeats)]))
    n = W * T
    parity = None
    if not case.fp8_input and case.combine_dtype == "bf16":
        got = case.out.view(torch.int16).cpu().numpy().view(np.uint16)
        got_w = case.out_w.cpu().numpy()
        same = bool(np.array_equal(got, out)) and \
            bool(np.array_equal(got_w.view(np.uint32), out_w.view(np.uint32)))
        parity = (f"{'bit-exact' if same else 'DIFFERS'}: device combined output and "
                  f"weights of all {n} tokens against the oracle's, same batch")
    return {"value": n / multi, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": (f"the whole {wl.name} batch ({n} tokens, H={H}): layout + "
                       f"dispatch + combine, {multi:.3f} s on {cores} host threads "
                       f"(dispatch and combine over token ranges; layout on one); "
                       f"{'median of 3' if repeats == 3 else 'one run'}"),
            "seconds": multi,
            "host_cores": os.cpu_count(),
            "single_thread": {"value": n / single, "unit": "tokens/s", "cores": 1,
                              "seconds": single}}, parity


def workload_text(wl, args):
    """The workload as both arms name it in `config`."""
    return (f"{wl.name}: W={wl.world_size} logical ranks on one GPU, E={wl.num_experts}, "
            f"k={wl.topk}, T={wl.max_tokens_per_rank} tokens/rank, H={wl.hidden}, "
            f"{'fp8 e4m3' if wl.fp8 else 'bf16'} dispatch"
            f"{' of a pre-quantised payload' if args.fp8_input else ''}, "
            f"fp32-accumulate bf16 combine of {args.combine_dtype} expert rows "
            f"with weights, {wl.routing} routing")


def run_reference(args):
    """--impl reference: the CPU oracle, timed per step on a bounded sample
    (256 tokens per rank of the workload's recipe) on every host core."""
    from combine_ep_layout_06_gb300 import inputs as gen
    import oracle
    wl = gen.WORKLOADS[args.workload]
    sample = 256
    swl = wl.scaled(sample)
    inp = gen.make_inputs(swl)
    W, H, k = swl.world_size, swl.hidden, swl.topk
    n = W * sample
    rc = oracle.layout(swl, inp.indices, inp.num_tokens)[2]
    cap = max(1, int(rc.max()))
    bufs = oracle.dispatch_buffers(swl, cap)
    y = np.empty((W, cap, H), np.uint16)
    out = np.empty((W, sample, H), np.uint16)
    out_w = np.empty((W, sample, k), np.float32)
    for a in (*bufs.values(), y, out, out_w):
        a.fill(0)
    cores = host_cores()
    for _ in range(args.warmup):
        oracle_step_seconds(swl, inp, cores, cap, bufs, y, out, out_w)
    steps = max(1, args.steps)
    tsec = sum(oracle_step_seconds(swl, inp, cores, cap, bufs, y, out, out_w)
               for _ in range(steps)) / steps
    v = n / tsec
    return {
        "impl": "reference",
        "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": tsec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8" if wl.fp8 else "bf16", "data": "synthetic",
        "config": {"workload": workload_text(wl, args),
                   "tokens_per_step": wl.world_size * wl.max_tokens_per_rank,
                   "sample": f"each timed step runs the oracle on {sample} tokens/rank "
                             f"({n} tokens) of this workload; value = tokens/s of that sample"},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{n} tokens of the {wl.name} recipe per step: layout + "
                                   f"dispatch + combine on {cores} host threads (dispatch and "
                                   f"combine over token ranges; the identity expert between "
                                   f"them untimed)"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
