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
output copied back inside every step.  `--impl reference` times the CPU
oracle (plain scalar C) on a bounded sample of the same workload instead.
With torchrun (N>1) every rank runs an independent replica ("replicas
only": the path has no exchange between GPUs on one device's segments).
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

def run_ours(args, rank, world, local_rank):
    import torch
    from combine_ep_layout_06_gb300 import inputs as gen
    from combine_ep_layout_06_gb300.op import (EpDispatchCombineConfig,
                                               EpDispatchCombineOp)

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = gen.WORKLOADS[args.workload]
    if args.tokens:
        wl = wl.scaled(args.tokens)
    W, T, H, k = wl.world_size, wl.max_tokens_per_rank, wl.hidden, wl.topk
    inp = gen.make_inputs(wl)
    N = W * T
    Er = wl.experts_per_rank
    P = int(sum(len(set((inp.indices[s, t] // Er).tolist()))
                for s in range(W) for t in range(T)))

    if args.fp8_input and not wl.fp8:
        raise SystemExit("--fp8-input needs an FP8 workload")
    cfg = EpDispatchCombineConfig(W, wl.num_experts, k, H, T,
                                  max_recv_tokens_per_rank=args.cap,
                                  dispatch_dtype="fp8_e4m3" if wl.fp8 else "bf16",
                                  combine_dtype=args.combine_dtype,
                                  max_grouped_rows_per_rank=args.moe_group,
                                  combine_mode=args.combine_mode)
    op = EpDispatchCombineOp(cfg, device=dev)
    x = torch.from_numpy(inp.x_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    xsc = None
    if args.fp8_input:        # pre-quantised payload: E4M3 codes + block scales
        x8, sc8 = gen.draw_fp8_payload(wl)
        x = torch.from_numpy(x8).to(dev)
        xsc = torch.from_numpy(sc8).to(dev)
    w = torch.from_numpy(inp.weights).to(dev)
    idx = torch.from_numpy(inp.indices).to(dev)
    out = torch.empty((W, T, H), dtype=torch.bfloat16, device=dev)
    out_w = torch.empty((W, T, k), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    nt = [T] * W

    # identity expert fills the registered combine buffer (not timed) and
    # the combined output must give back the input
    with torch.cuda.stream(stream):
        op.dispatch(x, w, xsc, idx, num_tokens=nt, stream=stream)
        op.identity_expert(stream=stream)
        op.combine(weights=op.out_w, out=out, out_weights=out_w, stream=stream)
    stream.synchronize()
    if xsc is not None:       # expected: the dequantised payload
        xs = x.view(torch.float8_e4m3fn).float() * xsc.repeat_interleave(128, dim=2)
    else:
        xs = x.float()
    ys = out.float()
    # tolerance: bf16 rounding of the expert product and of the sum; an E4M3
    # step (2^-4 relative) where a payload is quantised on the way
    quantised = (wl.fp8 and xsc is None) or args.combine_dtype == "fp8_e4m3"
    if quantised:
        ident_ok = bool(((ys - xs).abs() <= xs.abs() * 0.15 + xs.abs().amax() * 2.0 ** -8).all())
    else:
        ident_ok = bool(((ys - xs).abs() <= xs.abs() * (2.0 ** -8 * 10) + 1e-30).all())
    st, mask = op.get_error(stream)
    ident_ok = ident_ok and st == 0
    del xs, ys

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        op.layout(idx, num_tokens=nt, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        op.dispatch_send_replay(x, w, idx, num_tokens=nt, stream=stream, scales=xsc)
        op.dispatch_recv(stream=stream)
        if ev is not None:
            ev[2].record(stream)
        op.combine(weights=op.out_w, out=out, out_weights=out_w, stream=stream)
        if ev is not None:
            ev[3].record(stream)

    stream2 = torch.cuda.Stream(device=dev)

    def step_split(ev=None):
        # sender side on `stream`, receiver / expert side on `stream2`
        if ev is not None:
            ev[0].record(stream)
            ev[1].record(stream)
        stream2.wait_stream(stream)
        op.dispatch_send(x, w, xsc, idx, num_tokens=nt, stream=stream)
        op.dispatch_recv(stream=stream2)
        op.combine_send(stream=stream2)
        if ev is not None:
            ev[2].record(stream)
        op.combine_recv(weights=op.out_w, out=out, out_weights=out_w, stream=stream)
        stream.wait_stream(stream2)
        if ev is not None:
            ev[3].record(stream)

    def step_onecall():
        # what a user calls: one-call dispatch (layout, then the copy launched
        # programmatically after it) and combine; `step` runs the same work as
        # separate calls so that CUDA events can split it per kernel
        op.dispatch(x, w, xsc, idx, num_tokens=nt, stream=stream)
        op.combine(weights=op.out_w, out=out, out_weights=out_w, stream=stream)

    timed_step = step_onecall
    if args.split:
        step = step_split   # noqa: F811  (split phases replace the one-stream step)
        timed_step = step_split

    graph = None
    if not args.eager:
        with torch.cuda.stream(stream):
            for _ in range(3):
                timed_step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            timed_step()
        torch.cuda.synchronize()

    sampler = ClockSampler(local_rank) if rank == 0 else None
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            timed_step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
           for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_host0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    if args.flush_l2:
        # cold L2: a write of twice the L2 size before every step, outside
        # the step's own events; the step times are summed
        flush = torch.empty(2 * torch.cuda.get_device_properties(dev).L2_cache_size,
                            dtype=torch.uint8, device=dev)
        fev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
               for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(args.steps):
            if args.flush_l2:
                flush.fill_(i & 0xFF)
                fev[i][0].record(stream)
            if graph is not None:
                graph.replay()
            else:
                timed_step()
            if args.flush_l2:
                fev[i][1].record(stream)
        stop.record(stream)
    stop.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_host1 = time.time()
    total_ms = start.elapsed_time(stop)
    if args.flush_l2:
        total_ms = float(sum(e[0].elapsed_time(e[1]) for e in fev))
    with torch.cuda.stream(stream):   # per-kernel split: the same work, eagerly
        for i in range(args.steps):
            step(evs[i])
    torch.cuda.synchronize()
    lay = np.array([e[0].elapsed_time(e[1]) for e in evs])
    dis = np.array([e[1].elapsed_time(e[2]) for e in evs])
    com = np.array([e[2].elapsed_time(e[3]) for e in evs])
    clocks = sampler.summary(t_host0, t_host1) if sampler else None
    if sampler:
        sampler.stop()
    st, mask = op.get_error(stream)

    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(N, world, ms_per_step)

    ab = algorithmic_bytes(wl, P, N, wl.fp8, fp8_input=args.fp8_input,
                           y_bytes={"fp32": 4, "bf16": 2, "fp8_e4m3": 1 + 4 / 128}[args.combine_dtype],
                           scatter=args.combine_mode == "scatter")
    step_bytes = ab["dispatch"] + ab["combine"]
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    peak, peak_kind = measured_peak()
    d_ms, c_ms = float(dis.mean()), float(com.mean())
    dominant = "combine" if c_ms >= d_ms else "dispatch"
    dom_ms = c_ms if dominant == "combine" else d_ms
    achieved = ab[dominant] / (dom_ms / 1e3) / 1e9
    kname = ("combine_kernel" if dominant == "combine"
             else ("dispatch_kernel" if wl.fp8 and not args.fp8_input
                   else "dispatch_bulk_kernel"))

    # end to end: pinned host inputs -> device, path, combined output -> host.
    # Every step copies its own inputs in and its combined output out; the
    # copies of neighbouring steps overlap the compute through three streams
    # (H2D of step i+1 | dispatch + combine of step i | D2H of step i-1) and
    # double-buffered device inputs and outputs.
    e2e = None
    if args.e2e_steps > 0:
        hx = x.cpu().pin_memory()
        hsc = None if xsc is None else xsc.cpu().pin_memory()
        hw = torch.from_numpy(inp.weights).pin_memory()
        hi = torch.from_numpy(inp.indices).pin_memory()
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
        e2e = {"value": job_throughput(N, world, e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e_ms, "pipelined": "H2D / compute / D2H on three streams",
               "output_check": "pass" if e2e_ok else "FAIL",
               "host_link": {"copy_ms": link_ms,
                             "h2d_gb_per_s": h2d / (link_ms / 1e3) / 1e9,
                             "d2h_gb_per_s": d2h / (link_ms / 1e3) / 1e9,
                             "frac": link_ms / e_ms,
                             "what": "the step's H2D and D2H bytes copied concurrently, "
                                     "alone: the bound of the pipelined step"}}

    moe = None
    if args.moe_group:
        # standard-MoE conversion after the step's dispatch: grouping, identity
        # experts (a copy, untimed), un-grouping into the combine buffer
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
        moe = {"entries": n_ent, "gcap": args.moe_group, "errors": int(mask_m),
               "group_ms": g_ms, "ungroup_ms": u_ms,
               "group_gb_per_s": g_bytes / (g_ms / 1e3) / 1e9,
               "ungroup_gb_per_s": u_bytes / (u_ms / 1e3) / 1e9,
               "group_algorithmic_bytes": int(g_bytes),
               "ungroup_algorithmic_bytes": int(u_bytes)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, inp)

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
            "l2": ("L2 flushed before every timed step (a write of twice its size), "
                   "the flush outside the step's events" if args.flush_l2 else
                   f"no flush: each step moves {step_bytes / 1e6:.0f} MB "
                   f"({step_bytes / l2_bytes:.1f}x the {l2_bytes / 1e6:.0f} MB L2) between "
                   "two reads of any input (every input and output is read or written once "
                   "per step)"
                   if step_bytes >= 2 * l2_bytes else
                   f"warm L2: the step's {step_bytes / 1e6:.1f} MB fit in the "
                   f"{l2_bytes / 1e6:.0f} MB L2 (--flush-l2 gives the cold figure)"),
            "parallelism": f"replicas x{world}",
            "step": ("dispatch_send (layout + copy) on stream A, dispatch_recv + "
                     "combine_send on stream B, combine_recv on A" if args.split else
                     "dispatch (layout kernel, then the copy launched programmatically "
                     "after it) + combine, one stream; per-kernel times from the same "
                     "work as layout + dispatch_send (routing replay) + dispatch_recv + "
                     "combine")
                    + ("" if args.eager else
                       "; timed as a CUDA-graph replay of the step (per-kernel times eager)"),
        },
        "gb_per_s": step_bytes / (ms_per_step / 1e3) / 1e9,
        "frac_of_nominal_8tbs": step_bytes / (ms_per_step / 1e3) / 1e9 / NOMINAL_HBM_GBS,
        "frac_of_measured_hbm": step_bytes / (ms_per_step / 1e3) / 1e9 / peak,
        "algorithmic_bytes_per_step": int(step_bytes),
        "layout_ms": float(lay.mean()),
        "dispatch_ms": d_ms,
        "combine_ms": c_ms,
        "dispatch_gb_per_s": ab["dispatch"] / (d_ms / 1e3) / 1e9,
        "combine_gb_per_s": ab["combine"] / (c_ms / 1e3) / 1e9,
        "roofline": {
            "bound": "hbm",
            "kernel": kname,
            "achieved": achieved,
            "peak": peak,
            "peak_kind": f"of {peak_kind} (hbm_gbs copy bandwidth)",
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": recorded_traffic(kname, wl.name),
            "algorithmic_bytes_per_launch": int(ab[dominant]),
        },
        "identity_check": "pass" if ident_ok else "FAIL",
        "device_errors": int(mask),
        # this library's kernels per timed step: layout, copy, (receive,) combine
        "gpu_launches": (3 + (1 if args.split else 0) +
                         (1 if args.combine_mode == "scatter" else 0)) * args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if moe is not None:
        res["standard_moe"] = moe
    return res


# ------------------------------------------------------------ CPU oracle

def cpu_baseline(wl, inp, repeats=1):
    """The oracle as it stands (scalar C, one thread) on one batch of the
    benchmark's own inputs (a bounded sample: one step's worth, about
    5-15 s of CPU work): layout + dispatch + combine, the combine reading
    the dispatched rows as the expert output."""
    import oracle
    swl = wl
    cap = swl.world_size * swl.max_tokens_per_rank
    sample_tokens = swl.max_tokens_per_rank
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        pos, C, rc = oracle.layout(swl, inp.indices, inp.num_tokens)
        d = oracle.dispatch(swl, inp.x_bits, inp.weights, inp.indices,
                            inp.num_tokens, pos, cap)
        y = d["out"] if not swl.fp8 else np.zeros((swl.world_size, cap, swl.hidden), np.uint16)
        oracle.combine(swl, inp.num_tokens, pos, y, d["out_w"], cap)
        times.append(time.perf_counter() - t0)
    tsec = float(np.median(times))
    n = swl.world_size * swl.max_tokens_per_rank
    return {"value": n / tsec, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{wl.name} recipe at T={sample_tokens} tokens/rank "
                      f"({n} tokens, H={swl.hidden}); layout+dispatch+combine; "
                      f"{tsec:.2f} s wall, single thread",
            "seconds": tsec}


def workload_text(wl, args):
    """The workload as both arms name it in `config`."""
    return (f"{wl.name}: W={wl.world_size} logical ranks on one GPU, E={wl.num_experts}, "
            f"k={wl.topk}, T={wl.max_tokens_per_rank} tokens/rank, H={wl.hidden}, "
            f"{'fp8 e4m3' if wl.fp8 else 'bf16'} dispatch"
            f"{' of a pre-quantised payload' if args.fp8_input else ''}, "
            f"fp32-accumulate bf16 combine of {args.combine_dtype} expert rows "
            f"with weights, {wl.routing} routing")


def run_reference(args):
    """--impl reference: the CPU oracle, timed per step on a bounded sample."""
    import oracle
    from combine_ep_layout_06_gb300 import inputs as gen
    wl = gen.WORKLOADS[args.workload]
    sample = 256
    swl = wl.scaled(sample)
    inp = gen.make_inputs(swl)
    cap = swl.world_size * sample
    n = swl.world_size * sample

    def step():
        pos, C, rc = oracle.layout(swl, inp.indices, inp.num_tokens)
        d = oracle.dispatch(swl, inp.x_bits, inp.weights, inp.indices,
                            inp.num_tokens, pos, cap)
        y = d["out"] if not swl.fp8 else np.zeros((swl.world_size, cap, swl.hidden), np.uint16)
        oracle.combine(swl, inp.num_tokens, pos, y, d["out_w"], cap)

    for _ in range(args.warmup):
        step()
    steps = max(1, args.steps)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    tsec = (time.perf_counter() - t0) / steps
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
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1,
                         "kind": "oracle",
                         "sample": f"{n} tokens of the {wl.name} recipe per step"},
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
