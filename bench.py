#!/usr/bin/env python
"""Benchmark of the MoE dispatch / combine hot path on one GB300 (or N replicas).

One step = dispatch layout (2 kernels) -> bf16 dispatch -> combine over the
DeepSeek-V3-shaped workload: 4096 tokens, hidden 7168, 256 experts over 8
virtual ranks, top-8 (seeded synthetic routing and activations).  Inputs are
resident in HBM; L2 is flushed (a 256 MB write, then a 256 MB read of another
buffer) between timed steps, outside the CUDA-event brackets.  Prints one
JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (single-threaded C) on bounded samples
of the same workload -- the only reference there is for this path.
Under torchrun (N > 1) each rank runs an independent replica (weak scaling,
no collective on the data path); rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dispatch / combine HBM GB/s and tokens/s on 1 GB300, % of HBM roofline"
WORKLOAD = "dsv3"
L2_FLUSH_BYTES = 256 << 20


# ------------------------------------------------------------ byte accounting

# Secondary legs run after the timed step (each reported under "ops"); the
# headline step and its layout / dispatch split always run.
LEGS = ("fp8", "mxfp8", "backward", "ll", "sources", "workloads", "channels", "e2e")
# the other routing shapes, measured as an eager flushed step each (secondary figures)
OTHER_WORKLOADS = ("qwen_skew", "ds16_wide")
# CTA counts of the channel sweep (the pages fill NVLink with 4 SMs; HBM needs many more)
SWEEP_CTAS = (4, 8, 16, 32, 64, 152, 304, 608, 1216)


def workload_label(wl):
    """What the workload is, with its sizes."""
    kind = {"dsv3": "DeepSeek-V3 shape", "dsv3_fp8": "DeepSeek-V3 shape",
            "qwen_skew": "Qwen3-235B-like shape, Zipf-skewed routing",
            "ds16_wide": "DeepSeek-16B-like shape over 32 ranks", "tiny": "toy shape"}.get(wl.name, wl.name)
    return (f"{kind}: {wl.T} tokens, hidden {wl.H}, {wl.E} experts / {wl.R} virtual ranks, top-{wl.K}")


def algorithmic_bytes(T, H, E, R, K, n_pairs, n_valid, capacity):
    """Minimum HBM bytes of each operator: every input byte read once, every
    output byte written once (x is read once, not once per destination)."""
    layout = 4 * T * K * 2 + 4 * T * R + 4 * T * K * 3 + 4 * capacity + 4 * (3 * E + 2 * R + 4)
    dispatch = 2 * T * H + 2 * H * n_pairs + 4 * T * R
    dispatch_fp8 = 2 * T * H + n_pairs * (H + 4 * (H // 128)) + 4 * T * R
    dispatch_mxfp8 = 2 * T * H + n_pairs * (H + H // 32) + 4 * T * R
    combine = 2 * H * n_valid + 2 * T * H + 8 * T * K
    dispatch_bwd = 2 * H * n_pairs + 2 * T * H + 4 * T * R
    combine_bwd = 2 * T * H + 4 * H * n_valid + 12 * T * K
    return {"dispatch_backward": dispatch_bwd, "combine_backward": combine_bwd, "layout": layout, "dispatch": dispatch, "dispatch_fp8": dispatch_fp8, "dispatch_mxfp8": dispatch_mxfp8,
            "combine": combine}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def committed_traffic(kernel_file: str, profile_name: str):
    """DRAM bytes per launch from a committed ncu summary, or None if the
    summary is missing or the kernel source changed since it was taken."""
    prof = os.path.join(ROOT, "profiles", profile_name)
    src = os.path.join(ROOT, "combine_moe_dispatch_02_gb300", "csrc", kernel_file)
    if not os.path.exists(prof):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    vals = {}
    for line in open(prof):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256_16") != sha:
        return None
    try:
        return int(float(vals["dram_bytes_per_full_launch"]))
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------- multi-rank

def max_over_ranks(ms: float, world: int, device=None) -> float:
    """Slowest rank's time (replicas run in lock step between barriers)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbps(step_bytes: int, ms_step_max: float, world: int) -> float:
    """Whole-job throughput: every replica moves step_bytes per step; the job
    takes as long as its slowest rank."""
    return world * step_bytes / (ms_step_max * 1e-3) / 1e9


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, log_path: str | None = None):
        self.gpu = gpu_index
        self.proc = None
        self.log_path = log_path        # where to keep the raw samples; a temporary file if None
        self.path = None

    def start(self):
        try:
            if self.log_path:
                os.makedirs(os.path.dirname(os.path.abspath(self.log_path)), exist_ok=True)
                self.path = self.log_path
            else:
                fd, self.path = tempfile.mkstemp(prefix=f"clocks_rank{self.gpu}_", suffix=".csv")
                os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            if self.path and not self.log_path and os.path.exists(self.path):
                os.unlink(self.path)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not self.log_path:
            os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ L2 flush

class L2Flush:
    """Between timed steps: write a 256 MB buffer (twice the 129 MB L2), then
    read a second one, so that the step starts with an L2 holding only clean
    lines of unrelated data -- no cached inputs, and no dirty flush lines whose
    write-back would be charged to the next kernel."""

    def __init__(self, dev):
        import torch
        self.a = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.b = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.n = 0

    def __call__(self):
        self.n += 1
        self.a.fill_(self.n)
        self.b.max()


# ------------------------------------------------------------------ our arm

def run_ours(args, rank, world, local_rank):
    import torch
    from combine_moe_dispatch_02_gb300 import build as cuda_build
    from combine_moe_dispatch_02_gb300 import ep
    from combine_moe_dispatch_02_gb300.inputs import WORKLOADS, make_inputs

    cuda_build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = WORKLOADS[args.workload]
    inp = make_inputs(wl, seed=rank)
    T, H, E, R, K = wl.T, wl.H, wl.E, wl.R, wl.K

    L = ep.Layout(T, K, E, R, device=dev)
    x = inp.x.to(dev)
    idx = inp.topk_idx.to(dev)
    w = inp.topk_w.to(dev)
    y = inp.y.to(dev)
    recv, _ = ep.alloc_recv(L, H, False, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None, split=False):
        if evs:
            evs[0].record(stream)
        ep.moe_dispatch_layout(idx, w, E, R, L, stream)
        if split:
            evs[1].record(stream)
        ep.moe_dispatch(x, L, False, recv, None, stream)
        if evs:
            evs[2 if split else 1].record(stream)
        ep.moe_combine(y, L, w, out, stream)
        if evs:
            evs[3 if split else 2].record(stream)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize(dev)
    st, flags = ep.moe_layout_read_status(L, stream)
    if st != 0:
        raise RuntimeError(f"device status {st} ({ep.moe_status_string(st)}) flags {flags:#x}")
    n_pairs = int(L.rank_offset[R].item())
    n_valid = int(L.expert_offset[E].item())
    ab = algorithmic_bytes(T, H, E, R, K, n_pairs, n_valid, L.capacity)
    step_bytes = ab["layout"] + ab["dispatch"] + ab["combine"]

    # The timed steps replay the whole step as one CUDA graph, captured once (the
    # programmatic launch chain layout -> dispatch is kept as graph edges), with
    # events only at the step's two ends: an event between two kernels costs
    # ~2 us of GPU time and cuts the programmatic overlap.  Per-operator times
    # come from a separate pass with events between the operators.
    cap = torch.cuda.Stream(dev)
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=cap):
        ep.moe_dispatch_layout(idx, w, E, R, L, cap)
        ep.moe_dispatch(x, L, False, recv, None, cap)
        ep.moe_combine(y, L, w, out, cap)
    for _ in range(3):
        flush()
        g_step.replay()

    def graph_step(evs):
        evs[0].record(stream)
        g_step.replay()
        evs[1].record(stream)

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local_rank, args.clocks_log.replace("{rank}", str(rank)) if args.clocks_log else None)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.perf_counter()
    for s in range(args.steps):
        flush()                   # L2 flush, outside the event brackets
        graph_step(events[s])
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    st, flags = ep.moe_layout_read_status(L, stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after timed steps")

    tot = [e[0].elapsed_time(e[1]) for e in events]
    ms_step = statistics.mean(tot)
    # per-operator split: a separate eager pass of the same step with events
    # between the operators (each after an L2 flush, like the timed steps)
    n_split = max(args.steps // 4, 3)
    ev_split = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_split)]
    for e in ev_split:
        flush()
        step(e, split=True)
    torch.cuda.synchronize(dev)
    lay = [e[0].elapsed_time(e[1]) for e in ev_split]
    dis = [e[1].elapsed_time(e[2]) for e in ev_split]
    com = [e[2].elapsed_time(e[3]) for e in ev_split]
    ms_step = max_over_ranks(ms_step, world, dev)

    peak, peak_kind = measured_peaks()
    gbps = lambda b, ms: b / (ms * 1e-3) / 1e9
    n_sec = max(args.steps // 4, 3)
    legs = set(LEGS) if args.legs == "all" else set() if args.legs == "none" else set(args.legs.split(","))

    def timed(body, n, marks):
        """n flushed repetitions of body(events) with `marks` events each;
        the mean time between consecutive events in ms."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(marks)] for _ in range(n)]
        for e in evs:
            flush()
            body(e)
        torch.cuda.synchronize(dev)
        return [statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs) for i in range(marks - 1)]

    def pct(ms_list):
        """p10 / p50 / p90 of per-repetition times, in us."""
        q = statistics.quantiles(ms_list, n=10, method="inclusive") if len(ms_list) > 1 else [ms_list[0]] * 9
        return {"p10": round(q[0] * 1e3, 2), "p50": round(statistics.median(ms_list) * 1e3, 2), "p90": round(q[8] * 1e3, 2)}

    def hbm_op(us_ms, nbytes, **extra):
        return {"us": round(us_ms * 1e3, 2), "bytes": nbytes, "GB/s": round(gbps(nbytes, us_ms), 1),
                "frac": round(gbps(nbytes, us_ms) / peak, 4), **extra}

    com_ms = statistics.mean(com)
    achieved = ab["combine"] / (com_ms * 1e-3) / 1e9
    ops = {
        "note": "per-operator times from an eager pass of the step with events between the operators",
        "step_us": pct(tot),
        "layout": {"us": round(statistics.mean(lay) * 1e3, 2), "bytes": ab["layout"], "us_pct": pct(lay)},
        "dispatch_bf16": hbm_op(statistics.mean(dis), ab["dispatch"],
                                tokens_per_s=round(T / (statistics.mean(dis) * 1e-3), 1), us_pct=pct(dis)),
        "combine": hbm_op(com_ms, ab["combine"], tokens_per_s=round(T / (com_ms * 1e-3), 1), us_pct=pct(com)),
    }

    # FP8 and MXFP8 dispatch on the same layout (secondary figures)
    for fmt, key, leg in ((ep.MOE_FORMAT_FP8, "dispatch_fp8", "fp8"), (ep.MOE_FORMAT_MXFP8, "dispatch_mxfp8", "mxfp8")):
        if leg not in legs:
            continue
        rq, rs = ep.alloc_recv(L, H, fmt, device=dev)

        def body(e, fmt=fmt, rq=rq, rs=rs):
            e[0].record(stream)
            ep.moe_dispatch(x, L, fmt, rq, rs, stream)
            e[1].record(stream)
        ops[key] = hbm_op(timed(body, n_sec, 2)[0], ab[key])
        del rq, rs

    # backward pair: gradients of the receive rows and of the output
    if "backward" in legs:
        grad_recv = torch.empty_like(recv).normal_()
        grad_out = torch.empty_like(out).normal_()
        grad_x = torch.empty_like(x)
        grad_y = torch.empty_like(y)
        grad_w = torch.empty_like(w)

        def body(e):
            e[0].record(stream)
            ep.moe_dispatch_backward(grad_recv, L, grad_x, stream)
            e[1].record(stream)
            ep.moe_combine_backward(grad_out, y, L, w, grad_y, grad_w, stream)
            e[2].record(stream)
        dbwd, cbwd = timed(body, n_sec, 3)
        ops["dispatch_backward"] = hbm_op(dbwd, ab["dispatch_backward"])
        ops["combine_backward"] = hbm_op(cbwd, ab["combine_backward"])
        del grad_recv, grad_out, grad_x, grad_y, grad_w
    st, flags = ep.moe_layout_read_status(L, stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after the secondary legs")

    # low-latency (decode) path: 128 tokens of the same shape, fixed capacity 128 per expert
    if "ll" in legs:
        T_ll = 128
        x_ll, idx_ll, w_ll = x[:T_ll].contiguous(), idx[:T_ll].contiguous(), w[:T_ll].contiguous()
        recv_ll = torch.empty(E * T_ll, H, dtype=torch.bfloat16, device=dev)
        tpe_ll = torch.empty(E, dtype=torch.int32, device=dev)
        slot_ll = torch.empty(T_ll, K, dtype=torch.int32, device=dev)
        st_ll = torch.zeros(1, dtype=torch.int32, device=dev)
        out_ll = torch.empty(T_ll, H, dtype=torch.bfloat16, device=dev)

        def body(e):
            e[0].record(stream)
            ep.moe_ll_dispatch(x_ll, idx_ll, E, T_ll, recv_ll, tpe_ll, slot_ll, st_ll, stream)
            e[1].record(stream)
            ep.moe_ll_combine(recv_ll, slot_ll, w_ll, E, T_ll, out_ll, st_ll, stream)
            e[2].record(stream)
        lld, llc = timed(body, n_sec, 3)
        if int(st_ll.item()) != 0:
            raise RuntimeError("low-latency path reported a device error")
        ll_bytes = 2 * T_ll * H + 2 * H * T_ll * K + 4 * T_ll * K    # rows read, one row per entry written
        ops["ll_dispatch_T128"] = {"us": round(lld * 1e3, 2), "bytes": ll_bytes, "GB/s": round(gbps(ll_bytes, lld), 1)}
        ops["ll_combine_T128"] = {"us": round(llc * 1e3, 2), "bytes": ll_bytes, "GB/s": round(gbps(ll_bytes, llc), 1)}
        del recv_ll

    # multi-source receive: all eight ranks' tokens of this shape at once (S = 8
    # sources of T tokens, one region of 8T rows per destination rank)
    if "sources" in legs:
        S_ms = 8
        inp_ms = make_inputs(wl.scaled(S_ms * T), seed=1000 + rank, with_y=False)
        L_ms = ep.Layout(S_ms * T, K, E, R, device=dev, sources=S_ms)
        x_ms, idx_ms, w_ms = inp_ms.x.to(dev), inp_ms.topk_idx.to(dev), inp_ms.topk_w.to(dev)
        gen = torch.Generator(device=dev).manual_seed(77 + rank)
        y_ms = torch.randn(S_ms * T * K, H, device=dev, generator=gen).to(torch.bfloat16)
        recv_ms, _ = ep.alloc_recv(L_ms, H, False, device=dev)
        out_ms = torch.empty(S_ms * T, H, dtype=torch.bfloat16, device=dev)

        def body(e):
            e[0].record(stream)
            ep.moe_dispatch_layout(idx_ms, w_ms, E, R, L_ms, stream)
            e[1].record(stream)
            ep.moe_dispatch(x_ms, L_ms, False, recv_ms, None, stream)
            e[2].record(stream)
            ep.moe_combine(y_ms, L_ms, w_ms, out_ms, stream)
            e[3].record(stream)
        msl, msd, msc = timed(body, max(args.steps // 10, 3), 4)
        st, flags = ep.moe_layout_read_status(L_ms, stream)
        if st != 0:
            raise RuntimeError(f"device status {st} in the multi-source leg")
        ab_ms = algorithmic_bytes(S_ms * T, H, E, R, K, int(L_ms.tokens_per_rank.sum().item()),
                                  int(L_ms.expert_offset[E].item()), L_ms.capacity)
        ops["multi_source_S8"] = {"note": f"8 sources x {T} tokens, one region of {8 * T} rows per destination rank",
                                  "layout_us": round(msl * 1e3, 2),
                                  "dispatch_bf16": hbm_op(msd, ab_ms["dispatch"]),
                                  "combine": hbm_op(msc, ab_ms["combine"])}
        del x_ms, y_ms, recv_ms, out_ms, L_ms

    # the other routing shapes: Zipf-skewed Qwen3-235B-like routing (one rank
    # receives nearly every token) and DeepSeek-16B-like routing over 32 ranks
    # with a narrow hidden size; each an eager flushed step of its own
    if "workloads" in legs:
        wls = {}
        for name in OTHER_WORKLOADS:
            if name == args.workload:
                continue
            wo = WORKLOADS[name]
            To, Ho, Eo, Ro, Ko = wo.T, wo.H, wo.E, wo.R, wo.K
            inp_o = make_inputs(wo, seed=rank, with_y=False)
            L_o = ep.Layout(To, Ko, Eo, Ro, device=dev)
            x_o, idx_o, w_o = inp_o.x.to(dev), inp_o.topk_idx.to(dev), inp_o.topk_w.to(dev)
            gen = torch.Generator(device=dev).manual_seed(99 + rank)
            y_o = torch.randn(To * Ko, Ho, device=dev, generator=gen).to(torch.bfloat16)
            recv_o, _ = ep.alloc_recv(L_o, Ho, False, device=dev)
            out_o = torch.empty(To, Ho, dtype=torch.bfloat16, device=dev)

            def body(e):
                e[0].record(stream)
                ep.moe_dispatch_layout(idx_o, w_o, Eo, Ro, L_o, stream)
                e[1].record(stream)
                ep.moe_dispatch(x_o, L_o, False, recv_o, None, stream)
                e[2].record(stream)
                ep.moe_combine(y_o, L_o, w_o, out_o, stream)
                e[3].record(stream)
            ol, od, oc = timed(body, n_sec, 4)
            st, flags = ep.moe_layout_read_status(L_o, stream)
            if st != 0:
                raise RuntimeError(f"device status {st} in the {name} leg")
            tpr = L_o.tokens_per_rank.cpu()
            ab_o = algorithmic_bytes(To, Ho, Eo, Ro, Ko, int(tpr.sum()), int(L_o.expert_offset[Eo].item()),
                                     L_o.capacity)
            wls[name] = {"shape": workload_label(wo), "n_pairs": int(tpr.sum()),
                         "rows_per_rank_min_max": [int(tpr.min()), int(tpr.max())],
                         "layout_us": round(ol * 1e3, 2),
                         "dispatch_bf16": hbm_op(od, ab_o["dispatch"], tokens_per_s=round(To / (od * 1e-3), 1)),
                         "combine": hbm_op(oc, ab_o["combine"], tokens_per_s=round(To / (oc * 1e-3), 1))}
            del x_o, y_o, recv_o, out_o, L_o
        ops["other_workloads"] = wls

    # how many CTAs ("channels") the HBM-bound operators need: bf16 dispatch (one
    # warp per CTA) and combine (256 threads per CTA) at fixed CTA counts
    if "channels" in legs:
        sweep = {"note": "GB/s at a fixed number of CTAs; default = the operator's own grid", "dispatch_bf16": {},
                 "combine": {}}
        for n_cta in SWEEP_CTAS + (0,):
            def body_d(e, n_cta=n_cta):
                e[0].record(stream)
                ep.moe_dispatch(x, L, False, recv, None, stream, num_channels=n_cta, variant=1)
                e[1].record(stream)

            def body_c(e, n_cta=n_cta):
                e[0].record(stream)
                ep.moe_combine(y, L, w, out, stream, num_channels=n_cta)
                e[1].record(stream)
            key = str(n_cta) if n_cta else "default"
            sweep["dispatch_bf16"][key] = round(gbps(ab["dispatch"], timed(body_d, 10, 2)[0]), 1)
            sweep["combine"][key] = round(gbps(ab["combine"], timed(body_c, 10, 2)[0]), 1)
        ops["channel_sweep"] = sweep

    e2e = run_e2e(args, inp, L, dev, ab, step_bytes) if (rank == 0 and "e2e" in legs) else None

    result = {
        "metric": METRIC,
        "value": round(aggregate_gbps(step_bytes, ms_step, world), 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": f"synthetic (seeded N(0,1) activations, softmax top-{K} routing of N(0,1) logits"
                + (f", Zipf s={wl.zipf_s} expert bias)" if wl.zipf_s else ")"),
        "config": {"workload": workload_label(wl),
                   "T": T, "H": H, "E": E, "R": R, "K": K, "n_pairs": n_pairs, "capacity": L.capacity,
                   "step": "layout + bf16 dispatch + combine", "l2": "flushed between steps (256 MB write, then 256 MB read of another buffer)",
                   "launch": "timed steps replay one CUDA graph (layout -> dispatch -> combine)",
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": round(world * T / (ms_step * 1e-3), 1),
        "ops": ops,
        "roofline": {"bound": "hbm", "kernel": f"combine_kernel<{K if K in (1, 2, 4, 6, 8) else 0}>", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s",
                     "traffic": committed_traffic("combine.cu", "combine_dsv3_ncu.md") if args.workload == WORKLOAD
                     else None,
                     "timing": "combine between events in the eager per-operator pass, after the dispatch",
                     "algorithmic_bytes": ab["combine"]},
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(t_wall, 3),
    }
    if e2e is not None:
        result["e2e"] = e2e
    return result


def run_e2e(args, inp, L, dev, ab, step_bytes):
    """Same step through the public API with host buffers: pinned host ->
    device copies of the inputs, the three calls, device -> host copy of the
    combine output and the per-expert counts, every step inside the timed
    region.  Two device buffer sets: the inputs of step i+1 are copied on a
    copy stream while step i computes and copies its result back, as a
    serving or training loop would overlap them."""
    import torch
    from combine_moe_dispatch_02_gb300 import ep
    wl = inp.wl
    hx = inp.x.pin_memory()
    hidx = inp.topk_idx.pin_memory()
    hw = inp.topk_w.pin_memory()
    hy = inp.y.pin_memory()
    hout = torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
    hcnt = torch.empty(wl.E, dtype=torch.int32).pin_memory()
    bufs = [{"x": torch.empty_like(inp.x, device=dev), "idx": torch.empty_like(inp.topk_idx, device=dev),
             "w": torch.empty_like(inp.topk_w, device=dev), "y": torch.empty_like(inp.y, device=dev)}
            for _ in range(2)]
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    recv, _ = ep.alloc_recv(L, wl.H, False, device=dev)
    comp = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    n = max(3, min(args.steps // 10, 50))

    def run(steps):
        for i in range(steps):
            b = bufs[i % 2]
            if i >= 2:
                copy.wait_event(consumed[i % 2])       # step i-2 is done with this buffer set
            with torch.cuda.stream(copy):
                b["x"].copy_(hx, non_blocking=True)
                b["idx"].copy_(hidx, non_blocking=True)
                b["w"].copy_(hw, non_blocking=True)
                b["y"].copy_(hy, non_blocking=True)
            copied[i % 2].record(copy)
            comp.wait_event(copied[i % 2])
            ep.moe_dispatch_layout(b["idx"], b["w"], wl.E, wl.R, L, comp)
            ep.moe_dispatch(b["x"], L, False, recv, None, comp)
            ep.moe_combine(b["y"], L, b["w"], out, comp)
            consumed[i % 2].record(comp)
            hout.copy_(out, non_blocking=True)
            hcnt.copy_(L.tokens_per_expert, non_blocking=True)

    run(3)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    copy.wait_event(e0)
    run(n)
    comp.wait_stream(copy)
    e1.record(comp)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / n
    st, _ = ep.moe_layout_read_status(L, comp)
    if st != 0:
        raise RuntimeError(f"device status {st} in the end-to-end leg")
    h2d = hx.numel() * 2 + hidx.numel() * 4 + hw.numel() * 4 + hy.numel() * 2
    d2h = hout.numel() * 2 + hcnt.numel() * 4
    return {"value": round(step_bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "overlap": "inputs of step i+1 copied while step i computes (two device buffer sets)"}


# ------------------------------------------------------------ CPU baselines

def oracle_step_fn(wl, inp, T_s):
    """One oracle pass (layout, bf16 dispatch, combine) over the first T_s
    tokens of the workload; returns (callable, algorithmic bytes)."""
    import numpy as np
    import oracle
    from combine_moe_dispatch_02_gb300.inputs import bf16_bits
    idx = inp.topk_idx[:T_s].numpy()
    w = inp.topk_w[:T_s].numpy()
    xb = bf16_bits(inp.x[:T_s])
    # y rows for these tokens: the first T_s * K expert-major rows stand in
    yb = bf16_bits(inp.y[: T_s * wl.K])
    Lo = oracle.layout(idx, w, wl.E, wl.R)
    ab = algorithmic_bytes(T_s, wl.H, wl.E, wl.R, wl.K, Lo.n_pairs, int(Lo.expert_offset[wl.E]), Lo.capacity)

    def run():
        L = oracle.layout(idx, w, wl.E, wl.R)
        oracle.dispatch_bf16(xb, L)
        oracle.combine(yb, L.expert_slot, w)
    return run, ab["layout"] + ab["dispatch"] + ab["combine"]


def cpu_baseline(wl, inp, budget_s=10.0):
    """The oracle as it stands, single-threaded, timed on this host over the
    full workload repeated until about `budget_s` seconds have passed."""
    run, nbytes = oracle_step_fn(wl, inp, wl.T)
    run()  # warm-up
    t0 = time.perf_counter()
    n = 0
    while True:
        run()
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = (time.perf_counter() - t0) / n
    return {"value": round(nbytes / dt / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"full workload ({wl.T} tokens) x {n} passes of layout + bf16 dispatch + combine, "
                      f"{dt:.3f} s each, 1 thread", "host_cpu": _cpu_name(), "host_cores": os.cpu_count()}


def _cpu_name():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def run_reference(args):
    """Reference arm: the CPU oracle on bounded per-step samples of the
    workload (the first T_s tokens, T_s sized so the run stays short)."""
    from combine_moe_dispatch_02_gb300.inputs import WORKLOADS, make_inputs
    import oracle
    oracle.build()
    wl = WORKLOADS[args.workload]
    inp = make_inputs(wl, seed=0)
    probe, _ = oracle_step_fn(wl, inp, 128)
    t0 = time.perf_counter()
    probe()
    per_tok = (time.perf_counter() - t0) / 128
    target = 60.0 / max(args.steps + args.warmup, 1)         # about a minute in total
    T_s = int(max(32, min(wl.T, target / max(per_tok, 1e-9))))
    run, nbytes = oracle_step_fn(wl, inp, T_s)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    dt = statistics.mean(times)
    v = round(nbytes / dt / 1e9, 3)
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": f"DeepSeek-V3 shape, first {T_s} of {wl.T} tokens per step",
                                            "T_sample": T_s, "H": wl.H, "E": wl.E, "R": wl.R, "K": wl.K},
            "cpu_baseline": {"value": v, "unit": "GB/s", "kind": "oracle", "cores": 1,
                             "sample": f"{T_s} tokens of the 4096-token workload per step, 1 thread",
                             "host_cpu": _cpu_name()},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-log", default=None,
                    help="keep the raw nvidia-smi samples of the timed region here ({rank} is replaced)")
    ap.add_argument("--legs", default="all",
                    help="secondary legs after the timed step: 'all', 'none' or a comma list of " + ",".join(LEGS))
    args = ap.parse_args()
    if args.legs not in ("all", "none") and not set(args.legs.split(",")) <= set(LEGS):
        ap.error(f"--legs: choose 'all', 'none' or from {','.join(LEGS)}")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)))
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            from combine_moe_dispatch_02_gb300.inputs import WORKLOADS, make_inputs
            wl = WORKLOADS[args.workload]
            res["cpu_baseline"] = cpu_baseline(wl, make_inputs(wl, seed=0))
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
