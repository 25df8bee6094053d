#!/usr/bin/env python
"""Benchmark of the MoE dispatch / combine hot path on one GB300 (or N replicas).

One step = dispatch layout (2 kernels) -> dispatch -> combine over the
DeepSeek-V3-shaped workload: 4096 tokens, hidden 7168, 256 experts over 8
virtual ranks, top-8 (seeded synthetic routing and activations), made with
the library's moe_dispatch_with_layout call (layout and dispatch in one
call) and moe_combine; the three separate calls are timed as
ops.step_separate_calls.  The dispatch writes bf16 rows, or FP8 E4M3 rows
with 1x128 fp32 scales under ``--workload dsv3_fp8``.  Inputs are resident in HBM; L2 is flushed (a 256 MB
write, then a 256 MB read of another buffer) between timed steps, outside the
CUDA-event brackets.  Prints one JSON line.

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
# GB300 datasheet HBM3e bandwidth (~8 TB/s): the second denominator of every
# fraction, next to the measured copy rate
SPEC_HBM_GBS = 8000.0
L2_POLICY = ("GPU arm: L2 flushed between timed repetitions (256 MB write, then 256 MB read of another "
             "buffer), outside the event brackets; CPU oracle arm: host memory, no flush")

# Secondary legs run after the timed step (each reported under "ops"); the
# headline step and its per-operator split always run.
LEGS = ("formats", "backward", "ll", "sources", "workloads", "channels", "e2e")
# the other routing shapes, measured as steps of their own (secondary figures)
OTHER_WORKLOADS = ("qwen_skew", "ds16_wide")
# CTA counts of the channel sweep (the pages fill NVLink with 4 SMs; HBM needs many more)
SWEEP_CTAS = (4, 8, 16, 32, 64, 152, 304, 608, 1216)

FORMAT_NAMES = {0: "bf16", 1: "fp8", 2: "mxfp8"}


# ------------------------------------------------------------ byte accounting

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


def dispatch_key(fmt: int) -> str:
    """Key of algorithmic_bytes for a receive format."""
    return {0: "dispatch", 1: "dispatch_fp8", 2: "dispatch_mxfp8"}[int(fmt)]


def step_label(fmt: int) -> str:
    return {0: "layout + bf16 dispatch + combine",
            1: "layout + FP8 E4M3 dispatch (1x128 fp32 scales) + combine of bf16 expert outputs"}[int(fmt)]


# the calls a step makes: the layout and the dispatch in one moe_dispatch_with_layout call (its
# dispatch may read x while the layout is computed), then moe_combine
STEP_CALLS = "moe_dispatch_with_layout (layout + dispatch in one call) + moe_combine"


def step_config(wl, fmt, n_pairs, capacity, world, T_sample=None):
    """The `config` object of both arms: the workload, the step and the L2
    policy; a CPU sample of fewer tokens than the workload says so in its
    workload string."""
    label = workload_label(wl)
    if T_sample is not None and T_sample < wl.T:
        label += f" (first {T_sample} of {wl.T} tokens per step)"
    return {"workload": label, "T": wl.T if T_sample is None else T_sample, "H": wl.H, "E": wl.E, "R": wl.R,
            "K": wl.K, "n_pairs": n_pairs, "capacity": capacity, "step": step_label(fmt), "l2": L2_POLICY,
            "parallelism": f"replicas x{world}"}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def committed_traffic(record: str):
    """DRAM bytes per launch from a committed one-launch ncu record
    (profiles/<record>.json), with the capture it came from; (None, why) if
    the record is missing or a source it names has changed since."""
    path = os.path.join(ROOT, "profiles", record + ".json")
    if not os.path.exists(path):
        return None, "no committed capture"
    with open(path) as f:
        rec = json.load(f)
    for src, sha in rec["source_sha256_16"].items():
        with open(os.path.join(ROOT, "combine_moe_dispatch_02_gb300", "csrc", src), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != sha:
                return None, f"{src} changed since the committed capture"
    return int(rec["dram_bytes_per_launch"]), f"profiles/{record}.json: {rec['capture']}"


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


# ------------------------------------------------------------------ timers

class Timer:
    """Flushed, warmed-up CUDA-event timing on one stream.

    eager(body, n, marks): `warmup` untimed repetitions of body(mark), then n
    recorded ones; body calls mark(i) for i = 0 .. marks-1 between its
    launches; returns, per interval, the list of per-repetition times (ms).
    graph(fn, n): fn(stream) captured once as a CUDA graph, then replayed the
    same way with events only at its two ends; returns per-replay times (ms).
    """

    def __init__(self, torch, dev, stream, flush, warmup):
        self.torch, self.dev, self.stream, self.flush, self.warmup = torch, dev, stream, flush, warmup

    def _ev(self):
        return self.torch.cuda.Event(enable_timing=True)

    def eager(self, body, n, marks):
        for _ in range(self.warmup):
            self.flush()
            body(lambda i: None)
        evs = []
        for _ in range(n):
            e = [self._ev() for _ in range(marks)]
            self.flush()
            body(lambda i, e=e: e[i].record(self.stream))
            evs.append(e)
        self.torch.cuda.synchronize(self.dev)
        return [[e[i].elapsed_time(e[i + 1]) for e in evs] for i in range(marks - 1)]

    def capture(self, fn):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream(self.dev)
        cs.wait_stream(self.stream)
        with torch.cuda.graph(g, stream=cs):
            fn(cs)
        self.stream.wait_stream(cs)
        return g

    def replay(self, g, n):
        for _ in range(self.warmup):
            self.flush()
            g.replay()
        evs = []
        for _ in range(n):
            e0, e1 = self._ev(), self._ev()
            self.flush()
            e0.record(self.stream)
            g.replay()
            e1.record(self.stream)
            evs.append((e0, e1))
        self.torch.cuda.synchronize(self.dev)
        return [a.elapsed_time(b) for a, b in evs]

    def graph(self, fn, n):
        return self.replay(self.capture(fn), n)

    def back_to_back(self, fns, n):
        """fns (each fn(stream) one launch, typically on its own buffer set)
        captured back to back in one graph, replayed like graph(); per-launch
        times (ms): a replay's time over len(fns)."""
        g = self.capture(lambda s: [f(s) for f in fns])
        return [t / len(fns) for t in self.replay(g, n)]


def pct(ms_list):
    """p10 / p50 / p90 of per-repetition times, in us."""
    q = statistics.quantiles(ms_list, n=10, method="inclusive") if len(ms_list) > 1 else [ms_list[0]] * 9
    return {"p10": round(q[0] * 1e3, 2), "p50": round(statistics.median(ms_list) * 1e3, 2),
            "p90": round(q[8] * 1e3, 2)}


def gbps(nbytes, ms):
    return nbytes / (ms * 1e-3) / 1e9


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
    fmt = ep.MOE_FORMAT_FP8 if wl.fp8 else ep.MOE_FORMAT_BF16
    inp = make_inputs(wl, seed=rank)
    T, H, E, R, K = wl.T, wl.H, wl.E, wl.R, wl.K

    L = ep.Layout(T, K, E, R, device=dev)
    x = inp.x.to(dev)
    idx = inp.topk_idx.to(dev)
    w = inp.topk_w.to(dev)
    y = inp.y.to(dev)
    recv, recv_s = ep.alloc_recv(L, H, fmt, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    tm = Timer(torch, dev, stream, flush, args.warmup)
    peak, peak_kind = measured_peaks()
    # repetitions of each secondary figure (each after its own warm-up)
    n_sec = max(20, min(args.steps // 4, 400))
    n_stream = max(10, n_sec // 8)

    def check(layout, what):
        st, flags = ep.moe_layout_read_status(layout, stream)
        if st != 0:
            raise RuntimeError(f"device status {st} ({ep.moe_status_string(st)}) flags {flags:#x} {what}")

    def step_ops(s, f=fmt, rq=recv, rs=recv_s):
        ep.moe_dispatch_with_layout(idx, w, E, R, L, x, f, rq, rs, s)
        ep.moe_combine(y, L, w, out, s)

    def step_ops_separate(s, f=fmt, rq=recv, rs=recv_s):
        ep.moe_dispatch_layout(idx, w, E, R, L, s)
        ep.moe_dispatch(x, L, f, rq, rs, s)
        ep.moe_combine(y, L, w, out, s)

    for _ in range(args.warmup):
        flush()
        step_ops(stream)
    torch.cuda.synchronize(dev)
    check(L, "after the warm-up steps")
    n_pairs = int(L.rank_offset[R].item())
    n_valid = int(L.expert_offset[E].item())
    ab = algorithmic_bytes(T, H, E, R, K, n_pairs, n_valid, L.capacity)
    dkey = dispatch_key(fmt)
    step_bytes = ab["layout"] + ab[dkey] + ab["combine"]

    def hbm_op(nbytes, ms_list, eager_ms=None, stream_ms=None, **extra):
        """Graph-replayed figure (the fraction's time) and, if given, the
        eager one with events between launches and the back-to-back one over
        rotating buffer sets (frac_stream)."""
        ms = statistics.mean(ms_list)
        d = {"us": round(ms * 1e3, 2), "us_pct": pct(ms_list), "bytes": nbytes, "GB/s": round(gbps(nbytes, ms), 1),
             "frac": round(gbps(nbytes, ms) / peak, 4), "frac_spec": round(gbps(nbytes, ms) / SPEC_HBM_GBS, 4)}
        if eager_ms is not None:
            d["eager_us"] = round(statistics.mean(eager_ms) * 1e3, 2)
        if stream_ms is not None:
            sm = statistics.mean(stream_ms)
            d["stream_us"] = round(sm * 1e3, 2)
            d["frac_stream"] = round(gbps(nbytes, sm) / peak, 4)
        d.update(extra)
        return d

    # back-to-back launches over NB rotating buffer sets: every launch's inputs
    # were last touched NB launches earlier, with well over L2's 129 MB of
    # other traffic in between, so none is served from L2, and the launches
    # pay the write-back of their predecessors' dirty lines as a pipeline of
    # layers would; no event or launch gap sits inside the figure
    NB = 4
    xs = [x] + [x.clone() for _ in range(NB - 1)]
    ys = [y] + [y.clone() for _ in range(NB - 1)]
    outs = [out] + [torch.empty_like(out) for _ in range(NB - 1)]

    def rotating(op, bufs):
        return [lambda s, i=i: op(s, bufs[i % NB], i % NB) for i in range(2 * NB)]

    def stream_dispatch(f):
        sets = [ep.alloc_recv(L, H, f, device=dev) for _ in range(NB)]
        ms = tm.back_to_back(rotating(lambda s, b, i: ep.moe_dispatch(xs[i], L, f, b[0], b[1], s), sets), n_stream)
        del sets
        return ms

    # The timed steps replay the whole step as one CUDA graph, captured once (the
    # programmatic launch chain layout -> dispatch is kept as graph edges), with
    # events only at the step's two ends: an event between two kernels costs
    # ~2 us of GPU time and cuts the programmatic overlap.  Per-operator times
    # come from separate passes.
    # The steps rotate over NPLACE independently allocated buffer sets (layout,
    # routing, x, receive rows, y, out; set 0 is the one above), one graph
    # each: on GB300 the step moves by up to ~2 us with where its buffers land
    # in HBM (six placements in one process: 149.2-151.2 us), so the mean over
    # several placements is the steadier figure.  No placement is selected.
    NPLACE = 4
    places = [(L, idx, w, recv, recv_s)]
    for i in range(1, NPLACE):
        L_i = ep.Layout(T, K, E, R, device=dev)
        rq_i, rs_i = ep.alloc_recv(L_i, H, fmt, device=dev)
        places.append((L_i, idx.clone(), w.clone(), rq_i, rs_i))

    def place_step(i):
        L_i, idx_i, w_i, rq_i, rs_i = places[i]

        def fn(s):
            ep.moe_dispatch_with_layout(idx_i, w_i, E, R, L_i, xs[i], fmt, rq_i, rs_i, s)
            ep.moe_combine(ys[i], L_i, w_i, outs[i], s)
        return fn

    g_steps = [tm.capture(place_step(i)) for i in range(NPLACE)]
    for _ in range(3):
        for g_ in g_steps:
            flush()
            g_.replay()

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
        events[s][0].record(stream)
        g_steps[s % NPLACE].replay()
        events[s][1].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()
    for i in range(NPLACE):
        check(places[i][0], f"after the timed steps (buffer set {i})")
    tot = [e[0].elapsed_time(e[1]) for e in events]
    ms_step = max_over_ranks(statistics.mean(tot), world, dev)

    # per-operator split: an eager pass of the same step with events between
    # the operators (the combine runs after the dispatch, as in the step)
    def split_body(mark):
        mark(0)
        ep.moe_dispatch_layout(idx, w, E, R, L, stream)
        mark(1)
        ep.moe_dispatch(x, L, fmt, recv, recv_s, stream)
        mark(2)
        ep.moe_combine(y, L, w, out, stream)
        mark(3)
    lay, dis, com = tm.eager(split_body, n_sec, 4)
    # each operator alone, graph-replayed after a flush (the layout is complete)
    g_lay = tm.graph(lambda s: ep.moe_dispatch_layout(idx, w, E, R, L, s), n_sec)
    g_dis = tm.graph(lambda s: ep.moe_dispatch(x, L, fmt, recv, recv_s, s), n_sec)
    g_com = tm.graph(lambda s: ep.moe_combine(y, L, w, out, s), n_sec)
    # dispatch + combine as a pair (graph-replayed; the combine pays the
    # write-back of the dispatch's dirty receive rows)
    g_pair = tm.graph(lambda s: (ep.moe_dispatch(x, L, fmt, recv, recv_s, s), ep.moe_combine(y, L, w, out, s)), n_sec)
    # the same step through the three separate calls
    g_sep = tm.graph(step_ops_separate, n_sec)
    s_dis = stream_dispatch(fmt)
    s_com = tm.back_to_back(rotating(lambda s, o, i: ep.moe_combine(ys[i], L, w, o, s), outs), n_stream)
    check(L, "after the per-operator passes")

    legs = set(LEGS) if args.legs == "all" else set() if args.legs == "none" else set(args.legs.split(","))
    ops = {
        "note": ("us: graph-replayed (one CUDA graph per figure, events at its two ends, L2 flushed before "
                 "each replay, after warm-up replays); eager_us: eager launches with events between the "
                 "operators; stream_us: per launch in one graph of 8 back-to-back launches over 4 rotating "
                 "buffer sets (each launch's buffers untouched for the 3 launches before it, well over L2's "
                 "size; frac_stream from it); back_to_back_us (low-latency legs): per launch, 8 launches on the "
                 "same L2-resident buffers; frac: of the measured HBM copy rate, frac_spec: of the 8 TB/s "
                 "datasheet HBM3e bandwidth; the timed steps rotate over 4 independently allocated buffer sets "
                 "(step_us_by_placement: the mean of each)"),
        "step_us": pct(tot),
        "step_us_by_placement": [round(statistics.mean(tot[i::NPLACE]) * 1e3, 2)
                                 for i in range(min(NPLACE, len(tot)))],
        "layout": {"us": round(statistics.mean(g_lay) * 1e3, 2), "us_pct": pct(g_lay),
                   "eager_us": round(statistics.mean(lay) * 1e3, 2), "bytes": ab["layout"]},
        f"dispatch_{FORMAT_NAMES[fmt]}": hbm_op(ab[dkey], g_dis, dis, s_dis,
                                                tokens_per_s=round(T / (statistics.mean(g_dis) * 1e-3), 1)),
        "combine": hbm_op(ab["combine"], g_com, com, s_com, tokens_per_s=round(T / (statistics.mean(g_com) * 1e-3), 1),
                          eager_note="eager_us: after the dispatch, inside the step"),
        "dispatch_combine_pair": hbm_op(ab[dkey] + ab["combine"], g_pair),
        "step_separate_calls": hbm_op(step_bytes, g_sep, calls="moe_dispatch_layout + moe_dispatch + moe_combine",
                                      tokens_per_s=round(T / (statistics.mean(g_sep) * 1e-3), 1)),
    }

    # the step in the other receive format, graph-replayed like the timed steps
    # (bf16 step: layout -> FP8 dispatch -> combine; FP8 step: the bf16 one)
    if "formats" in legs:
        ofmt = ep.MOE_FORMAT_BF16 if fmt else ep.MOE_FORMAT_FP8
        oq, os_ = ep.alloc_recv(L, H, ofmt, device=dev)
        g_other = tm.graph(lambda s: step_ops(s, ofmt, oq, os_), n_sec)
        ob = ab["layout"] + ab[dispatch_key(ofmt)] + ab["combine"]
        ops[f"step_{FORMAT_NAMES[ofmt]}"] = hbm_op(ob, g_other, step=step_label(ofmt),
                                                   tokens_per_s=round(T / (statistics.mean(g_other) * 1e-3), 1))
        del oq, os_
        # each quantised format's dispatch alone on the same layout
        for f in (ep.MOE_FORMAT_FP8, ep.MOE_FORMAT_MXFP8):
            key = f"dispatch_{FORMAT_NAMES[f]}"
            if key in ops:
                continue
            rq, rs = ep.alloc_recv(L, H, f, device=dev)

            def body(mark, f=f, rq=rq, rs=rs):
                mark(0)
                ep.moe_dispatch(x, L, f, rq, rs, stream)
                mark(1)
            eg = tm.eager(body, n_sec, 2)[0]
            gr = tm.graph(lambda s, f=f, rq=rq, rs=rs: ep.moe_dispatch(x, L, f, rq, rs, s), n_sec)
            del rq, rs
            ops[key] = hbm_op(ab[dispatch_key(f)], gr, eg, stream_dispatch(f),
                              tokens_per_s=round(T / (statistics.mean(gr) * 1e-3), 1))
        check(L, "after the format legs")

    # backward pair: gradients of the receive rows and of the output
    if "backward" in legs:
        grad_recv = torch.empty(L.capacity, H, dtype=torch.bfloat16, device=dev).normal_()
        grad_out = torch.empty_like(out).normal_()
        grad_x = torch.empty_like(x)
        grad_y = torch.empty_like(y)
        grad_w = torch.empty_like(w)

        def body(mark):
            mark(0)
            ep.moe_dispatch_backward(grad_recv, L, grad_x, stream)
            mark(1)
            ep.moe_combine_backward(grad_out, y, L, w, grad_y, grad_w, stream)
            mark(2)
        dbwd, cbwd = tm.eager(body, n_sec, 3)
        gd = tm.graph(lambda s: ep.moe_dispatch_backward(grad_recv, L, grad_x, s), n_sec)
        gc = tm.graph(lambda s: ep.moe_combine_backward(grad_out, y, L, w, grad_y, grad_w, s), n_sec)
        ops["dispatch_backward"] = hbm_op(ab["dispatch_backward"], gd, dbwd)
        ops["combine_backward"] = hbm_op(ab["combine_backward"], gc, cbwd)
        del grad_recv, grad_out, grad_x, grad_y, grad_w
        check(L, "after the backward legs")

    # low-latency (decode) path: 128 tokens of the same shape, fixed capacity 128 per expert
    if "ll" in legs:
        T_ll = 128
        x_ll, idx_ll, w_ll = x[:T_ll].contiguous(), idx[:T_ll].contiguous(), w[:T_ll].contiguous()
        recv_ll = torch.empty(E * T_ll, H, dtype=torch.bfloat16, device=dev)
        tpe_ll = torch.empty(E, dtype=torch.int32, device=dev)
        slot_ll = torch.empty(T_ll, K, dtype=torch.int32, device=dev)
        st_ll = torch.zeros(1, dtype=torch.int32, device=dev)
        out_ll = torch.empty(T_ll, H, dtype=torch.bfloat16, device=dev)

        def body(mark):
            mark(0)
            ep.moe_ll_dispatch(x_ll, idx_ll, E, T_ll, recv_ll, tpe_ll, slot_ll, st_ll, stream)
            mark(1)
            ep.moe_ll_combine(recv_ll, slot_ll, w_ll, E, T_ll, out_ll, st_ll, stream)
            mark(2)
        lld, llc = tm.eager(body, n_sec, 3)
        ll_d = lambda s: ep.moe_ll_dispatch(x_ll, idx_ll, E, T_ll, recv_ll, tpe_ll, slot_ll, st_ll, s)
        ll_c = lambda s: ep.moe_ll_combine(recv_ll, slot_ll, w_ll, E, T_ll, out_ll, st_ll, s)
        gd, gc = tm.graph(ll_d, n_sec), tm.graph(ll_c, n_sec)
        # back to back on the same (L2-resident) buffers: the launch-to-launch time of a decode loop
        bd, bc = tm.back_to_back([ll_d] * 8, n_stream), tm.back_to_back([ll_c] * 8, n_stream)
        if int(st_ll.item()) != 0:
            raise RuntimeError("low-latency path reported a device error")
        ll_bytes = 2 * T_ll * H + 2 * H * T_ll * K + 4 * T_ll * K    # rows read, one row per entry written
        for key, g_, e_, b_ in (("ll_dispatch_T128", gd, lld, bd), ("ll_combine_T128", gc, llc, bc)):
            ops[key] = {"us": round(statistics.mean(g_) * 1e3, 2), "us_pct": pct(g_),
                        "eager_us": round(statistics.mean(e_) * 1e3, 2),
                        "back_to_back_us": round(statistics.mean(b_) * 1e3, 2), "bytes": ll_bytes,
                        "GB/s": round(gbps(ll_bytes, statistics.mean(g_)), 1), "bound": "latency"}
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

        def body(mark):
            mark(0)
            ep.moe_dispatch_layout(idx_ms, w_ms, E, R, L_ms, stream)
            mark(1)
            ep.moe_dispatch(x_ms, L_ms, False, recv_ms, None, stream)
            mark(2)
            ep.moe_combine(y_ms, L_ms, w_ms, out_ms, stream)
            mark(3)
        n_ms = max(10, n_sec // 4)
        msl, msd, msc = tm.eager(body, n_ms, 4)
        gl = tm.graph(lambda s: ep.moe_dispatch_layout(idx_ms, w_ms, E, R, L_ms, s), n_ms)
        gd = tm.graph(lambda s: ep.moe_dispatch(x_ms, L_ms, False, recv_ms, None, s), n_ms)
        gc = tm.graph(lambda s: ep.moe_combine(y_ms, L_ms, w_ms, out_ms, s), n_ms)
        check(L_ms, "in the multi-source leg")
        ab_ms = algorithmic_bytes(S_ms * T, H, E, R, K, int(L_ms.tokens_per_rank.sum().item()),
                                  int(L_ms.expert_offset[E].item()), L_ms.capacity)
        ops["multi_source_S8"] = {"note": f"8 sources x {T} tokens, one region of {8 * T} rows per destination rank",
                                  "layout": {"us": round(statistics.mean(gl) * 1e3, 2), "us_pct": pct(gl),
                                             "eager_us": round(statistics.mean(msl) * 1e3, 2)},
                                  "dispatch_bf16": hbm_op(ab_ms["dispatch"], gd, msd),
                                  "combine": hbm_op(ab_ms["combine"], gc, msc)}
        del x_ms, y_ms, recv_ms, out_ms, L_ms

    # the other routing shapes: Zipf-skewed Qwen3-235B-like routing (one rank
    # receives nearly every token) and DeepSeek-16B-like routing over 32 ranks
    # with a narrow hidden size; each a graph-replayed step of its own plus its
    # operators alone (bf16, FP8 and MXFP8 dispatch)
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

            def body(mark):
                mark(0)
                ep.moe_dispatch_layout(idx_o, w_o, Eo, Ro, L_o, stream)
                mark(1)
                ep.moe_dispatch(x_o, L_o, False, recv_o, None, stream)
                mark(2)
                ep.moe_combine(y_o, L_o, w_o, out_o, stream)
                mark(3)
            ol, od, oc = tm.eager(body, n_sec, 4)
            gs = tm.graph(lambda s: (ep.moe_dispatch_layout(idx_o, w_o, Eo, Ro, L_o, s),
                                     ep.moe_dispatch(x_o, L_o, False, recv_o, None, s),
                                     ep.moe_combine(y_o, L_o, w_o, out_o, s)), n_sec)
            gl = tm.graph(lambda s: ep.moe_dispatch_layout(idx_o, w_o, Eo, Ro, L_o, s), n_sec)
            gd = tm.graph(lambda s: ep.moe_dispatch(x_o, L_o, False, recv_o, None, s), n_sec)
            gc = tm.graph(lambda s: ep.moe_combine(y_o, L_o, w_o, out_o, s), n_sec)
            check(L_o, f"in the {name} leg")
            tpr = L_o.tokens_per_rank.cpu()
            ab_o = algorithmic_bytes(To, Ho, Eo, Ro, Ko, int(tpr.sum()), int(L_o.expert_offset[Eo].item()),
                                     L_o.capacity)
            tps = lambda g_: round(To / (statistics.mean(g_) * 1e-3), 1)
            del recv_o
            # back-to-back figures over rotating buffer sets, as for the step's shape
            xs_o = [x_o] + [x_o.clone() for _ in range(NB - 1)]

            def stream_o(f):
                sets = [ep.alloc_recv(L_o, Ho, f, device=dev) for _ in range(NB)]
                ms = tm.back_to_back(rotating(lambda s, b, i: ep.moe_dispatch(xs_o[i], L_o, f, b[0], b[1], s), sets),
                               n_stream)
                del sets
                return ms
            ys_o = [y_o] + [y_o.clone() for _ in range(NB - 1)]
            outs_o = [out_o] + [torch.empty_like(out_o) for _ in range(NB - 1)]
            sc = tm.back_to_back(rotating(lambda s, o, i: ep.moe_combine(ys_o[i], L_o, w_o, o, s), outs_o), n_stream)
            del ys_o, outs_o
            entry = {"shape": workload_label(wo), "n_pairs": int(tpr.sum()),
                     "rows_per_rank_min_max": [int(tpr.min()), int(tpr.max())],
                     "step": hbm_op(ab_o["layout"] + ab_o["dispatch"] + ab_o["combine"], gs, tokens_per_s=tps(gs),
                                    step=step_label(0)),
                     "layout": {"us": round(statistics.mean(gl) * 1e3, 2), "us_pct": pct(gl),
                                "eager_us": round(statistics.mean(ol) * 1e3, 2)},
                     "dispatch_bf16": hbm_op(ab_o["dispatch"], gd, od, stream_o(0), tokens_per_s=tps(gd)),
                     "combine": hbm_op(ab_o["combine"], gc, oc, sc, tokens_per_s=tps(gc),
                                       eager_note="eager_us: after the dispatch, inside the step")}
            for f in (ep.MOE_FORMAT_FP8, ep.MOE_FORMAT_MXFP8):
                rq, rs = ep.alloc_recv(L_o, Ho, f, device=dev)
                gf = tm.graph(lambda s, f=f, rq=rq, rs=rs: ep.moe_dispatch(x_o, L_o, f, rq, rs, s), n_sec)
                del rq, rs
                entry[f"dispatch_{FORMAT_NAMES[f]}"] = hbm_op(ab_o[dispatch_key(f)], gf, None, stream_o(f),
                                                              tokens_per_s=tps(gf))
            del xs_o
            check(L_o, f"in the {name} leg")
            wls[name] = entry
            del x_o, y_o, out_o, L_o
        ops["other_workloads"] = wls

    # how many CTAs ("channels") the HBM-bound operators need: the TMA-staged
    # bf16 dispatch (one warp per CTA), combine (256 threads per CTA, 16-byte
    # loads) and the TMA-staged combine (a producer warp stages the K rows,
    # four warps reduce), graph-replayed at fixed CTA counts
    if "channels" in legs:
        sweep = {"note": "GB/s at a fixed number of CTAs (graph-replayed, flushed); default = the operator's own grid",
                 "dispatch_bf16_tma": {}, "combine": {}, "combine_tma": {}}
        bq, _ = ep.alloc_recv(L, H, False, device=dev)
        for n_cta in SWEEP_CTAS + (0,):
            key = str(n_cta) if n_cta else "default"
            for name, fn, nb in (
                    ("dispatch_bf16_tma", lambda s, c=n_cta: ep.moe_dispatch(x, L, False, bq, None, s, num_channels=c,
                                                                         variant=1), ab["dispatch"]),
                    ("combine", lambda s, c=n_cta: ep.moe_combine(y, L, w, out, s, num_channels=c), ab["combine"]),
                    ("combine_tma", lambda s, c=n_cta: ep.moe_combine(y, L, w, out, s, num_channels=c, variant=1),
                     ab["combine"])):
                sweep[name][key] = round(gbps(nb, statistics.mean(tm.graph(fn, 10))), 1)
        ops["channel_sweep"] = sweep
        del bq

    e2e = run_e2e(args, inp, L, dev, fmt, step_bytes) if (rank == 0 and "e2e" in legs) else None

    # roofline of the dominant kernel (the combine), timed inside the step
    # (after the dispatch), plus the figures that bracket it
    com_ms = statistics.mean(com)
    achieved = gbps(ab["combine"], com_ms)
    traffic, traffic_src = (committed_traffic("combine_dsv3_ncu") if args.workload in ("dsv3", "dsv3_fp8")
                            else (None, "no committed capture of this shape"))
    pair_ms = statistics.mean(g_pair)
    roofline = {
        "bound": "hbm", "kernel": f"combine_kernel<{K if K in (1, 2, 4, 6, 8) else 0}>",
        "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
        "peak_source": (f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, torch copy)" if peak_kind == "measured"
                        else "fallback 6.8 TB/s"),
        "frac_spec": round(achieved / SPEC_HBM_GBS, 4), "peak_spec": SPEC_HBM_GBS,
        "traffic": traffic, "traffic_source": traffic_src,
        "timing": ("combine between events in the eager per-operator pass, after the dispatch: its window "
                   "includes the write-back of the dirty receive rows the dispatch leaves in L2 (up to ~100 MB); "
                   "combine_alone is the same kernel graph-replayed after an L2 flush, pair the dispatch and "
                   "the combine graph-replayed together, their bytes over their joint time"),
        "algorithmic_bytes": ab["combine"],
        "combine_alone": {"us": round(statistics.mean(g_com) * 1e3, 2),
                          "frac": round(gbps(ab["combine"], statistics.mean(g_com)) / peak, 4),
                          "frac_spec": round(gbps(ab["combine"], statistics.mean(g_com)) / SPEC_HBM_GBS, 4)},
        "pair": {"kernels": "dispatch_wide_kernel + combine_kernel",
                 "bytes": ab[dkey] + ab["combine"], "us": round(pair_ms * 1e3, 2),
                 "achieved": round(gbps(ab[dkey] + ab["combine"], pair_ms), 1),
                 "frac": round(gbps(ab[dkey] + ab["combine"], pair_ms) / peak, 4),
                 "frac_spec": round(gbps(ab[dkey] + ab["combine"], pair_ms) / SPEC_HBM_GBS, 4)},
    }

    value = aggregate_gbps(step_bytes, ms_step, world)
    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if fmt == 0 else "e4m3+bf16",
        "data": f"synthetic (seeded N(0,1) activations, softmax top-{K} routing of N(0,1) logits"
                + (f", Zipf s={wl.zipf_s} expert bias)" if wl.zipf_s else ")"),
        "config": step_config(wl, fmt, n_pairs, L.capacity, world),
        "launch": "timed steps replay one CUDA graph (layout -> dispatch -> combine), events at its two ends",
        "calls": STEP_CALLS,
        "frac": round(value / world / peak, 4),
        "frac_spec": round(value / world / SPEC_HBM_GBS, 4),
        "tokens_per_s": round(world * T / (ms_step * 1e-3), 1),
        "ops": ops,
        "roofline": roofline,
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(t_wall, 3),
    }
    if e2e is not None:
        result["e2e"] = e2e
    return result


def run_e2e(args, inp, L, dev, fmt, step_bytes):
    """Same step through the public API with host buffers: pinned host ->
    device copies of the inputs, the step's calls, device -> host copy of the
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
    recv, recv_s = ep.alloc_recv(L, wl.H, fmt, device=dev)
    comp = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    n = max(20, min(args.steps // 10, 50))

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
            ep.moe_dispatch_with_layout(b["idx"], b["w"], wl.E, wl.R, L, b["x"], fmt, recv, recv_s, comp)
            ep.moe_combine(b["y"], L, b["w"], out, comp)
            consumed[i % 2].record(comp)
            hout.copy_(out, non_blocking=True)
            hcnt.copy_(L.tokens_per_expert, non_blocking=True)

    run(max(3, args.warmup))
    torch.cuda.synchronize(dev)

    def link_gbs(dst, src):
        # one plain copy between the pinned host buffers and device memory,
        # the median of three (the host link's rate in this process)
        ts = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(comp)
            dst.copy_(src, non_blocking=True)
            b.record(comp)
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b))
        return round(src.numel() * src.element_size() / (statistics.median(ts) * 1e-3) / 1e9, 1)

    link = {"h2d_gbs": link_gbs(bufs[0]["y"], hy), "d2h_gbs": link_gbs(hout, out)}
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
            "overlap": "inputs of step i+1 copied while step i computes (two device buffer sets)",
            "link": link | {"note": "one plain copy of y host -> device and of out device -> host before the "
                                    "timed steps, this process"}}


# ------------------------------------------------------------ CPU baselines

def oracle_step_fn(wl, inp, T_s, fmt=0):
    """One oracle pass (layout, dispatch in the step's format, combine) over
    the first T_s tokens of the workload; returns (callable, algorithmic
    bytes, pairs, capacity)."""
    import oracle
    from combine_moe_dispatch_02_gb300.inputs import bf16_bits
    idx = inp.topk_idx[:T_s].numpy()
    w = inp.topk_w[:T_s].numpy()
    xb = bf16_bits(inp.x[:T_s])
    # y rows for these tokens: the first T_s * K expert-major rows stand in
    yb = bf16_bits(inp.y[: T_s * wl.K])
    Lo = oracle.layout(idx, w, wl.E, wl.R)
    ab = algorithmic_bytes(T_s, wl.H, wl.E, wl.R, wl.K, Lo.n_pairs, int(Lo.expert_offset[wl.E]), Lo.capacity)
    disp = oracle.dispatch_fp8 if fmt else oracle.dispatch_bf16

    def run():
        L = oracle.layout(idx, w, wl.E, wl.R)
        disp(xb, L)
        oracle.combine(yb, L.expert_slot, w)
    return run, ab["layout"] + ab[dispatch_key(fmt)] + ab["combine"], Lo.n_pairs, Lo.capacity


def cpu_baseline(wl, inp, budget_s=10.0):
    """The oracle as it stands, single-threaded, timed on this host over the
    full workload repeated until about `budget_s` seconds have passed."""
    fmt = 1 if wl.fp8 else 0
    run, nbytes, _, _ = oracle_step_fn(wl, inp, wl.T, fmt)
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
            "sample": f"full workload ({wl.T} tokens) x {n} passes of {step_label(fmt)}, {dt:.3f} s each, 1 thread",
            "host_cpu": cpu_model(), "host_cores": os.cpu_count()}


# Arm CPU part numbers (MIDR) of the cores these hosts carry, for hosts whose
# lscpu prints no model name
_ARM_PARTS = {"0xd4f": "Neoverse-V2 (NVIDIA Grace)", "0xd40": "Neoverse-V1", "0xd0c": "Neoverse-N1",
              "0xd49": "Neoverse-N2"}


def cpu_model():
    """The host's CPU model: lscpu's "Model name", else /proc/cpuinfo's."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name:"):
                name = line.split(":", 1)[1].strip()
                return _ARM_PARTS.get(name.lower(), name)
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        part = None
        for line in open("/proc/cpuinfo"):
            key = line.split(":", 1)[0].strip().lower()
            if key == "model name":
                return line.split(":", 1)[1].strip()
            if key == "cpu part" and part is None:
                part = line.split(":", 1)[1].strip().lower()
        if part:
            return _ARM_PARTS.get(part, f"Arm CPU part {part}")
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
    fmt = 1 if wl.fp8 else 0
    inp = make_inputs(wl, seed=0)
    probe, _, _, _ = oracle_step_fn(wl, inp, 128, fmt)
    t0 = time.perf_counter()
    probe()
    per_tok = (time.perf_counter() - t0) / 128
    target = 60.0 / max(args.steps + args.warmup, 1)         # about a minute in total
    T_s = int(max(32, min(wl.T, target / max(per_tok, 1e-9))))
    run, nbytes, n_pairs, capacity = oracle_step_fn(wl, inp, T_s, fmt)
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
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if fmt == 0 else "e4m3+bf16", "data": "synthetic",
            "config": step_config(wl, fmt, n_pairs, capacity, 1, T_sample=T_s),
            "cpu_baseline": {"value": v, "unit": "GB/s", "kind": "oracle", "cores": 1,
                             "sample": f"{T_s} of the workload's {wl.T} tokens per step, 1 thread",
                             "host_cpu": cpu_model(), "host_cores": os.cpu_count()},
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
