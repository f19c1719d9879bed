"""Benchmark of one MoE-layer forward (route -> dispatch -> grouped SwiGLU GEMM
-> combine) on GB300, printing one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config fine]
                    [--impl ours|reference] [--schedule interleaved|wave]

A step is one moe_layer_forward over one batch of T synthetic tokens with the
expert weights resident in HBM; L2 is flushed (a 256 MiB write) before every
timed step, outside the timed events. The default workload is the largest
single-GPU configuration, the fine-grained-expert layer (T=16384, d=4096,
E=256, top_k=8, ffn=2048: 6.6 TFLOP and 13 GB of weights per step). Under
torchrun each rank runs its own replica of the layer on its own tokens (weak
scaling, no collective on the data path); rank 0 prints the max-over-ranks
timing.

--impl reference times the fp64 CPU oracle on this machine's host cores on a
bounded sample of the same workload (there is no other implementation of this
path to run).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s and TFLOP/s on 1 GB300; fraction of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="fine", choices=sorted(synth.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--schedule", default="interleaved", choices=["interleaved", "wave"])
    ap.add_argument("--lead", type=int, default=0)
    ap.add_argument("--orientation", default="default", choices=["default", "tokens-m", "tokens-n"],
                    help="grouped GEMM operand orientation (which MMA operand holds the tokens)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the CUDA Graph replay of the layer (a secondary measurement)")
    ap.add_argument("--h-ring", type=int, default=0,
                    help="h as a ring of this many scheduler rows (0 = every row in place)")
    ap.add_argument("--l2-block-n", type=int, default=0, choices=[0, 64, 128, 192, 256],
                    help="Linear-2 tile width with tokens on the M side (0 = default)")
    ap.add_argument("--cta-group", type=int, default=0, choices=[0, 1, 2],
                    help="CTAs per grouped-GEMM tile (0 = default)")
    ap.add_argument("--row-order", default="default", choices=["default", "expert", "mixed"],
                    help="order of the grouped GEMM's scheduler rows")
    ap.add_argument("--router", default="default", choices=["default", "direct", "filter-verify"],
                    help="how the layer routes (the same bits either way)")
    ap.add_argument("--fused-combine", action="store_true",
                    help="combine inside the grouped GEMM (consumer warps) instead of a separate kernel")
    ap.add_argument("--timeline", action="store_true",
                    help="after the timed region, run one traced grouped GEMM and add its "
                         "per-tile timeline summary to the line")
    ap.add_argument("--stage", choices=["route", "dispatch", "combine"], default=None,
                    help="time one entry point alone (for profiling) instead of the layer")
    ap.add_argument("--experts", type=int, default=0,
                    help="profiling: the workload cut down to this many experts, with T scaled so the "
                         "tokens per expert (and d, ffn, top_k) stay the same")
    return ap.parse_args()


def scaled_config(cfg, experts):
    """The workload with fewer experts and proportionally fewer tokens: same d,
    ffn, top_k, routing skew and tokens per expert (T a multiple of the segments)."""
    if experts <= 0 or experts >= cfg.E:
        return cfg
    T = max(cfg.S, cfg.T * experts // cfg.E // cfg.S * cfg.S)
    return dataclasses.replace(cfg, name=f"{cfg.name}-{experts}e", T=T, E=experts)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_config(cfg):
    return {
        "workload": f"{cfg.name} MoE layer: T={cfg.T}, d={cfg.d}, E={cfg.E}, top_k={cfg.k}, "
                    f"SwiGLU ffn={cfg.F}, segments={cfg.S}, "
                    + (f"Zipf({cfg.zipf_s}) logit bias" if cfg.zipf_s else "balanced routing"),
        "T": cfg.T, "d": cfg.d, "E": cfg.E, "top_k": cfg.k, "ffn": cfg.F, "segments": cfg.S,
        "zipf_s": cfg.zipf_s, "seed": 0,
        "l2": "flushed before every timed step (256 MiB write, outside the timed events)",
    }


# ----------------------------------------------------------------- clocks
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        self.t0 = time.time()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        rows = []
        with open(self.f.name) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(parts[1]), max=float(parts[2]),
                                     power=float(parts[3]) if parts[3] not in ("", "[N/A]") else None,
                                     hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
                except ValueError:
                    continue
        os.unlink(self.f.name)
        if not rows:
            return None
        busy = [r for r in rows if r["power"] is None or r["power"] > 0] or rows
        top = max(r["sm"] for r in busy)
        load = [r for r in busy if r["sm"] >= 0.5 * top] or busy
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max((r["power"] or 0.0) for r in rows)}


# ----------------------------------------------------------------- oracle leg
def oracle_sample(cfg, inp_host, n_tokens, nthreads):
    """The fp64 oracle on the first n tokens of the workload: route, dispatch,
    expert FFN and combine. Returns elapsed seconds."""
    import oracle

    xb, wrb, bias, w1, w3, w2 = inp_host
    t0 = time.perf_counter()
    r = oracle.route(xb[:n_tokens], wrb, bias, cfg.k, nthreads=nthreads)
    oracle.dispatch(r.idx, cfg.E)
    oracle.layer_tokens(xb[:n_tokens], r.idx, r.gate, w1, w3, w2, np.arange(n_tokens, dtype=np.int32),
                        cfg.E, nthreads=nthreads)
    return time.perf_counter() - t0


def host_inputs(cfg, inp=None):
    if inp is None:
        inp = synth.make_inputs(cfg, seed=0, device="cuda" if torch.cuda.is_available() else "cpu")
    b = synth.bf16_bits
    bias = None if inp.bias is None else inp.bias.cpu().numpy()
    return b(inp.x), b(inp.wr), bias, b(inp.w1), b(inp.w3), b(inp.w2)


def pick_sample_tokens(cfg, inp_host, nthreads, budget_s):
    probe = min(cfg.T, max(2, nthreads))
    t = oracle_sample(cfg, inp_host, probe, nthreads)
    per_tok = t / probe
    return int(max(probe, min(cfg.T, budget_s / max(per_tok, 1e-9)))), per_tok


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, cfg):
    """--impl reference: the oracle, as it stands, timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    oracle.build()
    nth = cpu_threads()
    inp_host = host_inputs(cfg)
    total_steps = args.steps + args.warmup
    budget = min(8.0, 150.0 / max(total_steps, 1))  # the whole run stays within a few minutes
    n, _ = pick_sample_tokens(cfg, inp_host, nth, budget)
    for _ in range(args.warmup):
        oracle_sample(cfg, inp_host, n, nth)
    times = [oracle_sample(cfg, inp_host, n, nth) for _ in range(args.steps)]
    tsum = sum(times)
    value = n * args.steps / tsum
    sample = (f"first {n} of {cfg.T} tokens per step through route, dispatch, SwiGLU FFN and "
              f"combine (fp64 oracle)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        # measured: the mean wall time of one step as run (n tokens, not T)
        "ms_per_step": 1000.0 * tsum / args.steps,
        "tokens_per_step": n,
        # the same rate carried to a whole T-token step (not measured)
        "ms_per_full_step_extrapolated": 1000.0 * cfg.T / value,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nth, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- ranks
def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The largest of every rank's value (the job's time is its slowest rank)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, steps: int, world: int, slowest_ms: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (slowest_ms / 1000.0)


# ----------------------------------------------------------------- our leg
def traffic_record(cfg_name):
    """DRAM bytes per grouped-GEMM launch from the committed ncu summary, if its
    kernel source still matches."""
    p = os.path.join(ROOT, "profiles", f"grouped_gemm_{cfg_name}_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    src = os.path.join(ROOT, "grouped_gemm_softmax_gb300", "csrc", "grouped_gemm.cu")
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if rec.get("kernel_sha256") != h:
        return None
    return rec.get("dram_bytes_per_launch")


def timeline_summary(moe, cfg, shape, inp, ws, tuning, dev):
    """One extra layer call, outside the timed region, with the grouped GEMM's
    per-tile timeline switched on. Cycle counts are each SM's own clock64; only
    per-CTA differences are used. Summarises how much of each MMA issuer's
    span went to issuing tiles, the stage (operand) waits inside tiles, the
    gaps between consecutive tiles and the Linear-2 producers' waits for
    Linear-1 rows."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cap = moe.tile_trace_capacity(shape, sms)
    words = moe.TILE_TRACE_WORDS
    tt = torch.zeros(sms * cap * words, dtype=torch.int64, device=dev)
    tr = torch.zeros(sms * moe.TRACE_WORDS, dtype=torch.int64, device=dev)
    out = [torch.empty(cfg.T // cfg.S, cfg.d, dtype=torch.bfloat16, device=dev) for _ in range(cfg.S)]
    traced = dataclasses.replace(tuning, trace=tr, tile_trace=tt, tile_trace_cap=cap)
    moe.layer_forward(shape, inp.x, inp.wr, inp.bias, inp.w1, inp.w3, inp.w2, out, ws, tuning=traced)
    torch.cuda.synchronize(dev)
    st = moe.last_device_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status {st} {moe.last_device_detail()}")
    rec = tt.view(sms, cap, words).cpu().numpy().astype(np.int64)
    ctr = tr.view(sms, moe.TRACE_WORDS).cpu().numpy().astype(np.int64)
    kind = rec[:, :, 0] & 3
    issued = (rec[:, :, 3] > 0) & (rec[:, :, 4] > 0)
    busy = span = wait = 0
    gaps = []
    for c in range(sms):
        v = issued[c]
        if not v.any():
            continue
        st_, en = rec[c, v, 3], rec[c, v, 4]
        busy += int((en - st_).sum())
        span += int(en.max() - st_.min())
        wait += int(rec[c, v, 5].sum())
        if len(st_) > 1:
            gaps.append(st_[1:] - en[:-1])
    g = np.concatenate(gaps) if gaps else np.zeros(1, np.int64)
    produced = rec[:, :, 1] > 0
    l2 = produced & (kind == 1)
    t0 = ctr[:, 12][ctr[:, 12] > 0]
    t1 = ctr[:, 13][ctr[:, 13] > 0]
    return {
        "tiles_l1": int((issued & (kind == 0)).sum()), "tiles_l2": int((issued & (kind == 1)).sum()),
        "issuing_ctas": int(issued.any(1).sum()),
        "mma_issue_busy_frac": busy / max(span, 1),
        "stage_wait_frac_of_issue": wait / max(busy, 1),
        "gap_between_tiles_cycles_median": float(np.median(g)),
        "gap_between_tiles_cycles_p90": float(np.percentile(g, 90)),
        "l2_dependency_wait_cycles_mean": float(rec[:, :, 2][l2].mean()) if l2.any() else 0.0,
        "l2_tiles_that_waited_frac": float((rec[:, :, 2][l2] > 2000).mean()) if l2.any() else 0.0,
        "traced_kernel_us": float((t1.max() - t0.min()) / 1e3) if len(t0) and len(t1) else None,
        "truncated": bool((rec[:, -1, 1] > 0).any()),
    }


def run_ours(args, cfg):
    import grouped_gemm_softmax_gb300 as moe
    from grouped_gemm_softmax_gb300 import build as moe_build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if not moe_build.up_to_date():
        moe_build.build()
    moe.library()

    shape = moe.Shape(T=cfg.T, d=cfg.d, E=cfg.E, top_k=cfg.k, ffn=cfg.F, num_segments=cfg.S)
    inp = synth.make_inputs(cfg, seed=0, device=dev)
    if rank > 0:  # each replica routes its own tokens
        inp.x = synth.gaussian_bf16((cfg.T, cfg.d), 1.0, rank, synth.TID_X, dev)
    orient = {"default": moe.ORIENT_DEFAULT, "tokens-m": moe.ORIENT_TOKENS_M,
              "tokens-n": moe.ORIENT_TOKENS_N}[args.orientation]
    tuning = moe.Tuning(schedule=moe.SCHEDULE_EXPERT_WAVE if args.schedule == "wave"
                        else moe.SCHEDULE_INTERLEAVED, lead_rows=args.lead, orientation=orient,
                        h_ring_rows=args.h_ring, fused_combine=1 if args.fused_combine else 0,
                        row_order={"default": 0, "expert": 1, "mixed": 2}[args.row_order],
                        cta_group=args.cta_group, l2_block_n=args.l2_block_n,
                        router={"default": moe.ROUTER_DEFAULT, "direct": moe.ROUTER_DIRECT,
                                "filter-verify": moe.ROUTER_FILTER_VERIFY}[args.router])
    ws = moe.alloc_workspace(shape, dev, tuning if args.h_ring else None)
    rows = cfg.T // cfg.S
    out = [torch.empty(rows, cfg.d, dtype=torch.bfloat16, device=dev) for _ in range(cfg.S)]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        moe.layer_forward(shape, inp.x, inp.wr, inp.bias, inp.w1, inp.w3, inp.w2, out, ws,
                          tuning=tuning, stage_events=evs)

    sampler = ClockSampler(local) if rank == 0 else None
    for _ in range(args.warmup):
        flush.zero_()
        step()
    st = moe.last_device_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status {st} {moe.last_device_detail()}")

    # timed: one pair of events per step around the layer call, so the
    # layer's programmatic (overlapping) launches run as they do for a caller
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for evs in events:  # create the CUDA events
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    for k in range(args.steps):
        flush.zero_()
        events[k][0].record(stream)
        step()
        events[k][1].record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    st = moe.last_device_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status {st} {moe.last_device_detail()}")
    step_ms = np.array([a.elapsed_time(b) for a, b in events])
    total_ms = max_over_ranks(float(step_ms.sum()), dist, dev)

    # stage breakdown, outside the timed steps: events the library records
    # between its launches (they serialise the launches, so these stages sum
    # to a little more than the timed step)
    nstage = min(args.steps, 50)
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(nstage)]
    for evs in sev:
        for e in evs:
            e.record(stream)
    for k in range(nstage):
        flush.zero_()
        step(sev[k])
    torch.cuda.synchronize(dev)
    stage_ms = np.array([[evs[i].elapsed_time(evs[i + 1]) for i in range(4)] for evs in sev])
    value = job_throughput(cfg.T, args.steps, world, total_ms)
    ms_per_step = total_ms / args.steps
    ms_median = float(np.median(step_ms))

    # secondary: the same layer captured once in a CUDA Graph and replayed (the
    # library only enqueues stream work, so the whole layer is capturable); the
    # L2 flush stays outside the graph and outside the events, as above
    graph = None
    if not args.no_graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(max(args.warmup, 3)):
            flush.zero_()
            g.replay()
        gev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for k in range(args.steps):
            flush.zero_()
            gev[k][0].record(stream)
            g.replay()
            gev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        st = moe.last_device_status(ws)
        if st != moe.MOE_OK:
            raise RuntimeError(f"device status {st} {moe.last_device_detail()}")
        g_ms = np.array([a.elapsed_time(b) for a, b in gev])
        g_total = max_over_ranks(float(g_ms.sum()), dist, dev)
        graph = {"value": job_throughput(cfg.T, args.steps, world, g_total), "unit": "tokens/s",
                 "ms_per_step": g_total / args.steps, "ms_per_step_median": float(np.median(g_ms)),
                 "how": "one layer captured in a CUDA Graph, replayed once per step"}
        del g

    # secondary: the same layer calls back to back with no L2 flush between
    # them (what an inner loop over the same layer sees); the primary figure
    # above flushes L2 before every step
    bev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for evs in bev:
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize(dev)
    for k in range(args.steps):
        bev[k][0].record(stream)
        step()
        bev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    st = moe.last_device_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status {st} {moe.last_device_detail()}")
    b_ms = np.array([a.elapsed_time(b) for a, b in bev])
    b_total = max_over_ranks(float(b_ms.sum()), dist, dev)
    back_to_back = {"value": job_throughput(cfg.T, args.steps, world, b_total), "unit": "tokens/s",
                    "ms_per_step": b_total / args.steps, "ms_per_step_median": float(np.median(b_ms)),
                    "how": "the same layer calls back to back, no L2 flush between steps"}

    # e2e through the same C call with host buffers: every step copies its x
    # host->device (pinned) and its output device->host. Consecutive steps
    # overlap on three streams (H2D, layer, D2H: the two copy directions run on
    # their own copy engines), with two device buffers each for x and out;
    # the L2 flush stays in every step, on the layer's stream.
    e2e = None
    if not args.no_e2e:
        x_host = inp.x.cpu().pin_memory()
        out_host = [torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        x_dev = [torch.empty_like(inp.x) for _ in range(2)]
        out_dev = [[torch.empty(rows, cfg.d, dtype=torch.bfloat16, device=dev) for _ in range(cfg.S)]
                   for _ in range(2)]
        h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        h2d_done = [ev(), ev()]
        layer_done = [ev(), ev()]
        d2h_done = [ev(), ev()]

        def h2d(k):
            b = k % 2
            with torch.cuda.stream(h2d_s):
                if k >= 2:
                    h2d_s.wait_event(layer_done[b])  # step k-2 is done reading x_dev[b]
                x_dev[b].copy_(x_host, non_blocking=True)
                h2d_done[b].record(h2d_s)

        def pipeline(n):
            h2d(0)
            for k in range(n):
                b = k % 2
                if k + 1 < n:
                    h2d(k + 1)
                stream.wait_event(h2d_done[b])
                if k >= 2:
                    stream.wait_event(d2h_done[b])  # out_dev[b] copied out by step k-2
                flush.zero_()
                moe.layer_forward(shape, x_dev[b], inp.wr, inp.bias, inp.w1, inp.w3, inp.w2, out_dev[b], ws,
                                  tuning=tuning)
                layer_done[b].record(stream)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(layer_done[b])
                    for s_ in range(cfg.S):
                        out_host[b][s_ * rows:(s_ + 1) * rows].copy_(out_dev[b][s_], non_blocking=True)
                    d2h_done[b].record(d2h_s)
            for e_ in d2h_done:
                stream.wait_event(e_)

        pipeline(max(args.warmup, 2))
        torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h2d_s.wait_stream(stream)
        t0.record(h2d_s)
        stream.wait_event(t0)
        d2h_s.wait_event(t0)
        pipeline(args.steps)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_total = max_over_ranks(t0.elapsed_time(t1), dist, dev)
        st = moe.last_device_status(ws)
        if st != moe.MOE_OK:
            raise RuntimeError(f"device status {st} {moe.last_device_detail()}")
        e2e = {"value": job_throughput(cfg.T, args.steps, world, e2e_total), "unit": "tokens/s",
               "h2d_bytes_per_step": cfg.T * cfg.d * 2, "d2h_bytes_per_step": cfg.T * cfg.d * 2,
               "ms_per_step": e2e_total / args.steps,
               "overlap": "H2D, layer and D2H of consecutive steps on three streams"}

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    gemm_ms = float(stage_ms[:, 2].mean())
    gemm_flops = cfg.gemm_flops()
    achieved = gemm_flops / (gemm_ms / 1000.0) / 1e12
    burst = float(peaks["bf16_tflops"])
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    # a layer step lasts milliseconds, so the burst bf16 rate is the ceiling;
    # the power-capped sustained rate is reported beside it
    traffic = traffic_record(cfg.name)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": burst, "unit": "TFLOP/s",
                "frac": achieved / burst, "frac_of_sustained": achieved / sustained, "traffic": traffic,
                "kernel": "grouped_swiglu_gemm",
                "peak_source": ("measured bf16 dense burst (MEASURED_PEAKS.json)"
                                if peak_src == "measured" else "fallback bf16 burst")}
    hbm = float(peaks["hbm_gbs"])
    t_roof = max(cfg.flops() / (burst * 1e12), cfg.minimal_bytes() / (hbm * 1e9))
    t_roof_sus = max(cfg.flops() / (sustained * 1e12), cfg.minimal_bytes() / (hbm * 1e9))
    layer_frac = t_roof / (ms_per_step / 1000.0)
    layer_frac_sus = t_roof_sus / (ms_per_step / 1000.0)

    filtered = args.router == "filter-verify" or (args.router == "default" and cfg.E > 128)
    stage_roofline = stage_rooflines(cfg, stage_ms, hbm, float(peaks.get("sm_max_mhz", 2070.0)),
                                     torch.cuda.get_device_properties(dev).multi_processor_count, filtered)

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        nth = cpu_threads()
        inp_host = host_inputs(cfg, inp)
        n, _ = pick_sample_tokens(cfg, inp_host, nth, 10.0)
        el = oracle_sample(cfg, inp_host, n, nth)
        cpu = {"value": n / el, "unit": "tokens/s", "cores": nth, "kind": "oracle",
               "sample": f"first {n} of {cfg.T} tokens through route, dispatch, SwiGLU FFN and combine "
                         f"(fp64 oracle, {el:.1f} s)"}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "ms_per_step_median": ms_median,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(cfg), "gemm_schedule": args.schedule,
        "tflops": cfg.flops() / (ms_per_step / 1000.0) / 1e12 * world,
        "layer_roofline_frac": layer_frac, "layer_roofline_frac_of_sustained": layer_frac_sus,
        "stage_ms": {"route": float(stage_ms[:, 0].mean()), "dispatch": float(stage_ms[:, 1].mean()),
                     "grouped_gemm": gemm_ms, "combine": float(stage_ms[:, 3].mean())},
        "roofline": roofline, "stage_roofline": stage_roofline, "cpu_baseline": cpu, "e2e": e2e, "graph": graph,
        "back_to_back": back_to_back,
        "gpu_launches": moe.layer_kernel_launches(shape, tuning) * args.steps, "clocks": clocks,
        "wall_s_timed": t_wall,
    }
    if args.lead:
        line["config"]["lead_rows"] = args.lead
    if args.orientation != "default":
        line["config"]["orientation"] = args.orientation
    if args.cta_group:
        line["config"]["cta_group"] = args.cta_group
    if args.l2_block_n:
        line["config"]["l2_block_n"] = args.l2_block_n
    if args.row_order != "default":
        line["config"]["row_order"] = args.row_order
    if args.router != "default":
        line["config"]["router"] = args.router
    if args.fused_combine:
        line["config"]["fused_combine"] = True
    if args.h_ring:
        line["config"]["h_ring_rows"] = args.h_ring
        line["workspace_bytes"] = int(ws.numel())
    if args.timeline:
        line["timeline"] = timeline_summary(moe, cfg, shape, inp, ws, tuning, dev)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def stage_bytes(cfg, stage):
    """Algorithmic HBM bytes of one call of a memory-bound entry point: every
    input read once and every output written once (x read once by dispatch,
    although each token row is copied k times)."""
    T, d, E, k, R = cfg.T, cfg.d, cfg.E, cfg.k, cfg.R
    if stage == "route":
        return 2.0 * T * d + 2.0 * E * d + 4.0 * E + 8.0 * T * k
    if stage == "dispatch":
        return 4.0 * R + 2.0 * T * d + 2.0 * R * d + 8.0 * R + 8.0 * E
    return 2.0 * R * d + 8.0 * R + 2.0 * T * d  # combine


def stage_rooflines(cfg, stage_ms, hbm_gbs, sm_max_mhz, sms, filtered=False):
    """Each layer stage other than the GEMM against its own ceiling, from the
    stage events of the timed layer: achieved HBM bandwidth of its algorithmic
    bytes (stage_bytes) for route, dispatch and combine, and for route also
    the fp32 FMA rate (one logit is one thread's sequential sum on the CUDA
    cores) against the nominal 128 FMA/clk per SM at the maximum SM clock.
    A route that filters then verifies sums exactly only the candidate
    experts, so its dense FMA rate is an equivalent, not a fraction of a
    ceiling: it is reported as such, and the route's kernels are held to
    their own ceilings in the per-kernel profiles."""
    fp32_peak = sms * 128 * 2 * sm_max_mhz * 1e6 / 1e12
    out = {}
    for i, name in ((0, "route"), (1, "dispatch"), (3, "combine")):
        sec = float(stage_ms[:, i].mean()) / 1000.0
        gbs = stage_bytes(cfg, name) / sec / 1e9
        rec = {"ms": sec * 1000.0, "hbm_gbs": gbs, "hbm_frac": gbs / hbm_gbs}
        if name == "route" and filtered:
            rec.update({"router": "filter-verify",
                        "dense_equivalent_fp32_tflops": 2.0 * cfg.T * cfg.d * cfg.E / sec / 1e12,
                        "bound": "smem (exact candidate sums; see the route profile)"})
        elif name == "route":
            tf = 2.0 * cfg.T * cfg.d * cfg.E / sec / 1e12
            rec.update({"fp32_tflops": tf, "fp32_frac": tf / fp32_peak,
                        "fp32_peak": fp32_peak, "fp32_peak_source": "nominal: SMs x 128 FMA/clk x max SM clock"})
            rec["bound"] = "alu" if rec["fp32_frac"] > rec["hbm_frac"] else "hbm"
        else:
            rec["bound"] = "hbm"
        out[name] = rec
    return out


def run_stage(args, cfg):
    """Time one entry point alone on the config's inputs (no expert weights are
    generated): one JSON line with the stage's mean time. dispatch runs on the
    router's own indices; combine takes the dispatched token rows as its expert
    outputs (its work does not depend on their values), the router's gates and
    the dispatch's row map."""
    import grouped_gemm_softmax_gb300 as moe
    from grouped_gemm_softmax_gb300 import build as moe_build

    if not moe_build.up_to_date():
        moe_build.build()
    dev = torch.device("cuda", 0)
    shape = moe.Shape(T=cfg.T, d=cfg.d, E=cfg.E, top_k=cfg.k, ffn=cfg.F, num_segments=cfg.S)
    inp = synth.make_inputs(cfg, seed=0, device=dev, weights=False)
    i32 = dict(dtype=torch.int32, device=dev)
    idx = torch.empty(cfg.T, cfg.k, **i32)
    gate = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=dev)
    moe.route(shape, inp.x, inp.wr, inp.bias, idx, gate)
    if args.stage != "route":
        counts, offsets = torch.empty(cfg.E, **i32), torch.empty(cfg.E + 1, **i32)
        ros, sor = torch.empty(cfg.R, **i32), torch.empty(cfg.R, **i32)
        ws = moe.alloc_workspace(shape, dev)
        xp = moe.ws_view(ws, shape, moe.WS.X_PERM, torch.bfloat16, (cfg.R, cfg.d))
        moe.dispatch(shape, inp.x, idx, counts, offsets, ros, sor, xp, ws)
    if args.stage == "combine":
        y = xp  # the token rows stand in for the expert outputs
        segs = [torch.empty(cfg.T // cfg.S, cfg.d, dtype=torch.bfloat16, device=dev) for _ in range(cfg.S)]
    # the route stage as the layer runs it: filter then verify by default above
    # 128 experts (moe_route_filtered), else the direct kernels (moe_route)
    filtered = args.router == "filter-verify" or (args.router == "default" and cfg.E > 128)
    scratch = moe.alloc_route_scratch(shape, dev) if filtered else None

    def route_call():
        if filtered:
            moe.route_filtered(shape, inp.x, inp.wr, inp.bias, idx, gate, scratch)
        else:
            moe.route(shape, inp.x, inp.wr, inp.bias, idx, gate)

    calls = {
        "route": route_call,
        "dispatch": lambda: moe.dispatch(shape, inp.x, idx, counts, offsets, ros, sor, xp, ws),
        "combine": lambda: moe.combine(shape, y, gate, ros, segs),
    }
    call = calls[args.stage]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    # after the write that flushes L2, a read of another buffer larger than
    # L2 evicts the flush's dirty lines, so their write-back to HBM does not
    # land inside the timed call of a memory-bound kernel
    clean = torch.zeros(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
    ev = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        clean.sum()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        if i >= args.warmup:
            ev.append((a, b))
    torch.cuda.synchronize()
    if scratch is not None and moe.last_device_status(scratch) != moe.MOE_OK:
        raise RuntimeError(f"device status {moe.last_device_detail()}")
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    conf = workload_config(cfg)
    if args.stage == "route":
        conf["router"] = "filter-verify" if filtered else "direct"
    conf["l2"] = ("flushed before every timed call (256 MiB write, then a 256 MiB read of another "
                  "buffer so the flush's write-back lands before the timed events)")
    line = {"stage": args.stage, "config": conf, "ms": ms, "steps": args.steps,
            "hbm_gbs": stage_bytes(cfg, args.stage) / (ms / 1000.0) / 1e9,
            "algorithmic_bytes": stage_bytes(cfg, args.stage)}
    if args.stage == "route":
        line["fp32_tflops"] = 2.0 * cfg.T * cfg.d * cfg.E / (ms / 1000.0) / 1e12
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    cfg = scaled_config(synth.CONFIGS[args.config], args.experts)
    if args.stage:
        run_stage(args, cfg)
    elif args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
