"""Benchmark of the GB300 routed-expert MoE FFN layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode_bf16] [--tokens 64]

One step = one moe_ffn_forward over a batch of T tokens (router + top-8,
permutation, grouped gate/up with the clamped SwiGLU, grouped down with the
weighted scatter-add and the shared expert), weights resident in HBM.  Four
seeded x batches are cycled so the routed experts differ step to step, and
L2 is flushed (a 512 MB write) before every timed step; only the layer call
itself sits between the step's CUDA events.

Prints one JSON line (rank 0).  At N = 1 it also carries a per_config block:
every workload's configurations (decode bf16 / Int4 at 1, 8, 32 and 64
tokens, prefill bf16 at 4096, skewed Int4 prefill at 16384), each timed the
same way with its own clock record, roofline and oracle rate
(--no-per-config skips it).  --impl reference times the CPU oracle, the
plain implementation written from the method's description, on the host
cores, on a bounded sample of the same workload.

For N > 1 launch with torch.distributed.run: each rank runs its own replica
on its own GPU (the layer has no exchange step), "scaling": "weak".
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

METRIC = "MoE layer tokens/s"
L2_FLUSH_BYTES = 512 << 20
N_BATCHES = 4
THROTTLE_BITS = {
    0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
    0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
    0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
    0x100: "display_clock_setting"}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------ inputs

def host_layer(wl):
    """Seeded inputs on the host: x batches, router, expert stacks."""
    x_all = synthetic.gen_x(wl, T=wl.T * N_BATCHES)
    batches = [np.ascontiguousarray(x_all[i * wl.T:(i + 1) * wl.T]) for i in range(N_BATCHES)]
    w_router, b_router = synthetic.gen_router(wl)
    experts = synthetic.gen_experts(wl)
    shared = synthetic.gen_experts(wl, shared=True)
    return batches, w_router, b_router, experts, shared


def expert_bytes(wl):
    per = 3 * wl.H * wl.I
    if wl.fmt == "bf16":
        return per * 2
    return per // 2 + per // synthetic.INT4_GROUP * 2


def algorithmic_bytes(wl, distinct):
    """Weights of the distinct routed experts hit + the shared expert, router
    weight and bias, x in, fp32 out."""
    return ((distinct + 1) * expert_bytes(wl) + wl.E * wl.H * 2 + wl.E * 4
            + wl.T * wl.H * 2 + wl.T * wl.H * 4)


def gateup_bytes(wl, distinct):
    """Gate/up kernel: gate+up weights of distinct experts + shared, x_perm
    rows read, h written (two bf16 planes, or one fp16 plane)."""
    rows = (wl.top_k + 1) * wl.T
    w = (distinct + 1) * (2 * wl.I * wl.H) * (2 if wl.fmt == "bf16" else 0.5 + 2 / 32)
    h = rows * wl.I * (4 if wl.fmt == "bf16" else 2)
    return w + rows * wl.H * 2 + h


def down_bytes(wl, distinct):
    """Down projection: down weights of distinct experts + shared, h rows read
    (two bf16 planes, or one fp16 plane), out written once (fp32)."""
    rows = (wl.top_k + 1) * wl.T
    w = (distinct + 1) * (wl.I * wl.H) * (2 if wl.fmt == "bf16" else 0.5 + 2 / 32)
    return w + rows * wl.I * (4 if wl.fmt == "bf16" else 2) + wl.T * wl.H * 4


def traffic_per_launch(wl, units, record="gateup_traffic.json"):
    """DRAM bytes of one launch of the kernel a committed ncu capture covers
    (profiles/<record>: gateup_traffic.json for the gate/up kernel,
    decode_ffn_traffic.json for the one-launch decode FFN), scaled by the
    expert units processed; None when the record is absent, the kernel source
    changed since the capture, the workload shape differs, or the launch runs
    another kernel (above 64 tokens the token-major kernels serve)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", record)
    if (not os.path.exists(p) or wl.fmt != "bf16" or (wl.H, wl.I) != (4096, 1536)
            or wl.T > 64):
        return None
    with open(p) as f:
        rec = json.load(f)
    with open(os.path.join(ROOT, rec["source"]), "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    if not sha.startswith(rec["source_sha256_prefix"]):
        return None
    return rec["dram_bytes_per_unit"] * units


def flops_per_token(wl):
    return 2 * wl.E * wl.H + (wl.top_k + 1) * 2 * 3 * wl.H * wl.I


# ------------------------------------------------------------------ clocks

class ClockSampler:
    def __init__(self, gpu_index):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 5:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    mask = int(parts[4], 16)
                except ValueError:
                    continue
                for bit, name in THROTTLE_BITS.items():
                    if mask & bit and name != "gpu_idle":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle

def oracle_sample(wl, x, w_router, b_router, experts, shared, budget_s=12.0):
    """Times the oracle on successive token slices of x until budget_s.

    The oracle runs its tokens in parallel (one thread per token), so each
    slice holds as many tokens as it has threads (fewer if x is shorter).
    Returns (tokens done, seconds, threads used, tokens per slice)."""
    import oracle
    done, t0 = 0, time.perf_counter()
    chunk = max(1, min(x.shape[0], oracle.max_threads()))
    while True:
        start = (done // chunk * chunk) % x.shape[0]
        xs = np.ascontiguousarray(x[start:start + chunk])
        oracle.moe_forward(xs, w_router, b_router, experts, shared, wl.fmt)
        done += xs.shape[0]
        el = time.perf_counter() - t0
        if el >= budget_s:
            return done, el, min(chunk, oracle.max_threads()), chunk


# ------------------------------------------------------------------ main

def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="decode_bf16", choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--tokens", type=int, default=64)
    ap.add_argument("--experts", type=int, default=0,
                    help="override the routed expert count (small profiling cases only)")
    ap.add_argument("--deterministic", action="store_true",
                    help="fixed-order combination (bitwise reproducible output)")
    ap.add_argument("--accumulate", action="store_true",
                    help="out += layer(x) (residual add into the output)")
    ap.add_argument("--dense-ffn", type=int, default=0, metavar="I",
                    help="time the dense FFN (intermediate size I) instead of the MoE layer")
    ap.add_argument("--eager", action="store_true",
                    help="time eager layer calls instead of CUDA graph replays")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per_config block (every workload's configurations)")
    ap.add_argument("--per-config-cpu-s", type=float, default=1.5,
                    help="oracle seconds per per_config entry (0: no oracle timing)")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    args = ap.parse_args()
    # at least three untimed warm-up steps before any timed region; the JSON
    # line reports the number actually run
    args.warmup = max(args.warmup, 3)
    return args


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def config_of(wl, world, args=None, one_launch=False):
    modes = []
    if args is not None and args.deterministic:
        modes.append("deterministic combination")
    if args is not None and args.accumulate:
        modes.append("residual accumulate")
    return {"workload": f"{wl.name} T={wl.T} H={wl.H} E={wl.E} top_k={wl.top_k} I={wl.I} "
                        f"shared I={wl.I_shared} {wl.fmt} weights",
            "modes": modes or ["default (atomic fp32 scatter-add)"],
            "tokens_per_step": wl.T, "weights": wl.fmt,
            "expert_weight_bytes": wl.E * expert_bytes(wl),
            "x_batches_cycled": N_BATCHES,
            "l2": "flushed before every step (512 MB write); weights read per step exceed L2",
            "launch": ("eager layer calls" if args is not None and args.eager else
                       "CUDA graph replay, one captured layer call per x batch, timed by "
                       "events around each replay"),
            "stage_split": ("events between the stages of each call" if args is not None
                            and args.eager else
                            "second pass of K replays of graphs with event nodes between the "
                            "stages (gate/up duration for the roofline)")
                           + ("; gate/up and down are one launch (the gate/up stage holds both)"
                              if one_launch else ""),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference(args, wl, rank, world):
    if rank != 0:
        return
    batches, w_router, b_router, experts, shared = host_layer(wl)
    per_step = []
    tokens = 0
    for _ in range(args.warmup):
        pass  # the oracle has no warm state; warm-up steps are not timed
    t_all = 0.0
    import oracle
    # the oracle runs one thread per token: each step takes as many of the
    # step's tokens as it has threads
    n_per_step = min(wl.T, oracle.max_threads())
    cores = n_per_step
    for s in range(args.steps):
        x = batches[s % N_BATCHES]
        n = n_per_step
        t0 = time.perf_counter()
        oracle.moe_forward(np.ascontiguousarray(x[:n]), w_router, b_router, experts, shared,
                           wl.fmt)
        dt = time.perf_counter() - t0
        per_step.append(dt)
        tokens += n
        t_all += dt
    value = tokens / t_all
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t_all / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(wl, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"first {n_per_step} tokens of each step's batch "
                                       f"(one oracle thread per token)"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, wl, rank, world, local):
    import torch
    import routed_expert_ffn_sigmoid_gb300 as moe
    from routed_expert_ffn_sigmoid_gb300 import replicas

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    batches, w_router, b_router, experts, shared = host_layer(wl)

    def up16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev) if a.dtype == np.uint8 else up16(a)

    xs = [up16(b) for b in batches]
    wr, b = up16(w_router), torch.from_numpy(b_router).to(dev)
    ex = {k: up(v) for k, v in experts.items()}
    sh = {k: up(v) for k, v in shared.items()}
    exw = moe.make_weights(ex["gate"], ex["up"], ex["down"], ex.get("gate_scale"),
                           ex.get("up_scale"), ex.get("down_scale"))
    shw = moe.make_weights(sh["gate"], sh["up"], sh["down"], sh.get("gate_scale"),
                           sh.get("up_scale"), sh.get("down_scale"))
    flags = ((moe.MOE_FLAG_DETERMINISTIC if args.deterministic else 0)
             | (moe.MOE_FLAG_ACCUMULATE if args.accumulate else 0))
    dims = moe.make_dims(wl.T, wl.H, wl.E, wl.I, wl.I_shared, wl.top_k, wl.fmt, flags)
    ws = torch.zeros(moe.moe_workspace_size(dims), dtype=torch.uint8, device=dev)
    out = torch.zeros((wl.T, wl.H), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # distinct routed experts per batch (from the library's own routing, untimed)
    distinct = []
    idx = torch.empty((wl.T, wl.top_k), dtype=torch.int32, device=dev)
    wts = torch.empty((wl.T, wl.top_k), dtype=torch.float32, device=dev)
    for x in xs:
        moe.moe_router_topk(dims, x, wr, b, idx, wts, ws)
        distinct.append(int(torch.unique(idx).numel()))

    nst = moe.MOE_STAGE_COUNT
    def new_events():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)]
        for e in evs:
            e.record(stream)  # materialise the handle
        se = moe.MoeStageEvents()
        for i, e in enumerate(evs):
            se.ev[i] = e.cuda_event
        return evs, se

    for s in range(args.warmup):
        moe.moe_ffn_forward(dims, xs[s % N_BATCHES], wr, b, exw, shw, out, ws)
    torch.cuda.synchronize(dev)
    st = moe.moe_workspace_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(moe.moe_status_string(st))

    step_events = [new_events() for _ in range(args.steps)] if args.eager else []
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    if args.eager:
        with ClockSampler(local) as clk:
            time.sleep(0.3)  # let the sampler start before the timed steps
            for s in range(args.steps):
                flush.zero_()
                moe.moe_ffn_forward_timed(dims, xs[s % N_BATCHES], wr, b, exw, shw, out, ws,
                                          step_events[s][1])
            torch.cuda.synchronize(dev)
        step_ms = [evs[0].elapsed_time(evs[nst]) for evs, _ in step_events]
        stage_ms = [[evs[i].elapsed_time(evs[i + 1]) for evs, _ in step_events]
                    for i in range(nst)]
    else:
        # One graph per x batch: the layer call (all its kernels) captured
        # once, replayed every step, timed by events recorded on the stream
        # around the replay; the L2 flush runs between replays, outside the
        # graphs.  A second pass of K replays times the stages with graphs
        # of moe_ffn_forward_timed: their event nodes between the kernels
        # keep each kernel from starting early (programmatic dependent
        # launch), which costs ~13 us per step at 1-8 tokens, so that pass
        # gives the stage split and the kernel durations, not the step time.
        graphs, staged = [], []
        cap = torch.cuda.Stream(dev)
        for bi in range(N_BATCHES):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap, capture_error_mode="relaxed"):
                moe.moe_ffn_forward(dims, xs[bi], wr, b, exw, shw, out, ws)
            graphs.append(g)
            evs, se = new_events()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap, capture_error_mode="relaxed"):
                moe.moe_ffn_forward_timed(dims, xs[bi], wr, b, exw, shw, out, ws, se)
            staged.append((g, evs))
        for s in range(args.warmup):
            graphs[s % N_BATCHES].replay()
            staged[s % N_BATCHES][0].replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        step_ms, stage_ms = [], [[] for _ in range(nst)]
        with ClockSampler(local) as clk:
            time.sleep(0.3)
            for s in range(args.steps):
                flush.zero_()
                e0.record(stream)
                graphs[s % N_BATCHES].replay()
                e1.record(stream)
                e1.synchronize()
                step_ms.append(e0.elapsed_time(e1))
            for s in range(args.steps):
                flush.zero_()
                g, evs = staged[s % N_BATCHES]
                g.replay()
                # the graph's events are read before the graph runs again
                torch.cuda.synchronize(dev)
                for i in range(nst):
                    stage_ms[i].append(evs[i].elapsed_time(evs[i + 1]))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    st = moe.moe_workspace_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(moe.moe_status_string(st))
    value, ms_per_step = replicas.job_throughput(sum(step_ms), wl.T, args.steps, world, dev)

    # end to end through the C ABI with host buffers: H2D x, layer, D2H out
    host_x = [torch.from_numpy(bt.view(np.int16)).pin_memory() for bt in batches]
    host_out = torch.empty((wl.T, wl.H), dtype=torch.float32).pin_memory()
    xdev = torch.empty_like(xs[0])
    for s in range(args.warmup):
        xdev.copy_(host_x[s % N_BATCHES], non_blocking=True)
        moe.moe_ffn_forward(dims, xdev, wr, b, exw, shw, out, ws)
        host_out.copy_(out, non_blocking=True)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = 0.0
    for s in range(args.steps):
        flush.zero_()
        e0.record(stream)
        xdev.copy_(host_x[s % N_BATCHES], non_blocking=True)
        moe.moe_ffn_forward(dims, xdev, wr, b, exw, shw, out, ws)
        host_out.copy_(out, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    e2e_value, _ = replicas.job_throughput(e2e_ms, wl.T, args.steps, world, dev)

    hbm_peak, tc_peak, tc_sust, peak_src = peaks()
    mean_distinct = sum(distinct[s % N_BATCHES] for s in range(args.steps)) / args.steps
    # the dominant kernel: gate/up, or with one launch gate/up + down together
    # (the timed call's gate/up stage then brackets both projections)
    one_launch = moe.moe_ffn_one_launch(dims) == 1
    int4_gemv = moe.moe_ffn_int4_gemv(dims) == 1
    gu_ms = statistics.mean(stage_ms[2])
    gu_bytes = statistics.mean(
        gateup_bytes(wl, distinct[s % N_BATCHES])
        + (down_bytes(wl, distinct[s % N_BATCHES]) if one_launch else 0)
        for s in range(args.steps))
    achieved = gu_bytes / (gu_ms / 1e3) / 1e9
    layer_bytes = statistics.mean(algorithmic_bytes(wl, distinct[s % N_BATCHES])
                                  for s in range(args.steps))
    layer_gbs = layer_bytes / (ms_per_step / 1e3) / 1e9
    tflops = flops_per_token(wl) * wl.T / (ms_per_step / 1e3) / 1e12

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        n, el, cores, chunk = oracle_sample(wl, np.concatenate(batches), w_router, b_router,
                                            experts, shared, args.cpu_budget_s)
        cpu = {"value": n / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} tokens of the same workload's x batches, in slices of {chunk} "
                         f"tokens (one oracle thread per token), {el:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("bf16 operands, fp32 accumulate" if wl.fmt == "bf16" else
                      "int4 codes x 16-bit activations (two byte planes) in int8 dot products, "
                      "exact int32 group sums, scale per group in fp32" if int4_gemv else
                      "int4 weights as e5m2 (n - 8) x e4m3 activation planes, scale per group "
                      "after the MMA, fp32 accumulate" if wl.T <= 64 else
                      "int4 weights dequantised to fp16, fp32 accumulate"),
            "data": "synthetic (seeded generator; random-init weights)",
            "config": config_of(wl, world, args, one_launch),
            "roofline": {"bound": "hbm",
                         "kernel": ("decode_ffn (tcgen05 gate/up + down, one launch)" if one_launch
                                    else "int4_gemv_gateup (CUDA-core dp4a gate/up)" if int4_gemv
                                    else "gateup_swiglu (tcgen05 grouped gate/up)"),
                         "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak,
                         "traffic": (traffic_per_launch(wl, mean_distinct + 1,
                                                        "decode_ffn_traffic.json") if one_launch
                                     else traffic_per_launch(wl, mean_distinct + 1)),
                         "peak_source": f"{peak_src} hbm_gbs",
                         "algorithmic_bytes_per_launch": gu_bytes, "mean_launch_ms": gu_ms},
            "layer": {"algorithmic_GBps": layer_gbs, "hbm_frac": layer_gbs / hbm_peak,
                      "tflops": tflops, "tc_frac_sustained": tflops / (tc_sust or tc_peak),
                      "distinct_experts_mean": mean_distinct,
                      "stage_ms_mean": {n: statistics.mean(v) for n, v in
                                        zip(moe.STAGE_NAMES, stage_ms)}},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "tokens/s",
                    "h2d_bytes_per_step": wl.T * wl.H * 2, "d2h_bytes_per_step": wl.T * wl.H * 4},
            # T <= 128: logits, one-CTA routing, gather, gate/up, down; larger T:
            "gpu_launches": (layer_launches(wl.T, args.deterministic, wl.fmt, int4_gemv)
                             - (1 if one_launch else 0)) * args.steps,
            "clocks": clk.summary(),
        }
        if (world == 1 and not args.no_per_config and not args.deterministic
                and not args.accumulate and not args.experts):
            # every workload's configurations, each timed the same way (graph
            # replays, L2 flushed outside the events, its own clock record)
            line["per_config"] = per_config_block(
                args, dev, (wl.name, (wr, b, exw, shw), w_router, b_router, experts, shared))
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------------ every workload

# (workload, token counts) of the per-config block, in the order they run
PER_CONFIG = (("decode_bf16", (1, 8, 32, 64)), ("decode_int4", (1, 8, 32, 64)),
              ("prefill_bf16", (4096,)), ("skewed_prefill_int4", (16384,)))
PER_CONFIG_REGION_MS = 300.0  # timed region per entry (long enough for clock samples)


def upload_layer(moe, dev, w_router, b_router, experts, shared):
    import torch

    def up(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t if a.dtype == np.uint8 else t.view(torch.int16)).to(dev)

    ex = {k: up(v) for k, v in experts.items()}
    sh = {k: up(v) for k, v in shared.items()}
    exw = moe.make_weights(ex["gate"], ex["up"], ex["down"], ex.get("gate_scale"),
                           ex.get("up_scale"), ex.get("down_scale"))
    shw = moe.make_weights(sh["gate"], sh["up"], sh["down"], sh.get("gate_scale"),
                           sh.get("up_scale"), sh.get("down_scale"))
    return up(w_router), torch.from_numpy(b_router).to(dev), exw, shw


def time_config(moe, dev, wl, layer, host_x, w_router_np, b_router_np, experts_np, shared_np,
                warmup, cpu_budget_s, hbm_peak, tc_peak, tc_sust):
    """One per-config entry: CUDA-graph replays of moe_ffn_forward over the
    workload's seeded x batches, L2 flushed before each replay outside the
    events, clocks sampled during the timed region; roofline on the layer's
    algorithmic bytes or flops; the oracle timed on the same workload."""
    import torch

    wr, b, exw, shw = layer
    xs = [torch.from_numpy(bt.view(np.int16)).to(dev) for bt in host_x]
    dims = moe.make_dims(wl.T, wl.H, wl.E, wl.I, wl.I_shared, wl.top_k, wl.fmt, 0)
    ws = torch.zeros(moe.moe_workspace_size(dims), dtype=torch.uint8, device=dev)
    out = torch.zeros((wl.T, wl.H), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    distinct = []
    idx = torch.empty((wl.T, wl.top_k), dtype=torch.int32, device=dev)
    wts = torch.empty((wl.T, wl.top_k), dtype=torch.float32, device=dev)
    for x in xs:
        moe.moe_router_topk(dims, x, wr, b, idx, wts, ws)
        distinct.append(int(torch.unique(idx).numel()))
    graphs = []
    cap = torch.cuda.Stream(dev)
    for bi in range(N_BATCHES):
        moe.moe_ffn_forward(dims, xs[bi], wr, b, exw, shw, out, ws)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap, capture_error_mode="relaxed"):
            moe.moe_ffn_forward(dims, xs[bi], wr, b, exw, shw, out, ws)
        graphs.append(g)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_warm = []
    for s_ in range(max(warmup, 3)):
        flush.zero_()
        e0.record(stream)
        graphs[s_ % N_BATCHES].replay()
        e1.record(stream)
        e1.synchronize()
        t_warm.append(e0.elapsed_time(e1))
    est = min(t_warm)
    steps = int(min(3000, max(10, PER_CONFIG_REGION_MS / (est + 0.15))))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index or 0) as clk:
        time.sleep(0.3)
        for s_ in range(steps):
            flush.zero_()
            evs[s_][0].record(stream)
            graphs[s_ % N_BATCHES].replay()
            evs[s_][1].record(stream)
        torch.cuda.synchronize(dev)
    st = moe.moe_workspace_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(moe.moe_status_string(st))
    step_ms = [a.elapsed_time(c) for a, c in evs]
    ms = statistics.mean(step_ms)
    mean_distinct = sum(distinct[s_ % N_BATCHES] for s_ in range(steps)) / steps
    nbytes = statistics.mean(algorithmic_bytes(wl, distinct[s_ % N_BATCHES])
                             for s_ in range(steps))
    flops = flops_per_token(wl) * wl.T
    gbs = nbytes / (ms / 1e3) / 1e9
    tflops = flops / (ms / 1e3) / 1e12
    bound = "hbm" if flops / nbytes < tc_peak * 1e12 / (hbm_peak * 1e9) else "tensor"
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": gbs / hbm_peak, "peak_source": "measured hbm_gbs (copy)"}
    else:
        roof = {"bound": "tensor", "achieved": tflops, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": tflops / tc_peak, "peak_source": "measured bf16_tflops (burst)",
                "frac_of_sustained": tflops / tc_sust if tc_sust else None}
    roof.update({"algorithmic_bytes_per_step": nbytes, "flops_per_step": flops,
                 "hbm_frac": gbs / hbm_peak, "tc_frac_burst": tflops / tc_peak})
    cpu = None
    if cpu_budget_s > 0:
        n, el, cores, chunk = oracle_sample(wl, np.concatenate(host_x), w_router_np, b_router_np,
                                            experts_np, shared_np, cpu_budget_s)
        cpu = {"value": n / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} tokens of this workload's x batches in slices of {chunk}, "
                         f"{el:.1f} s"}
    del graphs, ws, out, flush, xs
    return {"workload": wl.name, "T": wl.T, "weights": wl.fmt,
            "config": config_of(wl, 1)["workload"],
            "steps": steps, "warmup": max(warmup, 3), "ms_per_step": ms,
            "ms_p10": float(np.percentile(step_ms, 10)), "ms_p90": float(np.percentile(step_ms, 90)),
            "value": wl.T / (ms / 1e3), "unit": "tokens/s", "GBps": gbs, "TFLOPps": tflops,
            "distinct_experts_mean": mean_distinct, "roofline": roof,
            "gpu_launches": (layer_launches(wl.T, False, wl.fmt,
                                            moe.moe_ffn_int4_gemv(dims) == 1)
                             - (1 if moe.moe_ffn_one_launch(dims) == 1 else 0)) * steps,
            "clocks": clk.summary(), "cpu_baseline": cpu}


def per_config_block(args, dev, resident=None):
    """Every workload's configurations timed the same way, one after another.

    resident: (workload name, uploaded layer, host router w, host bias,
    host experts, host shared) of a stack already on the device, reused for
    that workload."""
    import gc

    import torch
    import routed_expert_ffn_sigmoid_gb300 as moe

    hbm_peak, tc_peak, tc_sust, _ = peaks()
    entries = []
    for name, tokens in PER_CONFIG:
        base = synthetic.WORKLOADS[name]
        if resident is not None and resident[0] == name:
            _, layer, w_router, b_router, experts, shared = resident
        else:
            resident = None
            gc.collect()
            torch.cuda.empty_cache()
            w_router, b_router = synthetic.gen_router(base)
            experts = synthetic.gen_experts(base)
            shared = synthetic.gen_experts(base, shared=True)
            layer = upload_layer(moe, dev, w_router, b_router, experts, shared)
        for T in tokens:
            wl = base.with_tokens(T)
            x_all = synthetic.gen_x(wl, T=T * N_BATCHES)
            host_x = [np.ascontiguousarray(x_all[i * T:(i + 1) * T]) for i in range(N_BATCHES)]
            entries.append(time_config(moe, dev, wl, layer, host_x, w_router, b_router,
                                       experts, shared, args.warmup, args.per_config_cpu_s,
                                       hbm_peak, tc_peak, tc_sust))
        del layer, experts, shared
        resident = None
    gc.collect()
    torch.cuda.empty_cache()
    return entries


def layer_launches(T, deterministic, fmt="bf16", int4_gemv=False):
    """Kernels one moe_ffn_forward launches.  T <= 128: router partial logits,
    slice sum + top-k, the one-CTA permutation (for T <= 16 run by the top-k
    kernel's last CTA instead), gate/up, down.
    Larger T: logits (partial sums below 256 tokens, tensor cores from 256),
    top-k, count, scan, scatter, gate/up, down.  The bf16 gate/up GEMM gathers
    the token rows from x itself up to 8 tokens and from 512 tokens (its
    token-major form), and so does the CUDA-core Int4 gate/up (int4_gemv); in
    between, and otherwise for Int4, one more kernel writes x_perm.
    Deterministic mode adds the fixed-order combination."""
    gathers_itself = int4_gemv or (fmt == "bf16" and (T <= 8 or T >= 512))
    base = 4 if T <= 16 else (5 if T <= 128 else 7)
    return base + (0 if gathers_itself else 1) + (1 if deterministic else 0)


def run_dense(args, rank, world, local):
    """Times moe_dense_ffn: the dense FFN of the first layers (H = 4096,
    intermediate size --dense-ffn) over T tokens, weights resident."""
    import torch
    import routed_expert_ffn_sigmoid_gb300 as moe
    from routed_expert_ffn_sigmoid_gb300 import replicas

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    base = synthetic.WORKLOADS[args.workload]
    I = args.dense_ffn
    wl = synthetic.Workload("dense_ffn", args.tokens, base.H, 1, I, I, base.top_k, base.fmt, 60,
                            tokens=(args.tokens,))
    w = synthetic.gen_experts(wl, shared=True)
    x_all = synthetic.gen_x(wl, T=wl.T * N_BATCHES)

    def up(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t if a.dtype == np.uint8 else t.view(torch.int16)).to(dev)

    dw = {k: up(v) for k, v in w.items()}
    weights = moe.make_weights(dw["gate"], dw["up"], dw["down"], dw.get("gate_scale"),
                               dw.get("up_scale"), dw.get("down_scale"))
    xs = [up(x_all[i * wl.T:(i + 1) * wl.T]) for i in range(N_BATCHES)]
    flags = moe.MOE_FLAG_ACCUMULATE if args.accumulate else 0
    dims = moe.make_dims(wl.T, wl.H, 0, I, I, wl.top_k, wl.fmt, flags)
    ws = torch.zeros(moe.moe_dense_workspace_size(dims), dtype=torch.uint8, device=dev)
    out = torch.zeros((wl.T, wl.H), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for s_ in range(args.warmup):
        moe.moe_dense_ffn(dims, xs[s_ % N_BATCHES], weights, out, ws)
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    if not args.eager:  # one captured call per x batch, replayed
        graphs = []
        cap = torch.cuda.Stream(dev)
        for bi in range(N_BATCHES):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap, capture_error_mode="relaxed"):
                moe.moe_dense_ffn(dims, xs[bi], weights, out, ws)
            graphs.append(g)
        for s_ in range(args.warmup):
            graphs[s_ % N_BATCHES].replay()
        torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        for s_ in range(args.steps):
            flush.zero_()
            evs[s_][0].record(stream)
            if args.eager:
                moe.moe_dense_ffn(dims, xs[s_ % N_BATCHES], weights, out, ws)
            else:
                graphs[s_ % N_BATCHES].replay()
            evs[s_][1].record(stream)
        torch.cuda.synchronize(dev)
    st = moe.moe_workspace_status(ws)
    if st != moe.MOE_OK:
        raise RuntimeError(moe.moe_status_string(st))
    total = sum(a.elapsed_time(b) for a, b in evs)
    value, ms_per_step = replicas.job_throughput(total, wl.T, args.steps, world, dev)
    hbm_peak, tc_peak, tc_sust, peak_src = peaks()
    wbytes = 3 * wl.H * I * (2 if wl.fmt == "bf16" else 0.5 + 2 / 32)
    nbytes = wbytes + wl.T * wl.H * (2 + 4)
    flops = 2 * 3 * wl.H * I * wl.T
    gbs = nbytes / (ms_per_step / 1e3) / 1e9
    tflops = flops / (ms_per_step / 1e3) / 1e12
    ridge = tc_sust * 1e12 / (hbm_peak * 1e9)
    bound = "hbm" if flops / nbytes < ridge else "tensor"
    if rank == 0:
        roof = ({"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                 "frac": gbs / hbm_peak} if bound == "hbm" else
                {"bound": "tensor", "achieved": tflops, "peak": tc_sust, "unit": "TFLOP/s",
                 "frac": tflops / tc_sust})
        roof.update({"kernel": "moe_dense_ffn (grouped gate/up + down, one group)",
                     "traffic": None, "peak_source": f"{peak_src} peaks",
                     "algorithmic_bytes_per_call": nbytes, "flops_per_call": flops})
        print(json.dumps({
            "metric": "dense FFN tokens/s", "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 operands, fp32 accumulate" if wl.fmt == "bf16" else
                     "int4 weights dequantised to fp16, fp32 accumulate",
            "data": "synthetic (seeded generator; random-init weights)",
            "config": {"workload": f"dense FFN T={wl.T} H={wl.H} I={I} {wl.fmt} weights",
                       "l2": "flushed before every step (512 MB write)",
                       "launch": "eager layer calls" if args.eager else
                                 "CUDA graph replay, one captured call per x batch"},
            "roofline": roof, "gbs": gbs, "tflops": tflops,
            # dense-rows table, gate/up, down (+ the fp16 conversion of x for Int4)
            "gpu_launches": (3 + (1 if wl.fmt != "bf16" else 0)) * args.steps,
            "clocks": clk.summary()}), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    wl = synthetic.WORKLOADS[args.workload].with_tokens(args.tokens)
    if args.experts:
        from dataclasses import replace
        wl = replace(wl, E=args.experts)
    if args.impl == "reference":
        run_reference(args, wl, rank, world)
    elif args.dense_ffn:
        run_dense(args, rank, world, local)
    else:
        run_ours(args, wl, rank, world, local)


if __name__ == "__main__":
    main()
