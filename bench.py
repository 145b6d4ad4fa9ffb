#!/usr/bin/env python
"""Benchmark of one packed speculative-verification step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the hot path over one batch of the workload:
  * paged_n64_bf16 (default: the largest single-GPU workload, at the shared budget of 8
    slots per request), budget8n_bf16, full_width_bf16: verification attention (tile
    router -> split-KV work decomposition -> GQA-packed short tile -> online softmax ->
    PV -> combine), one launch;
  * wide_gqa_bf16: verification attention, draft-logit margin and the fused target
    margin + greedy acceptance (three launches).
The metric is verified candidate rows per second (rows = packed live rows M_live).
Inputs are resident in HBM when the timed region starts; consecutive steps rotate over
several independent input sets whose total footprint exceeds twice the L2 size, so a
step never finds its KV stream in L2.  Each step is one replay of a CUDA graph of its
launches, captured per input set (the C-ABI calls are capture-safe, as a serving loop
would replay its verify step), so the timed region holds no host work.  Timing events
recorded inside the graph around every launch give the per-kernel durations used for the
roofline: 16 copies of each graph are cycled, and the durations are those of the last
16 x sets steps of the timed region.  Rank 0 prints one JSON line.

--impl reference times the fp64 CPU oracle (the reference arm of this repository) on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
METRIC = "verified candidate rows/s and KV-stream HBM GB/s (% of GB300 peak) at N, budget"
NOMINAL_HBM_GBS = 8000.0

WORKLOAD_TEXT = {
    "full_width_bf16": "N=8 requests x 16 slots (128 packed rows), 32q/8kv heads, d=128, "
                       "contiguous KV context ~U[512,8192], bf16",
    "budget8n_bf16": "N=8 requests, shared budget 64 slots (8N), truncated-geometric "
                     "lengths, 32q/8kv, d=128, contiguous KV ~U[512,8192], bf16",
    "paged_n64_bf16": "N=64 requests, budget 512 slots (8N), 32q/8kv, d=128, paged KV "
                      "(16-token pages, shuffled block table) ~U[4096,32768], bf16",
    "wide_gqa_bf16": "N=32 x 7 slots (224 rows), 24q/2kv, d=256, KV ~U[1024,8192], plus "
                     "draft margin over [192,248320] and fused margin+greedy accept over "
                     "target logits [224,248320], bf16",
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default="paged_n64_bf16", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the contrast / other-workload measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill", action="store_true",
                    help="time only the wide-tile prefill contrast and print its JSON line")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value: float, world: int) -> float:
    """Max over ranks of a host float (timing plumbing only, not a data-path exchange)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ ours
def kv_bytes(b) -> int:
    """Algorithmic KV bytes of one attention launch: every context and candidate token's
    K and V row of each KV head is read once."""
    L = int(b.ctx_len.sum().item())
    k = int(b.cu_slots[-1].item())
    return (L + k) * b.hkv * b.d * 2 * b.q.element_size()


def attn_kwargs(b):
    if b.paged:
        return dict(k_cache=b.k_cache, v_cache=b.v_cache, block_table=b.block_table)
    return dict(k_ctx=b.k_ctx, v_ctx=b.v_ctx, cu_ctx=b.cu_ctx)


def build_step(b, svp, tile_mode=None):
    """Returns (launch list of (name, fn)), outputs preallocated; fixed workspaces."""
    import torch
    mode = svp.TILE_AUTO if tile_mode is None else tile_mode
    out = torch.empty_like(b.q)
    lse = torch.empty((b.m_cap, b.hq), dtype=torch.float32, device=b.q.device)
    kv = svp.make_kv(**attn_kwargs(b))
    ws = svp.Workspace(svp.verify_attn_workspace_size(b.n, b.m_cap, b.W, b.hq, b.hkv, b.d,
                                                      b.dtype, mode))

    def attn():
        svp.verify_attn_packed(b.q, b.k_new, b.v_new, b.ctx_len, b.cu_slots, w=b.W, kv=kv,
                               out=out, lse=lse, tile_mode=mode, ws=ws)

    launches = [("attn", attn)]
    if b.target_logits is not None and b.draft_logits is not None:
        V = b.target_logits.shape[1]
        dev = b.q.device
        rows_d = b.draft_logits.shape[0]
        d_outs = (torch.empty(rows_d, dtype=torch.int32, device=dev),) + tuple(
            torch.empty(rows_d, dtype=torch.float32, device=dev) for _ in range(3))
        ws_d = svp.Workspace(svp.draft_margin_workspace_size(rows_d, V))
        t_outs = (torch.empty(b.m_cap, dtype=torch.int32, device=dev),) + tuple(
            torch.empty(b.m_cap, dtype=torch.float32, device=dev) for _ in range(3)) + (
            torch.empty(b.n, dtype=torch.int32, device=dev),
            torch.empty(b.n, dtype=torch.int32, device=dev))
        ws_t = svp.Workspace(svp.margin_accept_workspace_size(b.n, b.m_cap, V))

        def draft():
            svp.draft_margin(b.draft_logits, ws=ws_d, outs=d_outs)

        def accept():
            svp.margin_accept(b.target_logits, b.tokens, b.cu_slots, ws=ws_t, outs=t_outs)

        launches += [("draft_margin", draft), ("margin_accept", accept)]
    return launches, (out, lse)


def step_bytes(b):
    kvb = kv_bytes(b)
    logit = 0
    if b.target_logits is not None and b.draft_logits is not None:
        logit = (b.m_live * b.target_logits.shape[1] + b.draft_logits.numel()) * 2
    return kvb, logit


def make_sets(name, nsets, seed, device):
    from speculative_decoding_verification_packed_gb300 import workloads as wl
    return [wl.make_batch(name, seed=seed + s, device=device) for s in range(nsets)]


def n_sets_for(b0) -> int:
    kvb, lg = step_bytes(b0)
    per = kvb + lg + 1
    return max(1, min(8, math.ceil(2 * L2_BYTES / per) + 1)) if per < 4 * L2_BYTES else 1


GRAPH_COPIES = 16   # step graphs per input set: the last replays of the timed region


def capture_step(plan, stream, copies=GRAPH_COPIES):
    """The whole step as one CUDA graph (the launches in order, as a serving loop replays
    its verify step), with a timing event recorded inside the graph before and after every
    launch.  `copies` graphs are captured, each with its own events, so that the timed
    loop can cycle through them and every copy keeps the durations of its last replay."""
    import torch
    # the workspaces were cleared on the default stream; the capture stream is non-blocking,
    # so the first calls below must not start before those clears are done
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _, fn in plan:
            fn()                      # first use: workspace signature, lazy init
    torch.cuda.synchronize()
    out = []
    for _ in range(copies):
        g = torch.cuda.CUDAGraph()
        evs = []
        with torch.cuda.graph(g, stream=stream):
            for name, fn in plan:
                e0 = torch.cuda.Event(enable_timing=True, external=True)
                e1 = torch.cuda.Event(enable_timing=True, external=True)
                e0.record()
                fn()
                e1.record()
                evs.append((name, e0, e1))
        out.append((g, evs))
    torch.cuda.synchronize()
    return out


def launch_dist(times_ms):
    """Median and nearest-rank p10 / p90 of per-launch device times (ms in, us out)."""
    xs = sorted(times_ms)
    if not xs:
        return None
    rank = lambda q: xs[min(len(xs) - 1, max(0, int(round(q * (len(xs) - 1)))))]
    return {"median": round(statistics.median(xs) * 1e3, 2), "p10": round(rank(0.1) * 1e3, 2),
            "p90": round(rank(0.9) * 1e3, 2)}


def timed_run(sets, steps, warmup, svp, tile_mode=None, clocks=None, dist_out=None):
    """K steps rotating over the input sets, each step one replay of a captured step graph
    (no host work inside the timed region).  ms per step from events on the stream around
    the K replays; per-launch device times from the events inside the graphs, i.e. from
    the last replay of every graph copy (the last copies x sets steps of the region)."""
    import torch
    stream = torch.cuda.current_stream()
    plans = [build_step(b, svp, tile_mode)[0] for b in sets]
    cap = torch.cuda.Stream()
    graphs = [capture_step(pl, cap) for pl in plans]
    nsets = len(graphs)
    pick = lambda s: graphs[s % nsets][(s // nsets) % GRAPH_COPIES]
    if clocks:
        clocks.start()          # sampling spans the warm-up and the timed region
        time.sleep(0.2)
    for w in range(warmup):
        pick(w)[0].replay()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    t0.record(stream)
    for s in range(steps):
        pick(s)[0].replay()
    t1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clk = clocks.stop() if clocks else None
    total_ms = t0.elapsed_time(t1)
    names = [n for n, _ in plans[0]]
    replayed = {(s % nsets, (s // nsets) % GRAPH_COPIES) for s in range(steps)}
    samples = [[] for _ in names]
    for (si, ci) in sorted(replayed):
        for li, (_, e0, e1) in enumerate(graphs[si][ci][1]):
            samples[li].append(e0.elapsed_time(e1))
    per_launch = [statistics.mean(x) for x in samples]
    if dist_out is not None:
        for li, name in enumerate(names):
            dist_out[name] = launch_dist(samples[li])
    return total_ms, dict(zip(names, per_launch)), clk, wall, steps * len(names)


def e2e_run(sets, steps, warmup, svp):
    """Same step through the public API with host (pinned) inputs: every step copies its
    inputs host->device, runs the step, and reads the outputs back."""
    import torch
    hosts = []
    for b in sets[:1]:        # one batch shape: every step re-uploads the same inputs
        h = {}
        for name in ("q", "k_new", "v_new", "ctx_len", "cu_slots", "k_ctx", "v_ctx", "cu_ctx",
                     "k_cache", "v_cache", "block_table", "tokens", "target_logits",
                     "draft_logits"):
            t = getattr(b, name)
            if t is not None:
                h[name] = t.cpu().pin_memory()
        hosts.append(h)
    b0 = sets[0]
    plan, (out, lse) = build_step(b0, svp)
    h2d = sum(t.numel() * t.element_size() for t in hosts[0].values())
    d2h_host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    d2h_host_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()
    stream = torch.cuda.current_stream()

    def one(s):
        h = hosts[s % len(hosts)]
        for name, t in h.items():
            getattr(b0, name).copy_(t, non_blocking=True)
        for _, fn in plan:
            fn()
        d2h_host_out.copy_(out, non_blocking=True)
        d2h_host_lse.copy_(lse, non_blocking=True)

    for w in range(warmup):
        one(w)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(steps):
        one(s)
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1), h2d, d2h


def traffic_record(workload: str, algorithmic_bytes: float):
    """DRAM bytes per launch of the attention kernel from the ncu capture summarised in
    profiles/attn_traffic.json, scaled from the captured launch to this launch's
    algorithmic bytes (traffic grows with the KV tiles streamed); None when the kernel
    source changed since the capture or no capture exists for the workload."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "attn_traffic.json")
    src = os.path.join(ROOT, "speculative_decoding_verification_packed_gb300", "csrc", "verify_tc.cu")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    r = rec.get(workload)
    if not r or r.get("kernel_src_sha") != h:
        return None
    return int(r["traffic_over_algorithmic"] * algorithmic_bytes)


def cpu_baseline(name, seed, budget_s=15.0):
    """The fp64 oracle timed on this host's cores on a bounded sample of the workload
    (whole requests, all heads, until about budget_s seconds of CPU work)."""
    import torch
    import oracle
    from speculative_decoding_verification_packed_gb300 import workloads as wl
    threads = os.cpu_count() or 1
    b = wl.make_batch(name, seed=seed, device="cpu", with_logits=False)
    cu = b.cu_slots.tolist()
    order = list(range(b.n)) * 64          # whole batch, repeated until the time budget
    done_rows, t_used, reqs = 0, 0.0, []
    for i in order:
        t0 = time.perf_counter()
        if b.paged:
            oracle.attention(b.q, b.k_new, b.v_new, b.ctx_len, b.cu_slots, hkv=b.hkv, scale=b.scale,
                             k_cache=b.k_cache, v_cache=b.v_cache, block_table=b.block_table,
                             cache_strides=b.cache_strides, requests=[i], threads=threads)
        else:
            oracle.attention(b.q, b.k_new, b.v_new, b.ctx_len, b.cu_slots, hkv=b.hkv, scale=b.scale,
                             k_ctx=b.k_ctx, v_ctx=b.v_ctx, cu_ctx=b.cu_ctx, requests=[i],
                             threads=threads)
        t_used += time.perf_counter() - t0
        done_rows += cu[i + 1] - cu[i]
        reqs.append(i)
        if t_used >= budget_s:
            break
    return {"value": done_rows / t_used, "unit": "rows/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(reqs)} request passes over the {b.n}-request batch in order "
                      f"({done_rows} rows, all {b.hq} heads) of {name}, seed {seed}, fp64 C "
                      f"oracle, {t_used:.1f} s"}


def run_ours(args):
    import torch
    import speculative_decoding_verification_packed_gb300 as svp
    from speculative_decoding_verification_packed_gb300 import build as svp_build

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    if rank == 0 or not os.path.exists(svp.LIB_PATH):
        svp_build.build()
    barrier(world)
    hbm_peak, tf_peak, peak_kind = measured_peaks()
    dev = torch.device("cuda", local)

    # the headline workload; each rank runs its own batch (weak scaling, no exchange)
    probe = make_sets(args.workload, 1, args.seed + 1000 * rank, dev)
    nsets = n_sets_for(probe[0])
    sets = probe + make_sets(args.workload, nsets - 1, args.seed + 1000 * rank + 1, dev)
    clocks = ClockSampler(local)
    barrier(world)
    dist = {}
    total_ms, per_launch, clk, wall, launches = timed_run(sets, args.steps, args.warmup, svp,
                                                          clocks=clocks, dist_out=dist)
    total_ms = reduce_max(total_ms, world)
    rows = reduce_sum(sum(int(sets[s % nsets].cu_slots[-1]) for s in range(args.steps)), world)
    ms_step = total_ms / args.steps
    value = rows / (total_ms / 1e3)
    kvb = statistics.mean(kv_bytes(b) for b in sets)
    attn_ms = per_launch["attn"]
    achieved = kvb / (attn_ms / 1e3) / 1e9
    tr = traffic_record(args.workload, kvb)
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; sizes and distributions of the workload)",
        "config": {"workload": args.workload, "description": WORKLOAD_TEXT[args.workload],
                   "n_requests": sets[0].n, "budget_slots": sets[0].m_cap,
                   "live_rows": int(sets[0].cu_slots[-1]),
                   "l2": f"{nsets} rotating input sets, {nsets * (kvb / 1e6):.0f} MB of KV "
                         f"(> 2x the 129 MB L2)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "traffic": tr, "kernel": "verify_tc_kernel",
                     "algorithmic_bytes_per_launch": int(kvb), "launch_us": round(attn_ms * 1e3, 2),
                     "peak_kind": peak_kind,
                     "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4)},
        "kv_gbs": round(achieved, 1),
        "per_launch_us": {k: round(v * 1e3, 2) for k, v in per_launch.items()},
        "per_launch_us_dist": dist,
        "gpu_launches": launches,
        "clocks": clk,
    }
    if "draft_margin" in per_launch:
        V = sets[0].target_logits.shape[1]
        lb = sets[0].draft_logits.numel() * 2
        result["draft_margin_gbs"] = round(lb / (per_launch["draft_margin"] / 1e3) / 1e9, 1)
        tb = int(sets[0].cu_slots[-1]) * V * 2
        result["margin_accept_gbs"] = round(tb / (per_launch["margin_accept"] / 1e3) / 1e9, 1)

    # end to end through the public API with host buffers (a step copies every input,
    # the KV context included, so large workloads take fewer steps)
    e2e_steps = max(3, min(args.steps // 5, int(2e10 // max(1, kvb))))
    e2e_ms, h2d, d2h = e2e_run(sets[:1], e2e_steps, 3, svp)
    e2e_rows = e2e_steps * int(sets[0].cu_slots[-1])
    result["e2e"] = {"value": round(e2e_rows / (e2e_ms / 1e3), 1), "unit": "rows/s",
                     "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                     "note": "all step inputs (incl. the KV context) copied from pinned host "
                             "memory every step"}

    if not args.no_extras and rank == 0:
        extras = {}
        # contrast: fixed 128-row tile, same inputs, same N
        fx_steps = max(5, min(200, args.steps // 4))
        fx_ms, fx_pl, _, _, _ = timed_run(sets, fx_steps, 3, svp, tile_mode=svp.TILE_FIXED128)
        fx_rows = sum(int(sets[s % nsets].cu_slots[-1]) for s in range(fx_steps))
        extras["fixed128_contrast"] = {
            "rows_per_s": round(fx_rows / (fx_ms / 1e3), 1),
            "kv_gbs": round(kvb / (fx_pl["attn"] / 1e3) / 1e9, 1),
            "short_tile_speedup": round(value / (fx_rows / (fx_ms / 1e3)), 3)}
        # contrast: the short tile without GQA packing (one query head per tile)
        un_ms, un_pl, _, _, _ = timed_run(sets, fx_steps, 3, svp, tile_mode=svp.TILE_SHORT_UNPACKED)
        un_rows = sum(int(sets[s % nsets].cu_slots[-1]) for s in range(fx_steps))
        extras["unpacked_short_contrast"] = {
            "rows_per_s": round(un_rows / (un_ms / 1e3), 1),
            "attn_us": round(un_pl["attn"] * 1e3, 2),
            "gqa_packing_speedup": round(value / (un_rows / (un_ms / 1e3)), 3)}
        for other in ("budget8n_bf16", "full_width_bf16", "paged_n64_bf16", "wide_gqa_bf16"):
            if other == args.workload:
                continue
            osets = make_sets(other, 1, args.seed, dev)
            n2 = n_sets_for(osets[0])
            osets += make_sets(other, n2 - 1, args.seed + 1, dev)
            st = max(5, min(100, args.steps // 20))
            oms, opl, _, _, _ = timed_run(osets, st, 3, svp)
            orows = sum(int(osets[s % n2].cu_slots[-1]) for s in range(st))
            okv = statistics.mean(kv_bytes(b) for b in osets)
            e = {"rows_per_s": round(orows / (oms / 1e3), 1),
                 "kv_gbs": round(okv / (opl["attn"] / 1e3) / 1e9, 1),
                 "kv_frac": round(okv / (opl["attn"] / 1e3) / 1e9 / hbm_peak, 4),
                 "per_launch_us": {k: round(v * 1e3, 2) for k, v in opl.items()}}
            # the attention launch also timed back to back (device time per call of a graph of
            # calls rotating over the sets); the step's events charge each launch its start-up gap
            bus = graph_us([dict(build_step(bb, svp)[0])["attn"] for bb in osets])
            e["attn_b2b_us"] = round(bus, 2)
            e["kv_frac_b2b"] = round(okv / (bus / 1e6) / 1e9 / hbm_peak, 4)
            fms, fpl, _, _, _ = timed_run(osets, st, 3, svp, tile_mode=svp.TILE_FIXED128)
            e["fixed128_rows_per_s"] = round(orows / (fms / 1e3), 1)
            ums, upl, _, _, _ = timed_run(osets, st, 3, svp, tile_mode=svp.TILE_SHORT_UNPACKED)
            e["unpacked_short_rows_per_s"] = round(orows / (ums / 1e3), 1)
            if "draft_margin" in opl:
                V = osets[0].target_logits.shape[1]
                e["draft_margin_gbs"] = round(osets[0].draft_logits.numel() * 2 /
                                              (opl["draft_margin"] / 1e3) / 1e9, 1)
                e["margin_accept_gbs"] = round(int(osets[0].cu_slots[-1]) * V * 2 /
                                               (opl["margin_accept"] / 1e3) / 1e9, 1)
                e["draft_margin_frac"] = round(e["draft_margin_gbs"] / hbm_peak, 4)
                e["margin_accept_frac"] = round(e["margin_accept_gbs"] / hbm_peak, 4)
            extras[other] = e
            del osets
            torch.cuda.empty_cache()
        extras["prefill_4096_causal"] = prefill_contrast(svp, dev, tf_peak)
        extras.update(next_rows_extras(svp, dev))
        # logit-stream kernels against the same measured HBM copy peak
        for key in ("stochastic_accept", "draft_features", "draft_margin_b2b", "margin_accept_b2b"):
            if key in extras:
                extras[key]["logit_frac"] = round(extras[key]["logit_gbs"] / hbm_peak, 4)
        result["extras"] = extras

    if not args.no_cpu_baseline and rank == 0 and world == 1:
        result["cpu_baseline"] = cpu_baseline(args.workload, args.seed)
    elif not args.no_cpu_baseline and rank == 0:
        result["cpu_baseline"] = cpu_baseline(args.workload, args.seed)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def prefill_contrast(svp, dev, tf_peak, reps: int = 10):
    """The wide-tile prefill contrast (tensor-bound): one causal sequence of 4096 rows,
    32 q / 8 KV heads, d = 128; 3 untimed launches, then `reps` launches timed with events."""
    import torch
    from speculative_decoding_verification_packed_gb300 import workloads as wl
    q, k, v = wl.make_prefill(device=dev)
    cu = torch.tensor([0, 4096], dtype=torch.int32, device=dev)
    pout = torch.empty_like(q)
    plse = torch.empty((4096, 32), dtype=torch.float32, device=dev)
    for _ in range(3):
        svp.prefill_attn(q, k, v, cu, max_s=4096, out=pout, lse=plse)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        svp.prefill_attn(q, k, v, cu, max_s=4096, out=pout, lse=plse)
    e1.record()
    torch.cuda.synchronize()
    pms = e0.elapsed_time(e1) / reps
    flops = 4.0 * 32 * 128 * (4096 * 4097 / 2)
    return {"us": round(pms * 1e3, 1), "tflops": round(flops / (pms / 1e3) / 1e12, 1),
            "frac_of_bf16_peak": round(flops / (pms / 1e3) / 1e12 / tf_peak, 4)}


def graph_us(fn, reps: int = 100, inner: int = 1) -> float:
    """Device time of one call (CUDA-graph replay, events on the replay stream).  fn may be a
    list of calls on different inputs (rotated so that consecutive calls do not find their
    input in L2); the time is per call.  inner > 1 captures the calls that many times in one
    graph, so that a call shorter than the host's replay overhead is still timed on the
    device."""
    import torch
    fns = (list(fn) if isinstance(fn, (list, tuple)) else [fn]) * inner
    for _ in range(3):
        for f in fns:
            f()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for f in fns:
                f()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps / len(fns) * 1e3


def next_rows_extras(svp, dev):
    """The allocator/packer, the captured step, the stochastic verifier, the draft features
    and the two margin launches back to back, each timed by graph replay (device time per
    call)."""
    import numpy as np
    import torch
    from speculative_decoding_verification_packed_gb300 import workloads as wl
    from speculative_decoding_verification_packed_gb300.pipeline import VerifyPipeline
    out = {}
    # DVL allocator + packer: budget 8N over W = 16, three batch sizes; retention of the
    # windows for labels drawn from the same prefix scores (a calibrated predictor)
    dv = {}
    for n in (8, 64, 512):
        rng = np.random.default_rng(n)
        sc = rng.beta(2.0, 1.2, (n, 15)).astype(np.float32)
        s_t = torch.from_numpy(sc).to(dev)
        gd = torch.Generator(device=dev)
        gd.manual_seed(n)
        tok = torch.randint(0, 150000, (n, 16), dtype=torch.int32, device=dev, generator=gd)
        pos = torch.randint(0, 1 << 20, (n, 16), dtype=torch.int32, device=dev, generator=gd)
        ws = svp.Workspace(256, dev)
        holder = {}

        def call():
            holder["r"] = svp.dvl_allocate_pack(s_t, budget_per_req=8, m_cap=16 * n, tokens=tok,
                                                positions=pos, kv_refs=tok, ws=ws)
        us = graph_us(call, inner=20)
        r = svp.dvl_allocate_pack(s_t, budget_per_req=8, m_cap=16 * n, ws=ws)
        q = np.minimum.accumulate(np.concatenate([np.ones((n, 1), np.float32), sc], axis=1), axis=1)
        u = rng.random((n, 15))
        passed = u < q[:, 1:]
        y = np.where(passed.all(axis=1), 15, np.argmin(passed, axis=1))
        k0 = r["k_init"].cpu().numpy().astype(np.int64)
        k = r["k"].cpu().numpy().astype(np.int64)
        ret = lambda kk: float(np.minimum(y, kk - 1).sum()) / max(1, int(y.sum()))
        dv[f"n{n}"] = {"us": round(us, 2), "retention_initial": round(ret(k0), 4),
                       "retention_adjusted": round(ret(k), 4),
                       "mean_window_initial": round(float(k0.mean()), 2),
                       "mean_window_adjusted": round(float(k.mean()), 2)}
    out["dvl_allocate_pack"] = dv
    # captured step: allocate/pack, gather, verify (full-width shapes), margin + accept
    n_bs, V = 8, 32000
    gc = torch.Generator().manual_seed(7)
    gd = torch.Generator(device=dev)
    gd.manual_seed(7)
    ctx = torch.randint(512, 8193, (n_bs,), dtype=torch.int32, generator=gc)
    cu_ctx = torch.zeros(n_bs + 1, dtype=torch.int64)
    cu_ctx[1:] = torch.cumsum(ctx.long(), 0)
    kc = torch.randn(int(cu_ctx[-1]), 8, 128, device=dev, generator=gd).to(torch.bfloat16)
    vc = torch.randn(int(cu_ctx[-1]), 8, 128, device=dev, generator=gd).to(torch.bfloat16)
    pipe = VerifyPipeline(n_bs, hq=32, hkv=8, d=128, vocab=V, ctx_len=ctx.to(dev),
                          kv_tensors=dict(k_ctx=kc, v_ctx=vc, cu_ctx=cu_ctx.to(dev)))
    pipe.scores.copy_(torch.rand(n_bs, 15, device=dev, generator=gd))
    pipe.q_full.normal_(generator=gd)
    pipe.k_full.normal_(generator=gd)
    pipe.v_full.normal_(generator=gd)
    pipe.logits_full.normal_(generator=gd)
    pipe.capture()
    for _ in range(3):
        pipe.step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(50):
        pipe.step()
    e1.record()
    torch.cuda.synchronize()
    out["captured_step"] = {"us": round(e0.elapsed_time(e1) / 50 * 1e3, 1),
                            "config": "8 requests, budget 8N = 64 slots, 32q/8kv d=128, ctx U[512,8192], vocab 32000"}
    del pipe, kc, vc
    torch.cuda.empty_cache()
    # stochastic verifier, draft features and the two margin launches on the wide-head
    # workload's logits, back-to-back calls in one graph rotating over three input sets
    # (2 x 207 MB of logits plus a copy of the first at its own address: no call finds its
    # logits in the 129 MB L2)
    bs = [wl.make_batch("wide_gqa_bf16", seed=sd, device=dev) for sd in (0, 1)]
    b = bs[0]
    V = b.target_logits.shape[1]
    lsets = [(bb.draft_logits, bb.target_logits, bb.tokens, bb.cu_slots) for bb in bs]
    lsets.append((b.draft_logits.clone(), b.target_logits.clone(), b.tokens, b.cu_slots))
    gu = torch.Generator(device=dev)
    gu.manual_seed(11)
    ua = torch.rand(b.m_cap, device=dev, generator=gu)
    un = torch.rand(b.n, device=dev, generator=gu)
    wss = svp.Workspace(svp.stochastic_accept_workspace_size(b.m_cap, V), dev)
    souts = (torch.empty(b.n, dtype=torch.int32, device=dev), torch.empty(b.n, dtype=torch.int32, device=dev),
             torch.empty(b.m_cap, dtype=torch.float32, device=dev))
    us = graph_us([lambda ls=ls: svp.stochastic_accept(ls[1], ls[2], ls[3], ua, un, temperature=1.0, ws=wss,
                                                       outs=souts) for ls in lsets])
    tb = int(b.cu_slots[-1]) * V * 2
    out["stochastic_accept"] = {"us": round(us, 2), "logit_gbs": round(tb / (us / 1e6) / 1e9, 1),
                                "config": "224 target rows x 248320 bf16, T = 1, 3 alternating input sets"}
    wsf = svp.Workspace(svp.draft_features_workspace_size(b.draft_logits.shape[0], V), dev)
    fout = torch.empty(b.draft_logits.shape[0], 18, dtype=torch.float32, device=dev)
    us = graph_us([lambda ls=ls: svp.draft_features(ls[0], ws=wsf, out=fout) for ls in lsets])
    db = b.draft_logits.numel() * 2
    out["draft_features"] = {"us": round(us, 2), "logit_gbs": round(db / (us / 1e6) / 1e9, 1),
                             "config": "192 draft rows x 248320 bf16, 18 values per row, 3 alternating input sets"}
    # the two margin launches of the wide-head step timed the same way; the step's
    # per-launch events (wide_gqa_bf16 extras) also charge each launch its start-up gap
    wsd = svp.Workspace(svp.draft_margin_workspace_size(b.draft_logits.shape[0], V), dev)
    dout = tuple(torch.empty(b.draft_logits.shape[0], dtype=t, device=dev)
                 for t in (torch.int32, torch.float32, torch.float32, torch.float32))
    us = graph_us([lambda ls=ls: svp.draft_margin(ls[0], ws=wsd, outs=dout) for ls in lsets])
    out["draft_margin_b2b"] = {"us": round(us, 2), "logit_gbs": round(db / (us / 1e6) / 1e9, 1),
                               "config": "192 draft rows x 248320 bf16, back-to-back calls, 3 alternating input sets"}
    wsm = svp.Workspace(svp.margin_accept_workspace_size(b.n, b.m_cap, V), dev)
    mout = tuple(torch.empty(b.m_cap, dtype=t, device=dev) for t in (torch.int32, torch.float32, torch.float32,
                                                                      torch.float32)) + \
        (torch.empty(b.n, dtype=torch.int32, device=dev), torch.empty(b.n, dtype=torch.int32, device=dev))
    us = graph_us([lambda ls=ls: svp.margin_accept(ls[1], ls[2], ls[3], ws=wsm, outs=mout) for ls in lsets])
    out["margin_accept_b2b"] = {"us": round(us, 2), "logit_gbs": round(tb / (us / 1e6) / 1e9, 1),
                                "config": "224 target rows x 248320 bf16 + greedy accept, back-to-back calls, "
                                          "3 alternating input sets"}
    return out


def run_reference(args):
    """The reference arm: the fp64 CPU oracle, one bounded sample per step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from speculative_decoding_verification_packed_gb300 import workloads as wl
    oracle.build()
    threads = os.cpu_count() or 1
    b = wl.make_batch(args.workload, seed=args.seed, device="cpu", with_logits=False)
    cu = b.cu_slots.tolist()
    kw = (dict(k_cache=b.k_cache, v_cache=b.v_cache, block_table=b.block_table,
               cache_strides=b.cache_strides) if b.paged else
          dict(k_ctx=b.k_ctx, v_ctx=b.v_ctx, cu_ctx=b.cu_ctx))

    # step s = request s mod n (all heads): the batch in order, one request per step,
    # so that a full cycle of steps is the whole workload
    def step(s):
        i = s % b.n
        oracle.attention(b.q, b.k_new, b.v_new, b.ctx_len, b.cu_slots, hkv=b.hkv, scale=b.scale,
                         requests=[i], threads=threads, **kw)
        return cu[i + 1] - cu[i]

    for w in range(min(args.warmup, 2)):      # warms the C library and page cache only
        step(w)
    t0 = time.perf_counter()
    rows = 0
    steps = 0
    # at most three passes over the batch and about a minute of host time, at least one step
    while steps < min(args.steps, 3 * b.n) and (steps == 0 or time.perf_counter() - t0 < 60.0):
        rows += step(steps)
        steps += 1
    dt = time.perf_counter() - t0
    value = rows / dt
    sample = (f"{steps} steps, step s = request s mod {b.n} of {args.workload} (all {b.hq} "
              f"heads), fp64 C oracle, {dt:.1f} s")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "rows/s",
        "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": round(dt / steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "description": WORKLOAD_TEXT[args.workload]},
        "cpu_baseline": {"value": round(value, 2), "unit": "rows/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 2), "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse_args()
    if args.prefill:
        import torch
        import speculative_decoding_verification_packed_gb300 as svp
        from speculative_decoding_verification_packed_gb300 import build as svp_build
        svp_build.build()
        torch.cuda.set_device(0)
        _, tf_peak, kind = measured_peaks()
        r = prefill_contrast(svp, torch.device("cuda", 0), tf_peak, reps=max(1, args.steps))
        r.update({"workload": "prefill_4096_causal", "peak_tflops": tf_peak, "peak_kind": kind})
        print(json.dumps(r), flush=True)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
