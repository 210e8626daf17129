#!/usr/bin/env python3
"""Benchmark of FP8 paged MLA decode on one GB300 (or N replicas).

Workload (default): the MTP decode shape of the FlashMLA "update fp8
support" page -- b=64, s_q=2 (causal), h_q=64, d=576 (512 latent + 64 RoPE),
dv=512, one KV head, page 64, seeded synthetic inputs with cache lengths
uniform in [2048, 6144] (mean 4096), E4M3 KV with a per-tensor scale, FP8
Q/P dots.  One step = the whole hot path over one batch: the tile
scheduler (metadata), the decode kernel and the split-KV combine.

Metric: TFLOPS with FLOPs = 2 * b * s_q * h_q * s_k * (576 + 512) summed
over sequences (the convention that reproduces the page's TFLOPS column);
the JSON line also carries us/call, KV GB/s and the roofline fraction.

Timing: CUDA events on the launching stream around exactly K steps after W
warm-up steps, a barrier and a synchronize on both sides, max over ranks.
Three copies of the inputs (3 x ~165 MB, more than twice the 129 MB L2)
rotate between steps, so every step reads its KV from HBM.

Multi-GPU: the batch is data-parallel and needs no exchange, so N GPUs run
N independent replicas of the per-GPU batch ("scaling": "weak").

``--impl reference`` times the fp64 CPU oracle on the same workload (a
bounded sample of sequences per step) on the host cores.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

MLA_D, MLA_DV = 576, 512
METRIC = "FP8-KV MLA decode µs/call, TFLOPS, KV GB/s and % roofline (b=64,s_q=2,s_k=4096)"
WORKLOAD = dict(workload="mla_mtp_decode", b=64, s_q=2, h_q=64, h_kv=1, d=576, dv=512, page=64,
                seqlens="uniform[2048,6144] seed 2", causal=True)
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "mla_decode_fp8_b64_sq2_traffic.txt")
KERNEL_SOURCE = os.path.join(ROOT, "paged_decode_attention_fp8_gb300", "csrc", "mla_decode.cu")


# ----------------------------------------------------------- accounting ----


def replica_seed(rank: int) -> int:
    """Seed of rank's batch: every replica draws its own Q and KV values (the
    sequence lengths stay those of seed 2, so every replica does the same work)."""
    return 2 + 1000 * rank


def slowest_rank_ms(ms: float, world: int, device=None) -> float:
    """The timed region's length on the slowest rank: a MAX all-reduce over
    the default process group (NCCL on GPUs, gloo in the CPU tests)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_replica: float, ms_per_step: float) -> float:
    """TFLOPS of the whole job: the work of all `world` replicas over one step
    of the slowest rank."""
    return world * flops_per_replica / (ms_per_step * 1e-3) / 1e12


def mla_flops(seqlens, s_q, h_q, d=MLA_D, dv=MLA_DV):
    """2 * s_q * h_q * s_k * (d + dv) per sequence (causal mask not discounted)."""
    return sum(2.0 * s_q * h_q * int(s) * (d + dv) for s in seqlens)


def mla_split_flops(seqlens, s_q, h_q):
    """(FP8 flops, bf16 flops): latent Q.K and P.V run in E4M3, the 64-wide RoPE chunk in bf16."""
    keys = sum(int(s) for s in seqlens)
    return 2.0 * s_q * h_q * keys * (512 + MLA_DV), 2.0 * s_q * h_q * keys * 64


def mla_bytes(seqlens, b, s_q, h_q):
    """Algorithmic bytes: valid KV rows (576 B each), Q (bf16), out (bf16), lse (f32),
    the block-table entries of the used pages and the seqlens."""
    kv = sum(int(s) for s in seqlens) * MLA_D
    pages = sum((int(s) + 63) // 64 for s in seqlens)
    rows = b * s_q * h_q
    return kv + rows * MLA_D * 2 + rows * MLA_DV * 2 + rows * 4 + pages * 4 + b * 4


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, src="fallback")


def traffic_from_profile():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel source."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(KERNEL_SOURCE, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    vals = {}
    with open(PROFILE_TRAFFIC) as f:
        for line in f:
            m = re.match(r"^(\w+):\s*(\S+)", line.strip())
            if m:
                vals[m.group(1)] = m.group(2)
    if vals.get("kernel_source_sha256_16") != sha:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------------- clocks ----


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"], samples=0)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["no samples"], samples=0)
        return dict(sm_mhz=statistics.median(sm), sm_max_mhz=max(smax), reasons=sorted(reasons), samples=len(sm))


# ---------------------------------------------------------- our arm ----


def build_inputs(seed, device, copies=3):
    import torch

    from paged_decode_attention_fp8_gb300 import synthetic as syn
    w = WORKLOAD
    seqlens = syn.uniform_seqlens(2, w["b"], 2048, 6144)
    inp = syn.mla_inputs(seed, w["b"], w["s_q"], w["h_q"], seqlens, causal=True, spare_pages=64)
    sets = []
    for c in range(copies):
        q = inp.q.to(device)
        kv = inp.kv_cache.to(device)
        sets.append((q, kv))
    bt = inp.block_table.to(device)
    sl = inp.seqlens.to(device)
    scale = torch.tensor([inp.kv_scale], dtype=torch.float32, device=device)
    return inp, seqlens, sets, bt, sl, scale


def run_ours(args):
    import torch
    import torch.distributed as dist

    import paged_decode_attention_fp8_gb300 as fm

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOAD
    b, s_q, h_q = w["b"], w["s_q"], w["h_q"]
    inp, seqlens, sets, bt, sl, scale = build_inputs(replica_seed(rank), dev)
    units = fm.metadata_units()
    tile_sched = torch.empty((units, 8), dtype=torch.int32, device=dev)
    num_splits = torch.empty((b + 1,), dtype=torch.int32, device=dev)
    out = torch.empty((b, s_q, h_q, MLA_DV), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((b, s_q, h_q), dtype=torch.float32, device=dev)
    ws = torch.empty((fm.workspace_bytes(b, s_q, h_q, units),), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    dot = args.dot

    def step(i, ev=None):
        q, kv = sets[i % len(sets)]
        fm.get_metadata(sl, h_q, s_q, num_units=units, tile_sched=tile_sched, num_splits=num_splits)
        if ev is not None:
            ev[0].record(stream)
        fm.decode(q, kv, bt, sl, scale, inp.softmax_scale, True, tile_sched, num_splits, dot_mode=dot,
                  out=out, lse=lse, workspace=ws)
        if ev is not None:
            ev[1].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert fm.last_device_error() == 0

    kernel_events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    host0 = time.perf_counter()
    host_n, host_us = min(args.steps, 100), 0.0
    for i in range(args.steps):
        step(i)
        if i + 1 == host_n:  # enqueue cost of the first steps, before the launch queue fills and the host
            host_us = (time.perf_counter() - host0) * 1e6 / host_n  # waits on the GPU: below the step time
                                                                    # means the loop is GPU-bound
    t1.record(stream)
    torch.cuda.synchronize()
    # The decode call's own duration: the same steps again with events around
    # the call (events between the launches would break their programmatic
    # overlap, so they stay out of the pass above).
    for i in range(args.steps):
        step(i, kernel_events[i])
    torch.cuda.synchronize()
    # Each kernel of the call alone: a third pass with the library's stage
    # events between its launches (they stop the launches overlapping, so this
    # pass times the kernels, not the call).
    fm.set_stage_timing(True)
    stages = []
    for i in range(min(args.steps, 500)):
        step(i)
        stages.append(fm.stage_times())
    fm.set_stage_timing(False)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = slowest_rank_ms(t0.elapsed_time(t1), world, dev)
    dec_ms = [a.elapsed_time(b_) for a, b_ in kernel_events]
    assert fm.last_device_error() == 0

    ms_per_step = total_ms / args.steps
    flops = mla_flops(seqlens, s_q, h_q)
    nbytes = mla_bytes(seqlens, b, s_q, h_q)
    kv_bytes = sum(seqlens) * MLA_D
    value = whole_job_tflops(world, flops, ms_per_step)

    peaks = measured_peaks()
    dec_avg_ms = sum(dec_ms) / len(dec_ms)
    stage_ms = [sum(x[k] for x in stages) / len(stages) for k in range(3)]
    kern_ms = stage_ms[1]
    achieved = nbytes / (kern_ms * 1e-3) / 1e9
    f8, f16 = mla_split_flops(seqlens, s_q, h_q)
    fp8_peak = 2.0 * peaks["bf16"]        # nominal E4M3 / bf16 dense ratio (4.5 / 2.25)
    t_hbm = nbytes / (peaks["hbm"] * 1e9)
    t_tensor = f8 / (fp8_peak * 1e12) + f16 / (peaks["bf16"] * 1e12)
    call_achieved = nbytes / (dec_avg_ms * 1e-3) / 1e9
    roofline = dict(bound="hbm" if t_hbm >= t_tensor else "tensor", achieved=round(achieved, 1),
                    peak=peaks["hbm"], unit="GB/s", frac=round(achieved / peaks["hbm"], 4),
                    traffic=traffic_from_profile(),
                    kernel=("mla_fp8_kernel" if dot == "fp8" else "mla_fp8_kernel (two-term 16-bit dots)") +
                    " alone (stage events around its launch, separate pass)",
                    kernel_us=round(kern_ms * 1e3, 2),
                    call_us=round(dec_avg_ms * 1e3, 2),
                    call_achieved=round(call_achieved, 1),
                    call_frac=round(call_achieved / peaks["hbm"], 4),
                    stages_us=dict(q_prep=round(stage_ms[0] * 1e3, 2), decode=round(stage_ms[1] * 1e3, 2),
                                   combine=round(stage_ms[2] * 1e3, 2)),
                    algorithmic_bytes_per_launch=nbytes,
                    t_hbm_us=round(t_hbm * 1e6, 2), t_tensor_us=round(t_tensor * 1e6, 2),
                    roofline_frac_of_time=round(max(t_hbm, t_tensor) / (kern_ms * 1e-3), 4),
                    peak_source=f"{peaks['src']} (MEASURED_PEAKS.json hbm_gbs; fp8 = 2 x bf16_tflops)")

    e2e = None if args.no_e2e else measure_e2e(args, inp, seqlens, sets, bt, sl, scale, dev, units, flops, world)

    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3" if dot == "fp8" else "e4m3 two-term (16-bit dots)",
        "data": "synthetic (seeded N(0,1) Q/KV, E4M3 per-tensor scale)",
        "config": dict(WORKLOAD, dot=dot, l2="3 rotating input copies (~495 MB) > 2x L2",
                       parallelism=f"replicas x{world}"),
        "us_per_call": round(dec_avg_ms * 1e3, 2),
        "us_per_step": round(ms_per_step * 1e3, 2),
        "host_enqueue_us_per_step": round(host_us, 1),
        "tflops_decode_call": round(flops / (dec_avg_ms * 1e-3) / 1e12, 1),
        "kv_gbs": round(kv_bytes / (dec_avg_ms * 1e-3) / 1e9, 1),
        "roofline": roofline,
        "clocks": clk,
        "e2e": e2e,
        # per step: schedule, Q quantisation, decode, combine
        "gpu_launches": 4 * args.steps,
    }
    if rank == 0 and world == 1 and not args.no_legs:
        # the other rows of the path, each on its own workload (not part of the headline value)
        del sets
        res["legs"] = run_legs(dev, max(20, min(args.steps, 200)), 5)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(inp, seqlens, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        dist.destroy_process_group()


def measure_e2e(args, inp, seqlens, sets, bt, sl, scale, dev, units, flops, world):
    """Same metric through the public API with host buffers: each step copies Q, the block
    table and the seqlens from pinned host memory, runs metadata + decode, and reads out + lse
    back.  The KV cache is the model's resident state (like weights) and stays in HBM.  The
    copies run on two copy streams (one per direction) into double-buffered device and host
    buffers, so a step's transfers overlap its neighbours' compute, as a serving loop would
    overlap them; every step still moves its own inputs in and its own results out inside the
    timed region."""
    import torch

    import paged_decode_attention_fp8_gb300 as fm
    w = WORKLOAD
    b, s_q, h_q = w["b"], w["s_q"], w["h_q"]
    q_h = inp.q.pin_memory()
    bt_h = inp.block_table.pin_memory()
    sl_h = inp.seqlens.pin_memory()
    nbuf = 2
    out_h = [torch.empty((b, s_q, h_q, MLA_DV), dtype=torch.bfloat16).pin_memory() for _ in range(nbuf)]
    lse_h = [torch.empty((b, s_q, h_q), dtype=torch.float32).pin_memory() for _ in range(nbuf)]
    q_d = [torch.empty_like(inp.q, device=dev) for _ in range(nbuf)]
    bt_d = [torch.empty_like(inp.block_table, device=dev) for _ in range(nbuf)]
    sl_d = [torch.empty_like(inp.seqlens, device=dev) for _ in range(nbuf)]
    out = [torch.empty((b, s_q, h_q, MLA_DV), dtype=torch.bfloat16, device=dev) for _ in range(nbuf)]
    lse = [torch.empty((b, s_q, h_q), dtype=torch.float32, device=dev) for _ in range(nbuf)]
    ts = torch.empty((units, 8), dtype=torch.int32, device=dev)
    ns = torch.empty((b + 1,), dtype=torch.int32, device=dev)
    ws = torch.empty((fm.workspace_bytes(b, s_q, h_q, units),), dtype=torch.uint8, device=dev)
    h2d_s = torch.cuda.Stream(dev)
    d2h_s = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]    # a slot's inputs are on the device
    ev_done = [torch.cuda.Event() for _ in range(nbuf)]  # a slot's decode finished reading and writing
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]   # a slot's results are back on the host
    steps = max(args.steps // 10, 20)

    def step(i, stream, first):
        k = i % nbuf
        _, kv = sets[i % len(sets)]
        with torch.cuda.stream(h2d_s):
            if not first:
                h2d_s.wait_event(ev_done[k])  # the decode two steps back has read this slot
            q_d[k].copy_(q_h, non_blocking=True)
            bt_d[k].copy_(bt_h, non_blocking=True)
            sl_d[k].copy_(sl_h, non_blocking=True)
            ev_in[k].record(h2d_s)
        stream.wait_event(ev_in[k])
        if not first:
            stream.wait_event(ev_out[k])  # this slot's previous results have left the device
        fm.get_metadata(sl_d[k], h_q, s_q, num_units=units, tile_sched=ts, num_splits=ns)
        fm.decode(q_d[k], kv, bt_d[k], sl_d[k], scale, inp.softmax_scale, True, ts, ns, dot_mode=args.dot,
                  out=out[k], lse=lse[k], workspace=ws)
        ev_done[k].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(ev_done[k])
            out_h[k].copy_(out[k], non_blocking=True)
            lse_h[k].copy_(lse[k], non_blocking=True)
            ev_out[k].record(d2h_s)

    def timed(run, n_steps, stream):
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        h2d_s.wait_event(t0)
        d2h_s.wait_event(t0)
        host0 = time.perf_counter()
        run()
        host_us = (time.perf_counter() - host0) * 1e6 / n_steps
        stream.wait_stream(h2d_s)  # the timed region ends when the last results are on the host
        stream.wait_stream(d2h_s)
        t1.record(stream)
        torch.cuda.synchronize()
        return slowest_rank_ms(t0.elapsed_time(t1), world, dev) / n_steps, host_us

    # eager: every step's copies, calls and events enqueued from Python
    stream = torch.cuda.current_stream(dev)
    for i in range(3):
        step(i, stream, i < nbuf)
    eager_ms, eager_host_us = timed(lambda: [step(i, stream, False) for i in range(steps)], steps, stream)

    # graph: the same calls captured once as a chain of `per_graph` steps and replayed, so
    # that Python's per-call cost leaves the loop (every step still copies its own inputs in
    # and its own results out); consecutive replays run one after another
    per_graph = 50
    replays = max(1, steps // per_graph)
    graph_ms = graph_host_us = None
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=cap):
            h2d_s.wait_stream(cap)
            d2h_s.wait_stream(cap)
            for i in range(per_graph):
                step(i, cap, i < nbuf)
            cap.wait_stream(h2d_s)
            cap.wait_stream(d2h_s)
        for _ in range(2):
            g.replay()
        graph_ms, graph_host_us = timed(lambda: [g.replay() for _ in range(replays)], replays * per_graph, stream)
    except Exception as exc:  # capture unsupported here: report the eager loop alone
        print(f"e2e graph capture failed: {exc!r}", file=sys.stderr)
    use_graph = graph_ms is not None and graph_ms < eager_ms
    ms = graph_ms if use_graph else eager_ms
    h2d = q_h.numel() * 2 + bt_h.numel() * 4 + sl_h.numel() * 4
    d2h = out_h[0].numel() * 2 + lse_h[0].numel() * 4
    return dict(value=round(whole_job_tflops(world, flops, ms), 2), unit="TFLOPS", ms_per_step=round(ms, 5),
                h2d_bytes_per_step=int(h2d), d2h_bytes_per_step=int(d2h),
                steps=replays * per_graph if use_graph else steps,
                launch="cuda graph of %d steps, replayed" % per_graph if use_graph else "eager",
                eager_ms_per_step=round(eager_ms, 5), eager_host_us_per_step=round(eager_host_us, 1),
                graph_ms_per_step=None if graph_ms is None else round(graph_ms, 5),
                note="KV cache resident in HBM; per-step Q/block table/seqlens in, out/lse back, on two copy "
                     "streams overlapping the neighbouring steps' compute (double-buffered)")


# ------------------------------------------------------- measurement legs ----
#
# Every other row of the path, timed on one GPU after the headline: each leg
# builds its seeded inputs, times `steps` calls with CUDA events around each
# call (after warm-up), and reports us/call with the roofline of its own
# algorithmic bytes and flops.  L2: every leg reads more than L2 (129 MB) per
# call or rotates input copies that together exceed it.


def _time_calls(call, steps, warmup, stream):
    import torch

    import paged_decode_attention_fp8_gb300 as fm
    for i in range(warmup):
        call(i)
    torch.cuda.synchronize()
    assert fm.last_device_error() == 0
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        evs[i][0].record(stream)
        call(warmup + i)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    assert fm.last_device_error() == 0
    ms = sorted(a.elapsed_time(b) for a, b in evs)
    _graph_time.last = _graph_replay_ms(call, warmup + steps, stream)
    return sum(ms) / len(ms), ms


def _graph_replay_ms(call, base, stream, per_graph=20, replays=10):
    """Per-call device time of `per_graph` calls captured as one CUDA graph and replayed
    back to back (no host enqueue in the timed region), or None if capture fails here."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=cap):
            for i in range(per_graph):
                call(base + i)
        g.replay()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(replays):
            g.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / (per_graph * replays)
    except Exception as exc:
        print(f"graph timing unavailable: {exc!r}", file=sys.stderr)
        return None


class _graph_time:  # the last _time_calls' graph-replayed per-call time (ms), for _leg_result
    last = None


def _leg_result(metric, avg_ms, ms, nbytes, flops_fp8, flops_16, peaks, cfg, launches):
    t_hbm = nbytes / (peaks["hbm"] * 1e9)
    t_tensor = flops_fp8 / (2.0 * peaks["bf16"] * 1e12) + flops_16 / (peaks["bf16"] * 1e12)
    flops = flops_fp8 + flops_16
    achieved = nbytes / (avg_ms * 1e-3) / 1e9
    return {
        "metric": metric, "value": round(avg_ms * 1e3, 2), "unit": "us/call", "higher_is_better": False,
        "graph_us_per_call": None if _graph_time.last is None else round(_graph_time.last * 1e3, 2),
        "config": cfg, "p10_us": round(ms[len(ms) // 10] * 1e3, 2),
        "p90_us": round(ms[(9 * len(ms)) // 10] * 1e3, 2), "calls": len(ms),
        "tflops": round(flops / (avg_ms * 1e-3) / 1e12, 2) if flops else None,
        "roofline": dict(bound="hbm" if t_hbm >= t_tensor else "tensor", achieved=round(achieved, 1),
                         peak=peaks["hbm"], unit="GB/s", frac=round(achieved / peaks["hbm"], 4),
                         algorithmic_bytes_per_launch=int(nbytes), t_hbm_us=round(t_hbm * 1e6, 2),
                         t_tensor_us=round(t_tensor * 1e6, 2),
                         roofline_frac_of_time=round(max(t_hbm, t_tensor) / (avg_ms * 1e-3), 4)),
        "gpu_launches_per_call": launches,
    }


def leg_mla(dev, peaks, steps, warmup, dot, seqlens, seed, label, value_pages=None, rows=False):
    """Dense MLA decode call (FP8 or 16-bit dots) on b = len(seqlens), s_q = 2, h_q = 64; with
    rows, one KV scale per cached row ([num_pages, 1, 64], FP8 dots)."""
    import torch

    import paged_decode_attention_fp8_gb300 as fm
    from paged_decode_attention_fp8_gb300 import synthetic as syn
    b, s_q, h_q = len(seqlens), 2, 64
    if rows:
        inp, row_scales = syn.mla_row_scaled_inputs(seed, b, s_q, h_q, seqlens, causal=True, spare_pages=16,
                                                    value_pages=value_pages)
    else:
        inp = syn.mla_inputs(seed, b, s_q, h_q, seqlens, causal=True, spare_pages=16, value_pages=value_pages)
    kv_bytes = sum(seqlens) * MLA_D
    copies = max(1, min(3, math.ceil(2 * 129e6 / kv_bytes)))
    kvs = [inp.kv_cache.to(dev) for _ in range(copies)]
    q, bt, sl = inp.q.to(dev), inp.block_table.to(dev), inp.seqlens.to(dev)
    scale = row_scales.to(dev) if rows else torch.tensor([inp.kv_scale], dtype=torch.float32, device=dev)
    units = fm.metadata_units()
    ts, ns = fm.get_metadata(sl, h_q, s_q, num_units=units)
    out = torch.empty((b, s_q, h_q, MLA_DV), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((b, s_q, h_q), dtype=torch.float32, device=dev)
    ws = torch.empty((fm.workspace_bytes(b, s_q, h_q, units),), dtype=torch.uint8, device=dev)

    def call(i):
        fm.decode(q, kvs[i % copies], bt, sl, scale, inp.softmax_scale, True, ts, ns, dot_mode=dot, out=out,
                  lse=lse, workspace=ws)

    avg, ms = _time_calls(call, steps, warmup, torch.cuda.current_stream(dev))
    f8, f16 = mla_split_flops(seqlens, s_q, h_q)
    if dot != "fp8":
        f8, f16 = 0.0, f8 + f16
    cfg = dict(workload="mla_decode", b=b, s_q=s_q, h_q=h_q, d=576, dv=512, page=64, seqlens=label, causal=True,
               dot=dot, l2=f"{copies} rotating cache copies ({copies * kv_bytes / 1e6:.0f} MB)",
               values="pooled N(0,1) pages" if value_pages else "N(0,1)",
               scales="per row [num_pages, 1, 64], (amax/448) 2^U[0,3]" if rows else "per tensor")
    nbytes = mla_bytes(seqlens, b, s_q, h_q) + (sum((x + 63) // 64 for x in seqlens) * 64 * 4 if rows else 0)
    what = f"{label}, {dot} dots" + (", per-row KV scales" if rows else "")
    res = _leg_result(f"dense MLA decode us/call ({what})", avg, ms, nbytes, f8, f16, peaks, cfg, 3)
    res["tflops_convention"] = round(mla_flops(seqlens, s_q, h_q) / (avg * 1e-3) / 1e12, 1)
    return res


def leg_sparse(dev, peaks, steps, warmup, s_q):
    import torch

    import paged_decode_attention_fp8_gb300 as fm
    from paged_decode_attention_fp8_gb300 import synthetic as syn
    rule = "affine" if s_q > 256 else "permutation"  # prefill-sized batches: vectorised index draw
    inp = syn.sparse_inputs(4, s_q, index_rule=rule)
    sets = [(inp.q.to(dev), inp.kv_cache.to(dev)) for _ in range(3)]
    idx = inp.topk_idx.to(dev)
    scale = torch.tensor([inp.kv_scale], dtype=torch.float32, device=dev)
    h_q, topk = inp.q.shape[1], idx.shape[1]
    ws = torch.empty((max(fm.sparse_workspace_bytes(s_q, h_q, topk, 0), 256),), dtype=torch.uint8, device=dev)
    out = torch.empty((s_q, h_q, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((s_q, h_q), dtype=torch.float32, device=dev)

    def call(i):
        q, kv = sets[i % len(sets)]
        fm.sparse_mla_decode(q, kv, idx, scale, inp.softmax_scale, out=out, lse=lse, workspace=ws)

    avg, ms = _time_calls(call, steps, warmup, torch.cuda.current_stream(dev))
    nbytes = s_q * topk * 512 + 2 * s_q * h_q * 512 * 2 + s_q * h_q * 4 + s_q * topk * 4
    flops = 2.0 * s_q * h_q * topk * 1024
    cfg = dict(workload="sparse_topk_mla_decode", s_q=s_q, h_q=h_q, d=512, topk=topk, num_tokens=131072,
               dot="fp8", splits="auto", indices=rule, l2="3 rotating cache copies (192 MiB) > L2")
    launches = 1 if fm.sparse_workspace_bytes(s_q, h_q, topk, 0) == 0 else 2
    return _leg_result(f"sparse top-k MLA decode us/call (s_q={s_q}, 16 heads, top-k 2048)", avg, ms, nbytes,
                       flops, 0.0, peaks, cfg, launches)


def leg_gqa(dev, peaks, steps, warmup, variant="plain"):
    """Paged GQA decode, bs = 32, 32/8 heads, hd 128, ctx U[1024, 16384].  variant "plain": one
    query token, per-tensor scales (paged_gqa_decode); "rows": one KV scale per cached row;
    "xqa": a speculative block of 4 query tokens with a seeded block mask, a 4096-key sliding
    window and attention sinks (paged_gqa_decode_ext)."""
    import torch

    import paged_decode_attention_fp8_gb300 as fm
    from paged_decode_attention_fp8_gb300 import synthetic as syn
    seqlens = syn.uniform_seqlens(5, 32, 1024, 16384)
    inp = syn.gqa_inputs(5, 32, seqlens, value_blocks=4096)
    sets = [(inp.k_cache.to(dev), inp.v_cache.to(dev)) for _ in range(2)]
    bt, sl = inp.block_table.to(dev), inp.seqlens.to(dev)
    bs, h_q, hd = inp.q.shape
    h_kv = inp.k_cache.shape[1]
    q_len, window = (4, 4096) if variant == "xqa" else (1, 0)
    if variant == "rows":
        shape = tuple(inp.k_cache.shape[:3])
        ks = syn.per_row_scales(5, 50, shape, inp.k_scale).to(dev)
        vs = syn.per_row_scales(5, 51, shape, inp.v_scale).to(dev)
    else:
        ks = torch.tensor([inp.k_scale], dtype=torch.float32, device=dev)
        vs = torch.tensor([inp.v_scale], dtype=torch.float32, device=dev)
    q = (syn.gqa_block_q(5, bs, q_len, h_q) if variant == "xqa" else inp.q.unsqueeze(1)).to(dev)
    mask = syn.spec_mask(5, bs, q_len).to(dev) if variant == "xqa" else None
    sinks = syn.sink_logits(5, h_q).to(dev) if variant == "xqa" else None
    # the split count each entry point will choose (the extended one is window-aware)
    splits = (fm.gqa_num_splits(bs, h_kv, bt.shape[1] * 16) if variant == "plain"
              else fm.gqa_ext_num_splits(bs, h_kv, bt.shape[1] * 16, q_len, window))
    ws = torch.empty((max(fm.gqa_workspace_bytes(bs, h_q, hd, splits), 256),), dtype=torch.uint8, device=dev)
    out = torch.empty((bs, q_len, h_q, hd), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((bs, q_len, h_q), dtype=torch.float32, device=dev)

    def call(i):
        kc, vc = sets[i % len(sets)]
        if variant == "plain":
            fm.paged_gqa_decode(q[:, 0], kc, vc, bt, sl, ks, vs, inp.softmax_scale, num_splits=0, out=out[:, 0],
                                lse=lse[:, 0], workspace=ws)
        else:
            fm.paged_gqa_decode_ext(q, kc, vc, bt, sl, ks, vs, inp.softmax_scale, spec_mask=mask, window=window,
                                    sinks=sinks, num_splits=0, out=out, lse=lse, workspace=ws)

    avg, ms = _time_calls(call, steps, warmup, torch.cuda.current_stream(dev))
    # keys a call must read: all of them, or with the window the last W + q_len - 1 of each sequence
    keys = sum(min(x, window + q_len - 1) if window else x for x in seqlens)
    nbytes = (keys * h_kv * hd * 2 + 2 * bs * q_len * h_q * hd * 2 + bs * q_len * h_q * 4 +
              sum((x + 15) // 16 for x in seqlens) * 4)
    if variant == "rows":
        nbytes += keys * h_kv * 2 * 4
    flops = 2.0 * keys * q_len * h_q * hd * 2
    cfg = dict(workload="paged_gqa_decode", bs=bs, h_q=h_q, h_kv=h_kv, head_dim=hd, page=16,
               seqlens="uniform[1024,16384] seed 5", splits=splits, values="pooled N(0,1) blocks",
               l2="2 rotating cache copies (~1.1 GB) > L2")
    if variant == "plain":
        cfg.update(dot="e4m3 operands, Q and P as two E4M3 terms", scales="per tensor")
        what = "bs=32, 32/8 heads, hd 128, ctx U[1024,16384]"
    elif variant == "rows":
        cfg.update(dot="e4m3 operands, Q and P as two E4M3 terms", scales="per row [num_blocks, h_kv, 16], base 2^U[-2,2]")
        what = "bs=32, 32/8 heads, hd 128, ctx U[1024,16384], per-row KV scales"
    else:
        cfg.update(dot="e4m3 operands, Q and P as two E4M3 terms", scales="per tensor", q_len=q_len,
                   mask="seeded block mask", window=window,
                   sinks="seeded logits U[-2,6]")
        what = "bs=32, 32/8 heads, hd 128, ctx U[1024,16384], 4-token speculative block, window 4096, sinks"
    return _leg_result(f"paged GQA decode us/call ({what})", avg, ms, nbytes, 0.0, flops, peaks, cfg,
                       1 if splits == 1 else 2)


def leg_kvwrite(dev, peaks, steps, warmup):
    import torch

    import paged_decode_attention_fp8_gb300 as fm
    from paged_decode_attention_fp8_gb300 import synthetic as syn
    seqlens = syn.uniform_seqlens(5, 32, 1024, 16384)
    kin, vin = syn.cache_write_inputs(5, seqlens), syn.cache_write_inputs(6, seqlens)
    xk, xv = syn.materialise(kin, device=dev), syn.materialise(vin, device=dev)
    slots = kin.slot_mapping.to(dev)
    n_tok, h_kv, hd = xk.shape
    caches = [torch.empty((kin.num_blocks, h_kv, 16, hd), dtype=torch.uint8, device=dev) for _ in range(2)]
    scales = [torch.empty((kin.num_blocks, h_kv, 16), dtype=torch.float32, device=dev) for _ in range(2)]

    def call(i):
        fm.paged_cache_write(xk, slots, caches[0], token_scales=scales[0])
        fm.paged_cache_write(xv, slots, caches[1], token_scales=scales[1])

    avg, ms = _time_calls(call, steps, warmup, torch.cuda.current_stream(dev))
    # per call: K and V rows read (bf16), codes and per-row scales written, slot mapping read twice
    nbytes = 2 * (n_tok * h_kv * hd * 3 + n_tok * h_kv * 4 + n_tok * 4)
    cfg = dict(workload="paged_kv_cache_write", tokens=n_tok, h_kv=h_kv, head_dim=hd, page=16,
               seqlens="uniform[1024,16384] seed 5, 32 sequences", scales="per row (amax/448)",
               tensors="K and V (2 launches per call)",
               l2="inputs 2 x %.0f MB bf16 > L2" % (n_tok * h_kv * hd * 2 / 1e6))
    return _leg_result("paged KV-cache write (quantise on write) us/call, a call = the K and V writes of "
                       "32 sequences", avg, ms, nbytes, 0.0, 0.0, peaks, cfg, 2)


def run_leg(name, dev, peaks, steps, warmup):
    from paged_decode_attention_fp8_gb300 import synthetic as syn
    if name == "mla_bf16":
        return leg_mla(dev, peaks, steps, warmup, "bf16", syn.uniform_seqlens(2, 64, 2048, 6144), 2,
                       "uniform[2048,6144] seed 2")
    if name == "mla_fixed4096":
        return leg_mla(dev, peaks, steps, warmup, "fp8", [4096] * 64, 12, "fixed 4096")
    if name.startswith("mla_long_b"):
        b = int(name[len("mla_long_b"):])
        return leg_mla(dev, peaks, steps, warmup, "fp8", [8196] * b, 3, "fixed 8196", value_pages=512)
    if name.startswith("sparse_sq"):
        return leg_sparse(dev, peaks, steps, warmup, int(name[len("sparse_sq"):]))
    if name == "gqa_bs32":
        return leg_gqa(dev, peaks, steps, warmup)
    if name == "gqa_bs32_rows":
        return leg_gqa(dev, peaks, steps, warmup, "rows")
    if name == "gqa_bs32_xqa":
        return leg_gqa(dev, peaks, steps, warmup, "xqa")
    if name == "mla_rows":
        return leg_mla(dev, peaks, steps, warmup, "fp8", syn.uniform_seqlens(2, 64, 2048, 6144), 2,
                       "uniform[2048,6144] seed 2", value_pages=96, rows=True)
    if name == "kvwrite":
        return leg_kvwrite(dev, peaks, steps, warmup)
    raise ValueError(name)


LEGS = ("mla_bf16", "mla_fixed4096", "mla_long_b32", "mla_long_b48", "mla_long_b64", "mla_long_b128", "mla_rows",
        "sparse_sq2", "sparse_sq16", "sparse_sq16384", "gqa_bs32", "gqa_bs32_rows", "gqa_bs32_xqa", "kvwrite")


def run_legs(dev, steps, warmup, names=LEGS):
    import gc

    import torch
    peaks = measured_peaks()
    legs = {}
    for name in names:
        leg_steps = min(steps, 30) if name == "sparse_sq16384" else steps
        legs[name] = run_leg(name, dev, peaks, leg_steps, warmup)
        gc.collect()
        torch.cuda.empty_cache()
    return legs


def run_secondary(args):
    """One leg as its own JSON line (``--workload``)."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    names = {"sparse": f"sparse_sq{args.sq}", "gqa": "gqa_bs32", "gqa_rows": "gqa_bs32_rows",
             "gqa_xqa": "gqa_bs32_xqa", "kvwrite": "kvwrite", "mla_bf16": "mla_bf16",
             "mla_fixed4096": "mla_fixed4096", "mla_long": f"mla_long_b{args.b}", "mla_rows": "mla_rows"}
    res = run_leg(names[args.workload], dev, measured_peaks(), args.steps, args.warmup)
    res.update(steps=args.steps, warmup=args.warmup, n_gpus=1, data="synthetic")
    print(json.dumps(res), flush=True)


# ------------------------------------------------------ oracle baseline ----


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(inp, seqlens, budget_s=15.0):
    """The fp64 oracle as it stands, timed on a bounded sample of the batch's sequences."""
    import oracle
    w = WORKLOAD
    done, t_used, flops = [], 0.0, 0.0
    order = list(range(w["b"]))
    t_start = time.perf_counter()
    for bi in order:
        t0 = time.perf_counter()
        oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens, inp.kv_scale, inp.softmax_scale,
                          True, batches=[bi])
        t_used += time.perf_counter() - t0
        done.append(bi)
        flops += mla_flops([seqlens[bi]], w["s_q"], w["h_q"])
        if time.perf_counter() - t_start > budget_s:
            break
    tflops = flops / t_used / 1e12
    full_ms = mla_flops(seqlens, w["s_q"], w["h_q"]) / (tflops * 1e12) * 1e3
    return dict(value=round(tflops, 6), unit="TFLOPS", cores=cpu_cores(), kind="oracle",
                sample=f"{len(done)} of {w['b']} sequences ({t_used:.1f} s); full batch ~{full_ms:.0f} ms/call",
                threads_note="numpy fp64 (BLAS matmul may use up to `cores` threads)")


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from paged_decode_attention_fp8_gb300 import synthetic as syn
    import oracle
    w = WORKLOAD
    seqlens = syn.uniform_seqlens(2, w["b"], 2048, 6144)
    inp = syn.mla_inputs(2, w["b"], w["s_q"], w["h_q"], seqlens, causal=True, spare_pages=64)
    per_step = max(1, int(args.ref_seqs))

    def step(i):
        picks = [(i * per_step + k) % w["b"] for k in range(per_step)]
        oracle.mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.seqlens, inp.kv_scale, inp.softmax_scale,
                          True, batches=picks)
        return mla_flops([seqlens[p] for p in picks], w["s_q"], w["h_q"])

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    flops = 0.0
    for i in range(args.steps):
        flops += step(args.warmup + i)
    dt = time.perf_counter() - t0
    tflops = flops / dt / 1e12
    ms_per_step = dt / args.steps * 1e3
    res = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(tflops, 6),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) Q/KV, E4M3 per-tensor scale)",
        "config": dict(WORKLOAD, dot="exact fp64", sample=f"{per_step} of {w['b']} sequences per step"),
        "cpu_baseline": dict(value=round(tflops, 6), unit="TFLOPS", cores=cpu_cores(), kind="oracle",
                             sample=f"{per_step} of {w['b']} sequences per step, {args.steps} steps"),
        "e2e": dict(value=round(tflops, 6), unit="TFLOPS", h2d_bytes_per_step=0, d2h_bytes_per_step=0),
    }
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--dot", choices=["fp8", "bf16"], default="fp8")
    ap.add_argument("--workload", choices=["mla", "sparse", "gqa", "gqa_rows", "gqa_xqa", "kvwrite", "mla_bf16",
                                           "mla_fixed4096", "mla_long", "mla_rows"],
                    default="mla", help="mla = the headline line (which also carries every leg under 'legs'); "
                    "the others print one measurement leg alone")
    ap.add_argument("--sq", type=int, default=2,
                    help="query tokens of the sparse leg (2 or 16 for decode, 16384 for the prefill-sized batch)")
    ap.add_argument("--b", type=int, default=64, help="batch of the mla_long leg (32, 48, 64 or 128)")
    ap.add_argument("--no-legs", action="store_true", help="headline only (skip the other rows' legs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (short runs under a profiler)")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-seqs", type=int, default=2, help="sequences of the batch per reference step")
    args = ap.parse_args()
    if args.impl == "reference":
        args.steps = 5 if args.steps is None else args.steps
        args.warmup = 1 if args.warmup is None else args.warmup
        run_reference(args)
        return
    args.steps = 20000 if args.steps is None else args.steps
    args.warmup = 50 if args.warmup is None else max(args.warmup, 3)
    if args.workload != "mla":
        args.steps = min(args.steps, 2000)
        run_secondary(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
