"""Benchmark: paged-attention decode, µs per call and achieved KV-read HBM GB/s.

Workload (one "step"): the decode step of the hybrid model's 16 full-attention
layers -- per layer, reshape_and_cache of the new token's K/V, then split-KV
paged-attention decode: batch 1, 24 query / 4 KV heads, head_dim 256, bf16
N(0,1) data, context 32768, 784-token pages scattered at random through a
pool 1.1x the context.  Every layer has its own 128 MiB cache (2 GiB per
step, far larger than the 129 MB L2), so no L2 flush is needed between steps.
Each layer is one pa_paged_attention_decode_append call, which does both in
one kernel (the same result as the two calls; `step_two_calls_ms` times the
step as two calls per layer).  The calls carry PA_FLAG_EARLY_KV_READ (the
step satisfies its contract: only the new row is written ahead of each
decode), which streams the old context ahead of each call's stream
dependency and leaves the outputs bit-identical.

`value` is whole-job KV-read GB/s (algorithmic bytes: 4096 B per context token
per layer) with all inputs resident in HBM; the step runs as a CUDA graph and
is timed with CUDA events on the launching stream.  `e2e` is the same metric
through the Python binding with the step's inputs copied from pinned host
memory and its outputs copied back inside the timed region.  `roofline`
covers the decode kernel (split kernel + reduce launch per layer call), timed
with CUDA events on the same stream over replays of a graph holding the 16
layers' decode calls alone (no events inside the graphs, which would break
the launch overlap between kernels).

After the headline line's measurements, the other workloads of the pages are
timed as graph replays of attention calls with PA_FLAG_EARLY_KV_READ set (the
graphs hold nothing that writes the caches) (`workloads`): the 512-token case (L2-warm and
L2-flushed), the 11-depth context sweep for the hybrid and dense shapes with a
fitted per-token slope and a flatness check, batch-32 decode, verify, a
chunked-prefill step, sliding-window decode, 12-heads-per-KV-head decode and
verify, and decode over an fp8 e4m3 cache.

`--impl reference` times the CPU fp64 oracle on the host cores instead (a
bounded sample of the same workload) and prints the same line shape.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "hybrid_step_l32768_bs784_x16"
METRIC = "paged-attn decode µs/call & achieved KV-read HBM GB/s vs context length"
KV_BYTES_PER_TOKEN_LAYER = 4096  # 2 (K, V) x 4 KV heads x 256 dims x 2 bytes
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e datasheet rate (secondary denominator)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_digest() -> str:
    """Digest of the decode kernel's source (the headline instantiation's code,
    not the launch table of the other shapes)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_attention_decode_split_gb300", "csrc")
    for name in ("pa_device.cuh", "decode_split.cuh", "decode_mma.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic():
    """DRAM bytes per decode call from the committed ncu summary, if it was
    taken on the current decode kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "decode_l32768_bs784_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_source_digest") != kernel_source_digest():
        return None
    return rec.get("dram_bytes_per_call")


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.result = None
        if self.proc is None:
            return False
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return False
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        loaded = [v for v in sm if smax and v > 0.5 * max(smax)] or sm
        self.result = {"sm_mhz": statistics.median(loaded) if loaded else None,
                       "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows)}
        return False


def dist_setup(n_gpus):
    """One process per GPU under torchrun (NCCL); replicas exchange only the
    barrier and the max of their timings.  Without a GPU (host-side tests of
    this logic) the group runs on gloo."""
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def _device_sync():
    import torch
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def barrier(world):
    import torch.distributed as dist
    if world > 1:
        dist.barrier()
    _device_sync()


def max_over_ranks(world, value: float) -> float:
    import torch
    import torch.distributed as dist
    if world == 1:
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, bytes_per_rank_step: int, ms_per_step: float) -> float:
    """Whole-job throughput: the bytes every replica processed in one step over
    the slowest replica's step time (weak scaling: fixed work per GPU)."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------------------------

def _bits(t):
    """bf16 tensor -> uint16 numpy bit patterns on the host (the oracle's input form)."""
    import numpy as np
    import torch
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def run_oracle_sample(layers, block_table, seq_lens, scale, budget_s: float):
    """Times the oracle over whole layers of the workload until about budget_s
    seconds of CPU work; returns (seconds, layers, threads)."""
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    done, t_total = 0, 0.0
    layers = list(layers)
    while True:  # whole passes over the layers until the budget is used
        for q, kc, vc in layers:
            t0 = time.perf_counter()
            oracle.paged_attention(q, kc, vc, block_table, seq_lens, scale, num_threads=threads)
            t_total += time.perf_counter() - t0
            done += 1
            if t_total >= budget_s:
                return t_total, done, threads


def bench_reference(args, world, rank):
    """The oracle as the reference arm: the same 16-layer step as our arm (one
    oracle call per layer over that layer's cache), timed step by step on the
    host cores within a time budget."""
    import torch
    from paged_attention_decode_split_gb300.inputs import WORKLOADS, make_problem
    if rank != 0:
        return
    spec = dict(WORKLOADS[WORKLOAD])
    spec["num_layers"] = args.layers
    prob = make_problem(1002, **spec)
    layers = [(_bits(prob.q[l]), _bits(prob.k_cache[l]), _bits(prob.v_cache[l])) for l in range(prob.num_layers)]
    bt, sl = prob.block_table.numpy(), prob.seq_lens.numpy()
    L = int(prob.seq_lens[0])
    bytes_step = prob.num_layers * L * KV_BYTES_PER_TOKEN_LAYER
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    times = []
    t_start = time.perf_counter()
    warm = max(3, args.warmup)
    for i in range(warm + args.steps):
        t0 = time.perf_counter()
        for q, kc, vc in layers:
            oracle.paged_attention(q, kc, vc, bt, sl, prob.scale, num_threads=threads)
        dt = time.perf_counter() - t0
        if i >= warm:
            times.append(dt)
        if time.perf_counter() - t_start > args.reference_budget and times:
            break  # keep the reference arm within a few minutes
    per_step = sum(times) / len(times)
    gbs = bytes_step / per_step / 1e9
    sample = (f"{len(times)} timed steps of all {prob.num_layers} layers (batch 1, 24 heads, context {L}, "
              f"block 784), fp64 oracle on {threads} host threads, after {warm} warm-up steps")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": len(times), "steps_requested": args.steps, "warmup": warm, "ms_per_step": per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers": prob.num_layers, "batch": 1, "context": L, "block_size": 784,
                   "q_heads": 24, "kv_heads": 4, "head_dim": 256},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def bench_gpu(args, world, rank, local):
    import torch
    import paged_attention_decode_split_gb300 as pa
    from paged_attention_decode_split_gb300 import _build
    from paged_attention_decode_split_gb300.inputs import WORKLOADS, make_new_tokens, make_problem

    _build.build()
    pa.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    spec = dict(WORKLOADS[WORKLOAD])
    spec["num_layers"] = args.layers
    prob = make_problem(1002 + rank, **spec, device="cuda")
    n_layers = prob.num_layers
    L = int(prob.seq_lens[0])
    B = prob.num_seqs
    bt = prob.block_table.to(dev)
    sl = prob.seq_lens.to(dev)
    # The step is reshape_and_cache then decode per layer, so nothing still
    # running writes the block table, seq_lens or the cached rows before the
    # new one: the calls may stream the old context ahead of their stream
    # dependency (PA_FLAG_EARLY_KV_READ; outputs are bit-identical either way).
    desc = pa.make_desc(num_seqs=B, num_q_heads=24, num_kv_heads=4, head_dim=256, block_size=prob.block_size,
                        max_pages_per_seq=prob.max_pages_per_seq, max_seq_len=L, num_pages=prob.num_pages,
                        scale=prob.scale, flags=pa.PA_FLAG_EARLY_KV_READ)
    ws = torch.empty(max(1, pa.workspace_bytes(desc)), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    k_new, v_new = make_new_tokens(77 + rank, n_layers * B, 4, 256, device="cuda")
    k_new = k_new.view(n_layers, B, 4, 256)
    v_new = v_new.view(n_layers, B, 4, 256)
    slots = prob.new_token_slots().to(dev)
    out = torch.empty((n_layers, B, 24, 256), dtype=torch.float32, device=dev)

    def layer_call(l):
        # one call per layer: the new token's K/V appended (reshape_and_cache)
        # and the decode that reads it, fused in one kernel
        pa.paged_attention_decode_append(prob.q[l], k_new[l], v_new[l], prob.k_cache[l], prob.v_cache[l], bt, sl,
                                         desc, out[l], ws, status=status)

    def layer_two_calls(l):
        pa.reshape_and_cache(k_new[l], v_new[l], prob.k_cache[l], prob.v_cache[l], slots, status=status)
        pa.paged_attention_decode(prob.q[l], prob.k_cache[l], prob.v_cache[l], bt, sl, desc, out[l], ws,
                                  status=status)

    stream = torch.cuda.Stream(device=dev)
    # eager warm-up (sets kernel attributes, loads modules) outside any capture
    with torch.cuda.stream(stream):
        for l in range(n_layers):
            layer_call(l)
    torch.cuda.synchronize()
    plan = pa.last_plan()

    # The step graph: 16 x (fused append + decode split kernel, reduce).
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for l in range(n_layers):
            layer_call(l)
    # The same step as two calls per layer (reshape_and_cache, then decode).
    graph2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph2, stream=stream):
        for l in range(n_layers):
            layer_two_calls(l)
    # The decode calls alone (same launches, no reshape) for the kernel's roofline.
    dec_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(dec_graph, stream=stream):
        for l in range(n_layers):
            pa.paged_attention_decode(prob.q[l], prob.k_cache[l], prob.v_cache[l], bt, sl, desc, out[l], ws,
                                      status=status)
    torch.cuda.synchronize()
    launches_per_step = n_layers * (1 + (1 if plan["reduce_launched"] else 0))

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            graph.replay()
            graph2.replay()
            dec_graph.replay()
    barrier(world)

    step_events = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    dec_reps = max(20, args.steps // 4)
    dec_events = [torch.cuda.Event(enable_timing=True) for _ in range(dec_reps + 1)]
    with ClockSampler(local) as clocks:
        barrier(world)
        with torch.cuda.stream(stream):
            step_events[0].record()
            for k in range(args.steps):
                graph.replay()
                step_events[k + 1].record()
        torch.cuda.synchronize()
        barrier(world)
        # kernel timing region: the decode calls alone, events on the same stream
        with torch.cuda.stream(stream):
            dec_events[0].record()
            for k in range(dec_reps):
                dec_graph.replay()
                dec_events[k + 1].record()
        torch.cuda.synchronize()
        # the unfused step (reshape_and_cache and decode as two calls per layer)
        two_events = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        with torch.cuda.stream(stream):
            two_events[0].record()
            for k in range(dec_reps):
                graph2.replay()
            two_events[1].record()
        torch.cuda.synchronize()
        barrier(world)
    per_step_ms = [step_events[k].elapsed_time(step_events[k + 1]) for k in range(args.steps)]
    total_ms = step_events[0].elapsed_time(step_events[-1])
    total_ms = max_over_ranks(world, total_ms)
    ms_per_step = total_ms / args.steps
    call_us = [dec_events[k].elapsed_time(dec_events[k + 1]) * 1e3 / n_layers for k in range(dec_reps)]

    bytes_step = n_layers * B * L * KV_BYTES_PER_TOKEN_LAYER
    value = whole_job_gbs(world, bytes_step, ms_per_step)
    peak, peak_kind = load_peaks()
    avg_call_us = dec_events[0].elapsed_time(dec_events[-1]) * 1e3 / (dec_reps * n_layers)
    achieved = (B * L * KV_BYTES_PER_TOKEN_LAYER) / (avg_call_us * 1e-6) / 1e9
    st = int(status.item())

    # ---- end to end through the binding with host buffers ----
    # The step's inputs travel in one pinned host buffer and one copy (q, the
    # new K/V rows, their slots, seq_lens and the block table, each at a
    # 256-byte aligned offset); the outputs come back in one copy.
    srcs = [torch.stack([q for q in prob.q]), k_new, v_new, slots, prob.seq_lens, prob.block_table]
    offs, total = [], 0
    for t in srcs:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    in_host = torch.empty(total, dtype=torch.uint8).pin_memory()
    in_dev = torch.empty(total, dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(srcs, offs):
        n = t.numel() * t.element_size()
        in_host[o:o + n].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
        views.append(in_dev[o:o + n].view(t.dtype).view(t.shape))
    q_dev, kn_dev, vn_dev, slots_dev, sl_dev, bt_dev = views
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = total
    d2h = out_host.numel() * out_host.element_size()

    sh = stream.cuda_stream  # the handle the calls are issued on

    def e2e_step():
        in_dev.copy_(in_host, non_blocking=True)
        for l in range(n_layers):
            pa.paged_attention_decode_append(q_dev[l], kn_dev[l], vn_dev[l], prob.k_cache[l], prob.v_cache[l], bt_dev,
                                             sl_dev, desc, out[l], ws, status=status, stream=sh)
        out_host.copy_(out, non_blocking=True)

    e2e_steps = max(5, min(args.steps, 200))
    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
            torch.cuda.current_stream().synchronize()  # the result is on the host each step
        e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(world, e2e_s)
    e2e_value = world * bytes_step * e2e_steps / e2e_s / 1e9

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        layer_cpu = [(_bits(prob.q[l]), _bits(prob.k_cache[l]), _bits(prob.v_cache[l])) for l in range(n_layers)]
        secs, layers_done, threads = run_oracle_sample(layer_cpu, prob.block_table.numpy(),
                                                       prob.seq_lens.numpy(), prob.scale, args.cpu_budget)
        cpu = {"value": layers_done * B * L * KV_BYTES_PER_TOKEN_LAYER / secs / 1e9, "unit": "GB/s",
               "cores": threads, "kind": "oracle",
               "sample": f"{layers_done} layer calls (passes over the {n_layers} layers; all 24 heads, context {L}), "
                         f"fp64, {secs:.1f} s on {threads} host threads"}

    if rank != 0:
        return
    suite = None if args.no_suite else secondary_workloads(args, dev, stream, peak)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "accum_dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers": n_layers, "batch": B, "context": L, "block_size": prob.block_size,
                   "q_heads": 24, "kv_heads": 4, "head_dim": 256, "num_pages_per_layer": prob.num_pages,
                   "l2": "no flush: 16 distinct 128 MiB layer caches (2 GiB per step) exceed the 129 MB L2",
                   "parallelism": f"replicas x{world}", "plan": plan, "flags": "PA_FLAG_EARLY_KV_READ",
                   "step": "per layer one pa_paged_attention_decode_append: the new token's K/V written into its "
                           "slot (reshape_and_cache) and the split-KV decode, in one kernel, plus the reduce"},
        "us_per_call": ms_per_step * 1e3 / n_layers,
        "us_per_context_token": ms_per_step * 1e3 / L,
        "ms_per_step_range": [min(per_step_ms), statistics.median(per_step_ms), max(per_step_ms)],
        "decode_call_us": {"mean": avg_call_us, "min": min(call_us), "max": max(call_us),
                           "how": f"CUDA events around {dec_reps} replays of a graph of the {n_layers} layers' "
                                  "decode calls (split kernel + reduce), timed after the step region"},
        "step_two_calls_ms": {"mean": two_events[0].elapsed_time(two_events[1]) / dec_reps,
                              "how": "the same step with reshape_and_cache and decode as two calls per layer "
                                     f"(graph of {n_layers} x 3 launches), CUDA events around {dec_reps} replays"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} copy bandwidth", "traffic": load_traffic(),
                     "algorithmic_bytes_per_call": B * L * KV_BYTES_PER_TOKEN_LAYER,
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "nominal_peak": NOMINAL_HBM_GBS},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "the Python API (its compiled tensor binding checks every tensor), eager calls on an explicit stream; the step's inputs copied in from one pinned host buffer and its outputs copied out every step"},
        "gpu_launches": launches_per_step * args.steps,
        "device_status": st,
        "clocks": clocks.result,
        "cpu_baseline": cpu,
        "workloads": suite,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------
# The other workloads of the pages, timed after the headline step (rank 0).

def _time_graph(calls, stream, reps, warm=3):
    """Captures the callables into one CUDA graph; returns ms per replay."""
    import torch
    with torch.cuda.stream(stream):
        for c in calls:
            c()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in calls:
            c()
    with torch.cuda.stream(stream):
        for _ in range(warm):
            g.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


# The suite's graphs hold attention calls only, so nothing still running
# writes the block table, seq_lens or cached K/V ahead of a call: like the
# headline step they set PA_FLAG_EARLY_KV_READ (1).
SUITE_FLAGS = 1


def _attention_calls(pa, prob, dev):
    """One decode (or verify) call per layer of the problem, with its buffers."""
    import torch
    bt, sl = prob.block_table.to(dev), prob.seq_lens.to(dev)
    desc = pa.make_desc(num_seqs=prob.num_seqs, q_len=prob.q_len, num_q_heads=prob.num_q_heads,
                        num_kv_heads=prob.num_kv_heads, head_dim=prob.head_dim, block_size=prob.block_size,
                        max_pages_per_seq=prob.max_pages_per_seq, max_seq_len=prob.max_seq_len,
                        num_pages=prob.num_pages, scale=prob.scale, flags=SUITE_FLAGS)
    ws = torch.empty(max(1, pa.workspace_bytes(desc)), dtype=torch.uint8, device=dev)
    out = torch.empty((prob.num_seqs * prob.q_len, prob.num_q_heads, prob.head_dim), dtype=torch.float32,
                      device=dev)
    fn = pa.paged_attention_decode if prob.q_len == 1 else pa.paged_attention_verify
    calls = [(lambda l=l: fn(prob.q[l], prob.k_cache[l], prob.v_cache[l], bt, sl, desc, out, ws))
             for l in range(prob.num_layers)]
    return calls


def _layers_beyond_l2(bytes_per_layer, minimum, l2_bytes=256 << 20):
    return max(minimum, -(-l2_bytes // max(1, bytes_per_layer)))


SECONDARY = ("decode_l512_bs16", "context_sweep", "batch32_uniform_bs784", "verify_b8_q16_l8192_bs832",
             "prefill_q2048_l16384_bs832", "decode_window2048_l32768_bs784", "decode_g12_l32768_bs784",
             "verify_g12_b32_q5_l2048_bs784", "decode_fp8_l32768_bs784", "verify_fp8_b8_q16_l8192_bs832",
             "decode_dense_l32768_bs16")


def secondary_workloads(args, dev, stream, peak, names=SECONDARY):
    import torch
    import paged_attention_decode_split_gb300 as pa
    from paged_attention_decode_split_gb300.inputs import SWEEP_DEPTHS, WORKLOADS, make_problem, sweep_workload
    res = {}

    if "decode_l512_bs16" in names:
        _short_context(pa, torch, dev, stream, res, WORKLOADS, make_problem)
    if "context_sweep" in names:
        res["context_sweep"] = _context_sweep(pa, dev, stream, SWEEP_DEPTHS, make_problem, sweep_workload)
    if "batch32_uniform_bs784" in names:
        _batch32(pa, dev, stream, peak, res, WORKLOADS, make_problem)
    if "verify_b8_q16_l8192_bs832" in names:
        _verify(pa, dev, stream, peak, res, WORKLOADS, make_problem)
    if "prefill_q2048_l16384_bs832" in names:
        _prefill(pa, dev, stream, res, WORKLOADS, make_problem)
    if "decode_window2048_l32768_bs784" in names:
        _window(pa, dev, stream, peak, res, WORKLOADS, make_problem)
    if "decode_g12_l32768_bs784" in names:
        _wide_group(pa, dev, stream, peak, res, WORKLOADS, make_problem)
    if "decode_dense_l32768_bs16" in names:
        _dense(pa, dev, stream, peak, res, WORKLOADS, make_problem)
    if "decode_fp8_l32768_bs784" in names:
        _fp8_decode(pa, dev, stream, peak, res, WORKLOADS, make_problem)
    if "verify_fp8_b8_q16_l8192_bs832" in names:
        _verify_fp8(pa, dev, stream, peak, res, WORKLOADS, make_problem)
    if "verify_g12_b32_q5_l2048_bs784" in names:
        _verify(pa, dev, stream, peak, res, WORKLOADS, make_problem, name="verify_g12_b32_q5_l2048_bs784",
                layers=2)
    return res


def _fp8_decode(pa, dev, stream, peak, res, WORKLOADS, make_problem):
    # The 32K hybrid layer over an fp8 e4m3 cache: 2048 B of K+V per token
    # (half of bf16), 64 MiB per layer, 16 layers (1 GiB) cycled against L2.
    prob = make_problem(1009, **WORKLOADS["decode_fp8_l32768_bs784"], device=dev)
    bt, sl = prob.block_table.to(dev), prob.seq_lens.to(dev)
    desc = pa.make_desc(num_seqs=prob.num_seqs, num_q_heads=prob.num_q_heads, num_kv_heads=prob.num_kv_heads,
                        head_dim=prob.head_dim, block_size=prob.block_size, max_pages_per_seq=prob.max_pages_per_seq,
                        max_seq_len=prob.max_seq_len, num_pages=prob.num_pages, scale=prob.scale, flags=SUITE_FLAGS)
    import torch
    ws = torch.empty(max(1, pa.workspace_bytes(desc)), dtype=torch.uint8, device=dev)
    out = torch.empty((prob.num_seqs, prob.num_q_heads, prob.head_dim), dtype=torch.float32, device=dev)
    calls = [(lambda l=l: pa.paged_attention_decode_fp8(prob.q[l], prob.k_cache[l], prob.v_cache[l], prob.k_scale[l],
                                                        prob.v_scale[l], bt, sl, desc, out, ws))
             for l in range(prob.num_layers)]
    us = _time_graph(calls, stream, 100) * 1e3 / len(calls)
    kv = prob.context_tokens() * KV_BYTES_PER_TOKEN_LAYER // 2
    res["decode_fp8_l32768_bs784"] = {"us_per_call": us, "kv_bytes_per_call": kv, "GBps": kv / (us * 1e-6) / 1e9,
                                      "frac_of_peak": kv / (us * 1e-6) / 1e9 / peak, "plan": pa.last_plan()}
    del prob, calls


def _verify_fp8(pa, dev, stream, peak, res, WORKLOADS, make_problem):
    # The verify workload over an fp8 e4m3 cache: 8 x 8208 tokens x 2048 B =
    # 134 MiB of codes per call; 4 layer copies cycled against L2.
    import torch
    prob = make_problem(1010, **dict(WORKLOADS["verify_b8_q16_l8192_bs832"], num_layers=4, kv_fp8=True), device=dev)
    bt, sl = prob.block_table.to(dev), prob.seq_lens.to(dev)
    desc = pa.make_desc(num_seqs=prob.num_seqs, q_len=prob.q_len, num_q_heads=prob.num_q_heads,
                        num_kv_heads=prob.num_kv_heads, head_dim=prob.head_dim, block_size=prob.block_size,
                        max_pages_per_seq=prob.max_pages_per_seq, max_seq_len=prob.max_seq_len,
                        num_pages=prob.num_pages, scale=prob.scale, flags=SUITE_FLAGS)
    ws = torch.empty(max(1, pa.workspace_bytes(desc)), dtype=torch.uint8, device=dev)
    out = torch.empty((prob.num_seqs * prob.q_len, prob.num_q_heads, prob.head_dim), dtype=torch.float32, device=dev)
    calls = [(lambda l=l: pa.paged_attention_verify_fp8(prob.q[l], prob.k_cache[l], prob.v_cache[l], prob.k_scale[l],
                                                        prob.v_scale[l], bt, sl, desc, out, ws))
             for l in range(prob.num_layers)]
    us = _time_graph(calls, stream, 100) * 1e3 / len(calls)
    kv = prob.context_tokens() * KV_BYTES_PER_TOKEN_LAYER // 2
    res["verify_fp8_b8_q16_l8192_bs832"] = {"us_per_call": us, "kv_bytes_per_call": kv, "GBps": kv / (us * 1e-6) / 1e9,
                                            "frac_of_peak": kv / (us * 1e-6) / 1e9 / peak,
                                            "TFLOPs": _causal_flops(prob) / (us * 1e-6) / 1e12, "plan": pa.last_plan()}
    del prob, calls


def _wide_group(pa, dev, stream, peak, res, WORKLOADS, make_problem):
    # 12 query heads per KV head at 32K: the same 128 MiB of K+V per layer as
    # the hybrid step with twice the arithmetic per byte; 16 layers (2 GiB).
    prob = make_problem(1008, **WORKLOADS["decode_g12_l32768_bs784"], device=dev)
    calls = _attention_calls(pa, prob, dev)
    us = _time_graph(calls, stream, 50) * 1e3 / len(calls)
    kv = prob.context_tokens() * KV_BYTES_PER_TOKEN_LAYER
    res["decode_g12_l32768_bs784"] = {"us_per_call": us, "GBps": kv / (us * 1e-6) / 1e9,
                                      "frac_of_peak": kv / (us * 1e-6) / 1e9 / peak, "plan": pa.last_plan()}
    del prob, calls


def _dense(pa, dev, stream, peak, res, WORKLOADS, make_problem):
    # The dense control at 32K: 32 query heads on 8 KV heads of 128 dims,
    # 16-token pages; 128 MiB of K+V per layer, 16 layers (2 GiB).
    prob = make_problem(1011, **WORKLOADS["decode_dense_l32768_bs16"], device=dev)
    calls = _attention_calls(pa, prob, dev)
    us = _time_graph(calls, stream, 50) * 1e3 / len(calls)
    kv = prob.context_tokens() * KV_BYTES_PER_TOKEN_LAYER
    res["decode_dense_l32768_bs16"] = {"us_per_call": us, "GBps": kv / (us * 1e-6) / 1e9,
                                       "frac_of_peak": kv / (us * 1e-6) / 1e9 / peak, "plan": pa.last_plan()}
    del prob, calls


def _short_context(pa, torch, dev, stream, res, WORKLOADS, make_problem):
    # 512-token decode on 16-token pages: 2 MiB of KV, launch-bound.  Timed with
    # the caches L2-resident, and again after writing a 256 MiB buffer each call.
    prob = make_problem(1001, **dict(WORKLOADS["decode_l512_bs16"], num_layers=16), device=dev)
    calls = _attention_calls(pa, prob, dev)
    warm_us = _time_graph(calls, stream, 200) * 1e3 / len(calls)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * 50)]
    with torch.cuda.stream(stream):
        for k in range(50):
            flush.fill_(k & 0xff)
            ev[2 * k].record()
            calls[k % len(calls)]()
            ev[2 * k + 1].record()
    torch.cuda.synchronize()
    flushed = sorted(ev[2 * k].elapsed_time(ev[2 * k + 1]) * 1e3 for k in range(50))
    kv = 512 * KV_BYTES_PER_TOKEN_LAYER
    res["decode_l512_bs16"] = {"us_per_call_l2_warm": warm_us, "us_per_call_l2_flushed_median": flushed[25],
                               "GBps_l2_flushed": kv / (flushed[25] * 1e-6) / 1e9, "plan": pa.last_plan()}
    del prob, calls, flush


def _context_sweep(pa, dev, stream, SWEEP_DEPTHS, make_problem, sweep_workload):
    # Context sweep: a 16-layer step at 11 depths, hybrid (832-token pages) and
    # dense control (32Q/8KV, head_dim 128, 16-token pages).  Enough distinct
    # layer copies are cycled to keep the caches out of L2.
    sweep = {}
    for dense in (False, True):
        rows = []
        for depth in SWEEP_DEPTHS:
            n = _layers_beyond_l2(depth * KV_BYTES_PER_TOKEN_LAYER, 16)
            prob = make_problem(1003 + depth + dense, **sweep_workload(depth, dense, num_layers=n), device=dev)
            calls = _attention_calls(pa, prob, dev)
            us = _time_graph(calls, stream, max(10, 3200 // n)) * 1e3 / n
            rows.append({"depth": depth, "us_per_call": us, "us_per_step_16": 16 * us,
                         "GBps": depth * KV_BYTES_PER_TOKEN_LAYER / (us * 1e-6) / 1e9,
                         "splits": pa.last_plan()["num_splits"]})
            del prob, calls
        xs = [r["depth"] for r in rows]
        ys = [r["us_per_step_16"] for r in rows]
        mx, my = sum(xs) / len(xs), sum(ys) / len(ys)
        slope = sum((x - mx) * (y - my) for x, y in zip(xs, ys)) / sum((x - mx) ** 2 for x in xs)
        icpt = my - slope * mx
        dev_pct = [100.0 * ((y - icpt) / x / slope - 1.0) for x, y in zip(xs, ys) if x >= 4096]
        sweep["dense_control" if dense else "hybrid"] = {
            "rows": rows, "fit_us_per_context_token_16_layers": slope, "fit_intercept_us": icpt,
            "max_abs_deviation_pct_depth_ge_4k": max(abs(d) for d in dev_pct),
            "flat_within_15pct": all(abs(d) <= 15.0 for d in dev_pct)}
    return sweep


def _batch32(pa, dev, stream, peak, res, WORKLOADS, make_problem):
    # Batched decode: 32 sequences, lengths uniform in [1024, 32768].
    prob = make_problem(1004, **dict(WORKLOADS["batch32_uniform_bs784"], num_layers=2), device=dev)
    calls = _attention_calls(pa, prob, dev)
    us = _time_graph(calls, stream, 50) * 1e3 / len(calls)
    kv = prob.context_tokens() * KV_BYTES_PER_TOKEN_LAYER
    res["batch32_uniform_bs784"] = {"us_per_call": us, "context_tokens": prob.context_tokens(),
                                    "GBps": kv / (us * 1e-6) / 1e9, "frac_of_peak": kv / (us * 1e-6) / 1e9 / peak,
                                    "plan": pa.last_plan()}


def _verify(pa, dev, stream, peak, res, WORKLOADS, make_problem, name="verify_b8_q16_l8192_bs832", layers=4):
    # Speculative verify: 8 sequences x 16 new rows over 8192 prior tokens
    # (256 MiB of K+V), or 32 sequences x 5 rows x 12 heads per KV head over
    # 2048 positions (256 MiB); 4 or 2 layer copies cycled against L2.
    prob = make_problem(1005, **dict(WORKLOADS[name], num_layers=layers), device=dev)
    calls = _attention_calls(pa, prob, dev)
    us = _time_graph(calls, stream, 100) * 1e3 / len(calls)
    kv = prob.context_tokens() * KV_BYTES_PER_TOKEN_LAYER
    flops = _causal_flops(prob)
    res[name] = {"us_per_call": us, "GBps": kv / (us * 1e-6) / 1e9,
                                        "frac_of_peak": kv / (us * 1e-6) / 1e9 / peak,
                                        "TFLOPs": flops / (us * 1e-6) / 1e12, "plan": pa.last_plan()}


def _window(pa, dev, stream, peak, res, WORKLOADS, make_problem):
    # Sliding-window decode: the 32K hybrid layer with a 2048-key window, so
    # a call reads 2048 x 4096 B = 8 MiB of K+V.  32 distinct layer copies
    # (256 MiB) keep the reads out of L2.
    import torch
    spec = dict(WORKLOADS["hybrid_step_l32768_bs784_x16"], num_layers=32)
    prob = make_problem(1007, **spec, device=dev)
    bt, sl = prob.block_table.to(dev), prob.seq_lens.to(dev)
    desc = pa.make_desc(num_seqs=1, num_q_heads=24, num_kv_heads=4, head_dim=256, block_size=784,
                        max_pages_per_seq=prob.max_pages_per_seq, max_seq_len=32768, num_pages=prob.num_pages,
                        scale=1 / 16, window=2048, flags=SUITE_FLAGS)
    ws = torch.empty(max(1, pa.workspace_bytes(desc)), dtype=torch.uint8, device=dev)
    out = torch.empty((1, 24, 256), dtype=torch.float32, device=dev)
    calls = [(lambda l=l: pa.paged_attention_decode(prob.q[l], prob.k_cache[l], prob.v_cache[l], bt, sl, desc,
                                                     out, ws)) for l in range(prob.num_layers)]
    us = _time_graph(calls, stream, 50) * 1e3 / len(calls)
    kv = 2048 * KV_BYTES_PER_TOKEN_LAYER
    res["decode_window2048_l32768_bs784"] = {"us_per_call": us, "GBps": kv / (us * 1e-6) / 1e9,
                                             "frac_of_peak": kv / (us * 1e-6) / 1e9 / peak,
                                             "plan": pa.last_plan()}
    del prob, calls


def _causal_flops(prob):
    """Useful flops of a q_len-row call: 4 D per (row, head, visible key)."""
    total = 0
    for L in prob.seq_lens.tolist():
        q = prob.q_len
        total += prob.num_q_heads * 4 * prob.head_dim * (q * (int(L) - q) + q * (q + 1) // 2)
    return total


def _prefill(pa, dev, stream, res, WORKLOADS, make_problem):
    # Chunked-prefill step: 2048 new rows of one sequence (L = 16384) on the
    # tensor cores, 96 row blocks per KV head, each reading only the keys its
    # rows can see.  Compute-bound: reported against the bf16 tensor peak.
    prob = make_problem(1006, **dict(WORKLOADS["prefill_q2048_l16384_bs832"], num_layers=2), device=dev)
    calls = _attention_calls(pa, prob, dev)
    us = _time_graph(calls, stream, 20) * 1e3 / len(calls)
    flops = _causal_flops(prob)
    tf_peak = load_tensor_peak()
    res["prefill_q2048_l16384_bs832"] = {
        "us_per_call": us, "TFLOPs": flops / (us * 1e-6) / 1e12, "useful_flops": flops,
        "bf16_peak_TFLOPs": tf_peak, "frac_of_bf16_peak": flops / (us * 1e-6) / 1e12 / tf_peak,
        "note": "useful flops (4 D per row, head and visible key); the kernel also runs the P residual MMA "
                "and pads each 128-row block's causal edge", "plan": pa.last_plan()}


def load_tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def only_workload(args):
    """Times one secondary workload on cuda:0 (used for small profiling runs)."""
    import torch
    import paged_attention_decode_split_gb300 as pa
    from paged_attention_decode_split_gb300 import _build
    _build.build()
    pa.load_library()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    peak, _ = load_peaks()
    res = secondary_workloads(args, dev, stream, peak, names=(args.only,))
    print(json.dumps({"workloads": res}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=16,
                    help="layers per step (16 = the workload; fewer only for small profiling runs)")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-suite", action="store_true", help="skip the other workloads (sweep, batch 32, verify)")
    ap.add_argument("--reference-budget", type=float, default=60.0,
                    help="wall seconds after which --impl reference stops taking steps")
    ap.add_argument("--only", choices=SECONDARY, default=None,
                    help="time one of the other workloads alone and print its record (no headline line)")
    args = ap.parse_args()
    import torch  # noqa: F401
    if args.only is not None:
        only_workload(args)
        return
    world, rank, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            bench_reference(args, world, rank)
        else:
            bench_gpu(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
