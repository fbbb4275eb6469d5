"""Benchmark: Flash-LoRA-Attention decode queries/s and achieved HBM bandwidth on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--legs all|none]

Headline workload (one GPU): the Llama-3-8B-shaped single-layer decode -
3 agents, 32 query / 8 kv heads, head_dim 128, r 16, shared context 16384
tokens, one query token per agent, bf16 storage, fp32 accumulation.
One step = one flash_lora_attn_decode call (scores, online softmax, P.V_base,
P.L_i in the decode kernel; split merge and the B_i epilogue in the merge
kernel behind it).

Timing: W warm-up steps, then K steps replayed from a CUDA graph between a
barrier + synchronize on both sides, timed with CUDA events on the launching
stream, right after 0.25 s of untimed replays (load clocks).  The step inputs
rotate over enough copies of the cache (> 4x the 126 MB L2) that no step finds
its K/V/L tiles in L2.  `e2e` re-times K steps through the C-ABI call with host
buffers (flash_lora_attn_decode_host_io): each step copies the queries from
pinned host memory to the device, decodes, and copies O back to pinned host
memory.  The other legs time each remaining hot-path row alone, plus the
naive-materialisation and non-shared-cache baselines on the headline workload.

Under torchrun each rank runs its own independent copy of the workload
(weak scaling, no collective on the data path); value = all ranks' queries
divided by the slowest rank's time.

`--impl reference` times the CPU oracle (fp64, numpy) on this host on a
bounded sample of the same workload; it is a baseline, not a target.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LoRA-attn decode queries/s + achieved HBM GB/s (fraction of B300 peak)"
HEADLINE = "llama8b_decode"
L2_BYTES = 126 * 1024 * 1024


# ----------------------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return dict(hbm_gbs=float(pk["hbm_gbs"]), bf16_tflops=float(pk["bf16_tflops"]),
                    bf16_tflops_sustained=float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                    source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


# Sources the headline decode kernels (decode_tc_kernel and its merge kernels)
# are compiled from: their own header and the helpers it includes.
HEADLINE_KERNEL_SOURCES = ("decode_tc.cuh", "ptx.cuh", "fla_common.cuh")


def kernel_source_hash(files=HEADLINE_KERNEL_SOURCES) -> str:
    """Hash of the headline kernels' CUDA sources; a stored ncu traffic figure
    is used only while it matches (an edit to another kernel leaves it valid)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_flash_lora_attn_b300", "csrc")
    for fn in sorted(files):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def stored_traffic(workload: str):
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t.get(workload)
        if e and e.get("source_hash") == kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() in ("active", "1"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, world_size: int, device=None) -> float:
    if world_size == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world_size: int):
    if world_size > 1:
        import torch.distributed as dist

        dist.barrier()


PREROLL_S = 0.25
REPLAYS = 21      # timed replays of the headline's K-step graph (median reported)
E2E_ROUNDS = 5    # timed rounds of the host-buffer loop (median reported)


def preroll(fn, stream, seconds=PREROLL_S):
    """Untimed repetitions of a timed region's own work for `seconds`, ending
    right before it: the timed steps then start on a GPU running at its load
    clocks instead of after an idle gap (the clock sampler's start-up leaves
    the GPU idle), and the sampler's readings fall in this busy window."""
    import torch

    t_end = time.perf_counter() + seconds
    n = 0
    while n < 3 or time.perf_counter() < t_end:
        with torch.cuda.stream(stream):
            fn()
        stream.synchronize()
        n += 1
    return n


# ----------------------------------------------------------------------------- workload bytes / flops

def decode_algorithmic_bytes(w) -> int:
    """K_base + V_base + every agent's L + B + Q + O for one decode call (the expanded L_i.B_i is not counted)."""
    N = w.total_tokens
    kv = 2 * N * w.hkv * w.head_dim * 2
    lr = N * w.n_agents * w.rank * 2
    b = w.n_agents * w.rank * w.hkv * w.head_dim * 2
    q = w.n_req * w.n_agents * w.hq * w.head_dim * 2
    o = w.n_req * w.n_agents * w.hq * w.head_dim * 4
    return kv + lr + b + q + o


def decode_algorithmic_flops(w) -> int:
    A, hq, d, r = w.n_agents, w.hq, w.head_dim, w.rank
    return A * hq * w.total_tokens * (4 * d + 2 * r) + w.n_req * A * hq * 2 * r * d


# ----------------------------------------------------------------------------- our arm

def build_decode_copies(w, n_copies, device, seed=0):
    """n_copies independent seeded decode inputs on the device (drawn there: fast, large)."""
    import torch

    g = torch.Generator(device=device).manual_seed(seed)
    A, hq, hkv, d, r, N = w.n_agents, w.hq, w.hkv, w.head_dim, w.rank, w.total_tokens
    copies = []
    for _ in range(n_copies):
        c = dict(
            Q=torch.randn((w.n_req, A, hq, d), generator=g, device=device).to(torch.bfloat16),
            K_base=torch.randn((N, hkv, d), generator=g, device=device).to(torch.bfloat16),
            V_base=torch.randn((N, hkv, d), generator=g, device=device).to(torch.bfloat16),
            L=torch.randn((N, A * r), generator=g, device=device).to(torch.bfloat16),
            B=(0.02 * torch.randn((A, r, hkv * d), generator=g, device=device)).to(torch.bfloat16),
        )
        import numpy as np

        c["offsets"] = torch.tensor([0] + list(np.cumsum(w.lengths)), dtype=torch.int32, device=device)
        c["O"] = torch.empty((w.n_req, A, hq, d), dtype=torch.float32, device=device)
        copies.append(c)
    return copies


def time_graph(fn_list, steps, warmup, stream):
    """Capture `steps` calls (cycling fn_list) into one CUDA graph; return seconds per step."""
    import torch

    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            fn_list[i % len(fn_list)]()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(steps):
            fn_list[i % len(fn_list)]()
    # one untimed replay (warm the graph), then the timed one
    with torch.cuda.stream(stream):
        graph.replay()
    stream.synchronize()
    return graph


def run_ours(args, ws, rank, local):
    import torch

    import attention_flash_lora_attn_b300 as fla
    from attention_flash_lora_attn_b300 import build_lib
    from workloads import WORKLOADS

    build_lib.build()
    fla.load_library()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w = WORKLOADS[HEADLINE]
    per_copy = decode_algorithmic_bytes(w)
    n_copies = max(4, -(-4 * L2_BYTES // per_copy))  # rotating set > 4x L2
    copies = build_decode_copies(w, n_copies, device, seed=1000 + rank)
    stream = torch.cuda.Stream(device)
    workspace = torch.zeros(
        fla.load_library().flash_lora_attn_decode_workspace_size(
            __import__("ctypes").byref(fla.binding.make_dims(w.n_agents, w.hq, w.hkv, w.head_dim, w.rank, 1,
                                                             w.n_agents * w.rank, w.rank)),
            w.n_req, w.total_tokens) + 256, dtype=torch.uint8, device=device)

    def make_call(c):
        def call():
            fla.flash_lora_attn_decode(c["Q"], c["K_base"], c["V_base"], c["L"], c["B"], c["offsets"],
                                       rank=w.rank, O=c["O"], workspace=workspace, kernel="tensor")
        return call

    calls = [make_call(c) for c in copies]
    graph = time_graph(calls, args.steps, args.warmup, stream)

    # ---- timed regions: REPLAYS replays of the K-step graph, each bracketed by
    #      a barrier + synchronize and timed with CUDA events on the launching
    #      stream; the line reports the median (and the min-max spread)
    times = []
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk, torch.cuda.stream(stream):
        preroll(graph.replay, stream)
        for _ in range(REPLAYS):
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier(ws)
            torch.cuda.synchronize()
            # replay() launches on the current stream, which is `stream` here
            start.record(stream)
            graph.replay()
            end.record(stream)
            torch.cuda.synchronize()
            times.append(start.elapsed_time(end) / 1e3)
    barrier(ws)
    t_local = statistics.median(times)
    t = max_over_ranks(t_local, ws, device)
    queries_per_step = w.n_req * w.n_agents
    value = ws * queries_per_step * args.steps / t
    ms_per_step = t / args.steps * 1e3
    assert fla.device_error() == 0

    # ---- e2e: the C-ABI call with host buffers, every step: the step's queries
    #      from pinned host memory to the device, the decode, and its output back
    #      to pinned host memory, all enqueued by one flash_lora_attn_decode_host_io
    #      call (one prepared call per resident cache).
    Qh = [c["Q"].cpu().pin_memory() for c in copies]
    Oh = torch.empty(copies[0]["O"].shape, dtype=torch.float32).pin_memory()
    Qd = torch.empty_like(copies[0]["Q"])
    calls = [fla.PreparedDecodeHostIO(Qh[i], Qd, c["K_base"], c["V_base"], c["L"], c["B"], c["offsets"],
                                      rank=w.rank, O_dev=c["O"], O_host=Oh, workspace=workspace, stream=stream)
             for i, c in enumerate(copies)]
    for i in range(max(args.warmup, 3)):
        calls[i % n_copies]()
    stream.synchronize()

    def e2e_round():
        for c in calls:
            c()

    e2e_times = []
    barrier(ws)
    torch.cuda.synchronize()
    preroll(e2e_round, stream)
    for _ in range(E2E_ROUNDS):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(ws)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(args.steps):
            calls[i % n_copies]()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_times.append(e0.elapsed_time(e1) / 1e3)
    barrier(ws)
    t_e2e = max_over_ranks(statistics.median(e2e_times), ws, device)
    e2e_value = ws * queries_per_step * args.steps / t_e2e

    peaks = load_peaks()
    step_s = t_local / args.steps
    achieved_gbs = per_copy / step_s / 1e9
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "queries/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V/L, B ~ N(0, 0.02^2)); no dataset or trained weights",
        "config": {
            "workload": "Llama-3-8B-shaped single-layer decode: 3 agents, 32 q / 8 kv heads, head_dim 128, "
                        "r 16, shared context 16384 tokens, 1 query token per agent",
            "n_agents": w.n_agents, "hq": w.hq, "hkv": w.hkv, "head_dim": w.head_dim, "rank": w.rank,
            "context_tokens": w.total_tokens, "queries_per_step": queries_per_step,
            "parallelism": f"replicas x{ws} (independent workloads, no collective)",
            "l2": f"inputs rotate over {n_copies} copies ({n_copies * per_copy / 1e6:.0f} MB > 4x the 126 MB L2)",
            "timing": f"median of {REPLAYS} replays of a CUDA graph of K back-to-back decode calls, each "
                      "replay bracketed by a barrier + synchronize and timed with CUDA events on the launching "
                      f"stream, after {PREROLL_S:.2f} s of untimed replays of the same graph (load clocks)",
            "replays": REPLAYS,
            "ms_per_step_min": min(times) / args.steps * 1e3,
            "ms_per_step_max": max(times) / args.steps * 1e3,
        },
        "roofline": {
            "bound": "hbm",
            "achieved": achieved_gbs,
            "peak": peaks["hbm_gbs"],
            "unit": "GB/s",
            "frac": achieved_gbs / peaks["hbm_gbs"],
            "traffic": stored_traffic(HEADLINE),
            "kernel": "decode_tc_kernel",
            "algorithmic_bytes_per_launch": per_copy,
            "peak_source": peaks["source"],
            "frac_of_nominal_8tbs": achieved_gbs / 8000.0,
        },
        "e2e": {"value": e2e_value, "unit": "queries/s",
                "h2d_bytes_per_step": int(copies[0]["Q"].numel() * 2),
                "d2h_bytes_per_step": int(copies[0]["O"].numel() * 4),
                "api": "flash_lora_attn_decode_host_io (pinned host Q in, host O out, one call per step)",
                "timing": f"median of {E2E_ROUNDS} rounds of K steps",
                "ms_per_step_min": min(e2e_times) / args.steps * 1e3,
                "ms_per_step_max": max(e2e_times) / args.steps * 1e3},
        # per step: the decode kernel and the split-merge kernel behind it
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
    }
    del copies, calls, graph, Qh
    torch.cuda.empty_cache()
    if rank == 0 and args.legs == "all":
        line["legs"] = run_legs(args, device, peaks)
        iso = line["legs"].get(f"{HEADLINE}/decode")
        if iso:
            line["latency"] = {
                "isolated_call_us": iso["us"],
                "isolated_call_hbm_frac": iso["hbm_frac"],
                "pipelined_call_us": ms_per_step * 1e3,
                "pipelined_call_hbm_frac": achieved_gbs / peaks["hbm_gbs"],
                "note": "isolated: one call alone, L2 flushed before it, median of event-timed graph "
                        "replays; pipelined: the headline's back-to-back calls"}
    if rank == 0 and ws == 1:
        line["cpu_baseline"] = cpu_baseline(w)
    return line


def _median_launch_s(fn, reps, stream, flush=None, settle=False):
    """Median device time of one fn() call over reps replays.

    fn is captured once into a CUDA graph, so the events bracket only the
    kernels the call enqueues (no host-side argument handling); an optional
    L2 flush runs between replays, outside the events.  settle: start after
    one idle second, so that a tensor-bound leg is not measured under the power
    cap its predecessors in the same process pushed the GPU into; the timed
    replays then follow 20 ms of untimed ones, which bring the clocks back up
    from idle without heating the GPU into the power cap (the legs are burst
    measurements, against the burst peak).
    """
    import torch

    if settle:
        torch.cuda.synchronize()
        time.sleep(1.0)
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fn()
    if settle:
        t_end = time.perf_counter() + 0.02
        with torch.cuda.stream(stream):
            while time.perf_counter() < t_end:
                graph.replay()
                stream.synchronize()
    times = []
    with torch.cuda.stream(stream):
        graph.replay()
        for _ in range(reps):
            if flush is not None:
                flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b) / 1e3)
    return statistics.median(times)


def run_legs(args, device, peaks, only=None):
    """The other hot-path rows, each timed alone: median of event-timed launches.

    `only` (a leg name such as "llama70b_decode/decode") runs that leg alone,
    which is how the ncu captures select one kernel on one workload.

    Inputs larger than L2 need no flush; the 512-token chunk workloads are
    preceded by a 256 MB write that evicts L2.
    """
    import numpy as np
    import torch

    import attention_flash_lora_attn_b300 as fla
    from workloads import WORKLOADS

    reps = max(5, min(args.steps, 20)) if only is None else args.steps
    stream = torch.cuda.Stream(device)

    def want(name):
        return only is None or only == name
    g = torch.Generator(device=device).manual_seed(7)
    scratch = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)

    def flush():
        scratch.fill_(1.0)

    def rnd(shape, std=1.0):
        return (std * torch.randn(shape, generator=g, device=device)).to(torch.bfloat16)

    out = {}
    # ---- LR-cache build of a 512-token chunk (4 agents, r 16) and the causal chunked prefill
    w = WORKLOADS["llama8b_prefill"]
    A, r, D, c, n0 = w.n_agents, w.rank, w.d_model, w.chunk, w.n0
    X, A_cat = rnd((c, D)), rnd((D, A * r), D ** -0.5)
    L = rnd((n0 + c, A * r))
    if want("llama8b_prefill/lr_cache_build"):
        t = _median_launch_s(lambda: fla.lr_cache_build(X, A_cat, L[n0:], n_agents=A), reps, stream, flush)
        flops, byts = 2 * c * D * A * r, (c * D + A * r * D + c * A * r) * 2
        out["llama8b_prefill/lr_cache_build"] = {
            "us": t * 1e6, "tflops": flops / t / 1e12, "tensor_frac": flops / t / 1e12 / peaks["bf16_tflops"],
            "gbs": byts / t / 1e9, "hbm_frac": byts / t / 1e9 / peaks["hbm_gbs"]}
    if want("llama8b_prefill/prefill"):
        Q, K, V = rnd((A, c, w.hq, w.head_dim)), rnd((n0 + c, w.hkv, w.head_dim)), rnd((n0 + c, w.hkv, w.head_dim))
        B = rnd((A, r, w.hkv * w.head_dim), 0.02)
        O = torch.empty((A, c, w.hq, w.head_dim), dtype=torch.float32, device=device)
        t = _median_launch_s(lambda: fla.flash_lora_attn_prefill(Q, K, V, L, B, n0, rank=r, O=O),
                             max(3, reps // 4), stream, flush, settle=True)
        # causal: query p sees n0+p+1 keys; QK^T and PV over d, PL over r, (PL)B once per query
        keys = sum(n0 + p + 1 for p in range(c))
        flops = A * w.hq * keys * (4 * w.head_dim + 2 * r) + A * c * w.hq * 2 * r * w.head_dim
        out["llama8b_prefill/prefill"] = {"us": t * 1e6, "tflops": flops / t / 1e12,
                                          "tensor_frac": flops / t / 1e12 / peaks["bf16_tflops"]}
        del Q, K, V, B, O
    del X, A_cat, L
    # ---- decode legs (inputs larger than L2)
    for name in ("llama8b_decode", "llama8b_ragged", "llama70b_decode"):
        if not want(f"{name}/decode"):
            continue
        w = WORKLOADS[name]
        N, A, r = w.total_tokens, w.n_agents, w.rank
        Q, K, V = rnd((w.n_req, A, w.hq, w.head_dim)), rnd((N, w.hkv, w.head_dim)), rnd((N, w.hkv, w.head_dim))
        L, B = rnd((N, A * r)), rnd((A, r, w.hkv * w.head_dim), 0.02)
        offs = torch.tensor([0] + list(np.cumsum(w.lengths)), dtype=torch.int32, device=device)
        O = torch.empty((w.n_req, A, w.hq, w.head_dim), dtype=torch.float32, device=device)
        fits_l2 = decode_algorithmic_bytes(w) < L2_BYTES
        t = _median_launch_s(lambda: fla.flash_lora_attn_decode(Q, K, V, L, B, offs, rank=r, O=O), reps, stream,
                             flush if fits_l2 else None)
        byts = decode_algorithmic_bytes(w)
        out[f"{name}/decode"] = {"us": t * 1e6, "queries_per_s": w.n_req * A / t, "gbs": byts / t / 1e9,
                                 "hbm_frac": byts / t / 1e9 / peaks["hbm_gbs"]}
        del Q, K, V, L, B, O
    # ---- baselines on the 8B decode (not the hot path): naive materialisation
    #      (V_i = V_base + L_i.B_i expanded, then plain attention per agent)
    #      and non-shared caches (a full K/V cache per agent)
    base_legs = ("llama8b_decode/lora_value_expand", "llama8b_decode/naive_materialised",
                 "llama8b_decode/non_shared")
    if any(want(n) for n in base_legs):
        from attention_flash_lora_attn_b300 import baselines
        w = WORKLOADS["llama8b_decode"]
        N, A, r, hkv, d = w.total_tokens, w.n_agents, w.rank, w.hkv, w.head_dim
        Q, K, V = rnd((1, A, w.hq, d)), rnd((N, hkv, d)), rnd((N, hkv, d))
        L, B = rnd((N, A * r)), rnd((A, r, hkv * d), 0.02)
        offs = torch.tensor([0, N], dtype=torch.int32, device=device)
        kv = N * hkv * d * 2  # bytes of one K or V cache
        expand_bytes = kv + N * A * r * 2 + A * r * hkv * d * 2 + A * kv  # V_base, L, B in; A x V_i out
        plain_bytes = 2 * kv + N * baselines.ZERO_RANK * 2                # one agent's K, V (+ zero LR cache)
        fused = out.get("llama8b_decode/decode", {}).get("us")
        if want("llama8b_decode/lora_value_expand") or want("llama8b_decode/naive_materialised"):
            naive = baselines.PreparedBaselineDecode("naive", Q, offs, K_base=K, V_base=V, L=L, B=B, rank=r,
                                                     stream=stream)
            if want("llama8b_decode/lora_value_expand"):
                t = _median_launch_s(naive.expand, reps, stream, flush)
                out["llama8b_decode/lora_value_expand"] = {
                    "us": t * 1e6, "bytes": expand_bytes, "gbs": expand_bytes / t / 1e9,
                    "hbm_frac": expand_bytes / t / 1e9 / peaks["hbm_gbs"]}
            if want("llama8b_decode/naive_materialised"):
                t = _median_launch_s(naive, reps, stream, flush)
                byts = expand_bytes + A * plain_bytes
                leg = {"us": t * 1e6, "queries_per_s": A / t, "bytes": byts, "gbs": byts / t / 1e9,
                       "hbm_frac": byts / t / 1e9 / peaks["hbm_gbs"]}
                if fused:
                    leg["time_vs_fused_decode"] = t * 1e6 / fused
                out["llama8b_decode/naive_materialised"] = leg
            del naive
        if want("llama8b_decode/non_shared"):
            Ks = [rnd((N, hkv, d)) for _ in range(A)]
            Vs = [rnd((N, hkv, d)) for _ in range(A)]
            ns = baselines.PreparedBaselineDecode("non_shared", Q, offs, K=Ks, V=Vs, stream=stream)
            t = _median_launch_s(ns, reps, stream, flush)
            byts = A * plain_bytes
            leg = {"us": t * 1e6, "queries_per_s": A / t, "bytes": byts, "cache_bytes": A * 2 * kv,
                   "gbs": byts / t / 1e9, "hbm_frac": byts / t / 1e9 / peaks["hbm_gbs"]}
            if fused:
                leg["time_vs_fused_decode"] = t * 1e6 / fused
            out["llama8b_decode/non_shared"] = leg
            del ns, Ks, Vs
        del Q, K, V, L, B
    # ---- ReBaseShared base projection fused with the LR build:
    #      [K_base | V_base | L] = X . [W_k | W_v | A_cat], one pass over X
    # (the 16384-row case is the profiler-sized slice of the 70B one, run only when asked for)
    for leg, wname, rows in (("llama8b_prefill/rebase_kv_lr_build", "llama8b_prefill", None),
                             ("llama70b_decode/rebase_kv_lr_build", "llama70b_decode", None),
                             ("llama70b_decode/rebase_kv_lr_build_16k_rows", "llama70b_decode", 16384)):
        if not want(leg) or (only is None and rows is not None):
            continue
        w = WORKLOADS[wname]
        n = rows or w.build_tokens
        D, kv, lr = w.d_model, w.hkv * w.head_dim, w.n_agents * w.rank
        X, W = rnd((n, D)), rnd((D, 2 * kv + lr), D ** -0.5)
        K = torch.empty((n, w.hkv, w.head_dim), dtype=torch.bfloat16, device=device)
        V, L = torch.empty_like(K), torch.empty((n, lr), dtype=torch.bfloat16, device=device)
        t = _median_launch_s(lambda: fla.rebase_kv_lr_build(X, W, hkv=w.hkv, head_dim=w.head_dim,
                                                            n_agents=w.n_agents, rank=w.rank, K_base=K, V_base=V,
                                                            L=L), max(3, reps // 2), stream,
                             flush if n * D * 2 < L2_BYTES else None, settle=True)
        flops, byts = 2 * n * D * (2 * kv + lr), (n * D + D * (2 * kv + lr) + n * (2 * kv + lr)) * 2
        out[leg] = {
            "us": t * 1e6, "tflops": flops / t / 1e12, "tensor_frac": flops / t / 1e12 / peaks["bf16_tflops"],
            "gbs": byts / t / 1e9, "hbm_frac": byts / t / 1e9 / peaks["hbm_gbs"]}
        del X, W, K, V, L
    # ---- full LR-cache build, 131072 x 8192 . 8192 x 320
    w = WORKLOADS["llama70b_decode"]
    # the first 16384 rows of the 70B build: a profiler-sized case of the same kernel
    for leg, rows in (("llama70b_decode/lr_cache_build", w.build_tokens),
                      ("llama70b_decode/lr_cache_build_16k_rows", 16384)):
        if not want(leg) or (only is None and rows != w.build_tokens):
            continue
        n, D, Nc = rows, w.d_model, w.n_agents * w.rank
        X, A_cat = rnd((n, D)), rnd((D, Nc), D ** -0.5)
        L = torch.empty((n, Nc), dtype=torch.bfloat16, device=device)
        t = _median_launch_s(lambda: fla.lr_cache_build(X, A_cat, L, n_agents=w.n_agents), max(3, reps // 2), stream,
                             settle=True)
        flops, byts = 2 * n * D * Nc, (n * D + Nc * D + n * Nc) * 2
        out[leg] = {
            "us": t * 1e6, "tflops": flops / t / 1e12, "tensor_frac": flops / t / 1e12 / peaks["bf16_tflops"],
            "gbs": byts / t / 1e9, "hbm_frac": byts / t / 1e9 / peaks["hbm_gbs"]}
        del X, A_cat, L
    del scratch
    torch.cuda.empty_cache()
    assert fla.device_error() == 0
    return out


# ----------------------------------------------------------------------------- CPU oracle arm

def oracle_sample_rate(w, budget_s=10.0, max_reps=50):
    """Oracle queries/s on a bounded sample: one agent's query (all its heads) per repetition."""
    import numpy as np
    import torch

    import oracle
    from workloads import make_decode_inputs

    x = make_decode_inputs(w, seed=0)
    r = w.rank
    reps, t_total = 0, 0.0
    while reps < max_reps and t_total < budget_s:
        a = reps % w.n_agents
        t0 = time.perf_counter()
        oracle.decode(x["Q"][:, a:a + 1], x["K_base"], x["V_base"], x["L"][:, a * r:(a + 1) * r],
                      x["B"][a:a + 1], x["offsets"].numpy(), rank=r)
        t_total += time.perf_counter() - t0
        reps += 1
    cores = len(os.sched_getaffinity(0))
    threads = torch.get_num_threads()
    return reps / t_total, reps, t_total, cores, threads


def _rate(fn, budget_s, max_reps, min_reps=1):
    """(reps / seconds, reps, seconds) of fn() repeated until budget_s or max_reps."""
    reps, t_total = 0, 0.0
    while reps < min_reps or (reps < max_reps and t_total < budget_s):
        t0 = time.perf_counter()
        fn(reps)
        t_total += time.perf_counter() - t0
        reps += 1
    return reps / t_total, reps, t_total


def oracle_per_config():
    """The oracle timed on every workload (bounded samples, extrapolated where
    the full workload would take minutes); all host threads unless stated."""
    import dataclasses

    import numpy as np
    import torch
    import oracle
    from workloads import WORKLOADS, make_build_inputs, make_decode_inputs, make_prefill_inputs

    out = {}
    one_thread = os.environ.get("FLA_ORACLE_ONE_THREAD") == "1"

    def decode_one(x, q, a, r):
        o = x["offsets"]
        t0, t1 = int(o[q]), int(o[q + 1])
        oracle.decode(x["Q"][q:q + 1, a:a + 1], x["K_base"][t0:t1], x["V_base"][t0:t1],
                      x["L"][t0:t1, a * r:(a + 1) * r], x["B"][a:a + 1], np.array([0, t1 - t0]), rank=r)

    # c0: the whole tiny fp32 workload (2 queries) per repetition
    w = WORKLOADS["tiny_decode"]
    x = make_decode_inputs(w, seed=0)
    rate, reps, secs = _rate(lambda i: oracle.decode(x["Q"], x["K_base"], x["V_base"], x["L"], x["B"],
                                                     x["offsets"].numpy(), rank=w.rank), 1.0, 200)
    out["tiny_decode"] = {"value": rate * w.n_req * w.n_agents, "unit": "queries/s",
                          "sample": f"{reps} runs of the full workload, {secs:.2f} s"}
    # c1: single-agent queries of the headline decode
    w = WORKLOADS["llama8b_decode"]
    x = make_decode_inputs(w, seed=0)
    rate, reps, secs = _rate(lambda i: decode_one(x, 0, i % w.n_agents, w.rank), 4.0, 50)
    out["llama8b_decode"] = {"value": rate, "unit": "queries/s",
                             "sample": f"{reps} single-agent queries (all heads, 16384 tokens), {secs:.2f} s"}
    del x
    if one_thread:
        return out
    # c2: causal prefill positions (one agent, all heads) and the chunk's LR build
    w = WORKLOADS["llama8b_prefill"]
    x = make_prefill_inputs(w, seed=0)
    r = w.rank
    pos = [0, 255, 511]

    def prefill_one(i):
        a, p = i % w.n_agents, pos[i % len(pos)]
        oracle.prefill(x["Q"][a:a + 1], x["K_base"], x["V_base"], x["L"][:, a * r:(a + 1) * r], x["B"][a:a + 1],
                       n0=w.n0, rank=r, positions=[p])
    rate, reps, secs = _rate(prefill_one, 3.0, 30)
    out["llama8b_prefill/prefill"] = {
        "value": rate, "unit": "query tokens/s",
        "sample": f"{reps} (agent, chunk position) rows, all heads, {secs:.2f} s",
        "full_chunk_s_extrapolated": w.n_agents * w.chunk / rate}
    rate, reps, secs = _rate(lambda i: oracle.lr_cache_build(x["X"], x["A_cat"]), 2.0, 20)
    out["llama8b_prefill/lr_cache_build"] = {
        "value": rate * w.chunk, "unit": "rows/s",
        "gflops": rate * 2 * w.chunk * w.d_model * w.n_agents * r / 1e9,
        "sample": f"{reps} full 512x4096 . 4096x64 builds, {secs:.2f} s"}
    del x
    # c3: single-agent queries of the shortest, a middle and the longest request;
    #     the batch time is extrapolated by tokens (each query's cost grows with
    #     its request's length)
    w = WORKLOADS["llama8b_ragged"]
    lens = sorted(w.lengths)
    pick = [lens[0], lens[len(lens) // 2], lens[-1]]
    x = make_decode_inputs(dataclasses.replace(w, lengths=tuple(pick)), seed=0)
    rate, reps, secs = _rate(lambda i: decode_one(x, i % 3, i % w.n_agents, w.rank), 3.0, 30, min_reps=3)
    toks = sum(pick[i % 3] for i in range(reps))
    batch_s = secs / toks * w.total_tokens * w.n_agents
    out["llama8b_ragged"] = {"value": w.n_req * w.n_agents / batch_s, "unit": "queries/s",
                             "sample": f"{reps} single-agent queries on requests of {pick} tokens, {secs:.2f} s; "
                                       "batch time extrapolated by tokens",
                             "batch_s_extrapolated": batch_s}
    del x
    # c4: one agent's query over the full 131072-token context, and 512 sampled
    #     rows of the 131072 x 8192 . 8192 x 320 build (extrapolated to all rows)
    w = WORKLOADS["llama70b_decode"]
    x = make_decode_inputs(w, seed=0)
    rate, reps, secs = _rate(lambda i: decode_one(x, 0, i % w.n_agents, w.rank), 1.0, 2)
    out["llama70b_decode"] = {"value": rate, "unit": "queries/s",
                              "sample": f"{reps} single-agent queries (all 64 heads, 131072 tokens), {secs:.2f} s"}
    del x
    b = make_build_inputs(512, w.d_model, w.n_agents, w.rank, torch.bfloat16, seed=0)
    rate, reps, secs = _rate(lambda i: oracle.lr_cache_build(b["X"], b["A_cat"]), 2.0, 20)
    out["llama70b_decode/lr_cache_build"] = {
        "value": rate * 512, "unit": "rows/s",
        "gflops": rate * 2 * 512 * w.d_model * w.n_agents * w.rank / 1e9,
        "sample": f"{reps} builds of 512 sampled rows, {secs:.2f} s",
        "full_build_s_extrapolated": w.build_tokens / (rate * 512)}
    return out


def oracle_one_thread():
    """The c0 and c1 oracle rates with one host thread: a child process whose
    BLAS and OpenMP pools are limited to one thread before numpy loads."""
    env = dict(os.environ, FLA_ORACLE_ONE_THREAD="1", OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1",
               MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-per-config"], env=env,
                       capture_output=True, text=True, timeout=300)
    if r.returncode != 0:
        return {"error": (r.stderr or r.stdout)[-300:]}
    res = json.loads(r.stdout.strip().splitlines()[-1])
    return {f"{k}_1thread": v for k, v in res.items()}


def cpu_baseline(w):
    rate, reps, secs, cores, threads = oracle_sample_rate(w)
    per = oracle_per_config()
    per.update(oracle_one_thread())
    return {"value": rate, "unit": "queries/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} single-agent decode queries (all 32 heads, 16384 tokens) of the "
                      f"headline workload, fp64 numpy, {secs:.1f} s; BLAS threads {threads}",
            "per_config": per}


def run_reference(args):
    from workloads import WORKLOADS

    w = WORKLOADS[HEADLINE]
    import numpy as np
    import torch

    import oracle
    from workloads import make_decode_inputs

    x = make_decode_inputs(w, seed=0)
    r = w.rank

    def step(i):
        a = i % w.n_agents
        oracle.decode(x["Q"][:, a:a + 1], x["K_base"], x["V_base"], x["L"][:, a * r:(a + 1) * r],
                      x["B"][a:a + 1], x["offsets"].numpy(), rank=r)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    t = time.perf_counter() - t0
    value = args.steps / t
    cores = len(os.sched_getaffinity(0))
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "queries/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) Q/K/V/L, B ~ N(0, 0.02^2))",
        "config": {"workload": "Llama-3-8B-shaped single-layer decode: 3 agents, 32 q / 8 kv heads, head_dim "
                               "128, r 16, shared context 16384 tokens, 1 query token per agent",
                   "sample": "one agent's decode query (all 32 heads) per step"},
        "cpu_baseline": {"value": value, "unit": "queries/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} single-agent decode queries of the headline workload, fp64 "
                                   f"numpy, BLAS threads {torch.get_num_threads()}"},
        "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ----------------------------------------------------------------------------- main

def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--legs", choices=["all", "none"], default="all")
    ap.add_argument("--oracle-per-config", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--only", default=None,
                    help="run one leg alone (e.g. llama70b_decode/decode) and print its numbers")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_env()

    if args.oracle_per_config:  # child of oracle_one_thread()
        if os.environ.get("FLA_ORACLE_ONE_THREAD") == "1":
            import torch

            torch.set_num_threads(1)
        print(json.dumps(oracle_per_config()))
        return 0

    if args.only:
        import torch

        import attention_flash_lora_attn_b300 as fla
        from attention_flash_lora_attn_b300 import build_lib

        build_lib.build()
        fla.load_library()
        device = torch.device("cuda", local)
        torch.cuda.set_device(device)
        print(json.dumps({"only": args.only, **run_legs(args, device, load_peaks(), only=args.only)}))
        return 0

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0

    if ws > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    line = run_ours(args, ws, rank, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
