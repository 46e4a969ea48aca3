#!/usr/bin/env python3
"""Benchmark of the parallel-decode step on GB300.

One step = one full decode iteration over a batch of blocks: the fused softmax-statistics +
threshold-commit kernel, the smoothing probability rows, the tcgen05 smoothing GEMM and the
KV-refresh mask (workload "smooth_step": B=16 blocks of L=64 positions, V=126464, d=2048).
Other workloads (--workload threshold_loop | hierarchical_loop | credit_loop |
threshold_single) time the decode loops instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload smooth_step]

Prints ONE JSON line (rank 0).  With N > 1 (torchrun), every rank runs its own independent
batch (weak scaling, no collective on the data path); value = all ranks' block-iterations over
the slowest rank's time.  --impl reference times the oracle (plain single-threaded C++) on the
host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402
from synth.workloads import SEEDS, WORKLOADS  # noqa: E402

METRIC = "decode iters/s per block; logit GB/s as fraction of GB300 HBM peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024
# Decode loops stop on the device: a continue test every k iterations gates the rest of the
# loop.  A test costs ~6-8 us of graph scheduling (a nested conditional section), so k trades
# how soon a finished block stops against that cost, about a quarter of the loop's expected
# length: 2 for the threshold loop (its blocks end within a few iterations), 8 for the 24-step
# credit loops, 16 for the hierarchical loops (up to 64 steps, nearly all of them decoding).
LOOP_TEST_EVERY = {"threshold_loop": 2, "hierarchical_loop": 16, "hierarchical_levels_loop": 16}
LOOP_TEST_EVERY_DEFAULT = 8


# ------------------------------------------------------------------ environment helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        out = {}
        for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
            v = d.get(k)
            if isinstance(v, dict):
                v = v.get("value")
            out[k] = float(v) if v is not None else FALLBACK_PEAKS[k]
        return out, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="dllm_clocks_", suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "window": "1.5 s of the same step immediately before and through the timed "
                          "region, 100 ms sampling"}


def load_for(fn, seconds: float, dev) -> None:
    """Run fn repeatedly for about `seconds` (keeps the GPU under the step's own load while
    the clock sampler starts; the timed region follows immediately)."""
    t_end = time.perf_counter() + seconds
    while time.perf_counter() < t_end:
        for _ in range(20):
            fn()
        torch.cuda.synchronize(dev)


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda") if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base: int, rank: int) -> int:
    """Each rank decodes its own batch (independent problems: weak scaling)."""
    return base + 7919 * rank


# ------------------------------------------------------------------ our arm: smooth_step

# Translation units (with the headers they include) whose source a DRAM-traffic figure in
# profiles/traffic.md was measured on; a figure counts only while that source is unchanged.
_KERNEL_SOURCES = {
    "smooth_gemm_kernel": ["smooth.cu", "mbarrier.cuh", "vec_math.cuh"],
    "prob_rows_kernel": ["smooth.cu", "mbarrier.cuh", "vec_math.cuh"],
    "stats_partials_kernel": ["stats_commit.cu", "vec_math.cuh"],
    "stats_probs_kernel": ["stats_probs.cu", "mbarrier.cuh", "vec_math.cuh"],
}


# Loop workloads whose first iteration launches the statistics kernel exactly as another's does
# (same B, L, V, every position masked): the variants differ only in the commit kernel.
_FIRST_ITER_CAPTURE = {"credit_tracked_loop": "credit_loop",
                       "hierarchical_levels_loop": "hierarchical_loop"}


def kernel_source_hash(kernel: str) -> str:
    import hashlib
    root = os.path.dirname(os.path.abspath(__file__))
    csrc = os.path.join(root, "diffusion_decoding_gb300", "csrc")
    h = hashlib.sha256()
    for name in _KERNEL_SOURCES[kernel] + ["common.cuh", "internal.h"]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    with open(os.path.join(root, "include", "dllm.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch from the ncu capture recorded in profiles/traffic.md
    for this kernel and workload, or None when there is none or the kernel source changed."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(kernel)
    with open(path) as f:
        for line in f:
            cells = [c.strip().strip("`") for c in line.strip().strip("|").split("|")]
            if len(cells) >= 4 and cells[0] == kernel and cells[1] == workload:
                try:
                    nbytes = float(cells[3])
                except ValueError:
                    continue
                return nbytes if cells[2] == want else None
    return None


def host_numa(local: int) -> dict:
    """NUMA placement of the host memory the e2e copies come from: the nodes the host has, the
    node of this GPU's PCI function, and the nodes this process may allocate on."""
    info = {"host_nodes": None, "gpu_node": None, "allowed_mems": None}
    base = "/sys/devices/system/node"
    try:
        info["host_nodes"] = sorted(int(n[4:]) for n in os.listdir(base)
                                    if n.startswith("node") and n[4:].isdigit())
    except OSError:
        pass
    try:
        bus = torch.cuda.get_device_properties(local).pci_bus_id
        dom = torch.cuda.get_device_properties(local).pci_domain_id
        dev = torch.cuda.get_device_properties(local).pci_device_id
        path = f"/sys/bus/pci/devices/{dom:04x}:{bus:02x}:{dev:02x}.0/numa_node"
        with open(path) as f:
            info["gpu_node"] = int(f.read().strip())
    except (OSError, AttributeError, ValueError):
        pass
    try:
        with open("/proc/self/status") as f:
            for line in f:
                if line.startswith("Mems_allowed_list:"):
                    info["allowed_mems"] = line.split(":", 1)[1].strip()
    except OSError:
        pass
    return info


def plain_h2d_gbs(nbytes: int, dev) -> float:
    """One plain pinned host -> device copy of nbytes (cudaMemcpyAsync), best of 5."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = float("inf")
    for _ in range(6):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        d.copy_(h, non_blocking=True)
        b.record()
        torch.cuda.synchronize(dev)
        best = min(best, a.elapsed_time(b))
    return nbytes / (best * 1e-3) / 1e9


def algorithmic_bytes_stats(w, rows_read: int) -> int:
    """Logit bytes one stats launch must read (masked rows only) + state/stat writes."""
    es = 2 if w.dtype == "bf16" else 4
    return rows_read * w.V * es


def capture_graph(fn, dev, stream):
    """fn() captured once as a CUDA graph (on a side stream, joined back to `stream`)."""
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            fn()
    stream.wait_stream(cap)
    return g


def cold_replay_ms(g, flush, dev, stream, n=40):
    """Mean time of one replay of g between two events, each after an L2 flush (a write of a
    buffer twice the L2) on a GPU kept busy while the host enqueues the replay."""
    ts = []
    for _ in range(n):
        flush.fill_(1)
        torch.cuda._sleep(1_000_000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ts.append(a.elapsed_time(b))
    return statistics.mean(ts)


def run_smooth_step(args, rank, world, local):
    import diffusion_decoding_gb300 as dd

    w = WORKLOADS["smooth_step"]
    dev = torch.device("cuda", local)
    seed = rank_seed(SEEDS[w.key], rank)
    B, L, V, d = w.B, w.L, w.V, w.d
    R = B * L
    T = w.prefix_len + L
    lg_host = synth.logits(w, seed)                       # uint16 bf16 bits [B, L, V]
    E_host = synth.embedding_table(seed + 1, V, d)        # uint16 bf16 bits [V, d]
    logits = torch.from_numpy(lg_host.view(np.int16)).view(torch.bfloat16).to(dev)
    E = torch.from_numpy(E_host.view(np.int16)).to(dev)
    Et = torch.empty(dd.dllm_embedding_t_elems(V, d), dtype=torch.int16, device=dev)
    dd.dllm_prepare_embedding(E, Et)
    del E
    shape = dd.make_shape(B, L, V, dd.DLLM_BF16)
    state = dd.BlockState(B, L, device=dev)
    stats = dd.StatsBuffers(R, device=dev)
    ws = dd.workspace(dd.dllm_workspace_bytes(shape), dev)
    ws_s = dd.workspace(dd.dllm_smooth_workspace_bytes(shape, d), dev)
    out = torch.empty(R, d, dtype=torch.float32, device=dev)
    row_ids = torch.empty(R, dtype=torch.int32, device=dev)
    M = torch.zeros(1, dtype=torch.int32, device=dev)
    refresh = torch.empty(B * T, dtype=torch.uint8, device=dev)
    idx = torch.empty(B * T, dtype=torch.int32, device=dev)
    count = torch.empty(B, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def reset_state():
        # every step decodes a fresh block (every position masked): the library's reset kernel
        dd.dllm_block_state_reset(state, credit=False)

    ev = {}

    def step(lg):
        # the step: threshold commit + smoothing in one call (each logit read from HBM once),
        # then the KV refresh
        reset_state()
        dd.dllm_commit_threshold_smooth(lg, shape, stats, state, w.tau, w.eos_id, Et, d, out,
                                        row_ids, M, ws_s)
        dd.dllm_kv_refresh_mask(state, w.prefix_len, w.window, refresh, idx, count)

    def step_two_pass(lg, timed=False):
        # the same step through the separate calls (statistics + commit, probabilities, GEMM),
        # used for per-kernel timings and as the comparison point
        reset_state()
        if timed:
            # keep the GPU busy while the host enqueues the step, so that the events below
            # bracket the kernels back to back rather than host launch latency
            torch.cuda._sleep(3_000_000)
            ev["a0"].record(stream)
        dd.dllm_commit_threshold(lg, shape, stats, state, w.tau, w.eos_id, ws)
        if timed:
            ev["a1"].record(stream)
        dd.dllm_smooth_probs(lg, shape, stats, state, d, row_ids, M, ws_s)
        if timed:
            ev["b0"].record(stream)
        dd.dllm_smooth_gemm(shape, Et, d, out, M, ws_s)
        if timed:
            ev["b1"].record(stream)
        dd.dllm_kv_refresh_mask(state, w.prefix_len, w.window, refresh, idx, count)

    for _ in range(args.warmup):
        step_two_pass(logits)
        step(logits)
    torch.cuda.synchronize(dev)
    Mv = int(M.item())

    # the whole step (state reset + commit + smoothing + refresh) captured once into a CUDA
    # graph and replayed: the kernels run back to back without host launch gaps
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            step(logits)
    stream.wait_stream(cap)
    graph_two = torch.cuda.CUDAGraph()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph_two, stream=cap):
            step_two_pass(logits)
    stream.wait_stream(cap)
    for _ in range(args.warmup):
        graph.replay()
        graph_two.replay()
    torch.cuda.synchronize(dev)
    assert int(M.item()) == Mv
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        graph_two.replay()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    ms_two_pass = t0.elapsed_time(t1) / args.steps

    # per-kernel timing (events on the launching stream), then the whole-step timing
    t_stats, t_gemm, t_prob = [], [], []
    for _ in range(args.steps):
        ev.update({k: torch.cuda.Event(enable_timing=True) for k in ("a0", "a1", "b0", "b1")})
        step_two_pass(logits, timed=True)
        torch.cuda.synchronize(dev)
        t_stats.append(ev["a0"].elapsed_time(ev["a1"]))
        t_prob.append(ev["a1"].elapsed_time(ev["b0"]))
        t_gemm.append(ev["b0"].elapsed_time(ev["b1"]))

    # the statistics + commit call inside a graph, as a captured step runs it: a graph of the
    # block reset + the call against one of the reset alone, each replayed after an L2 flush
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    g_reset = capture_graph(reset_state, dev, stream)
    g_call = capture_graph(
        lambda: (reset_state(),
                 dd.dllm_commit_threshold(logits, shape, stats, state, w.tau, w.eos_id, ws)),
        dev, stream)
    stats_ms_graph = (cold_replay_ms(g_call, flush, dev, stream) -
                      cold_replay_ms(g_reset, flush, dev, stream))
    del flush

    clocks = ClockSampler(local)
    clocks.start()
    load_for(graph.replay, 1.5, dev)  # same step, so the sampler sees it under load
    barrier(world)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms, world)
    assert dd.dllm_get_status(ws_s) == dd.DLLM_OK

    # end to end through the public API with host buffers: H2D logits, step, D2H results
    # Two logits buffers, each with its own captured step: the host->device copy of step i+1's
    # logits (on a copy stream) overlaps step i; every step's copy in and result copy out are
    # inside the timed region.
    lg_pin = torch.from_numpy(lg_host.view(np.int16)).pin_memory()
    logits2 = torch.empty_like(logits)
    graph2 = torch.cuda.CUDAGraph()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph2, stream=cap):
            step(logits2)
    stream.wait_stream(cap)
    bufs = [logits.view(torch.int16), logits2.view(torch.int16)]
    graphs = [graph, graph2]
    res_dev = [state.tokens, state.masked, state.n_commit, row_ids, M, out, idx, count]
    res_pin = [torch.empty_like(t, device="cpu").pin_memory() for t in res_dev]
    h2d = lg_pin.numel() * 2
    d2h = sum(t.numel() * t.element_size() for t in res_dev)
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    consumed = [torch.cuda.Event(), torch.cuda.Event()]

    def h2d_into(j):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[j])      # the step that last read buffer j is done
            bufs[j].copy_(lg_pin, non_blocking=True)
            copied[j].record(copy_stream)

    def e2e_run(n):
        for j in range(2):
            consumed[j].record(stream)
        h2d_into(0)
        for i in range(n):
            cur = i % 2
            if i + 1 < n:
                h2d_into(1 - cur)
            stream.wait_event(copied[cur])
            graphs[cur].replay()
            for hp, dv in zip(res_pin, res_dev):
                hp.copy_(dv, non_blocking=True)
            consumed[cur].record(stream)

    e2e_run(max(2, args.warmup))
    torch.cuda.synchronize(dev)
    barrier(world)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    copy_stream.wait_stream(stream)
    e2e_run(args.steps)
    f1.record(stream)
    torch.cuda.synchronize(dev)
    ms_e2e = max_over_ranks(f0.elapsed_time(f1) / args.steps, world)
    link = host_numa(local)
    link["plain_h2d_gbs"] = plain_h2d_gbs(h2d, dev)
    link["e2e_h2d_gbs"] = h2d / (ms_e2e * 1e-3) / 1e9

    peaks, peak_src = load_peaks()
    gemm_ms = statistics.mean(t_gemm)
    stats_ms = statistics.mean(t_stats)
    prob_ms = statistics.mean(t_prob)
    flops = 2.0 * Mv * V * d
    gemm_tf = flops / (gemm_ms * 1e-3) / 1e12
    stats_bytes = algorithmic_bytes_stats(w, R)
    stats_gbs = stats_bytes / (stats_ms * 1e-3) / 1e9
    prob_bytes = Mv * V * 2 * 2  # read logits rows + write bf16 P rows
    prob_gbs = prob_bytes / (prob_ms * 1e-3) / 1e9
    step_bytes = R * V * 2
    plan = dd.dllm_smooth_plan_info(shape, d)
    # block reset, rows read, statistics + probabilities, commit, kept-row map, GEMM (+ split-K
    # reduction), refresh
    launches_per_step = 1 + 4 + (plan["launches"] - 2) + 1
    res = {
        "metric": METRIC,
        "value": world * B * 1e3 / ms,
        "unit": "block-iters/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,2) bf16 logits, N(0,0.02) bf16 embedding table)",
        "config": {"workload": "smooth_step: threshold commit (tau 0.9) + iteration smoothing "
                               "(softmax x E, d=2048) + KV refresh (prefix 1024, window 4); "
                               "statistics and probabilities from one read of the logits",
                   "B": B, "L_block": L, "V": V, "d": d, "M_smoothed": Mv, "gemm_plan": plan,
                   "l2": "inputs larger than L2 (259 MB logits + 518 MB table per step)",
                   "launch": "whole step captured in one CUDA graph, replayed per step",
                   "parallelism": f"replicas x{world}"},
        "iters_per_s": 1e3 / ms,
        "ms_per_step_two_pass": ms_two_pass,
        "logit_gbs_step": step_bytes / (ms * 1e-3) / 1e9,
        # the GEMM is timed on its own (events around one synchronised call), so its scale is
        # the burst figure; the sustained ratio is kept beside it
        "roofline": {"bound": "tensor", "kernel": "smooth_gemm_kernel", "achieved": gemm_tf,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": gemm_tf / peaks["bf16_tflops"],
                     "peak_source": f"{peak_src} bf16 burst (kernel timed alone)",
                     "frac_of_sustained": gemm_tf / peaks["bf16_tflops_sustained"],
                     "traffic": measured_traffic("smooth_gemm_kernel", "smooth_step"),
                     "traffic_unit": "DRAM bytes per launch", "ms": gemm_ms,
                     "algorithmic": f"2*M*V*d = {flops:.4g} FLOP per launch"},
        "roofline_stats": {"bound": "hbm", "kernel": "stats_partials_kernel + commit_only_kernel (one commit call)", "achieved": stats_gbs,
                           "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": stats_gbs / peaks["hbm_gbs"], "frac_of_8tbs": stats_gbs / 8000,
                           "peak_source": f"{peak_src} HBM copy",
                           "traffic": measured_traffic("stats_partials_kernel", "smooth_step"),
                           "traffic_unit": "DRAM bytes per launch (statistics kernel)",
                           "ms": stats_ms,
                           "ms_in_graph": stats_ms_graph,
                           "frac_in_graph": stats_bytes / (stats_ms_graph * 1e-3) / 1e9
                                            / peaks["hbm_gbs"],
                           "algorithmic": f"{stats_bytes} logit bytes per launch"},
        "roofline_probs": {"bound": "hbm", "kernel": "prob_rows_kernel", "achieved": prob_gbs,
                           "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": prob_gbs / peaks["hbm_gbs"], "ms": prob_ms,
                           "traffic": measured_traffic("prob_rows_kernel", "smooth_step")},
        "e2e": {"value": world * B * 1e3 / ms_e2e, "unit": "block-iters/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                "overlap": "double-buffered: step i+1's logits copy in while step i runs",
                "host_link": link},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    return res


# ------------------------------------------------------------------ our arm: sharded vocabulary

def run_tp_shards(args, rank, world, local, n_shards=8):
    """One credit-decoding step (B=32, L=32, V=126464) with the vocabulary split over n_shards
    tensor-parallel shards, all simulated on this GPU: each shard's statistics, the merge of the
    shards' statistics, and the commit from the merged statistics, replayed as one CUDA graph.
    (On n GPUs each rank would reduce only its own shard and all-gather R x 16 bytes.)"""
    import diffusion_decoding_gb300 as dd
    from diffusion_decoding_gb300.tp import vocab_range

    w = WORKLOADS["credit_loop"]
    dev = torch.device("cuda", local)
    seed = rank_seed(SEEDS["credit_loop"], rank)
    R = w.B * w.L
    lg = synth.logits(w, seed, 0).reshape(R, w.V)
    shards, stats_k, ws_k, shapes = [], [], [], []
    for k in range(n_shards):
        first, cnt = vocab_range(w.V, n_shards, k)
        stride = -(-cnt // 8) * 8
        buf = np.zeros((R, stride), np.uint16)
        buf[:, :cnt] = lg[:, first:first + cnt]
        shards.append(torch.from_numpy(buf.view(np.int16)).to(dev).view(torch.bfloat16))
        shapes.append(dd.make_shape(1, R, cnt, dd.DLLM_BF16, row_stride=stride))
        stats_k.append(dd.StatsBuffers(R, device=dev))
        ws_k.append(dd.workspace(dd.dllm_workspace_bytes(shapes[-1]), dev))
    offsets = [vocab_range(w.V, n_shards, k)[0] for k in range(n_shards)]
    shape = dd.make_shape(w.B, w.L, w.V, dd.DLLM_BF16)
    state = dd.BlockState(w.B, w.L, w.K, device=dev)
    merged = dd.StatsBuffers(R, device=dev)
    ws = dd.workspace(dd.dllm_workspace_bytes(shape), dev)
    stream = torch.cuda.current_stream(dev)
    ev = {}

    def step(timed=False):
        state.reset()
        for k in range(n_shards):
            dd.dllm_decode_stats(shards[k], shapes[k], state.masked, stats_k[k], ws_k[k])
        if timed:
            ev["m0"].record(stream)
        dd.dllm_merge_shard_stats(list(zip(stats_k, offsets)), R, merged)
        if timed:
            ev["m1"].record(stream)
        dd.dllm_commit_credit(None, shape, merged, state, w.K, w.decay, w.boost, w.tau,
                              w.eos_id, ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    t_merge = []
    for _ in range(args.steps):
        ev.update({k: torch.cuda.Event(enable_timing=True) for k in ("m0", "m1")})
        step(timed=True)
        torch.cuda.synchronize(dev)
        t_merge.append(ev["m0"].elapsed_time(ev["m1"]))
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            step()
    stream.wait_stream(cap)
    for _ in range(args.warmup):
        graph.replay()
    clocks = ClockSampler(local)
    clocks.start()
    load_for(graph.replay, 1.5, dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    peaks, peak_src = load_peaks()
    step_bytes = R * w.V * 2
    gbs = step_bytes / (ms * 1e-3) / 1e9
    return {
        "metric": METRIC, "value": world * w.B * 1e3 / ms, "unit": "block-iters/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded planted-peak logits)",
        "config": {"workload": f"tp{n_shards}_credit_step: vocabulary split over {n_shards} "
                               "simulated tensor-parallel shards on one GPU, B=32 L=32 "
                               "V=126464 bf16, credit commit from the merged statistics",
                   "launch": "whole step captured in one CUDA graph, replayed per step",
                   "parallelism": f"replicas x{world}"},
        "iters_per_s": 1e3 / ms,
        "roofline": {"bound": "hbm", "kernel": f"{n_shards} x statistics + merge + commit",
                     "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "peak_source": f"{peak_src} HBM copy",
                     "traffic": None, "ms": ms,
                     "algorithmic": f"{step_bytes} logit bytes per step"},
        "merge_kernel_us": 1e3 * statistics.mean(t_merge),
        "gpu_launches": (2 * n_shards + 2) * args.steps,
        "clocks": clk,
    }


# ------------------------------------------------------------------ our arm: decode loops

def run_loop(args, rank, world, local, key):
    import diffusion_decoding_gb300 as dd

    w = WORKLOADS[key]
    dev = torch.device("cuda", local)
    seed = rank_seed(SEEDS[key], rank)
    n_it = w.max_iters
    # pre-generate every iteration's logits in HBM (the generator is outside the timed region)
    lgs = [torch.from_numpy(synth.logits(w, seed, it).view(np.int16 if w.dtype == "bf16"
                                                            else np.float32)).to(dev)
           for it in range(n_it)]
    if w.dtype == "bf16":
        lgs = [t.view(torch.bfloat16) for t in lgs]
    shape = dd.make_shape(w.B, w.L, w.V, dd.DLLM_BF16 if w.dtype == "bf16" else dd.DLLM_F32)
    state = dd.BlockState(w.B, w.L, w.K, device=dev)
    stats = dd.StatsBuffers(w.B * w.L, device=dev)
    ws = dd.workspace(dd.dllm_workspace_bytes(shape), dev)
    stream = torch.cuda.current_stream(dev)

    def one(lg):
        if w.strategy == "threshold":
            dd.dllm_commit_threshold(lg, shape, stats, state, w.tau, w.eos_id, ws)
        elif w.strategy == "hierarchical":
            dd.dllm_commit_hierarchical(lg, shape, stats, state, w.tau_low, w.min_width,
                                        w.eos_id, ws)
        elif w.strategy == "hierarchical_levels":
            dd.dllm_commit_hierarchical_levels(lg, shape, stats, state, w.tau_low, w.min_width,
                                               w.eos_id, ws)
        elif w.strategy == "credit_tracked":
            dd.dllm_commit_credit_tracked(lg, shape, stats, state, w.K, w.decay, w.boost, w.tau,
                                          w.eos_id, ws)
        else:
            dd.dllm_commit_credit(lg, shape, stats, state, w.K, w.decay, w.boost, w.tau,
                                  w.eos_id, ws)

    def loop_eager():
        state.reset()
        for lg in lgs:
            one(lg)

    def capture(every: int):
        """The whole decode loop (state reset + every iteration) as one CUDA graph, replayed per
        step: no host round trip or launch gap between iterations.  With every = k > 0 the loop
        stops on the device: before iterations k, 2k, ... dllm_loop_continue tests the block and
        the rest of the loop sits in a conditional section on that test, each section nested in
        the one before, so a finished block skips all remaining iterations at the next test."""
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        bodies = [torch.cuda.Stream(dev) for _ in range((n_it - 1) // every if every else 0)]
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                state.reset()
                cur, level = cap, 0
                for it in range(n_it):
                    if every and it > 0 and it % every == 0:
                        h = dd.dllm_capture_condition(0, cur)
                        dd.dllm_loop_continue(state, h, cur)
                        dd.dllm_capture_if_begin(h, bodies[level], cur)
                        cur, level = bodies[level], level + 1
                    with torch.cuda.stream(cur):
                        one(lgs[it])
                for body in reversed(bodies):
                    dd.dllm_capture_if_end(body)
        stream.wait_stream(cap)
        return g

    for _ in range(2):
        loop_eager()
    torch.cuda.synchronize(dev)
    every = LOOP_TEST_EVERY.get(key, LOOP_TEST_EVERY_DEFAULT)
    graph_all, graph_es = capture(0), capture(every)

    def time_graph(g, with_clocks):
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize(dev)
        clocks = ClockSampler(local) if with_clocks else None
        if clocks:
            clocks.start()
        load_for(g.replay, 1.5, dev)
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        clk = clocks.stop() if clocks else None
        return max_over_ranks(e0.elapsed_time(e1) / args.steps, world), clk

    ms_all, _ = time_graph(graph_all, False)
    ms_loop, clk = time_graph(graph_es, True)
    # rows actually read per iteration (masked rows of running sequences), for GB/s; the
    # iterations the early-stop loop runs are those that start with a sequence still decoding
    rows = []
    state.reset()
    for lg in lgs:
        m = state.masked.view(w.B, w.L).clone()
        e = state.eos_hit.clone()
        rows.append(int((m.sum(1) * (e == 0)).sum().item()))
        one(lg)
    torch.cuda.synchronize(dev)
    n_live = 1 + sum(1 for r in rows[1:] if r > 0)  # iterations that start with work to do
    # iterations the early-stop graph runs: up to the first continue test after the end
    n_exec = min(n_it, -(-n_live // every) * every)
    n_tests = (n_exec - 1) // every + (1 if n_exec < n_it else 0)
    # first (fully masked) iteration alone, L2 flushed before each launch
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    t1 = []
    for _ in range(args.steps):
        state.reset()
        flush.fill_(1)
        torch.cuda._sleep(1_000_000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        one(lgs[0])
        b.record(stream)
        torch.cuda.synchronize(dev)
        t1.append(a.elapsed_time(b))
    # the same first iteration inside a graph (as the loops run it): a graph of the block reset
    # + the first call against a graph of the reset alone, each replayed cold; the difference is
    # what the first iteration adds to a captured loop
    g_reset = capture_graph(state.reset, dev, stream)
    g_first = capture_graph(lambda: (state.reset(), one(lgs[0])), dev, stream)
    ms1_graph = (cold_replay_ms(g_first, flush, dev, stream) -
                 cold_replay_ms(g_reset, flush, dev, stream))
    peaks, peak_src = load_peaks()
    es = 2 if w.dtype == "bf16" else 4
    ms1 = statistics.median(t1)
    gbs1 = rows[0] * w.V * es / (ms1 * 1e-3) / 1e9
    total_bytes = sum(rows) * w.V * es
    return {
        "metric": METRIC,
        "value": world * w.B * n_live * 1e3 / ms_loop,
        "unit": "block-iters/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_loop, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded planted-peak logits)",
        "config": {"workload": f"{key}: {w.title}", "max_iterations": n_it,
                   "iterations_decoding": n_live, "iterations_run": n_exec,
                   "launch": "whole loop captured in one CUDA graph, replayed per step; a "
                             f"device-side continue test every {every} iterations "
                             "gates the rest of the loop (nested conditional sections: early "
                             "stop once every sequence is finished)",
                   "l2": "per-iteration logits pre-generated in HBM and rotated; "
                         "single-iteration timing flushes L2 first"},
        "iters_per_s": n_live * 1e3 / ms_loop,
        "loops_per_s": 1e3 / ms_loop,
        "ms_per_step_all_iterations": ms_all,
        "loop_logit_gbs": total_bytes / (ms_loop * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": "stats_partials_kernel + commit_only_kernel (one commit call)", "achieved": gbs1,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs1 / peaks["hbm_gbs"],
                     "peak_source": f"{peak_src} HBM copy",
                     "traffic": measured_traffic("stats_partials_kernel",
                                                 _FIRST_ITER_CAPTURE.get(key, key)),
                     "ms": ms1, "ms_in_graph": ms1_graph,
                     "frac_in_graph": rows[0] * w.V * es / (ms1_graph * 1e-3) / 1e9
                                      / peaks["hbm_gbs"],
                     "algorithmic": f"{rows[0]} rows x V x {es} B"},
        # block reset, statistics + commit per iteration run, the continue tests reached
        "gpu_launches": (1 + 2 * n_exec + n_tests) * args.steps,
        "clocks": clk,
    }


# ------------------------------------------------------------------ reference arm: the oracle

_REF_INPUTS = {}


def cpu_sample_smooth(seed: int, smooth_rows: int):
    """Time the oracle on a bounded sample of smooth_step; returns (seconds per full step, info).

    Statistics, commit and refresh run over every row; the smoothing product runs on
    `smooth_rows` of the kept rows and is extrapolated to all of them.  Inputs are generated
    once per seed (outside the timed part)."""
    import oracle

    w = WORKLOADS["smooth_step"]
    if seed not in _REF_INPUTS:
        _REF_INPUTS[seed] = (synth.logits(w, seed), synth.embedding_table(seed + 1, w.V, w.d))
    lg, E = _REF_INPUTS[seed]
    st = oracle.BlockState(w.B, w.L)
    t0 = time.perf_counter()
    s = oracle.stats(lg, oracle.active_rows(st.masked, st.eos_hit))
    oracle.commit_threshold(st, s.conf.reshape(w.B, w.L), s.argmax.reshape(w.B, w.L),
                            float(np.float32(w.tau)), w.eos_id)
    ids = oracle.smooth_rows(st.masked, st.eos_hit)
    oracle.kv_refresh(st.committed_now, w.prefix_len, w.window)
    t_commit = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.smooth_embed(lg.reshape(-1, w.V), s.lse, ids[:smooth_rows], E)
    t_rows = time.perf_counter() - t0
    per_row = t_rows / smooth_rows
    est = t_commit + per_row * len(ids)
    info = (f"oracle, 1 thread: stats+commit+refresh over all {w.B * w.L} rows "
            f"({t_commit:.2f} s) + smoothing of {smooth_rows} of {len(ids)} rows "
            f"({per_row:.3f} s/row), extrapolated to the full step ({est:.1f} s)")
    return est, info


def run_reference(args, rank, world):
    if rank != 0:
        return None
    key = args.workload
    if key != "smooth_step":
        return {"impl": "reference", "unavailable": "reference arm implemented for smooth_step"}
    times, info = [], ""
    for i in range(args.warmup + args.steps):
        est, info = cpu_sample_smooth(SEEDS[key], smooth_rows=1)
        if i >= args.warmup:
            times.append(est)
    w = WORKLOADS[key]
    sec = statistics.mean(times)
    value = w.B / sec
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "block-iters/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": key, "B": w.B, "L_block": w.L, "V": w.V,
                                        "d": w.d},
        "cpu_baseline": {"value": value, "unit": "block-iters/s", "cores": 1, "kind": "oracle",
                         "sample": info},
        "e2e": {"value": value, "unit": "block-iters/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="smooth_step",
                    choices=sorted(WORKLOADS) + ["tp8_shards"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    from diffusion_decoding_gb300 import build as cuda_build
    cuda_build.build()
    if args.workload == "smooth_step":
        res = run_smooth_step(args, rank, world, local)
    elif args.workload == "tp8_shards":
        res = run_tp_shards(args, rank, world, local)
    else:
        res = run_loop(args, rank, world, local, args.workload)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline and args.workload == "smooth_step":
            import multiprocessing
            est, info = cpu_sample_smooth(SEEDS[args.workload], smooth_rows=8)
            res["cpu_baseline"] = {"value": WORKLOADS[args.workload].B / est,
                                   "unit": "block-iters/s", "cores": 1, "kind": "oracle",
                                   "sample": info,
                                   "host_cores": multiprocessing.cpu_count()}
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
