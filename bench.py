#!/usr/bin/env python3
"""Benchmark: one step = route metadata + dispatch (gather, fused quantisation) + weighted
combine over one batch of a seeded synthetic workload, on one GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload qwen3|prefill|nvfp4|decode|tiny]
                    [--per-config decode,prefill,nvfp4|none] [--impl ours|reference] [--graph] [--no-fuse]

Prints ONE JSON line (rank 0). The headline workload is the Qwen3-MoE-like batch (T=16384,
H=4096, E=128, top-8, 5 % empty slots, bf16 rows): the largest of the benchmark shapes. The
line's ``per_config`` object repeats the measurement, in the same process and under the same
clock sampler, for the other target shapes (DeepSeek-V3 decode in the low-latency masked FP8
layout, prefill FP8 with Zipf routing, the NVFP4 payload). ``value`` is whole-job dispatch+combine throughput in tokens/s
(tokens of all ranks / max-over-ranks mean step time), inputs resident in HBM, L2 flushed
(256 MiB write + 256 MiB read) before every step, CUDA events around every step only (an
event between two kernels would keep the second from launching early). A second pass of K
eager steps with an event after every library call gives the per-kernel durations.
``--graph`` replays one captured step in the first pass. ``e2e`` repeats the measurement
through the public Python API with pinned host inputs copied in and the combined output
copied out inside the timed region (pipelined, serial and graph-replayed schedules; the
fastest is reported). ``roofline`` reports the dominant kernel's algorithmic bytes /
CUDA-event duration against the measured HBM copy bandwidth. ``cpu_baseline`` times the CPU oracle on a bounded
sample of the same workload. ``--impl reference`` times that oracle as the reference arm.
Multi-GPU: one process per GPU (torchrun), each rank runs its own seeded batch (weak
scaling, no data-path collective; a max-reduce of the step time only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dispatch+combine tokens/s and achieved HBM GB/s (fraction of ~8 TB/s), 1 GB300"
FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # the "~8 TB/s" of the metric's name; `frac` uses the measured copy peak
_CSRC = "combine_moe_route_meta_gb300/csrc/"
KERNEL_SOURCES = {  # the files whose contents decide each kernel's machine code
    "route_meta": [_CSRC + "route_meta.cu", _CSRC + "moe_device.cuh"],
    "dispatch": [_CSRC + "dispatch.cu", _CSRC + "dispatch_slice.cuh", _CSRC + "moe_device.cuh"],
    "route_dispatch": [_CSRC + "route_dispatch.cu", _CSRC + "dispatch_slice.cuh", _CSRC + "moe_device.cuh"],
    "combine": [_CSRC + "combine.cu", _CSRC + "moe_device.cuh"],
}


# ---------------------------------------------------------------------------
# byte model (algorithmic bytes each kernel must move; padding/capacity never counted)
# ---------------------------------------------------------------------------

def row_bytes(quant: str, H: int) -> int:
    if quant == "none":
        return 2 * H
    if quant == "fp8g128":
        return H + 4 * (H // 128)
    return H // 2 + H // 16


def algorithmic_bytes(w, n_valid: int, n_rows: int) -> dict:
    """n_valid: valid pairs; n_rows: rows actually written by dispatch / read by combine."""
    T, H, K, E = w.T, w.H, w.K, w.E
    masked = w.mode == "masked"
    meta = 4 * T * K + 4 * T * K + 4 * n_valid + 8 * (E + 1) + 4 * E + 4 * w.P
    disp = 2 * T * H + 4 * T * K + (4 * T * K + 8 * E if masked else 0) + n_rows * row_bytes(w.quant, H)
    comb = n_rows * 2 * H + 8 * T * K + (4 * T * K + 8 * E if masked else 0) + 2 * T * H
    return {"route_meta": meta, "dispatch": disp, "combine": comb}


def measured_hbm_gbs():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digest(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        p = os.path.join(ROOT, rel)
        if os.path.exists(p):
            with open(p, "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current source."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(p):
        return None
    fields = {}
    with open(p) as f:
        for line in f:
            if ":" in line and line.lstrip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                fields[k.strip()] = v.strip()
    if fields.get("source_sha256") != source_digest(kernel):
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# clocks sampler
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t0 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

_ORACLE_OUT = {}


def _oracle_out(w, T_s, slot: int = 0):
    """Dispatch output arrays for a T_s-token sample, allocated once (outside any timing);
    `slot` gives each concurrent caller its own arrays."""
    import oracle
    key = (w.name, w.seed, T_s, slot)
    if key not in _ORACLE_OUT:
        rows = None if w.mode == "masked" else T_s * w.K
        qs, qd, ss, sd = oracle.out_shapes(w.mode, w.quant, T_s, w.H, w.K, w.E, w.M, rows)
        _ORACLE_OUT[key] = (np.zeros(qs, qd), np.zeros(ss, sd) if ss is not None else None)
    return _ORACLE_OUT[key]


def oracle_step(w, T_s: int, expert_rows, slot: int = 0):
    """One oracle pass (route meta + dispatch + combine) over the first T_s tokens."""
    import oracle
    ids = np.ascontiguousarray(w.topk_ids[:T_s])
    x = np.ascontiguousarray(w.x[:T_s])
    wt = np.ascontiguousarray(w.topk_weights[:T_s])
    meta = oracle.route_meta(ids, w.E, P=w.P, M=w.M)
    rows = None if w.mode == "masked" else T_s * w.K
    oracle.dispatch(w.mode, w.quant, x, ids, meta, w.E, M=w.M, global_scale=w.global_scale or 0.0, rows=rows,
                    out=_oracle_out(w, T_s, slot))
    if w.mode == "normal":
        eo = expert_rows[: max(meta.num_valid, 1)]
        oracle.combine("normal", eo, ids, wt, meta, w.E)
    else:
        # masked combine reads only rows e*M + rank < e*M + masked_m[e]; give it a layout
        # whose experts hold just the slots this sample fills
        M_s = int(meta.masked_m.max()) if meta.num_valid else 1
        meta_s = oracle.route_meta(ids, w.E, P=w.P, M=M_s)
        eo = expert_rows[: w.E * M_s]
        oracle.combine("masked", eo, ids, wt, meta_s, w.E, M=M_s)


def _expert_rows_needed(w, T_s: int) -> int:
    """Expert-output rows the oracle's combine reads for a T_s-token sample: T_s*K in the
    contiguous layout, E x (largest per-expert count of the sample) in the masked one."""
    if w.mode == "normal":
        return max(T_s * w.K, 1)
    import oracle
    meta = oracle.route_meta(np.ascontiguousarray(w.topk_ids[:T_s]), w.E, P=w.P, M=w.M)
    return w.E * max(int(meta.masked_m.max()) if meta.num_valid else 1, 1)


def time_oracle(w, budget_s: float, max_tokens: int):
    """Pick a token sample that takes ~budget_s per step and time one step of it."""
    from workloads import random_bf16
    rng = np.random.default_rng(99)
    T_probe = min(w.T, 16)
    er = random_bf16(rng, (_expert_rows_needed(w, T_probe), w.H))
    oracle_step(w, T_probe, er)  # allocates the sample's output arrays
    t0 = time.perf_counter()
    oracle_step(w, T_probe, er)
    per_tok = (time.perf_counter() - t0) / T_probe
    T_s = int(max(1, min(w.T, max_tokens, budget_s / max(per_tok, 1e-9))))
    er = random_bf16(rng, (_expert_rows_needed(w, T_s), w.H))
    _oracle_out(w, T_s)
    return T_s, er


def cpu_baseline(w, budget_s: float = 12.0) -> dict:
    T_s, er = time_oracle(w, budget_s / 3, w.T)
    times = []
    t_end = time.perf_counter() + budget_s
    while True:
        t0 = time.perf_counter()
        oracle_step(w, T_s, er)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() > t_end or len(times) >= 50:
            break
    med = statistics.median(times)
    return {"value": T_s / med, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"first {T_s} of {w.T} tokens of the {w.name} workload, route+dispatch+combine, "
                      f"median of {len(times)} passes, single-threaded C oracle"}


def cpu_baseline_all_cores(w, budget_s: float = 10.0) -> dict:
    """The same oracle, unchanged, run concurrently on every host core: one thread per core,
    each repeating the single-core sample on its own output arrays (the oracle's C calls
    release the interpreter lock). Tokens of all threads / wall time."""
    from concurrent.futures import ThreadPoolExecutor
    n = os.cpu_count() or 1
    T_s, er = time_oracle(w, budget_s / 4, w.T)
    for j in range(n):
        _oracle_out(w, T_s, j)
    oracle_step(w, T_s, er)
    t_one = time.perf_counter()
    oracle_step(w, T_s, er)
    t_one = time.perf_counter() - t_one
    passes = int(max(1, min(50, budget_s / max(t_one, 1e-9) / 2)))

    def work(j):
        for _ in range(passes):
            oracle_step(w, T_s, er, slot=j)

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=n) as ex:
        list(ex.map(work, range(n)))
    wall = time.perf_counter() - t0
    return {"value": n * passes * T_s / wall, "unit": "tokens/s", "cores": n, "kind": "oracle",
            "sample": f"{n} threads, each {passes} passes over the first {T_s} of {w.T} tokens of the "
                      f"{w.name} workload (route+dispatch+combine), single-threaded C oracle per thread"}


def run_reference(args, w, rank, world):
    if rank != 0:
        return None
    total_steps = args.steps + args.warmup
    budget = max(0.05, min(5.0, 90.0 / max(total_steps, 1)))
    T_s, er = time_oracle(w, budget, w.T)
    for _ in range(args.warmup):
        oracle_step(w, T_s, er)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(w, T_s, er)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    value = T_s / (ms / 1e3)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 combine / f32 quant", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {T_s} of {w.T} tokens per step, route+dispatch+combine, "
                                   f"single-threaded C oracle"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def max_over_ranks(x: float, dist, device="cpu") -> float:
    """Max of a per-rank scalar over all ranks (identity without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's step time."""
    return tokens_per_rank * world / (ms_per_step / 1e3)


def rank_seed(rank: int) -> int:
    """Each rank draws its own batch of the workload (weak scaling)."""
    return rank


def config_of(w) -> dict:
    return {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "K": w.K, "P": w.P, "M": w.M,
            "mode": w.mode, "quant": w.quant, "seed": w.seed, "recipe": w.recipe,
            "l2": f"flushed before every step ({FLUSH_BYTES >> 20} MiB write, then a {FLUSH_BYTES >> 20} MiB "
                  f"read so no dirty flush lines remain)"}


L2_BYTES = 129 << 20  # GB300 L2 (126 MiB reported by the device; rounded up)


def run_e2e(args, w, d, dev, x_h, ids_h, wt_h, g, fused, expert_out, dist):
    """Tokens/s through the public API with every step's inputs copied in from pinned host
    memory and its combined output copied back, K steps inside the timed region.

    Pipelined as a serving loop would run it: step i+1's host->device copy and step i-1's
    device->host copy overlap step i's kernels (three streams, two sets of device inputs,
    dispatcher outputs and pinned output buffers; events order every reuse of a buffer).
    The L2 is not flushed inside the region: each step's inputs arrive fresh from the host,
    and the combine reads rotate over enough expert-output buffers that the rows one step
    reads have left L2 before they are read again.

    Three more schedules are timed the same way: "serial" (copy in, kernels, copy out, one
    step after another, issued eagerly), "graph" (that serial step captured once per
    expert-output buffer as a CUDA graph and replayed, so small steps are not bound by the
    host's issue rate) and "graph_pipelined" (the pipelined schedule of a period of steps
    captured as one graph). The line reports the fastest and lists all of them."""
    import torch
    import combine_moe_route_meta_gb300 as moe

    nx, ni, nw = x_h.numel() * 2, ids_h.numel() * 4, wt_h.numel() * 4
    o_ids = (nx + 15) // 16 * 16
    o_w = (o_ids + ni + 15) // 16 * 16
    n_in = (o_w + nw + 15) // 16 * 16
    host_in = torch.empty(n_in, dtype=torch.uint8).pin_memory()
    host_in[:nx].copy_(x_h.view(torch.uint8).reshape(-1))
    host_in[o_ids:o_ids + ni].copy_(ids_h.view(torch.uint8).reshape(-1))
    host_in[o_w:o_w + nw].copy_(wt_h.view(torch.uint8).reshape(-1))
    dev_in = [torch.empty(n_in, dtype=torch.uint8, device=dev) for _ in range(2)]
    views = [(b[:nx].view(torch.bfloat16).view(w.T, w.H), b[o_ids:o_ids + ni].view(torch.int32).view(w.T, w.K),
              b[o_w:o_w + nw].view(torch.float32).view(w.T, w.K)) for b in dev_in]
    ds = [d, moe.MoEDispatcher(w.T, w.H, w.K, w.E, mode=w.mode, quant=w.quant, num_partitions=w.P,
                               max_tokens_per_expert=w.M, device=dev)]
    outp = [torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    # expert-output buffers: the combine of one step reads K rows per token
    read_per_step = max(1, w.T * w.K * w.H * 2)
    n_eo = int(min(32, max(1, -(-2 * L2_BYTES // read_per_step))))
    eos = [expert_out] + [torch.empty_like(expert_out).copy_(expert_out) for _ in range(n_eo - 1)]

    def kernels(slot, i):
        x2, ids2, wt2 = views[slot]
        dd = ds[slot]
        if fused:
            dd.route_dispatch(x2, ids2, g)
        else:
            dd.route(ids2)
            dd.dispatch(x2, ids2, g)
        dd.combine(eos[i % n_eo], ids2, wt2)

    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def issue_pipeline(n, ran, out):
        """Issue n pipelined steps on the three streams; ran / out carry the per-slot events
        of the previous steps (kernels done, device->host copy done)."""
        for i in range(n):
            b = i & 1
            if ran[b] is not None:
                s_in.wait_event(ran[b])
            with torch.cuda.stream(s_in):
                dev_in[b].copy_(host_in, non_blocking=True)
            e_in = torch.cuda.Event()
            e_in.record(s_in)
            s_run.wait_event(e_in)
            if out[b] is not None:
                s_run.wait_event(out[b])
            with torch.cuda.stream(s_run):
                kernels(b, i)
            ran[b] = torch.cuda.Event()
            ran[b].record(s_run)
            s_out.wait_event(ran[b])
            with torch.cuda.stream(s_out):
                outp[b].copy_(ds[b].out, non_blocking=True)
            out[b] = torch.cuda.Event()
            out[b].record(s_out)

    def pipelined(n):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        issue_pipeline(n, [None, None], [None, None])
        t1.record(s_out)
        return t0, t1

    def serial(n):
        evs = []
        with torch.cuda.stream(s_run):
            for i in range(n):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s_run)
                dev_in[0].copy_(host_in, non_blocking=True)
                kernels(0, i)
                outp[0].copy_(ds[0].out, non_blocking=True)
                e1.record(s_run)
                evs.append((e0, e1))
        return evs

    torch.cuda.synchronize()
    pipelined(max(args.warmup, 2))
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = pipelined(args.steps)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    for dd in ds:
        dd.check()
    last = (args.steps - 1) & 1
    assert torch.equal(outp[last], ds[last].out.cpu()), "e2e output differs from the device result"
    ms_pipe = max_over_ranks(t0.elapsed_time(t1) / args.steps, dist, dev)

    serial(max(args.warmup, 2))
    torch.cuda.synchronize()
    evs = serial(args.steps)
    torch.cuda.synchronize()
    ms_serial = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in evs), dist, dev)

    # one serial step per expert-output buffer, captured once (outside the timed region)
    ms_graph, graph_error = None, None
    try:
        graphs = []
        for j in range(n_eo):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=s_run):
                dev_in[0].copy_(host_in, non_blocking=True)
                kernels(0, j)
                outp[0].copy_(ds[0].out, non_blocking=True)
            graphs.append(gr)
    except RuntimeError as exc:  # capture refused: report the eager schedules only
        graph_error = str(exc).splitlines()[0][:200]
        torch.cuda.synchronize()
    if graph_error is None:
        for i in range(max(args.warmup, 2)):
            graphs[i % n_eo].replay()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s_run):
            g0.record(s_run)
            for i in range(args.steps):
                graphs[i % n_eo].replay()
            g1.record(s_run)
        torch.cuda.synchronize()
        ds[0].check()
        assert torch.equal(outp[0], ds[0].out.cpu()), "graph e2e output differs from the device result"
        ms_graph = max_over_ranks(g0.elapsed_time(g1) / args.steps, dist, dev)

    # the pipelined schedule of a period of steps captured as one graph (its streams forked
    # from and joined back to the capturing stream); replays run back to back, so the
    # pipeline drains once per period
    ms_gpipe = None
    if graph_error is None:
        period = max(n_eo, 8)

        def capture_period(n):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=s_run):
                fork = torch.cuda.Event()
                fork.record(s_run)
                s_in.wait_event(fork)
                s_out.wait_event(fork)
                issue_pipeline(n, [None, None], [None, None])
                for s_ in (s_in, s_out):
                    j = torch.cuda.Event()
                    j.record(s_)
                    s_run.wait_event(j)
            return gr

        full, rem = divmod(args.steps, period)
        try:
            g_full = capture_period(period) if full else None
            g_rem = capture_period(rem) if rem else None
        except RuntimeError as exc:  # capture refused: keep the other schedules
            graph_error = "graph_pipelined: " + str(exc).splitlines()[0][:200]
            torch.cuda.synchronize()
    if ms_graph is not None and graph_error is None:
        for _ in range(2):
            (g_full or g_rem).replay()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s_run):
            p0.record(s_run)
            for _ in range(full):
                g_full.replay()
            if g_rem is not None:
                g_rem.replay()
            p1.record(s_run)
        torch.cuda.synchronize()
        for dd in ds:
            dd.check()
        last = ((rem or period) - 1) & 1
        assert torch.equal(outp[last], ds[last].out.cpu()), "graph-pipelined e2e output differs"
        ms_gpipe = max_over_ranks(p0.elapsed_time(p1) / args.steps, dist, dev)

    world = dist.get_world_size() if dist else 1
    variants = {
        "pipelined": {"ms_per_step": ms_pipe, "value": job_throughput(w.T, world, ms_pipe),
                      "schedule": "copies of neighbouring steps overlap this step's kernels (3 streams, 2 buffer sets)"},
        "serial": {"ms_per_step": ms_serial, "value": job_throughput(w.T, world, ms_serial),
                   "schedule": "copy in, kernels, copy out, one step after another, issued eagerly"},
    }
    if ms_graph is not None:
        variants["graph"] = {"ms_per_step": ms_graph, "value": job_throughput(w.T, world, ms_graph),
                             "schedule": "the serial step (copy in, kernels, copy out) replayed as a CUDA graph"}
    if ms_gpipe is not None:
        variants["graph_pipelined"] = {
            "ms_per_step": ms_gpipe, "value": job_throughput(w.T, world, ms_gpipe),
            "schedule": f"the pipelined schedule of {max(n_eo, 8)} steps captured as one CUDA graph, replayed"}
    best = min(variants, key=lambda k: variants[k]["ms_per_step"])
    return {"value": variants[best]["value"], "unit": "tokens/s", "ms_per_step": variants[best]["ms_per_step"],
            "h2d_bytes_per_step": n_in, "d2h_bytes_per_step": w.T * w.H * 2,
            "copies": "one pinned H2D of the step's inputs, one D2H of the combined output, every step",
            "schedule": best,
            "l2": f"not flushed; inputs arrive by H2D each step; combine reads rotate over {n_eo} expert-output buffers",
            "schedules": variants, **({"graph_capture_error": graph_error} if graph_error else {})}


def run_gpu(args, w, rank, world, dist):
    """The JSON line of one workload (the caller samples the clocks around it)."""
    import torch
    import combine_moe_route_meta_gb300 as moe

    dev = torch.device("cuda", torch.cuda.current_device())
    x_h = torch.from_numpy(w.x.view(np.int16)).view(torch.bfloat16)
    ids_h = torch.from_numpy(w.topk_ids)
    wt_h = torch.from_numpy(w.topk_weights)
    x, ids, wt = x_h.to(dev), ids_h.to(dev), wt_h.to(dev)
    d = moe.MoEDispatcher(w.T, w.H, w.K, w.E, mode=w.mode, quant=w.quant, num_partitions=w.P,
                          max_tokens_per_expert=w.M, device=dev)
    g = w.global_scale or 0.0
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + rank)
    eo_rows = w.T * w.K if w.mode == "normal" else w.E * w.M
    expert_out = torch.randn((eo_rows, w.H), dtype=torch.bfloat16, device=dev, generator=gen)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    flush_out = torch.empty((), dtype=torch.int32, device=dev)

    def flush_l2(i: int):
        """Evict L2: write a buffer larger than L2, then read another one, so that the
        step starts with an L2 full of clean, unrelated lines (no write-back of the
        flush itself lands inside the timed step)."""
        flush.fill_(i & 0xff)
        torch.amax(flush_rd, dim=0, out=flush_out)
    stream = torch.cuda.current_stream()
    route_launches = 1 if moe.moe_route_meta_workspace_size(w.T, w.K, w.E) == 0 else 2
    # small batches: route + dispatch as one fused kernel (moe_route_dispatch)
    fused = not args.no_fuse and w.T <= 512 and w.T * w.K <= 4096

    def step():
        if fused:
            d.route_dispatch(x, ids, g)
        else:
            d.route(ids)
            d.dispatch(x, ids, g)
        d.combine(expert_out, ids, wt)

    # metadata facts for the byte model
    step()
    torch.cuda.synchronize()
    d.check()
    seg = d.seg_indptr.cpu().numpy()
    n_valid = int(seg[-1])
    n_rows = int(d.masked_m.sum().item()) if w.mode == "masked" else n_valid
    algo = algorithmic_bytes(w, n_valid, n_rows)

    def timed_step(i, e):
        """One step between events e[0] and e[3] (no event between its kernels)."""
        flush_l2(i)
        e[0].record(stream)
        if graph is not None:
            graph.replay()
        else:
            step()
        e[3].record(stream)

    def kernel_timed_step(i, e):
        """One eager step with an event after every kernel (e[1] route, e[2] dispatch)."""
        flush_l2(i)
        e[0].record(stream)
        if fused:
            d.route_dispatch(x, ids, g)
            e[2].record(stream)
        else:
            d.route(ids)
            e[1].record(stream)
            d.dispatch(x, ids, g)
            e[2].record(stream)
        d.combine(expert_out, ids, wt)
        e[3].record(stream)

    graph = None
    if args.graph:
        # one step (the library's launches only) captured once and replayed per step
        s2 = torch.cuda.Stream()
        s2.wait_stream(stream)
        with torch.cuda.stream(s2):
            step()
        stream.wait_stream(s2)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()

    for i in range(args.warmup):
        flush_l2(i)
        graph.replay() if graph is not None else step()
    def timed_pass(fn):
        """K steps bracketed by a barrier and a device synchronisation on both sides."""
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            fn(i, ev[i])
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        return ev

    # pass 1: the step time (an event between two kernels would stop the second one from
    # launching early under programmatic dependent launch, so none is recorded there)
    ev = timed_pass(timed_step)
    # pass 2: the same K steps, eager, with an event after every kernel: per-kernel durations
    ev_k = timed_pass(kernel_timed_step)
    # pass 3: one step captured as a CUDA graph, replayed K times after an L2 flush each (cold)
    # and K times back to back (warm: the step's working set may stay in L2)
    g_step = graph
    if g_step is None:
        s3 = torch.cuda.Stream()
        s3.wait_stream(stream)
        with torch.cuda.stream(s3):
            step()
        stream.wait_stream(s3)
        g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step):
            step()

    def graph_cold(i, e):
        flush_l2(i)
        e[0].record(stream)
        g_step.replay()
        e[3].record(stream)

    ev_g = timed_pass(graph_cold)
    for _ in range(args.warmup):
        g_step.replay()
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    w0.record(stream)
    for _ in range(args.steps):
        g_step.replay()
    w1.record(stream)
    torch.cuda.synchronize()
    d.check()
    ms_gc = max_over_ranks(statistics.mean(e[0].elapsed_time(e[3]) for e in ev_g), dist, dev)
    ms_gw = max_over_ranks(w0.elapsed_time(w1) / args.steps, dist, dev)
    graph_replay = {"cold_l2": {"ms_per_step": ms_gc, "value": job_throughput(w.T, world, ms_gc)},
                    "warm_l2": {"ms_per_step": ms_gw, "value": job_throughput(w.T, world, ms_gw)},
                    "timing": "one step captured as a CUDA graph; cold: L2 flushed before each replay; "
                              "warm: K replays back to back"}

    step_ms = [e[0].elapsed_time(e[3]) for e in ev]
    ms = max_over_ranks(statistics.mean(step_ms), dist, dev)
    ms_median = max_over_ranks(statistics.median(step_ms), dist, dev)
    value = job_throughput(w.T, world, ms)
    ms_k = max_over_ranks(statistics.mean(e[0].elapsed_time(e[3]) for e in ev_k), dist, dev)

    kernels = {}
    if fused:
        algo = {"route_dispatch": algo["route_meta"] + algo["dispatch"], "combine": algo["combine"]}
        spans = {"route_dispatch": (0, 2), "combine": (2, 3)}
    else:
        spans = {"route_meta": (0, 1), "dispatch": (1, 2), "combine": (2, 3)}
    for name, (a, b) in spans.items():
        us = 1e3 * max_over_ranks(statistics.mean(e[a].elapsed_time(e[b]) for e in ev_k), dist, dev)
        kernels[name] = {"us": us, "bytes": algo[name], "gbs": algo[name] / (us * 1e-6) / 1e9}
    peak, peak_kind = measured_hbm_gbs()
    roofline = None
    if kernels:
        dom = max(kernels, key=lambda k: kernels[k]["us"])
        ach = kernels[dom]["gbs"]
        roofline = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": peak, "unit": "GB/s",
                    "frac": ach / peak, "peak_source": f"{peak_kind} (hbm_gbs copy bandwidth)",
                    "frac_vs_8tbs": ach / NOMINAL_HBM_GBS,
                    "algorithmic_bytes_per_launch": algo[dom],
                    "traffic": profiled_traffic(dom, w.name)}
    step_bytes = sum(algo.values())

    # ---- end to end through the public API: pinned host in, host out ----
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, d, dev, x_h, ids_h, wt_h, g, fused, expert_out, dist)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded numpy PCG64 inputs, random expert outputs)",
        "dtypes": "f32 arithmetic (quantiser, combine accumulation) on bf16 rows; fp8 / nvfp4 / bf16 rows out; "
                  "int32 metadata",
        "ms_per_step_median": ms_median,
        "ms_per_step_with_kernel_events": ms_k,
        "graph_replay": graph_replay,
        "config": config_of(w),
        "timing": (("CUDA graph of one step, replayed per step" if graph is not None else "eager launches")
                   + ", CUDA events around each step; then K more eager steps with an event after every "
                     "kernel give the per-kernel durations; graph_replay: the step as a CUDA graph, cold "
                     "and warm L2"),
        "run": {"fused_route_dispatch": fused, "n_valid_pairs": n_valid, "rows_moved": n_rows},
        "achieved_gbs_step": step_bytes / (ms * 1e-3) / 1e9 / max(world, 1) * world,
        "frac_step": step_bytes / (ms * 1e-3) / 1e9 / peak,
        "frac_step_vs_8tbs": step_bytes / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
        "step_algorithmic_bytes": step_bytes,
        "kernels": kernels,
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": args.steps * ((1 if fused else route_launches + 1) + 1),
        "gpu_launches_kernel_pass": args.steps * ((1 if fused else route_launches + 1) + 1),
    }
    return line


# ---------------------------------------------------------------------------
# the NEXT rows (FlashInfer layout, dispatch layout, DeepGEMM formats, int64 ids, FP8
# pass-through): one timed call each, inputs in HBM, L2 flushed before every call
# ---------------------------------------------------------------------------

def run_next_rows(args):
    """One JSON line per NEXT-row call: median CUDA-event time of K calls after an L2 flush,
    the call's algorithmic bytes, GB/s and fraction of the measured copy bandwidth."""
    import torch
    import combine_moe_route_meta_gb300 as moe
    from workloads import make_workload

    dev = torch.device("cuda", 0)
    peak, peak_src = measured_hbm_gbs()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    flush_out = torch.empty((), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def timed_us(fn):
        for _ in range(args.warmup):
            fn()
        ev = []
        for i in range(args.steps):
            flush.fill_(i & 0xff)
            torch.amax(flush_rd, dim=0, out=flush_out)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            ev.append((a, b))
        torch.cuda.synchronize()
        return statistics.median(x.elapsed_time(y) for x, y in ev) * 1e3

    def emit(row, call, workload, T, us, nbytes, kernels, launches):
        gbs = nbytes / us / 1e3
        print(json.dumps({"row": row, "call": call, "workload": workload, "T": T, "us": us,
                          "tokens_per_s": T / us * 1e6, "algorithmic_bytes": nbytes, "gbs": gbs,
                          "peak": peak, "peak_source": peak_src, "frac": gbs / peak,
                          "kernels": kernels, "launches_per_call": launches,
                          "steps": args.steps, "warmup": args.warmup,
                          "l2": "flushed before every call"}), flush=True)

    def dev_in(w):
        x = torch.from_numpy(w.x.view(np.int16)).to(dev).view(torch.bfloat16)
        return x, torch.from_numpy(w.topk_ids).to(dev), torch.from_numpy(w.topk_weights).to(dev)

    st = moe.new_status(dev)
    only = {g for g in args.only.split(",") if g}
    want = lambda g: not only or g in only

    # f1: FlashInfer one-row-per-partition layout (the NVFP4 workload's tokens, 8 partitions,
    # one receive slot per token)
    if want("f1"):
        next_rows_f1(args, dev, st, timed_us, emit, dev_in)
    if want("f2"):
        next_rows_f2(dev, st, timed_us, emit)
    if want("f3f4"):
        next_rows_f3f4(dev, st, timed_us, emit, dev_in)
    if want("f3-swizzled"):
        next_rows_f3_swizzled(args, dev, st, timed_us, emit, dev_in)
    torch.cuda.synchronize()
    moe.check_status(st, "next rows")


def next_rows_f1(args, dev, st, timed_us, emit, dev_in):
    import torch
    import combine_moe_route_meta_gb300 as moe
    from workloads import make_workload
    w = make_workload("nvfp4", seed=0)
    x, ids, wt = dev_in(w)
    T, H, K, E, P = w.T, w.H, w.K, w.E, w.P
    S = T
    ep = E // P
    flat = w.topk_ids
    parts = np.zeros((T, P), bool)
    for k in range(K):
        e = flat[:, k]
        ok = (e >= 0) & (e < E)
        parts[np.nonzero(ok)[0], e[ok] // ep] = True
    routed = int(parts.sum())
    g = w.global_scale
    for quant, layout in (("nvfp4b16", "row"), ("nvfp4b16", "swizzled"), ("none", "row")):
        rx = torch.empty((P, S, H // 2 if quant == "nvfp4b16" else H),
                         dtype=torch.uint8 if quant == "nvfp4b16" else torch.bfloat16, device=dev)
        rsf = None
        if quant == "nvfp4b16":
            rsf = torch.empty((moe.swizzled_scale_bytes(P * S, H),) if layout == "swizzled" else (P, S, H // 16),
                              dtype=torch.uint8, device=dev)
        rids = torch.empty((P, S, K), dtype=torch.int32, device=dev)
        rw = torch.empty((P, S, K), dtype=torch.float32, device=dev)
        rb = row_bytes(quant, H)
        nbytes = 2 * T * H + 8 * T * K + P * S * 4 * K + routed * (rb + 4 * K)
        fn = lambda: moe.moe_dispatch_partitioned_ex(quant, layout, x, ids, wt, E, P, rx, rsf, rids, rw, st,
                                                     input_global_scale=g)
        us = timed_us(fn)
        emit("f1", f"moe_dispatch_partitioned_ex({quant}, {layout} scales)", "nvfp4", T, us, nbytes,
             ["dispatch_partitioned_tiles_kernel"] if layout == "swizzled" else
             (["dispatch_partitioned_ring_kernel"] if quant == "nvfp4b16" else ["dispatch_bulk_copy_kernel"]), 1)
        del rx, rsf, rids, rw
    partial = torch.randn((P, S, H), dtype=torch.bfloat16, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    us = timed_us(lambda: moe.moe_combine_partitioned(partial, ids, E, P, out, st))
    emit("f1", "moe_combine_partitioned", "nvfp4", T, us, routed * 2 * H + 4 * T * K + 2 * T * H,
         ["combine_partitioned_ring_kernel"], 1)
    del partial, out


def next_rows_f2(dev, st, timed_us, emit):
    import torch
    import combine_moe_route_meta_gb300 as moe
    from workloads import make_workload
    # f2: get_dispatch_layout outputs (decode and prefill routing, 8 partitions)
    for name in ("decode", "prefill"):
        w2 = make_workload(name, seed=0)
        ids2 = torch.from_numpy(w2.topk_ids).to(dev)
        P2 = 8
        ntr = torch.empty(P2, dtype=torch.int32, device=dev)
        itr = torch.empty((w2.T, P2), dtype=torch.uint8, device=dev)
        nte = torch.empty(w2.E, dtype=torch.int32, device=dev)
        us = timed_us(lambda: moe.moe_dispatch_layout(ids2, w2.E, P2, ntr, itr, st, nte))
        emit("f2", "moe_dispatch_layout", name, w2.T, us, 4 * w2.T * w2.K + w2.T * P2 + 4 * P2 + 4 * w2.E,
             ["dispatch_layout_kernel"], 1)


def next_rows_f3f4(dev, st, timed_us, emit, dev_in):
    import torch
    import combine_moe_route_meta_gb300 as moe
    from workloads import make_workload
    # f3 / f4 on the prefill workload: expert-aligned metadata from int64 ids, then the FP8
    # dispatch with UE8M0 column-major scales into the aligned segments; FP8 pass-through rows
    w = make_workload("prefill", seed=0)
    x, ids, wt = dev_in(w)
    T, H, K, E = w.T, w.H, w.K, w.E
    A = 128
    cap = T * K + E * (A - 1)
    ids64 = ids.to(torch.int64)
    seg = torch.empty(E + 1, dtype=torch.int64, device=dev)
    s2d = torch.empty(T * K, dtype=torch.int32, device=dev)
    reo = torch.empty(cap, dtype=torch.int32, device=dev)
    mm = torch.empty(E, dtype=torch.int32, device=dev)
    pc = torch.empty(8, dtype=torch.int32, device=dev)
    i32 = torch.empty((T, K), dtype=torch.int32, device=dev)
    ws = moe.new_workspace(T, K, E, dev)
    fn = lambda: moe.moe_route_meta_ex(ids64, E, seg, s2d, reo, mm, st, ws, 8, 0, A, pc, topk_ids_i32_out=i32)
    fn()
    torch.cuda.synchronize()
    n_rows = int(seg[-1].item())
    n_valid = int((s2d >= 0).sum().item())
    meta_bytes = 8 * T * K + 4 * T * K + 4 * T * K + 4 * n_rows + 8 * (E + 1) + 4 * E + 4 * 8
    emit("f3+f4", "moe_route_meta_ex(int64 ids, expert_alignment=128, int32 copy)", "prefill", T, timed_us(fn),
         meta_bytes, ["route_meta_count_kernel", "route_meta_place_kernel"], 2)
    q = torch.empty((cap, H), dtype=torch.uint8, device=dev)
    R4 = (cap + 3) // 4 * 4
    G = H // 128
    sc = torch.empty(((G + 3) // 4, R4, 4), dtype=torch.uint8, device=dev)
    fn = lambda: moe.moe_dispatch_ex("normal", "fp8g128_ue8m0", "col", x, i32, E, s2d, seg, q, sc, st, out_rows=cap)
    emit("f3", "moe_dispatch_ex(fp8g128_ue8m0, column-major scales, aligned segments)", "prefill", T,
         timed_us(fn), 2 * T * H + 4 * T * K + n_valid * (H + G), ["dispatch_bulk_quant_kernel"], 1)
    codes = torch.randint(0, 256, (T, H), dtype=torch.uint8, device=dev)
    om = moe.route_meta(ids, E, dev_status=st)
    fn = lambda: moe.moe_dispatch_ex("normal", "fp8_passthrough", "row", codes, ids, E, om.src2dst, om.seg_indptr,
                                     q, None, st)
    nv = int(om.seg_indptr[-1].item())
    emit("f4", "moe_dispatch_ex(fp8_passthrough)", "prefill", T, timed_us(fn), T * H + 4 * T * K + nv * H,
         ["dispatch_bulk_copy_kernel"], 1)
    del q, sc, codes


def next_rows_f3_swizzled(args, dev, st, timed_us, emit, dev_in):
    import torch
    import combine_moe_route_meta_gb300 as moe
    from workloads import make_workload
    # f3: NVFP4 masked dispatch with block scales written in the 128 x 4 swizzled layout
    w = make_workload("nvfp4", seed=0)
    x, ids, wt = dev_in(w)
    T, H, K, E, M = w.T, w.H, w.K, w.E, (args.masked_capacity or w.M)
    d = moe.MoEDispatcher(T, H, K, E, mode="masked", quant="nvfp4b16", num_partitions=w.P,
                          max_tokens_per_expert=M, device=dev)
    d.route(ids)
    torch.cuda.synchronize()
    rows = int(d.masked_m.sum().item())
    qm = torch.empty((E, M, H // 2), dtype=torch.uint8, device=dev)
    sfm = torch.empty((moe.swizzled_scale_bytes(E * M, H),), dtype=torch.uint8, device=dev)
    fn = lambda: moe.moe_dispatch_ex("masked", "nvfp4b16", "swizzled", x, ids, E, d.src2dst, d.seg_indptr, qm, sfm,
                                     st, M, input_global_scale=w.global_scale)
    emit("f3", "moe_dispatch_ex(nvfp4b16 masked, swizzled 128x4 scales)",
         "nvfp4" if M == w.M else f"nvfp4 (M={M})", T, timed_us(fn),
         2 * T * H + 8 * T * K + 8 * E + rows * row_bytes("nvfp4b16", H),
         ["dispatch_bulk_quant_kernel", "sf_tiles_interleave_kernel"], 2)


WORKLOAD_NAMES = ("tiny", "decode", "prefill", "qwen3", "nvfp4")


def summarise(ln: dict) -> dict:
    """The per_config entry of one workload's line: its config, step time and throughput, per-kernel
    times, roofline of the dominant kernel, graph replay, end to end and CPU baselines."""
    keep = ("config", "value", "unit", "ms_per_step", "ms_per_step_median", "achieved_gbs_step",
            "step_algorithmic_bytes", "kernels", "roofline", "graph_replay", "run", "gpu_launches",
            "cpu_baseline", "cpu_baseline_all_cores")
    keep += ("frac_step", "frac_step_vs_8tbs")
    out = {k: ln[k] for k in keep if k in ln}
    e2e = ln.get("e2e")
    if e2e:
        out["e2e"] = {k: e2e[k] for k in ("value", "unit", "ms_per_step", "h2d_bytes_per_step",
                                          "d2h_bytes_per_step", "schedule")}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="qwen3", choices=["tiny", "decode", "prefill", "qwen3", "nvfp4"])
    ap.add_argument("--per-config", default="decode,prefill,nvfp4",
                    help="other workloads measured in the same run (comma list, or 'none'); reported "
                         "under per_config")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--graph", action="store_true",
                    help="capture one step's launches in a CUDA graph and replay it (step time only)")
    ap.add_argument("--no-fuse", action="store_true", help="separate route_meta and dispatch calls")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--next-rows", action="store_true",
                    help="instead of the step: time each NEXT-row call (one JSON line per call)")
    ap.add_argument("--only", default="",
                    help="--next-rows: comma list of groups to run (f1, f2, f3f4, f3-swizzled); default all")
    ap.add_argument("--masked-capacity", type=int, default=0,
                    help="--next-rows: slots per expert M of the masked NVFP4 row (default: the workload's "
                         "8192; a smaller M moves the same rows with smaller buffers, e.g. for a profiler)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from workloads import make_workload

    if args.impl == "reference":
        w = make_workload(args.workload, seed=0)
        line = run_reference(args, w, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch
    dist = None
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
    else:
        torch.cuda.set_device(0)

    from combine_moe_route_meta_gb300 import build as _build
    if rank == 0 or not _build.up_to_date():
        _build.build()
    if dist:
        dist.barrier()

    if args.next_rows:
        if rank == 0:
            run_next_rows(args)
        if dist:
            dist.barrier()
            dist.destroy_process_group()
        return

    others = [n for n in args.per_config.split(",") if n and n != "none" and n != args.workload]
    for n in others:
        if n not in WORKLOAD_NAMES:
            raise SystemExit(f"--per-config: unknown workload {n!r}")

    def one(name, budget):
        w = make_workload(name, seed=rank_seed(rank))
        cpu = cpu_all = None
        if world == 1 and not args.no_cpu_baseline:
            cpu = cpu_baseline(w, budget)
            cpu_all = cpu_baseline_all_cores(w, budget * 0.8)
        ln = run_gpu(args, w, rank, world, dist)
        ln["cpu_baseline"] = cpu
        ln["cpu_baseline_all_cores"] = cpu_all
        del w
        torch.cuda.empty_cache()
        return ln

    # one clock sampler over every timed region of the run (headline and per_config)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    line = one(args.workload, 12.0)
    per = {n: summarise(one(n, 5.0)) for n in others}
    clocks = sampler.stop()
    line["clocks"] = clocks
    if per:
        line["per_config"] = per
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
