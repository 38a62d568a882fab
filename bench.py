#!/usr/bin/env python3
"""Benchmark: MoE route top-k -> dispatch count -> dispatch pack -> combine.

One step is one pass of the whole routing path over one batch of the
DeepSeek-V3-shaped decode workload (N=32 ranks x T=128 tokens, E=256, R=8,
H=7168 bf16), with the inputs already in HBM.  The expert op between pack
and combine stands in for the grouped expert GEMM and is not timed; in its
place the L2 is flushed (a GPU-side read of 2x the L2 size), as it is
before every step, so no kernel reads data a previous kernel left in L2.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on
the host cores instead (bounded samples of the same workload).
With N > 1 (torchrun) every rank runs an independent replica: the path has
no exchange step across GPUs, so value = N * tokens / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dispatch+combine tokens/s and achieved HBM GB/s (fraction of GB300 peak), 1 GPU"
DEFAULT_WORKLOAD = "dsv3_decode"
KERNELS = ("route", "count", "pack", "combine")
KERNEL_SOURCES = {"route": "route_topk.cu", "count": "dispatch_count.cu",
                  "pack": "dispatch_pack.cu", "combine": "combine.cu"}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--e2e-steps", type=int, default=100)
    p.add_argument("--e2e-lanes", type=int, default=3,
                   help="independent buffer sets the end-to-end steps alternate between")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="CPU work for the oracle baseline (0 disables it)")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--tokens-per-rank", type=int, default=0,
                   help="T of the workload (0: its own); a smaller batch of the same shape, for "
                        "profiling captures that must stay small")
    p.add_argument("--no-extras", action="store_true",
                   help="time the step and its breakdown only (no graphs, variants, end-to-end "
                        "run or other workloads)")
    p.add_argument("--no-other-workloads", dest="other_workloads", action="store_false",
                   help="leave out the table of the other workloads")
    p.add_argument("--workload-steps", type=int, default=100,
                   help="timed steps per workload of the workloads table")
    p.add_argument("--cap-rows", type=int, default=0,
                   help="per-rank receive capacity (0: the bound N*T*max(R,E/N)); a smaller "
                        "capacity shrinks the allocation, not the work")
    return p.parse_args()


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def dist_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def reduce_max(value: float, dist=None) -> float:
    """Max of `value` over all ranks (the slowest replica sets the step
    time).  Works with NCCL (CUDA tensor) and gloo (CPU tensor)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_replica: int, world: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every replica processes its own batch per step."""
    return world * tokens_per_replica / (ms_per_step / 1e3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# headers that only declare host functions: of these, only the macro
# definitions (status codes, dtypes, flags) can change a kernel
DECLARATION_HEADERS = ("moe_internal.cuh", "moe_route.h")


def source_hash(name: str) -> str:
    """Hash of a kernel source file and every local header it includes (the
    declaration headers through their #define lines only)."""
    dirs = [os.path.join(ROOT, "combine_moe_route_topk_gb300", "csrc"), os.path.join(ROOT, "include")]
    h = hashlib.sha256()
    todo, seen = [name], set()
    while todo:
        f = todo.pop(0)
        path = next((os.path.join(d, f) for d in dirs if os.path.exists(os.path.join(d, f))), None)
        if f in seen or path is None:
            continue
        seen.add(f)
        with open(path, "rb") as fh:
            data = fh.read()
        part = data
        if f in DECLARATION_HEADERS:
            part = b"\n".join(l for l in data.splitlines() if l.lstrip().startswith(b"#define")
                              and not re.match(rb"\s*#define\s+MOE_VERSION\b", l))
        h.update(f.encode() + b"\0" + part)
        todo += [m.decode() for m in re.findall(rb'#include "([^"]+)"', data)]
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current source of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_sha256_16") != source_hash(KERNEL_SOURCES[kernel]):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled in the background."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def wait_first(self, timeout=10.0):
        t0 = time.time()
        while self.proc is not None and not self.samples and time.time() - t0 < timeout:
            time.sleep(0.02)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [s for (t, s) in self.samples if t0 <= t <= t1 and len(s) >= 9]
        if not rows:  # very short window: take the samples closest to it
            rows = [s for (t, s) in self.samples if t0 - 0.5 <= t <= t1 + 0.5 and len(s) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][2]), "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# --------------------------------------------------------------------------
# CPU oracle timing (baseline / reference arm)
# --------------------------------------------------------------------------

def oracle_pass(w, inp, tokens=None, phases=None):
    """One oracle pass of route -> count -> pack -> combine (identity expert)
    over the whole batch, or over the first `tokens` tokens treated as a
    smaller batch of the same shape (T' = tokens / N per rank).  With a
    `phases` dict, the seconds of each step are added to it."""
    import numpy as np
    import oracle
    logits, bias = inp.logits.numpy(), None if inp.bias is None else inp.bias.numpy()
    xb = oracle.x_as_bytes(inp.x)
    T = w.T
    if tokens is not None:
        T = max(1, tokens // w.N)
        logits, xb = logits[:w.N * T], xb[:w.N * T]
    t = [time.perf_counter()]
    idx, tw, _ = oracle.route(logits, bias, w.R, w.score_fn, w.renormalize)
    t.append(time.perf_counter())
    cap = w.N * T * max(w.R, w.E // w.N)
    cnt, _ = oracle.count(w.N, T, w.E, cap, idx)
    t.append(time.perf_counter())
    px, _, _ = oracle.pack(xb, None, cnt["pos"], cnt["rank_offsets"], cap)
    t.append(time.perf_counter())
    y = px.view(np.uint16) if w.y_dtype == 0 else px.view(np.float32)
    oracle.combine(y, w.y_dtype, cnt["pos"], cnt["rank_offsets"], tw, cap, w.H)
    t.append(time.perf_counter())
    if phases is not None:
        for k, a, b in zip(KERNELS, t, t[1:]):
            phases[k] = phases.get(k, 0.0) + (b - a)
    return w.N * T


def cpu_baseline(w, inp, seconds):
    n_tok, passes, phases = 0, 0, {}
    t0 = time.perf_counter()
    while True:
        n_tok += oracle_pass(w, inp, phases=phases)
        passes += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": n_tok / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "phase_ms_per_pass": {k: v / passes * 1e3 for k, v in phases.items()},
            "sample": f"{passes} full pass(es) of the {w.name} batch ({w.NT} tokens): "
                      f"route, count, pack, combine; single-threaded C, {dt:.1f} s"}


def run_reference(args):
    rank, _, world = dist_info()
    if rank != 0:
        return 0
    import torch  # noqa: F401  (seeded generator)
    from combine_moe_route_topk_gb300 import workloads as W
    import oracle
    oracle.build_lib()
    w = W.WORKLOADS[args.workload]
    inp = W.make_inputs(w)
    # size the sample so the whole run stays within ~2 minutes
    probe = 256
    t0 = time.perf_counter()
    oracle_pass(w, inp, probe)
    per_tok = (time.perf_counter() - t0) / probe
    budget = 120.0 / max(1, args.steps + args.warmup)
    sample = int(min(w.NT, max(w.N, (budget / per_tok) // w.N * w.N)))
    for _ in range(args.warmup):
        oracle_pass(w, inp, sample)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        n = oracle_pass(w, inp, sample)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    value = n / (ms / 1e3)
    desc = (f"batches of {n} tokens ({n // w.N} per rank) of the {w.name} shape: route, count, "
            f"pack, combine; single-threaded C oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))
    return 0


def workload_config(w):
    from combine_moe_route_topk_gb300 import workloads as W
    return {"workload": w.name, "N": w.N, "T": w.T, "tokens": w.NT, "E": w.E, "R": w.R,
            "H": w.H, "x_dtype": {0: "bf16", 1: "f32", 2: "fp8e4m3+f32/128"}[w.x_dtype],
            "scores": ("softmax" if w.score_fn == W.SOFTMAX else "sigmoid")
                      + ("+renorm" if w.renormalize else ""),
            "cap_rows_per_rank": W.default_cap(w),
            "l2": "flushed before every step and between pack and combine by reading a 2x L2 "
                  "buffer (untimed; evicts everything, leaves clean lines)",
            "expert_op": "not timed (stands in for the grouped expert GEMM)",
            "parallelism": "replicas"}


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

class nvtx_range:
    """NVTX range around a part of the run (lets a profiler select, e.g., the
    launches of the timed region); does nothing where NVTX is unavailable."""

    def __init__(self, name):
        self.name = name

    def __enter__(self):
        try:
            import torch
            torch.cuda.nvtx.range_push(self.name)
            self.ok = True
        except Exception:
            self.ok = False
        return self

    def __exit__(self, *exc):
        if self.ok:
            import torch
            torch.cuda.nvtx.range_pop()
        return False


def new_events(n):
    import torch
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def mean_interval(pairs):
    return statistics.mean(a.elapsed_time(b) for a, b in pairs)


class PathRunner:
    """One workload on one GPU: its seeded inputs in HBM, its buffers, and the
    four calls of the path.  The expert op between pack and combine stands in
    for the grouped expert GEMM and is not run: combine reads y as pack left
    it (identity) or as it was zeroed once (a separate y)."""

    def __init__(self, moe, W, w, dev, stream, flush):
        self.moe, self.w, self.dev, self.stream, self.flush = moe, w, dev, stream, flush
        self.dims = moe.dims_of(w)
        self.inp_cpu = W.make_inputs(w)
        self.inp = W.Inputs(*(t.to(dev) if t is not None else None
                              for t in (self.inp_cpu.logits, self.inp_cpu.bias, self.inp_cpu.x,
                                        self.inp_cpu.x_scales)))
        self.b = moe.Buffers(self.dims, device=dev,
                             separate_y=False if w.x_dtype == w.y_dtype else None)
        if self.b.y.data_ptr() != self.b.packed_x.data_ptr():
            self.b.y.zero_()

    def launch(self, k, s=None):
        moe, w, b, inp, dims = self.moe, self.w, self.b, self.inp, self.dims
        s = self.stream if s is None else s
        if k == "route":
            moe.route_topk(dims, inp.logits, inp.bias, w.score_fn, w.renormalize, b.topk_idx,
                           b.topk_w, s)
        elif k == "count":
            moe.dispatch_count(dims, b.topk_idx, b.expert_counts, b.expert_offsets,
                               b.rank_counts, b.rank_offsets, b.send_counts, b.pos, b.status, s)
        elif k == "pack":
            moe.dispatch_pack(dims, inp.x, inp.x_scales, b.pos, b.packed_x, b.packed_scales,
                              b.packed_src, s)
        else:
            moe.combine(dims, b.y, b.pos, b.topk_w, b.out, s)

    def step(self, ev):
        """dispatch (route -> count -> pack back to back, so each launch
        overlaps the tail of the previous kernel), the expert-op stand-in (an
        L2 flush, untimed), combine, and the L2 flush before the next step.
        Events: [0] dispatch [1] flush [2] combine [3] flush [4]."""
        st = self.stream
        ev[0].record(st)
        self.launch("route")
        self.launch("count")
        self.launch("pack")
        ev[1].record(st)
        self.flush()
        ev[2].record(st)
        self.launch("combine")
        ev[3].record(st)
        self.flush()
        ev[4].record(st)

    def check_status(self):
        st = self.moe.read_status(self.b.status, self.stream)
        if st != self.moe.MOE_OK:
            raise SystemExit(f"dispatch_count status {self.moe.STATUS_NAMES.get(st, st)} on {self.w.name}")

    def steps(self, n):
        """n steps, each self-contained (it ends with the flush the next one
        starts after).  Returns the per-step events."""
        evs = [new_events(5) for _ in range(n)]
        for e in evs:
            self.step(e)
        return evs

    def clean_flush_ms(self, n):
        """An L2 flush on an L2 that holds only clean lines (the previous
        flush's): the baseline that the flushes inside a step are compared
        with, to charge the write-back of the dirty lines a kernel left."""
        pool = [new_events(2) for _ in range(n)]
        self.flush()
        for e in pool:
            e[0].record(self.stream)
            self.flush()
            e[1].record(self.stream)
        import torch
        torch.cuda.synchronize(self.dev)
        return mean_interval(pool)

    def breakdown(self, n, host_lead):
        """Per-kernel times: an event between every two kernels (the events
        serialise the launches, so these sum to a little more than a step);
        and route -> count back to back, what the dispatch segment spends
        before pack's own work."""
        import torch
        st = self.stream
        pool = [new_events(6) for _ in range(n)]
        host_lead(n)
        for ev in pool:
            self.flush()
            ev[0].record(st)
            for i, k in enumerate(("route", "count", "pack")):
                self.launch(k)
                ev[i + 1].record(st)
            self.flush()
            ev[4].record(st)
            self.launch("combine")
            ev[5].record(st)
        rc = [new_events(2) for _ in range(n)]
        host_lead(n)
        for e in rc:
            self.flush()
            e[0].record(st)
            self.launch("route")
            self.launch("count")
            e[1].record(st)
        torch.cuda.synchronize(self.dev)
        per = {"route": [e[0].elapsed_time(e[1]) for e in pool],
               "count": [e[1].elapsed_time(e[2]) for e in pool],
               "pack": [e[2].elapsed_time(e[3]) for e in pool],
               "combine": [e[4].elapsed_time(e[5]) for e in pool]}
        return per, mean_interval(rc)

    def timed_repeat(self, fn, n, host_lead):
        """Mean event time of fn() run alone after an L2 flush, n times."""
        import torch
        pool = [new_events(2) for _ in range(n + 3)]
        host_lead(n + 3)
        for e in pool:
            self.flush()
            e[0].record(self.stream)
            fn()
            e[1].record(self.stream)
        torch.cuda.synchronize(self.dev)
        return mean_interval(pool[3:])

    def fused_ms(self, n, host_lead):
        """moe_dispatch_fused on the same batch, or why it does not take it."""
        import torch
        moe, w, b, inp, dims = self.moe, self.w, self.b, self.inp, self.dims
        try:
            ws = torch.zeros(moe.buffer_sizes(dims)["fused_workspace_bytes"], dtype=torch.uint8,
                             device=self.dev)

            def call():
                moe.dispatch_fused(dims, inp.logits, inp.bias, w.score_fn, w.renormalize, inp.x,
                                   inp.x_scales, b.topk_idx, b.topk_w, b.expert_counts,
                                   b.expert_offsets, b.rank_counts, b.rank_offsets,
                                   b.send_counts, b.pos, b.status, b.packed_x, b.packed_scales,
                                   b.packed_src, ws, self.stream)
            ms = self.timed_repeat(call, n, host_lead)
            if moe.read_status(b.status, self.stream) != moe.MOE_OK:
                raise RuntimeError("fused dispatch status")
            return {"ms": ms}
        except moe.MoeError as ex:
            return {"unsupported": str(ex)}

    def ep_local(self, n, host_lead, rank=0):
        """The expert-parallel local path of one rank: rank-restricted pack,
        then (after an L2 flush) its local accumulation; events around each."""
        import torch
        moe, w, b, inp, dims = self.moe, self.w, self.b, self.inp, self.dims
        from combine_moe_route_topk_gb300 import workloads as W
        # the default routing in place
        self.launch("route")
        self.launch("count")
        self.launch("pack")
        torch.cuda.synchronize(self.dev)
        cap = moe.buffer_sizes(dims)["cap_rows"]
        rows = int(b.rank_counts[rank].item())
        toks = int(((b.pos >= rank * cap) & (b.pos < (rank + 1) * cap)).any(dim=1).sum().item())
        out2 = torch.empty_like(b.out)
        pool = [(new_events(2), new_events(2)) for _ in range(n + 3)]
        host_lead(n + 3)
        for e, e2 in pool:
            self.flush()
            e[0].record(self.stream)
            moe.dispatch_pack_rank(dims, rank, inp.x, inp.x_scales, b.pos, b.packed_x,
                                   b.packed_scales, b.packed_src, self.stream)
            e[1].record(self.stream)
            self.flush()
            e2[0].record(self.stream)
            moe.combine_rank(dims, rank, b.y, b.pos, b.topk_w, out2, self.stream)
            e2[1].record(self.stream)
        torch.cuda.synchronize(self.dev)
        t_pr = mean_interval([e for e, _ in pool[3:]])
        t_cr = mean_interval([e2 for _, e2 in pool[3:]])
        del out2
        rb, yb = W.row_bytes(w), W.y_row_bytes(w)
        sb = 4 * (w.H // 128) if w.x_dtype == W.FP8E4M3_BLK128 else 0
        b_pr = toks * (rb + sb) + rows * (rb + sb) + rows * 4 + w.NT * w.R * 4
        b_cr = rows * yb + w.NT * yb + w.NT * w.R * 8
        peak = measured_peaks()[0]
        return {"rank": rank, "rows": rows, "tokens": toks,
                "pack_rank_ms": t_pr, "pack_rank_alg_bytes": b_pr,
                "pack_rank_alg_gbs": b_pr / (t_pr / 1e3) / 1e9,
                "pack_rank_frac": b_pr / (t_pr / 1e3) / 1e9 / peak,
                "combine_rank_ms": t_cr, "combine_rank_alg_bytes": b_cr,
                "combine_rank_alg_gbs": b_cr / (t_cr / 1e3) / 1e9,
                "combine_rank_frac": b_cr / (t_cr / 1e3) / 1e9 / peak}

    def free(self):
        del self.b, self.inp


def roofline_of(w, kern, launch_ms, writeback_ms, peak, peak_kind):
    """Roofline entry of the dominant kernel (the slower of pack and combine by
    median): algorithmic bytes over its mean event time; the DRAM-level
    fraction from the committed ncu traffic of the same source; and the
    fraction with the write-back of its dirty L2 lines charged to it."""
    from combine_moe_route_topk_gb300 import workloads as W
    alg = W.algorithmic_bytes(w)
    dom = max(("pack", "combine"), key=lambda k: kern[k]["median_ms"])
    ms = launch_ms[dom]
    achieved = alg[dom] / (ms / 1e3) / 1e9
    traffic = ncu_traffic(dom, w.name)
    wb = max(0.0, writeback_ms[dom])
    r = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
         "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
         if peak_kind == "measured" else "fallback 6.8 TB/s",
         "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
         "frac_dram": None if traffic is None else traffic / (ms / 1e3) / 1e9 / peak,
         "frac_with_writeback": alg[dom] / ((ms + wb) / 1e3) / 1e9 / peak,
         "alg_bytes_per_launch": alg[dom], "launch_ms": ms, "writeback_ms": wb}
    return r


def measure_workload(runner, steps, nb, host_lead, sampler_window=None):
    """The step, its per-kernel breakdown, the write-back of the dirty lines
    pack and combine leave in L2, and the fused and expert-parallel local
    variants, for one workload: the entry of the `workloads` table."""
    import torch
    w = runner.w
    from combine_moe_route_topk_gb300 import workloads as W
    runner.flush()
    runner.steps(3)
    runner.check_status()
    torch.cuda.synchronize(runner.dev)
    host_lead(steps)
    evs = runner.steps(steps)
    torch.cuda.synchronize(runner.dev)
    runner.check_status()
    disp = [e[0].elapsed_time(e[1]) for e in evs]
    comb = [e[2].elapsed_time(e[3]) for e in evs]
    fl_p = [e[1].elapsed_time(e[2]) for e in evs]
    fl_c = [e[3].elapsed_time(e[4]) for e in evs]
    clean = runner.clean_flush_ms(nb)
    per, rc_ms = runner.breakdown(nb, host_lead)
    alg = W.algorithmic_bytes(w)
    peak, peak_kind = measured_peaks()
    kern = {k: {"ms": statistics.mean(v), "median_ms": statistics.median(v),
                "alg_gbs": alg[k] / (statistics.mean(v) / 1e3) / 1e9} for k, v in per.items()}
    step_ms = statistics.mean(a + c for a, c in zip(disp, comb))
    wb = {"pack": statistics.mean(fl_p) - clean, "combine": statistics.mean(fl_c) - clean}
    launch_ms = {"pack": kern["pack"]["ms"], "combine": statistics.mean(comb)}
    pc_ms = launch_ms["pack"] + launch_ms["combine"]
    pc_gbs = (alg["pack"] + alg["combine"]) / (pc_ms / 1e3) / 1e9
    pc_wb_ms = pc_ms + max(0.0, wb["pack"]) + max(0.0, wb["combine"])
    pc_wb_gbs = (alg["pack"] + alg["combine"]) / (pc_wb_ms / 1e3) / 1e9
    entry = {
        "config": {"N": w.N, "T": w.T, "tokens": w.NT, "E": w.E, "R": w.R, "H": w.H,
                   "x_dtype": {0: "bf16", 1: "f32", 2: "fp8e4m3+f32/128"}[w.x_dtype]},
        "steps": steps, "ms_per_step": step_ms, "tokens_per_s": w.NT / (step_ms / 1e3),
        "dispatch_ms": statistics.mean(disp), "combine_ms": statistics.mean(comb),
        "route_count_chain_ms": rc_ms,
        "kernels": kern,
        "pack_plus_combine": {"ms": pc_ms, "alg_gbs": pc_gbs, "frac": pc_gbs / peak,
                              "ms_with_writeback": pc_wb_ms,
                              "frac_with_writeback": pc_wb_gbs / peak},
        "writeback_ms": {"after_pack": wb["pack"], "after_combine": wb["combine"],
                         "clean_flush_ms": clean,
                         "note": "L2 flush right after the kernel minus a flush of an L2 "
                                 "holding only clean lines: the write-back of the dirty "
                                 "lines the kernel left, which the step does not time"},
        "step_with_writeback_ms": step_ms + max(0.0, wb["pack"]) + max(0.0, wb["combine"]),
        "roofline": roofline_of(w, kern, launch_ms, wb, peak, peak_kind),
    }
    entry["fused_dispatch"] = runner.fused_ms(nb, host_lead)
    entry["ep_local_rank0"] = runner.ep_local(nb, host_lead)
    return entry, (disp, comb, fl_p, fl_c, clean, per, rc_ms)


def run_ours(args):
    import torch
    import combine_moe_route_topk_gb300 as moe
    from combine_moe_route_topk_gb300 import workloads as W

    rank, local_rank, world = dist_info()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    moe.lib()  # fails loudly if the library was not built

    w = W.WORKLOADS[args.workload]
    if args.tokens_per_rank:
        w = w.replace(T=args.tokens_per_rank)
    if args.cap_rows:
        w = w.replace(cap_rows=args.cap_rows)
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    # L2 flush: read a buffer twice the L2 size.  Every line a step left in
    # L2 is evicted (dirty ones are written back during the flush, outside
    # the timed segments) and the L2 is left holding clean lines, so no
    # kernel pays for write-backs of the flush itself.
    flush_buf = torch.zeros(2 * l2 // 4, dtype=torch.float32, device=dev)
    flush_out = torch.zeros((), dtype=torch.float32, device=dev)

    def flush():
        torch.sum(flush_buf, dim=0, out=flush_out)

    def host_lead(iters):
        # The loops after the timed region bracket single short kernels with
        # events, and Python needs tens of microseconds per call: a GPU sleep
        # long enough for the host to enqueue the whole loop first keeps that
        # host time out of every interval.
        sleep = getattr(torch.cuda, "_sleep", None)  # a private helper of torch
        if sleep is not None:
            sleep(int(iters * 150e-6 * 2.0e9))

    run = PathRunner(moe, W, w, dev, stream, flush)
    dims, b, inp, inp_cpu = run.dims, run.b, run.inp, run.inp_cpu
    launch = run.launch

    flush()
    run.steps(max(3, args.warmup))
    run.check_status()

    sampler = None if args.no_clocks else ClockSampler(local_rank)
    if sampler is not None:
        sampler.wait_first()
    evs = [new_events(5) for _ in range(args.steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    with nvtx_range("timed"):
        for e in evs:
            run.step(e)
        torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    t_wall1 = time.time()
    clocks = None
    if sampler is not None:
        time.sleep(0.05)
        sampler.stop()
        clocks = sampler.summary(t_wall0, t_wall1)
    run.check_status()

    dispatch_ms = [e[0].elapsed_time(e[1]) for e in evs]
    combine_ms = [e[2].elapsed_time(e[3]) for e in evs]
    step_ms = [a + c for a, c in zip(dispatch_ms, combine_ms)]
    ms = reduce_max(statistics.mean(step_ms), pg)
    value = job_throughput(w.NT, world, ms)
    fl_pack = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    fl_comb = statistics.mean(e[3].elapsed_time(e[4]) for e in evs)

    # ---- after the timed region: breakdown, write-back, variants ---------
    nb = max(10, min(args.steps, 200))
    clean = run.clean_flush_ms(nb)
    wb = {"pack": fl_pack - clean, "combine": fl_comb - clean}
    per, route_count_chain_ms = run.breakdown(nb, host_lead)
    per_timed = {"dispatch (route+count+pack)": statistics.mean(dispatch_ms),
                 "combine": statistics.mean(combine_ms),
                 "route+count alone, back to back (diagnostic)": route_count_chain_ms}
    step_wb_ms = reduce_max(statistics.mean(step_ms) + max(0.0, wb["pack"]) + max(0.0, wb["combine"]), pg)

    with nvtx_range("ep_local"):
        ep_main = run.ep_local(nb, host_lead)
    ep_main["note"] = ("moe_dispatch_pack_rank + moe_combine_rank for rank 0 (the all-reduce "
                       "over ranks that completes it is not part of the library)")
    graph_replay = extra = e2e = None
    if not args.no_extras:
        graph_replay = graph_replay_of(args, run, host_lead, pg, world)
        extra = variants_of(args, run, nb, host_lead, per_timed)
        extra["next_rows"]["ep_local_rank0"] = ep_main
        e2e = run_e2e(args, w, dims, inp_cpu, b, dev, stream, flush, moe)

    alg = W.algorithmic_bytes(w)
    peak, peak_kind = measured_peaks()
    kern = {}
    for k in KERNELS:
        mean_ms = statistics.mean(per[k])
        kern[k] = {"ms": mean_ms, "median_ms": statistics.median(per[k]),
                   "alg_bytes": alg[k], "alg_gbs": alg[k] / (mean_ms / 1e3) / 1e9}
    # combine has its own events inside the timed region; pack's come from
    # the breakdown pass right after it
    launch_ms = {"pack": kern["pack"]["ms"], "combine": per_timed["combine"]}
    roofline = roofline_of(w, kern, launch_ms, wb, peak, peak_kind)
    pc_ms = launch_ms["pack"] + launch_ms["combine"]
    pc_gbs = (alg["pack"] + alg["combine"]) / (pc_ms / 1e3) / 1e9
    pc_wb_ms = pc_ms + max(0.0, wb["pack"]) + max(0.0, wb["combine"])
    pc_wb_gbs = (alg["pack"] + alg["combine"]) / (pc_wb_ms / 1e3) / 1e9

    # ---- the other workloads, each on its own buffers ---------------------
    workloads = None
    if not args.no_extras and args.other_workloads:
        run.free()
        del run, b, inp
        torch.cuda.empty_cache()
        workloads = {}
        wsampler = None if args.no_clocks else ClockSampler(local_rank)
        if wsampler is not None:
            wsampler.wait_first()
        tw0 = time.time()
        for name in W.WORKLOADS:
            if name == w.name:
                continue
            r2 = PathRunner(moe, W, W.WORKLOADS[name], dev, stream, flush)
            entry, _ = measure_workload(r2, args.workload_steps, max(10, min(args.workload_steps, 50)),
                                        host_lead)
            workloads[name] = entry
            r2.free()
            del r2
            torch.cuda.empty_cache()
        if wsampler is not None:
            time.sleep(0.05)
            wsampler.stop()
            workloads["clocks"] = wsampler.summary(tw0, time.time())

    if rank != 0:
        return 0
    cpu = None
    if world == 1 and args.cpu_seconds > 0:
        import oracle
        oracle.build_lib()
        cpu = cpu_baseline(w, inp_cpu, args.cpu_seconds)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "io_dtype": "bf16", "data": "synthetic", "config": workload_config(w),
        "gpu_launches": 4 * args.steps,
        "roofline": roofline,
        "pack_plus_combine": {"ms": pc_ms, "alg_gbs": pc_gbs, "frac": pc_gbs / peak,
                              "frac_of_8tbs_nominal": pc_gbs / 8000.0,
                              "ms_with_writeback": pc_wb_ms,
                              "frac_with_writeback": pc_wb_gbs / peak},
        "step_with_writeback_ms": step_wb_ms,
        "writeback_ms": {"after_pack": wb["pack"], "after_combine": wb["combine"],
                         "clean_flush_ms": clean,
                         "note": "the L2 flush that follows pack (and combine) inside every "
                                 "step, minus a flush of an L2 holding only clean lines: the "
                                 "write-back of the dirty lines the kernel left in L2, which "
                                 "the timed segments do not include; step_with_writeback_ms "
                                 "charges it"},
        "timed_segments_ms": per_timed,
        "graph_replay": graph_replay,
        "kernels": kern,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "wall_s_timed_region": t_wall1 - t_wall0,
    }
    if extra is not None:
        line.update(extra)
    else:
        line["next_rows"] = {"ep_local_rank0": ep_main}
    if workloads is not None:
        line["workloads"] = workloads
    print(json.dumps(line))
    return 0


def graph_replay_of(args, run, host_lead, pg, world):
    """The same step replayed from CUDA graphs, as a serving loop runs it:
    dispatch (route -> count -> pack, with their programmatic-dependency
    edges) and combine captured once each, the L2 flush between replays."""
    import torch
    dev, stream, flush = run.dev, run.stream, run.flush
    cap_stream = torch.cuda.Stream(dev)
    g_disp, g_comb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    cap_stream.wait_stream(stream)
    with torch.cuda.graph(g_disp, stream=cap_stream):
        for k in ("route", "count", "pack"):
            run.launch(k, cap_stream)
    with torch.cuda.graph(g_comb, stream=cap_stream):
        run.launch("combine", cap_stream)
    stream.wait_stream(cap_stream)
    n_g = args.steps + max(3, args.warmup)
    gpool = [new_events(4) for _ in range(n_g)]
    gevs = []
    host_lead(n_g)
    for i in range(n_g):
        flush()
        e = gpool[i]
        e[0].record(stream)
        g_disp.replay()
        e[1].record(stream)
        flush()
        e[2].record(stream)
        g_comb.replay()
        e[3].record(stream)
        if i >= max(3, args.warmup):
            gevs.append(e)
    torch.cuda.synchronize(dev)
    run.check_status()
    g_step = [e[0].elapsed_time(e[1]) + e[2].elapsed_time(e[3]) for e in gevs]
    g_ms = reduce_max(statistics.mean(g_step), pg)
    del g_disp, g_comb
    return {"ms_per_step": g_ms, "median_ms_per_step": statistics.median(g_step),
            "dispatch_ms": statistics.mean(e[0].elapsed_time(e[1]) for e in gevs),
            "combine_ms": statistics.mean(e[2].elapsed_time(e[3]) for e in gevs),
            "value": job_throughput(run.w.NT, world, g_ms), "replays": len(gevs),
            "note": "two CUDA graphs (dispatch, combine) replayed per step"}


def variants_of(args, run, nb, host_lead, per_timed):
    """The quantising pack, the decode-fused dispatch, the bias-for-selection
    router, the send-side combine and the expert-parallel local path, each on
    the headline batch."""
    import torch
    moe, w, b, inp, dims, dev, stream = run.moe, run.w, run.b, run.inp, run.dims, run.dev, run.stream
    from combine_moe_route_topk_gb300 import workloads as W
    out = {}

    # the quantising pack (bf16 rows -> e4m3 + per-128 scales), timed alone
    # on the same routing; it replaces pack when the experts take fp8 input
    quant = None
    if w.x_dtype == W.BF16 and w.H % 128 == 0:
        qs = moe.buffer_sizes(moe.fp8_dims(dims))
        pq = torch.empty(qs["packed_x_bytes"], dtype=torch.uint8, device=dev)
        ps = torch.empty(qs["packed_scales_bytes"] // 4, dtype=torch.float32, device=dev)

        def qpack():
            moe.dispatch_pack_quant(dims, inp.x, b.pos, pq, ps, b.packed_src, stream)

        def chain():
            run.launch("route")
            run.launch("count")
            qpack()
        with nvtx_range("pack_quant"):
            qm = run.timed_repeat(qpack, nb, host_lead)
        cm = run.timed_repeat(chain, nb, host_lead)
        # the same fp8 dispatch as one call (decode batches only)
        fused_fp8 = None
        try:
            ws = torch.zeros(max(16, moe.buffer_sizes(dims)["fused_workspace_bytes"]), dtype=torch.uint8,
                             device=dev)

            def fused_q():
                moe.dispatch_fused_quant(dims, inp.logits, inp.bias, w.score_fn, w.renormalize, inp.x,
                                         b.topk_idx, b.topk_w, b.expert_counts, b.expert_offsets,
                                         b.rank_counts, b.rank_offsets, b.send_counts, b.pos, b.status,
                                         pq, ps, b.packed_src, ws, stream)
            with nvtx_range("fused_quant"):
                fused_fp8 = run.timed_repeat(fused_q, nb, host_lead)
            if moe.read_status(b.status, stream) != moe.MOE_OK:
                raise RuntimeError("fused fp8 dispatch status")
        except moe.MoeError:
            fused_fp8 = None
        qbytes = w.NT * (2 * w.H + w.R * (w.H + 4 * (w.H // 128))) + w.NT * w.R * 8
        quant = {"ms": qm, "alg_bytes": qbytes, "alg_gbs": qbytes / (qm / 1e3) / 1e9,
                 "frac": qbytes / (qm / 1e3) / 1e9 / measured_peaks()[0],
                 "fp8_dispatch_ms": cm,
                 "fused_fp8_dispatch_ms": fused_fp8,
                 "vs_bf16_dispatch_ms": per_timed["dispatch (route+count+pack)"],
                 "note": "moe_dispatch_pack_quant on the same routing, timed alone; "
                         "fp8_dispatch_ms: route + count + quantising pack back to back; "
                         "fused_fp8_dispatch_ms: moe_dispatch_fused_quant (the same outputs in one "
                         "call; null where the batch is not a decode batch)"}
        del pq, ps
    out["pack_quant"] = quant

    # decode-fused dispatch (route + count + pack in one launch) on the same
    # inputs, when the batch is a decode batch it supports
    with nvtx_range("fused"):
        fused = run.fused_ms(nb, host_lead)
    if "ms" in fused:
        fused.update({"vs_separate_dispatch_ms": per_timed["dispatch (route+count+pack)"],
                      "step_ms_if_used": fused["ms"] + per_timed["combine"],
                      "note": "moe_dispatch_fused on the same batch (one thread-block cluster "
                              "for batches of up to 512 tokens, else a route kernel that also "
                              "counts, then the pack kernel deriving the rows)"})
    out["fused_dispatch"] = fused

    # the router with the bias in the selection key only (score of the raw
    # logit + bias decides; weights are the raw scores), against the default
    rtimes = {}
    for label, fn in (("default", w.score_fn), ("bias_select_only", w.score_fn | moe.MOE_BIAS_SELECT_ONLY)):
        rtimes[label] = run.timed_repeat(
            lambda fn=fn: moe.route_topk(dims, inp.logits, inp.bias, fn, w.renormalize, b.topk_idx,
                                         b.topk_w, stream), nb, host_lead)
    # restore the default routing for the steps below
    run.launch("route")
    run.launch("count")
    torch.cuda.synchronize(dev)

    # send-side accumulation (partial rows per token and destination rank,
    # then their sum)
    next_rows = {}
    sz = moe.buffer_sizes(dims)
    P = sz["partial_slots"]
    part = torch.empty(sz["partial_bytes"] // b.y.element_size(), dtype=b.y.dtype, device=dev)
    slot_rank = torch.empty(w.NT * P, dtype=torch.int32, device=dev)
    out2 = torch.empty_like(b.out)
    evs2 = []
    ppool = [new_events(3) for _ in range(nb + 3)]
    host_lead(nb + 3)
    send_range = nvtx_range("send_side")
    send_range.__enter__()
    for i in range(nb + 3):
        run.flush()
        e = ppool[i]
        e[0].record(stream)
        moe.combine_partials(dims, b.y, b.pos, b.topk_w, part, slot_rank, stream)
        e[1].record(stream)
        moe.combine_reduce_partials(dims, part, slot_rank, out2, stream)
        e[2].record(stream)
        if i >= 3:
            evs2.append(e)
    torch.cuda.synchronize(dev)
    send_range.__exit__(None, None, None)
    used = int((slot_rank >= 0).sum().item())
    yb = W.y_row_bytes(w)
    t_part = statistics.mean(e[0].elapsed_time(e[1]) for e in evs2)
    t_red = statistics.mean(e[1].elapsed_time(e[2]) for e in evs2)
    b_part = w.NT * (yb * w.R + yb * P) + w.NT * w.R * 8
    b_red = yb * used + w.NT * yb + w.NT * P * 4
    next_rows["route_bias_select_only"] = {
        "ms": rtimes["bias_select_only"], "default_route_ms": rtimes["default"],
        "note": "moe_route_topk with MOE_BIAS_SELECT_ONLY (DeepSeek-V3 convention) vs the "
                "default reading, each timed alone after an L2 flush"}
    next_rows["send_side_combine"] = {
        "partials_ms": t_part, "reduce_ms": t_red, "ms": t_part + t_red,
        "alg_bytes": b_part + b_red, "alg_gbs": (b_part + b_red) / ((t_part + t_red) / 1e3) / 1e9,
        "partial_rows_per_token": used / w.NT,
        "note": "moe_combine_partials + moe_combine_reduce_partials; one GPU moves more bytes "
                "this way than the plain combine (the saving is in data sent between GPUs)"}
    del part, slot_rank, out2
    out["next_rows"] = next_rows
    return out


def run_e2e(args, w, dims, inp_cpu, b, dev, stream, flush, moe):
    """Same path through the public API with host buffers: every step copies
    its inputs from pinned host memory, runs the four calls and copies `out`
    back, all inside the timed region.

    Steps alternate between `--e2e-lanes` independent sets of device buffers
    and streams, so one step's copies overlap another step's kernels (a
    serving pipeline; the copy engines and the SMs work at the same time).
    The value is steps / time from the first step's start to the last step's
    end.  A single-lane run (no overlap) is timed too and reported beside it.
    """
    import torch
    h_logits = inp_cpu.logits.pin_memory()
    h_bias = None if inp_cpu.bias is None else inp_cpu.bias.pin_memory()
    h_x = inp_cpu.x.pin_memory()
    h_xs = None if inp_cpu.x_scales is None else inp_cpu.x_scales.pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_logits, h_bias, h_x, h_xs) if t is not None)

    class Lane:
        def __init__(self, bufs, strm):
            self.b = bufs
            self.s = strm
            self.logits = torch.empty_like(h_logits, device=dev)
            self.bias = None if h_bias is None else torch.empty_like(h_bias, device=dev)
            self.x = torch.empty_like(h_x, device=dev)
            self.xs = None if h_xs is None else torch.empty_like(h_xs, device=dev)
            self.out = torch.empty(bufs.out.shape, dtype=bufs.out.dtype).pin_memory()

    def one(L):
        with torch.cuda.stream(L.s):
            L.logits.copy_(h_logits, non_blocking=True)
            if L.bias is not None:
                L.bias.copy_(h_bias, non_blocking=True)
            L.x.copy_(h_x, non_blocking=True)
            if L.xs is not None:
                L.xs.copy_(h_xs, non_blocking=True)
            bb = L.b
            moe.route_topk(dims, L.logits, L.bias, w.score_fn, w.renormalize, bb.topk_idx,
                           bb.topk_w, L.s)
            moe.dispatch_count(dims, bb.topk_idx, bb.expert_counts, bb.expert_offsets,
                               bb.rank_counts, bb.rank_offsets, bb.send_counts, bb.pos,
                               bb.status, L.s)
            moe.dispatch_pack(dims, L.x, L.xs, bb.pos, bb.packed_x, bb.packed_scales,
                              bb.packed_src, L.s)
            moe.combine(dims, bb.y, bb.pos, bb.topk_w, bb.out, L.s)
            L.out.copy_(bb.out, non_blocking=True)

    def timed(lanes, n):
        for i in range(2 * len(lanes)):
            one(lanes[i % len(lanes)])
        torch.cuda.synchronize(dev)
        flush()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for L in lanes:
            L.s.wait_event(t0)
        for i in range(n):
            one(lanes[i % len(lanes)])
        for L in lanes:
            stream.wait_stream(L.s)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1) / n

    n = max(1, args.e2e_steps)
    lanes = [Lane(b, torch.cuda.Stream(dev))]
    serial_ms = timed(lanes, n)
    for _ in range(max(1, args.e2e_lanes) - 1):
        lanes.append(Lane(moe.Buffers(dims, device=dev,
                                      separate_y=False if w.x_dtype == w.y_dtype else None),
                          torch.cuda.Stream(dev)))
    ms = timed(lanes, n) if len(lanes) > 1 else serial_ms
    d2h = lanes[0].out.numel() * lanes[0].out.element_size()
    return {"value": w.NT / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "lanes": len(lanes), "serial_ms_per_step": serial_ms,
            "serial_value": w.NT / (serial_ms / 1e3)}


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
