#!/usr/bin/env python3
"""Benchmark of single-token split-KV decode attention on GB300.

A step is one decode step's attention over L layers of one geometry: every
layer has its own Q and its own K/V cache, all resident in HBM, and the step
runs the whole hot path (split kernel + merge kernel) once per layer. For the
Gemma local sliding ring (the headline workload) L = 40, the sliding-window
layers of Gemma 4 12B (48 layers, 8 of them global, per "Hand-Writing Gemma 4
Flash-Decoding + an FP4 Matvec Bonus (Part 2)", section "The starting point",
and mlxcel issue #683). The live-band bytes of all layers (tens to hundreds of
MB) exceed the 129 MB L2, so no layer's K/V is still in L2 when it is read
again one step later.

Metric: live-band KV GB/s = sum over layers and sequences of
band_b * NKV * HS * 2 (K and V) * 2 bytes, divided by the step time, and the
same time as microseconds per layer. Device time comes from CUDA events around
CUDA-graph replays of the step; e2e repeats the step through the public call
(fd_decode_attn_ex via the Python binding, with the step's plan and
workspace) with each step's queries and lengths copied from pinned host memory
and the outputs copied back inside the timed region. The plan is made once per
geometry, as a decode loop makes it: for the whole cache, with the step's
shortest length as its lower bound (fd_plan_min_len; --no-min-len drops it).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fd|reference]
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
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import torch  # noqa: E402

HEADLINE = "gemma_local_ring"
METRIC = "decode-attn live-band KV GB/s (% of HBM peak) and µs/layer per geometry"
L2_BYTES = 129 * 1024 * 1024


def live_band_bytes(w, lens) -> int:
    keep = w.capacity if w.window <= 0 else min(w.window, w.capacity)
    tot = 0
    for L in lens.tolist():
        L = max(0, int(L))
        tot += L - max(0, L - keep)
    return tot * w.NKV * w.HS * 2 * 2


def max_over_ranks(x: float, device) -> float:
    """Largest value of x over the ranks of the default process group (x
    itself without one): a replica job is as slow as its slowest rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbps(bytes_per_step_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job live-band GB/s: every rank's bytes over the slowest step."""
    return bytes_per_step_per_rank * world / (ms_per_step * 1e-3) / 1e9


def kernels_per_call(plan) -> int:
    """Kernels one call launches: the split kernel, plus the merge kernel
    unless one block/cluster spans every split or the fused merge is on."""
    return 1 if (plan.num_splits == plan.cluster or plan.fused) else 2


def measured_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """Samples nvidia-smi every 20 ms while the timed regions run; entering
    waits (up to 5 s) for the first sample so the sampler is live before the
    timed region starts."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.skip = 0

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
                time.sleep(0.01)
            self.skip = len(self.lines)  # samples taken before the timed region are not counted
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=5)

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[self.skip:]:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def layers_for(w, live, cap_layers=256):
    """Enough layers that one step's live bytes exceed twice the L2, at least 4
    (the headline ring uses its model's 40 layers)."""
    if w.name == HEADLINE:
        return 40
    n = max(4, math.ceil(2 * L2_BYTES / max(1, live)))
    alloc = 2 * w.B * w.NKV * w.capacity * w.HS * 2
    n = min(n, cap_layers, max(2, (64 << 30) // alloc))
    return n


class Step:
    """L layers of one geometry resident on the device; kv = "bf16" or "e4m3"
    (E4M3 codes with per-(sequence, KV head) scales: half the live bytes)."""

    def __init__(self, w, layers, device, seed_base=0, kv="bf16", path=0, min_len=True):
        from decode_attention_04_gb300.inputs import draw_lens, make_inputs, make_inputs_fp8

        self.w = w
        self.L = layers
        self.kv = kv
        self.lens_h = draw_lens(w)
        self.q, self.k, self.v, self.ks, self.vs = [], [], [], [], []
        for i in range(layers):
            seed = w.seed * 1000 + seed_base + i
            if kv == "e4m3":
                q, k, v, ks, vs, _ = make_inputs_fp8(w, device=device, seed=seed, lens=self.lens_h)
                self.ks.append(ks)
                self.vs.append(vs)
            else:
                q, k, v, _ = make_inputs(w, device=device, seed=seed, lens=self.lens_h)
            self.q.append(q)
            self.k.append(k)
            self.v.append(v)
        self.lens = self.lens_h.to(device)
        self.out = [torch.empty_like(x) for x in self.q]
        self.live = live_band_bytes(w, self.lens_h) // (2 if kv == "e4m3" else 1)
        # One plan for the step, made the way a decode loop makes it: for the
        # cache's whole capacity (max_len 0), with the step's shortest length
        # as the lower bound on every length (decode lengths only grow, so it
        # holds for every later replay of a captured step); a forced kernel
        # family overrides the plan's. One workspace serves the layers in turn.
        import decode_attention_04_gb300 as fd
        kvt = fd.FD_KV_E4M3 if kv == "e4m3" else fd.FD_KV_BF16
        self.the_plan = fd.fd_plan_kv(w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, kv_dtype=kvt)
        if path:
            fd.fd_plan_override(self.the_plan, 0, path)
        if min_len:
            fd.fd_plan_min_len(self.the_plan, int(self.lens_h.min().item()))
        self.ws = torch.zeros(max(16, self.the_plan.workspace_bytes), dtype=torch.uint8, device=device)

    def plan(self):
        return self.the_plan

    def run(self, stream=None):
        """The step: one fd_decode_attn_ex (or _fp8_ex) call per layer."""
        import decode_attention_04_gb300 as fd
        w, p = self.w, self.the_plan
        for i in range(self.L):
            if self.kv == "e4m3":
                fd.fd_decode_attn_fp8_ex(p, self.ws, p.workspace_bytes, None, self.q[i], self.k[i], self.v[i],
                                         self.ks[i], self.vs[i], self.out[i], self.lens, w.B, w.NH, w.NKV, w.HS,
                                         w.capacity, w.window, w.scale, stream)
            else:
                fd.fd_decode_attn_ex(p, self.ws, p.workspace_bytes, None, self.q[i], self.k[i], self.v[i],
                                     self.out[i], self.lens, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window,
                                     w.scale, stream)


def time_graph(step: Step, steps: int, warmup: int, stream, bracket=None):
    """Capture the L-layer step in a CUDA graph; time `steps` replays with CUDA
    events on the capture stream. Returns per-step milliseconds (list)."""
    with torch.cuda.stream(stream):
        for _ in range(max(3, warmup)):
            step.run(stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step.run(stream)
    with torch.cuda.stream(stream):
        for _ in range(max(3, warmup)):
            g.replay()
    stream.synchronize()
    if bracket:
        bracket()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(steps):
            g.replay()
            ev[i + 1].record(stream)
    stream.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)], g


def time_e2e(step: Step, steps: int, warmup: int, stream, bracket=None):
    """Each step: pinned host Q (all layers) and lens -> device, the L public
    calls, outputs -> pinned host; CUDA events around the whole step."""
    w = step.w
    qh = torch.stack([x.cpu() for x in step.q]).pin_memory()
    lh = step.lens_h.clone().pin_memory()
    oh = torch.empty_like(qh).pin_memory()
    qd = torch.stack(step.q)  # staging on the device, one copy per step
    saved_q, saved_out = step.q, step.out
    step.q = list(qd.unbind(0))
    od = torch.empty_like(qd)
    step.out = list(od.unbind(0))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]

    def one():
        qd.copy_(qh, non_blocking=True)
        step.lens.copy_(lh, non_blocking=True)
        step.run(stream)
        oh.copy_(od, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(max(3, warmup)):
            one()
        stream.synchronize()
        if bracket:
            bracket()
        ev[0].record(stream)
        for i in range(steps):
            one()
            ev[i + 1].record(stream)
    stream.synchronize()
    step.q, step.out = saved_q, saved_out
    ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    h2d = qh.numel() * qh.element_size() + lh.numel() * lh.element_size()
    d2h = oh.numel() * oh.element_size()
    return ms, h2d, d2h


def cpu_baseline(w, step: Step, budget_s: float = 10.0):
    """The FP64 oracle, as it stands, on this host's cores: the step's layers in
    turn, repeated until about `budget_s` seconds of oracle time are used (at
    least one layer)."""
    import oracle

    oracle.build()
    host = {}
    done, t_used, nbytes = 0, 0.0, 0
    while done == 0 or t_used < budget_s:
        i = done % step.L
        if i not in host:  # copies to host memory stay outside the timed calls
            host[i] = (step.q[i].cpu(), step.k[i].cpu(), step.v[i].cpu())
        q, k, v = host[i]
        t0 = time.perf_counter()
        oracle.decode(q, k, v, step.lens_h, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, w.scale)
        t_used += time.perf_counter() - t0
        nbytes += step.live
        done += 1
    cores = os.cpu_count() or 1
    return {"value": nbytes / t_used / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} layer calls ({done / step.L:.1f} passes over the {step.L} layers of one step of "
                      f"{w.name}, {nbytes / 1e6:.1f} MB live band), FP64, {cores} threads, {t_used:.2f} s"}


def time_single_calls(step: Step, n: int, stream):
    """Plain launches (no graph) of layer 0, one at a time: CUDA events around
    each call, a synchronize between calls. Returns the median in µs."""
    one = Step.__new__(Step)
    one.__dict__.update(step.__dict__)
    one.L = 1
    ts = []
    with torch.cuda.stream(stream):
        for i in range(n + 3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            one.run(stream)
            b.record(stream)
            stream.synchronize()
            if i >= 3:
                ts.append(a.elapsed_time(b) * 1e3)
    return statistics.median(ts)


def time_l2_hot(step: Step, steps: int, stream):
    """A graph of layer 0 alone, replayed back to back: its K/V stay in L2 when
    they fit (labelled L2-hot; not the metric). Returns µs per call."""
    one = Step.__new__(Step)
    one.__dict__.update(step.__dict__)
    one.L = 1
    ms, g = time_graph(one, steps, 3, stream)
    del g
    return statistics.median(ms) * 1e3


def cpu_oracle_sample(w, step: Step, budget_s: float = 1.5):
    """The FP64 oracle on layer 0 of a geometry, on all host cores and on one
    thread: the first k (sequence, head) rows, k sized from one timed row so
    each timing takes about `budget_s`; the bytes counted are those rows' share
    of the live band (its K/V rows are read once per query row)."""
    import numpy as np
    import oracle

    oracle.build()
    q, k, v = step.q[0].cpu(), step.k[0].cpu(), step.v[0].cpu()
    rows_total = w.B * w.NH
    per_row_bytes = step.live / rows_total

    def timed(nrows, nthreads, reps=1):
        want = np.zeros(rows_total, dtype=bool)
        want[:nrows] = True
        t0 = time.perf_counter()
        for _ in range(reps):
            oracle.decode(q, k, v, step.lens_h, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, w.scale, want=want,
                          nthreads=nthreads)
        return time.perf_counter() - t0

    out = {}
    for label, nthreads in (("all_cores", 0), ("one_thread", 1)):
        threads = (os.cpu_count() or 1) if nthreads == 0 else 1
        t1 = max(timed(1, nthreads), 1e-6)
        nrows = max(1, min(rows_total, int(budget_s / t1) * threads))
        reps = 1
        if nrows == rows_total:  # the whole layer is cheap: repeat it to fill the budget
            reps = max(1, int(budget_s / max(timed(nrows, nthreads), 1e-6)))
        t = timed(nrows, nthreads, reps)
        out[label] = {"GBps": per_row_bytes * nrows * reps / t / 1e9, "rows": nrows, "calls": reps,
                      "seconds": round(t, 3)}
    out["threads_all_cores"] = os.cpu_count() or 1
    return out


def run_geometry(w, steps, warmup, stream, device, peak, kv="bf16", min_len=True):
    from decode_attention_04_gb300.inputs import draw_lens
    lens = draw_lens(w)
    live = live_band_bytes(w, lens)
    L = layers_for(w, live)
    st = Step(w, L, device, kv=kv, min_len=min_len)
    ms, _ = time_graph(st, steps, warmup, stream)
    t = statistics.median(ms)
    plan = st.plan()
    gbs = st.live * L / (t * 1e-3) / 1e9
    res = {"us_per_layer": t * 1e3 / L, "us_per_layer_min": min(ms) * 1e3 / L, "live_GBps": gbs,
           "frac_of_peak": gbs / peak, "layers": L, "live_bytes_per_layer": st.live,
           "num_splits": plan.num_splits, "desc": w.desc,
           "us_single_call_plain_launch": time_single_calls(st, 20, stream),
           "us_l2_hot_one_layer": time_l2_hot(st, steps, stream),
           "l2_hot_fits": st.live <= L2_BYTES // 2}
    if kv == "bf16":
        res["cpu_oracle"] = cpu_oracle_sample(w, st)
    del st
    torch.cuda.empty_cache()
    return res


# Share of the library's device time taken by the split kernel in the
# committed ncu launch list of the headline workload (profiles/); the split
# and merge kernels of one call run back to back under programmatic dependent
# launch, so events cannot separate them without changing what is timed.
SPLIT_SHARE = {"gemma_local_ring": (0.612, "profiles/launches_gemma_local_ring.md",
                                    "split_tc_kernel<TcCfg<256,1,8,1,4096>> (16 x 8 blocks of one tile)")}


def dominant_kernel(name, per_layer_us, live, peak):
    """The split kernel's part of the timed per-layer time (its launch-list
    share) and the live-band rate over that part, against the same peak."""
    if name not in SPLIT_SHARE:
        return None
    share, src, kernel = SPLIT_SHARE[name]
    us = per_layer_us * share
    gbs = live / (us * 1e-6) / 1e9
    return {"kernel": kernel, "share_of_device_time": share, "share_source": src, "us_per_launch": us,
            "achieved": gbs, "frac": gbs / peak, "unit": "GB/s",
            "how": "timed per-layer CUDA-event time x the kernel's share in the ncu launch list"}


def geometry_summary(geoms, geoms8):
    """Compact per-geometry rows for the end of the JSON line: workload,
    µs per layer, live-band GB/s, fraction of the HBM peak, splits."""
    if not geoms:
        return None

    def rows(g):
        return [[name, round(r["us_per_layer"], 2), round(r["live_GBps"], 1), round(r["frac_of_peak"], 3),
                 r["num_splits"]] for name, r in g.items()]

    return {"cols": ["workload", "us_per_layer", "live_GBps", "frac_of_peak", "splits"],
            "bf16": rows(geoms), "e4m3": rows(geoms8) if geoms8 else None}


def allocation_independence(steps, stream, device, caps=(4096, 32768, 131072), min_len=True):
    """Gemma global MQA at len 4096 with the cache allocated at several
    capacities: the time must not grow with the allocation (the page's 537 MB
    of whole-allocation reads was the bug this op fixes)."""
    from dataclasses import replace
    from decode_attention_04_gb300.inputs import WORKLOADS
    base = WORKLOADS["gemma_global_mqa_4k"]
    out = {}
    for cap in caps:
        w = replace(base, name=f"mqa_len4096_cap{cap}", capacity=cap)
        L = 32  # 32 x 8.4 MB live > 2 x L2
        st = Step(w, L, device, min_len=min_len)
        ms, g = time_graph(st, steps, 3, stream)
        out[str(cap)] = {"us_per_layer": statistics.median(ms) * 1e3 / L, "num_splits": st.plan().num_splits}
        del st, g
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="fd", choices=["fd", "reference"])
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--no-geometries", action="store_true", help="skip the per-geometry table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-min-len", action="store_true",
                    help="plans without the lengths' lower bound (nothing read before the lengths)")
    ap.add_argument("--only", default="", help="comma-separated geometries for the per-geometry tables")
    ap.add_argument("--no-e4m3", action="store_true", help="skip the E4M3 per-geometry table")
    ap.add_argument("--profile-calls", type=int, default=0,
                    help="profiling mode: N plain fd_decode_attn calls on one layer of --workload, then exit")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "e4m3"],
                    help="cache type of --profile-calls (the timed step and its line are bf16)")
    ap.add_argument("--path", type=int, default=0,
                    help="kernel family of --profile-calls (0 = the plan's, 1 SIMT, 2 mma tiles, 3 tcgen05)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from decode_attention_04_gb300.inputs import PROFILE_WORKLOADS, WORKLOADS
    w = WORKLOADS[args.workload] if args.workload in WORKLOADS else PROFILE_WORKLOADS[args.workload]

    if args.impl == "reference":
        return reference_arm(args, w, rank, world)
    if args.profile_calls:
        return profile_calls(w, args.profile_calls, args.kv, args.path, not args.no_min_len)

    import decode_attention_04_gb300 as fd
    from decode_attention_04_gb300 import build as libbuild
    if rank == 0:
        libbuild.build()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        torch.cuda.set_device(local)
        dist.barrier()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    fd.load_library()
    peak, peak_kind = measured_peaks()
    stream = torch.cuda.Stream(device)

    use_min_len = not args.no_min_len
    step = Step(w, layers_for(w, 0), device, min_len=use_min_len)
    L = step.L
    plan = step.plan()
    launches_per_call = kernels_per_call(plan)

    # ---- device-timed steps (graph replay), clocks sampled during the region
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    def bracket():  # a barrier and a device synchronize on each side of a timed region
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    with ClockSampler(local) as clk:
        ms, graph = time_graph(step, args.steps, args.warmup, stream, bracket)
        bracket()
        # ---- end to end through the public call, host buffers (sampled too)
        e2e_ms, h2d, d2h = time_e2e(step, args.steps, args.warmup, stream, bracket)
        bracket()
    tot_ms = max_over_ranks(sum(ms), device)
    ms_per_step = tot_ms / args.steps
    value = job_gbps(step.live * L, world, ms_per_step)
    per_layer_us = ms_per_step * 1e3 / L
    achieved = step.live / (per_layer_us * 1e-6) / 1e9
    e2e_ms_per_step = max_over_ranks(statistics.mean(e2e_ms), device)
    e2e_value = job_gbps(step.live * L, world, e2e_ms_per_step)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    cpu = None if args.no_cpu_baseline else cpu_baseline(w, step)
    live = step.live
    del graph
    clocks = clk.summary()
    geoms = geoms8 = alloc = None
    if not args.no_geometries:
        del step
        torch.cuda.empty_cache()
        geoms, geoms8 = {}, {}
        only = [x for x in args.only.split(",") if x]
        todo = {n: g for n, g in WORKLOADS.items() if not only or n in only}
        for name, gw in todo.items():
            geoms[name] = run_geometry(gw, max(10, min(args.steps, 30)), 3, stream, device, peak,
                                       min_len=use_min_len)
        if not args.no_e4m3:
            for name, gw in todo.items():
                geoms8[name] = run_geometry(gw, max(10, min(args.steps, 30)), 3, stream, device, peak, kv="e4m3",
                                            min_len=use_min_len)
        if not only:
            alloc = allocation_independence(max(10, min(args.steps, 30)), stream, device, min_len=use_min_len)

    traffic = None
    tf = ROOT / "profiles" / "traffic.txt"
    if tf.exists():
        try:
            traffic = json.loads(tf.read_text()).get(w.name)
        except (ValueError, OSError):
            traffic = None
    dominant = dominant_kernel(w.name, per_layer_us, live, peak)

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "us_per_layer": per_layer_us,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: Q,K,V iid N(0,1) rounded to bf16, seeded",
        "config": {
            "workload": w.name,
            "desc": w.desc,
            "layers_per_step": L,
            "live_band_bytes_per_layer": live,
            "B": w.B, "NH": w.NH, "NKV": w.NKV, "HS": w.HS, "capacity": w.capacity, "window": w.window,
            "num_splits": plan.num_splits,
            "l2": f"inputs larger than L2: {L} layers x {live / 1e6:.1f} MB live band = {L * live / 1e6:.0f} MB per step vs 129 MB L2",
            "timing": "CUDA events around CUDA-graph replays of the step, on the launching stream",
            "plan": {"num_splits": plan.num_splits, "min_len": plan.min_len, "path": plan.path,
                     "call": "fd_decode_attn_ex, one plan and workspace for the step"},
            "parallelism": f"replicas x{world}",
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "one fd_decode_attn_ex call (split kernel + merge kernel), averaged over the timed step",
            "achieved": achieved,
            "peak": peak,
            "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback 6.8 TB/s",
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": traffic,
            "dominant_kernel": dominant,
        },
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms_per_step},
        "gpu_launches": args.steps * L * launches_per_call,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "geometries": geoms,
        "geometries_e4m3": geoms8,
        "allocation_independence": alloc,
        # last, so a reader that keeps only the end of the line still has
        # every geometry: [workload, us/layer, live GB/s, fraction of peak, splits]
        "geometry_summary": geometry_summary(geoms, geoms8),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def profile_calls(w, n, kv="bf16", path=0, min_len=True):
    """N plain calls on one layer (for ncu launch lists and captures)."""
    from decode_attention_04_gb300 import build as libbuild
    libbuild.build()
    device = torch.device("cuda", 0)
    st = Step(w, 1, device, kv=kv, path=path, min_len=min_len)
    for _ in range(n):
        st.run()
    torch.cuda.synchronize()
    print(json.dumps({"profile_calls": n, "workload": w.name, "kv": kv, "live_bytes": st.live}), flush=True)
    return 0


def reference_arm(args, w, rank, world):
    """--impl reference: the FP64 oracle as it stands on this host's cores, on
    the same workload, metric and unit; each step is one layer of the step (a
    bounded sample of the workload)."""
    if rank != 0:
        return 0
    import oracle
    from decode_attention_04_gb300.inputs import draw_lens, make_inputs

    oracle.build()
    lens = draw_lens(w)
    live = live_band_bytes(w, lens)
    q, k, v, _ = make_inputs(w, lens=lens)
    for _ in range(args.warmup):
        oracle.decode(q, k, v, lens, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, w.scale)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode(q, k, v, lens, w.B, w.NH, w.NKV, w.HS, w.capacity, w.window, w.scale)
    dt = time.perf_counter() - t0
    value = live * args.steps / dt / 1e9
    cores = os.cpu_count() or 1
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic: Q,K,V iid N(0,1) rounded to bf16, seeded",
        "config": {"workload": w.name, "desc": w.desc, "layers_per_step": 1,
                   "note": "each step is one layer of the fd step (bounded CPU sample)"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} timed calls on one layer of {w.name}, FP64, {cores} threads"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
