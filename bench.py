"""Benchmark of content-routed sparse attention on B300.

Headline (``value``): decode tok/s per attention layer at a 1M-token cache
(B=1, Hq=32, Hkv=4, d=128, S=1024, k=16, bf16): one step = route one new
query token per head (scores over 1023 span summaries + top-16) and attend
its selected spans plus its local span.  ``roofline`` divides the step's
gathered K/V bytes plus the summary bytes its route reads by the whole
step's time.  ``e2e`` repeats the decode through the same C-ABI calls with
the query copied in from pinned host memory and the output copied back
every step.

Further lines, each with its own roofline and, on rank 0 of a one-GPU run,
the oracle timed on the host cores (``cpu_baseline``):
  prefill          8192 queries against a 1M cache (summaries + route + attend)
  prefill_128k     the whole 128K prefill, 16 chunks of 8192
  tiny_prefill     the 4096-query fp32 case
  decode_10m       decode at a 10M-token cache
  decode_group_shared, decode_q8, decode_q4   decode with one top-k per
                   kv-head group, and over the 8-bit and 4-bit caches
  dense_comparison the same shapes through dense attention (PyTorch SDPA)

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Multi-GPU (torchrun, one process per GPU): every rank runs an independent
replica of the workload; value = tokens of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import content_routed_sparse_build_b300 as ssa  # noqa: E402
from synth import workloads as W  # noqa: E402

METRIC = "routed-attention decode tok/s and prefill tok/s per layer at 1M ctx; % of roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")


# --------------------------------------------------------------------- helpers
def peaks():
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.proc = None
        self.rows = []
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            self.sel = ["-i", str(device)]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *self.sel, "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if len(r) > 3 + i and r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(self.rows)}


def dist_setup(backend: str = "nccl"):
    """One process per GPU, launched by torchrun: (world size, rank, local rank).

    The ranks run independent replicas of the workload (the path has no
    exchange step); the process group only carries the barrier around the
    timed region and the max over ranks of its duration.
    """
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if backend == "nccl":
        torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        if backend == "nccl":
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    """The largest of the ranks' values (the job's time is its slowest rank's)."""
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, seconds: float, ws: int) -> float:
    """Whole-job throughput: the units every rank processed over the max-over-ranks time."""
    return units_per_rank * ws / seconds


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) that ncu measured
# for the roofline's unit, as the kernels stand in this tree; each figure
# names the profile summary it comes from.  The decode step's figure was
# captured on a 256K cache (a full-size capture may take one counter pass
# only) and scaled to the 1M step by each kernel's unit: the attend reads by
# the gathered bytes, the route's by the candidate count; the partial and
# merge bytes do not change.  The prefill attend kernel changed after its last
# full-size capture, so its line reports no traffic.
NCU_TRAFFIC = {
    "decode_1m": (2.214e8, "profiles/decode_1m_launches.md: route + attend + merge of one step, "
                           "256K capture scaled to 1M"),
    "decode_1m_q8": (1.155e8, "profiles/decode_1m_launches.md: route + 8-bit attend + merge, 256K capture "
                              "scaled to 1M"),
    "decode_1m_q4": (6.108e7, "profiles/decode_attend_q4_256k.md: route + 4-bit attend + merge, 256K capture "
                              "scaled to 1M"),
}


def traffic_of(workload: str):
    t = NCU_TRAFFIC.get(workload)
    return (t[0], t[1]) if t else (None, None)


def flush_l2(buf):
    buf.zero_()


# --------------------------------------------------------------------- decode
class DecodeBench:
    """The decode workload: 256 distinct queries at the last 256 positions of
    the cache.  A step routes one query token per head and attends it; the
    256 steps are captured once in a CUDA graph and replayed."""

    def __init__(self, w: W.Workload, dev, group: bool = False, q8: bool = False, q4: bool = False):
        self.w = w
        self.dev = dev
        self.group = group                                     # group-shared selection
        self.q8 = q8                                           # attend over the 8-bit cache
        self.q4 = q4                                           # attend over the 4-bit cache
        self.inp = W.Inputs(w)
        self.K = self.inp.k(dev)
        self.V = self.inp.v(dev)
        self.Q = self.inp.q(dev)                               # [steps, B, Hq, d]
        self.p = ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L, w.S, w.topk, w.dtype)
        self.summ = torch.zeros((w.B, w.Hkv, w.n_spans, w.d), dtype=torch.float32, device=dev)
        self.ws = ssa.workspace(self.p, 1, ssa.SSA_OP_DECODE, dev)
        self.wsg = ssa.workspace(self.p, 1, ssa.SSA_OP_ROUTE_GROUP, dev) if group else None
        self.sels = [torch.empty((w.B, w.Hq, 1, w.topk), dtype=torch.int32, device=dev)
                     for _ in range(w.n_q)]
        self.sel = self.sels[0]
        self.O = torch.empty((w.B, w.Hq, w.d), dtype=w.dtype, device=dev)
        self.lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
        self.qs = [self.Q[s].contiguous() for s in range(w.n_q)]
        if q8:
            self.Kq, self.Ks, self.Vq, self.Vs = ssa.q8_cache(self.p, dev)
            ssa.ssa_quantize_kv(self.p, self.K, self.V, 0, w.L, self.Kq, self.Ks, self.Vq, self.Vs)
        if q4:
            self.Kq, self.Ks, self.Vq, self.Vs = ssa.q4_cache(self.p, dev)
            ssa.ssa_quantize_kv4(self.p, self.K, self.V, 0, w.L, self.Kq, self.Ks, self.Vq, self.Vs)
        if q8 or q4:
            del self.K, self.V                                 # the quantised cache is what a step reads
            torch.cuda.empty_cache()

    def build_summaries(self):
        if self.q8:
            ssa.ssa_build_summaries_q8(self.p, self.Kq, self.Ks, 0, self.w.n_spans, self.summ)
        elif self.q4:
            ssa.ssa_build_summaries_q4(self.p, self.Kq, self.Ks, 0, self.w.n_spans, self.summ)
        else:
            ssa.ssa_build_summaries(self.p, self.K, 0, self.w.n_spans, self.summ)

    def route(self, i):
        if self.group:
            ssa.ssa_route_group(self.p, self.qs[i], 1, self.w.q_pos0 + i, self.summ, self.sels[i], None,
                                self.wsg)
        else:
            ssa.ssa_route(self.p, self.qs[i], 1, self.w.q_pos0 + i, self.summ, self.sels[i])

    def attend(self, i):
        if self.q8:
            ssa.ssa_attend_decode_q8(self.p, self.qs[i], self.w.q_pos0 + i, self.Kq, self.Ks, self.Vq, self.Vs,
                                     self.sels[i], self.O, self.lse, self.ws)
        elif self.q4:
            ssa.ssa_attend_decode_q4(self.p, self.qs[i], self.w.q_pos0 + i, self.Kq, self.Ks, self.Vq, self.Vs,
                                     self.sels[i], self.O, self.lse, self.ws)
        else:
            ssa.ssa_attend_decode(self.p, self.qs[i], self.w.q_pos0 + i, self.K, self.V, self.sels[i],
                                  self.O, self.lse, self.ws)

    def step(self, i):
        # the whole step in one call where the library has one: route (which
        # also plans) + attend + merge
        if self.q8:
            ssa.ssa_decode_step_q8(self.p, self.qs[i], self.w.q_pos0 + i, self.summ, self.Kq, self.Ks, self.Vq,
                                   self.Vs, self.sels[i], self.O, self.lse, self.ws)
            return
        if self.q4:
            ssa.ssa_decode_step_q4(self.p, self.qs[i], self.w.q_pos0 + i, self.summ, self.Kq, self.Ks, self.Vq,
                                   self.Vs, self.sels[i], self.O, self.lse, self.ws)
            return
        if self.group:
            ssa.ssa_decode_step_group(self.p, self.qs[i], self.w.q_pos0 + i, self.summ, self.K, self.V,
                                      self.sels[i], self.O, self.lse, self.ws)
            return
        ssa.ssa_decode_step(self.p, self.qs[i], self.w.q_pos0 + i, self.summ, self.K, self.V, self.sels[i],
                            self.O, self.lse, self.ws)

    def graph(self, fn, n):
        """A CUDA graph of fn(0 .. n-1) (query index modulo the 256 queries)."""
        side = torch.cuda.Stream(self.dev)
        side.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(side):
            for i in range(min(n, 3)):
                fn(i % self.w.n_q)
        torch.cuda.current_stream(self.dev).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                fn(i % self.w.n_q)
        return g

    def algorithmic_bytes(self):
        """Per query index: (attend bytes, route bytes), from the actual selections."""
        w = self.w
        el = 2 if w.dtype != torch.float32 else 4
        out = []
        for i in range(w.n_q):
            self.route(i)
        torch.cuda.synchronize()
        for i in range(w.n_q):
            pos = w.q_pos0 + i
            ell = pos // w.S
            sel = self.sels[i].reshape(w.B, w.Hkv, w.g * w.topk).cpu().numpy()
            kv_rows = 0
            for b in range(w.B):
                for g in range(w.Hkv):
                    u = np.unique(sel[b, g][sel[b, g] >= 0])
                    kv_rows += len(u) * w.S + (pos - ell * w.S + 1)
            # K + V (+ two fp32 scales)
            row_bytes = (2 * w.d + 8) if self.q8 else (w.d + 8) if self.q4 else w.d * el * 2
            attend = kv_rows * row_bytes + 2 * w.B * w.Hq * w.d * el + w.B * w.Hq * w.topk * 4
            route = w.B * w.Hkv * ell * w.d * 4 + w.B * w.Hq * w.d * el + w.B * w.Hq * w.topk * 4
            out.append((attend, route))
        return out


def hold_device(stream):
    """Queues about half a millisecond of device-side sleep on `stream` (a
    torch utility kernel, outside the timed region), so that the host has
    queued the timed launches before the start event executes: the
    device-timed region then holds the steps' execution and not the host's
    submission latency, which the e2e figure includes."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(1_000_000)


def replay_ms(g, reps, stream):
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_device(stream)
    a.record(stream)
    for _ in range(reps):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def decode_graphs(db, steps):
    """CUDA graphs whose replays run exactly `steps` decode steps: a graph of
    the workload's n_q distinct queries replayed steps // n_q times, then a
    graph of the remainder.  Returns [(graph, replays)]."""
    n = db.w.n_q
    reps, rem = divmod(steps, n)
    plan = []
    if reps:
        plan.append((db.graph(db.step, n), reps, n))
    if rem:
        plan.append((db.graph(db.step, rem), 1, rem))
    return plan


def replay_plan(plan):
    for g, r, _ in plan:
        for _ in range(r):
            g.replay()


def plan_text(plan, steps):
    return ("%d decode steps as CUDA-graph replays (%s); every graph was replayed during warm-up; the "
            "replays are queued behind a 0.5 ms device-side sleep so that host submission is outside the "
            "device-timed region (e2e includes it)" % (
                steps, " + ".join("%d-step graph x %d" % (k, r) for _, r, k in plan)))


def bench_decode(w, dev, steps, warmup, ws_n, cpu_leg):
    db = DecodeBench(w, dev)
    st = torch.cuda.current_stream(dev)
    # summaries of the whole cache (the decode steps read them), timed on its own
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    db.build_summaries()
    torch.cuda.synchronize()
    e0.record(st)
    db.build_summaries()
    e1.record(st)
    torch.cuda.synchronize()
    summ_ms = e0.elapsed_time(e1)
    summ_bytes = w.B * w.Hkv * w.L * w.d * 2 + w.B * w.Hkv * w.n_spans * w.d * 4
    per_q = db.algorithmic_bytes()

    n = w.n_q
    plan = decode_graphs(db, steps)
    g_att = db.graph(db.attend, n)          # attend only, on the selections routed above
    g_att.replay()
    torch.cuda.synchronize()
    # end to end through the C ABI first, before this process starts the
    # nvidia-smi clock sampler: its polling slows host-side CUDA calls (the
    # stream synchronise, the copies' submission) for as long as it runs and
    # about a second after, which a host-bound loop measures (72 -> 108 us
    # per step on one box), while the device-timed regions below, queued
    # behind a device-side sleep, do not see it
    e2e = bench_decode_e2e(db, min(max(steps, 256), 2048))
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        # warm-up, right before the timed region (the sampler's start leaves
        # the GPU idle for a moment): every graph the timed region replays is
        # replayed first, at least `warmup` steps in all
        done = 0
        while done < max(warmup, 1):
            replay_plan(plan)
            done += steps
        barrier(ws_n)
        torch.cuda.synchronize()
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_device(st)
        start.record(st)
        replay_plan(plan)
        stop.record(st)
        torch.cuda.synchronize()
        barrier(ws_n)
    total_ms = start.elapsed_time(stop)
    att_reps = max(1, -(-steps // n))
    attend_ms = replay_ms(g_att, att_reps, st) / (att_reps * n) * steps
    err = ssa.ssa_workspace_error(db.ws)
    total_ms_max = max_over_ranks(total_ms, ws_n)

    attend_bytes = sum(per_q[s % n][0] for s in range(steps))
    route_bytes = sum(per_q[s % n][1] for s in range(steps))
    pk = peaks()
    step_gbs = (attend_bytes + route_bytes) / (total_ms_max * 1e-3) / 1e9
    att_gbs = attend_bytes / (attend_ms * 1e-3) / 1e9
    tr, tr_src = traffic_of(w.name)
    res = {
        "tok_s": job_throughput(steps, total_ms_max * 1e-3, ws_n),
        "ms_per_step": total_ms_max / steps,
        "attend_ms_per_step": attend_ms / steps,
        "route_plus_gaps_ms_per_step": (total_ms - attend_ms) / steps,
        "attend_bytes_per_step": attend_bytes / steps,
        "route_bytes_per_step": route_bytes / steps,
        # the headline fraction: gathered K/V plus summary bytes of a step
        # over the whole step's time (route, attend and every gap between)
        "roofline": {"bound": "hbm", "achieved": round(step_gbs, 1), "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": round(step_gbs / pk["hbm_gbs"], 4),
                     "traffic": tr, "traffic_source": tr_src,
                     "kernel": "whole decode step (route + attend), %d launches per step, timed as "
                               "CUDA-graph replays" % launches_per_decode_step(w),
                     "bytes": "gathered K/V of the union of each kv-head group's selected spans plus "
                              "the causal local span, plus the candidate summaries the route reads, "
                              "per step, from the run's own selections",
                     "peak_source": pk["source"],
                     "attend_only": {"achieved": round(att_gbs, 1), "frac": round(att_gbs / pk["hbm_gbs"], 4),
                                     "what": "the attend launches alone, replayed apart from the route"}},
        "summaries": {"ms": summ_ms, "gbs": summ_bytes / (summ_ms * 1e-3) / 1e9,
                      "frac": summ_bytes / (summ_ms * 1e-3) / 1e9 / pk["hbm_gbs"]},
        "clocks": clk.summary(),
        "device_error_bits": err,
        "timing": plan_text(plan, steps),
    }
    res["e2e"] = e2e
    if cpu_leg:
        res["cpu_baseline"] = cpu_baseline_decode(db)
    return res, db


def time_decode_variant(db, steps, ws_n):
    """Times `steps` decode steps of a variant (graphs warmed first) and the
    attend launches alone; returns (step ms, attend ms, per-query bytes, plan)."""
    st = torch.cuda.current_stream(db.dev)
    db.build_summaries()
    per_q = db.algorithmic_bytes()
    n = db.w.n_q
    plan = decode_graphs(db, steps)
    g_att = db.graph(db.attend, n)
    g_att.replay()
    replay_plan(plan)                       # warm-up, right before the timed region
    torch.cuda.synchronize()
    barrier(ws_n)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_device(st)
    a.record(st)
    replay_plan(plan)
    b.record(st)
    torch.cuda.synchronize()
    step_ms = max_over_ranks(a.elapsed_time(b), ws_n) / steps
    att_reps = max(1, -(-steps // n))
    attend_ms = replay_ms(g_att, att_reps, st) / (att_reps * n)
    return step_ms, attend_ms, per_q, plan


def variant_line(db, steps, ws_n, extra):
    w = db.w
    step_ms, attend_ms, per_q, plan = time_decode_variant(db, steps, ws_n)
    n = w.n_q
    attend_bytes = sum(per_q[s % n][0] for s in range(steps)) / steps
    route_bytes = sum(per_q[s % n][1] for s in range(steps)) / steps
    err = ssa.ssa_workspace_error(db.ws)
    if db.wsg is not None:
        err |= ssa.ssa_workspace_error(db.wsg)
    pk = peaks()
    step_gbs = (attend_bytes + route_bytes) / (step_ms * 1e-3) / 1e9
    att_gbs = attend_bytes / (attend_ms * 1e-3) / 1e9
    out = {"workload": w.name, "value": job_throughput(1, step_ms * 1e-3, ws_n), "unit": "tok/s",
           "ms_per_step": step_ms, "steps": steps, "timing": plan_text(plan, steps),
           "attend_ms_per_step": attend_ms, "attend_bytes_per_step": attend_bytes,
           "route_bytes_per_step": route_bytes,
           "roofline": {"bound": "hbm", "achieved": round(step_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": round(step_gbs / pk["hbm_gbs"], 4), "traffic": None,
                        "kernel": "whole decode step (route + attend)", "peak_source": pk["source"],
                        "attend_only": {"achieved": round(att_gbs, 1), "frac": round(att_gbs / pk["hbm_gbs"], 4)}},
           "device_error_bits": err}
    out.update(extra)
    return out


def bench_decode_group(w, dev, steps, ws_n):
    """The same decode workload with group-shared selection (one top-k per
    kv-head group): each group's heads attend the same k spans, so a step
    streams k spans plus the local span per kv-head."""
    db = DecodeBench(w, dev, group=True)
    return variant_line(db, steps, ws_n, {"routing": "group-shared (one top-k per kv-head group), "
                                                     "ssa_decode_step_group"})


def bench_decode_10m(dev, steps, ws_n, cpu_leg):
    """Decode with a 10M-token cache (S 3072, 3255 candidate spans), per-head
    selection, to set against the 1M line: the pages report decode slowing by
    about 30% from 1M to 10M."""
    w = W.DECODE_10M
    db = DecodeBench(w, dev)
    out = variant_line(db, steps, ws_n, {"L": w.L, "S": w.S})
    if cpu_leg:
        out["cpu_baseline"] = cpu_baseline_decode_10m(db)
    del db
    torch.cuda.empty_cache()
    return out


def bench_decode_q8(w, dev, steps, ws_n):
    """The same decode workload over the 8-bit cache (per-head selection on
    the summaries of the dequantised keys): a step streams the same spans
    at 2 d + 8 bytes per token instead of 4 d."""
    db = DecodeBench(w, dev, q8=True)
    out = variant_line(db, steps, ws_n, {"cache": "8-bit K / V, one fp32 scale per token row; fp32 summaries"})
    tr, tr_src = traffic_of(w.name + "_q8")
    out["roofline"]["traffic"], out["roofline"]["traffic_source"] = tr, tr_src
    return out


def bench_decode_q4(w, dev, steps, ws_n):
    """The same decode workload over the 4-bit cache: a step streams the
    same spans at d + 8 bytes per token."""
    db = DecodeBench(w, dev, q4=True)
    out = variant_line(db, steps, ws_n, {"cache": "4-bit K / V, one fp32 scale per token row; fp32 summaries"})
    tr, tr_src = traffic_of(w.name + "_q4")
    out["roofline"]["traffic"], out["roofline"]["traffic_source"] = tr, tr_src
    del db
    torch.cuda.empty_cache()
    return out


def bench_decode_e2e(db: DecodeBench, steps: int):
    """Same decode through the C ABI with host buffers, one token in and one
    out per step, each step waited for.  Two forms:

    * the headline: cudaMemcpyAsync of Q in from page-locked host memory,
      ssa_decode_step on device buffers, cudaMemcpyAsync of O out, then a
      stream synchronise;
    * mapped host buffers: ssa_decode_step on page-locked host Q, sel and O
      (the route kernel reads the step's query over the host link, the
      merge writes the output back over it), then a stream synchronise.

    The calls go straight to the C ABI and to the CUDA runtime (ctypes,
    arguments prepared once), so the loop measures the library and the data
    movement, not Python tensor calls."""
    w = db.w
    st = torch.cuda.current_stream(db.dev)
    el = db.Q.element_size()
    nbytes = w.B * w.Hq * w.d * el
    q_host = db.Q.cpu().pin_memory()                       # [steps, B, Hq, d]
    o_host = torch.empty((w.B, w.Hq, w.d), dtype=w.dtype).pin_memory()
    q_dev = torch.empty((w.B, w.Hq, w.d), dtype=w.dtype, device=db.dev)
    rt = ctypes.CDLL("libcudart.so.13")
    rt.cudaMemcpyAsync.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                                   ctypes.c_void_p]
    rt.cudaStreamSynchronize.argtypes = [ctypes.c_void_p]
    L = ssa.lib()
    sp = ctypes.c_void_p(st.cuda_stream)
    pp = ctypes.byref(db.p)
    qd, od = ctypes.c_void_p(q_dev.data_ptr()), ctypes.c_void_p(db.O.data_ptr())
    oh = ctypes.c_void_p(o_host.data_ptr())
    summ, sel = ctypes.c_void_p(db.summ.data_ptr()), ctypes.c_void_p(db.sel.data_ptr())
    K, V = ctypes.c_void_p(db.K.data_ptr()), ctypes.c_void_p(db.V.data_ptr())
    ws, wsn = ctypes.c_void_p(db.ws.data_ptr()), db.ws.numel()
    qh = [ctypes.c_void_p(q_host.data_ptr() + i * nbytes) for i in range(w.n_q)]

    sel_host = torch.empty(db.sel.shape, dtype=torch.int32).pin_memory()
    selh = ctypes.c_void_p(sel_host.data_ptr())

    def copies(s):
        i = s % w.n_q
        pos = w.q_pos0 + i
        rc = rt.cudaMemcpyAsync(qd, qh[i], nbytes, 1, sp)
        rc |= L.ssa_decode_step(pp, qd, pos, summ, K, V, sel, od, None, ws, wsn, sp)
        rc |= rt.cudaMemcpyAsync(oh, od, nbytes, 2, sp)
        rc |= rt.cudaStreamSynchronize(sp)
        return rc

    def mapped(s):
        i = s % w.n_q
        rc = L.ssa_decode_step(pp, qh[i], w.q_pos0 + i, summ, K, V, selh, oh, None, ws, wsn, sp)
        rc |= rt.cudaStreamSynchronize(sp)
        return rc

    # at least 512 timed steps after 64 warm-up ones: a few tens of steps
    # (about a millisecond of wall time) mostly time the host thread and the
    # GPU coming out of idle, not the steady per-token cost
    n_e2e = max(steps, 512)

    def rate(one):
        for s in range(64):
            if one(s):
                raise RuntimeError("e2e decode step failed")
        t0 = time.perf_counter()
        bad = 0
        for s in range(n_e2e):
            bad |= one(s)
        dt = time.perf_counter() - t0
        if bad:
            raise RuntimeError("e2e decode step failed")
        return n_e2e / dt

    sel_bytes = sel_host.numel() * 4
    return {"value": rate(copies), "unit": "tok/s", "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes,
            "steps": n_e2e, "warmup": 64,
            "clocks": "not sampled during this loop: the nvidia-smi sampler's polling slows host-side CUDA "
                      "calls, so it runs only around the device-timed regions",
            "how": "cudaMemcpyAsync Q in from page-locked host memory, ssa_decode_step, cudaMemcpyAsync O out, "
                   "stream synchronise",
            "mapped_host": {"value": rate(mapped), "unit": "tok/s", "h2d_bytes_per_step": nbytes,
                            "d2h_bytes_per_step": nbytes + sel_bytes,
                            "how": "ssa_decode_step on page-locked host Q / sel / O: the route reads Q and the "
                                   "merge writes O over the host link; stream synchronise"}}


def cpu_baseline_decode(db: DecodeBench, budget_s: float = 15.0):
    """The oracle (as it stands) on the host cores, on a bounded sample of decode steps."""
    import oracle
    w = db.w
    inp = db.inp
    K = inp.k("cpu")
    V = inp.v("cpu")
    Q = inp.q("cpu")
    summ = oracle.summaries(K, w.L, w.S)
    n = 0
    t0 = time.perf_counter()
    while n < w.n_q:
        q = Q[n].reshape(w.B, w.Hq, 1, w.d).contiguous()
        sel, _ = oracle.route(q, w.q_pos0 + n, summ, w.Hkv, w.S, w.topk)
        oracle.attend(q, K, V, w.q_pos0 + n, w.S, sel)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    del K, V
    return {"value": n / dt, "unit": "tok/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": "%d of the %d decode steps (route + attend per step; summaries of the 1M "
                      "cache built beforehand, untimed)" % (n, w.n_q)}


def cpu_baseline_decode_10m(db: DecodeBench, n_steps: int = 12):
    """The oracle on the host cores on sampled steps of the 10M decode.  The
    20 GB cache is never held on the host: the oracle's summaries come from
    host regenerations of span ranges and each step's attention runs on the
    compacted cache of its selected spans (both prepared untimed); the timed
    part is the oracle's route and attend of every sampled step."""
    import oracle
    from oracle import streamed
    w = db.w
    inp = db.inp
    Q = inp.q("cpu")
    summ = streamed.summaries_streamed(inp)
    steps = np.linspace(0, w.n_q - 1, n_steps).astype(int)
    tot = 0.0
    for s in steps:
        t = w.q_pos0 + int(s)
        q = Q[s].reshape(w.B, w.Hq, 1, w.d).contiguous()
        t0 = time.perf_counter()
        sel, _ = oracle.route(q, t, summ, w.Hkv, w.S, w.topk)
        tot += time.perf_counter() - t0
        for _, qc, Kc, Vc, pos, sel_c in streamed.compact_decode_step(inp, Q[s], sel, t):
            t0 = time.perf_counter()
            oracle.attend(qc, Kc, Vc, pos, w.S, sel_c)
            tot += time.perf_counter() - t0
    return {"value": len(steps) / tot, "unit": "tok/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": "%d of the %d decode steps, evenly spaced (route over the 3255 candidate summaries + "
                      "attend on each step's compacted cache of selected spans; summaries and compaction "
                      "untimed)" % (len(steps), w.n_q)}


def cpu_baseline_prefill_rows(w: W.Workload, inp: W.Inputs, Q, K, V, q_pos0: int, n_q: int,
                              budget_s: float = 10.0, batch: int = 512, seed: int = 5):
    """The oracle's route + attend on random (query, head) rows of one chunk
    of queries, for about budget_s seconds.  Returns (rows per second, rows)."""
    import oracle
    summ = oracle.summaries(K, q_pos0 + n_q, w.S, 0, (q_pos0 + n_q) // w.S)
    n_rows = w.B * w.Hq * n_q
    rng = np.random.default_rng(seed)
    order = rng.permutation(n_rows)
    done, tot = 0, 0.0
    while done < n_rows and tot < budget_s:
        rows = np.sort(order[done: done + batch])
        t0 = time.perf_counter()
        sel, _ = oracle.route(Q, q_pos0, summ, w.Hkv, w.S, w.topk, rows=rows)
        oracle.attend(Q, K, V, q_pos0, w.S, sel, rows=rows)
        tot += time.perf_counter() - t0
        done += len(rows)
    return done / tot, done


# --------------------------------------------------------------------- prefill
class PrefillBench:
    """One chunk of queries against an existing cache (summaries of the chunk's
    spans, route, attend)."""

    def __init__(self, w: W.Workload, dev):
        self.w = w
        self.dev = dev
        self.inp = W.Inputs(w)
        self.K = self.inp.k(dev)
        self.V = self.inp.v(dev)
        self.Q = self.inp.q(dev)                               # [B, Hq, n_q, d]
        self.p = ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L, w.S, w.topk, w.dtype)
        self.summ = torch.zeros((w.B, w.Hkv, w.n_spans, w.d), dtype=torch.float32, device=dev)
        self.sel = torch.empty((w.B, w.Hq, w.n_q, w.topk), dtype=torch.int32, device=dev)
        self.O = torch.empty_like(self.Q)
        self.lse = torch.empty((w.B, w.Hq, w.n_q), dtype=torch.float32, device=dev)
        self.ws = ssa.workspace(self.p, w.n_q, ssa.SSA_OP_PREFILL, dev)
        self.ws_route = ssa.workspace(self.p, w.n_q, ssa.SSA_OP_ROUTE, dev)
        self.stream = torch.cuda.current_stream(dev)
        self.j0 = w.q_pos0 // w.S
        self.j1 = w.n_spans
        pre = ssa.params(w.B, w.Hq, w.Hkv, w.d, w.q_pos0, w.S, w.topk, w.dtype, L_cap=w.L)
        if self.j0 > 0:
            ssa.ssa_build_summaries(pre, self.K, 0, self.j0, self.summ)

    def step(self, ev=None):
        """One chunk; ev (optional): three events, recorded before the route,
        before the attend path and at the end."""
        w = self.w
        ssa.ssa_build_summaries(self.p, self.K, self.j0, self.j1, self.summ, self.stream)
        if ev is not None:
            ev[0].record(self.stream)
        ssa.ssa_route(self.p, self.Q, w.n_q, w.q_pos0, self.summ, self.sel, None, self.ws_route,
                      self.stream)
        if ev is not None:
            ev[1].record(self.stream)
        ssa.ssa_attend_prefill(self.p, self.Q, w.n_q, w.q_pos0, self.K, self.V, self.sel, self.O,
                               self.lse, self.ws, self.stream)
        if ev is not None:
            ev[2].record(self.stream)

    def route_flops(self):
        """2 * d FLOP per candidate span per (query, head): the scores the router must compute."""
        w = self.w
        cand = (w.q_pos0 + np.arange(w.n_q)) // w.S
        return float(2 * w.d * w.B * w.Hq * cand.sum())

    def flops(self):
        w = self.w
        self.step()
        sel = self.sel.cpu().numpy()
        nsel = (sel >= 0).sum(axis=-1)                         # [B, Hq, n_q]
        pos = w.q_pos0 + np.arange(w.n_q)
        local = pos - (pos // w.S) * w.S + 1
        tokens = nsel * w.S + local[None, None, :]
        return float(4 * w.d * tokens.sum())


def time_ms(fn, reps, warmup, stream, flush=None):
    """Mean CUDA-event time of fn() over reps calls (L2 flushed before each when given)."""
    for _ in range(warmup):
        fn()
    tot = 0.0
    for _ in range(reps):
        if flush is not None:
            flush_l2(flush)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        tot += a.elapsed_time(b)
    return tot / reps


def bench_dense_comparison(dev, flush, decode_step_ms, prefill_1m_ms):
    """The pages' comparison point: dense attention over the whole context,
    here PyTorch's scaled_dot_product_attention (a library call, used for this
    measurement only; GQA native, bf16), on the same shapes as the routed
    lines.  The dense prefill chunk attends every query to the whole cache
    without a mask, so it also counts the chunk's own causal triangle (0.4%
    of its work at 1M); the dense decode step attends the whole cache."""
    import torch.nn.functional as F
    st = torch.cuda.current_stream(dev)
    out = {"dense": "torch scaled_dot_product_attention, enable_gqa, bf16, no mask"}
    # decode at 1M: one query per head
    w = W.DECODE_1M
    inp = W.Inputs(w)
    K, V = inp.k(dev), inp.v(dev)
    q = inp.q(dev)[0].reshape(w.B, w.Hq, 1, w.d)
    dense_dec = time_ms(lambda: F.scaled_dot_product_attention(q, K, V, enable_gqa=True), 20, 3, st, flush)
    out["decode_1m"] = {"routed_ms_per_step": decode_step_ms, "dense_ms_per_step": dense_dec,
                        "speedup": dense_dec / decode_step_ms if decode_step_ms else None}
    # prefill chunk of 8192 queries against 1M
    wp = W.PREFILL_1M
    Qp = W.Inputs(wp.with_(needles=0)).q(dev)
    dense_pre = time_ms(lambda: F.scaled_dot_product_attention(Qp, K, V, enable_gqa=True), 3, 1, st, flush)
    out["prefill_1m"] = {"routed_ms_per_chunk": prefill_1m_ms, "dense_ms_per_chunk": dense_pre,
                         "speedup": dense_pre / prefill_1m_ms if prefill_1m_ms else None}
    del K, V, q, Qp
    torch.cuda.empty_cache()
    # prefill: the last 8192-query chunk of the 128K workload, routed and dense
    w1 = W.PREFILL_128K.with_(n_q=8192, chunk=8192, q_pos0=W.PREFILL_128K.L - 8192)
    pb = PrefillBench(w1, dev)
    routed = time_ms(pb.step, 5, 2, st, flush)
    dense = time_ms(lambda: F.scaled_dot_product_attention(pb.Q, pb.K, pb.V, enable_gqa=True), 5, 2, st, flush)
    out["prefill_128k_last_chunk"] = {"routed_ms_per_chunk": routed, "dense_ms_per_chunk": dense,
                                      "speedup": dense / routed}
    del pb
    torch.cuda.empty_cache()
    return out


def tensor_roofline(flop: float, ms: float, what: str, traffic=None, traffic_source=None):
    """Selected-span FLOP over time against the measured burst bf16 peak (a
    chunk of a few milliseconds is a kernel timed on its own, not a seconds-
    long loop under the power cap); the sustained-peak fraction rides along."""
    pk = peaks()
    achieved = flop / (ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": round(achieved, 2), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
            "frac": round(achieved / pk["bf16_tflops"], 4), "traffic": traffic, "traffic_source": traffic_source,
            "kernel": what, "peak_source": pk["source"] + " burst bf16",
            "frac_of_sustained": round(achieved / pk["bf16_tflops_sustained"], 4)}


def bench_prefill(w, dev, steps, warmup, ws_n, flush, cpu_leg):
    pb = PrefillBench(w, dev)
    st = pb.stream
    fl = pb.flops()
    for _ in range(warmup):
        pb.step()
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    tot = 0.0
    barrier(ws_n)
    torch.cuda.synchronize()
    for s in range(steps):
        flush_l2(flush)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        pb.step(evs[s])
        b.record(st)
        torch.cuda.synchronize()
        tot += a.elapsed_time(b)
    barrier(ws_n)
    route_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / steps
    attend_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / steps
    rfl = pb.route_flops()
    ms = max_over_ranks(tot / steps, ws_n)
    err = ssa.ssa_workspace_error(pb.ws)
    tr, tr_src = traffic_of(w.name)
    out = {
        "workload": w.name, "value": job_throughput(w.n_q, ms * 1e-3, ws_n), "unit": "tok/s",
        "ms_per_step": ms, "attend_ms": attend_ms, "steps": steps,
        "l2": "flushed before every timed chunk (256 MiB write)",
        "roofline": tensor_roofline(fl, ms, "whole chunk: summaries + route + attend (4*d FLOP per attended "
                                            "token per query head over the selected spans and the local span)"),
        "attend_roofline": tensor_roofline(fl, attend_ms, "attend path alone (dispatch + attend + merge)", tr, tr_src),
        "route_ms": route_ms,
        "route_roofline": tensor_roofline(rfl, route_ms, "route alone (split + tensor-core scores + top-k): "
                                                         "2*d FLOP per candidate span per query head; the split "
                                                         "summaries make the tensor cores issue 3x that"),
        "selected_span_tflop_per_step": fl / 1e12,
        "device_error_bits": err,
    }
    if cpu_leg:
        inp = pb.inp
        Q, K, V = inp.q("cpu"), inp.k("cpu"), inp.v("cpu")
        rps, n = cpu_baseline_prefill_rows(w, inp, Q, K, V, w.q_pos0, w.n_q)
        import oracle
        out["cpu_baseline"] = {"value": rps / w.Hq, "unit": "tok/s", "cores": oracle.threads(), "kind": "oracle",
                               "sample": "%d random (query, head) rows of the chunk's %d, route + attend; "
                                         "tok/s = rows/s / Hq" % (n, w.B * w.Hq * w.n_q)}
        del Q, K, V
    del pb
    torch.cuda.empty_cache()
    return out


class Prefill128kBench:
    """The whole 128K prefill: 16 chunks of 8192 queries, each one's K / V
    already in the cache; a chunk builds the summaries of the spans it
    completes, routes its queries and attends them."""

    def __init__(self, w: W.Workload, dev):
        self.w = w
        self.dev = dev
        self.inp = W.Inputs(w)
        self.K = self.inp.k(dev)
        self.V = self.inp.v(dev)
        Q = self.inp.q(dev)                                   # [B, Hq, L, d]
        self.chunks = []
        for c0 in range(0, w.n_q, w.chunk):
            n = min(w.chunk, w.n_q - c0)
            self.chunks.append((c0, n, Q[:, :, c0:c0 + n].contiguous()))
        del Q
        self.p_full = ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L, w.S, w.topk, w.dtype)
        self.summ = torch.zeros((w.B, w.Hkv, w.n_spans, w.d), dtype=torch.float32, device=dev)
        self.sel = [torch.empty((w.B, w.Hq, n, w.topk), dtype=torch.int32, device=dev) for _, n, _ in self.chunks]
        self.O = [torch.empty_like(q) for _, _, q in self.chunks]
        self.lse = [torch.empty((w.B, w.Hq, n), dtype=torch.float32, device=dev) for _, n, _ in self.chunks]
        self.ws = ssa.workspace(self.p_full, w.chunk, ssa.SSA_OP_PREFILL, dev)
        self.ws_route = ssa.workspace(self.p_full, w.chunk, ssa.SSA_OP_ROUTE, dev)
        self.stream = torch.cuda.current_stream(dev)
        self.rstream = torch.cuda.Stream(dev)     # summaries + route, a chunk ahead

    def run(self, evs=None):
        """The chunks as a two-stream pipeline: chunk c + 1's summaries and
        route (which read the cache and its own queries only) run on a second
        stream while chunk c attends and merges; each chunk's attention
        waits for its own selections.  Every launch is the same as in a
        one-stream loop; only their overlap differs."""
        w = self.w
        start = torch.cuda.Event()
        start.record(self.stream)
        self.rstream.wait_event(start)
        for c, (c0, n, q) in enumerate(self.chunks):
            L_now = c0 + n
            p = ssa.params(w.B, w.Hq, w.Hkv, w.d, L_now, w.S, w.topk, w.dtype, L_cap=w.L)
            ssa.ssa_build_summaries(p, self.K, c0 // w.S, (L_now + w.S - 1) // w.S, self.summ, self.rstream)
            ssa.ssa_route(p, q, n, c0, self.summ, self.sel[c], None, self.ws_route, self.rstream)
            routed = torch.cuda.Event()
            routed.record(self.rstream)
            self.stream.wait_event(routed)
            ssa.ssa_attend_prefill(p, q, n, c0, self.K, self.V, self.sel[c], self.O[c], self.lse[c], self.ws,
                                   self.stream)
            if evs is not None:
                evs[c].record(self.stream)

    def flops(self):
        w = self.w
        self.run()
        tot = 0.0
        for c, (c0, n, _) in enumerate(self.chunks):
            sel = self.sel[c].cpu().numpy()
            nsel = (sel >= 0).sum(axis=-1)
            pos = c0 + np.arange(n)
            local = pos - (pos // w.S) * w.S + 1
            tot += float(4 * w.d * (nsel * w.S + local[None, None, :]).sum())
        return tot


def bench_prefill_128k(dev, steps, ws_n, flush, cpu_leg):
    """The 128K chunked prefill as a whole: 131072 / (time of all 16 chunks)."""
    w = W.PREFILL_128K
    pb = Prefill128kBench(w, dev)
    st = pb.stream
    fl = pb.flops()
    pb.run()
    torch.cuda.synchronize()
    nch = len(pb.chunks)
    tot, per_chunk = 0.0, np.zeros(nch)
    barrier(ws_n)
    for _ in range(steps):
        flush_l2(flush)
        a = torch.cuda.Event(enable_timing=True)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(nch)]
        a.record(st)
        pb.run(evs)
        torch.cuda.synchronize()
        tot += a.elapsed_time(evs[-1])
        prev = a
        for c in range(nch):
            per_chunk[c] += prev.elapsed_time(evs[c])
            prev = evs[c]
    barrier(ws_n)
    ms = max_over_ranks(tot / steps, ws_n)
    err = ssa.ssa_workspace_error(pb.ws)
    out = {"workload": w.name, "value": job_throughput(w.n_q, ms * 1e-3, ws_n), "unit": "tok/s",
           "ms_per_prefill": ms, "steps": steps, "chunks": nch,
           "ms_per_chunk": [round(x / steps, 4) for x in per_chunk],
           "l2": "flushed before every timed prefill (256 MiB write); K / V are 512 MiB",
           "schedule": "two streams: chunk c + 1's summaries and route run while chunk c attends and merges; "
                       "each chunk's attention waits for its own route",
           "roofline": tensor_roofline(fl, ms, "all 16 chunks: summaries + route + attend (4*d FLOP per attended "
                                               "token per query head)"),
           "selected_span_tflop": fl / 1e12, "device_error_bits": err}
    if cpu_leg:
        import oracle
        inp = pb.inp
        Q, K, V = inp.q("cpu"), inp.k("cpu"), inp.v("cpu")
        c0 = w.n_q - w.chunk
        # rows drawn from the whole prefill at once: each row's oracle cost is
        # its route over its own candidates plus its attention, so the sample
        # stands for every chunk, early and late
        rps, n = cpu_baseline_prefill_rows(w, inp, Q, K, V, 0, w.n_q, budget_s=10.0)
        out["cpu_baseline"] = {"value": rps / w.Hq, "unit": "tok/s", "cores": oracle.threads(), "kind": "oracle",
                               "sample": "%d random (query, head) rows drawn from all 131072 queries, route + "
                                         "attend; tok/s = rows/s / Hq" % n}
        del Q, K, V
    del pb
    torch.cuda.empty_cache()
    return out


def bench_tiny(dev, steps, ws_n, cpu_leg):
    """The tiny fp32 prefill (4096 queries, 4 heads, d 64, S 64, k 8) in one
    chunk: summaries + route + attend, tok/s = 4096 / time."""
    w = W.TINY_PREFILL
    inp = W.Inputs(w)
    Q, K, V = inp.q(dev), inp.k(dev), inp.v(dev)
    p = ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L, w.S, w.topk, w.dtype)
    summ = torch.zeros((w.B, w.Hkv, w.n_spans, w.d), dtype=torch.float32, device=dev)
    sel = torch.empty((w.B, w.Hq, w.n_q, w.topk), dtype=torch.int32, device=dev)
    O = torch.empty_like(Q)
    lse = torch.empty((w.B, w.Hq, w.n_q), dtype=torch.float32, device=dev)
    ws = ssa.workspace(p, w.n_q, ssa.SSA_OP_PREFILL, dev)
    wsr = ssa.workspace(p, w.n_q, ssa.SSA_OP_ROUTE, dev)
    st = torch.cuda.current_stream(dev)

    def run():
        ssa.ssa_build_summaries(p, K, 0, w.n_spans, summ)
        ssa.ssa_route(p, Q, w.n_q, 0, summ, sel, None, wsr)
        ssa.ssa_attend_prefill(p, Q, w.n_q, 0, K, V, sel, O, lse, ws)

    ms = max_over_ranks(time_ms(run, max(steps, 3), 3, st), ws_n)
    out = {"workload": w.name, "value": job_throughput(w.n_q, ms * 1e-3, ws_n), "unit": "tok/s",
           "ms_per_step": ms, "steps": max(steps, 3),
           "roofline": {"bound": "n/a", "note": "fp32 parity workload of 4096 queries; no roofline claimed"},
           "device_error_bits": ssa.ssa_workspace_error(ws)}
    if cpu_leg:
        import oracle
        Qh, Kh, Vh = inp.q("cpu"), inp.k("cpu"), inp.v("cpu")
        t0 = time.perf_counter()
        summ_o = oracle.summaries(Kh, w.L, w.S)
        sel_o, _ = oracle.route(Qh, 0, summ_o, w.Hkv, w.S, w.topk)
        oracle.attend(Qh, Kh, Vh, 0, w.S, sel_o)
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": w.n_q / dt, "unit": "tok/s", "cores": oracle.threads(), "kind": "oracle",
                               "sample": "the whole workload: summaries + route + attend of all 4096 queries"}
    return out


# --------------------------------------------------------------------- reference arm
def run_reference(args, ws_n, rank):
    """The oracle timed on the host cores on the decode workload (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    w = W.DECODE_1M
    inp = W.Inputs(w)
    K, V, Q = inp.k("cpu"), inp.v("cpu"), inp.q("cpu")
    summ = oracle.summaries(K, w.L, w.S)

    def one(s):
        i = s % w.n_q
        q = Q[i].reshape(w.B, w.Hq, 1, w.d).contiguous()
        sel, _ = oracle.route(q, w.q_pos0 + i, summ, w.Hkv, w.S, w.topk)
        oracle.attend(q, K, V, w.q_pos0 + i, w.S, sel)

    for s in range(args.warmup):
        one(s)
    t0 = time.perf_counter()
    for s in range(args.steps):
        one(s)
    dt = time.perf_counter() - t0
    v = args.steps / dt
    line = {"metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": ws_n, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                       "L": w.L, "S": w.S, "topk": w.topk},
            "cpu_baseline": {"value": v, "unit": "tok/s", "cores": oracle.threads(),
                             "kind": "oracle",
                             "sample": "%d decode steps of the 1M-cache workload" % args.steps},
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--prefill-steps", type=int, default=5)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-L", type=int, default=None,
                    help="shrink the decode cache (profiling runs on a smaller case)")
    ap.add_argument("--prefill-L", type=int, default=None,
                    help="shrink the prefill cache (profiling runs on a smaller case)")
    ap.add_argument("--prefill-chunk", type=int, default=None,
                    help="queries of the prefill chunk (profiling runs on a smaller case)")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-main-decode", action="store_true",
                    help="skip the 16-bit per-head decode line only (the decode variant lines still run)")
    ap.add_argument("--no-dense", action="store_true",
                    help="skip the dense-attention comparison (PyTorch SDPA on the same shapes)")
    ap.add_argument("--no-group", action="store_true",
                    help="skip the decode line with group-shared selection")
    ap.add_argument("--no-q8", action="store_true",
                    help="skip the decode line over the 8-bit cache")
    ap.add_argument("--no-q4", action="store_true",
                    help="skip the decode line over the 4-bit cache")
    ap.add_argument("--no-10m", action="store_true",
                    help="skip the decode line with a 10M-token cache")
    ap.add_argument("--no-128k", action="store_true",
                    help="skip the whole 128K chunked prefill")
    ap.add_argument("--no-chunk", action="store_true",
                    help="skip the 8192-query chunk against the 1M cache")
    ap.add_argument("--no-tiny", action="store_true",
                    help="skip the tiny fp32 prefill")
    args = ap.parse_args()
    if args.impl == "reference":
        # the oracle runs on the host cores only: no process group, no GPU
        args.steps = args.steps if args.steps is not None else 3
        args.warmup = args.warmup if args.warmup is not None else 1
        run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
        return
    ws_n, rank, local = dist_setup()
    steps = args.steps if args.steps is not None else 2048
    warmup = max(3, args.warmup if args.warmup is not None else 256)
    dev = torch.device("cuda", local)
    ssa.lib()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # > L2 (126 MB)
    cpu_leg = rank == 0 and ws_n == 1 and not args.no_cpu_baseline
    small = bool(args.decode_L or args.prefill_L or args.prefill_chunk)

    w = W.DECODE_1M
    if args.decode_L:
        w = w.with_(name="decode_%d" % args.decode_L, L=args.decode_L, q_pos0=args.decode_L - w.n_q)
    if args.no_decode or args.no_main_decode:
        dec = {"tok_s": None, "ms_per_step": None, "roofline": None, "e2e": None, "clocks": None,
               "attend_ms_per_step": None, "route_plus_gaps_ms_per_step": None,
               "attend_bytes_per_step": None, "route_bytes_per_step": None,
               "summaries": None, "device_error_bits": None, "timing": None}
    else:
        dec, db = bench_decode(w, dev, steps, warmup, ws_n, cpu_leg)
        del db
    torch.cuda.empty_cache()
    line = {
        "metric": METRIC, "value": dec["tok_s"], "unit": "tok/s", "n_gpus": ws_n, "steps": steps,
        "warmup": warmup, "ms_per_step": dec["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "L": w.L,
                   "S": w.S, "topk": w.topk, "queries": "%d distinct decode queries at positions "
                   "%d..%d, cycled" % (w.n_q, w.q_pos0, w.last_pos),
                   "l2": "inputs larger than L2: 2 GiB K/V cache, ~220 MB gathered per step",
                   "parallelism": "replicas" if ws_n > 1 else "single GPU"},
        "roofline": dec["roofline"],
        "e2e": dec["e2e"],
        "clocks": dec["clocks"],
        "gpu_launches": steps * launches_per_decode_step(w) if dec["tok_s"] is not None else 0,
        "decode_detail": {k: dec[k] for k in ("attend_ms_per_step", "route_plus_gaps_ms_per_step",
                                               "attend_bytes_per_step", "route_bytes_per_step",
                                               "summaries", "device_error_bits", "timing")},
    }
    if "cpu_baseline" in dec:
        line["cpu_baseline"] = dec["cpu_baseline"]
    if not args.no_decode and not args.no_group:
        line["decode_group_shared"] = bench_decode_group(w, dev, steps, ws_n)
        torch.cuda.empty_cache()
    if not args.no_decode and not args.no_q8:
        line["decode_q8"] = bench_decode_q8(w, dev, steps, ws_n)
        torch.cuda.empty_cache()
    if not args.no_decode and not args.no_q4:
        line["decode_q4"] = bench_decode_q4(w, dev, steps, ws_n)
        torch.cuda.empty_cache()
    if not args.no_decode and not args.no_10m and not small:
        d10 = bench_decode_10m(dev, steps, ws_n, cpu_leg)
        d10["vs_1m"] = d10["value"] / dec["tok_s"] if dec["tok_s"] else None
        line["decode_10m"] = d10
        torch.cuda.empty_cache()
    pre = None
    if not args.no_prefill and not args.no_chunk:
        wp = W.PREFILL_1M
        if args.prefill_L or args.prefill_chunk:
            L = args.prefill_L or wp.L
            n = args.prefill_chunk or wp.n_q
            wp = wp.with_(name="prefill_%d_vs_%d" % (n, L), L=L, n_q=n, chunk=n, q_pos0=L - n)
        pre = bench_prefill(wp, dev, args.prefill_steps, 2, ws_n, flush, cpu_leg)
        line["prefill"] = pre
        torch.cuda.empty_cache()
    if not args.no_prefill and not args.no_128k and not small:
        line["prefill_128k"] = bench_prefill_128k(dev, max(1, args.prefill_steps // 2), ws_n, flush, cpu_leg)
        torch.cuda.empty_cache()
    if not args.no_tiny and not small:
        line["tiny_prefill"] = bench_tiny(dev, args.prefill_steps, ws_n, cpu_leg)
        torch.cuda.empty_cache()
    if (not args.no_dense and dec["ms_per_step"] is not None and pre is not None and ws_n == 1 and not small):
        torch.cuda.empty_cache()
        line["dense_comparison"] = bench_dense_comparison(dev, flush, dec["ms_per_step"], pre["ms_per_step"])
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def launches_per_decode_step(w) -> int:
    """Kernels one ssa_decode_step launches: on the 16-bit path the route
    (which also builds the attend plan), the split attention and the merge;
    the fp32 path runs the route and one row kernel."""
    p = ssa.params(w.B, w.Hq, w.Hkv, w.d, w.L, w.S, w.topk, w.dtype)
    fast = ssa.ssa_workspace_size(p, 1, ssa.SSA_OP_DECODE) > 256
    return 3 if fast else 2


if __name__ == "__main__":
    main()
