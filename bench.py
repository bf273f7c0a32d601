#!/usr/bin/env python3
"""Benchmark of the hierarchical KV cache resolver on GB300: top-k selections resolved per second.

A step is one decode step of a synthetic workload: hs_step_begin plus the resolution of every layer for every
request, captured once per step of the workload's selection sequence into a CUDA graph and replayed. The
sequence starts from an empty cache, so the first step is the all-miss cold start; when K exceeds the sequence
the pool is reset (outside the timed intervals) and the sequence restarts. One selection = one request-layer's
top-k list for one step.

Default run: every workload. The headline (the top-level value, roofline, noio, e2e and cpu_baseline) is the
largest one, the shared-selection workload (8 requests x 78 layers, context 1,048,576, one top-k 2048 selection
per request and step shared by all layers) with hs_prefetch(l+1) on a second stream overlapped with
hs_resolve(l). The other workloads, and the shared one with a single hs_resolve_shared per step, are in
``per_workload`` with the same fields. ``--workload NAME`` measures one workload.

Timing: W warm-up steps, then K steps, each bracketed by CUDA events on the launching stream with a 256 MiB L2
flush between steps (outside the events), barrier + synchronize around the whole region, max over ranks. A GPU-side
spin of about 5 ms precedes each timed pass (outside the events) so that every step is enqueued before the GPU
reaches it. Clocks are sampled with nvidia-smi during the timed regions.

Roofline (the slower of two terms): miss-row bytes over the measured host link, and metadata + hot-buffer bytes
over HBM (measured copy peak). The resolve kernels' duration is bounded by the step graph's, which is used.
``floor`` is the same step with every resolve replaced by a kernel that does nothing, launched with the resolve's
exact configuration (hs_probe_launch): the cost of launching alone.

Also reported: e2e (the same steps through the public API on the host clock, host buffers in and out), a no-IO
run (misses sourced from an HBM copy of the pool), and the CPU oracle on a bounded sample (``cpu_baseline``).

``--gpus N`` without an external launcher starts N replica processes (one GPU and one pool each; gloo only for
the barrier and the max-over-ranks time). ``--impl reference`` times the CPU oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import socket
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workload as wl  # noqa: E402

METRIC = "top-k selections resolved/s"
UNIT = "selections/s"
FLUSH_BYTES = 256 << 20
MLA_SCALE = 1.0 / math.sqrt(192.0)  # softmax scale of the attention consumer: 1/sqrt(128 + 64)
HEADLINE = ("shared", {"prefetch": True})
# The headline workload's 78 layers need 429 GB of host pool, so its layers share one pool; a layer reading the pages
# the previous layer just read (the same tokens, shifted rows) is much faster than one reading a pool of its own. The
# same pipeline on 16 of its layers, each with a host pool of its own (88 GB), measures the per-layer cost without
# that reuse.
OWN_POOL_LAYERS = 16
# (workload, mode) of the default run after the headline; modes of one workload are adjacent so its pool is reused
DEFAULT_SET = [("shared", {"prefetch": True, "prefetch_depth": 2}), ("shared", {"prefetch": True, "prefetch_depth": 4}),
               ("shared", {"shared_call": True}), ("shared", {"full_offload": True}),
               (f"shared_own{OWN_POOL_LAYERS}", {"prefetch": True}), ("tiny", {}), ("dsa", {}),
               ("dsa", {"full_offload": True}), ("multilayer", {}), ("quest", {})]
HIDING_WORK_MB = 64.0  # per-layer work stand-in of the prefetch-hiding measurement on the headline workload
# Before a timed pass the stream first runs a spin of this many GPU cycles (about 97 ms at 2.07 GHz), outside the
# timed intervals: the host then enqueues every step of the pass while the GPU is still busy, so a stall of the host
# thread (the host may be a shared virtual machine) cannot fall between a step's start event and its graph launch. A
# 5 ms spin was seen to run out on a pass whose host thread took about 1 ms per step to enqueue, and the steps after
# that point then measured the host (0.2-1 ms each against 0.05 ms); stalls of more than 48 ms were seen too. (A
# kernel that holds the stream until the host releases it does not serve: with the GPU held, the launch queue fills
# and the host blocks before it can release, and first launches wait for the device to go idle.)
LEAD_CYCLES = 200_000_000
HBM_NOMINAL_GBS = 8000.0  # the nominal HBM3e rate ("about 8 TB/s"), reported beside the measured copy peak


def workload_of(name: str) -> wl.Workload:
    """A workload by name; `shared_own<N>` is the headline workload on N layers (each with a host pool of its own
    wherever they fit)."""
    if name.startswith("shared_own") and name[len("shared_own"):].isdigit():
        return dataclasses.replace(wl.WORKLOADS["shared"], layers=int(name[len("shared_own"):]))
    return wl.WORKLOADS[name]


def describe(w: wl.Workload) -> str:
    sel = "shared by all layers" if w.shared_across_layers else "per layer"
    return (f"{w.name}: {w.requests} requests x {w.layers} layers, ctx {w.ctx}, top-k {w.topk} ({sel}), "
            f"{w.slots} hot slots, {w.row_bytes}-B rows, {w.steps} steps")


def mode_name(mode: dict) -> str:
    on = [k for k in ("prefetch", "shared_call", "full_offload", "work_only", "attention") if mode.get(k)]
    if mode.get("prefetch") and mode.get("prefetch_depth", 1) != 1:
        on[on.index("prefetch")] = f"prefetch_depth={mode['prefetch_depth']}"
    if mode.get("layer_work_mb"):
        on.append(f"layer_work_mb={mode['layer_work_mb']:g}")
    if mode.get("tiered_frac") is not None:
        on.append(f"tiered_frac={mode['tiered_frac']:g}")
    return "+".join(on) if on else "per-layer resolve"


def mem_available() -> int:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def choose_host_layers(w: wl.Workload, alias: bool = False) -> int:
    """All layers get their own host pool when it fits in half of the available host memory (and aliasing is not
    asked for); otherwise every layer reads one shared pool, shifted per layer (see Resources). Loads use
    ld.global.cv, so a shared pool still sends every miss over the link."""
    if w.layers == 1:
        return 1
    if alias:
        return 1
    return w.layers if w.host_bytes() < 0.5 * mem_available() else 1


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running (start/stop around each timed
    region; the summary covers all of them)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, args=(self.proc,), daemon=True).start()
        except OSError:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        time.sleep(0.15)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.proc = None

    def __enter__(self):
        self.start()
        return self

    def __exit__(self, *exc):
        self.stop()

    def _read(self, proc):
        for line in proc.stdout:
            self.lines.append(line.strip())

    def summary(self) -> dict:
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _sources_sha16(names) -> str:
    import hashlib

    from hierarchical_sparse_attention_hs_gb300 import build as hs_build

    csrc = os.path.join(os.path.dirname(hs_build.__file__), "csrc")
    parts = [hashlib.sha256(open(os.path.join(csrc, n), "rb").read()).hexdigest() for n in names]
    return hashlib.sha256("".join(parts).encode()).hexdigest()[:16]


def kernel_sources_sha16() -> str:
    """Hash of the files the resolve kernel is compiled from (its translation unit and the headers it includes),
    which a committed ncu capture of that kernel must match."""
    return _sources_sha16(("hs_resolve.cu", "hs_block.cuh", "hs_pool.hpp"))


def attention_sources_sha16() -> str:
    """Hash of the files the attention kernel is compiled from, which its committed ncu capture must match."""
    return _sources_sha16(("hs_attention.cu", "hs_pool.hpp"))


def _load_capture(name: str, sha_key: str, sha: str):
    try:
        with open(os.path.join(ROOT, "profiles", name)) as f:
            cap = json.load(f)
    except (OSError, ValueError):
        return None
    return cap if cap.get(sha_key) == sha else None


def captured_traffic(w: wl.Workload, cold_launches: int, steady_launches: int, noio: bool = False):
    """DRAM bytes per launch from the committed ncu capture of this workload (its no-IO form when `noio`), when
    the kernel sources are the ones it was taken on; else None."""
    suffix = "_noio" if noio else ""
    cap = _load_capture(f"hs_resolve_kernel_{w.name}{suffix}_ncu.json", "kernel_sources_sha16", kernel_sources_sha16())
    if cap is None:
        return None
    d = cap["dram_bytes_per_launch"]
    if d.get("cold") is None:  # a capture of steady launches only stands for every launch of the pass
        return d["steady"]
    n = cold_launches + steady_launches
    return (cold_launches * d["cold"] + steady_launches * d["steady"]) / n if n else None


def captured_attention_traffic(w: wl.Workload):
    """DRAM bytes per launch of the attention kernel from its committed ncu capture on this workload, when the
    kernel sources are the ones it was taken on; else None."""
    cap = _load_capture(f"hs_mla_decode_kernel_{w.name}_ncu.json", "attention_sources_sha16",
                        attention_sources_sha16())
    return None if cap is None else cap["dram_read_bytes"] + cap["dram_write_bytes"]


def meta_bytes_per_launch(w: wl.Workload, batch: int) -> int:
    """Metadata bytes of one resolve of one layer that do not depend on hits/misses: selection read, tok2slot
    gather, out_slots write (4k each) and the stamp + slot-token reads (8H), per request-layer."""
    return batch * (12 * w.topk + 8 * w.slots)


class Resources:
    """Device and host memory of one workload: the pool buffers (host pool, hot buffer, metadata), one pool handle
    that fetches over the host link and, for the no-IO runs, a second handle over the same hot buffer and metadata
    whose misses come from an HBM copy of the host pool; the selections of every step in device memory."""

    def __init__(self, w: wl.Workload, alias_host: bool = False, noio: bool = True, attention: bool = False,
                 tiered_frac: float | None = None, layer_shift_rows: int | None = None):
        import torch

        import hierarchical_sparse_attention_hs_gb300 as hs

        self.torch, self.hs, self.w = torch, hs, w
        self.host_layers = choose_host_layers(w, alias_host)
        # Layers that share one host pool read it shifted by ctx / layers rows per layer, so that layers selecting
        # the same tokens (a shared selection) read different host rows, as with a pool per layer. They still read
        # largely the same host pages, which keeps their fetches faster than a pool per layer's (scattered rows are
        # bound on the host's side, most likely by address translation); the own-pool entry measures the difference.
        if layer_shift_rows is None:
            layer_shift_rows = w.ctx // w.layers if self.host_layers == 1 and w.layers > 1 else 0
        self.buf = hs.PoolBuffers(w.layers, w.requests, w.ctx, w.slots, w.topk, w.row_bytes,
                                  host_layers=self.host_layers, noio=noio, layer_shift_rows=layer_shift_rows)
        wl.fill_host_pool(w, self.buf.host.ptr, self.host_layers, extra_rows=self.buf.extra_rows)
        self.pool = self.buf.create()
        self.noio_pool = None
        if noio:
            self.buf.upload_noio()
            self.noio_pool = hs.hs_pool_create(self.buf.desc)
        self.sel_host = wl.gen_selections(w)  # [steps][selection layers][B][k]
        self.sel = torch.from_numpy(self.sel_host).cuda()
        self.out = torch.full((w.layers, w.requests, w.topk), -1, dtype=torch.int32, device="cuda")
        self.flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.q = self.att_out = self.att_lse = None
        if attention:
            if w.row_bytes != hs.MLA_D_QK * 2:
                raise ValueError("attention needs 1152-byte rows (the mla workload)")
            self.q = torch.from_numpy(wl.gen_queries(w.requests, hs.MLA_HEADS, hs.MLA_D_QK, w.seed).view(np.int16)).cuda()
            self.att_out = torch.empty((w.requests, hs.MLA_HEADS, hs.MLA_D_V), dtype=torch.float32, device="cuda")
            self.att_lse = torch.empty((w.requests, hs.MLA_HEADS), dtype=torch.float32, device="cuda")
        self.res = None
        if tiered_frac is not None:
            self.res = torch.from_numpy(wl.gen_resident(w.ctx, w.requests, w.steps, w.seed, frac=tiered_frac)).cuda()
        torch.cuda.synchronize()

    def host_rows_layer0(self) -> np.ndarray:
        """Layer 0 of the host pool as uint8 [requests][ctx][row_bytes] (a view of the mapped buffer)."""
        w = self.w
        n = self.host_layers * w.requests * w.ctx * w.row_bytes
        return self.buf.host.numpy()[:n].reshape(self.host_layers, w.requests, w.ctx, w.row_bytes)[0]

    def counters(self) -> np.ndarray:
        return self.buf.view("counters").cpu().numpy().astype(np.int64).sum(axis=0)

    def close(self):
        if self.noio_pool:
            self.hs.hs_pool_destroy(self.noio_pool)
            self.noio_pool = None
        self.buf.close()
        self.buf.host.close()


class StepGraphs:
    """One CUDA graph per decode step of the sequence for a pool handle and a mode (prefetch, one shared call,
    per-layer work stand-in, full offload, three tiers, attention, or the launch floor). `sel_of(s, ls)` and
    `out_of(l)` give the selection and out_slots addresses (device tensors or mapped host memory); with
    `single` one graph serves every step (its selection buffer is refilled between replays)."""

    def __init__(self, res: Resources, pool: int, mode: dict, floor: bool = False, sel_of=None, out_of=None,
                 single: bool = False):
        torch, hs, w = res.torch, res.hs, res.w
        self.res, self.pool, self.mode, self.floor = res, pool, dict(mode), floor
        self.torch, self.hs, self.w = torch, hs, w
        self.sel_of = sel_of or (lambda s, ls: res.sel[s][ls])
        self.out_of = out_of or (lambda l: res.out[l])
        self.stream = torch.cuda.Stream()
        self.depth = int(mode.get("prefetch_depth", 1)) if mode.get("prefetch") else 0
        self.sides = [torch.cuda.Stream() for _ in range(self.depth)]
        self.shared_call = bool(mode.get("shared_call")) and w.shared_across_layers
        self.layer_work = bool(mode.get("layer_work_mb")) or bool(mode.get("work_only"))
        if mode.get("full_offload"):
            self.offload_buf = torch.empty(w.requests * w.topk * w.row_bytes, dtype=torch.uint8, device="cuda")
        if self.layer_work:
            self.gather_buf = torch.empty(w.requests * w.topk * w.row_bytes, dtype=torch.uint8, device="cuda")
            nb = max(16, int(mode.get("layer_work_mb", 0.0) * (1 << 20)) // 16 * 16)
            self.work_src = torch.ones(nb, dtype=torch.uint8, device="cuda")
            self.work_dst = torch.empty(nb, dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()
        self.graphs = [self._capture(s) for s in range(1 if single else w.steps)]
        torch.cuda.synchronize()

    def _lsel(self, l):
        return 0 if self.w.shared_across_layers else l

    # one resolve-like call: the real one, or an empty kernel with its launch configuration
    def _resolve(self, l, sel, out, st):
        if self.floor:
            self.hs.hs_probe_launch(self.pool, l, 1, self.w.requests, self.w.topk, st)
        elif self.res.res is not None:
            self.hs.hs_resolve_tiered(self.pool, l, self.w.requests, sel, self.w.topk, self._res_step, self.w.ctx,
                                      out, st)
        else:
            self.hs.hs_resolve(self.pool, l, self.w.requests, sel, self.w.topk, out, st)

    def _prefetch(self, l, sel, st):
        if self.floor:
            self.hs.hs_probe_launch(self.pool, l, 1, self.w.requests, self.w.topk, st)
        else:
            self.hs.hs_prefetch(self.pool, l, self.w.requests, sel, self.w.topk, st)

    def _shared(self, sel, out, st):
        w = self.w
        if self.floor:
            self.hs.hs_probe_launch(self.pool, 0, w.layers, w.requests, w.topk, st)
        else:
            self.hs.hs_resolve_shared(self.pool, 0, w.layers, w.requests, sel, w.topk, out, st)

    def _layer_work(self, l):
        w, st = self.w, self.stream
        if self.mode.get("attention"):
            r = self.res
            self.hs.hs_mla_decode(self.pool, l, w.requests, r.q, self.out_of(l), w.topk, None, 0, MLA_SCALE,
                                  r.att_out, r.att_lse, st)
        if not self.layer_work:
            return
        self.hs.hs_gather(self.pool, l, w.requests, self.out_of(l), w.topk, self.gather_buf, st)
        with self.torch.cuda.stream(st):
            self.work_dst.copy_(self.work_src)

    def enqueue(self, s):
        """Enqueue decode step s on self.stream."""
        torch, hs, w, st = self.torch, self.hs, self.w, self.stream
        sel = lambda ls: self.sel_of(s, ls)  # noqa: E731
        if self.mode.get("work_only"):
            for l in range(w.layers):
                self._layer_work(l)
            return
        if self.mode.get("full_offload"):
            for l in range(w.layers):
                hs.hs_gather_history(self.pool, l, w.requests, sel(self._lsel(l)), w.topk, self.offload_buf, st)
            return
        if self.mode.get("prefetch"):
            hs.hs_step_begin(self.pool, st)  # a prefetch on a side stream reads the step: its own launch
        elif not self.floor:
            hs.hs_step_begin_fused(self.pool)  # carried by the step's first resolve (no launch of its own)
        self._res_step = None if self.res.res is None else self.res.res[s % w.steps]
        if self.shared_call:
            self._shared(sel(0), self.out_of(0), st)
            for l in range(w.layers):
                self._layer_work(l)
            return
        if not self.mode.get("prefetch"):
            for l in range(w.layers):
                self._resolve(l, sel(self._lsel(l)), self.out_of(l), st)
                self._layer_work(l)
            return
        # exact layer-wise prefetch, D layers ahead on D side streams: when layer l starts on the main stream, layer
        # l + D is resolved on side stream (l + D) % D (at layer 0, layers 1 .. D); layer l's own resolve waits for
        # its prefetch and then only re-stamps and emits its slots. D = 1: prefetch(l+1) beside resolve(l).
        D = self.depth
        done = [None] * w.layers
        for l in range(w.layers):
            if done[l] is not None:
                st.wait_event(done[l])
            ahead = range(1, min(D, w.layers - 1) + 1) if l == 0 else ([l + D] if l + D < w.layers else [])
            if ahead:
                started = torch.cuda.Event()
                started.record(st)
                for j in ahead:
                    side = self.sides[j % D]
                    side.wait_event(started)
                    self._prefetch(j, sel(self._lsel(j)), side)
                    done[j] = torch.cuda.Event()
                    done[j].record(side)
            self._resolve(l, sel(self._lsel(l)), self.out_of(l), st)
            self._layer_work(l)

    def _capture(self, s):
        g = self.torch.cuda.CUDAGraph()
        with self.torch.cuda.graph(g, stream=self.stream):
            self.enqueue(s)
        return g

    def launches_per_step(self) -> int:
        """Kernels of this library launched per step."""
        w = self.w
        per_layer_work = (1 if self.mode.get("attention") else 0) + (1 if self.layer_work else 0)
        if self.mode.get("work_only"):
            return w.layers * per_layer_work
        if self.mode.get("full_offload"):
            return w.layers
        if self.shared_call:
            return 1 + w.layers * per_layer_work
        if self.mode.get("prefetch"):
            return 1 + w.layers * (1 + per_layer_work) + (w.layers - 1)
        return w.layers * (1 + per_layer_work)

    def flush(self):
        with self.torch.cuda.stream(self.stream):
            self.res.flush_buf.fill_(1)

    def reset(self):
        self.hs.hs_pool_reset(self.pool, self.stream)

    def run(self, k_steps: int, timed: bool = True, snapshots: bool = False):
        """Replay k_steps decode steps of the sequence from the cold start (the pool is reset first, and again
        whenever the sequence wraps, outside the timed intervals). Returns a list of (sequence position, step ms,
        counters after the step or None) and the counters (hits, misses, evictions, bytes) summed over layers
        and steps."""
        torch = self.torch
        rows, pending = [], []
        totals = np.zeros(4, dtype=np.int64)
        cview = self.res.buf.view("counters")
        snaps = torch.empty((k_steps,) + tuple(cview.shape), dtype=torch.int64, device="cuda") if snapshots else None

        def collect():
            self.stream.synchronize()
            for i, p, e0, e1 in pending:
                c = snaps[i].sum(dim=0).cpu().numpy() if snapshots else None
                rows.append((p, e0.elapsed_time(e1) if timed else 0.0, c))
            pending.clear()

        def lead():
            if timed:
                with torch.cuda.stream(self.stream):
                    torch.cuda._sleep(LEAD_CYCLES)

        self.reset()
        lead()
        pos = 0
        for i in range(k_steps):
            if pos == len(self.graphs) or pos == self.w.steps:
                collect()
                totals += self.res.counters()
                pos = 0
                self.reset()
                lead()
            self.flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(self.stream):
                if timed:
                    e0.record(self.stream)
                self.graphs[pos].replay()
                if timed:
                    e1.record(self.stream)
                if snapshots:
                    snaps[i].copy_(cview)
            pending.append((i, pos, e0, e1))
            pos += 1
        collect()
        totals += self.res.counters()
        return rows, totals

    def close(self):
        self.graphs = []


def step_stats(rows, w: wl.Workload, link_gbs: float) -> dict:
    """Cold, churn and steady step times; the link fraction of miss-heavy steps (cold start, churn steps) from
    their own miss bytes."""
    cold = [r[1] for r in rows if r[0] == 0]
    churn = [r[1] for r in rows if r[0] in w.churn]
    steady = [r[1] for r in rows if r[0] != 0 and r[0] not in w.churn]
    heavy = []
    prev = None
    for p, ms, c in rows:
        if c is not None:
            step_bytes = int(c[3]) - (int(prev[3]) if (prev is not None and p != 0) else 0)
            if (p == 0 or p in w.churn) and ms > 0:
                heavy.append({"step": p, "miss_bytes": step_bytes, "ms": ms,
                              "link_gbs": step_bytes / (ms / 1e3) / 1e9,
                              "frac": step_bytes / (link_gbs * 1e9) / (ms / 1e3)})
        prev = c
    out = {
        "cold_step_ms": statistics.mean(cold) if cold else None,
        "churn_step_ms": statistics.mean(churn) if churn else None,
        "steady_step_ms": statistics.mean(steady) if steady else None,
        "steady_step_ms_p10_p50_p90": ([float(np.percentile(steady, q)) for q in (10, 50, 90)] if steady else None),
    }
    if heavy:
        out["miss_heavy_steps"] = {"n": len(heavy),
                                   "link_frac_mean": statistics.mean(h["frac"] for h in heavy),
                                   "link_gbs_mean": statistics.mean(h["link_gbs"] for h in heavy),
                                   "first": heavy[0]}
    return out


def measure_link(hs, torch, host_ptr: int, nbytes: int, chunk: int = 1 << 30) -> tuple:
    """Best zero-copy and memcpy host-to-device GB/s over the host buffer, read in chunks of at most 1 GiB
    (so every page of the buffer is read at least once)."""
    dev = torch.empty(min(nbytes, chunk), dtype=torch.uint8, device="cuda")
    best_zc = best_cp = 0.0
    for off in range(0, nbytes, chunk):
        n = min(chunk, nbytes - off) // 16 * 16
        if n < 16:
            break
        zc, cp = hs.hs_probe_link(host_ptr + off, dev, n, 3 if off else 5)
        best_zc, best_cp = max(best_zc, zc), max(best_cp, cp)
    del dev
    return best_zc, best_cp


def e2e_passes(res: Resources, mode: dict, k_steps: int, ref_graphs: StepGraphs) -> dict:
    """The same steps through the public API on the host clock (time.perf_counter), host buffers in and out.

    zero-copy: one graph whose kernels read the selection from, and write out_slots to, mapped page-locked host
    memory. Per step the timed region covers the host writing that step's selection into the mapped buffer, the
    graph launch, the stream synchronisation and the host reading every layer's out_slots back.
    with_copies: the same with a device selection buffer and device out_slots: the host writes the selection into
    pinned memory, cudaMemcpyAsync copies it in, the graph runs, cudaMemcpyAsync copies out_slots out, the stream
    is synchronised and the host reads them.
    The L2 flush and its synchronisation happen before each timed region. out_slots are compared with a replay of
    the same sequence through the device-memory graphs."""
    torch, hs, w = res.torch, res.hs, res.w
    nsel = w.selection_layers * w.requests * w.topk
    # one shared call writes the slot list of its first layer only (every layer's is the same)
    out_layers = 1 if (mode.get("shared_call") and w.shared_across_layers) else w.layers
    nout = out_layers * w.requests * w.topk
    writes_slots = not (mode.get("full_offload") or mode.get("work_only"))
    # reference out_slots of every step of the sequence, from the device-memory graphs
    ref = []
    ref_graphs.reset()
    for pos in range(w.steps):
        with torch.cuda.stream(ref_graphs.stream):
            ref_graphs.graphs[pos].replay()
        ref_graphs.stream.synchronize()
        ref.append(res.out[:out_layers].cpu().numpy().copy())

    host_sel = hs.HostBuffer(nsel * 4)
    host_out = hs.HostBuffer(nout * 4)
    sel_np = np.frombuffer(host_sel.numpy(), dtype=np.int32).reshape(w.selection_layers, w.requests, w.topk)
    out_np = np.frombuffer(host_out.numpy(), dtype=np.int32).reshape(out_layers, w.requests, w.topk)
    result = np.empty((out_layers, w.requests, w.topk), dtype=np.int32)
    per_ls = w.requests * w.topk * 4
    per_l = w.requests * w.topk * 4
    zc = StepGraphs(res, res.pool, mode, sel_of=lambda s, ls: host_sel.ptr + ls * per_ls,
                    out_of=lambda l: host_out.ptr + l * per_l, single=True)
    # device-buffer graph for the copy variant
    dsel = torch.empty((w.selection_layers, w.requests, w.topk), dtype=torch.int32, device="cuda")
    cp = StepGraphs(res, res.pool, mode, sel_of=lambda s, ls: dsel[ls], single=True)
    pin_sel = torch.empty((w.selection_layers, w.requests, w.topk), dtype=torch.int32).pin_memory()
    pin_out = torch.empty((out_layers, w.requests, w.topk), dtype=torch.int32).pin_memory()
    pin_sel_np, pin_out_np = pin_sel.numpy(), pin_out.numpy()

    def loop(g: StepGraphs, body):
        times, match = [], (True if writes_slots else None)
        g.reset()
        pos = 0
        for _ in range(k_steps):
            if pos == w.steps:
                pos = 0
                g.reset()
            g.flush()
            g.stream.synchronize()
            t0 = time.perf_counter()
            body(g, pos)
            times.append(time.perf_counter() - t0)
            if writes_slots:
                match = match and bool(np.array_equal(result, ref[pos]))
            pos += 1
        return sum(times), match

    def zc_body(g, pos):
        sel_np[...] = res.sel_host[pos]
        with torch.cuda.stream(g.stream):
            g.graphs[0].replay()
        g.stream.synchronize()
        np.copyto(result, out_np)

    def cp_body(g, pos):
        pin_sel_np[...] = res.sel_host[pos]
        with torch.cuda.stream(g.stream):
            dsel.copy_(pin_sel, non_blocking=True)
            g.graphs[0].replay()
            pin_out.copy_(res.out[:out_layers], non_blocking=True)
        g.stream.synchronize()
        np.copyto(result, pin_out_np)

    zc_s, zc_match = loop(zc, zc_body)
    cp_s, cp_match = loop(cp, cp_body)
    zc.close()
    cp.close()
    torch.cuda.synchronize()
    host_sel.close()
    host_out.close()
    sel_per_step = w.layers * w.requests
    return {
        "value": k_steps * sel_per_step / zc_s, "unit": UNIT, "h2d_bytes_per_step": nsel * 4,
        "d2h_bytes_per_step": nout * 4 if writes_slots else 0, "ms_per_step": zc_s * 1e3 / k_steps,
        "clock": "host (time.perf_counter) around each step",
        "path": "per step: host writes the selection into mapped page-locked memory, one graph launch whose kernels "
                "read it and write out_slots back over the host link, stream sync, host reads every layer's "
                "out_slots",
        "out_slots_match_device_path": zc_match,
        "with_copies": {"value": k_steps * sel_per_step / cp_s, "unit": UNIT, "h2d_bytes_per_step": nsel * 4,
                        "d2h_bytes_per_step": nout * 4 if writes_slots else 0, "ms_per_step": cp_s * 1e3 / k_steps,
                        "out_slots_match_device_path": cp_match,
                        "path": "per step: host writes the selection into pinned memory, cudaMemcpyAsync in, graph "
                                "launch, cudaMemcpyAsync of out_slots out, stream sync, host reads them"},
    }


def _oracle_requests(w: wl.Workload, lo: int, hi: int, sel: np.ndarray, host: np.ndarray, res, budget_s: float,
                     t0: float, ls: int = 0) -> tuple:
    """Steps of one layer (selection layer ls) for requests lo..hi-1 from the cold start, the sequence replayed from a
    fresh cache each time it ends (as the GPU passes do), until the budget; (selections, steps)."""
    import oracle

    n = steps = 0
    while time.perf_counter() - t0 < budget_s:
        pool = oracle.OraclePool(w.ctx, w.slots, w.row_bytes, 1, hi - lo, track_rows=True)
        for s in range(w.steps):
            if time.perf_counter() - t0 >= budget_s:
                break
            pool.step_begin()
            pool.resolve(0, sel[s, ls, lo:hi], host[lo:hi], resident=None if res is None else res[s, lo:hi])
            n += hi - lo
            steps += 1
    return n, steps


def cpu_baseline(w: wl.Workload, budget_s: float = 12.0, tiered_frac: float | None = None, threads: int = 1,
                 host: np.ndarray | None = None) -> dict:
    """The CPU oracle on a bounded sample of the same workload: request-layers of layer 0, hot rows tracked in
    host memory, steps in order from the cold start until the time budget. With threads > 1 the request-layers are
    split over that many threads (the oracle's C routine runs without the interpreter lock), each resolving its
    own, which are independent: the requests of layer 0, and with more threads than requests whole layers of
    requests (threads // requests layers, one request-layer per thread; their rows are layer 0's, which costs the
    same). `host` is layer 0's host rows [requests][ctx][row_bytes] (generated when not given)."""
    reqs = w.requests
    nl = max(1, min(w.layers, threads // reqs)) if threads > reqs else 1
    sel = wl.gen_selections(w, layers=(0, 1 if w.shared_across_layers else nl), requests=(0, reqs))
    if host is None:
        host = np.stack([wl.rows(w, 0, b) for b in range(reqs)])
    res = None if tiered_frac is None else wl.gen_resident(w.ctx, reqs, w.steps, w.seed, frac=tiered_frac)
    if nl > 1:  # one request-layer per thread
        units = [(0 if w.shared_across_layers else l, b, b + 1) for l in range(nl) for b in range(reqs)]
    else:
        th = max(1, min(threads, reqs))
        units = [(0, reqs * i // th, reqs * (i + 1) // th) for i in range(th)]
    threads = len(units)
    results = [None] * threads
    t0 = time.perf_counter()

    def work(i):
        ls, lo, hi = units[i]
        results[i] = _oracle_requests(w, lo, hi, sel, host, res, budget_s, t0, ls)

    ths = [threading.Thread(target=work, args=(i,)) for i in range(threads)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    dt = time.perf_counter() - t0
    n = sum(r[0] for r in results)
    steps = min(r[1] for r in results)
    how = ("single-threaded" if threads == 1 else
           f"{threads} threads, one request-layer each" if nl > 1 else f"{threads} threads over the requests")
    which = f"layers 0..{nl - 1}" if nl > 1 else "layer 0"
    return {"value": n / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{which} of {w.name}, {reqs} requests, at least {steps} decode steps (the {w.steps}-step "
                      f"sequence replayed from the cold start; {n} selections, hot rows tracked" +
                      (", resident maps" if res is not None else "") + f", {dt:.1f} s {how})"}


def max_over_ranks(ms: float, dist=None) -> float:
    """The slowest rank's time (every rank processes the same number of units)."""
    if dist is None:
        return ms
    import torch

    t = torch.tensor([ms], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(world: int, units_per_rank: int, max_ms: float) -> float:
    """Whole-job throughput: all ranks' units over the slowest rank's time (weak scaling)."""
    return world * units_per_rank / (max_ms / 1e3)


class Env:
    """Per-process measurement context: ranks, peaks, link, clock sampler."""

    def __init__(self, args, dist, world: int, rank: int, local: int):
        self.args, self.dist, self.world, self.rank, self.local = args, dist, world, rank, local
        peaks = {}
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                peaks = json.load(f)
        except OSError:
            pass
        self.peaks = peaks
        self.hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
        self.hbm_src = "measured" if "hbm_gbs" in peaks else "fallback"
        self.clk = ClockSampler(local)

    def barrier(self):
        import torch

        if self.dist:
            self.dist.barrier()
        torch.cuda.synchronize()


def roofline_of(w, mode, env: Env, n_launch_layers: int, n_kernels: int, tot, kern_ms: float, link, res, rows,
                noio: bool = False) -> dict:
    """Roofline of the resolve kernel over a pass: link term (miss bytes over the measured link) and HBM term
    (metadata + hot-buffer bytes; in no-IO mode the rows are read from HBM too), over the measured time."""
    hits, misses, evictions, miss_bytes = (int(x) for x in tot)
    # the committed captures are of the plain per-layer resolve; no other mode's launches are what they measured
    plain = not any(mode.get(k) for k in ("prefetch", "shared_call", "full_offload", "work_only", "tiered_frac",
                                          "attention", "layer_work_mb"))
    if mode.get("full_offload"):  # every selected row crossed the link
        hits, misses = 0, n_launch_layers * w.requests * w.topk
        miss_bytes = misses * w.row_bytes
    link_peak = max(link)
    meta = n_launch_layers * meta_bytes_per_launch(w, w.requests) + 4 * hits + 16 * misses
    if res.res is not None:  # the resident-map lookup of every selected token
        meta += 4 * n_launch_layers * w.requests * w.topk
    kern_s = kern_ms / 1e3
    if noio:
        hbm = meta + 2 * miss_bytes
        return {"bound": "hbm", "achieved": hbm / kern_s / 1e9, "peak": env.hbm_peak, "unit": "GB/s",
                "frac": hbm / (env.hbm_peak * 1e9) / kern_s,
                "frac_of_nominal": hbm / (HBM_NOMINAL_GBS * 1e9) / kern_s, "hbm_bytes_per_launch": hbm / n_kernels,
                "traffic": captured_traffic(w, sum(w.layers for r in rows if r[0] == 0),
                                            sum(w.layers for r in rows if r[0] != 0), noio=True) if plain else None,
                "peak_source": f"HBM {env.hbm_peak:.1f} GB/s {env.hbm_src} (MEASURED_PEAKS.json copy); "
                               f"frac_of_nominal: against {HBM_NOMINAL_GBS:.0f} GB/s nominal"}
    hbm = meta + miss_bytes
    t_link = miss_bytes / (link_peak * 1e9)
    t_hbm = hbm / (env.hbm_peak * 1e9)
    bound = "host_link" if t_link >= t_hbm else "hbm"
    return {
        "bound": bound,
        "achieved": (miss_bytes / kern_s / 1e9) if bound == "host_link" else (hbm / kern_s / 1e9),
        "peak": link_peak if bound == "host_link" else env.hbm_peak,
        "unit": "GB/s",
        "frac": max(t_link, t_hbm) / kern_s,
        "hbm_frac": t_hbm / kern_s,
        "hbm_frac_of_nominal": hbm / (HBM_NOMINAL_GBS * 1e9) / kern_s,
        "traffic": captured_traffic(w, sum(w.layers for r in rows if r[0] == 0),
                                    sum(w.layers for r in rows if r[0] != 0)) if plain else None,
        "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum per launch from the committed ncu capture "
                          "(profiles/) of this workload's steady launches, null unless taken on these kernel sources",
        "kernel": "hs_gather_kernel" if mode.get("full_offload") else "hs_resolve_kernel",
        "kernel_ms_per_launch": kern_ms / n_kernels,
        "launches": n_kernels,
        "timing": ("CUDA events around each step's graph in the timed region: " +
                   ("the step's hs_gather_history launches (every selected row of every layer from host memory)"
                    if mode.get("full_offload") else
                    "the step increment plus the step's resolves, an upper bound on the resolve launches" +
                    (" (layer-wise prefetch on side streams included)" if mode.get("prefetch") else ""))),
        "algorithmic_bytes_per_launch": {"link": miss_bytes / n_kernels, "hbm": hbm / n_kernels},
        "peak_source": f"host link measured in this run (zero-copy {link[0]:.1f}, memcpy {link[1]:.1f} GB/s); "
                       f"HBM {env.hbm_peak:.1f} GB/s {env.hbm_src} (hbm_frac_of_nominal: against "
                       f"{HBM_NOMINAL_GBS:.0f} GB/s nominal)",
    }


def measure(env: Env, res: Resources, mode: dict, K: int, W: int, legs: set, cpu_budget: float,
            cpu_threads: int, link: tuple, headline: bool = False) -> dict:
    """All legs of one (workload, mode): the timed pass, its launch floor, e2e, no-IO (with its floor) and the CPU
    oracle. Returns the per-workload dict."""
    torch, w = res.torch, res.w
    nvtx = torch.cuda.nvtx
    g = StepGraphs(res, res.pool, mode)
    nvtx.range_push(f"warm-up: {W} steps of {w.name} ({mode_name(mode)})")
    g.run(W, timed=False)
    nvtx.range_pop()
    env.barrier()
    env.clk.start()
    nvtx.range_push(f"timed: {K} steps of {w.name} ({mode_name(mode)})")
    rows, tot = g.run(K, snapshots=True)
    nvtx.range_pop()
    env.barrier()
    env.clk.stop()
    step_ms = [r[1] for r in rows]
    kern_ms = sum(step_ms)
    total_ms = max_over_ranks(kern_ms, env.dist)
    sel_per_step = w.layers * w.requests
    value = aggregate_rate(env.world, K * sel_per_step, total_ms)
    shared_call = g.shared_call
    n_kernels = K if shared_call else K * w.layers
    out = {
        "workload": describe(w), "mode": mode_name(mode), "value": value, "unit": UNIT, "steps": K,
        "ms_per_step": total_ms / K, "selected_entries_per_s": value * w.topk,
        "miss_gbs": int(tot[3]) / (total_ms / 1e3) / 1e9 * env.world,
        "gpu_launches": K * g.launches_per_step(),
        "host_pool": ("one pool per layer" if res.host_layers == w.layers else
                      f"layers share one host pool, layer l reading token t from row t + l * "
                      f"{res.buf.layer_shift_rows} (host_layer_stride = that many rows), so no two layers read the "
                      f"same row for the same token; every miss crosses the link"),
    }
    out.update(step_stats(rows, w, max(link)))
    out["step_ms"] = [round(r[1], 4) for r in rows]
    out["roofline"] = roofline_of(w, mode, env, K * w.layers, n_kernels, tot, kern_ms, link, res, rows)
    # run-to-run spread: two more passes of the same K steps (after the timed region)
    if "spread" in legs:
        vals = [value]
        for _ in range(2):
            r2, _ = g.run(K)
            vals.append(aggregate_rate(env.world, K * sel_per_step, max_over_ranks(sum(r[1] for r in r2), env.dist)))
        out["repeats"] = {"n": len(vals), "values": vals, "min": min(vals), "median": statistics.median(vals),
                          "max": max(vals)}
    if "floor" in legs and not (mode.get("work_only") or mode.get("full_offload")):
        fg = StepGraphs(res, res.pool, mode, floor=True)
        fg.run(3, timed=False)
        frows, _ = fg.run(K)
        fg.close()
        fms = sum(r[1] for r in frows) / K
        out["floor"] = {"ms_per_step": fms, "frac_of_step": fms / (total_ms / K),
                        "what": "the same step graph with every resolve replaced by an empty kernel launched with "
                                "the resolve's configuration (hs_probe_launch): grid, cluster, shared memory, "
                                "programmatic dependent launch; hs_step_begin kept where the step has it (prefetch "
                                "pipelines), elsewhere the step increment rides on the first resolve"}
    if "e2e" in legs:
        nvtx.range_push("end to end")
        out["e2e"] = e2e_passes(res, mode, K, g)
        nvtx.range_pop()
    g.close()
    if "noio" in legs and res.noio_pool:
        ng = StepGraphs(res, res.noio_pool, mode)
        nvtx.range_push(f"no-IO: {w.name}")
        ng.run(W, timed=False)
        nrows, ntot = ng.run(K)
        nvtx.range_pop()
        ng.close()
        nms = max_over_ranks(sum(r[1] for r in nrows), env.dist)
        nk_ms = sum(r[1] for r in nrows)
        noio = {"value": aggregate_rate(env.world, K * sel_per_step, nms), "unit": UNIT, "ms_per_step": nms / K,
                "kernel_ms_per_launch": nk_ms / n_kernels,
                "roofline": roofline_of(w, mode, env, K * w.layers, n_kernels, ntot, nk_ms, link, res, nrows,
                                        noio=True)}
        if "floor" in legs and not (mode.get("work_only") or mode.get("full_offload")):
            fg = StepGraphs(res, res.noio_pool, mode, floor=True)
            fg.run(3, timed=False)
            frows, _ = fg.run(K)
            fg.close()
            fms = sum(r[1] for r in frows) / K
            noio["floor"] = {"ms_per_step": fms, "frac_of_step": fms / (nms / K)}
            # the HBM roofline of what is left once launching alone is paid
            rf = noio["roofline"]
            t_hbm = rf["frac"] * (nk_ms / K)
            noio["roofline"]["frac_above_floor"] = t_hbm / max(1e-9, nk_ms / K - fms)
        out["noio"] = noio
    if "cpu" in legs and env.rank == 0 and not (mode.get("full_offload") or mode.get("work_only")):
        host = res.host_rows_layer0()
        tiered = mode.get("tiered_frac")
        out["cpu_baseline"] = cpu_baseline(w, budget_s=cpu_budget, tiered_frac=tiered, host=host)
        if headline and cpu_threads > 1:
            out["cpu_baseline_threads"] = cpu_baseline(w, budget_s=cpu_budget, tiered_frac=tiered,
                                                       threads=cpu_threads, host=host)
    return out


def prefetch_hiding(env: Env, res: Resources, K: int, W: int, work_mb: float) -> dict:
    """Exposed resolve time with a per-layer work stand-in (hs_gather of the layer's rows plus a work_mb MB device
    copy after each layer, on the main stream): work alone, per-layer resolves + work, with layer-wise prefetch,
    and with one shared call. Exposed = (resolve + work) - work; hidden = the share of it prefetch removes."""
    out = {"layer_work_mb": work_mb}
    for key, mode in (("work_only", {"work_only": True, "layer_work_mb": work_mb}),
                      ("resolve_work", {"layer_work_mb": work_mb}),
                      ("prefetch_work", {"prefetch": True, "layer_work_mb": work_mb}),
                      ("prefetch2_work", {"prefetch": True, "prefetch_depth": 2, "layer_work_mb": work_mb}),
                      ("shared_call_work", {"shared_call": True, "layer_work_mb": work_mb})):
        g = StepGraphs(res, res.pool, mode)
        g.run(W, timed=False)
        rows, _ = g.run(K)
        g.close()
        steady = [r[1] for r in rows if r[0] != 0]
        out[key + "_steady_ms"] = statistics.mean(steady) if steady else None
        out[key + "_ms_per_step"] = sum(r[1] for r in rows) / K
    exposed = out["resolve_work_steady_ms"] - out["work_only_steady_ms"]
    exposed_pf = out["prefetch_work_steady_ms"] - out["work_only_steady_ms"]
    exposed_sc = out["shared_call_work_steady_ms"] - out["work_only_steady_ms"]
    out["exposed_resolve_ms"] = exposed
    out["exposed_with_prefetch_ms"] = exposed_pf
    out["exposed_with_shared_call_ms"] = exposed_sc
    out["hidden_by_prefetch_frac"] = 1.0 - exposed_pf / exposed if exposed > 0 else None
    exposed_pf2 = out["prefetch2_work_steady_ms"] - out["work_only_steady_ms"]
    out["exposed_with_prefetch2_ms"] = exposed_pf2
    out["hidden_by_prefetch2_frac"] = 1.0 - exposed_pf2 / exposed if exposed > 0 else None
    out["hidden_by_shared_call_frac"] = 1.0 - exposed_sc / exposed if exposed > 0 else None
    return out


def attention_leg(env: Env, K: int, W: int) -> dict:
    """The attention consumer on the mla workload: resolve the sequence to its steady state, then one graph of a
    single hs_mla_decode launch on the last step's slot lists, replayed K times with L2 flushed before each and
    CUDA events on its stream. Roofline: HBM (the rows and queries it must read), with the tensor rate beside."""
    import hierarchical_sparse_attention_hs_gb300 as hs
    import torch

    w = wl.WORKLOADS["mla"]
    res = Resources(w, noio=False, attention=True)
    try:
        g = StepGraphs(res, res.pool, {})
        g.run(w.steps, timed=False)
        g.close()
        st = torch.cuda.Stream()
        ag = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ag, stream=st):
            hs.hs_mla_decode(res.pool, 0, w.requests, res.q, res.out[0], w.topk, None, 0, MLA_SCALE, res.att_out,
                             res.att_lse, st)
        torch.cuda.synchronize()
        times = []
        for i in range(W + K):
            with torch.cuda.stream(st):
                res.flush_buf.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(st):
                e0.record(st)
                ag.replay()
                e1.record(st)
            if i >= W:
                times.append((e0, e1))
        st.synchronize()
        ms = [a.elapsed_time(b) for a, b in times]
        slots = res.out[0].cpu().numpy()
        valid = int(((slots >= 0) & (slots < w.slots)).sum())
        flops = 2.0 * hs.MLA_HEADS * valid * (hs.MLA_D_QK + hs.MLA_D_V)
        nbytes = valid * w.row_bytes + res.q.numel() * 2 + res.att_out.numel() * 4 + res.att_lse.numel() * 4 + \
            w.requests * w.topk * 4
        mean_ms = statistics.mean(ms)
        bf16_peak = float(env.peaks.get("bf16_tflops", 1900.0))
        tflops = flops / (mean_ms / 1e3) / 1e12
        gbs = nbytes / (mean_ms / 1e3) / 1e9
        return {
            "kernel": "hs_mla_decode_kernel", "workload": describe(w), "bound": "hbm", "achieved": gbs,
            "peak": env.hbm_peak, "unit": "GB/s", "frac": gbs / env.hbm_peak, "ms_per_launch": mean_ms,
            "ms_per_launch_p50": float(np.percentile(ms, 50)), "launches": len(ms),
            "algorithmic_bytes_per_launch": nbytes,
            "bytes_definition": "valid rows x 1152 B + queries (bf16) + out (fp32) + lse + the slot list",
            "tensor": {"achieved": tflops, "peak": bf16_peak, "unit": "TFLOP/s", "frac": tflops / bf16_peak,
                       "flops_per_launch": flops,
                       "flops_definition": "2 * 128 heads * valid rows * (576 + 512): the score and value products"},
            "valid_rows_per_launch": valid,
            "traffic": captured_attention_traffic(w),
            "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum per launch from the committed ncu "
                              "capture (profiles/), null unless taken on these kernel sources",
            "timing": "CUDA events around one graph launch each, L2 flushed before each, on the launch stream",
        }
    finally:
        res.close()


def run_reference(args) -> int:
    """Reference arm: the CPU oracle as it stands on the headline workload (or --workload), one layer per step
    (the layers of the shared workload resolve identically), timed on the host clock."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle

    name = HEADLINE[0] if args.workload == "all" else args.workload
    w = wl.WORKLOADS[name]
    reqs = w.requests
    sel = wl.gen_selections(w, layers=(0, 1), requests=(0, reqs))
    host = np.empty((reqs, w.ctx, w.row_bytes), dtype=np.uint8)
    for b in range(reqs):
        wl.fill_rows_at(w, host[b].ctypes.data, 0, b, 0, w.ctx)
    layers_per_step = max(1, min(w.layers, args.ref_layers))

    def one_step(pool, s):
        pool.step_begin()
        for l in range(layers_per_step):
            pool.resolve(l, sel[s % w.steps, 0], host)

    pool = oracle.OraclePool(w.ctx, w.slots, w.row_bytes, layers_per_step, reqs, track_rows=True)
    for s in range(args.warmup):
        one_step(pool, s)
    pool = oracle.OraclePool(w.ctx, w.slots, w.row_bytes, layers_per_step, reqs, track_rows=True)
    t0 = time.perf_counter()
    for s in range(args.steps):
        if s and s % w.steps == 0:
            pool = oracle.OraclePool(w.ctx, w.slots, w.row_bytes, layers_per_step, reqs, track_rows=True)
        one_step(pool, s)
    dt = time.perf_counter() - t0
    n = args.steps * reqs * layers_per_step
    value = n / dt
    mode = dict(HEADLINE[1]) if args.workload == "all" else {}
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": describe(w), "mode": mode_name(mode),
                   "sample": f"{layers_per_step} of {w.layers} layer(s) per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} decode steps of {layers_per_step} layer(s) x {reqs} requests of "
                                   f"{w.name}, hot rows tracked, single-threaded"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _setup_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo")
    return world, rank, local, dist


def gpu_measure(args, env: Env) -> dict:
    """Every leg of the run on this rank's GPU; returns the line (rank 0 prints it)."""
    import torch

    import hierarchical_sparse_attention_hs_gb300 as hs
    from hierarchical_sparse_attention_hs_gb300 import build as hs_build

    torch.cuda.set_device(env.local)
    if env.rank == 0:
        hs_build.build()
    if env.dist:
        env.dist.barrier()
    hs.load()
    K, W = args.steps, args.warmup
    legs = set(args.legs.split(","))
    if args.workload == "all":
        head_name, head_mode = HEADLINE
        others = [] if args.headline_only else DEFAULT_SET
    else:
        head_name = args.workload if not args.own_pool_layers else f"shared_own{args.own_pool_layers}"
        head_mode = {"prefetch": args.prefetch, "prefetch_depth": args.prefetch_depth if args.prefetch else 1,
                     "shared_call": args.shared_call,
                     "layer_work_mb": args.layer_work_mb, "work_only": args.work_only,
                     "full_offload": args.full_offload, "tiered_frac": args.tiered_frac, "attention": args.attention}
        head_mode = {k: v for k, v in head_mode.items() if v not in (None, False, 0.0) and
                     not (k == "prefetch_depth" and v == 1)}
        others = []
    alias = args.alias_host  # otherwise layers share a host pool only where their own pools do not fit
    cache = {}

    def resources(name, mode):
        key = (name, mode.get("tiered_frac"), bool(mode.get("attention")))
        if key not in cache:
            for k in list(cache):
                cache.pop(k).close()
            torch.cuda.empty_cache()
            w = workload_of(name)
            # (the own-pool comparison needs no HBM copy of its 88 GB pool: its no-IO mode is the headline's)
            r = Resources(w, alias_host=alias, noio="noio" in legs and not name.startswith("shared_own"),
                          attention=bool(mode.get("attention")),
                          tiered_frac=mode.get("tiered_frac"))
            # the GPU reads the whole host pool once (as a long-running server has long since done), so that
            # first-touch address translation of host pages is not charged to the timed steps; it also measures
            # the link
            r.link = measure_link(hs, torch, r.buf.host.ptr, r.buf.host.nbytes // 16 * 16)
            torch.cuda.empty_cache()  # the probe's staging buffer goes back to the device
            cache[key] = r
        return cache[key]

    t_start = time.perf_counter()
    res = resources(head_name, head_mode)
    head = measure(env, res, head_mode, K, W, legs, args.cpu_budget, args.cpu_threads, res.link, headline=True)
    head["pool_bytes"] = {"host": res.buf.host.nbytes, "hot_buffer": res.buf.hot.numel(),
                          "metadata": res.buf.meta.numel()}
    if args.workload == "all" and "hiding" in legs and res.w.shared_across_layers:
        head["prefetch_hiding"] = prefetch_hiding(env, res, K, W, HIDING_WORK_MB)
    per = {}
    for name, mode in others:
        key = name if not mode else f"{name} ({mode_name(mode)})"
        try:
            r = resources(name, mode)
            per[key] = measure(env, r, mode, K, W, legs, args.cpu_budget_other, 1, r.link)
        except Exception as e:  # one workload failing must not lose the others
            per[key] = {"error": f"{type(e).__name__}: {e}"}
    attention = None
    if args.workload == "all" and "attention" in legs:
        for k in list(cache):
            cache.pop(k).close()
        torch.cuda.empty_cache()
        try:
            attention = attention_leg(env, K, W)
        except Exception as e:
            attention = {"error": f"{type(e).__name__}: {e}"}
    for k in list(cache):
        cache.pop(k).close()
    w = workload_of(head_name)
    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": env.world, "steps": K, "warmup": W,
        "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int32", "data": "synthetic",
        "config": {"workload": describe(w), "mode": mode_name(head_mode),
                   "parallelism": f"replicas x{env.world} (independent requests per GPU)",
                   "l2": "flushed between steps (256 MiB write)", "host_pool": head["host_pool"],
                   "graphs": "one CUDA graph per decode step"},
        "selected_entries_per_s": head["selected_entries_per_s"],
        "gpu_launches": head["gpu_launches"],
        "roofline": head["roofline"],
        "noio": head.get("noio"),
        "e2e": head.get("e2e"),
        "clocks": env.clk.summary(),
        "headline": head,
        "per_workload": per or None,
        "attention": attention,
        "run_s": time.perf_counter() - t_start,
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    return line


def run_gpu(args, measure_fn=None) -> int:
    """One rank: set up the process group (gloo, for the barrier and the max over ranks), measure, and print the
    line on rank 0. `measure_fn(args, env) -> dict` is the GPU work (replaced by a stub in CPU tests)."""
    world, rank, local, dist = _setup_dist()
    env = Env(args, dist, world, rank, local)
    line = (measure_fn or gpu_measure)(args, env)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank: int, world: int, port: int, argv: list, measure_fn) -> None:
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    args = parse_args(argv)
    sys.exit(run_gpu(args, measure_fn))


def spawn_replicas(n: int, argv: list, measure_fn=None) -> int:
    """Start n replica processes (one per GPU, RANK = LOCAL_RANK = GPU index) when no launcher set WORLD_SIZE;
    returns the first non-zero exit code, else 0."""
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_replica, args=(r, n, port, argv, measure_fn)) for r in range(n)]
    for p in procs:
        p.start()
    rc = 0
    for p in procs:
        p.join()
        if p.exitcode and not rc:
            rc = p.exitcode
    return rc


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["hs", "reference"], default="hs")
    ap.add_argument("--workload", choices=["all"] + list(wl.WORKLOADS), default="all",
                    help="all (default): every workload, headlined on the shared workload with layer-wise prefetch")
    ap.add_argument("--headline-only", action="store_true", help="with --workload all: only the headline")
    ap.add_argument("--legs", default="io,floor,e2e,noio,cpu,spread,hiding,attention",
                    help="comma-separated legs: floor, e2e, noio, cpu, spread, hiding, attention")
    ap.add_argument("--alias-host", action="store_true", help="all layers read one host pool")
    ap.add_argument("--own-pool-layers", type=int, default=0,
                    help="with --workload shared: that many of its layers, each with a host pool of its own")
    ap.add_argument("--prefetch", action="store_true", help="layer-wise prefetch on a second stream")
    ap.add_argument("--prefetch-depth", type=int, default=1,
                    help="with --prefetch: prefetch this many layers ahead, on as many side streams")
    ap.add_argument("--layer-work-mb", type=float, default=0.0,
                    help="per-layer work stand-in after each resolve: hs_gather + a copy of this many MB")
    ap.add_argument("--work-only", action="store_true",
                    help="replay only the per-layer work stand-in (no resolve): the reference for exposed time")
    ap.add_argument("--shared-call", action="store_true",
                    help="workloads whose layers share one selection: one hs_resolve_shared call per step")
    ap.add_argument("--full-offload", action="store_true",
                    help="comparator without a GPU cache: fetch every selected row from host memory every step")
    ap.add_argument("--cpu-budget", type=float, default=8.0, help="seconds of CPU-oracle time for the headline")
    ap.add_argument("--cpu-budget-other", type=float, default=3.0,
                    help="seconds of CPU-oracle time for each other workload")
    ap.add_argument("--cpu-threads", type=int, default=os.cpu_count() or 1,
                    help="threads of the second, multi-threaded CPU-oracle line of the headline (1 = skip it)")
    ap.add_argument("--tiered-frac", type=float, default=None,
                    help="three-tier resolution: fraction of pages still held in the HBM KV pool (plus the newest "
                         "256 tokens), one resident map per request and step")
    ap.add_argument("--attention", action="store_true",
                    help="sparse MLA decode (hs_mla_decode) after each layer's resolve; needs 1152-byte rows (the "
                         "mla workload)")
    ap.add_argument("--ref-layers", type=int, default=1, help="reference arm: layers resolved per step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if args.attention and (args.tiered_frac is not None or args.full_offload or args.work_only):
        ap.error("--attention reads the slot lists of plain resolves; it combines with none of --tiered-frac, "
                 "--full-offload, --work-only")
    if args.own_pool_layers and (args.workload != "shared" or args.own_pool_layers < 2):
        ap.error("--own-pool-layers takes --workload shared and at least 2 layers")
    if args.tiered_frac is not None and (args.prefetch or args.shared_call or args.full_offload):
        ap.error("--tiered-frac resolves each layer with its own call; it combines with none of --prefetch, "
                 "--shared-call, --full-offload")
    world_env = os.environ.get("WORLD_SIZE")
    if world_env is not None and int(world_env) != args.gpus:
        ap.error(f"--gpus {args.gpus} does not match WORLD_SIZE={world_env} set by the launcher")
    return args


def main(argv=None) -> int:
    argv = sys.argv[1:] if argv is None else argv
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return spawn_replicas(args.gpus, argv)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
