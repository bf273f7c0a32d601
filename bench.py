#!/usr/bin/env python3
"""Benchmark of the hierarchical KV cache resolver on GB300: top-k selections resolved per second.

A step is one decode step of a synthetic workload: hs_step_begin plus one hs_resolve per layer for every
request (captured once per step of the workload's selection sequence into a CUDA graph and replayed). The
sequence starts from an empty cache, so the first step is the all-miss cold start; when K exceeds the sequence
the pool is reset (outside the timed intervals) and the sequence restarts. One selection = one request-layer's
top-k list for one step.

Timing: W warm-up steps, then K steps, each bracketed by CUDA events on the launching stream with a 256 MiB L2
flush between steps (outside the events), barrier + synchronize around the whole region, max over ranks. Clocks
are sampled with nvidia-smi during the timed region.

Roofline (the slower of two terms): miss-row bytes over the measured host link, and metadata + hot-buffer bytes
over HBM (measured copy peak). The resolve kernels' duration is bounded by the step graph's (hs_step_begin + the
resolves), which is what is used.

Also reported: e2e (the same steps through the public API with the selection copied in from pinned host memory
and out_slots copied back inside the timed region), a no-IO run (misses sourced from an HBM copy of the pool),
and the CPU oracle on a bounded sample (``cpu_baseline``).

`--impl reference` times the CPU oracle itself as the reference arm.
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

import numpy as np  # noqa: E402

import workload as wl  # noqa: E402

METRIC = "top-k selections resolved/s"
UNIT = "selections/s"
FLUSH_BYTES = 256 << 20
MLA_SCALE = 1.0 / math.sqrt(192.0)  # softmax scale of the attention consumer: 1/sqrt(128 + 64)


def describe(w: wl.Workload) -> str:
    sel = "shared by all layers" if w.shared_across_layers else "per layer"
    return (f"{w.name}: {w.requests} requests x {w.layers} layers, ctx {w.ctx}, top-k {w.topk} ({sel}), "
            f"{w.slots} hot slots, {w.row_bytes}-B rows, {w.steps} steps")


def mem_available() -> int:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def choose_host_layers(w: wl.Workload) -> int:
    """All layers get their own host pool when it fits in half of the available host memory; otherwise every
    layer reads one shared pool (host_layer_stride 0). Loads use ld.global.cv, so a shared pool still sends
    every miss over the link."""
    if w.layers == 1:
        return 1
    return w.layers if w.host_bytes() < 0.5 * mem_available() else 1


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        time.sleep(0.15)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

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


def kernel_sources_sha16() -> str:
    """Hash of the files the resolve kernel is compiled from (its translation unit and the headers it includes),
    which a committed ncu capture of that kernel must match."""
    import hashlib

    from hierarchical_sparse_attention_hs_gb300 import build as hs_build

    csrc = os.path.join(os.path.dirname(hs_build.__file__), "csrc")
    files = [os.path.join(csrc, n) for n in ("hs_resolve.cu", "hs_block.cuh", "hs_pool.hpp")]
    parts = [hashlib.sha256(open(f, "rb").read()).hexdigest() for f in files]
    return hashlib.sha256("".join(parts).encode()).hexdigest()[:16]


def captured_traffic(w: wl.Workload, cold_launches: int, steady_launches: int):
    """DRAM bytes per launch from the committed ncu capture of this workload, when the kernel sources are the
    ones it was taken on; else None."""
    path = os.path.join(ROOT, "profiles", f"hs_resolve_kernel_{w.name}_ncu.json")
    try:
        with open(path) as f:
            cap = json.load(f)
    except (OSError, ValueError):
        return None
    if cap.get("kernel_sources_sha16") != kernel_sources_sha16():
        return None
    d = cap["dram_bytes_per_launch"]
    n = cold_launches + steady_launches
    return (cold_launches * d["cold"] + steady_launches * d["steady"]) / n if n else None


def attention_sources_sha16() -> str:
    """Hash of the files the attention kernel is compiled from, which its committed ncu capture must match."""
    import hashlib

    from hierarchical_sparse_attention_hs_gb300 import build as hs_build

    csrc = os.path.join(os.path.dirname(hs_build.__file__), "csrc")
    files = [os.path.join(csrc, n) for n in ("hs_attention.cu", "hs_pool.hpp")]
    parts = [hashlib.sha256(open(f, "rb").read()).hexdigest() for f in files]
    return hashlib.sha256("".join(parts).encode()).hexdigest()[:16]


def captured_attention_traffic(w: wl.Workload):
    """DRAM bytes per launch of the attention kernel from its committed ncu capture on this workload, when the
    kernel sources are the ones it was taken on; else None."""
    path = os.path.join(ROOT, "profiles", f"hs_mla_decode_kernel_{w.name}_ncu.json")
    try:
        with open(path) as f:
            cap = json.load(f)
    except (OSError, ValueError):
        return None
    if cap.get("attention_sources_sha16") != attention_sources_sha16():
        return None
    return cap["dram_read_bytes"] + cap["dram_write_bytes"]


def meta_bytes_per_launch(w: wl.Workload, batch: int) -> int:
    """Metadata bytes of one resolve launch that do not depend on hits/misses: selection read, tok2slot gather,
    out_slots write (4k each) and the stamp + slot-token reads (8H), per request-layer."""
    return batch * (12 * w.topk + 8 * w.slots)


class GpuRun:
    """One pool for a workload, its per-step graphs, and the measurement passes."""

    def __init__(self, w: wl.Workload, noio: bool = False, prefetch: bool = False, host: object = None,
                 host_layers: int | None = None, layer_work_mb: float = 0.0, work_only: bool = False,
                 full_offload: bool = False, shared_call: bool = False, tiered_frac: float | None = None,
                 attention: bool = False):
        import torch

        import hierarchical_sparse_attention_hs_gb300 as hs

        self.torch, self.hs, self.w = torch, hs, w
        self.noio, self.prefetch = noio, prefetch
        self.host_layers = choose_host_layers(w) if host_layers is None else host_layers
        self.buf = hs.PoolBuffers(w.layers, w.requests, w.ctx, w.slots, w.topk, w.row_bytes,
                                  host_layers=self.host_layers, noio=noio, host=host)
        if host is None:
            wl.fill_host_pool(w, self.buf.host.ptr, self.host_layers)
        if noio:
            self.buf.upload_noio()
        self.pool = self.buf.create()
        sel = wl.gen_selections(w)  # [steps][selection layers][B][k]
        self.sel_host = sel
        self.sel = torch.from_numpy(sel).cuda()
        self.out = torch.empty((w.layers, w.requests, w.topk), dtype=torch.int32, device="cuda")
        self.stream = torch.cuda.Stream()
        self.side = torch.cuda.Stream() if prefetch else None
        self.host_io = None
        self.flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        # Stand-in for the rest of a decoder layer, run after each layer's resolve on the main stream: the
        # sparse-attention read of the selected rows (hs_gather) plus a copy of layer_work_mb MB (the layer's
        # other memory traffic). work_only replays the same per-layer work without any resolve.
        self.layer_work = layer_work_mb > 0 or work_only
        self.work_only = work_only
        # Comparator without a GPU cache: every step fetches all selected rows of every layer from the host
        # history (the traffic the resolution avoids), into a dense buffer.
        self.full_offload = full_offload
        # Layers that share one selection resolved by a single hs_resolve_shared call per step
        self.shared_call = shared_call and w.shared_across_layers
        # Three-tier resolution: per step, a resident map of the tokens still held in the HBM KV pool (one map per
        # request, shared by all layers as a block table is), kept in device memory like the pool's block table
        # Sparse MLA decode after each layer's resolve, reading the rows through out_slots (576 bf16 per row)
        self.attention = attention
        if attention:
            if w.row_bytes != hs.MLA_D_QK * 2:
                raise ValueError("--attention needs 1152-byte rows (the mla workload)")
            self.q = torch.from_numpy(wl.gen_queries(w.requests, hs.MLA_HEADS, hs.MLA_D_QK, w.seed).view(np.int16)).cuda()
            self.att_out = torch.empty((w.requests, hs.MLA_HEADS, hs.MLA_D_V), dtype=torch.float32, device="cuda")
            self.att_lse = torch.empty((w.requests, hs.MLA_HEADS), dtype=torch.float32, device="cuda")
        self.res = None
        if tiered_frac is not None:
            self.res = torch.from_numpy(wl.gen_resident(w.ctx, w.requests, w.steps, w.seed, frac=tiered_frac)).cuda()
        if full_offload:
            self.offload_buf = torch.empty(w.requests * w.topk * w.row_bytes, dtype=torch.uint8, device="cuda")
        if self.layer_work:
            self.gather_buf = torch.empty(w.requests * w.topk * w.row_bytes, dtype=torch.uint8, device="cuda")
            nb = max(16, int(layer_work_mb * (1 << 20)) // 16 * 16)
            self.work_src = torch.ones(nb, dtype=torch.uint8, device="cuda")
            self.work_dst = torch.empty(nb, dtype=torch.uint8, device="cuda")
            self.out.fill_(-1)
        torch.cuda.synchronize()
        self.graphs = [self._capture(s) for s in range(w.steps)]
        torch.cuda.synchronize()

    def _lsel(self, l):
        return 0 if self.w.shared_across_layers else l

    def _sel(self, s, ls):
        """Selection rows of step s, selection layer ls: the device copy, or (while graphs for the zero-copy
        end-to-end pass are captured) the address in the mapped host buffer."""
        if self.host_io is None:
            return self.sel[s][ls]
        host_sel, _ = self.host_io
        w = self.w
        return host_sel.ptr + ((s * w.selection_layers + ls) * w.requests * w.topk) * 4

    def _out(self, l):
        if self.host_io is None:
            return self.out[l]
        _, host_out = self.host_io
        return host_out.ptr + l * self.w.requests * self.w.topk * 4

    def enqueue(self, s):
        """Enqueue decode step s on self.stream: hs_step_begin, then the step's resolves."""
        if self.work_only:
            for l in range(self.w.layers):
                self.enqueue_layer_work(l)
            return
        if self.full_offload:
            w = self.w
            for l in range(w.layers):
                self.hs.hs_gather_history(self.pool, l, w.requests, self._sel(s, self._lsel(l)), w.topk,
                                          self.offload_buf, self.stream)
            return
        self.hs.hs_step_begin(self.pool, self.stream)
        self.enqueue_resolves(s)

    def enqueue_attention(self, l):
        w = self.w
        self.hs.hs_mla_decode(self.pool, l, w.requests, self.q, self._out(l), w.topk, None, 0, MLA_SCALE,
                              self.att_out, self.att_lse, self.stream)

    def enqueue_layer_work(self, l):
        if self.attention:
            self.enqueue_attention(l)
        if not self.layer_work:
            return
        w = self.w
        self.hs.hs_gather(self.pool, l, w.requests, self._out(l), w.topk, self.gather_buf, self.stream)
        with self.torch.cuda.stream(self.stream):
            self.work_dst.copy_(self.work_src)

    def enqueue_resolves(self, s):
        """Enqueue the resolves of decode step s (all layers, all requests) on self.stream, each followed by the
        layer's work stand-in when there is one."""
        torch, hs, w = self.torch, self.hs, self.w
        st = self.stream
        def src(ls):
            return self._sel(s, ls)

        if self.shared_call:
            hs.hs_resolve_shared(self.pool, 0, w.layers, w.requests, src(0), w.topk, self._out(0), st)
            for l in range(w.layers):
                self.enqueue_layer_work(l)
            return
        if self.res is not None:
            for l in range(w.layers):
                hs.hs_resolve_tiered(self.pool, l, w.requests, src(self._lsel(l)), w.topk, self.res[s], w.ctx,
                                     self._out(l), st)
                self.enqueue_layer_work(l)
            return
        if not self.prefetch:
            for l in range(w.layers):
                hs.hs_resolve(self.pool, l, w.requests, src(self._lsel(l)), w.topk, self._out(l), st)
                self.enqueue_layer_work(l)
            return
        # exact layer-wise prefetch: once layer l starts on the main stream, layer l+1 is resolved on the side
        # stream; layer l+1's own resolve waits for it and then only re-stamps and emits its slots
        side = self.side
        done = [None] * w.layers
        for l in range(w.layers):
            if done[l] is not None:
                st.wait_event(done[l])
            if l + 1 < w.layers:
                started = torch.cuda.Event()
                started.record(st)
                side.wait_event(started)
                hs.hs_prefetch(self.pool, l + 1, w.requests, src(self._lsel(l + 1)), w.topk, side)
                done[l + 1] = torch.cuda.Event()
                done[l + 1].record(side)
            hs.hs_resolve(self.pool, l, w.requests, src(self._lsel(l)), w.topk, self._out(l), st)
            self.enqueue_layer_work(l)

    def _capture(self, s):
        """One graph per decode step: hs_step_begin, then the step's resolves (programmatic dependent launch lets
        each kernel's launch overlap the one before it)."""
        g = self.torch.cuda.CUDAGraph()
        with self.torch.cuda.graph(g, stream=self.stream):
            self.enqueue(s)
        return g

    def launches_per_step(self) -> int:
        if self.attention:
            return 1 + 2 * self.w.layers
        if self.work_only or self.full_offload:
            return self.w.layers
        if self.shared_call:
            return 2 + (self.w.layers if self.layer_work else 0)
        return 1 + self.w.layers * (2 if self.layer_work else 1) + (self.w.layers - 1 if self.prefetch else 0)

    def flush(self):
        with self.torch.cuda.stream(self.stream):
            self.flush_buf.fill_(1)

    def reset(self):
        self.hs.hs_pool_reset(self.pool, self.stream)

    def run_steps(self, k_steps: int, timed: bool = True):
        """Replay k_steps decode steps of the sequence from the cold start (the pool must have just been reset),
        resetting it whenever the sequence wraps (outside the timed intervals). Returns a list of
        (sequence position, step ms) and the counters (hits, misses, evictions, bytes) summed over layers and
        steps."""
        torch = self.torch
        rows, pending = [], []
        totals = np.zeros(4, dtype=np.int64)

        def collect():
            self.stream.synchronize()
            for p, e0, e1 in pending:
                rows.append((p, e0.elapsed_time(e1)))
            pending.clear()

        pos = 0
        for _ in range(k_steps):
            if pos == self.w.steps:
                collect()
                totals += self.counters_total()
                pos = 0
                self.reset()
            self.flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(self.stream):
                if timed:
                    e0.record(self.stream)
                self.graphs[pos].replay()
                if timed:
                    e1.record(self.stream)
            if timed:
                pending.append((pos, e0, e1))
            pos += 1
        collect()
        totals += self.counters_total()
        return rows, totals

    def counters_total(self) -> np.ndarray:
        return self.buf.view("counters").cpu().numpy().astype(np.int64).sum(axis=0)

    def e2e_pass(self, k_steps: int):
        """Public-API loop with host buffers, zero-copy: the step graphs are captured again with the selections
        and out_slots in mapped page-locked host memory, which the kernels read and write over the host link
        themselves; events bracket each whole step. Returns (ms, h2d bytes, d2h bytes, out_slots match)."""
        torch, hs, w = self.torch, self.hs, self.w
        host_sel = hs.HostBuffer(self.sel_host.nbytes)
        host_out = hs.HostBuffer(self.out.numel() * 4)
        np.frombuffer(host_sel.numpy(), dtype=np.int32)[:] = self.sel_host.reshape(-1)
        self.host_io = (host_sel, host_out)
        try:
            graphs = [self._capture(s) for s in range(w.steps)]
        finally:
            self.host_io = None
        torch.cuda.synchronize()
        # first pass of the sequence on the device-memory graphs, kept for comparison with the zero-copy pass
        self.reset()
        ref = []
        for pos in range(w.steps):
            with torch.cuda.stream(self.stream):
                self.graphs[pos].replay()
            self.stream.synchronize()
            ref.append(self.out.cpu().numpy().copy())
        self.reset()
        host_out_np = np.frombuffer(host_out.numpy(), dtype=np.int32).reshape(tuple(self.out.shape))
        writes_slots = not (self.full_offload or self.work_only)
        match = True if writes_slots else None
        times = []
        pos = 0
        for _ in range(k_steps):
            if pos == w.steps:
                pos = 0
                self.reset()
            self.flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            with torch.cuda.stream(self.stream):
                graphs[pos].replay()
            e1.record(self.stream)
            times.append((e0, e1))
            e1.synchronize()
            if writes_slots:
                match = match and bool(np.array_equal(host_out_np, ref[pos]))
            pos += 1
        self.stream.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in times)
        del graphs
        host_sel.close()
        host_out.close()
        return ms, self.sel[0].numel() * 4, self.out.numel() * 4, match

    def attention_pass(self, k_steps: int) -> dict:
        """The attention consumer alone, on the slot lists the last step left: one graph per layer's launch
        replayed k_steps times, L2 flushed before each, CUDA events around each launch on its stream."""
        torch, w = self.torch, self.w
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            self.enqueue_attention(0)
        torch.cuda.synchronize()
        times = []
        for _ in range(k_steps):
            self.flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(self.stream):
                e0.record(self.stream)
                g.replay()
                e1.record(self.stream)
            times.append((e0, e1))
        self.stream.synchronize()
        ms = [a.elapsed_time(b) for a, b in times]
        slots = self.out[0].cpu().numpy()
        valid = int(((slots >= 0) & (slots < w.slots)).sum())
        flops = 2.0 * self.hs.MLA_HEADS * valid * (self.hs.MLA_D_QK + self.hs.MLA_D_V)
        return {"ms": statistics.mean(ms), "ms_p50": float(np.percentile(ms, 50)), "valid_rows": valid,
                "flops": flops}

    def e2e_copy_pass(self, k_steps: int):
        """The same loop with explicit copies: per step, copy the selections in from pinned host memory, run the
        step's graph, copy out_slots back to pinned host memory; events bracket the whole step."""
        torch = self.torch
        w = self.w
        self.reset()
        host_sel = torch.from_numpy(self.sel_host).pin_memory()  # [steps][Lsel][B][k]
        host_out = torch.empty(tuple(self.out.shape), dtype=torch.int32).pin_memory()
        times = []
        pos = 0
        for _ in range(k_steps):
            if pos == w.steps:
                pos = 0
                self.reset()
            self.flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            with torch.cuda.stream(self.stream):
                self.sel[pos].copy_(host_sel[pos], non_blocking=True)
                self.graphs[pos].replay()
                host_out.copy_(self.out, non_blocking=True)
            e1.record(self.stream)
            times.append((e0, e1))
            pos += 1
        self.stream.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in times)
        h2d = self.sel[0].numel() * 4
        d2h = self.out.numel() * 4
        return ms, h2d, d2h

    def close(self):
        self.buf.close()


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


def _oracle_requests(w: wl.Workload, lo: int, hi: int, sel: np.ndarray, host: np.ndarray, res, budget_s: float,
                     t0: float) -> tuple:
    """Steps of layer 0 for requests lo..hi-1 from the cold start, the sequence replayed from a fresh cache each
    time it ends (as the GPU passes do), until the budget; (selections, steps)."""
    import oracle

    n = steps = 0
    while time.perf_counter() - t0 < budget_s:
        pool = oracle.OraclePool(w.ctx, w.slots, w.row_bytes, 1, hi - lo, track_rows=True)
        for s in range(w.steps):
            if time.perf_counter() - t0 >= budget_s:
                break
            pool.step_begin()
            pool.resolve(0, sel[s, 0, lo:hi], host[lo:hi], resident=None if res is None else res[s, lo:hi])
            n += hi - lo
            steps += 1
    return n, steps


def cpu_baseline(w: wl.Workload, budget_s: float = 12.0, tiered_frac: float | None = None,
                 threads: int = 1) -> dict:
    """The CPU oracle on a bounded sample of the same workload: request-layers of layer 0, hot rows tracked in
    host memory, steps in order from the cold start until the time budget. With threads > 1 the requests are
    split over that many threads (the oracle's C routine runs without the interpreter lock), each resolving its
    own requests, which are independent."""
    import threading

    reqs = w.requests
    sel = wl.gen_selections(w, layers=(0, 1), requests=(0, reqs))
    host = np.stack([wl.rows(w, 0, b) for b in range(reqs)])
    res = None if tiered_frac is None else wl.gen_resident(w.ctx, reqs, w.steps, w.seed, frac=tiered_frac)
    threads = max(1, min(threads, reqs))
    bounds = [reqs * i // threads for i in range(threads + 1)]
    results = [None] * threads
    t0 = time.perf_counter()

    def work(i):
        results[i] = _oracle_requests(w, bounds[i], bounds[i + 1], sel, host, res, budget_s, t0)

    ths = [threading.Thread(target=work, args=(i,)) for i in range(threads)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    dt = time.perf_counter() - t0
    n = sum(r[0] for r in results)
    steps = min(r[1] for r in results)
    mode = "single-threaded" if threads == 1 else f"{threads} threads over the requests"
    return {"value": n / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"layer 0 of {w.name}, {reqs} requests, at least {steps} decode steps (the {w.steps}-step "
                      f"sequence replayed from the cold start; {n} selections, hot rows tracked" +
                      (", resident maps" if res is not None else "") + f", {dt:.1f} s {mode})"}


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


def run_reference(args) -> int:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle

    w = wl.WORKLOADS[args.workload]
    reqs = w.requests
    sel = wl.gen_selections(w, layers=(0, 1), requests=(0, reqs))
    host = np.stack([wl.rows(w, 0, b) for b in range(reqs)])
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
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": describe(w), "sample": f"{layers_per_step} layer(s) per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} decode steps of {layers_per_step} layer(s) x {reqs} requests of "
                                   f"{w.name}, hot rows tracked, single-threaded"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args) -> int:
    import torch

    import hierarchical_sparse_attention_hs_gb300 as hs
    from hierarchical_sparse_attention_hs_gb300 import build as hs_build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    if rank == 0:
        hs_build.build()
    if dist:
        dist.barrier()
    hs.load()
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    hbm_src = "measured" if "hbm_gbs" in peaks else "fallback"

    w = wl.WORKLOADS[args.workload]
    K, W = args.steps, args.warmup
    run = GpuRun(w, prefetch=args.prefetch, layer_work_mb=args.layer_work_mb, work_only=args.work_only,
                 full_offload=args.full_offload, shared_call=args.shared_call, tiered_frac=args.tiered_frac,
                 attention=args.attention)
    # The GPU reads the whole host pool once (as a long-running server has long since done), so that first-touch
    # address translation of host pages is not charged to the timed steps; it also measures the link.
    link_zc, link_cp = measure_link(hs, torch, run.buf.host.ptr, run.buf.host.nbytes // 16 * 16)
    pool_bytes = {"host": run.buf.host.nbytes, "hot_buffer": run.buf.hot.numel(), "metadata": run.buf.meta.numel()}
    # warm-up, then a cold start for the timed region
    nvtx = torch.cuda.nvtx
    nvtx.range_push(f"warm-up: {W} steps of {w.name}")
    run.run_steps(W, timed=False)
    run.reset()
    run.stream.synchronize()
    nvtx.range_pop()

    def barrier():
        if dist:
            dist.barrier()
        torch.cuda.synchronize()

    barrier()
    with ClockSampler(local) as clk:
        nvtx.range_push(f"timed: {K} steps of {w.name}")
        per_step, tot = run.run_steps(K)
        nvtx.range_pop()
        barrier()
    step_ms = [r[1] for r in per_step]
    # The resolve launches of a step run back to back in the step's graph behind hs_step_begin, their launches
    # overlapped by programmatic dependent launch; their duration is bounded by the step's, which is used.
    kern_ms = sum(step_ms)
    total_ms = max_over_ranks(sum(step_ms), dist)
    sel_per_step = w.layers * w.requests
    value = aggregate_rate(world, K * sel_per_step, total_ms)
    n_launch = K * w.layers  # per-layer resolutions (one launch each, or one launch per step with --shared-call)
    n_kernels = K if run.shared_call else n_launch

    hits, misses, evictions, miss_bytes = (int(x) for x in tot)
    if args.full_offload:  # every selected row crossed the link
        hits, misses = 0, K * w.layers * w.requests * w.topk
        miss_bytes = misses * w.row_bytes
    link_peak = max(link_zc, link_cp)
    meta = n_launch * meta_bytes_per_launch(w, w.requests) + 4 * hits + 16 * misses
    if run.res is not None:  # the resident-map lookup of every selected token
        meta += 4 * n_launch * w.requests * w.topk
    hbm_bytes = meta + miss_bytes
    t_link = miss_bytes / (link_peak * 1e9)
    t_hbm = hbm_bytes / (hbm_peak * 1e9)
    kern_s = kern_ms / 1e3
    bound = "host_link" if t_link >= t_hbm else "hbm"
    roofline = {
        "bound": bound,
        "achieved": (miss_bytes / kern_s / 1e9) if bound == "host_link" else (hbm_bytes / kern_s / 1e9),
        "peak": link_peak if bound == "host_link" else hbm_peak,
        "unit": "GB/s",
        "frac": max(t_link, t_hbm) / kern_s,
        "traffic": captured_traffic(w, sum(w.layers for r in per_step if r[0] == 0),
                                    sum(w.layers for r in per_step if r[0] != 0)),
        "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum per launch from the committed ncu capture "
                          "(profiles/), null unless taken on these kernel sources",
        "kernel": "hs_resolve_kernel",
        "kernel_ms_per_launch": kern_ms / n_kernels,
        "launches": n_kernels,
        "timing": ("CUDA events around each step's graph in the timed region: hs_step_begin plus the step's "
                   "resolves, an upper bound on the resolve launches" +
                   (" (layer-wise prefetch included)" if args.prefetch else "")),
        "algorithmic_bytes_per_launch": {"link": miss_bytes / n_kernels, "hbm": hbm_bytes / n_kernels},
        "peak_source": f"host link measured in this run (zero-copy {link_zc:.1f}, memcpy {link_cp:.1f} GB/s); "
                       f"HBM {hbm_peak:.1f} GB/s {hbm_src}",
    }

    attention = None
    if args.attention:
        # the consumer alone, on the slot lists of the sequence's last step (steady state)
        a = run.attention_pass(K)
        bf16_peak = float(peaks.get("bf16_tflops", 1900.0))
        tflops = a["flops"] / (a["ms"] / 1e3) / 1e12
        attention = {
            "kernel": "hs_mla_decode_kernel", "bound": "tensor", "achieved": tflops, "peak": bf16_peak,
            "unit": "TFLOP/s", "frac": tflops / bf16_peak, "ms_per_launch": a["ms"], "ms_per_launch_p50": a["ms_p50"],
            "flops_per_launch": a["flops"], "valid_rows_per_launch": a["valid_rows"],
            "flops_definition": "2 * 128 heads * valid rows * (576 + 512): the score and value products; no "
                                "score work is repeated (each CTA of a pair computes the scores over its own columns)",
            "row_bytes_per_launch": a["valid_rows"] * w.row_bytes,
            "traffic": captured_attention_traffic(w),
            "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum per launch from the committed ncu capture "
                              "(profiles/), null unless taken on these kernel sources",
            "peak_source": "bf16_tflops (cuBLAS bf16 GEMM, burst) in MEASURED_PEAKS.json" if "bf16_tflops" in peaks
                           else "fallback 1900 TFLOP/s",
            "timing": "CUDA events around one graph launch each, L2 flushed before each, on the launch stream",
        }

    # end to end through the public API with host buffers: zero-copy (the kernels read the selections from and
    # write out_slots to mapped host memory), and with explicit staging copies
    nvtx.range_push("end to end, zero-copy")
    e2e_ms, h2d, d2h, e2e_match = run.e2e_pass(K)
    nvtx.range_pop()
    e2e_ms = max_over_ranks(e2e_ms, dist)
    c_ms, c_h2d, c_d2h = run.e2e_copy_pass(K)
    c_ms = max_over_ranks(c_ms, dist)
    e2e = {"value": aggregate_rate(world, K * sel_per_step, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h,
           "path": "selections and out_slots in mapped page-locked host memory, read and written by the kernels "
                   "over the host link (no staging copies); L2 flushed between steps",
           "out_slots_match_device_path": e2e_match,
           "with_copies": {"value": aggregate_rate(world, K * sel_per_step, c_ms), "unit": UNIT,
                           "h2d_bytes_per_step": c_h2d, "d2h_bytes_per_step": c_d2h,
                           "path": "cudaMemcpyAsync of the selections in and out_slots out around each step's graph"}}
    host = run.buf.host
    run.buf.host = None
    run.close()
    torch.cuda.empty_cache()

    # no-IO mode on the same workload: misses sourced from an HBM copy of the pool
    noio = None
    if not args.skip_noio:
        nrun = GpuRun(w, noio=True, prefetch=args.prefetch, host=host, host_layers=run.host_layers,
                      layer_work_mb=args.layer_work_mb, work_only=args.work_only, full_offload=args.full_offload,
                      shared_call=args.shared_call, tiered_frac=args.tiered_frac)
        nvtx.range_push("no-IO")
        nrun.run_steps(W, timed=False)
        nrun.reset()
        nper, _ = nrun.run_steps(K)
        nvtx.range_pop()
        nms = max_over_ranks(sum(r[1] for r in nper), dist)
        nk_ms = sum(r[1] for r in nper)
        n_hbm = meta + 2 * miss_bytes
        noio = {"value": aggregate_rate(world, K * sel_per_step, nms), "unit": UNIT, "ms_per_step": nms / K,
                "kernel_ms_per_launch": nk_ms / n_kernels,
                "roofline": {"bound": "hbm", "achieved": n_hbm / (nk_ms / 1e3) / 1e9, "peak": hbm_peak,
                             "unit": "GB/s", "frac": (n_hbm / (hbm_peak * 1e9)) / (nk_ms / 1e3)}}
        nrun.buf.host = None
        nrun.close()
    host.close()

    clocks = clk.summary()
    cold = [r[1] for r in per_step if r[0] == 0]
    churn = [r[1] for r in per_step if r[0] in w.churn]  # steps whose selection shares nothing with the last
    steady = [r[1] for r in per_step if r[0] != 0 and r[0] not in w.churn]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int32", "data": "synthetic",
        "config": {"workload": describe(w), "parallelism": f"replicas x{world} (independent requests per GPU)",
                   "l2": "flushed between steps (256 MiB write)",
                   "host_pool": ("one pool per layer" if run.host_layers == w.layers else
                                 "layers share one host pool (host_layer_stride 0); every miss still crosses the link"),
                   "graphs": "one CUDA graph per decode step", "prefetch": bool(args.prefetch),
                   "pool_bytes": pool_bytes,
                   "layer_work_mb": args.layer_work_mb, "work_only": bool(args.work_only),
                   "full_offload": bool(args.full_offload), "shared_call": bool(args.shared_call),
                   "tiered_frac": args.tiered_frac, "attention": bool(args.attention)},
        "selected_entries_per_s": value * w.topk,
        "miss_gbs": miss_bytes / (total_ms / 1e3) / 1e9 * world,
        "cold_step_ms": statistics.mean(cold) if cold else None,
        "churn_step_ms": statistics.mean(churn) if churn else None,
        "steady_step_ms": statistics.mean(steady) if steady else None,
        "steady_step_ms_p10_p50_p90": ([float(np.percentile(steady, q)) for q in (10, 50, 90)] if steady else None),
        "roofline": roofline,
        "noio": noio,
        "e2e": e2e,
        "gpu_launches": K * run.launches_per_step(),
        "attention": attention,
        "clocks": clocks,
    }
    if rank == 0 and not args.skip_cpu:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget, tiered_frac=args.tiered_frac)
        if min(args.cpu_threads, w.requests) > 1:
            line["cpu_baseline_threads"] = cpu_baseline(w, budget_s=args.cpu_budget, tiered_frac=args.tiered_frac,
                                                        threads=args.cpu_threads)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main() -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["hs", "reference"], default="hs")
    ap.add_argument("--workload", choices=list(wl.WORKLOADS), default="dsa")
    ap.add_argument("--prefetch", action="store_true", help="layer-wise prefetch on a second stream")
    ap.add_argument("--layer-work-mb", type=float, default=0.0,
                    help="per-layer work stand-in after each resolve: hs_gather + a copy of this many MB")
    ap.add_argument("--work-only", action="store_true",
                    help="replay only the per-layer work stand-in (no resolve): the reference for exposed time")
    ap.add_argument("--shared-call", action="store_true",
                    help="workloads whose layers share one selection: one hs_resolve_shared call per step")
    ap.add_argument("--full-offload", action="store_true",
                    help="comparator without a GPU cache: fetch every selected row from host memory every step")
    ap.add_argument("--skip-noio", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--cpu-threads", type=int, default=os.cpu_count() or 1,
                    help="threads of the second, multi-threaded CPU-oracle line (1 = skip it)")
    ap.add_argument("--tiered-frac", type=float, default=None,
                    help="three-tier resolution: fraction of pages still held in the HBM KV pool (plus the newest "
                         "256 tokens), one resident map per request and step")
    ap.add_argument("--attention", action="store_true",
                    help="sparse MLA decode (hs_mla_decode) after each layer's resolve; needs 1152-byte rows (the "
                         "mla workload); adds the attention kernel's tensor-core roofline")
    ap.add_argument("--ref-layers", type=int, default=1, help="reference arm: layers resolved per step")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.attention and (args.tiered_frac is not None or args.full_offload or args.work_only):
        ap.error("--attention reads the slot lists of plain resolves; it combines with none of --tiered-frac, "
                 "--full-offload, --work-only")
    if args.tiered_frac is not None and (args.prefetch or args.shared_call or args.full_offload):
        ap.error("--tiered-frac resolves each layer with its own call; it combines with none of --prefetch, "
                 "--shared-call, --full-offload")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
