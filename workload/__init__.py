"""Seeded synthetic workloads for the hierarchical KV cache resolver.

This module only draws inputs: top-k selection streams and host KV row contents. It holds none of the
resolution method's arithmetic, so the CPU oracle and the CUDA path can both consume its output without sharing
any of the method's code.

The five workloads stand in for the unnamed long-context sparse-attention serving workloads of the HiSparse paper
("HiSparse: Scaling Sparse-Attention Decoding with Hierarchical KV Cache Management", Abstract: DSA, NSA and Quest
families) and the 1M-token setting of the "Hybrid HiSparse" knowledge card (Timeline: GLM 5.3, 8xH200, 1M tokens).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wl_gen.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libhs_workload.so")
_lib = None
_lock = threading.Lock()

UNIFORM, ZIPF = 0, 1
ROWS_BF16_NORMAL, ROWS_HASH = 0, 1
BASE_SEED = 20260807


def build(force: bool = False) -> str:
    """Compile the generator into a shared library next to this file (plain C, gcc)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, i64, u64, f64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p
            lib.wl_gen_selections.argtypes = [u64, i32, i32, i32, i32, i32, f64, vp, i32, i32, i32, i32, i32, vp]
            lib.wl_gen_selections.restype = ctypes.c_int
            lib.wl_fill_rows.argtypes = [u64, i32, i32, i32, i32, i64, i64, vp]
            lib.wl_fill_rows.restype = ctypes.c_int
            lib.wl_splitmix64.argtypes = [ctypes.POINTER(u64)]
            lib.wl_splitmix64.restype = u64
            lib.wl_xoshiro_sequence.argtypes = [u64, u64, u64, u64, ctypes.c_int, vp]
            lib.wl_xoshiro_sequence.restype = None
            lib.wl_stream_seed.argtypes = [u64, i32, i32]
            lib.wl_stream_seed.restype = u64
            _lib = lib
    return _lib


@dataclass(frozen=True)
class Workload:
    """Shapes and selection-stream recipe of one synthetic workload.

    layers x requests request-layers (independent cache instances), each with a host history of `ctx` selection
    units (tokens, or pages), a hot buffer of `slots` rows of `row_bytes` bytes, and `topk` selections per step.
    """

    name: str
    index: int
    layers: int
    requests: int
    ctx: int
    topk: int
    slots: int
    row_bytes: int
    steps: int
    keep_pct: int
    dist: int
    zipf_s: float = 0.0
    churn: tuple = field(default_factory=tuple)
    shared_across_layers: bool = False
    row_kind: int = ROWS_HASH

    @property
    def seed(self) -> int:
        return BASE_SEED + self.index

    @property
    def selection_layers(self) -> int:
        """Number of independent selection streams per request (1 when all layers share one selection)."""
        return 1 if self.shared_across_layers else self.layers

    def host_bytes(self, host_layers: int | None = None) -> int:
        hl = self.layers if host_layers is None else host_layers
        return hl * self.requests * self.ctx * self.row_bytes

    def hot_bytes(self) -> int:
        return self.layers * self.requests * self.slots * self.row_bytes


WORKLOADS = {
    "tiny": Workload("tiny", 1, layers=1, requests=1, ctx=4096, topk=64, slots=512, row_bytes=1152, steps=16,
                     keep_pct=70, dist=UNIFORM, row_kind=ROWS_BF16_NORMAL),
    "dsa": Workload("dsa", 2, layers=1, requests=32, ctx=131072, topk=2048, slots=4096, row_bytes=656, steps=64,
                    keep_pct=80, dist=ZIPF, zipf_s=1.1),
    "multilayer": Workload("multilayer", 3, layers=61, requests=16, ctx=262144, topk=2048, slots=4096,
                           row_bytes=656, steps=32, keep_pct=60, dist=UNIFORM, churn=(8, 16, 24)),
    "quest": Workload("quest", 4, layers=32, requests=8, ctx=8192, topk=256, slots=512, row_bytes=32768,
                      steps=128, keep_pct=75, dist=UNIFORM),
    "shared": Workload("shared", 5, layers=78, requests=8, ctx=1048576, topk=2048, slots=8192, row_bytes=656,
                       steps=32, keep_pct=85, dist=ZIPF, zipf_s=1.05, shared_across_layers=True),
    # the dsa stream with rows an attention kernel can read: 576 bf16 values (512 latent + 64 rotary)
    "mla": Workload("mla", 6, layers=1, requests=32, ctx=131072, topk=2048, slots=4096, row_bytes=1152, steps=32,
                    keep_pct=80, dist=ZIPF, zipf_s=1.1, row_kind=ROWS_BF16_NORMAL),
}


def gen_selections(w: Workload, layers=None, requests=None, steps: int | None = None) -> np.ndarray:
    """Selections int32 [steps][len(layers)][len(requests)][topk] for a contiguous layer/request range.

    `layers` / `requests` are (start, count) tuples; by default all selection layers and all requests.
    For a workload shared across layers there is one selection layer (index 0).
    """
    lib = _load()
    l0, nl = layers if layers is not None else (0, w.selection_layers)
    r0, nr = requests if requests is not None else (0, w.requests)
    ns = w.steps if steps is None else steps
    if l0 < 0 or nl < 1 or l0 + nl > w.selection_layers or r0 < 0 or nr < 1 or r0 + nr > w.requests:
        raise ValueError("layer/request range outside the workload")
    out = np.empty((ns, nl, nr, w.topk), dtype=np.int32)
    churn = np.asarray(w.churn if w.churn else [-1], dtype=np.int32)
    rc = lib.wl_gen_selections(w.seed, w.ctx, w.topk, ns, w.keep_pct, w.dist, w.zipf_s,
                               churn.ctypes.data, len(w.churn), l0, nl, r0, nr, out.ctypes.data)
    if rc != 0:
        raise RuntimeError("selection generator rejected its arguments")
    return out


def fill_rows_at(w: Workload, address: int, layer: int, request: int, tok0: int, ntok: int) -> None:
    """Write host rows (layer, request, tok0 .. tok0+ntok-1) to raw host memory at `address`."""
    rc = _load().wl_fill_rows(w.seed, w.row_kind, w.row_bytes, layer, request, tok0, ntok, ctypes.c_void_p(address))
    if rc != 0:
        raise RuntimeError("row generator rejected its arguments")


def rows(w: Workload, layer: int, request: int, tok0: int = 0, ntok: int | None = None) -> np.ndarray:
    """Host rows of one request-layer as uint8 [ntok][row_bytes]."""
    n = w.ctx - tok0 if ntok is None else ntok
    out = np.empty((n, w.row_bytes), dtype=np.uint8)
    fill_rows_at(w, out.ctypes.data, layer, request, tok0, n)
    return out


def fill_host_pool(w: Workload, address: int, host_layers: int, threads: int | None = None,
                   extra_rows: int = 0) -> None:
    """Fill a host pool laid out [host_layers][requests][ctx][row_bytes] at raw address `address`, followed by
    `extra_rows` more rows (a shared pool read with a per-layer shift reaches past its last request's rows).

    Layer l of the pool holds the rows of layer l (host_layers == layers) or, when layers alias a smaller pool,
    of pool layer l; the extra rows hold rows ctx, ctx + 1, ... of the last request of the last pool layer.
    Filled in parallel chunks (the C routine releases the GIL through ctypes).
    """
    per_rl = w.ctx * w.row_bytes
    jobs = [(l, b) for l in range(host_layers) for b in range(w.requests)]
    nthreads = threads or min(16, os.cpu_count() or 1)
    chunk = max(1, w.ctx // 8)

    tasks = []
    for (l, b) in jobs:
        for t0 in range(0, w.ctx, chunk):
            n = min(chunk, w.ctx - t0)
            tasks.append((l, b, t0, n))
    # rows ctx .. of (last layer, last request) continue the pool contiguously
    for t0 in range(w.ctx, w.ctx + extra_rows, chunk):
        tasks.append((host_layers - 1, w.requests - 1, t0, min(chunk, w.ctx + extra_rows - t0)))

    def worker(idx):
        for i in range(idx, len(tasks), nthreads):
            l, b, t0, n = tasks[i]
            fill_rows_at(w, address + (l * w.requests + b) * per_rl + t0 * w.row_bytes, l, b, t0, n)

    ths = [threading.Thread(target=worker, args=(i,)) for i in range(nthreads)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()


def splitmix64_sequence(seed: int, n: int) -> list:
    lib = _load()
    st = ctypes.c_uint64(seed)
    return [lib.wl_splitmix64(ctypes.byref(st)) for _ in range(n)]


def xoshiro_sequence(state, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().wl_xoshiro_sequence(*[ctypes.c_uint64(s) for s in state], n, out.ctypes.data)
    return out


def gen_resident(ctx: int, batch: int, steps: int, seed: int, window: int = 256, page: int = 64,
                 frac: float = 0.3) -> np.ndarray:
    """Resident-tier maps int32 [steps][batch][ctx] for the three-tier resolver: entry t is the row of token t in
    the ordinary HBM KV pool, or -1 when the token's KV lives only in host memory.

    Recipe: the newest `window` tokens are resident (they were written by the latest decode steps), and every
    other page of `page` tokens is resident with probability `frac`, drawn afresh each step. Resident pages take
    distinct pool blocks in random order, so rows are distinct within a request.
    """
    if ctx % page:
        raise ValueError("ctx must be a multiple of page")
    rng = np.random.default_rng([seed, 0x5E5D, ctx, batch])
    npages = ctx // page
    out = np.full((steps, batch, ctx), -1, dtype=np.int32)
    first_window_page = max(0, (ctx - window) // page)
    for s in range(steps):
        for b in range(batch):
            res = rng.random(npages) < frac
            res[first_window_page:] = True
            pages = np.flatnonzero(res)
            blocks = rng.permutation(npages)[: len(pages)]
            rows = (blocks[:, None] * page + np.arange(page)[None, :]).astype(np.int32)
            out[s, b].reshape(npages, page)[pages] = rows
    return out


def gen_queries(batch: int, heads: int, dim: int, seed: int) -> np.ndarray:
    """Decode queries as bf16 bit patterns uint16 [batch][heads][dim]: N(0,1) float32 draws (numpy generator
    seeded by (seed, batch, heads, dim)) rounded to nearest even."""
    rng = np.random.default_rng([seed, 0x9E37, batch, heads, dim])
    f = rng.standard_normal((batch, heads, dim), dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)
