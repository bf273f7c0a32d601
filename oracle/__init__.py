"""CPU oracle for the hierarchical KV cache resolver -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import this package. The
library path (``hierarchical_sparse_attention_hs_gb300``) never does, and the two share no code.

The arithmetic lives in ``hs_oracle.c`` (plain C, one request-layer at a time, library ``qsort`` for every ordering
step). It follows the per-layer resolution of the HiSparse paper (Abstract): each layer's selections are looked
up in the GPU cache, least recently used entries make room, and the missing rows come from host memory, within the
decode step; only where the KV rows sit changes, so the model computes the same outputs. The policy is fully
specified: hits take the current decode step as stamp; victims are the
non-selected slots with the oldest stamp, ties to the lowest slot index; misses go to victims in ascending token
order; empty slots (stamp 0) are used first.

:class:`OraclePool` keeps that state for a chosen subset of (layer, request) cache instances, so the large
workloads can be checked on sampled request-layers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hs_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libhs_oracle.so")
_lib = None
_lock = threading.Lock()

ERR_RANGE = 1
ERR_DUP = 2


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, -O2, no vectorisation pragmas) into oracle/_build/."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Open a compiled oracle and declare its entry points."""
    lib = ctypes.CDLL(path)
    i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    lib.ora_resolve_rl.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i32, vp, vp]
    lib.ora_resolve_rl.restype = ctypes.c_int
    lib.ora_resolve_batch.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, i64, vp, i32, vp, vp]
    lib.ora_resolve_batch.restype = ctypes.c_int
    lib.ora_resolve_batch_tiered.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, i64, vp, i32, vp, vp, vp]
    lib.ora_resolve_batch_tiered.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


class OraclePool:
    """Oracle state for `n_layers` x `n_requests` request-layers of one cache geometry.

    Arrays mirror the device metadata: ``tok2slot`` int32 [n_layers][n_requests][ctx] (-1 = not resident),
    ``slot_tok`` int32 [n_layers][n_requests][slots] (-1 = empty), ``slot_stamp`` int32 (0 = never used),
    ``hot`` uint8 [n_layers][n_requests][slots][row_bytes] (optional), ``counters`` uint64 [n_layers][4] =
    (hits, misses, evictions, bytes). ``step`` is the decode step counter, ``error`` the OR of rejected-row bits.
    """

    def __init__(self, ctx: int, slots: int, row_bytes: int, n_layers: int = 1, n_requests: int = 1,
                 track_rows: bool = True, library=None):
        self._lib = library if library is not None else _load()
        self.ctx, self.slots, self.row_bytes = ctx, slots, row_bytes
        self.n_layers, self.n_requests = n_layers, n_requests
        self.tok2slot = np.full((n_layers, n_requests, ctx), -1, dtype=np.int32)
        self.slot_tok = np.full((n_layers, n_requests, slots), -1, dtype=np.int32)
        self.slot_stamp = np.zeros((n_layers, n_requests, slots), dtype=np.int32)
        self.hot = np.zeros((n_layers, n_requests, slots, row_bytes), dtype=np.uint8) if track_rows else None
        self.counters = np.zeros((n_layers, 4), dtype=np.uint64)
        self.step = 0
        self.error = 0

    def step_begin(self) -> None:
        self.step += 1

    def resolve(self, layer: int, sel: np.ndarray, host_rows: np.ndarray | None = None,
                want_slots: bool = True, resident: np.ndarray | None = None) -> np.ndarray | None:
        """Resolve one call for oracle layer `layer` over its requests.

        sel: int32 [n_requests][k]; host_rows: uint8 [n_requests][ctx][row_bytes] (needed when rows are tracked);
        resident: optional int32 [n_requests][ctx], the row of each token still held in the HBM KV pool (or -1),
        for the three-tier variant. Returns out_slots int32 [n_requests][k] (or None when want_slots is False,
        the prefetch form).
        """
        sel = np.ascontiguousarray(sel, dtype=np.int32)
        nb, k = sel.shape
        if nb != self.n_requests:
            raise ValueError("selection batch must cover every tracked request")
        out = np.empty((nb, k), dtype=np.int32) if want_slots else None
        hot = self.hot[layer] if self.hot is not None else None
        if hot is not None:
            if host_rows is None or host_rows.shape != (nb, self.ctx, self.row_bytes):
                raise ValueError("host rows [requests][ctx][row_bytes] are needed when rows are tracked")
            host_rows = np.ascontiguousarray(host_rows, dtype=np.uint8)
        cnt = np.zeros(4, dtype=np.uint64)
        if resident is not None:
            resident = np.ascontiguousarray(resident, dtype=np.int32)
            if resident.shape != (nb, self.ctx):
                raise ValueError("resident map must be [requests][ctx]")
        rc = self._lib.ora_resolve_batch_tiered(self.step, self.ctx, self.slots, self.row_bytes, nb,
                                                _ptr(self.tok2slot[layer]), _ptr(self.slot_tok[layer]),
                                                _ptr(self.slot_stamp[layer]), _ptr(hot),
                                                _ptr(host_rows) if hot is not None else None,
                                                self.ctx * self.row_bytes, _ptr(sel), k, _ptr(resident),
                                                _ptr(out), _ptr(cnt))
        if rc < 0:
            raise RuntimeError(f"oracle precondition failed ({rc})")
        self.error |= rc
        self.counters[layer] += cnt
        return out

    def resolve_one(self, layer: int, req: int, sel: np.ndarray, host_rows: np.ndarray | None = None) -> tuple:
        """Resolve a single request-layer; returns (out_slots, error_bits)."""
        sel = np.ascontiguousarray(sel, dtype=np.int32)
        k = sel.shape[0]
        out = np.empty(k, dtype=np.int32)
        hot = self.hot[layer, req] if self.hot is not None else None
        rows = None
        if hot is not None:
            if host_rows is None or host_rows.shape != (self.ctx, self.row_bytes):
                raise ValueError("host rows [ctx][row_bytes] are needed when rows are tracked")
            rows = np.ascontiguousarray(host_rows, dtype=np.uint8)
        cnt = np.zeros(4, dtype=np.uint64)
        rc = self._lib.ora_resolve_rl(self.step, self.ctx, self.slots, self.row_bytes,
                                      _ptr(self.tok2slot[layer, req]), _ptr(self.slot_tok[layer, req]),
                                      _ptr(self.slot_stamp[layer, req]), _ptr(hot), _ptr(rows),
                                      _ptr(sel), k, _ptr(out), _ptr(cnt))
        if rc < 0:
            raise RuntimeError(f"oracle precondition failed ({rc})")
        self.error |= rc
        self.counters[layer] += cnt
        return out, rc
