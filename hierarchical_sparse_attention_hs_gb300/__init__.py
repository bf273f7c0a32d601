"""Python binding of the hs C ABI (include/hs.h): argument marshalling only.

Every step of the resolution runs in the CUDA kernels of ``libhs.so``; this module only converts torch tensors,
streams and integers into the plain pointers and sizes of the C entry points, and raises :class:`HsError` on a
negative return code. PyTorch is used for device memory and streams. There is no CPU fallback: if the library
has not been built, loading it raises.

The method is the per-layer selection resolution of "HiSparse: Scaling Sparse-Attention Decoding with
Hierarchical KV Cache Management" (Abstract); the policy and the memory layout are documented in hs.h.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build_mod

__all__ = [
    "HsError", "hs_pool_desc", "hs_meta_layout", "load", "hs_meta_bytes", "hs_get_meta_layout", "hs_pool_create",
    "hs_pool_reset", "hs_step_begin", "hs_resolve", "hs_prefetch", "hs_get_error", "hs_get_counters",
    "hs_pool_destroy", "hs_host_alloc", "hs_host_free", "hs_error_string", "HS_DEVERR_RANGE", "HS_DEVERR_DUP",
    "HS_DEVERR_STATE", "HostBuffer", "PoolBuffers", "hs_probe_link", "hs_gather", "hs_gather_history",
    "hs_resolve_shared", "hs_resolve_tiered", "hs_mla_decode", "hs_mla_decode_history", "HS_DEVERR_TIMEOUT",
    "MLA_HEADS", "MLA_D_QK", "MLA_D_V", "hs_probe_launch", "hs_debug_attention", "hs_step_begin_fused", "hs_probe_link_static", "HS_ERR_TOO_LARGE",
    "hs_resolve_ids", "hs_prefetch_ids",
]

HS_OK = 0
HS_ERR_INVALID_ARG = -1
HS_ERR_CUDA = -2
HS_ERR_NOT_MAPPED = -3
HS_ERR_NO_MEMORY = -4
HS_ERR_UNSUPPORTED = -5
HS_ERR_TOO_LARGE = -6
HS_DEVERR_RANGE = 1
HS_DEVERR_DUP = 2
HS_DEVERR_STATE = 4
HS_DEVERR_TIMEOUT = 8
MLA_HEADS, MLA_D_QK, MLA_D_V = 128, 576, 512  # shape of the sparse MLA decode consumer

LIB_PATH = _build_mod.LIB_PATH
_lib = None
_lock = threading.Lock()


class HsError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {hs_error_string(code)} ({code})")
        self.code = code


class hs_pool_desc(ctypes.Structure):
    _fields_ = [
        ("layers", ctypes.c_int32), ("max_batch", ctypes.c_int32), ("ctx", ctypes.c_int32),
        ("slots", ctypes.c_int32), ("topk_max", ctypes.c_int32), ("row_bytes", ctypes.c_int32),
        ("host_pool", ctypes.c_void_p), ("host_layer_stride", ctypes.c_int64), ("host_req_stride", ctypes.c_int64),
        ("hot_buf", ctypes.c_void_p), ("meta", ctypes.c_void_p), ("noio_src", ctypes.c_void_p),
    ]


class hs_meta_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("step", "error", "counters", "tok2slot", "slot_tok", "slot_stamp", "total")]


def load():
    """Open libhs.so (built by ``build.build()``); raises if it is missing -- there is no other path."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run hierarchical_sparse_attention_hs_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        P, vp, i32, sz = ctypes.POINTER, ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        sig = {
            "hs_meta_bytes": (sz, [P(hs_pool_desc)]),
            "hs_get_meta_layout": (ctypes.c_int, [P(hs_pool_desc), P(hs_meta_layout)]),
            "hs_pool_create": (ctypes.c_int, [P(hs_pool_desc), vp, P(vp)]),
            "hs_pool_reset": (ctypes.c_int, [vp, vp]),
            "hs_step_begin": (ctypes.c_int, [vp, vp]),
            "hs_step_begin_fused": (ctypes.c_int, [vp]),
            "hs_resolve": (ctypes.c_int, [vp, i32, i32, vp, i32, vp, vp]),
            "hs_prefetch": (ctypes.c_int, [vp, i32, i32, vp, i32, vp]),
            "hs_resolve_ids": (ctypes.c_int, [vp, i32, i32, vp, vp, i32, vp, vp]),
            "hs_prefetch_ids": (ctypes.c_int, [vp, i32, i32, vp, vp, i32, vp]),
            "hs_gather": (ctypes.c_int, [vp, i32, i32, vp, i32, vp, vp]),
            "hs_resolve_shared": (ctypes.c_int, [vp, i32, i32, i32, vp, i32, vp, vp]),
            "hs_resolve_tiered": (ctypes.c_int, [vp, i32, i32, vp, i32, vp, ctypes.c_int64, vp, vp]),
            "hs_gather_history": (ctypes.c_int, [vp, i32, i32, vp, i32, vp, vp]),
            "hs_mla_decode": (ctypes.c_int, [vp, i32, i32, vp, vp, i32, vp, ctypes.c_int64, ctypes.c_float, vp, vp,
                                             vp]),
            "hs_mla_decode_history": (ctypes.c_int, [vp, i32, i32, vp, vp, i32, ctypes.c_float, vp, vp, vp]),
            "hs_get_error": (ctypes.c_int, [vp, P(i32), i32]),
            "hs_get_counters": (ctypes.c_int, [vp, i32, P(ctypes.c_uint64)]),
            "hs_pool_destroy": (ctypes.c_int, [vp]),
            "hs_host_alloc": (ctypes.c_int, [sz, P(vp)]),
            "hs_host_free": (ctypes.c_int, [vp]),
            "hs_error_string": (ctypes.c_char_p, [ctypes.c_int]),
            "hs_probe_link": (ctypes.c_int, [vp, vp, sz, i32, vp, P(ctypes.c_double), P(ctypes.c_double)]),
            "hs_probe_launch": (ctypes.c_int, [vp, i32, i32, i32, i32, vp]),
            "hs_probe_link_static": (ctypes.c_int, [vp, sz, i32, vp, P(ctypes.c_double), P(ctypes.c_double)]),
            "hs_debug_attention": (ctypes.c_int, [ctypes.c_uint32, i32, P(i32)]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int, what: str) -> None:
    if rc != HS_OK:
        raise HsError(rc, what)


def hs_probe_link(host_ptr: int, dev, nbytes: int, iters: int = 5, stream=None) -> tuple:
    """(zero-copy SM read GB/s, cudaMemcpyAsync H2D GB/s) over `nbytes` of mapped host memory."""
    zc, cp = ctypes.c_double(), ctypes.c_double()
    _check(load().hs_probe_link(host_ptr, _addr(dev), nbytes, iters, _stream(stream), ctypes.byref(zc),
                                ctypes.byref(cp)), "hs_probe_link")
    return zc.value, cp.value


def hs_probe_link_static(host_ptr: int, nbytes: int, iters: int = 5, stream=None) -> tuple:
    """(zero-copy SM read GB/s, cudaMemcpyAsync H2D GB/s) with the library's own fixed device scratch (at most
    16 MiB); for callers that have no device allocator."""
    zc, cp = ctypes.c_double(), ctypes.c_double()
    _check(load().hs_probe_link_static(host_ptr, nbytes, iters, _stream(stream), ctypes.byref(zc), ctypes.byref(cp)),
           "hs_probe_link_static")
    return zc.value, cp.value


def hs_probe_launch(pool: int, layer: int, nlayers: int, batch: int, k: int, stream=None) -> None:
    _check(load().hs_probe_launch(pool, layer, nlayers, batch, k, _stream(stream)), "hs_probe_launch")


def hs_debug_attention(wait_limit: int = 0, stall: bool = False) -> int:
    """Test hook: set the attention kernel's wait limit (0 = default) and stall switch; returns the largest batch
    whose keys are split over two CTA pairs on the current device."""
    n = ctypes.c_int32()
    _check(load().hs_debug_attention(wait_limit, int(bool(stall)), ctypes.byref(n)), "hs_debug_attention")
    return int(n.value)


def hs_error_string(code: int) -> str:
    return load().hs_error_string(code).decode()


def hs_meta_bytes(desc: hs_pool_desc) -> int:
    return int(load().hs_meta_bytes(ctypes.byref(desc)))


def hs_get_meta_layout(desc: hs_pool_desc) -> dict:
    lay = hs_meta_layout()
    _check(load().hs_get_meta_layout(ctypes.byref(desc), ctypes.byref(lay)), "hs_get_meta_layout")
    return {n: int(getattr(lay, n)) for n, _ in hs_meta_layout._fields_}


def hs_pool_create(desc: hs_pool_desc, stream=None) -> int:
    h = ctypes.c_void_p()
    _check(load().hs_pool_create(ctypes.byref(desc), _stream(stream), ctypes.byref(h)), "hs_pool_create")
    return h.value


def hs_pool_reset(pool: int, stream=None) -> None:
    _check(load().hs_pool_reset(pool, _stream(stream)), "hs_pool_reset")


def hs_step_begin(pool: int, stream=None) -> None:
    _check(load().hs_step_begin(pool, _stream(stream)), "hs_step_begin")


def hs_step_begin_fused(pool: int) -> None:
    _check(load().hs_step_begin_fused(pool), "hs_step_begin_fused")


def hs_resolve(pool: int, layer: int, batch: int, topk_idx, k: int, out_slots, stream=None) -> None:
    _check(load().hs_resolve(pool, layer, batch, _addr(topk_idx), k, _addr(out_slots), _stream(stream)),
           "hs_resolve")


def hs_prefetch(pool: int, layer: int, batch: int, topk_idx, k: int, stream=None) -> None:
    _check(load().hs_prefetch(pool, layer, batch, _addr(topk_idx), k, _stream(stream)), "hs_prefetch")


def hs_resolve_ids(pool: int, layer: int, batch: int, req_ids, topk_idx, k: int, out_slots, stream=None) -> None:
    _check(load().hs_resolve_ids(pool, layer, batch, _addr(req_ids), _addr(topk_idx), k, _addr(out_slots),
                                 _stream(stream)), "hs_resolve_ids")


def hs_prefetch_ids(pool: int, layer: int, batch: int, req_ids, topk_idx, k: int, stream=None) -> None:
    _check(load().hs_prefetch_ids(pool, layer, batch, _addr(req_ids), _addr(topk_idx), k, _stream(stream)),
           "hs_prefetch_ids")


def hs_resolve_shared(pool: int, layer0: int, nlayers: int, batch: int, topk_idx, k: int, out_slots,
                      stream=None) -> None:
    _check(load().hs_resolve_shared(pool, layer0, nlayers, batch, _addr(topk_idx), k, _addr(out_slots),
                                    _stream(stream)), "hs_resolve_shared")


def hs_resolve_tiered(pool: int, layer: int, batch: int, topk_idx, k: int, resident_row, resident_stride: int,
                      out_slots, stream=None) -> None:
    _check(load().hs_resolve_tiered(pool, layer, batch, _addr(topk_idx), k, _addr(resident_row), resident_stride,
                                    _addr(out_slots), _stream(stream)), "hs_resolve_tiered")


def hs_gather(pool: int, layer: int, batch: int, out_slots, k: int, dst, stream=None) -> None:
    _check(load().hs_gather(pool, layer, batch, _addr(out_slots), k, _addr(dst), _stream(stream)), "hs_gather")


def hs_mla_decode(pool: int, layer: int, batch: int, q, out_slots, k: int, resident_rows, resident_count: int,
                  sm_scale: float, out, lse, stream=None) -> None:
    _check(load().hs_mla_decode(pool, layer, batch, _addr(q), _addr(out_slots), k, _addr(resident_rows),
                                resident_count, sm_scale, _addr(out), _addr(lse), _stream(stream)), "hs_mla_decode")


def hs_mla_decode_history(pool: int, layer: int, batch: int, q, topk_idx, k: int, sm_scale: float, out, lse,
                          stream=None) -> None:
    _check(load().hs_mla_decode_history(pool, layer, batch, _addr(q), _addr(topk_idx), k, sm_scale, _addr(out),
                                        _addr(lse), _stream(stream)), "hs_mla_decode_history")


def hs_gather_history(pool: int, layer: int, batch: int, topk_idx, k: int, dst, stream=None) -> None:
    _check(load().hs_gather_history(pool, layer, batch, _addr(topk_idx), k, _addr(dst), _stream(stream)),
           "hs_gather_history")


def hs_get_error(pool: int, clear: bool = False) -> int:
    v = ctypes.c_int32()
    _check(load().hs_get_error(pool, ctypes.byref(v), int(clear)), "hs_get_error")
    return int(v.value)


def hs_get_counters(pool: int, layer: int) -> list:
    arr = (ctypes.c_uint64 * 4)()
    _check(load().hs_get_counters(pool, layer, arr), "hs_get_counters")
    return [int(x) for x in arr]


def hs_pool_destroy(pool: int) -> None:
    _check(load().hs_pool_destroy(pool), "hs_pool_destroy")


def hs_host_alloc(nbytes: int) -> int:
    p = ctypes.c_void_p()
    _check(load().hs_host_alloc(nbytes, ctypes.byref(p)), "hs_host_alloc")
    return p.value


def hs_host_free(ptr: int) -> None:
    _check(load().hs_host_free(ptr), "hs_host_free")


class HostBuffer:
    """Page-locked, device-mapped host memory from hs_host_alloc, freed on close()."""

    def __init__(self, nbytes: int):
        self.nbytes = nbytes
        self.ptr = hs_host_alloc(nbytes)

    def numpy(self):
        import numpy as np

        return np.ctypeslib.as_array((ctypes.c_uint8 * self.nbytes).from_address(self.ptr))

    def close(self):
        if self.ptr:
            hs_host_free(self.ptr)
            self.ptr = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class PoolBuffers:
    """Caller-side memory for one pool, allocated with torch (device) and hs_host_alloc (host), plus the handle.

    ``host_layers`` host-pool layers are allocated; with fewer than ``layers`` the pool's layer stride is 0 only
    when host_layers == 1 (all layers read one pool). ``layer_shift_rows`` S > 0 (with host_layers == 1) makes the
    layer stride S rows instead: the pool grows by (layers - 1) * S rows and layer l reads token t of request b from
    flat row b * ctx + t + l * S, so layers that select the same tokens read different rows. ``noio`` keeps a
    device copy of the host pool and selects the no-IO source. Views of the metadata arrays are exposed as torch
    tensors for inspection.
    """

    def __init__(self, layers, max_batch, ctx, slots, topk_max, row_bytes, host_layers=None, noio=False,
                 host: HostBuffer | None = None, stream=None, layer_shift_rows: int = 0):
        import torch

        self.layers, self.max_batch, self.ctx, self.slots = layers, max_batch, ctx, slots
        self.topk_max, self.row_bytes = topk_max, row_bytes
        self.host_layers = layers if host_layers is None else host_layers
        if self.host_layers not in (1, layers):
            raise ValueError("host_layers must be 1 (shared pool) or equal to layers")
        if layer_shift_rows < 0 or (layer_shift_rows and self.host_layers != 1):
            raise ValueError("layer_shift_rows applies to a shared host pool only")
        self.layer_shift_rows = layer_shift_rows if layers > 1 else 0
        per_layer = max_batch * ctx * row_bytes
        self.extra_rows = (layers - 1) * self.layer_shift_rows
        host_bytes = self.host_layers * per_layer + self.extra_rows * row_bytes
        self.host = host if host is not None else HostBuffer(host_bytes)
        self.hot = torch.zeros(layers * max_batch * slots * row_bytes, dtype=torch.uint8, device="cuda")
        self.noio_src = None
        if noio:
            self.noio_src = torch.empty(host_bytes, dtype=torch.uint8, device="cuda")
        layer_stride = per_layer if self.host_layers == layers else self.layer_shift_rows * row_bytes
        self.desc = hs_pool_desc(layers, max_batch, ctx, slots, topk_max, row_bytes, self.host.ptr, layer_stride, 0,
                                 self.hot.data_ptr(), None, None)
        nbytes = hs_meta_bytes(self.desc)
        if nbytes == 0:
            raise HsError(HS_ERR_INVALID_ARG, "hs_meta_bytes")
        self.meta = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.desc.meta = self.meta.data_ptr()
        self.layout = hs_get_meta_layout(self.desc)
        self.handle = None
        self._stream = stream

    def upload_noio(self):
        """Copy the host pool into the no-IO device source (call after filling the host pool)."""
        import torch

        if self.noio_src is None:
            raise ValueError("pool was not created with noio=True")
        src = torch.frombuffer(self.host.numpy(), dtype=torch.uint8)
        self.noio_src.copy_(src)
        self.desc.noio_src = self.noio_src.data_ptr()

    def create(self):
        self.handle = hs_pool_create(self.desc, self._stream)
        return self.handle

    def view(self, name):
        """torch view of a metadata array: step, error (int32 scalar), counters [layers][4] (int64 bit pattern),
        tok2slot [layers][max_batch][ctx], slot_tok / slot_stamp [layers][max_batch][slots]."""
        import torch

        off = self.layout[name]
        L, B = self.layers, self.max_batch
        if name in ("step", "error"):
            return self.meta[off:off + 4].view(torch.int32)
        if name == "counters":
            return self.meta[off:off + 32 * L].view(torch.int64).view(L, 4)
        n = self.ctx if name == "tok2slot" else self.slots
        return self.meta[off:off + 4 * L * B * n].view(torch.int32).view(L, B, n)

    def hot_view(self):
        return self.hot.view(self.layers, self.max_batch, self.slots, self.row_bytes)

    def close(self):
        if self.handle:
            hs_pool_destroy(self.handle)
            self.handle = None
