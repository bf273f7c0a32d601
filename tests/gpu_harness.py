"""Helpers for the GPU parity tests: run a workload through the C ABI and the CPU oracle side by side."""
from __future__ import annotations

import numpy as np
import torch

import hierarchical_sparse_attention_hs_gb300 as hs
import oracle
import workload as wl


def make_pool(w: wl.Workload, host_layers: int = 1, noio: bool = False, max_batch: int | None = None,
              layer_shift_rows: int = 0):
    buf = hs.PoolBuffers(w.layers, max_batch or w.requests, w.ctx, w.slots, w.topk, w.row_bytes,
                         host_layers=host_layers, noio=noio, layer_shift_rows=layer_shift_rows)
    wl.fill_host_pool(w, buf.host.ptr, buf.host_layers, extra_rows=buf.extra_rows)
    if noio:
        buf.upload_noio()
    buf.create()
    return buf


def host_rows(buf) -> np.ndarray:
    n = buf.host_layers * buf.max_batch * buf.ctx * buf.row_bytes
    return buf.host.numpy()[:n].reshape(buf.host_layers, buf.max_batch, buf.ctx, buf.row_bytes)


def layer_rows(buf, l: int, b: int) -> np.ndarray:
    """The ctx host rows layer l of request b reads: its own pool layer, the shared pool, or the shared pool
    from row l * layer_shift_rows on."""
    if buf.host_layers == buf.layers:
        return host_rows(buf)[l, b]
    flat = buf.host.numpy().reshape(-1, buf.row_bytes)
    start = b * buf.ctx + l * buf.layer_shift_rows
    return flat[start:start + buf.ctx]


def check_hot_rows(buf, layers=None) -> None:
    """Hot-buffer bytes equal the oracle's: occupied slot v holds host row slot_tok[v], empty slots are zero.

    (The oracle's own hot buffer satisfies exactly this, pinned by invariant I2; slot_tok is compared with the
    oracle separately.)"""
    st_all = buf.view("slot_tok").cpu().numpy()
    for l in (range(buf.layers) if layers is None else layers):
        hot = buf.hot_view()[l].cpu().numpy()
        for b in range(buf.max_batch):
            st = st_all[l, b]
            occ = st >= 0
            assert np.array_equal(hot[b][occ], layer_rows(buf, l, b)[st[occ]]), (l, b)
            assert not hot[b][~occ].any(), (l, b)


def compare_state(buf, ora: oracle.OraclePool, tag="") -> None:
    for name, ref in (("tok2slot", ora.tok2slot), ("slot_tok", ora.slot_tok), ("slot_stamp", ora.slot_stamp)):
        got = buf.view(name).cpu().numpy()
        if not np.array_equal(got, ref):
            bad = np.argwhere(got != ref)
            raise AssertionError(f"{tag} {name} differs at {bad[:5].tolist()} ({len(bad)} entries)")
    cnt = buf.view("counters").cpu().numpy().astype(np.uint64)
    assert np.array_equal(cnt, ora.counters), f"{tag} counters {cnt.tolist()} vs {ora.counters.tolist()}"


def replay(w: wl.Workload, steps: int | None = None, host_layers: int = 1, noio: bool = False,
           prefetch: bool = False, graphs: bool = False, mid_check: bool = True, shared_call: bool = False,
           depth: int = 0, fused: bool = False, layer_shift_rows: int = 0):
    """Run `steps` decode steps of workload w on the GPU and in the oracle; compare out_slots after every step
    and the whole state at the midpoint and at the end. Returns (buf, oracle pool)."""
    ns = w.steps if steps is None else steps
    sel = wl.gen_selections(w, steps=ns)  # [ns][selection layers][B][k]
    buf = make_pool(w, host_layers=host_layers, noio=noio, layer_shift_rows=layer_shift_rows)
    pool = buf.handle
    L, B, k = w.layers, w.requests, w.topk
    ora = oracle.OraclePool(w.ctx, w.slots, w.row_bytes, L, B, track_rows=False)
    topk_all = torch.from_numpy(sel).cuda()
    out = torch.full((L, B, k), -7, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    s0 = torch.cuda.Stream()  # a non-default stream, so the same code can be captured into a graph
    s1 = torch.cuda.Stream() if prefetch else None
    sides = [torch.cuda.Stream() for _ in range(depth)]

    def lsel(l):
        return 0 if w.shared_across_layers else l

    def enqueue(s):
        if fused:
            hs.hs_step_begin_fused(pool)  # carried by the first resolve below
        else:
            hs.hs_step_begin(pool, s0)
        if shared_call:
            # one call resolves every layer; all layers' out_slots are the same, written once
            hs.hs_resolve_shared(pool, 0, L, B, topk_all[s, 0], k, out[0], s0)
            for l in range(1, L):
                out[l].copy_(out[0])
            return
        if not prefetch:
            for l in range(L):
                hs.hs_resolve(pool, l, B, topk_all[s, lsel(l)], k, out[l], s0)
            return
        if depth:
            # layer-wise, `depth` layers ahead on `depth` side streams: when layer l starts on s0, layer l + depth
            # is prefetched (at layer 0, layers 1 .. depth); layer l's resolve waits for its own prefetch
            done = [None] * L
            for l in range(L):
                if done[l] is not None:
                    s0.wait_event(done[l])
                ahead = range(1, min(depth, L - 1) + 1) if l == 0 else ([l + depth] if l + depth < L else [])
                if ahead:
                    started = torch.cuda.Event()
                    started.record(s0)
                    for j in ahead:
                        side = sides[j % depth]
                        side.wait_event(started)
                        hs.hs_prefetch(pool, j, B, topk_all[s, lsel(j)], k, side)
                        done[j] = torch.cuda.Event()
                        done[j].record(side)
                hs.hs_resolve(pool, l, B, topk_all[s, lsel(l)], k, out[l], s0)
            return
        # layer-wise prefetch: layer l+1 is resolved ahead on s1 while layer l is resolved on s0
        ev_begin = torch.cuda.Event()
        ev_begin.record(s0)
        s1.wait_event(ev_begin)
        evs = [None] * L
        for l in range(1, L):
            hs.hs_prefetch(pool, l, B, topk_all[s, lsel(l)], k, s1)
            evs[l] = torch.cuda.Event()
            evs[l].record(s1)
        for l in range(L):
            if evs[l] is not None:
                s0.wait_event(evs[l])
            hs.hs_resolve(pool, l, B, topk_all[s, lsel(l)], k, out[l], s0)
        ev_end = torch.cuda.Event()
        ev_end.record(s1)
        s0.wait_event(ev_end)

    graph_list = []
    if graphs:
        # one graph per decode step (its selection pointers differ); captured up front, replayed in order
        for s in range(ns):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s0):
                enqueue(s)
            graph_list.append(g)
        torch.cuda.synchronize()

    for s in range(ns):
        with torch.cuda.stream(s0):
            if graphs:
                graph_list[s].replay()
            else:
                enqueue(s)
        s0.synchronize()
        ora.step_begin()
        if prefetch:
            # the oracle makes the same calls: counters count every call, so a resolve after a prefetch adds
            # its (all-hit) lookups; the state equals a lone resolve's (pinned on the CPU)
            for l in range(1, L):
                ora.resolve(l, sel[s, lsel(l)], None, want_slots=False)
        for l in range(L):
            expect = ora.resolve(l, sel[s, lsel(l)], None)
            got = out[l].cpu().numpy()
            if not np.array_equal(got, expect):
                bad = np.argwhere(got != expect)
                raise AssertionError(f"{w.name} step {s} layer {l}: out_slots differ at {bad[:5].tolist()}")
        if mid_check and s == ns // 2:
            compare_state(buf, ora, f"{w.name} step {s}")
    torch.cuda.synchronize()
    compare_state(buf, ora, f"{w.name} end")
    assert hs.hs_get_error(buf.handle) == 0
    return buf, ora
