"""Pins for the CPU oracle: checks that do not go through the oracle's own code.

Each pin raises AssertionError when the oracle under test disagrees with it. They are used twice: against the
real oracle (all must pass) and against deliberately broken copies of it (each copy must fail at least one), which
shows the pins can catch a plausible mistake anywhere in the oracle.

The policy being pinned is the per-layer resolution of "HiSparse: Scaling Sparse-Attention Decoding with
Hierarchical KV Cache Management" (Abstract): per layer, find which selected tokens are already cached, choose
least recently used victims for the rest and bring their rows over from the host, which moves KV rows without
changing what attention reads. The stated readings: stamp = decode step, oldest stamp first, ties to the lowest slot, misses paired with victims in
ascending token order, empties (stamp 0) first, rows with out-of-range or duplicate tokens rejected whole.
"""
from __future__ import annotations

import heapq
import itertools
import json
import os
from collections import OrderedDict

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _pool(lib, ctx, slots, row_bytes=16, n_layers=1, n_requests=1, track_rows=True):
    return oracle.OraclePool(ctx, slots, row_bytes, n_layers, n_requests, track_rows=track_rows, library=lib)


def _rows(ctx, row_bytes, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 256, size=(ctx, row_bytes), dtype=np.uint8)


# ---------------------------------------------------------------------------------------------------------------
# P1: brute force on tiny inputs. The victim set is found by exhaustive search over all subsets of the candidate
# slots: the unique size-m subset whose every key is smaller than every key outside it.
# ---------------------------------------------------------------------------------------------------------------
def brute_force_step(tok2slot, slot_tok, stamp, sel, step, resident=None):
    """Advance plain-Python state (lists) by one call; returns (out_slots, hits, misses, evictions, fills).
    With a resident map, a token outside the hot buffer but held in the HBM pool is served in place (counted as a
    hit, out_slot -2 - row, no slot, no stamp)."""
    sel = [int(t) for t in sel]
    valid = [t for t in sel if t >= 0]
    hit_slots = set()
    misses = []
    inplace = 0
    for t in valid:
        if tok2slot[t] >= 0:
            hit_slots.add(tok2slot[t])
        elif resident is not None and resident[t] >= 0:
            inplace += 1
        else:
            misses.append(t)
    for v in hit_slots:
        stamp[v] = step
    misses.sort()
    cands = [v for v in range(len(slot_tok)) if v not in hit_slots]
    key = {v: (stamp[v], v) for v in cands}
    m = len(misses)
    chosen = None
    for sub in itertools.combinations(cands, m):
        inside = set(sub)
        if all(key[a] < key[b] for a in sub for b in cands if b not in inside):
            assert chosen is None, "victim set must be unique"
            chosen = sub
    assert chosen is not None
    victims = sorted(chosen, key=lambda v: key[v])
    evictions = 0
    fills = []
    for t, v in zip(misses, victims):
        u = slot_tok[v]
        if u >= 0:
            tok2slot[u] = -1
            evictions += 1
        tok2slot[t] = v
        slot_tok[v] = t
        stamp[v] = step
        fills.append((t, v))
    out = [tok2slot[t] if t >= 0 else -1 for t in sel]
    if resident is not None:
        out = [(-2 - int(resident[t])) if (t >= 0 and o < 0) else o for t, o in zip(sel, out)]
    return out, len(valid) - m, m, evictions, fills


def pin_brute_force(lib, n_traces=300, seed=1):
    rng = np.random.default_rng(seed)
    for trace in range(n_traces):
        ctx = int(rng.integers(4, 17))
        slots = int(rng.integers(1, 9))
        R = 8
        rows = _rows(ctx, R, 1000 + trace)
        pool = _pool(lib, ctx, slots, R)
        t2s = [-1] * ctx
        s2t = [-1] * slots
        st = [0] * slots
        hot = [bytes(R)] * slots
        cnt = np.zeros(4, dtype=np.uint64)
        step = 0
        for call in range(int(rng.integers(2, 14))):
            # most calls open a new decode step; some repeat the step (a second call on the same layer in one
            # step, as a prefetch followed by a resolve with a different selection does)
            if call == 0 or rng.random() < 0.75:
                pool.step_begin()
                step += 1
            k = int(rng.integers(1, min(slots, ctx) + 1))
            sel = rng.choice(ctx, size=k, replace=False).astype(np.int32)
            if k > 1 and rng.random() < 0.2:
                sel[int(rng.integers(0, k))] = -1  # padding entry
            out_o = pool.resolve(0, sel[None, :], rows[None])
            out_b, h, m, e, fills = brute_force_step(t2s, s2t, st, sel, step)
            for t, v in fills:
                hot[v] = rows[t].tobytes()
            cnt += np.array([h, m, e, m * R], dtype=np.uint64)
            assert out_o[0].tolist() == out_b, (trace, call)
            assert pool.tok2slot[0, 0].tolist() == t2s, (trace, call)
            assert pool.slot_tok[0, 0].tolist() == s2t, (trace, call)
            assert pool.slot_stamp[0, 0].tolist() == st, (trace, call)
            assert all(pool.hot[0, 0, v].tobytes() == hot[v] for v in range(slots)), (trace, call)
            assert pool.counters[0].tolist() == cnt.tolist(), (trace, call)


def pin_brute_force_tiered(lib, n_traces=200, seed=11):
    """The three-tier variant against the brute force, with a fresh random resident map for every call."""
    rng = np.random.default_rng(seed)
    for trace in range(n_traces):
        ctx = int(rng.integers(4, 17))
        slots = int(rng.integers(1, 9))
        R = 8
        rows = _rows(ctx, R, 5000 + trace)
        pool = _pool(lib, ctx, slots, R)
        t2s, s2t, st = [-1] * ctx, [-1] * slots, [0] * slots
        hot = [bytes(R)] * slots
        cnt = np.zeros(4, dtype=np.uint64)
        step = 0
        for call in range(int(rng.integers(2, 14))):
            if call == 0 or rng.random() < 0.75:
                pool.step_begin()
                step += 1
            k = int(rng.integers(1, min(slots, ctx) + 1))
            sel = rng.choice(ctx, size=k, replace=False).astype(np.int32)
            resident = np.where(rng.random(ctx) < 0.4, rng.integers(0, 1000, size=ctx), -1).astype(np.int32)
            out_o = pool.resolve(0, sel[None, :], rows[None], resident=resident[None, :])
            out_b, h, m, e, fills = brute_force_step(t2s, s2t, st, sel, step, resident)
            for t, v in fills:
                hot[v] = rows[t].tobytes()
            cnt += np.array([h, m, e, m * R], dtype=np.uint64)
            assert out_o[0].tolist() == out_b, (trace, call)
            assert pool.tok2slot[0, 0].tolist() == t2s, (trace, call)
            assert pool.slot_tok[0, 0].tolist() == s2t, (trace, call)
            assert pool.slot_stamp[0, 0].tolist() == st, (trace, call)
            assert all(pool.hot[0, 0, v].tobytes() == hot[v] for v in range(slots)), (trace, call)
            assert pool.counters[0].tolist() == cnt.tolist(), (trace, call)


def pin_tiered_all_resident(lib, seed=12):
    """Closed form: when every selected token outside the hot buffer is held in the HBM pool, nothing is
    fetched, no slot changes, and each such entry reports -2 - its pool row."""
    rng = np.random.default_rng(seed)
    ctx, slots, R = 500, 40, 8
    rows = _rows(ctx, R, 9)
    pool = _pool(lib, ctx, slots, R)
    first = rng.choice(ctx, size=30, replace=False).astype(np.int32)
    pool.step_begin()
    pool.resolve(0, first[None, :], rows[None])
    snap = (pool.tok2slot.copy(), pool.slot_tok.copy(), pool.slot_stamp.copy(), pool.hot.copy())
    resident = np.arange(ctx, dtype=np.int32) * 3 + 1
    sel = np.setdiff1d(rng.choice(ctx, size=60, replace=False), first)[:25].astype(np.int32)
    c0 = pool.counters[0].copy()
    pool.step_begin()
    out = pool.resolve(0, sel[None, :], rows[None], resident=resident[None, :])
    assert out[0].tolist() == (-2 - resident[sel]).tolist()
    for a, b in zip(snap, (pool.tok2slot, pool.slot_tok, pool.slot_stamp, pool.hot)):
        assert np.array_equal(a, b)
    assert (pool.counters[0] - c0).tolist() == [len(sel), 0, 0, 0]
    # a hot-buffer copy takes precedence over the resident one, and is re-stamped
    both = first[:5]
    pool.step_begin()
    out = pool.resolve(0, both[None, :], rows[None], resident=resident[None, :])
    assert np.array_equal(out[0], pool.tok2slot[0, 0][both])
    assert np.all(pool.slot_stamp[0, 0][out[0]] == pool.step)


# ---------------------------------------------------------------------------------------------------------------
# P2: with one selection per step the policy is textbook LRU (capacity = slots), empty slots taken lowest first.
# ---------------------------------------------------------------------------------------------------------------
class TextbookLRU:
    def __init__(self, capacity):
        self.od = OrderedDict()  # token -> slot, least recently used first
        self.free = list(range(capacity))
        heapq.heapify(self.free)

    def access(self, t):
        if t in self.od:
            self.od.move_to_end(t)
            return True, self.od[t]
        if self.free:
            slot = heapq.heappop(self.free)
        else:
            _, slot = self.od.popitem(last=False)
        self.od[t] = slot
        return False, slot


def pin_textbook_lru(lib, seed=2):
    rng = np.random.default_rng(seed)
    for ctx, slots, steps in [(64, 8, 3000), (200, 37, 3000), (16, 16, 500), (1000, 1, 300)]:
        pool = _pool(lib, ctx, slots, 8, track_rows=False)
        lru = TextbookLRU(slots)
        # a skewed trace so that both hits and evictions are frequent
        hot_set = rng.choice(ctx, size=min(ctx, 2 * slots), replace=False)
        for _ in range(steps):
            t = int(hot_set[rng.integers(0, len(hot_set))]) if rng.random() < 0.7 else int(rng.integers(0, ctx))
            before = pool.counters[0, 0]
            pool.step_begin()
            out = pool.resolve(0, np.array([[t]], dtype=np.int32))
            hit, slot = lru.access(t)
            assert bool(pool.counters[0, 0] - before) == hit
            assert int(out[0, 0]) == slot
        resident = {int(tk): int(s) for tk, s in lru.od.items()}
        t2s = pool.tok2slot[0, 0]
        assert {int(tk): int(t2s[tk]) for tk in np.nonzero(t2s >= 0)[0]} == resident


# ---------------------------------------------------------------------------------------------------------------
# P3: no eviction possible (slots >= ctx): token t sits in the slot numbered by its first appearance in the global
# fill order (ascending tokens within each step); its stamp is the last step that selected it.
# ---------------------------------------------------------------------------------------------------------------
def pin_no_eviction_closed_form(lib, seed=3):
    rng = np.random.default_rng(seed)
    for ctx, slots, k, steps in [(50, 50, 7, 20), (40, 64, 12, 15), (300, 300, 33, 30)]:
        pool = _pool(lib, ctx, slots, 8, track_rows=False)
        seen = []
        last = {}
        for s in range(1, steps + 1):
            sel = rng.choice(ctx, size=k, replace=False).astype(np.int32)
            new = sorted(set(sel.tolist()) - set(seen))
            seen.extend(new)
            for t in sel.tolist():
                last[t] = s
            before = pool.counters[0].copy()
            pool.step_begin()
            pool.resolve(0, sel[None, :])
            assert int(pool.counters[0, 1] - before[1]) == len(new)
            assert int(pool.counters[0, 2]) == 0
        expect = np.full(ctx, -1, dtype=np.int32)
        expect[np.array(seen, dtype=np.int64)] = np.arange(len(seen), dtype=np.int32)
        assert np.array_equal(pool.tok2slot[0, 0], expect)
        stamps = np.zeros(slots, dtype=np.int32)
        for t, s in last.items():
            stamps[seen.index(t)] = s
        assert np.array_equal(pool.slot_stamp[0, 0], stamps)


# ---------------------------------------------------------------------------------------------------------------
# P4: full churn (slots == k, consecutive selections disjoint): every call misses and evicts everything, and the
# slots hold the selection in ascending token order.
# ---------------------------------------------------------------------------------------------------------------
def pin_churn_closed_form(lib, seed=4):
    rng = np.random.default_rng(seed)
    for ctx, k, steps in [(64, 8, 12), (1000, 100, 10)]:
        R = 8
        rows = _rows(ctx, R, seed + ctx)
        pool = _pool(lib, ctx, k, R)
        prev = set()
        for s in range(1, steps + 1):
            pool_choices = np.array(sorted(set(range(ctx)) - prev))
            sel = rng.choice(pool_choices, size=k, replace=False).astype(np.int32)
            before = pool.counters[0].copy()
            pool.step_begin()
            out = pool.resolve(0, sel[None, :], rows[None])
            d = pool.counters[0] - before
            assert d.tolist() == [0, k, k if s > 1 else 0, k * R]
            order = np.sort(sel)
            assert np.array_equal(pool.slot_tok[0, 0], order)
            assert np.array_equal(out[0], np.searchsorted(order, sel))
            assert np.array_equal(pool.hot[0, 0], rows[order])
            assert np.all(pool.slot_stamp[0, 0] == s)
            prev = set(sel.tolist())


# ---------------------------------------------------------------------------------------------------------------
# Hand-worked trace, stored with its derivation under tests/golden/.
# ---------------------------------------------------------------------------------------------------------------
def pin_hand_trace(lib):
    with open(os.path.join(GOLDEN, "hand_trace_ctx8_slots3.json")) as f:
        g = json.load(f)
    pool = _pool(lib, g["ctx"], g["slots"], 8, track_rows=False)
    for st in g["steps"]:
        pool.step_begin()
        out = pool.resolve(0, np.array([st["sel"]], dtype=np.int32))
        assert out[0].tolist() == st["out_slots"], st
        assert pool.slot_tok[0, 0].tolist() == st["slot_tok"], st
        assert pool.slot_stamp[0, 0].tolist() == st["slot_stamp"], st
        assert int(pool.error) == st.get("error", 0), st
    assert pool.counters[0].tolist() == g["counters"]


# ---------------------------------------------------------------------------------------------------------------
# Rejected rows: out-of-range or duplicate tokens reject the whole row and change nothing.
# ---------------------------------------------------------------------------------------------------------------
def pin_rejection(lib):
    ctx, slots, R = 32, 6, 8
    rows = _rows(ctx, R, 7)
    pool = _pool(lib, ctx, slots, R)
    pool.step_begin()
    pool.resolve(0, np.array([[3, 9, 4]], dtype=np.int32), rows[None])
    snap = (pool.tok2slot.copy(), pool.slot_tok.copy(), pool.slot_stamp.copy(), pool.hot.copy(),
            pool.counters.copy())
    for bad, bit in [([5, 32, 1], oracle.ERR_RANGE), ([7, 3, 7], oracle.ERR_DUP), ([3, 3, -1], oracle.ERR_DUP),
                     ([40, 2, 2], oracle.ERR_RANGE | oracle.ERR_DUP)]:
        pool.step_begin()
        pool.error = 0
        out, rc = pool.resolve_one(0, 0, np.array(bad, dtype=np.int32), rows)
        assert rc == bit, (bad, rc)
        assert out.tolist() == [-1, -1, -1]
        for a, b in zip(snap, (pool.tok2slot, pool.slot_tok, pool.slot_stamp, pool.hot, pool.counters)):
            assert np.array_equal(a, b), bad
    # padding only: nothing happens, nothing is counted
    pool.step_begin()
    out, rc = pool.resolve_one(0, 0, np.array([-1, -5, -1], dtype=np.int32), rows)
    assert rc == 0 and out.tolist() == [-1, -1, -1]
    assert np.array_equal(snap[4], pool.counters)


# ---------------------------------------------------------------------------------------------------------------
# Invariants I1-I6 (checked after every call of a workload replay).
# ---------------------------------------------------------------------------------------------------------------
def check_invariants(pool, layer, req, sel, out, host_rows, step, before, misses):
    """I1-I6 for one request-layer after one call. `before` = (slot_tok, hot) copies taken before the call,
    `misses` = this call's miss count from the counters."""
    t2s = pool.tok2slot[layer, req]
    s2t = pool.slot_tok[layer, req]
    st = pool.slot_stamp[layer, req]
    sel = np.asarray(sel)
    valid = sel[sel >= 0]
    # I1: every selected token is resident, and out_slots points at it
    assert np.all(t2s[valid] >= 0)
    assert np.array_equal(out[sel >= 0], t2s[valid])
    assert np.all(out[sel < 0] == -1)
    # I4: residency <= slots and the two maps are mutual inverses
    res_t = np.nonzero(t2s >= 0)[0]
    res_s = np.nonzero(s2t >= 0)[0]
    assert len(res_t) == len(res_s) <= pool.slots
    assert np.array_equal(s2t[t2s[res_t]], res_t)
    assert np.array_equal(t2s[s2t[res_s]], res_s)
    # I6: stamps never exceed the step; the selected slots carry this step
    assert np.all(st <= step)
    assert np.all(st[out[sel >= 0]] == step)
    # I3: exactly `misses` slots were (re)filled, and they now hold selected tokens
    changed = np.nonzero(before[0] != s2t)[0]
    refilled = set(changed.tolist())
    if pool.hot is not None:
        hot = pool.hot[layer, req]
        row_changed = np.nonzero(np.any(before[1] != hot, axis=1))[0]
        refilled |= set(row_changed.tolist())
        # I2: every occupied slot holds its token's host row
        assert np.array_equal(hot[res_s], host_rows[s2t[res_s]])
        # I5: gathering through out_slots equals gathering the full host history by the selection
        assert np.array_equal(hot[out[sel >= 0]], host_rows[valid])
    assert len(refilled) <= misses
    assert np.all(np.isin(s2t[sorted(refilled)], valid))


ALL_PINS = [pin_hand_trace, pin_rejection, pin_brute_force, pin_textbook_lru, pin_no_eviction_closed_form,
            pin_churn_closed_form, pin_brute_force_tiered, pin_tiered_all_resident]
