"""Invariants I1-I6 of the oracle after every call, replaying the synthetic workloads (sampled request-layers
for the large ones) with host rows tracked byte for byte."""
import numpy as np
import pytest

import oracle
import pins
import workload as wl

# (workload, layers sampled, requests sampled, steps replayed)
CASES = [
    ("tiny", (0, 1), (0, 1), None),
    ("dsa", (0, 1), (5, 2), 12),
    ("multilayer", (17, 1), (3, 1), 10),   # covers the churn step 8
    ("quest", (4, 1), (2, 2), 24),
    ("shared", (0, 1), (6, 1), 6),
]


@pytest.mark.parametrize("name,layers,reqs,steps", CASES, ids=[c[0] for c in CASES])
def test_invariants_hold_after_every_call(name, layers, reqs, steps):
    w = wl.WORKLOADS[name]
    ns = w.steps if steps is None else steps
    sel_layer = (0, 1) if w.shared_across_layers else layers
    sel = wl.gen_selections(w, layers=sel_layer, requests=reqs, steps=ns)
    host = np.stack([wl.rows(w, layers[0], reqs[0] + b) for b in range(reqs[1])])
    pool = oracle.OraclePool(w.ctx, w.slots, w.row_bytes, 1, reqs[1], track_rows=True)
    for s in range(ns):
        pool.step_begin()
        before = [(pool.slot_tok[0, b].copy(), pool.hot[0, b].copy()) for b in range(reqs[1])]
        c0 = pool.counters[0].copy()
        out = pool.resolve(0, sel[s, 0], host)
        d = pool.counters[0] - c0
        assert int(d[3]) == int(d[1]) * w.row_bytes
        assert int(d[0] + d[1]) == np.count_nonzero(sel[s, 0] >= 0)
        for b in range(reqs[1]):
            # per-request miss count: selected tokens that no slot held before the call
            valid = sel[s, 0, b][sel[s, 0, b] >= 0]
            misses = int(np.count_nonzero(~np.isin(valid, before[b][0])))
            pins.check_invariants(pool, 0, b, sel[s, 0, b], out[b], host[b], pool.step, before[b], misses)
    assert pool.error == 0


@pytest.mark.parametrize("same", [True, False])
def test_prefetch_then_resolve_equals_resolve_alone(same):
    """Exact layer-wise prefetch (HiSparse paper, Abstract): prefetch(l) then resolve(l) in the same step leaves
    the state and out_slots of a lone resolve(l). With a different selection in the resolve (same=False) the
    second call is an ordinary resolve at the same step, which the brute-force pin covers; here it only has
    to keep the invariants."""
    w = wl.WORKLOADS["shared"]
    sel = wl.gen_selections(w, requests=(0, 2), steps=6)[:, 0]
    other = wl.gen_selections(wl.WORKLOADS["dsa"], requests=(0, 2), steps=6)[:, 0] % w.ctx
    host = np.stack([wl.rows(w, 0, b) for b in range(2)])
    lone = oracle.OraclePool(w.ctx, w.slots, w.row_bytes, 1, 2)
    pre = oracle.OraclePool(w.ctx, w.slots, w.row_bytes, 1, 2)
    for s in range(6):
        lone.step_begin()
        pre.step_begin()
        target = sel[s] if same else other[s]
        out_lone = lone.resolve(0, target, host)
        assert pre.resolve(0, sel[s], host, want_slots=False) is None
        before = [(pre.slot_tok[0, b].copy(), pre.hot[0, b].copy()) for b in range(2)]
        m0 = pre.counters[0, 1]
        out_pre = pre.resolve(0, target, host)
        if same:
            assert pre.counters[0, 1] == m0  # everything was resident
            assert np.array_equal(out_pre, out_lone)
            for name in ("tok2slot", "slot_tok", "slot_stamp", "hot"):
                assert np.array_equal(getattr(pre, name), getattr(lone, name)), name
        else:
            for b in range(2):
                valid = target[b][target[b] >= 0]
                misses = int(np.count_nonzero(~np.isin(valid, before[b][0])))
                pins.check_invariants(pre, 0, b, target[b], out_pre[b], host[b], pre.step, before[b], misses)
        if same:
            lone_hits = lone.counters[0, 0]
            assert pre.counters[0, 0] == lone_hits + (s + 1) * 2 * w.topk
