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
