"""The seeded input generators: published PRNG outputs and the stated properties of every selection stream."""
import numpy as np
import pytest

import workload as wl


def test_splitmix64_published_outputs():
    # splitmix64 (Vigna) seeded with 1234567: the first outputs of the reference C implementation
    assert wl.splitmix64_sequence(1234567, 5) == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                                                  4593380528125082431, 16408922859458223821]


def test_xoshiro256starstar_published_outputs():
    # xoshiro256** from state (1, 2, 3, 4). The first three follow by hand: s1*5=10, rotl(10,7)*9=11520; the
    # second output uses s1 = 2^2 = 0; the third rotl(262149*5, 7)*9 = 1509978240.
    got = wl.xoshiro_sequence((1, 2, 3, 4), 10).tolist()
    assert got[:3] == [11520, 0, 1509978240]
    assert got == [11520, 0, 1509978240, 1215971899390074240, 1216172134540287360, 607988272756665600,
                   16172922978634559625, 8476171486693032832, 10595114339597558777, 2904607092377533576]


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_selection_stream_properties(name):
    w = wl.WORKLOADS[name]
    nl = min(2, w.selection_layers)
    nr = min(3, w.requests)
    steps = min(w.steps, 30)
    sel = wl.gen_selections(w, layers=(0, nl), requests=(0, nr), steps=steps)
    assert sel.shape == (steps, nl, nr, w.topk)
    assert sel.min() >= 0 and sel.max() < w.ctx
    keep = (w.keep_pct * w.topk + 50) // 100
    for l in range(nl):
        for r in range(nr):
            rows = sel[:, l, r]
            for s in range(steps):
                assert len(np.unique(rows[s])) == w.topk  # no duplicates
                assert not np.all(np.diff(rows[s]) > 0)  # shuffled, not sorted
                if s:
                    ov = len(np.intersect1d(rows[s], rows[s - 1]))
                    assert ov == (0 if s in w.churn else keep)
    # deterministic, and a sub-range equals the same slice of a wider draw (independent streams)
    again = wl.gen_selections(w, layers=(0, nl), requests=(0, nr), steps=steps)
    assert np.array_equal(sel, again)
    if nr > 1:
        sub = wl.gen_selections(w, layers=(0, 1), requests=(1, 1), steps=steps)
        assert np.array_equal(sub[:, 0, 0], sel[:, 0, 1])


def test_zipf_recency_skew():
    # Zipf over recency ranks: the newest positions dominate the first draw of the dsa stream
    w = wl.WORKLOADS["dsa"]
    sel = wl.gen_selections(w, requests=(0, 4), steps=1)[0, 0]
    top = np.mean(sel >= w.ctx - 4096)
    assert top > 0.5  # ranks 1..4096 hold most of the mass for s = 1.1
    uni = wl.gen_selections(wl.WORKLOADS["multilayer"], layers=(0, 1), requests=(0, 4), steps=1)[0, 0]
    assert np.mean(uni >= wl.WORKLOADS["multilayer"].ctx - 4096) < 0.05


def test_host_rows_distinct_and_reproducible():
    w = wl.WORKLOADS["dsa"]
    a = wl.rows(w, 0, 3, 100, 50)
    b = wl.rows(w, 0, 3, 100, 50)
    assert np.array_equal(a, b)
    assert len({r.tobytes() for r in a}) == 50
    c = wl.rows(w, 0, 4, 100, 50)
    assert not np.any(np.all(a == c, axis=1))
    # tag word: (layer, request, token)
    tag = a[:, :8].copy().view(np.uint64)[:, 0]
    assert np.array_equal(tag & 0xFFFFFFFF, np.arange(100, 150))
    assert np.all((tag >> 32) & 0xFFFF == 3)


def test_tiny_rows_are_bf16_standard_normal():
    w = wl.WORKLOADS["tiny"]
    r = wl.rows(w, 0, 0)
    vals = (r.view(np.uint16).astype(np.uint32) << 16).view(np.float32)
    assert vals.shape == (w.ctx, w.row_bytes // 2)
    assert abs(vals.mean()) < 0.01 and abs(vals.std() - 1.0) < 0.01


def test_host_pool_extra_rows_continue_the_last_request():
    """A shared pool read with a per-layer shift reaches past its last request's rows: the extra rows are rows ctx,
    ctx + 1, ... of that request, written right after its row ctx - 1."""
    import dataclasses

    w = dataclasses.replace(wl.WORKLOADS["dsa"], requests=2, ctx=1024)
    extra = 37
    pool = np.zeros((w.requests * w.ctx + extra, w.row_bytes), dtype=np.uint8)
    wl.fill_host_pool(w, pool.ctypes.data, 1, threads=3, extra_rows=extra)
    for b in range(w.requests):
        assert np.array_equal(pool[b * w.ctx:(b + 1) * w.ctx], wl.rows(w, 0, b))
    assert np.array_equal(pool[w.requests * w.ctx:], wl.rows(w, 0, w.requests - 1, w.ctx, extra))
    # a layer shifted by s rows reads, for token t of request b, the row of token t + s (past the end: the extra rows)
    s = 29
    flat = pool.reshape(-1, w.row_bytes)
    t = w.ctx - 5
    assert np.array_equal(flat[(w.requests - 1) * w.ctx + t + s], wl.rows(w, 0, w.requests - 1, t + s, 1)[0])
