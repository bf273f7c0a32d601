"""Outputs unchanged (HiSparse paper, Abstract: only KV placement changes): after every resolve, the rows a
sparse-attention kernel reads through out_slots from the hot buffer are byte-identical to the rows it would read
through the selection from the full history -- both read on the GPU, through the C ABI."""
import numpy as np
import pytest
import torch

import gpu_harness as gh
import hierarchical_sparse_attention_hs_gb300 as hs
import workload as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g

    g.build()


@pytest.mark.parametrize("name,steps,layers,noio", [
    ("tiny", 16, [0], False),
    ("dsa", 10, [0], False),
    ("dsa", 6, [0], True),
    ("quest", 6, [0, 31], False),
    ("shared", 4, [0, 77], False),
])
def test_gathers_through_slots_equal_gathers_from_history(name, steps, layers, noio):
    w = wl.WORKLOADS[name]
    sel = wl.gen_selections(w, steps=steps)
    buf = gh.make_pool(w, host_layers=1 if w.layers > 1 else w.layers, noio=noio)
    pool = buf.handle
    L, B, k = w.layers, w.requests, w.topk
    topk = torch.from_numpy(sel).cuda()
    out = torch.empty((L, B, k), dtype=torch.int32, device="cuda")
    a = torch.empty((B, k, w.row_bytes), dtype=torch.uint8, device="cuda")
    h = torch.empty_like(a)
    lsel = (lambda l: 0) if w.shared_across_layers else (lambda l: l)
    for s in range(steps):
        hs.hs_step_begin(pool)
        for l in range(L):
            hs.hs_resolve(pool, l, B, topk[s, lsel(l)], k, out[l])
        for l in layers:
            a.fill_(0x5A)
            h.fill_(0xA5)
            hs.hs_gather(pool, l, B, out[l], k, a)
            hs.hs_gather_history(pool, l, B, topk[s, lsel(l)], k, h)
            assert torch.equal(a, h), (name, s, l)
    # padding: both sides give zero rows
    pad = topk[0, 0].clone()
    pad[:, ::7] = -1
    slots = torch.empty((B, k), dtype=torch.int32, device="cuda")
    hs.hs_step_begin(pool)
    hs.hs_resolve(pool, 0, B, pad, k, slots)
    hs.hs_gather(pool, 0, B, slots, k, a)
    hs.hs_gather_history(pool, 0, B, pad, k, h)
    assert torch.equal(a, h)
    assert not a[:, ::7].any()
    assert hs.hs_get_error(pool) == 0
    buf.close()


@pytest.mark.parametrize("name,noio", [("tiny", False), ("tiny", True), ("dsa", False), ("dsa", True),
                                       ("quest", False), ("quest", True)])
def test_gathers_equal_a_numpy_gather_of_the_host_rows(name, noio):
    """Each gather kernel on its own against host rows gathered on the CPU (not against the other gather): rows
    through out_slots from the hot buffer, and by token from the full history, equal host[layer][b][token] byte
    for byte; padding and out-of-range entries give zero rows. Both the host-link source and the no-IO source."""
    w = wl.WORKLOADS[name]
    steps = 3
    sel = wl.gen_selections(w, steps=steps)
    buf = gh.make_pool(w, host_layers=1, noio=noio)
    host = gh.host_rows(buf)[0]  # [B][ctx][R]; every layer reads this pool
    pool = buf.handle
    L, B, k, R = w.layers, w.requests, w.topk, w.row_bytes
    topk = torch.from_numpy(sel).cuda()
    out = torch.empty((L, B, k), dtype=torch.int32, device="cuda")
    a = torch.empty((B, k, R), dtype=torch.uint8, device="cuda")
    lsel = (lambda l: 0) if w.shared_across_layers else (lambda l: l)
    rng = np.random.default_rng([w.seed, 0x6A7E])
    check_layers = sorted({0, L - 1})
    for s in range(steps):
        hs.hs_step_begin(pool)
        for l in range(L):
            hs.hs_resolve(pool, l, B, topk[s, lsel(l)], k, out[l])
        for l in check_layers:
            idx = sel[s, lsel(l)].copy()  # [B][k]
            expect = host[np.arange(B)[:, None], idx]  # [B][k][R]
            a.fill_(0x5A)
            hs.hs_gather(pool, l, B, out[l], k, a)
            assert np.array_equal(a.cpu().numpy(), expect), (name, s, l, "through out_slots")
            # the history read with planted padding and out-of-range tokens
            bad = rng.random((B, k)) < 0.05
            idx[bad] = rng.choice(np.array([-1, -5, w.ctx, w.ctx + 17, 2**31 - 1], dtype=np.int64),
                                  size=int(bad.sum())).astype(np.int32)
            keep = (idx >= 0) & (idx < w.ctx)
            expect = np.zeros((B, k, R), dtype=np.uint8)
            expect[keep] = host[np.nonzero(keep)[0], idx[keep]]
            a.fill_(0xA5)
            hs.hs_gather_history(pool, l, B, torch.from_numpy(idx).cuda(), k, a)
            assert np.array_equal(a.cpu().numpy(), expect), (name, s, l, "from the history")
            # the hot read with planted padding and out-of-range slots
            slots = out[l].cpu().numpy()
            bad = rng.random((B, k)) < 0.05
            slots[bad] = rng.choice(np.array([-1, -3, w.slots, w.slots + 9], dtype=np.int64),
                                    size=int(bad.sum())).astype(np.int32)
            idx = sel[s, lsel(l)]
            expect = host[np.arange(B)[:, None], idx].copy()
            expect[bad] = 0
            a.fill_(0x33)
            hs.hs_gather(pool, l, B, torch.from_numpy(slots).cuda(), k, a)
            assert np.array_equal(a.cpu().numpy(), expect), (name, s, l, "planted slots")
    assert hs.hs_get_error(pool) == 0
    buf.close()
    buf.host.close()
