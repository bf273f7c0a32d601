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
