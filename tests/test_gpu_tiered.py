"""Three-tier resolution on the GPU against the CPU oracle ("Hybrid HiSparse" knowledge card, Timeline: resident,
hot and missing rows resolved in one pass, the hot pages coming from ordinary KV blocks of the same pool).

A token still held in the HBM KV pool is served in place (out_slot = -2 - its pool row), a hot-buffer hit takes
precedence over it, and only tokens in neither tier are fetched. Both miss-ranking modes are covered: the token
bitmap (short contexts) and the radix sort (contexts above 2^18 tokens), each with its own check for a repeated
in-place token."""
import numpy as np
import pytest
import torch

import hierarchical_sparse_attention_hs_gb300 as hs
import oracle
import workload as wl
from gpu_harness import compare_state, make_pool

pytestmark = pytest.mark.gpu

# bitmap ranking (ctx <= 2^18) and radix ranking (ctx > 2^18); 3 and 9 requests give clusters of 8 and 4
SHORT = wl.Workload("tiered_short", 21, layers=2, requests=9, ctx=16384, topk=512, slots=1024, row_bytes=272,
                    steps=10, keep_pct=70, dist=wl.ZIPF, zipf_s=1.1)
LONG = wl.Workload("tiered_long", 22, layers=1, requests=3, ctx=1 << 19, topk=1024, slots=2048, row_bytes=64,
                   steps=8, keep_pct=60, dist=wl.UNIFORM, churn=(5,))


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g

    g.build()


def _tiered_replay(w, frac):
    sel = wl.gen_selections(w)  # [steps][layers][B][k]
    res = wl.gen_resident(w.ctx, w.requests, w.steps, w.seed, frac=frac)  # [steps][B][ctx]
    buf = make_pool(w, host_layers=w.layers)
    L, B, k = w.layers, w.requests, w.topk
    ora = oracle.OraclePool(w.ctx, w.slots, w.row_bytes, L, B, track_rows=False)
    host = buf.host.numpy().reshape(L, B, w.ctx, w.row_bytes)
    s0 = torch.cuda.Stream()
    out = torch.full((L, B, k), -7, dtype=torch.int32, device="cuda")
    n_inplace = 0
    for s in range(w.steps):
        res_d = torch.from_numpy(res[s]).cuda()
        sel_d = torch.from_numpy(sel[s]).cuda()
        with torch.cuda.stream(s0):
            hs.hs_step_begin(buf.handle, s0)
            for l in range(L):
                hs.hs_resolve_tiered(buf.handle, l, B, sel_d[l], k, res_d, w.ctx, out[l], s0)
        s0.synchronize()
        ora.step_begin()
        got = out.cpu().numpy()
        hot = buf.hot_view().cpu().numpy()
        for l in range(L):
            expect = ora.resolve(l, sel[s, l], None, resident=res[s])
            assert np.array_equal(got[l], expect), (w.name, s, l, np.argwhere(got[l] != expect)[:5].tolist())
            # what a sparse-attention kernel would read: hot slot, or the in-place row of the HBM pool (built
            # here from the host rows by the resident map), equals the selected token's host row
            for b in range(B):
                o, t = got[l, b], sel[s, l, b]
                hit, inpl = o >= 0, o <= -2
                assert np.array_equal(hot[l, b][o[hit]], host[l, b][t[hit]])
                rows = -2 - o[inpl]
                tok_of_row = np.full(w.ctx, -1, dtype=np.int64)
                held = res[s, b] >= 0
                tok_of_row[res[s, b][held]] = np.flatnonzero(held)
                assert np.array_equal(tok_of_row[rows], t[inpl])
                n_inplace += int(inpl.sum())
        if s == w.steps // 2:
            compare_state(buf, ora, f"{w.name} step {s}")
    compare_state(buf, ora, f"{w.name} end")
    assert hs.hs_get_error(buf.handle) == 0
    assert n_inplace > 0
    return buf, ora


@pytest.mark.parametrize("w", [SHORT, LONG], ids=lambda w: w.name)
def test_tiered_matches_oracle(w):
    _tiered_replay(w, frac=0.3)


def test_tiered_without_resident_rows_equals_two_tier():
    """An all -1 map makes the three-tier call the plain resolve (same outputs, same state)."""
    w = SHORT
    sel = wl.gen_selections(w, steps=4)
    a = make_pool(w, host_layers=w.layers)
    c = make_pool(w, host_layers=w.layers)
    B, k = w.requests, w.topk
    none = torch.full((B, w.ctx), -1, dtype=torch.int32, device="cuda")
    oa = torch.empty((B, k), dtype=torch.int32, device="cuda")
    oc = torch.empty_like(oa)
    s0 = torch.cuda.Stream()
    for s in range(4):
        t = torch.from_numpy(sel[s, 0]).cuda()
        with torch.cuda.stream(s0):
            hs.hs_step_begin(a.handle, s0)
            hs.hs_step_begin(c.handle, s0)
            hs.hs_resolve_tiered(a.handle, 0, B, t, k, none, w.ctx, oa, s0)
            hs.hs_resolve(c.handle, 0, B, t, k, oc, s0)
        s0.synchronize()
        assert torch.equal(oa, oc)
    for name in ("tok2slot", "slot_tok", "slot_stamp", "counters"):
        assert torch.equal(a.view(name), c.view(name)), name
    assert torch.equal(a.hot_view(), c.hot_view())


@pytest.mark.parametrize("w", [SHORT, LONG], ids=lambda w: w.name)
def test_tiered_all_resident_fetches_nothing(w):
    """Every selected token resident and none hot: all served in place, no slot, stamp or byte changes."""
    sel = wl.gen_selections(w, steps=1)[0, 0]
    buf = make_pool(w, host_layers=w.layers)
    B, k = w.requests, w.topk
    res = np.arange(w.ctx, dtype=np.int32)[::-1].copy()
    res_d = torch.from_numpy(np.tile(res, (B, 1))).cuda()
    out = torch.empty((B, k), dtype=torch.int32, device="cuda")
    before = {n: buf.view(n).clone() for n in ("tok2slot", "slot_tok", "slot_stamp")}
    s0 = torch.cuda.Stream()
    with torch.cuda.stream(s0):
        hs.hs_step_begin(buf.handle, s0)
        hs.hs_resolve_tiered(buf.handle, 0, B, torch.from_numpy(sel).cuda(), k, res_d, w.ctx, out, s0)
    s0.synchronize()
    assert np.array_equal(out.cpu().numpy(), -2 - res[sel])
    for n, v in before.items():
        assert torch.equal(buf.view(n), v), n
    cnt = buf.view("counters").cpu().numpy()[0]
    assert cnt.tolist() == [B * k, 0, 0, 0]
    assert not buf.hot_view().any()


@pytest.mark.parametrize("w", [SHORT, LONG], ids=lambda w: w.name)
def test_tiered_repeated_inplace_token_rejects_row(w):
    """A token repeated among the in-place entries rejects its row like any repeat: out_slots -1, the duplicate
    error bit, and no state change; the other rows resolve normally."""
    sel = wl.gen_selections(w, steps=2)[:, 0]  # [2][B][k]
    res = wl.gen_resident(w.ctx, w.requests, 2, w.seed, frac=0.3)
    buf = make_pool(w, host_layers=w.layers)
    B, k = w.requests, w.topk
    ora = oracle.OraclePool(w.ctx, w.slots, w.row_bytes, w.layers, B, track_rows=False)
    s0 = torch.cuda.Stream()
    out = torch.empty((B, k), dtype=torch.int32, device="cuda")
    bad = sel[1].copy()
    b_bad = B // 2
    inpl = np.flatnonzero(res[1, b_bad][bad[b_bad]] >= 0)
    assert len(inpl) >= 2
    bad[b_bad, inpl[-1]] = bad[b_bad, inpl[0]]  # one in-place token twice
    for s, row in enumerate((sel[0], bad)):
        with torch.cuda.stream(s0):
            hs.hs_step_begin(buf.handle, s0)
            hs.hs_resolve_tiered(buf.handle, 0, B, torch.from_numpy(row).cuda(), k,
                                 torch.from_numpy(res[s]).cuda(), w.ctx, out, s0)
        s0.synchronize()
        ora.step_begin()
        expect = ora.resolve(0, row, None, resident=res[s])
        assert np.array_equal(out.cpu().numpy(), expect), s
    assert (out.cpu().numpy()[b_bad] == -1).all()
    compare_state(buf, ora, w.name)
    assert hs.hs_get_error(buf.handle, clear=True) == ora.error == 2


def test_tiered_argument_errors():
    w = SHORT
    buf = make_pool(w, host_layers=w.layers)
    B, k = w.requests, w.topk
    t = torch.zeros((B, k), dtype=torch.int32, device="cuda")
    out = torch.empty((B, k), dtype=torch.int32, device="cuda")
    res = torch.full((B, w.ctx), -1, dtype=torch.int32, device="cuda")
    with pytest.raises(RuntimeError):
        hs.hs_resolve_tiered(buf.handle, 0, B, t, k, None, w.ctx, out)
    with pytest.raises(RuntimeError):
        hs.hs_resolve_tiered(buf.handle, 0, B, t, k, res, w.ctx - 1, out)
    torch.cuda.synchronize()
