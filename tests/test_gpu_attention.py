"""The sparse MLA decode consumer on the tensor cores, against the float64 oracle and against itself reading the
full history ("HiSparse" paper, Abstract: model outputs are unchanged because only KV placement changes).

Tolerance, from the arithmetic. Scores: bf16 products are exact in fp32 and 576 of them accumulate in fp32, so a
score is off by at most 576 * 2^-24 * sum|q_d r_d| (about 0.013 for N(0,1) data before the scale, 1e-3 after).
Weights: P = 2^(s - m) is rounded to bf16 (relative 2^-9) and the normaliser sums the rounded weights, so each
normalised weight is off by at most about 2 * 2^-9 + the score error, relative. The output, a weighted mean of
value rows, is then off by at most max|value| * (that relative error) summed over weights = max|value| * ~5e-3;
lse by about 2^-8. The tests allow max|err| <= 6e-3 * max|value| + 1e-3 for the output and 5e-3 for lse. The
rounding errors are independent, so the typical error is far smaller: about 2^-9/sqrt(3) * sqrt(sum_i w_i^2) *
RMS(value) (3.7e-4 for 190 N(0,1) rows at the default scale); the tests also require the RMS error to stay below
2^-9 * RMS(value), which any systematic mistake (a wrong scale, row or mask) exceeds by orders of magnitude.
"""
import math

import numpy as np
import pytest
import torch

import hierarchical_sparse_attention_hs_gb300 as hs
import workload as wl
from gpu_harness import make_pool
from oracle import mla_attention as mla

pytestmark = pytest.mark.gpu

H, DQK, DV = hs.MLA_HEADS, hs.MLA_D_QK, hs.MLA_D_V
SCALE = 1.0 / math.sqrt(192.0)  # 1/sqrt(128 + 64): the query-key head dimension of the unabsorbed heads


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g

    g.build()


def _w(name, index, requests, ctx, topk, slots, steps=3, keep=70):
    return wl.Workload(name, index, layers=1, requests=requests, ctx=ctx, topk=topk, slots=slots, row_bytes=1152,
                       steps=steps, keep_pct=keep, dist=wl.UNIFORM, row_kind=wl.ROWS_BF16_NORMAL)


def _value_stats(host):
    v = mla.bf16_bits_to_f64(host.view(np.uint16)[..., :DV])
    return float(np.abs(v).max()), math.sqrt(float(np.mean(v ** 2)))


def _check(out, lse, ref_out, ref_lse, vstats, tag):
    vmax, vrms = vstats
    err = np.abs(out - ref_out)
    assert err.max() <= 6e-3 * vmax + 1e-3, f"{tag}: max |out err| {err.max()}"
    rms_err = math.sqrt(float(np.mean(err ** 2)))
    assert rms_err <= 2.0 ** -9 * vrms, f"{tag}: rms err {rms_err}"
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), f"{tag}: lse finiteness"
    assert np.abs(lse[fin] - ref_lse[fin]).max(initial=0.0) <= 5e-3, f"{tag}: lse"


def _run_pair(buf, q, slots_d, topk_d, k, scale, resident=None, resident_count=0):
    """hs_mla_decode through the slot list and hs_mla_decode_history through the tokens; both outputs."""
    B = q.shape[0]
    out_a = torch.full((B, H, DV), float("nan"), device="cuda")
    lse_a = torch.full((B, H), float("nan"), device="cuda")
    out_b, lse_b = torch.full_like(out_a, float("nan")), torch.full_like(lse_a, float("nan"))
    hs.hs_mla_decode(buf.handle, 0, B, q, slots_d, k, resident, resident_count, scale, out_a, lse_a)
    hs.hs_mla_decode_history(buf.handle, 0, B, q, topk_d, k, scale, out_b, lse_b)
    torch.cuda.synchronize()
    return out_a, lse_a, out_b, lse_b


def _oracle(w, host, q_bits, sel, scale):
    """Oracle on the rows each request's selection names (by token, from the host rows)."""
    B, k = sel.shape
    rows = np.zeros((B, k, DQK), dtype=np.uint16)
    valid = (sel >= 0) & (sel < w.ctx)
    for b in range(B):
        rows[b][valid[b]] = host[b][sel[b][valid[b]]].view(np.uint16).reshape(-1, DQK)
    return mla.decode_batch(q_bits, rows, valid, scale)


@pytest.mark.parametrize("k,pad", [(200, 0.05), (64, 0.0), (1, 0.0), (2048, 0.02)])
def test_decode_after_resolve_matches_history_and_oracle(k, pad):
    w = _w(f"mla_k{k}", 40 + k % 7, requests=3, ctx=8192, topk=k, slots=max(4 * k, 64))
    sel_all = wl.gen_selections(w)[:, 0]  # [steps][B][k]
    rng = np.random.default_rng(k)
    buf = make_pool(w, noio=True)
    host = buf.host.numpy().reshape(w.requests, w.ctx, w.row_bytes)
    q_bits = wl.gen_queries(w.requests, H, DQK, w.seed)
    q = torch.from_numpy(q_bits.view(np.int16)).cuda()
    B = w.requests
    vstats = _value_stats(host)
    out_slots = torch.empty((B, k), dtype=torch.int32, device="cuda")
    for s in range(w.steps):
        sel = sel_all[s].copy()
        if pad:
            sel[rng.random(sel.shape) < pad] = -1
        topk = torch.from_numpy(sel).cuda()
        hs.hs_step_begin(buf.handle)
        hs.hs_resolve(buf.handle, 0, B, topk, k, out_slots)
        out_a, lse_a, out_b, lse_b = _run_pair(buf, q, out_slots, topk, k, SCALE)
        # placement changes nothing: bit-identical results through the hot buffer and from the history
        assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b), s
        ref_out, ref_lse = _oracle(w, host, q_bits, sel, SCALE)
        _check(out_a.cpu().numpy(), lse_a.cpu().numpy(), ref_out, ref_lse, vstats, f"k={k} step {s}")
    assert hs.hs_get_error(buf.handle) == 0


def test_decode_large_batch_one_pair_per_request():
    """Up to the number of four-CTA clusters the device holds at once, a request's keys are split in two and the
    halves merged (the batches above); a larger batch runs one CTA pair over all of a request's keys. Both agree
    with the oracle, and the slot-list and history reads stay bit-identical."""
    split_max = hs.hs_debug_attention()  # defaults kept; the largest batch whose keys are split on this device
    w = _w("mla_wide", 52, requests=split_max + 10, ctx=2048, topk=200, slots=800, steps=2)
    assert w.requests > split_max  # so this launch runs one pair per request
    sel_all = wl.gen_selections(w)[:, 0]
    rng = np.random.default_rng(52)
    buf = make_pool(w, noio=True)
    host = buf.host.numpy().reshape(w.requests, w.ctx, w.row_bytes)
    q_bits = wl.gen_queries(w.requests, H, DQK, w.seed)
    q = torch.from_numpy(q_bits.view(np.int16)).cuda()
    B = w.requests
    vstats = _value_stats(host)
    out_slots = torch.empty((B, w.topk), dtype=torch.int32, device="cuda")
    for s in range(w.steps):
        sel = sel_all[s].copy()
        sel[rng.random(sel.shape) < 0.05] = -1
        sel[5, :] = -1  # a request with nothing valid
        topk = torch.from_numpy(sel).cuda()
        hs.hs_step_begin(buf.handle)
        hs.hs_resolve(buf.handle, 0, B, topk, w.topk, out_slots)
        out_a, lse_a, out_b, lse_b = _run_pair(buf, q, out_slots, topk, w.topk, SCALE)
        assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b), s
        ref_out, ref_lse = _oracle(w, host, q_bits, sel, SCALE)
        _check(out_a.cpu().numpy(), lse_a.cpu().numpy(), ref_out, ref_lse, vstats, f"wide step {s}")
        assert not out_a[5].any() and torch.isneginf(lse_a[5]).all()
    assert hs.hs_get_error(buf.handle) == 0


def test_decode_full_size_sampled():
    """The benchmark's configuration (32 requests, contexts of 131072 rows, top-k 2048 from 4096 hot slots, the
    same launch as the timed one): every request's slot-list read equals its history read bit for bit, and a
    sample of requests equals the oracle."""
    w = wl.WORKLOADS["mla"]
    sel_all = wl.gen_selections(w, steps=2)[:, 0]
    buf = make_pool(w)
    host = buf.host.numpy().reshape(w.requests, w.ctx, w.row_bytes)
    q_bits = wl.gen_queries(w.requests, H, DQK, w.seed)
    q = torch.from_numpy(q_bits.view(np.int16)).cuda()
    B, k = w.requests, w.topk
    out_slots = torch.empty((B, k), dtype=torch.int32, device="cuda")
    sample = [0, 13, B - 1]
    for s in range(2):
        topk = torch.from_numpy(sel_all[s]).cuda()
        hs.hs_step_begin(buf.handle)
        hs.hs_resolve(buf.handle, 0, B, topk, k, out_slots)
        out_a, lse_a, out_b, lse_b = _run_pair(buf, q, out_slots, topk, k, SCALE)
        assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b), s
        sel = sel_all[s][sample]
        rows = np.zeros((len(sample), k, DQK), dtype=np.uint16)
        valid = (sel >= 0) & (sel < w.ctx)
        for i, b in enumerate(sample):
            rows[i][valid[i]] = host[b][sel[i][valid[i]]].view(np.uint16).reshape(-1, DQK)
        ref_out, ref_lse = mla.decode_batch(q_bits[sample], rows, valid, SCALE)
        vstats = _value_stats(rows[valid].view(np.uint8))
        _check(out_a[sample].cpu().numpy(), lse_a[sample].cpu().numpy(), ref_out, ref_lse, vstats, f"full step {s}")
    assert hs.hs_get_error(buf.handle) == 0


def test_decode_peaked_scores_rescale_path():
    """sm_scale = 1 spreads the scores over hundreds of log2 units, so the running maximum rises by more than 8
    many times and the output accumulator is rescaled in tensor memory; padding rows and a request with no valid
    entry at all are mixed in."""
    w = _w("mla_peaked", 47, requests=4, ctx=4096, topk=300, slots=1024, steps=1)
    sel = wl.gen_selections(w)[0, 0].copy()
    sel[1, ::3] = -1
    sel[2, :] = -1  # nothing valid: zero output, lse -inf
    buf = make_pool(w, noio=True)
    host = buf.host.numpy().reshape(w.requests, w.ctx, w.row_bytes)
    q_bits = wl.gen_queries(w.requests, H, DQK, 77)
    q = torch.from_numpy(q_bits.view(np.int16)).cuda()
    topk = torch.from_numpy(sel).cuda()
    out_slots = torch.empty_like(topk)
    hs.hs_step_begin(buf.handle)
    hs.hs_resolve(buf.handle, 0, w.requests, topk, w.topk, out_slots)
    out_a, lse_a, out_b, lse_b = _run_pair(buf, q, out_slots, topk, w.topk, 1.0)
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)
    ref_out, ref_lse = _oracle(w, host, q_bits, sel, 1.0)
    _check(out_a.cpu().numpy(), lse_a.cpu().numpy(), ref_out, ref_lse, _value_stats(host), "peaked")
    assert not out_a[2].any() and torch.isneginf(lse_a[2]).all()
    assert hs.hs_get_error(buf.handle) == 0


def test_decode_three_tier_rows_in_place():
    """After hs_resolve_tiered, entries -2 - row are read from the ordinary HBM pool in place; the result equals
    the history read and the oracle."""
    w = _w("mla_tiered", 48, requests=3, ctx=8192, topk=512, slots=2048, steps=4)
    sel_all = wl.gen_selections(w)[:, 0]
    res = wl.gen_resident(w.ctx, w.requests, w.steps, w.seed, frac=0.4)
    B = w.requests
    res = np.where(res >= 0, res + (np.arange(B, dtype=np.int32) * w.ctx)[None, :, None], -1).astype(np.int32)
    buf = make_pool(w, noio=True)
    host = buf.host.numpy().reshape(B, w.ctx, w.row_bytes)
    q_bits = wl.gen_queries(B, H, DQK, w.seed)
    q = torch.from_numpy(q_bits.view(np.int16)).cuda()
    out_slots = torch.empty((B, w.topk), dtype=torch.int32, device="cuda")
    vstats = _value_stats(host)
    pool_rows = np.zeros((B * w.ctx, w.row_bytes), dtype=np.uint8)
    for s in range(w.steps):
        for b in range(B):  # the HBM pool holds each resident token's row at its block-table row
            held = res[s, b] >= 0
            pool_rows[res[s, b][held]] = host[b][held]
        pool_d = torch.from_numpy(pool_rows).cuda()
        topk = torch.from_numpy(sel_all[s]).cuda()
        hs.hs_step_begin(buf.handle)
        hs.hs_resolve_tiered(buf.handle, 0, B, topk, w.topk, torch.from_numpy(res[s]).cuda(), w.ctx, out_slots)
        n_inplace = int((out_slots <= -2).sum())
        out_a, lse_a, out_b, lse_b = _run_pair(buf, q, out_slots, topk, w.topk, SCALE, pool_d, B * w.ctx)
        assert n_inplace > 0
        assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b), s
        ref_out, ref_lse = _oracle(w, host, q_bits, sel_all[s], SCALE)
        _check(out_a.cpu().numpy(), lse_a.cpu().numpy(), ref_out, ref_lse, vstats, f"tiered step {s}")
    assert hs.hs_get_error(buf.handle) == 0


def test_decode_argument_errors():
    w = _w("mla_args", 49, requests=2, ctx=1024, topk=32, slots=128, steps=1)
    buf = make_pool(w, noio=True)
    q = torch.zeros((2, H, DQK), dtype=torch.int16, device="cuda")
    idx = torch.zeros((2, 32), dtype=torch.int32, device="cuda")
    out = torch.empty((2, H, DV), device="cuda")
    lse = torch.empty((2, H), device="cuda")
    with pytest.raises(hs.HsError):
        hs.hs_mla_decode(buf.handle, 1, 2, q, idx, 32, None, 0, SCALE, out, lse)  # layer out of range
    with pytest.raises(hs.HsError):
        hs.hs_mla_decode(buf.handle, 0, 3, q, idx, 32, None, 0, SCALE, out, lse)  # batch > max_batch
    with pytest.raises(hs.HsError):
        hs.hs_mla_decode(buf.handle, 0, 2, q, idx, 32, None, -1, SCALE, out, lse)
    other = wl.Workload("mla_rb", 50, layers=1, requests=1, ctx=256, topk=8, slots=16, row_bytes=656, steps=1,
                        keep_pct=0, dist=wl.UNIFORM)
    buf2 = make_pool(other)
    with pytest.raises(hs.HsError) as e:
        hs.hs_mla_decode_history(buf2.handle, 0, 1, q, idx, 8, SCALE, out, lse)
    assert e.value.code == hs.HS_ERR_UNSUPPORTED
    out.fill_(7.0)
    lse.fill_(7.0)
    hs.hs_mla_decode(buf.handle, 0, 0, q, idx, 32, None, 0, SCALE, out, lse)  # batch 0: no-op
    hs.hs_mla_decode(buf.handle, 0, 2, q, idx, 0, None, 0, SCALE, out, lse)  # k 0: no-op
    hs.hs_mla_decode_history(buf.handle, 0, 2, q, idx, 0, SCALE, out, lse)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())  # nothing written
    assert hs.hs_get_error(buf.handle) == 0


def test_decode_history_from_host_memory():
    """With no HBM copy of the history, hs_mla_decode_history reads the rows from page-locked host memory over
    the link; after resolves that fetched them from there too, it equals the read through the hot buffer."""
    w = _w("mla_host", 51, requests=2, ctx=4096, topk=160, slots=640, steps=3)
    sel_all = wl.gen_selections(w)[:, 0]
    buf = make_pool(w)  # rows come from the host pool
    host = buf.host.numpy().reshape(w.requests, w.ctx, w.row_bytes)
    q_bits = wl.gen_queries(w.requests, H, DQK, w.seed)
    q = torch.from_numpy(q_bits.view(np.int16)).cuda()
    out_slots = torch.empty((w.requests, w.topk), dtype=torch.int32, device="cuda")
    vstats = _value_stats(host)
    for s in range(w.steps):
        topk = torch.from_numpy(sel_all[s]).cuda()
        hs.hs_step_begin(buf.handle)
        hs.hs_resolve(buf.handle, 0, w.requests, topk, w.topk, out_slots)
        out_a, lse_a, out_b, lse_b = _run_pair(buf, q, out_slots, topk, w.topk, SCALE)
        assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b), s
        ref_out, ref_lse = _oracle(w, host, q_bits, sel_all[s], SCALE)
        _check(out_a.cpu().numpy(), lse_a.cpu().numpy(), ref_out, ref_lse, vstats, f"host step {s}")
    assert hs.hs_get_error(buf.handle) == 0


@pytest.mark.parametrize("split", [True, False])
def test_wait_timeout_is_reported_and_the_pool_stays_usable(split):
    """Failure detection without a GPU fault. With the test hook, the tensor-core issuer of every CTA waits on a
    barrier that nothing completes, under a short wait limit: the wait runs out before anything is issued, every
    role stops, the kernel frees its tensor memory and returns, and the pool's error word reads HS_DEVERR_TIMEOUT.
    The context stays usable: with the defaults restored, the same call gives the normal, exact result. Both
    launch shapes: keys split over two CTA pairs per request, and one pair per request."""
    split_max = hs.hs_debug_attention()
    B = 3 if split else split_max + 2
    w = _w(f"mla_to_{int(split)}", 61 + int(split), requests=B, ctx=4096, topk=64, slots=256, steps=2)
    sel = wl.gen_selections(w)[:, 0]
    buf = make_pool(w, noio=True)
    host = buf.host.numpy().reshape(w.requests, w.ctx, w.row_bytes)
    q_bits = wl.gen_queries(w.requests, H, DQK, w.seed)
    q = torch.from_numpy(q_bits.view(np.int16)).cuda()
    out_slots = torch.empty((B, w.topk), dtype=torch.int32, device="cuda")
    topk = torch.from_numpy(sel[1]).cuda()
    for s in range(2):
        hs.hs_step_begin(buf.handle)
        hs.hs_resolve(buf.handle, 0, B, torch.from_numpy(sel[s]).cuda(), w.topk, out_slots)
    out = torch.zeros((B, H, DV), device="cuda")
    lse = torch.zeros((B, H), device="cuda")
    torch.cuda.synchronize()
    hs.hs_debug_attention(64, True)
    try:
        hs.hs_mla_decode(buf.handle, 0, B, q, out_slots, w.topk, None, 0, SCALE, out, lse)
        torch.cuda.synchronize()
    finally:
        hs.hs_debug_attention(0, False)
    assert hs.hs_get_error(buf.handle, clear=True) == hs.HS_DEVERR_TIMEOUT
    assert hs.hs_get_error(buf.handle) == 0
    out_a, lse_a, out_b, lse_b = _run_pair(buf, q, out_slots, topk, w.topk, SCALE)
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)
    ref_out, ref_lse = _oracle(w, host, q_bits, sel[1], SCALE)
    _check(out_a.cpu().numpy(), lse_a.cpu().numpy(), ref_out, ref_lse, _value_stats(host), "after a timeout")
    assert hs.hs_get_error(buf.handle) == 0
    buf.close()
