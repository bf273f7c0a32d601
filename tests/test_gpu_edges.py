"""Edge cases of the GPU path against the CPU oracle: every cluster size, padding and ragged k, rejected rows,
empty calls, wide stamp ranges (multi-pass victim sort), long token keys, and host-side argument errors."""
import numpy as np
import pytest
import torch

import hierarchical_sparse_attention_hs_gb300 as hs
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g

    g.build()


def _pool(layers, batch, ctx, slots, topk_max, row_bytes, seed=0):
    buf = hs.PoolBuffers(layers, batch, ctx, slots, topk_max, row_bytes, host_layers=layers)
    rng = np.random.default_rng(seed)
    h = buf.host.numpy()
    h[:] = rng.integers(0, 256, size=h.shape, dtype=np.uint8)
    buf.create()
    return buf


def _rand_sel(rng, batch, k, ctx, prev=None, keep=0.6, pad=0.0):
    out = np.empty((batch, k), dtype=np.int32)
    for b in range(batch):
        n_keep = int(keep * k) if prev is not None else 0
        kept = rng.choice(prev[b][prev[b] >= 0], size=min(n_keep, int((prev[b] >= 0).sum())), replace=False) \
            if prev is not None else np.empty(0, dtype=np.int64)
        rest = np.setdiff1d(rng.choice(ctx, size=min(ctx, 3 * k), replace=False), kept)[: k - len(kept)]
        row = np.concatenate([kept, rest]).astype(np.int32)
        rng.shuffle(row)
        if pad:
            row[rng.random(k) < pad] = -1
        out[b] = row
    return out


def _run(buf, ora, sels, layer=0, set_step=None):
    stream = torch.cuda.Stream()
    batch, k = sels[0].shape
    for sel in sels:
        with torch.cuda.stream(stream):
            if set_step is not None:
                buf.view("step").fill_(set_step)
            hs.hs_step_begin(buf.handle, stream)
            t = torch.from_numpy(sel).cuda()
            out = torch.full((batch, k), -9, dtype=torch.int32, device="cuda")
            hs.hs_resolve(buf.handle, layer, batch, t, k, out, stream)
        stream.synchronize()
        if set_step is not None:
            ora.step = set_step
            set_step = None
        ora.step_begin()
        expect = ora.resolve(layer, sel, None)
        assert np.array_equal(out.cpu().numpy(), expect)
    for name, ref in (("tok2slot", ora.tok2slot), ("slot_tok", ora.slot_tok), ("slot_stamp", ora.slot_stamp)):
        assert np.array_equal(buf.view(name).cpu().numpy(), ref), name
    assert np.array_equal(buf.view("counters").cpu().numpy().astype(np.uint64), ora.counters)


def _check_rows(buf):
    host = buf.host.numpy().reshape(buf.layers, buf.max_batch, buf.ctx, buf.row_bytes)
    st = buf.view("slot_tok").cpu().numpy()
    hot = buf.hot_view().cpu().numpy()
    for l in range(buf.layers):
        for b in range(buf.max_batch):
            occ = st[l, b] >= 0
            assert np.array_equal(hot[l, b][occ], host[l, b][st[l, b][occ]])
            assert not hot[l, b][~occ].any()


@pytest.mark.parametrize("batch", [80, 32, 16, 5, 1])  # cluster sizes 1, 2, 4, 8, 8
def test_every_cluster_size(batch):
    rng = np.random.default_rng(batch)
    ctx, slots, k, R = 5000, 300, 120, 48
    buf = _pool(1, batch, ctx, slots, k, R, seed=batch)
    ora = oracle.OraclePool(ctx, slots, R, 1, batch, track_rows=False)
    sels, prev = [], None
    for s in range(12):
        prev = _rand_sel(rng, batch, k, ctx, prev, keep=0.0 if s == 6 else 0.6)
        sels.append(prev)
    _run(buf, ora, sels)
    _check_rows(buf)
    buf.close()


def test_padding_and_ragged_k():
    rng = np.random.default_rng(5)
    ctx, slots, kmax, R = 3000, 257, 200, 32
    buf = _pool(2, 6, ctx, slots, kmax, R, seed=5)
    ora = oracle.OraclePool(ctx, slots, R, 2, 6, track_rows=False)
    prev = None
    sels = []
    for s in range(10):
        prev = _rand_sel(rng, 6, 77, ctx, prev, keep=0.5, pad=0.15)  # k = 77 < topk_max, 15% padding
        sels.append(prev)
    _run(buf, ora, sels, layer=1)
    _check_rows(buf)
    buf.close()


def test_rejected_rows_change_nothing():
    rng = np.random.default_rng(9)
    ctx, slots, k, R = 1000, 64, 16, 16
    buf = _pool(1, 4, ctx, slots, k, R, seed=9)
    ora = oracle.OraclePool(ctx, slots, R, 1, 4, track_rows=False)
    base = _rand_sel(rng, 4, k, ctx)
    _run(buf, ora, [base])
    bad = _rand_sel(rng, 4, k, ctx, prev=base, keep=0.5)
    bad[0, 3] = ctx            # out of range
    bad[1, 5] = bad[1, 7]      # duplicate
    hit_tok = base[2, 0]
    bad[2, :2] = hit_tok       # duplicate of a resident token (caught among hits)
    _run(buf, ora, [bad])
    assert ora.error == (oracle.ERR_RANGE | oracle.ERR_DUP)
    assert hs.hs_get_error(buf.handle, clear=True) == (hs.HS_DEVERR_RANGE | hs.HS_DEVERR_DUP)
    assert hs.hs_get_error(buf.handle) == 0
    # row 3 was valid and was resolved normally; the next steps continue in lockstep with the oracle
    _run(buf, ora, [_rand_sel(rng, 4, k, ctx, prev=base, keep=0.3)])
    buf.close()


def test_empty_calls_are_noops():
    buf = _pool(1, 2, 100, 8, 4, 16)
    before = buf.meta.clone()
    t = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    hs.hs_resolve(buf.handle, 0, 0, t, 4, t)
    hs.hs_resolve(buf.handle, 0, 2, t, 0, t)
    hs.hs_prefetch(buf.handle, 0, 0, t, 4)
    torch.cuda.synchronize()
    assert torch.equal(before, buf.meta)
    buf.close()


def test_wide_stamp_range_multi_pass_victim_sort():
    # jump the step counter so stamps span > 2^16: the victim sort needs three 8-bit passes
    rng = np.random.default_rng(11)
    ctx, slots, k, R = 4000, 200, 40, 16
    buf = _pool(1, 3, ctx, slots, k, R, seed=11)
    ora = oracle.OraclePool(ctx, slots, R, 1, 3, track_rows=False)
    prev = None
    first = []
    for s in range(6):
        prev = _rand_sel(rng, 3, k, ctx, prev, keep=0.2)
        first.append(prev)
    _run(buf, ora, first)
    later = []
    for s in range(8):
        prev = _rand_sel(rng, 3, k, ctx, prev, keep=0.5)
        later.append(prev)
    _run(buf, ora, later, set_step=70000)
    assert int(buf.view("slot_stamp").max()) > 70000 and int(buf.view("slot_stamp")[buf.view("slot_stamp") > 0].min()) < 10
    _check_rows(buf)
    buf.close()


@pytest.mark.parametrize("shape", ["narrow", "wide", "few_old", "ties", "empties_late"])
def test_victim_choice_on_arbitrary_stamp_distributions(shape):
    """The victim choice against the oracle on stamp layouts a short replay rarely reaches: after a few ordinary
    steps, the stamps of the occupied slots are rewritten (identically on both sides, every stamp <= the step) and
    the next steps resolved. narrow: a few recent steps; wide: ages spread over 1000 steps, so stamp bins are
    clamped while the victims lie in exact bins; few_old: fewer very old slots than misses, so the threshold falls
    in the clamped bin and the full sort runs; ties: three distinct stamps; empties_late: empty slots remain at a
    late step."""
    rng = np.random.default_rng(sum(map(ord, shape)))
    batch, ctx, slots, k, R = 4, 5000, 300, 64, 16
    buf = _pool(1, batch, ctx, slots, k, R, seed=5)
    ora = oracle.OraclePool(ctx, slots, R, 1, batch, track_rows=False)
    prev, sels = None, []
    n_fill = 2 if shape == "empties_late" else 8
    for s in range(n_fill):
        prev = _rand_sel(rng, batch, k, ctx, prev, keep=0.3)
        sels.append(prev)
    _run(buf, ora, sels)
    step = 2000
    occ = ora.slot_tok[0] >= 0
    st = ora.slot_stamp[0].copy()
    for b in range(batch):
        n = int(occ[b].sum())
        if shape == "narrow":
            v = rng.integers(step - 6, step + 1, size=n)
        elif shape == "wide":
            v = rng.integers(step - 1000, step + 1, size=n)
        elif shape == "few_old":
            v = np.full(n, step - 1)
            v[rng.choice(n, size=5, replace=False)] = rng.integers(1, 20, size=5)
        elif shape == "ties":
            v = rng.choice(np.array([step - 300, step - 7, step]), size=n)
        else:
            v = rng.integers(step - 2, step + 1, size=n)
        st[b][occ[b]] = v
    ora.slot_stamp[0][...] = st
    buf.view("slot_stamp")[0].copy_(torch.from_numpy(st).cuda())
    later = []
    for s in range(4):
        prev = _rand_sel(rng, batch, k, ctx, prev, keep=0.25 if shape == "few_old" else 0.5)
        later.append(prev)
    _run(buf, ora, later, set_step=step)
    _check_rows(buf)
    assert hs.hs_get_error(buf.handle) == 0
    buf.close()


def test_long_token_keys():
    # ctx = 2^23: token keys need three 8-bit passes, the top pass nearly empty
    rng = np.random.default_rng(13)
    ctx, slots, k, R = 1 << 23, 96, 64, 16
    buf = _pool(1, 2, ctx, slots, k, R, seed=13)
    ora = oracle.OraclePool(ctx, slots, R, 1, 2, track_rows=False)
    prev = None
    sels = []
    for s in range(8):
        prev = _rand_sel(rng, 2, k, ctx, prev, keep=0.4)
        sels.append(prev)
    _run(buf, ora, sels)
    _check_rows(buf)
    buf.close()


def test_argument_errors():
    buf = _pool(2, 4, 100, 16, 8, 16)
    t = torch.zeros((4, 8), dtype=torch.int32, device="cuda")
    for args in [(2, 4, t, 8, t), (-1, 4, t, 8, t), (0, 5, t, 8, t), (0, 4, t, 9, t), (0, 4, None, 8, t),
                 (0, 4, t, 8, None)]:
        with pytest.raises(hs.HsError) as e:
            hs.hs_resolve(buf.handle, *args)
        assert e.value.code == hs.HS_ERR_INVALID_ARG
    # a host pool that is not page-locked mapped memory is refused
    plain = np.zeros(2 * 4 * 100 * 16, dtype=np.uint8)
    d = hs.hs_pool_desc(2, 4, 100, 16, 8, 16, plain.ctypes.data, 0, 0, buf.hot.data_ptr(), buf.meta.data_ptr(), None)
    with pytest.raises(hs.HsError) as e:
        hs.hs_pool_create(d)
    assert e.value.code == hs.HS_ERR_NOT_MAPPED
    # misaligned meta
    d = hs.hs_pool_desc(2, 4, 100, 16, 8, 16, buf.host.ptr, 0, 0, buf.hot.data_ptr(), buf.meta.data_ptr() + 16, None)
    with pytest.raises(hs.HsError) as e:
        hs.hs_pool_create(d)
    assert e.value.code == hs.HS_ERR_INVALID_ARG
    buf.close()


@pytest.mark.parametrize("batch", [3, 40])
def test_resolve_shared_small_and_ragged(batch):
    # layers 1..3 resolved together with one selection, layer 0 and 4 on their own; small miss counts leave
    # fewer blocks than first-wave warps
    rng = np.random.default_rng(21 + batch)
    ctx, slots, k, R = 3000, 200, 60, 48
    L = 5
    buf = _pool(L, batch, ctx, slots, k, R, seed=3)
    ora = oracle.OraclePool(ctx, slots, R, L, batch, track_rows=False)
    stream = torch.cuda.Stream()
    prev = None
    for step in range(10):
        prev = _rand_sel(rng, batch, k, ctx, prev, keep=0.0 if step == 5 else 0.7, pad=0.05)
        other = _rand_sel(rng, batch, k, ctx, None)
        t = torch.from_numpy(prev).cuda()
        t2 = torch.from_numpy(other).cuda()
        outs = torch.full((L, batch, k), -9, dtype=torch.int32, device="cuda")
        with torch.cuda.stream(stream):
            hs.hs_step_begin(buf.handle, stream)
            hs.hs_resolve(buf.handle, 0, batch, t2, k, outs[0], stream)
            hs.hs_resolve_shared(buf.handle, 1, 3, batch, t, k, outs[1], stream)
            hs.hs_resolve(buf.handle, 4, batch, t2, k, outs[4], stream)
        stream.synchronize()
        ora.step_begin()
        assert np.array_equal(outs[0].cpu().numpy(), ora.resolve(0, other, None))
        for l in (1, 2, 3):
            assert np.array_equal(outs[1].cpu().numpy(), ora.resolve(l, prev, None)), (step, l)
        assert np.array_equal(outs[4].cpu().numpy(), ora.resolve(4, other, None))
    for name, ref in (("tok2slot", ora.tok2slot), ("slot_tok", ora.slot_tok), ("slot_stamp", ora.slot_stamp)):
        assert np.array_equal(buf.view(name).cpu().numpy(), ref), name
    assert np.array_equal(buf.view("counters").cpu().numpy().astype(np.uint64), ora.counters)
    _check_rows(buf)
    with pytest.raises(hs.HsError):
        hs.hs_resolve_shared(buf.handle, 3, 3, batch, t, k, outs[0])  # past the last layer
    buf.close()


@pytest.mark.parametrize("ctx", [6000, 300000])  # token bitmap and radix miss ranking
def test_selection_and_slots_in_mapped_host_memory(ctx):
    """The selection is read from, and out_slots written to, page-locked mapped host memory by the kernel itself
    (no copies). The same host buffers are rewritten every step, so a stale copy of a host line would show; the
    results equal the device-memory path's and the oracle's. The gather reads its slot list from host memory too."""
    rng = np.random.default_rng(ctx)
    batch, slots, k, R = 6, 400, 96, 64
    dev = _pool(1, batch, ctx, slots, k, R, seed=5)
    hst = _pool(1, batch, ctx, slots, k, R, seed=5)
    ora = oracle.OraclePool(ctx, slots, R, 1, batch, track_rows=False)
    sel_h = hs.HostBuffer(batch * k * 4)
    out_h = hs.HostBuffer(batch * k * 4)
    gat_h = torch.empty((batch, k, R), dtype=torch.uint8, device="cuda")
    gat_d = torch.empty_like(gat_h)
    sel_np = np.frombuffer(sel_h.numpy(), dtype=np.int32).reshape(batch, k)
    out_np = np.frombuffer(out_h.numpy(), dtype=np.int32).reshape(batch, k)
    stream = torch.cuda.Stream()
    prev = None
    for step in range(12):
        prev = _rand_sel(rng, batch, k, ctx, prev, keep=0.0 if step == 6 else 0.6, pad=0.03)
        sel_np[:] = prev
        out_np[:] = -9
        t = torch.from_numpy(prev).cuda()
        out_d = torch.full((batch, k), -9, dtype=torch.int32, device="cuda")
        with torch.cuda.stream(stream):
            hs.hs_step_begin(dev.handle, stream)
            hs.hs_step_begin(hst.handle, stream)
            hs.hs_resolve(dev.handle, 0, batch, t, k, out_d, stream)
            hs.hs_resolve(hst.handle, 0, batch, sel_h.ptr, k, out_h.ptr, stream)
            hs.hs_gather(dev.handle, 0, batch, out_d, k, gat_d, stream)
            hs.hs_gather(hst.handle, 0, batch, out_h.ptr, k, gat_h, stream)
        stream.synchronize()
        ora.step_begin()
        expect = ora.resolve(0, prev, None)
        assert np.array_equal(out_d.cpu().numpy(), expect), step
        assert np.array_equal(out_np, expect), step
        assert torch.equal(gat_h, gat_d), step
    for name in ("tok2slot", "slot_tok", "slot_stamp", "counters"):
        assert torch.equal(dev.view(name), hst.view(name)), name
    assert torch.equal(dev.hot_view(), hst.hot_view())
    _check_rows(hst)
    for b in (dev, hst):
        b.close()
    sel_h.close()
    out_h.close()


def test_probe_link_measures_and_rejects():
    """The link probe reads a mapped host buffer with SM loads and copies it with cudaMemcpyAsync; both give a
    positive bandwidth below the device's own copy rate, and bad arguments are refused before anything runs."""
    host = hs.HostBuffer(64 << 20)
    dev = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    zc, cp = hs.hs_probe_link(host.ptr, dev, 64 << 20, 2)
    assert 1.0 < zc < 5000.0 and 1.0 < cp < 5000.0, (zc, cp)
    with pytest.raises(hs.HsError):
        hs.hs_probe_link(host.ptr, dev, (64 << 20) - 8, 2)  # not a multiple of 16
    with pytest.raises(hs.HsError):
        hs.hs_probe_link(host.ptr + 8, dev, 1 << 20, 2)  # misaligned host address
    with pytest.raises(hs.HsError):
        hs.hs_probe_link(host.ptr, dev, 1 << 20, 0)  # no iteration
    torch.cuda.synchronize()
    host.close()


def test_host_alloc_failure_is_reported_and_leaves_cuda_usable():
    """A page-locked allocation the host cannot satisfy (1 PiB) comes back as HS_ERR_CUDA with a null pointer,
    without a sticky error: a normal allocation and a device launch work right after."""
    with pytest.raises(hs.HsError) as e:
        hs.hs_host_alloc(1 << 50)
    assert e.value.code == hs.HS_ERR_CUDA
    host = hs.HostBuffer(1 << 20)
    dev = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    zc, cp = hs.hs_probe_link(host.ptr, dev, 1 << 20, 1)
    assert zc > 0 and cp > 0
    torch.cuda.synchronize()
    host.close()


def test_probe_launch_runs_and_checks_its_arguments():
    """The launch-floor probe enqueues the resolve's launch shape with an empty kernel: it touches no memory
    (the pool's state is unchanged) and refuses the arguments a resolve refuses."""
    buf = _pool(4, 8, 2000, 256, 64, 48)
    before = buf.meta.clone()
    for nl, batch in ((1, 8), (4, 3), (2, 1)):
        hs.hs_probe_launch(buf.handle, 0, nl, batch, 64)
    hs.hs_probe_launch(buf.handle, 0, 1, 0, 64)  # batch 0: no-op
    torch.cuda.synchronize()
    assert torch.equal(buf.meta, before)
    for bad in ((0, 5, 8, 64), (-1, 1, 8, 64), (0, 1, 9, 64), (0, 1, 8, 65), (0, 0, 8, 64)):
        with pytest.raises(hs.HsError):
            hs.hs_probe_launch(buf.handle, *bad)
    buf.close()


def test_fused_step_begins_add_up_and_reset_drops_them():
    """Two fused begins before a resolve advance the step by two; a reset drops a pending one; a call that launches
    nothing (batch 0) leaves it pending for the next."""
    rng = np.random.default_rng(3)
    buf = _pool(1, 2, 3000, 128, 32, 16)
    ora = oracle.OraclePool(3000, 128, 16, 1, 2, track_rows=False)
    out = torch.empty((2, 32), dtype=torch.int32, device="cuda")
    sel = _rand_sel(rng, 2, 32, 3000)
    hs.hs_step_begin_fused(buf.handle)
    hs.hs_step_begin_fused(buf.handle)
    hs.hs_resolve(buf.handle, 0, 0, torch.from_numpy(sel).cuda(), 32, out)  # batch 0: nothing launched
    hs.hs_resolve(buf.handle, 0, 2, torch.from_numpy(sel).cuda(), 32, out)
    ora.step_begin()
    ora.step_begin()
    expect = ora.resolve(0, sel, None)
    torch.cuda.synchronize()
    assert int(buf.view("step").item()) == 2
    assert np.array_equal(out.cpu().numpy(), expect)
    assert np.array_equal(buf.view("slot_stamp").cpu().numpy(), ora.slot_stamp)
    hs.hs_step_begin_fused(buf.handle)
    hs.hs_pool_reset(buf.handle)
    hs.hs_resolve(buf.handle, 0, 2, torch.from_numpy(sel).cuda(), 32, out)
    torch.cuda.synchronize()
    assert int(buf.view("step").item()) == 0  # the reset dropped the pending begin
    assert hs.hs_get_error(buf.handle) == 0
    buf.close()


def test_checkpoint_and_resume():
    """The pool's whole state is plain device arrays (metadata and hot buffer): copied out mid-sequence and copied
    back later, it makes the pool replay the same steps with the same outputs and state."""
    rng = np.random.default_rng(123)
    batch, ctx, slots, k, R = 4, 5000, 300, 80, 64
    buf = _pool(1, batch, ctx, slots, k, R, seed=9)
    stream = torch.cuda.Stream()
    sels, prev = [], None
    for step in range(8):
        prev = _rand_sel(rng, batch, k, ctx, prev, keep=0.5)
        sels.append(prev)

    def run(steps):
        outs = []
        for sel in steps:
            out = torch.empty((batch, k), dtype=torch.int32, device="cuda")
            with torch.cuda.stream(stream):
                hs.hs_step_begin(buf.handle, stream)
                hs.hs_resolve(buf.handle, 0, batch, torch.from_numpy(sel).cuda(), k, out, stream)
            stream.synchronize()
            outs.append(out.cpu().numpy())
        return outs

    run(sels[:4])
    snap_meta, snap_hot = buf.meta.clone(), buf.hot.clone()
    first = run(sels[4:])
    end_meta, end_hot = buf.meta.clone(), buf.hot.clone()
    buf.meta.copy_(snap_meta)  # restore the checkpoint
    buf.hot.copy_(snap_hot)
    torch.cuda.synchronize()
    second = run(sels[4:])
    assert all(np.array_equal(a, b) for a, b in zip(first, second))
    assert torch.equal(buf.meta, end_meta) and torch.equal(buf.hot, end_hot)
    buf.close()
