"""GPU path (through the C ABI) against the CPU oracle, bit for bit: out_slots after every call, the whole
metadata state (tok2slot, slot_tok, slot_stamp, counters) and every hot-buffer byte, on all five workloads at
their full sizes, in the launch configuration the benchmark uses."""
import numpy as np
import pytest
import torch

import gpu_harness as gh
import workload as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g

    g.build()


def test_tiny_full_state_and_rows():
    import oracle

    w = wl.WORKLOADS["tiny"]
    buf, ora = gh.replay(w)
    # the oracle with rows tracked: compare every hot-buffer byte directly
    ora2 = oracle.OraclePool(w.ctx, w.slots, w.row_bytes, 1, 1, track_rows=True)
    sel = wl.gen_selections(w)
    host = gh.host_rows(buf)[0]
    for s in range(w.steps):
        ora2.step_begin()
        ora2.resolve(0, sel[s, 0], host)
    assert np.array_equal(buf.hot_view().cpu().numpy(), ora2.hot)
    buf.close()


@pytest.mark.parametrize("name", ["dsa", "multilayer", "quest", "shared"])
def test_workload_parity(name):
    w = wl.WORKLOADS[name]
    buf, ora = gh.replay(w)
    gh.check_hot_rows(buf)
    buf.close()


def test_dsa_graph_replay_matches_oracle():
    w = wl.WORKLOADS["dsa"]
    buf, _ = gh.replay(w, steps=24, graphs=True)
    gh.check_hot_rows(buf)
    buf.close()


def test_dsa_noio_mode():
    w = wl.WORKLOADS["dsa"]
    buf, _ = gh.replay(w, steps=20, noio=True)
    gh.check_hot_rows(buf)
    buf.close()


def test_shared_with_layerwise_prefetch_is_exact():
    # prefetch(l+1) on a second stream + resolve(l): the state must equal a lone resolve's (the oracle's)
    w = wl.WORKLOADS["shared"]
    buf, _ = gh.replay(w, steps=8, prefetch=True)
    gh.check_hot_rows(buf)
    buf.close()


@pytest.mark.parametrize("depth", [1, 2, 3])
def test_shared_layerwise_prefetch_depth_is_exact(depth):
    # prefetch `depth` layers ahead on as many side streams, as the benchmark does, captured in graphs: the state
    # equals per-layer resolves (the oracle's)
    w = wl.WORKLOADS["shared"]
    buf, _ = gh.replay(w, steps=5, prefetch=True, graphs=True, depth=depth)
    gh.check_hot_rows(buf, layers=[0, 1, 2, 40, 77])
    buf.close()


def test_shared_prefetch_in_graph():
    w = wl.WORKLOADS["shared"]
    buf, _ = gh.replay(w, steps=4, prefetch=True, graphs=True)
    gh.check_hot_rows(buf, layers=[0, 1, 77])
    buf.close()


@pytest.mark.parametrize("shared_call", [False, True])
def test_shared_pool_read_with_a_layer_shift_is_exact(shared_call):
    # one host pool for all layers, layer l reading token t from row t + l * S (the benchmark's stand-in for a pool
    # per layer): the state equals the oracle's, and every layer's hot rows are its own shifted host rows
    w = wl.WORKLOADS["shared"]
    shift = w.ctx // w.layers
    if shared_call:
        buf, _ = gh.replay(w, steps=4, shared_call=True, layer_shift_rows=shift)
    else:
        buf, _ = gh.replay(w, steps=4, prefetch=True, graphs=True, depth=1, layer_shift_rows=shift)
    assert buf.layer_shift_rows == shift and buf.desc.host_layer_stride == shift * w.row_bytes
    gh.check_hot_rows(buf, layers=[0, 1, 40, 77])
    buf.close()


def test_shared_selection_one_call_for_all_layers():
    # hs_resolve_shared: one resolve per step drives all 78 layers; state, counters and rows equal the oracle's
    # per-layer resolves
    w = wl.WORKLOADS["shared"]
    buf, _ = gh.replay(w, steps=12, shared_call=True)
    gh.check_hot_rows(buf, layers=[0, 1, 40, 77])
    buf.close()


@pytest.mark.parametrize("name,graphs,shared_call", [("dsa", False, False), ("dsa", True, False),
                                                     ("multilayer", True, False), ("shared", True, True)])
def test_fused_step_begin_is_exact(name, graphs, shared_call):
    # the step increment carried by the first resolve of each step (no launch of its own): identical outputs and
    # state, and the step counter advances once per step
    w = wl.WORKLOADS[name]
    steps = 10 if name != "multilayer" else 6
    buf, ora = gh.replay(w, steps=steps, graphs=graphs, fused=True, shared_call=shared_call)
    assert int(buf.view("step").item()) == steps == ora.step
    assert int(buf.meta[8:12].view(torch.int32).item()) == 0  # the completion count is left at zero
    gh.check_hot_rows(buf, layers=[0, w.layers - 1])
    buf.close()
