"""bench.py's host-side bookkeeping on CPU: a committed ncu capture counts only while the kernel sources it was
taken on are unchanged (the hash it records matches), otherwise the bench line reports null; the roofline fractions
against the measured and nominal peaks; the CPU oracle's thread split; the own-pool entry's workload."""
import json

import bench
import workload as wl


def _write(tmp_path, name, payload):
    prof = tmp_path / "profiles"
    prof.mkdir(exist_ok=True)
    (prof / name).write_text(json.dumps(payload))


def test_attention_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    w = wl.WORKLOADS["mla"]
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.captured_attention_traffic(w) is None  # no capture at all
    good = {"attention_sources_sha16": bench.attention_sources_sha16(), "dram_read_bytes": 1000,
            "dram_write_bytes": 24}
    _write(tmp_path, f"hs_mla_decode_kernel_{w.name}_ncu.json", good)
    assert bench.captured_attention_traffic(w) == 1024
    _write(tmp_path, f"hs_mla_decode_kernel_{w.name}_ncu.json", dict(good, attention_sources_sha16="0" * 16))
    assert bench.captured_attention_traffic(w) is None  # taken on other sources


def test_steady_only_capture_stands_for_every_launch(tmp_path, monkeypatch):
    w = wl.WORKLOADS["dsa"]
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    cap = {"kernel_sources_sha16": bench.kernel_sources_sha16(), "dram_bytes_per_launch": {"cold": None, "steady": 77}}
    _write(tmp_path, f"hs_resolve_kernel_{w.name}_noio_ncu.json", cap)
    assert bench.captured_traffic(w, 1, 3, noio=True) == 77
    assert bench.captured_traffic(w, 1, 3) is None  # the host-link form has no capture here


def test_resolve_traffic_weights_cold_and_steady_launches(tmp_path, monkeypatch):
    w = wl.WORKLOADS["dsa"]
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    cap = {"kernel_sources_sha16": bench.kernel_sources_sha16(), "dram_bytes_per_launch": {"cold": 900, "steady": 100}}
    _write(tmp_path, f"hs_resolve_kernel_{w.name}_ncu.json", cap)
    assert bench.captured_traffic(w, 1, 3) == (900 + 3 * 100) / 4
    _write(tmp_path, f"hs_resolve_kernel_{w.name}_ncu.json", dict(cap, kernel_sources_sha16="f" * 16))
    assert bench.captured_traffic(w, 1, 3) is None


def test_committed_captures_name_their_sources():
    """Each committed capture records the hash of the sources it was taken on, and its command runs committed
    files only."""
    import os

    for name in ("hs_resolve_kernel_dsa_ncu.json", "hs_resolve_kernel_dsa_noio_ncu.json",
                 "hs_mla_decode_kernel_mla_ncu.json"):
        cap = json.load(open(os.path.join(bench.ROOT, "profiles", name)))
        key = "kernel_sources_sha16" if name.startswith("hs_resolve") else "attention_sources_sha16"
        assert len(cap[key]) == 16 and int(cap[key], 16) >= 0
        assert cap["command"].startswith("ncu ") and "--clock-control none" in cap["command"]
        assert "_work" not in cap["command"]


class _Env:
    hbm_peak = 6789.6
    hbm_src = "measured"


class _Res:
    res = None  # no resident maps


def test_only_the_plain_resolve_carries_captured_traffic(tmp_path, monkeypatch):
    """The committed captures are of the plain per-layer resolve: a full-offload pass (the gather kernel), a
    prefetch pipeline or a shared call must not borrow their DRAM bytes."""
    w = wl.WORKLOADS["dsa"]
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    cap = {"kernel_sources_sha16": bench.kernel_sources_sha16(), "dram_bytes_per_launch": {"cold": None, "steady": 100}}
    _write(tmp_path, f"hs_resolve_kernel_{w.name}_ncu.json", cap)
    rows = [(0, 1.0, None), (1, 1.0, None)]
    tot = [1000, 100, 50, 100 * w.row_bytes]
    args = (2, 2, tot, 2.0, (200.0, 200.0), _Res(), rows)
    plain = bench.roofline_of(w, {}, _Env(), *args)
    assert plain["traffic"] == 100 and plain["kernel"] == "hs_resolve_kernel"
    off = bench.roofline_of(w, {"full_offload": True}, _Env(), *args)
    assert off["traffic"] is None and off["kernel"] == "hs_gather_kernel"
    assert "hs_gather_history" in off["timing"]
    for mode in ({"prefetch": True}, {"shared_call": True}, {"tiered_frac": 0.3}):
        assert bench.roofline_of(w, mode, _Env(), *args)["traffic"] is None, mode
    assert bench.roofline_of(w, {"prefetch": True}, _Env(), *args, noio=True)["traffic"] is None


def test_hbm_fractions_against_measured_and_nominal_peaks():
    """The HBM term is reported against the measured copy peak and, beside it, the nominal rate: the same bytes over
    the same time, so the two fractions differ by exactly the ratio of the peaks."""
    w = wl.WORKLOADS["dsa"]
    rows = [(0, 1.0, None), (1, 1.0, None)]
    tot = [1000, 100, 50, 100 * w.row_bytes]
    args = (2, 2, tot, 2.0, (200.0, 200.0), _Res(), rows)
    ratio = _Env.hbm_peak / bench.HBM_NOMINAL_GBS
    io = bench.roofline_of(w, {}, _Env(), *args)
    assert abs(io["hbm_frac_of_nominal"] - io["hbm_frac"] * ratio) <= 1e-12 * io["hbm_frac"]
    noio = bench.roofline_of(w, {}, _Env(), *args, noio=True)
    assert abs(noio["frac_of_nominal"] - noio["frac"] * ratio) <= 1e-12 * noio["frac"]


def test_threaded_cpu_baseline_spreads_over_request_layers():
    """With more threads than requests the CPU oracle runs one request-layer per thread, several layers of requests
    (a workload with its own selection per layer reads each layer's)."""
    import dataclasses

    w = dataclasses.replace(wl.WORKLOADS["tiny"], requests=2, layers=4, ctx=512, slots=128, topk=16, steps=4)
    many = bench.cpu_baseline(w, budget_s=0.3, threads=8)
    assert many["cores"] == 8 and "layers 0..3" in many["sample"] and many["value"] > 0
    few = bench.cpu_baseline(w, budget_s=0.3, threads=2)
    assert few["cores"] == 2 and "layer 0 " in few["sample"]
    one = bench.cpu_baseline(w, budget_s=0.3, threads=1)
    assert one["cores"] == 1 and "single-threaded" in one["sample"]


def test_own_pool_entry_is_the_headline_workload_on_fewer_layers():
    w = bench.workload_of("shared_own16")
    head = wl.WORKLOADS[bench.HEADLINE[0]]
    assert w.layers == bench.OWN_POOL_LAYERS < head.layers
    assert (w.requests, w.ctx, w.topk, w.slots, w.row_bytes, w.shared_across_layers) == (
        head.requests, head.ctx, head.topk, head.slots, head.row_bytes, head.shared_across_layers)
    assert ("shared_own16", {"prefetch": True}) in bench.DEFAULT_SET
