"""The link probe that allocates nothing (hs_probe_link_static), against the ordinary one (hs_probe_link).

Some callers cannot allocate device memory: plain C code linking only this library (it has the page-locked host
memory of hs_host_alloc, but no device allocator), or a component whose framework hands out no scratch. The ordinary
probe needs a caller-provided device buffer that serves only as scratch; the allocation-free one uses a fixed 16 MiB
array inside the library instead. Both time the same two transfers over the same host buffer, so their results agree
within the spread of link measurements on this machine (35 %: they also differ in the clock, events against device
clock stamps); checked on two calls in a row, since the second call reuses the scratch and its looked-up address.
Sizes beyond the fixed scratch are refused with their own error code before anything runs.

This file is collected last (its name sorts after every other test file), so a run that stops at its first failure
has already run everything else; it also passes on its own in a fresh process.
"""
import pytest
import torch

import hierarchical_sparse_attention_hs_gb300 as hs

pytestmark = pytest.mark.gpu

TOLERANCE = 0.35  # relative difference allowed between two measurements of the same link


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g

    g.build()


def test_static_probe_agrees_with_the_ordinary_probe_on_two_calls():
    n = 16 << 20  # the whole fixed scratch
    host = hs.HostBuffer(n)
    host.numpy()[:] = 0x3C
    dev = torch.empty(n, dtype=torch.uint8, device="cuda")  # the ordinary probe's scratch, from the test's allocator
    for call in range(2):
        zc_static, cp_static = hs.hs_probe_link_static(host.ptr, n, 8)
        zc, cp = hs.hs_probe_link(host.ptr, dev, n, 8)
        for name, got, ref in (("zero-copy", zc_static, zc), ("memcpy", cp_static, cp)):
            assert 1.0 < got < 5000.0, (call, name, got)
            assert abs(got - ref) <= TOLERANCE * ref, (call, name, got, ref)
    torch.cuda.synchronize()
    host.close()


def test_static_probe_refuses_sizes_beyond_its_scratch():
    n = 16 << 20
    host = hs.HostBuffer(n + 4096)
    for bad in (n + 16, n + 4096):
        with pytest.raises(hs.HsError) as e:
            hs.hs_probe_link_static(host.ptr, bad, 1)
        assert e.value.code == hs.HS_ERR_TOO_LARGE
        assert "16 MiB" in str(e.value)
    with pytest.raises(hs.HsError) as e:
        hs.hs_probe_link_static(host.ptr, n - 8, 1)  # not a multiple of 16
    assert e.value.code == hs.HS_ERR_INVALID_ARG
    zc, cp = hs.hs_probe_link_static(host.ptr, 1 << 20, 2)  # a smaller size still works afterwards
    assert zc > 0 and cp > 0
    torch.cuda.synchronize()
    host.close()
