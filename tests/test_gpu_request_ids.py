"""hs_resolve_ids / hs_prefetch_ids: batch row b resolves against pool request req_ids[b].

Every step resolves a random subset of the pool's requests in a random order, compared with the oracle resolving
those requests (the others get an all-padding row, which the policy leaves untouched): out_slots of every row, the
whole metadata state, the counters and the hot-buffer bytes. Some steps prefetch first (the state must equal a lone
resolve), and one extra row carries an out-of-range id, which must be rejected alone."""
import numpy as np
import pytest
import torch

import hierarchical_sparse_attention_hs_gb300 as hs
import oracle
import workload as wl
from gpu_harness import check_hot_rows, compare_state, make_pool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g

    g.build()


def test_request_ids_map_rows_to_pool_requests():
    w = wl.WORKLOADS["dsa"]
    steps = 8
    sel = wl.gen_selections(w, steps=steps)  # [steps][1][B][k]
    buf = make_pool(w)
    pool = buf.handle
    B, k = w.requests, w.topk
    ora = oracle.OraclePool(w.ctx, w.slots, w.row_bytes, 1, B, track_rows=False)
    rng = np.random.default_rng(1234)
    st = torch.cuda.Stream()
    for s in range(steps):
        n = int(rng.integers(B // 2, B + 1))
        ids = rng.permutation(B)[:n].astype(np.int32)
        rows = sel[s, 0, ids]
        bad_row = s % 3 == 1  # one more row with an id past the pool's requests
        if bad_row:
            ids = np.append(ids, np.int32(B + 5))
            rows = np.concatenate([rows, sel[s, 0, :1]])
        ids_d = torch.from_numpy(ids).cuda()
        rows_d = torch.from_numpy(np.ascontiguousarray(rows)).cuda()
        out = torch.full((len(ids), k), -7, dtype=torch.int32, device="cuda")
        prefetch = s % 2 == 0
        with torch.cuda.stream(st):
            hs.hs_step_begin(pool, st)
            if prefetch:
                hs.hs_prefetch_ids(pool, 0, len(ids), ids_d, rows_d, k, st)
            hs.hs_resolve_ids(pool, 0, len(ids), ids_d, rows_d, k, out, st)
        st.synchronize()
        full = np.full((B, k), -1, dtype=np.int32)
        full[ids[:n]] = sel[s, 0, ids[:n]]
        ora.step_begin()
        if prefetch:
            ora.resolve(0, full, None, want_slots=False)
        expect = ora.resolve(0, full, None)
        got = out.cpu().numpy()
        assert np.array_equal(got[:n], expect[ids[:n]]), f"step {s}"
        err = hs.hs_get_error(pool, clear=True)
        if bad_row:
            assert (got[n] == -1).all(), f"step {s}: the rejected row's out_slots"
            assert err == hs.HS_DEVERR_RANGE, err
        else:
            assert err == 0, err
        compare_state(buf, ora, f"step {s}")
    check_hot_rows(buf, layers=[0])
    # argument checks: no ids
    with pytest.raises(hs.HsError):
        hs.hs_resolve_ids(pool, 0, 1, 0, rows_d, k, out)
    buf.close()
    buf.host.close()
