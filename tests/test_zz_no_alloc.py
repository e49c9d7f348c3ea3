"""dhs_select_noalloc, the entry point for callers that cannot allocate.

Callers recording a CUDA graph, plug-ins in engines that own all device
memory, or decode loops that must not synchronise on cudaMalloc use this
call; it keeps its scratch in a fixed array of the library image.  This test
calls it through the C ABI twice in a row (different queries, different
numbers of rows, so stale scratch from the first call would show) and
checks each result against the context-based dhs_select, which must agree
exactly (selections are integer results).  It lives in its own file, named
to be collected last.
"""
import numpy as np
import pytest

import workload as wl

pytestmark = pytest.mark.gpu


def test_noalloc_select_matches_context_select_twice():
    import torch
    import hierarchical_sparse_kv_int8_gb300 as dhs

    dhs.build()
    rec = wl.CONFIGS["cfg2"].scaled(N=1)
    S, E, K, k = rec.S, rec.idx_row, rec.K, rec.topk
    keys = torch.from_numpy(rec.index_keys(0, 1)[0]).cuda()
    host = torch.zeros((rec.s_max, rec.row_elems), dtype=torch.int16, pin_memory=True)
    cfg = dhs.make_config(n_slots=1, k_max=K, topk=k, s_max=rec.s_max, idx_heads=rec.H_idx,
                          idx_dim=rec.d_idx, q_heads=rec.Hq, kv_heads=rec.Hkv, qk_dim=rec.qk_dim,
                          v_dim=rec.v_dim, kv_layout=rec.kv_layout, budget=rec.B,
                          ring_window=rec.W, page_rows=rec.p, opt_rows_max=0)
    ctx = dhs.Context(cfg)
    ctx.bind(0, host, keys, S)
    kr = np.array([K], np.int32)
    for call, (rnd, n_rows) in enumerate([(0, S), (1, S - 4999)]):
        qi = torch.from_numpy(rec.index_queries(rnd, 0, 1)).cuda()
        want = torch.full((1, K, k), -1, dtype=torch.int32, device="cuda")
        pos = np.full((1, K), n_rows - 1, np.int64)   # every query sees rows [0, n_rows)
        ctx.select(qi, kr, want, pos)
        ctx.resolve(want, torch.empty_like(want))
        ctx.attend(torch.zeros((1, K, rec.Hq, rec.qk_dim), dtype=torch.int16, device="cuda"),
                   torch.zeros((1, K, rec.row_elems), dtype=torch.int16, device="cuda"),
                   torch.full_like(want, -1),
                   torch.empty((1, K, rec.Hq, rec.v_dim), dtype=torch.bfloat16, device="cuda"))
        ctx.commit(np.zeros(1, np.int32))
        got = torch.full((K, k), -7, dtype=torch.int32, device="cuda")
        dhs.select_noalloc(qi[0], keys, K, n_rows, E, k, got)
        torch.cuda.synchronize()
        assert torch.equal(got, want[0]), "call %d differs from dhs_select" % call
    assert ctx.stats()["device_error"] == 0
