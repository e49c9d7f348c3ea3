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


def _noalloc_vs_oracle(n_q, n_rows, row_bytes, topk, seed, lo=-8, hi=8):
    """dhs_select_noalloc on seeded keys and queries against the oracle's
    exact scores and ordered top-k, query by query."""
    import torch
    import hierarchical_sparse_kv_int8_gb300 as dhs
    from oracle.dhs_oracle import index_scores, topk_ordered

    dhs.build()
    keys = wl.i8(n_rows * row_bytes, seed, 1, 0, lo, hi).reshape(n_rows, row_bytes)
    q = wl.i8(n_q * row_bytes, seed, 2, 0, lo, hi).reshape(n_q, row_bytes)
    got = torch.full((n_q, topk), -7, dtype=torch.int32, device="cuda")
    dhs.select_noalloc(torch.from_numpy(q).cuda(), torch.from_numpy(keys).cuda(), n_q, n_rows,
                       row_bytes, topk, got)
    got = got.cpu().numpy()
    for j in range(n_q):
        sc = index_scores(q[j], keys, n_rows)
        want = topk_ordered(sc, topk)
        assert np.array_equal(got[j], want), "query %d differs from the oracle" % j
    return keys, q


@pytest.mark.parametrize("row_bytes", [16, 128, 1024])
def test_noalloc_full_range_multi_pass(row_bytes):
    """Full-range int8 keys and queries: every query's scores span more than
    2^13 values, so the radix select takes several passes; rows of 16, 128 and
    1024 bytes cover the shared-memory rotation for 1, 8 and 64 chunks."""
    n_rows = {16: 60000, 128: 40000, 1024: 6000}[row_bytes]
    keys, q = _noalloc_vs_oracle(8, n_rows, row_bytes, 2048, seed=61 + row_bytes,
                                 lo=-128, hi=127)
    sc = keys.astype(np.int64) @ q[0].astype(np.int64)
    assert sc.max() - sc.min() >= 1 << 13


def test_noalloc_domain_shorter_than_k():
    """n_rows < topk: every row is kept, ordered, and the list is padded with -1."""
    _noalloc_vs_oracle(3, 3000, 64, 4096, seed=71)


def test_noalloc_topk_4096():
    """The largest list (4096 entries, beyond the context's 2048), over a
    domain larger than it, with many ties (narrow int8 range)."""
    _noalloc_vs_oracle(5, 200000, 64, 4096, seed=72)


def test_noalloc_capacity_edge():
    """n_queries * n_rows = 2^21 fills the fixed scratch exactly and is
    served; one row more is refused with DHS_ERR_CAPACITY before any launch."""
    import torch
    import hierarchical_sparse_kv_int8_gb300 as dhs
    _noalloc_vs_oracle(8, 1 << 18, 16, 256, seed=73)
    keys = torch.zeros(((1 << 21) + 1, 16), dtype=torch.int8, device="cuda")
    q = torch.zeros((1, 16), dtype=torch.int8, device="cuda")
    out = torch.zeros((1, 256), dtype=torch.int32, device="cuda")
    with pytest.raises(dhs.DhsError) as e:
        dhs.select_noalloc(q, keys, 1, (1 << 21) + 1, 16, 256, out)
    assert e.value.code == 3
