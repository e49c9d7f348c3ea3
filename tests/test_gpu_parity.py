"""GPU path against the oracle, element by element, through the C ABI.

Small recipes run the oracle on every request and cover the edges: domains
shorter than k (padding), queries placed inside the history, idle slots,
union overflow of the hot cache, optional residency, ring hits after commits
over several rounds, both kv layouts, shared and per-query retrieval, and
both attention passes after a shared resolve (per query, and over the union
with query masks).  The full-size configurations run with the bench's launch
shapes and check sampled requests (every step is request-local, so a request
is checked completely).
"""
import numpy as np
import pytest

import workload as wl
from harness import build_oracle, compare_round, compare_state, oracle_round

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import hierarchical_sparse_kv_int8_gb300 as dhs
    dhs.build()
    dhs.load()


def _runner(rec, **kw):
    from hierarchical_sparse_kv_int8_gb300.runner import Runner
    return Runner(rec, **kw)


TINY_GQA = wl.Recipe("tiny_gqa", N=3, K=4, S=700, H_idx=2, d_idx=32, topk=64, Hq=8, Hkv=1,
                     qk_dim=128, v_dim=128, kv_layout=0, B=48, rho_within=0.6, rho_cross=0.7,
                     W=40, p=8, opt_frac=0.1, seed=11)
TINY_GQA2 = wl.Recipe("tiny_gqa_hkv2", N=2, K=3, S=333, H_idx=1, d_idx=48, topk=32, Hq=8, Hkv=2,
                      qk_dim=128, v_dim=128, kv_layout=0, B=20, rho_within=0.5, rho_cross=0.5,
                      W=16, p=4, seed=12)
TINY_MLA = wl.Recipe("tiny_mla", N=2, K=3, S=517, H_idx=1, d_idx=128, topk=32, Hq=16, Hkv=1,
                     qk_dim=576, v_dim=512, kv_layout=1, B=40, rho_within=0.5, rho_cross=0.6,
                     W=24, p=8, opt_frac=0.25, seed=13)
TINY_SHORT = wl.Recipe("tiny_short_history", N=2, K=2, S=45, H_idx=1, d_idx=64, topk=64, Hq=8,
                       Hkv=1, qk_dim=128, v_dim=128, kv_layout=0, B=32, rho_within=0.3,
                       rho_cross=0.5, W=8, p=4, seed=14)


# Index rows of other widths than the configurations': 16 B and 32 B (one
# thread per row, one or two chunks), 192 B (16 lanes share a row, four of
# them idle) and 768 B (32 lanes, two chunks each), with three or five queries
# (the wide rows' reduce-scatter pads them to eight).  The last recipe draws
# full-range int8 keys and queries, so every query's scores span far more
# than 2^13 values: top-k takes several radix passes and the per-CTA sort and
# merge path.
TINY_IDX16 = wl.Recipe("tiny_idx16", N=2, K=3, S=400, H_idx=1, d_idx=16, topk=64, Hq=8, Hkv=1,
                       qk_dim=128, v_dim=128, kv_layout=0, B=48, rho_within=0.5,
                       rho_cross=0.6, W=16, p=8, seed=23)
TINY_IDX32 = wl.Recipe("tiny_idx32", N=2, K=5, S=400, H_idx=2, d_idx=16, topk=64, Hq=8, Hkv=1,
                       qk_dim=128, v_dim=128, kv_layout=0, B=48, rho_within=0.5,
                       rho_cross=0.6, W=16, p=8, seed=24)
TINY_WIDE = wl.Recipe("tiny_wide_rows", N=2, K=5, S=900, H_idx=2, d_idx=96, topk=96, Hq=8,
                      Hkv=1, qk_dim=128, v_dim=128, kv_layout=0, B=64, rho_within=0.5,
                      rho_cross=0.6, W=16, p=8, seed=21)
TINY_WIDE_FULL = wl.Recipe("tiny_wide_full_range", N=2, K=3, S=1500, H_idx=4, d_idx=192,
                           topk=128, Hq=8, Hkv=1, qk_dim=128, v_dim=128, kv_layout=0, B=64,
                           rho_within=0.5, rho_cross=0.6, W=16, p=8, seed=22,
                           i8_lo=-128, i8_hi=127)

# Index rows for the remaining scoring paths: 512 B (eight 64-byte groups on
# the tensor-core path) with full-range int8 and eight queries, so a score
# reaches 2^23 in magnitude; 320 B, 256 B and 448 B (five, four and seven
# groups), 144 B and 272 B (the dp4a paths with 16 and 32 lanes per row).
TINY_TC512_FULL = wl.Recipe("tiny_tc512_full_range", N=3, K=8, S=2100, H_idx=4, d_idx=128,
                            topk=128, Hq=8, Hkv=1, qk_dim=128, v_dim=128, kv_layout=0, B=64,
                            rho_within=0.5, rho_cross=0.6, W=16, p=8, seed=31,
                            i8_lo=-128, i8_hi=127)
TINY_TC320 = wl.Recipe("tiny_tc320", N=2, K=5, S=800, H_idx=1, d_idx=320, topk=64, Hq=8,
                       Hkv=1, qk_dim=128, v_dim=128, kv_layout=0, B=48, rho_within=0.5,
                       rho_cross=0.6, W=16, p=8, seed=32, i8_lo=-128, i8_hi=127)
TINY_TC256 = wl.Recipe("tiny_tc256", N=2, K=8, S=700, H_idx=2, d_idx=128, topk=64, Hq=8,
                       Hkv=1, qk_dim=128, v_dim=128, kv_layout=0, B=48, rho_within=0.5,
                       rho_cross=0.6, W=16, p=8, seed=35, i8_lo=-128, i8_hi=127)
TINY_TC448 = wl.Recipe("tiny_tc448", N=2, K=2, S=500, H_idx=1, d_idx=448, topk=64, Hq=8,
                       Hkv=1, qk_dim=128, v_dim=128, kv_layout=0, B=48, rho_within=0.5,
                       rho_cross=0.6, W=16, p=8, seed=36)
TINY_IDX144 = wl.Recipe("tiny_idx144", N=2, K=3, S=600, H_idx=1, d_idx=144, topk=64, Hq=8,
                        Hkv=1, qk_dim=128, v_dim=128, kv_layout=0, B=48, rho_within=0.5,
                        rho_cross=0.6, W=16, p=8, seed=33)
TINY_IDX272 = wl.Recipe("tiny_idx272", N=2, K=4, S=600, H_idx=1, d_idx=272, topk=64, Hq=8,
                        Hkv=1, qk_dim=128, v_dim=128, kv_layout=0, B=48, rho_within=0.5,
                        rho_cross=0.6, W=16, p=8, seed=34)


def _rounds(rec, n_rounds, shared=True, k_sched=None, residency=True, attn_pass=0, label=""):
    run = _runner(rec, attn_pass=attn_pass)
    slots = list(range(rec.N))
    o = build_oracle(rec, slots)
    if residency and rec.opt_frac > 0:
        run.set_residency()
        for r in slots:
            o.set_residency(r, rec.residency_rows(r))
    for rnd in range(n_rounds):
        kr = rec.k_per_req() if k_sched is None else k_sched(rnd)
        acc = rec.accepted(rnd, kr)
        run.load_round(rnd)
        run.select(kr)
        run.resolve(shared)
        run.attend()
        ores = oracle_round(o, rec, rnd, slots, kr, None, shared)
        compare_round(run, o, ores, slots, kr, "%s round %d" % (label, rnd))
        run.commit(acc)
        o.commit(acc)
        compare_state(run, o, slots, "%s round %d" % (label, rnd))
    st = run.ctx.stats()
    assert st["device_error"] == 0
    return run, o, st


PER_QUERY, UNION, UNION_MMA = 1, 2, 3


@pytest.mark.parametrize("shared,attn_pass", [(True, PER_QUERY), (True, UNION), (True, UNION_MMA),
                                              (False, 0)],
                         ids=["per_query_pass", "union_tensor_cores", "union_mma_sync",
                              "per_query_retrieval"])
def test_tiny_gqa_rounds(shared, attn_pass):
    _, o, st = _rounds(TINY_GQA, 4, shared=shared, attn_pass=attn_pass, label="tiny_gqa")
    assert st["misses"] == o.stats.misses and st["hot_hits"] == o.stats.hot_hits
    assert st["ring_hits"] == o.stats.ring_hits and st["opt_hits"] == o.stats.opt_hits
    assert st["host_rows_fetched"] == o.stats.host_rows_fetched
    assert st["installs"] == o.stats.installs and st["evictions"] == o.stats.evictions
    assert st["direct_only"] == o.stats.direct_only
    assert st["selections"] == o.stats.selections
    assert st["miss_selections"] == o.stats.miss_selections
    assert o.stats.ring_hits > 0 and o.stats.opt_hits > 0 and o.stats.evictions > 0


@pytest.mark.parametrize("attn_pass", [PER_QUERY, UNION, UNION_MMA])
def test_tiny_two_kv_heads(attn_pass):
    _rounds(TINY_GQA2, 3, attn_pass=attn_pass, label="tiny_hkv2")


@pytest.mark.parametrize("attn_pass", [PER_QUERY, UNION])
def test_tiny_mla_latent(attn_pass):
    _rounds(TINY_MLA, 3, attn_pass=attn_pass, label="tiny_mla")


@pytest.mark.parametrize("rec", [TINY_IDX16, TINY_IDX32, TINY_WIDE, TINY_WIDE_FULL,
                                 TINY_TC512_FULL, TINY_TC320, TINY_IDX144, TINY_IDX272],
                         ids=["16B", "32B", "192B", "768B_full_range", "512B_full_range",
                              "320B_full_range", "144B", "272B"])
def test_index_row_widths(rec):
    if rec.i8_hi > 8:  # the full-range recipe must leave the single-pass top-k
        keys = rec.index_keys(0, 1)[0, :rec.S].astype(np.int64)
        sc = keys @ rec.index_queries(0, 0, 1)[0, 0].astype(np.int64)
        assert sc.max() - sc.min() >= 1 << 13
    _rounds(rec, 3, attn_pass=UNION, label=rec.name)


@pytest.mark.parametrize("rec", [TINY_GQA, TINY_GQA2, TINY_MLA, TINY_IDX16, TINY_WIDE,
                                 TINY_WIDE_FULL, TINY_TC512_FULL, TINY_TC320, TINY_IDX144,
                                 TINY_IDX272, TINY_TC256, TINY_TC448],
                         ids=["64B", "48B", "128B", "16B", "192B", "768B_full_range",
                              "512B_full_range", "320B_full_range", "144B", "272B",
                              "256B_full_range", "448B"])
def test_index_scores_exact(rec):
    """Every indexer score over every query's domain equals the exact integer
    dot product of eq. (1), on each scoring path."""
    from oracle.dhs_oracle import index_scores
    import torch
    run = _runner(rec)
    run.load_round(0)
    kr = rec.k_per_req()
    run.select(kr)
    ss = (rec.s_max + 31) // 32 * 32  # score rows are padded to 32
    sc = run.export("scores", torch.int32, (rec.N, run.Km, ss)).cpu().numpy()
    keys = rec.index_keys(0, rec.N)
    qi = rec.index_queries(0, 0, rec.N)
    for r in range(rec.N):
        for j in range(int(kr[r])):
            want = index_scores(qi[r, j], keys[r], rec.S)
            assert np.array_equal(sc[r, j, :rec.S].astype(np.int64), want), \
                "%s scores differ at r=%d j=%d" % (rec.name, r, j)
    assert run.ctx.stats()["device_error"] == 0


@pytest.mark.parametrize("d_idx,N,S", [(64, 64, 65536), (128, 64, 32768)], ids=["64B", "128B"])
def test_index_scores_exact_large_launch(d_idx, N, S):
    """64- and 128-byte index rows go to the tensor-core scorer once a launch
    streams 256 MB of keys or more: sampled requests' scores and top-k lists
    equal the oracle's."""
    from oracle.dhs_oracle import index_scores, topk_ordered
    import torch
    rec = wl.Recipe("large_launch_%dB_%d" % (d_idx, N), N=N, K=4, S=S, H_idx=1, d_idx=d_idx,
                    topk=256, Hq=8, Hkv=1, qk_dim=128, v_dim=128, kv_layout=0, B=64,
                    rho_within=0.5, rho_cross=0.6, W=16, p=8, seed=41, i8_lo=-128, i8_hi=127)
    key_bytes = rec.N * rec.S * rec.idx_row
    assert key_bytes >= 256 << 20
    run = _runner(rec)
    run.load_round(0)
    kr = rec.k_per_req()
    run.select(kr)
    ss = (rec.s_max + 31) // 32 * 32
    sc = run.export("scores", torch.int32, (rec.N, run.Km, ss)).cpu().numpy()
    topk = run.topk.cpu().numpy()
    qi = rec.index_queries(0, 0, rec.N)
    for r in (0, N // 2 + 5, N - 1):
        keys = rec.index_keys(r, r + 1)[0]
        for j in range(int(kr[r])):
            want = index_scores(qi[r, j], keys, rec.S)
            assert np.array_equal(sc[r, j, :rec.S].astype(np.int64), want), "r=%d j=%d" % (r, j)
            assert np.array_equal(topk[r, j], topk_ordered(want, rec.topk)), "r=%d j=%d" % (r, j)
    assert run.ctx.stats()["device_error"] == 0


@pytest.mark.parametrize("full_range", [False, True], ids=["one_pass", "multi_pass"])
def test_topk_parts_read_from_global_memory(full_range):
    """Domains whose quarter no longer fits in a top-k CTA's shared memory
    (here 40 000 scores per CTA) are read from global memory by every pass;
    with full-range int8 the scores span more than 2^13 values and the radix
    select takes several passes.  Every top-k list equals the oracle's."""
    from oracle.dhs_oracle import index_scores, topk_ordered
    kw = dict(i8_lo=-128, i8_hi=127) if full_range else {}
    rec = wl.Recipe("unstaged_%s" % ("multi" if full_range else "one"), N=2, K=2, S=160000,
                    H_idx=1, d_idx=128, topk=256, Hq=8, Hkv=1, qk_dim=128, v_dim=128,
                    kv_layout=0, B=64, rho_within=0.5, rho_cross=0.6, W=16, p=8, seed=43, **kw)
    run = _runner(rec)
    run.load_round(0)
    kr = rec.k_per_req()
    run.select(kr)
    topk = run.topk.cpu().numpy()
    qi = rec.index_queries(0, 0, rec.N)
    keys = rec.index_keys(0, rec.N)
    for r in range(rec.N):
        for j in range(int(kr[r])):
            want = index_scores(qi[r, j], keys[r], rec.S)
            assert np.array_equal(topk[r, j], topk_ordered(want, rec.topk)), "r=%d j=%d" % (r, j)
    assert run.ctx.stats()["device_error"] == 0


@pytest.mark.parametrize("rec", [TINY_TC512_FULL, TINY_GQA], ids=["512B", "64B"])
def test_index_scores_extreme_values(rec):
    """The largest magnitudes a row can produce: every product is
    (-128)(-128) or (-128)(127), so the scores are 16384 and -16256 times the
    row's bytes exactly (+2^23 and -2^23 + 65536 for 512 bytes), every row
    ties, and each top-k is the lowest rows in order."""
    import torch
    run = _runner(rec)
    run.load_round(0)
    run.keys.fill_(-128)
    run.q_idx.fill_(-128)
    run.q_idx[:, 1::2].fill_(127)
    kr = rec.k_per_req()
    run.select(kr)
    ss = (rec.s_max + 31) // 32 * 32  # score rows are padded to 32
    sc = run.export("scores", torch.int32, (rec.N, run.Km, ss)).cpu().numpy()
    topk = run.topk.cpu().numpy()
    for r in range(rec.N):
        for j in range(int(kr[r])):
            want = 16384 * rec.idx_row if j % 2 == 0 else -(128 * 127 * rec.idx_row)
            assert (sc[r, j, :rec.S] == want).all(), "r=%d j=%d" % (r, j)
            assert np.array_equal(topk[r, j], np.arange(rec.topk)), "r=%d j=%d" % (r, j)
    assert run.ctx.stats()["device_error"] == 0


@pytest.mark.parametrize("attn_pass", [PER_QUERY, UNION])
def test_history_shorter_than_k_and_idle_slots(attn_pass):
    sched = lambda rnd: np.array([2, 0] if rnd % 2 == 0 else [1, 2], np.int32)
    _rounds(TINY_SHORT, 4, k_sched=sched, attn_pass=attn_pass, label="short")


@pytest.mark.parametrize("attn_pass", [PER_QUERY, UNION])
def test_queries_inside_history(attn_pass):
    rec = TINY_GQA
    run = _runner(rec, attn_pass=attn_pass)
    slots = list(range(rec.N))
    o = build_oracle(rec, slots)
    kr = rec.k_per_req()
    pos = np.array([[5, 63, 64, 400], [0, 1, 699, 10_000], [-1, 30, 2, 100]], np.int64)
    run.load_round(0)
    run.select(kr, pos)
    run.resolve(True)
    run.attend()
    ores = oracle_round(o, rec, 0, slots, kr, None, True, pos)
    compare_round(run, o, ores, slots, kr, "pos")


def test_cfg1_full():
    rec = wl.CONFIGS["cfg1"]
    _rounds(rec, 2, label="cfg1")


@pytest.mark.parametrize("attn_pass", [0, UNION, UNION_MMA])
def test_cfg2_full(attn_pass):
    """The benchmark workload: round 0 is the previous step, round 1 is timed."""
    rec = wl.CONFIGS["cfg2"]
    _, o, st = _rounds(rec, 2, attn_pass=attn_pass, label="cfg2")
    assert o.stats.hot_hits > 0 and o.stats.misses > 0


# Sixteen query heads per kv head with the per-query pass split eight ways:
# the splits of an item merge as one cluster, each CTA finishing two heads.
CLUSTER16 = wl.Recipe("cluster_merge_16_heads", N=4, K=8, S=4096, H_idx=1, d_idx=64, topk=2048,
                      Hq=16, Hkv=1, qk_dim=128, v_dim=128, kv_layout=0, B=512,
                      rho_within=0.8, rho_cross=0.8, W=64, p=8, seed=51)


@pytest.mark.parametrize("shared", [True, False], ids=["shared", "per_query_retrieval"])
def test_cluster_merged_splits_16_heads(shared):
    _rounds(CLUSTER16, 2, shared=shared, attn_pass=PER_QUERY, label="cluster16")


def _sampled(rec, slots, rounds=2, shared=True, k_max=None, opt_rows_max=None, kr=None,
             residency=None):
    run = _runner(rec, k_max=k_max, opt_rows_max=opt_rows_max)
    o = build_oracle(rec, slots, k_max=k_max, opt_rows_max=opt_rows_max)
    if residency is not None or rec.opt_frac > 0:
        rows_of = residency or rec.residency_rows
        run.set_residency(rows_of)
        for r in slots:
            o.set_residency(r, rows_of(r))
    kr = rec.k_per_req() if kr is None else kr
    for rnd in range(rounds):
        acc = rec.accepted(rnd, kr)
        run.load_round(rnd)
        run.select(kr)
        run.resolve(shared)
        run.attend()
        ores = oracle_round(o, rec, rnd, slots, kr, None, shared)
        compare_round(run, o, ores, slots, kr, "%s round %d" % (rec.name, rnd))
        run.commit(acc)
        o.commit(acc)
        compare_state(run, o, slots, "%s round %d" % (rec.name, rnd), full_host=False)
    assert run.ctx.stats()["device_error"] == 0
    return run, o


def test_cfg3_full_sampled():
    rec = wl.CONFIGS["cfg3"]
    _sampled(rec, [0, 77, 127])


def test_cfg3_union_mma_sync_sampled():
    """The DFlash2-style configuration (a 24-request cut) with the union pass
    forced onto mma.sync tiles (the automatic choice takes the tensor-core
    pass, which the full-size sampled test covers)."""
    from hierarchical_sparse_kv_int8_gb300.runner import Runner
    rec = wl.CONFIGS["cfg3"].scaled(N=24)
    slots = [0, 23]
    run = Runner(rec, attn_pass=UNION_MMA)
    o = build_oracle(rec, slots)
    kr = rec.k_per_req()
    for rnd in range(2):
        acc = rec.accepted(rnd, kr)
        run.load_round(rnd)
        run.select(kr)
        run.resolve(True)
        run.attend()
        ores = oracle_round(o, rec, rnd, slots, kr, None, True)
        compare_round(run, o, ores, slots, kr, "cfg3 mma.sync union round %d" % rnd)
        run.commit(acc)
        o.commit(acc)
        compare_state(run, o, slots, "cfg3 mma.sync union round %d" % rnd, full_host=False)
    assert run.ctx.stats()["device_error"] == 0


def test_cfg4_full_sampled():
    rec = wl.CONFIGS["cfg4"]
    _sampled(rec, [5, 63])


def test_repeated_row_in_a_selection_is_flagged():
    """A selection is a set: a caller list that names a row twice is reported
    through the device check word (code 5), and nothing faults."""
    rec = TINY_GQA
    run = _runner(rec, attn_pass=UNION)
    kr = rec.k_per_req()
    run.load_round(0)
    run.select(kr)
    assert run.ctx.stats()["device_error"] == 0
    run.topk[1, 2, 7] = run.topk[1, 2, 3]
    run.resolve(True)
    run.attend()
    run.commit(rec.accepted(0))
    st = run.ctx.stats(check=False)
    assert st["device_error"] == 5


@pytest.mark.parametrize("attn_pass,pinned,big", [(PER_QUERY, True, False), (UNION, True, False),
                                                  (PER_QUERY, False, False), (UNION, True, True)],
                         ids=["per_query_pinned", "union_pinned", "per_query_pageable",
                              "union_pinned_20KB_index_rows"])
def test_round_through_host_buffers(attn_pass, pinned, big):
    """dhs_round_host gives the same outputs and cache state as the device
    calls, whether its host buffers are page-locked (used in place) or not
    (copied through device buffers), and whether the index rows fit in the
    indexer's launch parameters (16 KB) or go through a device buffer."""
    import torch
    rec = TINY_TC512_FULL.scaled(N=5) if big else TINY_GQA
    run = _runner(rec, attn_pass=attn_pass)
    run.set_residency()
    kr = rec.k_per_req()
    run.load_round(0)
    run.round(kr, rec.accepted(0))
    run.load_round(1)
    sid = run.ctx.snapshot()
    acc1 = rec.accepted(1)
    run.round(kr, acc1)
    want_out = run.out.cpu()
    want_lse = run.lse.cpu()
    B, N = rec.B, rec.N
    want_state = [run.export(w, torch.int32, (N, B)).cpu() for w in ("hot_row", "hot_stamp", "lru")]
    run.ctx.restore(sid)

    def host(t):
        h = t.cpu()
        return h.pin_memory() if pinned else h
    qi, q, bl = host(run.q_idx), host(run.q), host(run.block)
    out = torch.zeros(run.out.shape, dtype=run.out.dtype, pin_memory=pinned)
    lse = torch.zeros(run.lse.shape, dtype=run.lse.dtype, pin_memory=pinned)
    run.ctx.round_host(qi, kr, q, bl, acc1, out, lse)
    for r in range(N):
        for j in range(int(kr[r])):
            assert torch.equal(out[r, j], want_out[r, j]), "out r=%d j=%d" % (r, j)
            assert torch.equal(lse[r, j], want_lse[r, j]), "lse r=%d j=%d" % (r, j)
    got_state = [run.export(w, torch.int32, (N, B)).cpu() for w in ("hot_row", "hot_stamp", "lru")]
    for g, w in zip(got_state, want_state):
        assert torch.equal(g, w)
    assert run.ctx.stats()["device_error"] == 0


# ---------------------------------------------------------------- one-CTA-per-query top-k
TOPK_ROW = 2


@pytest.mark.parametrize("rec", [TINY_GQA, TINY_SHORT, TINY_WIDE_FULL, TINY_TC512_FULL],
                         ids=["64B", "short_history", "768B_full_range", "512B_full_range"])
def test_topk_row_kernel_rounds(rec):
    """The one-CTA-per-query top-k, forced on small recipes: whole rounds
    (lists, locations, outputs, cache state) equal the oracle's, including
    domains shorter than k and scores spanning more than 2^13 values."""
    from hierarchical_sparse_kv_int8_gb300.runner import Runner
    run = Runner(rec, topk_pass=TOPK_ROW)
    slots = list(range(rec.N))
    o = build_oracle(rec, slots)
    if rec.opt_frac > 0:
        run.set_residency()
        for r in slots:
            o.set_residency(r, rec.residency_rows(r))
    sched = (lambda rnd: np.array([2, 0] if rnd % 2 == 0 else [1, 2], np.int32)) \
        if rec is TINY_SHORT else (lambda rnd: rec.k_per_req())
    for rnd in range(3):
        kr = sched(rnd)
        acc = rec.accepted(rnd, kr)
        run.load_round(rnd)
        run.select(kr)
        run.resolve(True)
        run.attend()
        ores = oracle_round(o, rec, rnd, slots, kr, None, True)
        compare_round(run, o, ores, slots, kr, "%s row top-k round %d" % (rec.name, rnd))
        run.commit(acc)
        o.commit(acc)
        compare_state(run, o, slots, "%s row top-k round %d" % (rec.name, rnd))
    assert run.ctx.stats()["device_error"] == 0


# (rows of the 128-row chunks whose index is a multiple of 16 form the
# kernel's threshold sample on long domains)
ROW_SAMPLE_STRIDE = 16


def _sampled_rows(S):
    return (np.arange(S) // 128) % ROW_SAMPLE_STRIDE == 0


@pytest.mark.parametrize("S,fill,rescans",
                         [(3000, "ties", 0), (9000, "ties", 0), (160000, "one_pass", 0),
                          (160000, "multi_pass", 0), (160000, "sample_high", 4),
                          (160000, "sample_low", 4), (160000, "long_ties", 4)],
                         ids=["all_equal_collected", "all_equal_ordered_fallback",
                              "long_one_pass", "long_multi_pass", "estimate_too_high",
                              "estimate_too_low", "long_ties"])
def test_topk_row_kernel_lists(S, fill, rescans):
    """Lists of the one-CTA-per-query top-k against the oracle's ordered
    top-k: every score equal (3000 rows: all rows are candidates and sorted;
    9000 rows: too many ties for the candidate area, so the lowest rows equal
    to the threshold are placed by the ordered pass), and long domains read
    from global memory in one radix pass (uniform -8..8) or several
    (full-range int8).  Long domains first try the sampled single read; the
    last three cases defeat the sample (sampled rows scoring above the rest,
    below the rest, or a domain of ties) so that the exact passes run after
    it, which the rescan counter confirms for the four long domains."""
    import torch
    from oracle.dhs_oracle import index_scores, topk_ordered
    from hierarchical_sparse_kv_int8_gb300.runner import Runner
    kw = dict(i8_lo=-128, i8_hi=127) if fill == "multi_pass" else {}
    rec = wl.Recipe("row_topk_%s_%d" % (fill, S), N=3, K=3, S=S, H_idx=1, d_idx=128, topk=256,
                    Hq=8, Hkv=1, qk_dim=128, v_dim=128, kv_layout=0, B=64, rho_within=0.5,
                    rho_cross=0.6, W=16, p=8, seed=44, **kw)
    run = Runner(rec, topk_pass=TOPK_ROW)
    run.load_round(0)
    if fill == "ties":
        run.keys.fill_(3)
        run.q_idx.fill_(-2)
    elif fill in ("sample_high", "sample_low", "long_ties"):
        # one positive query word: a row's score is the sum of its key bytes
        run.q_idx.fill_(1)
        g = torch.Generator().manual_seed(7)
        samp = torch.from_numpy(_sampled_rows(S))
        if fill == "long_ties":
            keys = torch.full((rec.N, S, rec.idx_row), 3, dtype=torch.int8)
            keys[:, ::997] = 4  # 161 rows above a domain of ties
        else:
            high = torch.randint(0, 9, (rec.N, S, rec.idx_row), generator=g, dtype=torch.int8)
            low = torch.randint(-8, 1, (rec.N, S, rec.idx_row), generator=g, dtype=torch.int8)
            hi_rows = samp if fill == "sample_high" else ~samp
            keys = torch.where(hi_rows[None, :, None], high, low)
        run.keys[:, :S].copy_(keys.to(run.keys.device))
    kr = rec.k_per_req()
    pos = np.array([[S - 1, S // 2, 100], [S + 5, 700, 257], [0, 255, S - 2]], np.int64)
    run.ctx.reset_stats(run.stream)
    run.select(kr, pos)
    topk = run.topk.cpu().numpy()
    qi = run.q_idx.cpu().numpy()
    keys = run.keys.cpu().numpy()
    for r in range(rec.N):
        for j in range(int(kr[r])):
            dom = max(0, min(S, int(pos[r, j]) + 1))
            want = topk_ordered(index_scores(qi[r, j], keys[r], dom), rec.topk)
            assert np.array_equal(topk[r, j], want), "r=%d j=%d dom=%d" % (r, j, dom)
    st = run.ctx.stats()
    assert st["device_error"] == 0
    assert st["topk_rescans"] == rescans


# ---------------------------------------------------------------- one call per round, request groups
@pytest.mark.parametrize("rec,groups,attn_pass",
                         [(TINY_GQA, 2, PER_QUERY), (TINY_GQA, 3, UNION), (TINY_GQA2, 2, UNION),
                          (TINY_GQA, 2, UNION_MMA), (TINY_MLA, 2, 0)],
                         ids=["per_query_2", "union_tc_3", "hkv2_union_tc_2", "union_mma_2",
                              "latent_auto_2"])
def test_round_in_request_groups(rec, groups, attn_pass):
    """dhs_round issues select, resolve, attend and commit in one call, the
    request slots split into groups on internal streams (uneven groups when
    the slots do not divide) for the tensor-core union pass, as one group for
    the other passes: every round equals the oracle's, state included."""
    from hierarchical_sparse_kv_int8_gb300.runner import Runner
    run = Runner(rec, attn_pass=attn_pass, round_groups=groups)
    slots = list(range(rec.N))
    o = build_oracle(rec, slots)
    if rec.opt_frac > 0:
        run.set_residency()
        for r in slots:
            o.set_residency(r, rec.residency_rows(r))
    for rnd in range(3):
        kr = rec.k_per_req()
        if rnd == 1:
            kr = kr.copy()
            kr[0] = 0  # an idle slot in one group
        acc = rec.accepted(rnd, kr)
        run.load_round(rnd)
        run.round_fused(kr, acc)
        ores = oracle_round(o, rec, rnd, slots, kr, acc, True)
        compare_round(run, o, ores, slots, kr, "%s groups round %d" % (rec.name, rnd))
        compare_state(run, o, slots, "%s groups round %d" % (rec.name, rnd))
    st = run.ctx.stats()
    assert st["device_error"] == 0 and st["resolve_calls"] == 3


def test_cfg3_round_in_four_groups_sampled():
    """The DFlash2-style configuration in one dhs_round call with four request
    groups on internal streams: sampled requests of every group equal the oracle."""
    from hierarchical_sparse_kv_int8_gb300.runner import Runner
    rec = wl.CONFIGS["cfg3"]
    slots = [0, 40, 95, 127]
    run = Runner(rec, round_groups=4)
    o = build_oracle(rec, slots)
    kr = rec.k_per_req()
    for rnd in range(2):
        acc = rec.accepted(rnd, kr)
        run.load_round(rnd)
        run.round_fused(kr, acc)
        ores = oracle_round(o, rec, rnd, slots, kr, acc, True)
        compare_round(run, o, ores, slots, kr, "cfg3 groups round %d" % rnd)
        compare_state(run, o, slots, "cfg3 groups round %d" % rnd, full_host=False)
    assert run.ctx.stats()["device_error"] == 0


def test_round_host_in_request_groups():
    """dhs_round_host with request groups gives the outputs of the grouped
    device round (pinned host buffers used in place)."""
    import torch
    from hierarchical_sparse_kv_int8_gb300.runner import Runner
    rec = TINY_GQA
    run = Runner(rec, attn_pass=UNION, round_groups=2)
    kr = rec.k_per_req()
    run.load_round(0)
    run.round_fused(kr, rec.accepted(0, kr))
    run.load_round(1)
    sid = run.ctx.snapshot()
    acc1 = rec.accepted(1, kr)
    run.round_fused(kr, acc1)
    want_out, want_lse = run.out.cpu(), run.lse.cpu()
    run.ctx.restore(sid)
    qi, q, bl = run.q_idx.cpu().pin_memory(), run.q.cpu().pin_memory(), run.block.cpu().pin_memory()
    out = torch.zeros(run.out.shape, dtype=run.out.dtype, pin_memory=True)
    lse = torch.zeros(run.lse.shape, dtype=run.lse.dtype, pin_memory=True)
    run.ctx.round_host(qi, kr, q, bl, acc1, out, lse)
    for r in range(rec.N):
        for j in range(int(kr[r])):
            assert torch.equal(out[r, j], want_out[r, j]) and torch.equal(lse[r, j], want_lse[r, j])
    assert run.ctx.stats()["device_error"] == 0


# ---------------------------------------------------------------- index keys of kept rows
@pytest.mark.parametrize("fused", [False, True], ids=["separate_calls", "dhs_round"])
def test_kept_rows_take_their_index_keys(fused):
    """dhs_append_keys before each round's commit: the bound key buffers hold
    the block keys of the kept rows, and later rounds (which score those rows)
    equal the oracle's, through the separate calls and through dhs_round."""
    import torch
    from hierarchical_sparse_kv_int8_gb300.runner import Runner
    rec = TINY_GQA
    run = Runner(rec, attn_pass=UNION, round_groups=2 if fused else 0)
    slots = list(range(rec.N))
    o = build_oracle(rec, slots)
    bkeys = torch.zeros((rec.N, run.Km, rec.idx_row), dtype=torch.int8, device="cuda")
    for rnd in range(4):
        kr = rec.k_per_req()
        acc = rec.accepted(rnd, kr)
        bk = rec.block_index_keys(rnd, 0, rec.N)
        bkeys[:, :bk.shape[1]].copy_(torch.from_numpy(bk))
        run.load_round(rnd)
        if fused:
            run.ctx.append_keys(acc, bkeys, run.stream)
            run.round_fused(kr, acc)
        else:
            run.select(kr)
            run.resolve(True)
            run.attend()
            run.ctx.append_keys(acc, bkeys, run.stream)
            run.commit(acc)
        ores = oracle_round(o, rec, rnd, slots, kr, None, True)
        o.append_keys(acc, bk)
        o.commit(acc)
        compare_round(run, o, ores, slots, kr, "key append round %d" % rnd)
        compare_state(run, o, slots, "key append round %d" % rnd)
        keys = run.keys.cpu().numpy()
        for r in slots:
            assert np.array_equal(keys[r], o.req[r].keys), "key rows r=%d round %d" % (r, rnd)
    assert run.ctx.stats()["device_error"] == 0


# ---------------------------------------------------------------- graphs that keep launch priorities
def test_round_replayed_from_a_priority_graph():
    """dhs_graph_* capture a dhs_round (three request groups on prioritised
    streams) into a graph instantiated with the launches' priorities; replays
    from the same snapshot give the eager call's outputs and cache state."""
    import torch
    import hierarchical_sparse_kv_int8_gb300 as dhs
    from hierarchical_sparse_kv_int8_gb300.runner import Runner
    rec = TINY_GQA
    stream = torch.cuda.Stream()
    run = Runner(rec, attn_pass=UNION, round_groups=3, stream=stream)
    kr = rec.k_per_req()
    acc = rec.accepted(0, kr)
    run.load_round(0)
    sid = run.ctx.snapshot(stream)
    run.round_fused(kr, acc)
    stream.synchronize()
    names = ("hot_row", "hot_stamp", "lru")
    state = [run.export(w, torch.int32, (rec.N, rec.B)) for w in names]  # (on the runner's stream)
    stream.synchronize()
    want = [run.out.clone(), run.lse.clone()] + [t.clone() for t in state]
    run.ctx.restore(sid, stream)
    stream.synchronize()
    with dhs.Graph.capture(stream) as g:
        run.round_fused(kr, acc)
    for _ in range(2):
        run.ctx.restore(sid, stream)
        with torch.cuda.stream(stream):
            run.out.zero_()
            run.lse.zero_()
        g.replay()
        got = [run.out, run.lse] + [run.export(w, torch.int32, (rec.N, rec.B)) for w in names]
        stream.synchronize()
        for a, b in zip(got, want):
            assert torch.equal(a, b)
    g.close()
    assert run.ctx.stats()["device_error"] == 0
