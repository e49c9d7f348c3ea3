"""Pins of the oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: every expected value is a
number printed on the pages (tests/golden/*.json, each with its citation), a
brute-force enumeration on tiny inputs, a closed form, an invariant, or a
library routine computing the same quantity by another route.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import HOT, OPT, RING, STAGE, Config, Oracle, decode_loc, encode_loc

GOLD = os.path.join(os.path.dirname(__file__), "golden")
PAGES = json.load(open(os.path.join(GOLD, "pages_worked_examples.json")))
GiB = float(1 << 30)


# ---------------------------------------------------------------- sizing (3.4)
def test_ring_rows_worked_example():
    g = PAGES["ring_rows"]
    assert oracle.ring_rows(g["W"], g["p"], g["K_max"]) == g["R_d"]


def test_ring_rows_covers_window_and_block():
    # eq. (9): whole pages holding the window, the block and p-1 alignment rows
    for W, p, K in itertools.product([1, 63, 64, 2048, 4000], [1, 16, 64], [1, 4, 8]):
        R = oracle.ring_rows(W, p, K)
        assert R % p == 0 and W + K + p - 1 <= R < W + K + 2 * p - 1


def test_ring_bytes_example():
    g = PAGES["ring_bytes"]
    R = PAGES["ring_rows"]["R_d"]
    assert round(g["slots"] * R * g["row_bytes"] / GiB, 2) == g["GiB"]


def test_staging_example():
    g = PAGES["staging"]
    four = oracle.staging_bytes(g["chi"], g["N"], g["K_max"], g["k"], g["d_kv"]) / GiB
    all_ = oracle.staging_bytes(g["chi_all"], g["N"], g["K_max"], g["k"], g["d_kv"]) / GiB
    assert round(four, 2) == g["GiB"]
    assert round(all_, 1) == g["GiB_all"]
    assert all_ / four == g["ratio"]


def test_per_session_state():
    g, s, r = PAGES["per_session"], PAGES["staging"], PAGES["ring_rows"]
    ring = r["R_d"] * PAGES["ring_bytes"]["row_bytes"]
    stage = oracle.staging_bytes(s["chi"], 1, s["K_max"], s["k"], s["d_kv"])
    assert round((ring + stage) / GiB, 3) == g["GiB"]
    assert round(g["table1_with"] - g["table1_without"], 3) == g["GiB"]


def test_fig8_payload_and_shared_identity():
    g = PAGES["fig8_payload"]
    one = g["requests"] * g["k"] * g["row_bytes"] / 1e6
    assert round(one, 2) == g["MB_one"]
    assert round(8 * one) == g["MB_eight"]
    s = PAGES["shared_retrieval"]
    assert round(100 * (1 - 1 / s["selections_per_row"])) == s["saving_pct"]


def test_ring_address_disjoint():
    # eq. (10): live positions of one slot (span < R_d) never share a row, slots are disjoint
    R = oracle.ring_rows(64, 16, 4)
    for n in [0, 5, R - 3, 3 * R + 7]:
        live = range(max(0, n - 64), n + 4)
        addrs = [oracle.ring_address(2, t, R) for t in live]
        assert len(set(addrs)) == len(addrs)
        assert all(2 * R <= a < 3 * R for a in addrs)


# ---------------------------------------------------------------- selection
def test_index_scores_naive_loop():
    rng = np.random.default_rng(1)
    H, D, S = 3, 5, 11
    q = rng.integers(-128, 128, H * D, dtype=np.int64).astype(np.int8)
    keys = rng.integers(-128, 128, (S, H * D), dtype=np.int64).astype(np.int8)
    got = oracle.index_scores(q, keys, 9)
    for s in range(9):
        want = 0
        for h in range(H):
            for d in range(D):
                want += int(q[h * D + d]) * int(keys[s][h * D + d])
        assert got[s] == want
    assert got.shape == (9,)


def _is_topk(scores, sel, k):
    """The defining property: every kept row beats every dropped row under
    (score desc, row asc), kept rows are listed in that order, and the list
    has min(k, n) entries followed by -1 padding."""
    n = len(scores)
    m = min(k, n)
    kept = [int(s) for s in sel[:m]]
    if any(s != -1 for s in sel[m:]) or len(set(kept)) != m or not all(0 <= s < n for s in kept):
        return False
    beats = lambda a, b: scores[a] > scores[b] or (scores[a] == scores[b] and a < b)
    dropped = set(range(n)) - set(kept)
    if any(not beats(a, b) for a in kept for b in dropped):
        return False
    return all(beats(kept[i], kept[i + 1]) for i in range(m - 1))


@pytest.mark.parametrize("seed", range(40))
def test_topk_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(0, 40))
    k = int(rng.integers(1, 12))
    scores = rng.integers(-3, 4, n).astype(np.int64)  # many ties
    sel = oracle.topk_ordered(scores, k)
    assert sel.shape == (k,)
    assert _is_topk(scores, sel, k)


def test_topk_all_ties_takes_lowest_rows():
    sel = oracle.topk_ordered(np.zeros(100, np.int64), 7)
    assert list(sel) == list(range(7))


def test_topk_k_covers_domain():
    sel = oracle.topk_ordered(np.array([5, -1, 5, 9], np.int64), 6)
    assert list(sel) == [3, 0, 2, 1, -1, -1]


def test_select_constant_keys_ties():
    # constant keys: every row scores the same, so each query takes its lowest rows
    c = _tiny_cfg(topk=4, n_slots=1, k_max=2)
    o = Oracle(c)
    keys = np.ones((c.s_max, c.idx_heads * c.idx_dim), np.int8)
    o.bind(0, _host(c, 0), keys, 12)
    q = np.ones((1, 2, c.idx_heads * c.idx_dim), np.int8)
    sel = o.select(q, np.array([2], np.int32), pos=np.array([[12, 2]]))
    assert list(sel[0, 0]) == [0, 1, 2, 3]
    assert list(sel[0, 1]) == [0, 1, 2, -1]   # domain of a query at position 2 is rows 0..2


# ---------------------------------------------------------------- helpers
def _tiny_cfg(**kw):
    base = dict(n_slots=2, k_max=4, topk=3, s_max=40, idx_heads=2, idx_dim=4, q_heads=4, Hkv=2,
                qk_dim=8, v_dim=8, kv_layout=0, budget=4, ring_window=8, page_rows=4,
                opt_rows_max=8)
    base.update(kw)
    return Config(**base)


def _host(c, seed):
    rng = np.random.default_rng(100 + seed)
    vals = rng.standard_normal((c.s_max, c.row_elems)).astype(np.float32)
    return (vals.view(np.uint32) >> 16).astype(np.uint16)


def _bf16(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------- union / misses (eq. 6, Fig. 3)
def test_fig3_shared_retrieval_one_copy_per_row():
    g = PAGES["fig3_shared"]
    c = _tiny_cfg(n_slots=1, k_max=g["K"], topk=g["k"], budget=16)
    o = Oracle(c)
    o.bind(0, _host(c, 0), np.zeros((c.s_max, 8), np.int8), 30)
    a, b = 10, 11
    sel = np.array([[[a, 1, 2], [a, b, 3], [a, b, 4], [5, 6, 7]]], np.int64)
    o.req[0].K = 4
    o.resolve(sel, shared=True)
    assert sum(1 for j in range(4) for s in sel[0, j] if s == a) == g["a_selected_by"]
    assert sum(1 for j in range(4) for s in sel[0, j] if s == b) == g["b_selected_by"]
    assert list(o.misses[0]) == [1, 2, 3, 4, 5, 6, 7, a, b]
    assert o.stats.host_rows_fetched == 9           # each distinct row once
    # every query that selected a gets the same location
    la = {int(o.loc[0, j, i]) for j in range(4) for i in range(3) if sel[0, j, i] == a}
    assert len(la) == 1
    o2 = Oracle(c)
    o2.bind(0, _host(c, 0), np.zeros((c.s_max, 8), np.int8), 30)
    o2.req[0].K = 4
    o2.resolve(sel, shared=False)
    assert o2.stats.host_rows_fetched == 12         # one fetch per selection
    # the per-query baseline leaves the same cache state
    assert list(o.req[0].hot_row) == list(o2.req[0].hot_row)
    # per-query placement: selection (j, i) of a missing row is fetched into
    # staging row j*k + i, and that row holds the original c_s (eq. 11)
    for j in range(4):
        for i in range(3):
            assert decode_loc(int(o2.loc[0, j, i])) == (STAGE, j * 3 + i)
            assert np.array_equal(o2.staging[0][j * 3 + i], o2.req[0].host[int(sel[0, j, i])])
    o2.check_placement()
    o.check_placement()


def test_direct_only_means_every_row_resolved_in_step_one():
    """Fig. 2: steps 2 and 3 (hot-cache scan, host fetch) are skipped only
    when every selected row of the request resolves in step 1 (the live ring
    tail or the ready optional map).  Random rounds on a tiny source; the
    count is checked against set membership computed here, by brute force."""
    rng = np.random.default_rng(7)
    K, k, n0 = 2, 3, 24
    c = _tiny_cfg(n_slots=3, k_max=K, topk=k, budget=4, ring_window=6, s_max=64,
                  opt_rows_max=12)
    o = Oracle(c)
    for r in range(3):
        o.bind(r, _host(c, r), np.zeros((c.s_max, 8), np.int8), n0)
    want, seen_direct, seen_other = 0, 0, 0
    for rnd in range(40):
        sel = np.full((3, K, k), -1, np.int64)
        step1 = {}
        for r in range(3):
            q = o.req[r]
            q.K = K
            ring = set(range(max(q.ring_first, q.n - c.ring_window), q.n))
            step1[r] = ring | set(q.opt_slot)
            pool = sorted(step1[r]) if rng.random() < 0.5 and step1[r] else list(range(q.n))
            for j in range(K):
                m = min(int(rng.integers(1, k + 1)), len(pool))
                sel[r, j, :m] = rng.choice(pool, m, replace=False)
        before = o.stats.direct_only
        o.resolve(sel, shared=True)
        for r in range(3):
            U = set(int(x) for x in sel[r].reshape(-1) if x >= 0)
            d = U <= step1[r]
            want += d
            seen_direct += d
            seen_other += not d
        assert o.stats.direct_only == want
        o.attend(np.zeros((3, K, c.q_heads, c.qk_dim), np.uint16),
                 np.zeros((3, K, c.row_elems), np.uint16))
        o.commit(np.full(3, int(rng.integers(0, K + 1))))
        if rnd % 5 == 0:
            for r in range(3):
                rows = rng.choice(o.req[r].n, 8, replace=False).astype(np.int32)
                o.set_residency(r, rows)
    assert seen_direct > 10 and seen_other > 10


@pytest.mark.parametrize("seed", range(12))
def test_union_and_miss_set_invariants(seed):
    rng = np.random.default_rng(seed)
    K, k, B, n = 4, 6, 8, 30
    c = _tiny_cfg(n_slots=1, k_max=K, topk=k, budget=B, ring_window=5, s_max=48, opt_rows_max=6)
    o = Oracle(c)
    host = _host(c, seed)
    o.bind(0, host, np.zeros((c.s_max, 8), np.int8), n)
    # previous traffic fills the cache; commits put rows into the ring
    for rnd in range(3):
        sel = np.full((1, K, k), -1, np.int64)
        for j in range(K):
            m = int(rng.integers(0, k + 1))
            sel[0, j, :m] = rng.choice(o.req[0].n, m, replace=False)
        o.req[0].K = K
        before_hot = set(int(x) for x in o.req[0].hot_row if x >= 0)
        ring_lo = max(o.req[0].ring_first, o.req[0].n - c.ring_window)
        ring = set(range(ring_lo, o.req[0].n))
        opt = set(o.req[0].opt_slot)
        loc = o.resolve(sel, shared=True)
        U = set(int(s) for s in sel[0].reshape(-1) if s >= 0)
        assert list(o.union[0]) == sorted(U)                          # eq. (6)
        assert len(U) <= K * k                                        # |U| <= K k
        D = U - ring - opt - before_hot
        assert list(o.misses[0]) == sorted(D)                         # D = U \ R, ascending
        assert all(0 <= d < o.req[0].n for d in D)                    # D in H: host copy exists
        # protected rows: no hot row of U was evicted
        after = set(int(x) for x in o.req[0].hot_row if x >= 0)
        assert (before_hot & U) <= after
        assert len(after) <= B
        # promoted = min(|D|, B - |hot rows in U|)
        assert len(after - before_hot) == min(len(D), B - len(before_hot & U))
        o.check_placement()                                           # eq. (11)
        # shared fetches never exceed per-query fetches
        assert len(D) <= sum(1 for j in range(K) for s in sel[0, j] if s >= 0 and int(s) in D)
        q = _bf16(rng.standard_normal((1, K, c.q_heads, c.qk_dim)))
        blk = _bf16(rng.standard_normal((1, K, c.row_elems)))
        o.attend(q, blk)
        o.commit(np.array([int(rng.integers(0, K + 1))]))
        if rnd == 1:
            o.set_residency(0, np.array([0, 1, 2, 3], np.int32))


def test_disjoint_queries_shared_equals_independent():
    c = _tiny_cfg(n_slots=1, k_max=3, topk=4, budget=4)
    sel = np.array([[[0, 1, 2, 3], [4, 5, 6, 7], [8, 9, 10, 11]]], np.int64)
    fetched = []
    for shared in (True, False):
        o = Oracle(c)
        o.bind(0, _host(c, 0), np.zeros((c.s_max, 8), np.int8), 20)
        o.req[0].K = 3
        o.resolve(sel, shared=shared)
        fetched.append(o.stats.host_rows_fetched)
    assert fetched[0] == fetched[1] == 12


# ---------------------------------------------------------------- LRU hand-worked trace
def test_lru_hand_trace():
    g = json.load(open(os.path.join(GOLD, "lru_trace.json")))
    tiers = {"RING": RING, "OPT": OPT, "HOT": HOT, "STAGE": STAGE}
    c = _tiny_cfg(n_slots=1, k_max=2, topk=3, budget=g["budget"], s_max=16, opt_rows_max=2)
    o = Oracle(c)
    o.bind(0, _host(c, 0), np.zeros((c.s_max, 8), np.int8), g["n"])
    for st in g["steps"]:
        if st["opt"]:
            o.set_residency(0, np.array(st["opt"], np.int32))
        sel = np.full((1, 2, 3), -1, np.int64)
        for j, s in enumerate(st["sel"]):
            sel[0, j] = s
        o.req[0].K = len(st["sel"])
        loc = o.resolve(sel, shared=True)
        assert o.t == st["t"]
        for j, row in enumerate(st["loc"]):
            assert [decode_loc(int(x)) for x in loc[0, j]] == [(tiers[a], b) for a, b in row]
        assert list(o.req[0].hot_row) == st["rows"]
        assert list(o.req[0].hot_stamp) == st["stamps"]
        assert list(o.misses[0]) == st["misses"]
        o.check_placement()
        o.attend(np.zeros((1, 2, c.q_heads, c.qk_dim), np.uint16), np.zeros((1, 2, c.row_elems), np.uint16))
        o.commit(np.array([0]))
        for v, row in enumerate(st["rows"]):      # installed payload is the original row
            if row >= 0:
                assert np.array_equal(o.req[0].hot_payload[v], o.req[0].host[row])


# ---------------------------------------------------------------- attention
def _dense_reference(c, host, n, block, qa, j, h):
    """Dense causal attention by torch's scaled_dot_product_attention (float64):
    the query at position n + j sees history 0..n-1 and block rows 0..j."""
    torch = pytest.importorskip("torch")
    seq = np.concatenate([host[:n], block[:j + 1]])
    R = oracle.bf16_to_f64(seq)
    Kh, Vh = oracle.split_row(R, h // (c.q_heads // c.Hkv), c)
    q = torch.tensor(oracle.bf16_to_f64(qa), dtype=torch.float64)[None, None, None, :]
    out = torch.nn.functional.scaled_dot_product_attention(
        q, torch.tensor(Kh)[None, None], torch.tensor(Vh)[None, None], scale=c.scale)
    return out[0, 0, 0].numpy()


@pytest.mark.parametrize("layout", [0, 1])
def test_topk_equal_history_is_dense_causal_attention(layout):
    n, K = 13, 3
    if layout == 0:
        c = _tiny_cfg(n_slots=1, k_max=K, topk=n, kv_layout=0)
    else:
        c = _tiny_cfg(n_slots=1, k_max=K, topk=n, kv_layout=1, Hkv=1, qk_dim=12, v_dim=8)
    rng = np.random.default_rng(7)
    o = Oracle(c)
    host = _host(c, 3)
    keys = rng.integers(-8, 9, (c.s_max, c.idx_heads * c.idx_dim)).astype(np.int8)
    o.bind(0, host.copy(), keys, n)
    qi = rng.integers(-8, 9, (1, K, c.idx_heads * c.idx_dim)).astype(np.int8)
    sel = o.select(qi, np.array([K], np.int32))
    o.resolve(sel)
    qa = _bf16(rng.standard_normal((1, K, c.q_heads, c.qk_dim)))
    blk = _bf16(rng.standard_normal((1, K, c.row_elems)))
    out, lse = o.attend(qa, blk)
    for j in range(K):
        for h in range(c.q_heads):
            want = _dense_reference(c, host, n, blk[0], qa[0, j, h], j, h)
            np.testing.assert_allclose(out[0, j, h], want, rtol=1e-12, atol=1e-12)


def test_attention_two_rows_closed_form():
    # one selected row and the anchor's own block row: softmax over two logits
    c = _tiny_cfg(n_slots=1, k_max=1, topk=1, Hkv=1, q_heads=1)
    o = Oracle(c)
    host = _host(c, 5)
    o.bind(0, host, np.zeros((c.s_max, 8), np.int8), 10)
    o.req[0].K = 1
    o.resolve(np.array([[[4]]], np.int64))
    rng = np.random.default_rng(3)
    qa = _bf16(rng.standard_normal((1, 1, 1, c.qk_dim)))
    blk = _bf16(rng.standard_normal((1, 1, c.row_elems)))
    out, lse = o.attend(qa, blk)
    qv = oracle.bf16_to_f64(qa[0, 0, 0])
    r1, r2 = oracle.bf16_to_f64(host[4]), oracle.bf16_to_f64(blk[0, 0])
    a, b = c.scale * qv.dot(r1[:8]), c.scale * qv.dot(r2[:8])
    wa, wb = math.exp(a), math.exp(b)
    want = (wa * r1[8:16] + wb * r2[8:16]) / (wa + wb)
    np.testing.assert_allclose(out[0, 0, 0], want, rtol=1e-13)
    assert abs(lse[0, 0, 0] - math.log(wa + wb)) < 1e-12


def test_attention_equal_keys_is_mean_of_values():
    c = _tiny_cfg(n_slots=1, k_max=2, topk=5, Hkv=1, q_heads=2)
    host = _host(c, 9)
    host[:, :8] = _bf16(np.full(8, 0.5))          # identical keys everywhere
    o = Oracle(c)
    o.bind(0, host, np.zeros((c.s_max, 8), np.int8), 20)
    o.req[0].K = 2
    sel = np.array([[[3, 7, 1, 12, 5], [2, 4, 6, 8, -1]]], np.int64)
    o.resolve(sel)
    blk = _bf16(np.random.default_rng(2).standard_normal((1, 2, c.row_elems)))
    blk[0, :, :8] = host[0, :8]
    qa = _bf16(np.random.default_rng(4).standard_normal((1, 2, 2, c.qk_dim)))
    out, _ = o.attend(qa, blk)
    V = oracle.bf16_to_f64(host[:, 8:16])
    VB = oracle.bf16_to_f64(blk[0, :, 8:16])
    want0 = (V[[3, 7, 1, 12, 5]].sum(0) + VB[0]) / 6
    want1 = (V[[2, 4, 6, 8]].sum(0) + VB[:2].sum(0)) / 6
    np.testing.assert_allclose(out[0, 0, 0], want0, rtol=1e-13)
    np.testing.assert_allclose(out[0, 1, 1], want1, rtol=1e-13)


def test_attention_selection_order_irrelevant():
    c = _tiny_cfg(n_slots=1, k_max=1, topk=6)
    host = _host(c, 11)
    qa = _bf16(np.random.default_rng(5).standard_normal((1, 1, c.q_heads, c.qk_dim)))
    blk = _bf16(np.random.default_rng(6).standard_normal((1, 1, c.row_elems)))
    outs = []
    for perm in ([9, 2, 14, 0, 5, 7], [7, 5, 0, 14, 2, 9]):
        o = Oracle(c)
        o.bind(0, host, np.zeros((c.s_max, 8), np.int8), 20)
        o.req[0].K = 1
        o.resolve(np.array([[perm]], np.int64))
        outs.append(o.attend(qa, blk)[0])
    np.testing.assert_allclose(outs[0], outs[1], rtol=1e-13)


# ---------------------------------------------------------------- commit / rollback (eq. 7, 9, 10)
def test_fig3_commit_example():
    g = PAGES["fig3_commit"]
    c = _tiny_cfg(n_slots=1, k_max=g["K"], topk=2)
    o = Oracle(c)
    host = _host(c, 1)
    orig = host.copy()
    n = 17
    o.bind(0, host, np.zeros((c.s_max, 8), np.int8), n)
    o.req[0].K = g["K"]
    o.resolve(np.array([[[1, 2]] * g["K"]], np.int64))
    blk = _bf16(np.random.default_rng(8).standard_normal((1, g["K"], c.row_elems)))   # D, E, F, G
    o.attend(np.zeros((1, g["K"], c.q_heads, c.qk_dim), np.uint16), blk)
    kept = 1 + g["A"]                     # anchor D plus accepted E, F
    assert kept == g["kept"]
    o.commit(np.array([kept]))
    assert o.req[0].n == n + 1 + g["A"]
    live = o.ring_live(0)
    assert sorted(live) == [n, n + 1, n + 2]
    for u in range(3):
        assert np.array_equal(live[n + u], blk[0, u])
        assert np.array_equal(o.req[0].host[n + u], blk[0, u])
    assert np.array_equal(o.req[0].host[n + 3], orig[n + 3])   # G never published


@pytest.mark.parametrize("a", [1, 2, 3, 4])
def test_rollback_equals_never_staging_rejected(a):
    c = _tiny_cfg(n_slots=1, k_max=4, topk=2, ring_window=6)
    blk = _bf16(np.random.default_rng(9).standard_normal((1, 4, c.row_elems)))
    states = []
    for K in (4, a):
        o = Oracle(c)
        o.bind(0, _host(c, 2), np.zeros((c.s_max, 8), np.int8), 11)
        for rnd in range(3):              # several rounds wrap the ring window
            o.req[0].K = K
            o.resolve(np.array([[[0, 1]] * 4], np.int64))
            o.attend(np.zeros((1, 4, c.q_heads, c.qk_dim), np.uint16), blk)
            o.commit(np.array([a]))
        states.append((o.req[0].n, o.ring_live(0), o.req[0].host.copy()))
    assert states[0][0] == states[1][0]
    assert sorted(states[0][1]) == sorted(states[1][1])
    for t in states[0][1]:
        assert np.array_equal(states[0][1][t], states[1][1][t])
    assert np.array_equal(states[0][2], states[1][2])


def test_commit_validation():
    c = _tiny_cfg(n_slots=1, k_max=4, topk=2)
    o = Oracle(c)
    o.bind(0, _host(c, 2), np.zeros((c.s_max, 8), np.int8), 11)
    o.req[0].K = 2
    with pytest.raises(ValueError):
        o.commit(np.array([3]))
    with pytest.raises(ValueError):
        o.set_residency(0, np.array([1, 1], np.int32))
    with pytest.raises(ValueError):
        o.set_residency(0, np.arange(9, dtype=np.int32))


def test_location_encoding_roundtrip():
    for tier in (RING, OPT, HOT, STAGE):
        for idx in (0, 1, 12345, (1 << 28) - 1):
            l = encode_loc(tier, idx)
            assert l >= 0 and decode_loc(l) == (tier, idx)


# ---------------------------------------------------------------- source sharing (2.2, 3.2)
def _direct_attention(c, rows, block, q, j):
    """softmax(scale K q) V over the given original rows then block rows 0..j,
    written out in float64 here (per query head)."""
    R = oracle.bf16_to_f64(np.concatenate([rows, block[:j + 1]]))
    outs = []
    for h in range(c.q_heads):
        Kh, Vh = oracle.split_row(R, h // (c.q_heads // c.Hkv), c)
        lg = c.scale * (Kh @ oracle.bf16_to_f64(q[h]))
        w = np.exp(lg - lg.max())
        outs.append(w @ Vh / w.sum())
    return np.stack(outs)


def test_follower_attends_its_own_rows_at_the_producers_positions():
    """GLM-style index sharing (3.2): a follower payload layer takes the
    positions a producer selected, fetches its own rows for them and attends
    over its own bytes."""
    rng = np.random.default_rng(3)
    K, k = 3, 5
    c = _tiny_cfg(n_slots=1, k_max=K, topk=k, budget=4, s_max=48)
    prod, foll = Oracle(c), Oracle(c)
    prod.bind(0, _host(c, 1), rng.integers(-8, 9, (c.s_max, 8)).astype(np.int8), 30)
    foll.bind(0, _host(c, 2), np.zeros((c.s_max, 8), np.int8), 30)
    qi = rng.integers(-8, 9, (1, K, 8)).astype(np.int8)
    sel = prod.select(qi, np.array([K]))
    foll.adopt(sel, np.array([K]))
    foll.resolve(sel)
    foll.check_placement()                     # eq. (11) against the follower's own rows
    q = _bf16(rng.standard_normal((1, K, c.q_heads, c.qk_dim)))
    blk = _bf16(rng.standard_normal((1, K, c.row_elems)))
    out, _ = foll.attend(q, blk)
    host = foll.req[0].host
    for j in range(K):
        rows = host[[int(s) for s in sel[0, j] if s >= 0]]
        assert np.allclose(out[0, j], _direct_attention(c, rows, blk[0], q[0, j], j), atol=1e-12)
    assert not np.array_equal(_host(c, 1), host)   # the producer's bytes were not used


def test_reindex_fetches_only_rows_absent_after_the_first_selection():
    """A Reindex layer (2.2, 3.2) selects again over the shared source before
    the step commits: its misses are exactly its union less the rows ready
    after the first layer's update (ring, optional, hot rows including the
    first layer's promotions), and rows the first layer fetched and promoted
    are hits for it."""
    rng = np.random.default_rng(11)
    K, k, B = 2, 6, 10
    c = _tiny_cfg(n_slots=1, k_max=K, topk=k, budget=B, s_max=64, ring_window=6)
    o = Oracle(c)
    o.bind(0, _host(c, 4), np.zeros((c.s_max, 8), np.int8), 40)
    for step in range(6):
        q = o.req[0]
        q.K = K
        sel1 = np.full((1, K, k), -1, np.int64)
        for j in range(K):
            sel1[0, j] = rng.choice(q.n, k, replace=False)
        o.resolve(sel1)
        o.attend(np.zeros((1, K, c.q_heads, c.qk_dim), np.uint16), np.zeros((1, K, c.row_elems), np.uint16))
        ready = set(int(x) for x in q.hot_row if x >= 0) | set(q.opt_slot) | \
            set(range(max(q.ring_first, q.n - c.ring_window), q.n))
        sel2 = np.full((1, K, k), -1, np.int64)
        for j in range(K):
            # half the rows of the first selection, half fresh
            keep = rng.choice(sel1[0, j], k // 2, replace=False)
            rest = rng.choice(np.setdiff1d(np.arange(q.n), keep), k - k // 2, replace=False)
            sel2[0, j] = np.concatenate([keep, rest])
        q.K = K
        o.resolve(sel2)
        U2 = set(int(s) for s in sel2[0].reshape(-1))
        assert list(o.misses[0]) == sorted(U2 - ready)
        o.check_placement()
        o.attend(np.zeros((1, K, c.q_heads, c.qk_dim), np.uint16), np.zeros((1, K, c.row_elems), np.uint16))
        o.commit(np.array([int(rng.integers(0, K + 1))]))


def test_reuse_consumer_attends_the_inherited_rows():
    """A Reuse layer (2.2, 3.2) consumes the preceding selected-location
    vector with its own queries: its output is attention over the original
    rows of that selection (eq. 11), with no further resolution."""
    rng = np.random.default_rng(5)
    K, k = 3, 4
    c = _tiny_cfg(n_slots=1, k_max=K, topk=k, budget=3, s_max=40)
    o = Oracle(c)
    o.bind(0, _host(c, 6), rng.integers(-8, 9, (c.s_max, 8)).astype(np.int8), 25)
    sel = o.select(rng.integers(-8, 9, (1, K, 8)).astype(np.int8), np.array([K]))
    o.resolve(sel)
    blk = _bf16(rng.standard_normal((1, K, c.row_elems)))
    calls = o.stats.misses
    for layer in range(2):
        q = _bf16(rng.standard_normal((1, K, c.q_heads, c.qk_dim)))
        out, _ = o.attend(q, blk)
        for j in range(K):
            rows = o.req[0].host[[int(s) for s in sel[0, j] if s >= 0]]
            assert np.allclose(out[0, j], _direct_attention(c, rows, blk[0], q[0, j], j), atol=1e-12)
    assert o.stats.misses == calls and o.t == 1   # no second resolution


# ---------------------------------------------------------------- index keys of kept rows (3.3 with 2.2)
def test_kept_rows_join_the_history_with_their_index_keys():
    """Kept rows join the history with the index keys the target computed
    for them: key row n_r + u becomes block key u (u < a_r), earlier rows and
    rows past the kept prefix are untouched, and the next round ranks those
    rows by their keys.  The block keys here point along the sign of the next
    round's first query with the largest int8 magnitude, so each kept row
    reaches the maximum possible score 8 * sum|q| (computed here by hand), and
    the query's list starts with exactly the kept rows in row order."""
    rng = np.random.default_rng(11)
    c = _tiny_cfg(n_slots=2, k_max=3, topk=6, s_max=48, budget=8)
    row = c.idx_heads * c.idx_dim
    o = Oracle(c)
    keys = [rng.integers(-8, 9, (c.s_max, row)).astype(np.int8) for _ in range(2)]
    for r in range(2):
        o.bind(r, _host(c, r), keys[r], 30)
    q0 = rng.integers(-8, 9, (2, c.k_max, row)).astype(np.int8)
    q1 = rng.integers(-8, 9, (2, c.k_max, row)).astype(np.int8)
    q1[:, 0, 0] = 5  # (no all-zero query)
    kr = np.array([3, 2], np.int32)
    sel = o.select(q0, kr)
    o.resolve(sel, shared=True)
    o.attend(np.zeros((2, c.k_max, c.q_heads, c.qk_dim), np.uint16),
             np.zeros((2, c.k_max, c.row_elems), np.uint16))
    acc = np.array([2, 1], np.int32)
    block = np.zeros((2, c.k_max, row), np.int8)
    for r in range(2):
        block[r, :] = (8 * np.sign(q1[r, 0].astype(np.int64))).astype(np.int8)
    before = [k.copy() for k in keys]
    o.append_keys(acc, block)
    o.commit(acc)
    for r in range(2):
        a = int(acc[r])
        assert np.array_equal(keys[r][:30], before[r][:30])
        assert np.array_equal(keys[r][30:30 + a], block[r, :a])
        assert np.array_equal(keys[r][30 + a:], before[r][30 + a:])
        assert o.req[r].n == 30 + a
    sel1 = o.select(q1, np.array([1, 1], np.int32))
    for r in range(2):
        a = int(acc[r])
        top = 8 * sum(abs(int(x)) for x in q1[r, 0])
        for u in range(a):  # the kept rows' scores, element by element
            assert sum(int(q1[r, 0, e]) * int(keys[r][30 + u, e]) for e in range(row)) == top
        assert list(sel1[r, 0, :a]) == [30 + u for u in range(a)]
    with pytest.raises(ValueError):
        o.append_keys(np.array([4, 0]), block)  # more rows than the block holds


# ---------------------------------------------------------------- compressed sources, eq. (8)
def test_rows_completed_by_a_round_eq8():
    """[ADHS] eq. (8): with m positions per stored row, committing a of the
    block's positions from token frontier n completes the rows
    floor(n/m) <= s < floor((n+a)/m).  Worked by hand: 5 -> 12 with m = 4
    completes rows 1 and 2 (positions 4..11); 8 -> 11 completes none (row 2
    still lacks position 11); 7 -> 8 completes row 1; m = 1 completes exactly
    the kept positions."""
    from oracle.dhs_oracle import completed_rows, domain_length
    assert list(completed_rows(5, 7, 4)) == [1, 2]
    assert list(completed_rows(8, 3, 4)) == []
    assert list(completed_rows(7, 1, 4)) == [1]
    assert list(completed_rows(10, 0, 4)) == []
    assert list(completed_rows(9, 4, 1)) == [9, 10, 11, 12]
    # a query at position p sees the complete rows whose positions are all <= p
    assert domain_length(10, 17, 4) == 4     # rows 0..3 hold positions 0..15; row 4 ends at 19
    assert domain_length(10, 19, 4) == 5
    assert domain_length(3, 40, 4) == 3      # capped by the complete history
    assert domain_length(10, 2, 4) == 0


def test_compressed_source_rounds():
    """A source with m = 3: each round's commit publishes exactly the rows
    eq. (8) completes, with the compressor's payload and keys; the partial
    group stays out of every domain; the ring serves no history row (every
    union row resolves through the hot cache or the host); with m = 1 the
    compressed commit given the block rows leaves the host backing of the
    ordinary commit."""
    rng = np.random.default_rng(3)
    for m in (3, 1):
        c = _tiny_cfg(n_slots=2, k_max=4, topk=6, s_max=48, budget=6, tokens_per_row=m)
        row = c.idx_heads * c.idx_dim
        o = Oracle(c)
        ref = Oracle(_tiny_cfg(n_slots=2, k_max=4, topk=6, s_max=48, budget=6)) if m == 1 else None
        n_tok = [30, 31] if m == 3 else [10, 11]
        for r in range(2):
            keys = rng.integers(-8, 9, (c.s_max, row)).astype(np.int8)
            host = _host(c, r)
            o.bind(r, host.copy(), keys.copy(), n_tok[r])
            if ref:
                ref.bind(r, host.copy(), keys.copy(), n_tok[r])
            assert o.req[r].n == n_tok[r] // m
        for rnd in range(5):
            qi = rng.integers(-8, 9, (2, c.k_max, row)).astype(np.int8)
            kr = np.array([4, 3], np.int32)
            sel = o.select(qi, kr)
            for r in range(2):
                assert sel[r].max() < o.req[r].n  # only complete rows are selectable
            o.resolve(sel, shared=True)
            assert o.stats.ring_hits == 0 or m == 1
            qa = rng.standard_normal((2, c.k_max, c.q_heads, c.qk_dim)).astype(np.float32)
            bl = rng.standard_normal((2, c.k_max, c.row_elems)).astype(np.float32)
            o.attend(_bf16(qa), _bf16(bl))
            acc = rng.integers(0, kr + 1).astype(np.int32)
            cm = (c.k_max + m - 1) // m
            rows = _bf16(rng.standard_normal((2, cm, c.row_elems)))
            rkeys = rng.integers(-8, 9, (2, cm, row)).astype(np.int8)
            before = [(q.tok, q.n, q.host.copy(), q.keys.copy()) for q in (o.req[0], o.req[1])]
            if m == 1:
                ref.select(qi, kr)
                ref.resolve(sel, shared=True)
                ref.attend(_bf16(qa), _bf16(bl))
                ref.commit(acc)
                rows = np.stack([np.stack([ref.req[r].host[before[r][0] + u] if u < acc[r]
                                           else np.zeros(c.row_elems, np.uint16)
                                           for u in range(cm)]) for r in range(2)])
            o.commit_compressed(acc, rows, rkeys)
            for r in range(2):
                tok0, n0, host0, keys0 = before[r]
                q = o.req[r]
                done = list(range(tok0 // m, (tok0 + int(acc[r])) // m))
                assert q.tok == tok0 + int(acc[r]) and q.n == q.tok // m
                assert q.n == (done[-1] + 1 if done else n0)
                for i, s in enumerate(done):
                    assert np.array_equal(q.host[s], rows[r, i])
                    assert np.array_equal(q.keys[s], rkeys[r, i])
                keep = np.ones(c.s_max, bool)
                keep[done] = False
                assert np.array_equal(q.host[keep], host0[keep])
                assert np.array_equal(q.keys[keep], keys0[keep])
                if ref:
                    assert np.array_equal(q.host, ref.req[r].host)
    with pytest.raises(ValueError):
        Oracle(_tiny_cfg(tokens_per_row=2)).commit(np.zeros(2, np.int32))
