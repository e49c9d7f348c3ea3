"""Shared pieces of the GPU parity tests: build the oracle over the same seeded
inputs as a Runner, run rounds on both, and compare.

Bars (stated by the benchmark spec for this path): selections, locations, union and miss
lists, hot-cache and ring state bit-exact; attention outputs within max abs
2e-2 and max rel 1e-2, where "rel" is read per (request, query, head) output
vector as ||gpu - oracle||_inf / max(||oracle||_inf, 1e-6) (elementwise
relative error is ill-posed for outputs near zero).  The lse is held to the
same absolute bound.
"""
from __future__ import annotations

import numpy as np

import oracle
from oracle import HOT, INDEX_MASK, OPT, RING, STAGE, TIER_SHIFT

ABS_TOL = 2e-2
REL_TOL = 1e-2


def oracle_config(rec, k_max=None, opt_rows_max=None):
    return oracle.Config(n_slots=rec.N, k_max=k_max or rec.kmax, topk=rec.topk, s_max=rec.s_max,
                         idx_heads=rec.H_idx, idx_dim=rec.d_idx, q_heads=rec.Hq, Hkv=rec.Hkv,
                         qk_dim=rec.qk_dim, v_dim=rec.v_dim, kv_layout=rec.kv_layout,
                         budget=rec.B, ring_window=rec.W, page_rows=rec.p,
                         opt_rows_max=rec.opt_rows_max if opt_rows_max is None else opt_rows_max,
                         tokens_per_row=rec.m)


def build_oracle(rec, slots, k_max=None, opt_rows_max=None):
    o = oracle.Oracle(oracle_config(rec, k_max, opt_rows_max))
    for r in slots:
        o.bind(r, rec.host_rows(r, r + 1)[0], rec.index_keys(r, r + 1)[0], rec.S * rec.m)
    return o


def oracle_inputs(rec, rnd, slots, Km):
    """Round inputs of the sampled slots, laid out [N][Km][...] like the device buffers."""
    N = rec.N
    qi = np.zeros((N, Km, rec.idx_row), np.int8)
    qa = np.zeros((N, Km, rec.Hq, rec.qk_dim), np.uint16)
    bl = np.zeros((N, Km, rec.row_elems), np.uint16)
    for r in slots:
        qi[r, :rec.kmax] = rec.index_queries(rnd, r, r + 1)[0]
        qa[r, :rec.kmax] = rec.attn_queries(rnd, r, r + 1)[0]
        bl[r, :rec.kmax] = rec.block_rows(rnd, r, r + 1)[0]
    return qi, qa, bl


def oracle_round(o, rec, rnd, slots, k_per_req, accepted=None, shared=True, pos=None):
    Km = o.cfg.k_max
    qi, qa, bl = oracle_inputs(rec, rnd, slots, Km)
    kr = np.asarray(k_per_req, np.int32)
    sel = o.select(qi, kr, pos)
    o.resolve(sel, shared=shared)
    o.check_placement()
    out, lse = o.attend(qa, bl)
    res = dict(topk=sel.copy(), loc=o.loc.copy(), out=out, lse=lse,
               union={r: o.union[r].copy() for r in slots if r in o.union},
               misses={r: o.misses[r].copy() for r in slots if r in o.misses},
               staging={r: o.staging[r].copy() for r in slots if r in o.staging})
    if accepted is not None:
        o.commit(accepted)
    return res


def bf16_bits_to_f64(t):
    """bfloat16 torch tensor -> float64 numpy."""
    return t.float().cpu().numpy().astype(np.float64)


def compare_outputs(gpu_out, gpu_lse, ores, slots, k_per_req, label=""):
    worst_abs, worst_rel = 0.0, 0.0
    for r in slots:
        for j in range(int(k_per_req[r])):
            g = gpu_out[r, j]
            w = ores["out"][r, j]
            err = np.abs(g - w)
            worst_abs = max(worst_abs, float(err.max()))
            rel = err.max(axis=1) / np.maximum(np.abs(w).max(axis=1), 1e-6)
            worst_rel = max(worst_rel, float(rel.max()))
            lerr = np.abs(gpu_lse[r, j] - ores["lse"][r, j]).max()
            assert lerr <= ABS_TOL, "%s lse err %g at r=%d j=%d" % (label, lerr, r, j)
    assert worst_abs <= ABS_TOL, "%s max abs err %g" % (label, worst_abs)
    assert worst_rel <= REL_TOL, "%s max rel err %g" % (label, worst_rel)
    return worst_abs, worst_rel


def compare_round(run, o, ores, slots, k_per_req, label="", check_staging=True):
    """Selections, locations, union/miss lists, counts and outputs of one
    round (staging rows too, unless another source has reused the staging
    arena since: the outputs already show what attention read there)."""
    topk = run.topk.cpu().numpy()
    loc = run.loc.cpu().numpy()
    rec = run.rec
    KK = run.Km * rec.topk
    uni = run.export("union", run.torch.int32, (rec.N, KK)).cpu().numpy()
    mis = run.export("miss", run.torch.int32, (rec.N, KK)).cpu().numpy()
    cnt = run.export("counts", run.torch.int32, (rec.N, 4)).cpu().numpy()
    for r in slots:
        K = int(k_per_req[r])
        for j in range(K):
            assert np.array_equal(topk[r, j], ores["topk"][r, j]), \
                "%s topk differs at r=%d j=%d" % (label, r, j)
            assert np.array_equal(loc[r, j], ores["loc"][r, j]), \
                "%s loc differs at r=%d j=%d" % (label, r, j)
        if K:
            U, M = int(cnt[r, 0]), int(cnt[r, 1])
            assert np.array_equal(uni[r, :U], ores["union"][r]), "%s union r=%d" % (label, r)
            assert np.array_equal(mis[r, :M], ores["misses"][r]), "%s misses r=%d" % (label, r)
    # every staging row a location names holds the host row it stands for
    stage = run.export("stage", run.torch.int16, (rec.N, KK, rec.row_elems))  # stays on device
    for r in slots:
        K = int(k_per_req[r])
        if not K or r not in ores["staging"] or not check_staging:
            continue
        lr = ores["loc"][r, :K].reshape(-1)
        lr = lr[lr >= 0]
        idx = np.unique(lr[(lr >> TIER_SHIFT) == STAGE] & INDEX_MASK)
        if idx.size:
            got = stage[r][run.torch.from_numpy(idx).to(stage.device)].cpu().numpy()
            assert np.array_equal(got.view(np.uint16), ores["staging"][r][idx]), \
                "%s staging rows r=%d" % (label, r)
    out = bf16_bits_to_f64(run.out)
    lse = run.lse.cpu().numpy().astype(np.float64)
    return compare_outputs(out, lse, ores, slots, k_per_req, label)


def compare_state(run, o, slots, label="", full_host=True):
    """Hot cache (row, stamp, payload, LRU order), frontier, live ring rows and
    host backing of the sampled slots."""
    torch, rec = run.torch, run.rec
    N, B, row = rec.N, rec.B, rec.row_elems
    hot_row = run.export("hot_row", torch.int32, (N, B)).cpu().numpy()
    hot_stamp = run.export("hot_stamp", torch.int32, (N, B)).cpu().numpy()
    lru = run.export("lru", torch.int32, (N, B)).cpu().numpy()
    front = run.export("frontier", torch.int64, (N,)).cpu().numpy()
    hot_data = run.export("hot_data", torch.int16, (N, B, row))
    ring = run.export("ring", torch.int16, (N, run.ctx.ring_rows, row))
    for r in slots:
        q = o.req[r]
        assert np.array_equal(hot_row[r], q.hot_row), "%s hot rows r=%d" % (label, r)
        assert np.array_equal(hot_stamp[r], q.hot_stamp), "%s hot stamps r=%d" % (label, r)
        order = np.lexsort((np.arange(B), hot_stamp[r]))
        assert np.array_equal(lru[r], order), "%s lru order r=%d" % (label, r)
        assert front[r] == q.n, "%s frontier r=%d" % (label, r)
        hd = hot_data[r].cpu().numpy().view(np.uint16)
        filled = q.hot_row >= 0
        assert np.array_equal(hd[filled], q.hot_payload[filled]), "%s hot payload r=%d" % (label, r)
        rg = ring[r].cpu().numpy().view(np.uint16)
        for t, want in o.ring_live(r).items():
            assert np.array_equal(rg[t % run.ctx.ring_rows], want), "%s ring t=%d r=%d" % (label, t, r)
        hb = run.host[r].numpy().view(np.uint16)
        lo = 0 if full_host else rec.S
        assert np.array_equal(hb[lo:q.n], q.host[lo:q.n]), "%s host backing r=%d" % (label, r)
