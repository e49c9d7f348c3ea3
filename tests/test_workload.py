"""The seeded input generators: determinism, slicing, value ranges, and the
sharing structure each configuration names (measured with the oracle)."""
import numpy as np
import pytest

import oracle
import workload as wl


def test_slices_regenerate_identically():
    rec = wl.CONFIGS["cfg2"].scaled(S=1000, s_slack=24)
    full = rec.index_keys(0, 8)
    assert np.array_equal(full[5:7], rec.index_keys(5, 7))
    h = rec.host_rows(0, 8)
    assert np.array_equal(h[3:4], rec.host_rows(3, 4))
    q = rec.index_queries(1, 0, 8)
    assert np.array_equal(q[2:5], rec.index_queries(1, 2, 5))


def test_thread_count_does_not_change_values():
    a = np.empty(300000, np.uint16)
    b = np.empty(300000, np.uint16)
    wl._load().wl_gen_bf16_normal(a.ctypes.data, a.size, 7, 3, 11, 1)
    wl._load().wl_gen_bf16_normal(b.ctypes.data, b.size, 7, 3, 11, 13)
    assert np.array_equal(a, b)


def test_int8_uniform_range():
    x = wl.i8(200000, 0, 1)
    assert x.min() == -8 and x.max() == 8
    counts = np.bincount(x.astype(np.int64) + 8, minlength=17)
    assert counts.min() > 0.9 * x.size / 17 and counts.max() < 1.1 * x.size / 17


def test_bf16_normal_moments():
    v = wl.bf16_to_f64(wl.bf16_bits(400000, 0, 2))
    assert abs(v.mean()) < 0.01 and abs(v.var() - 1.0) < 0.02
    assert np.abs(v).max() < 5.0
    # bf16 rounding is to nearest even of the single-precision value
    raw = np.float32(1.0)
    assert wl.bf16_to_f64(np.array([0x3F80], np.uint16))[0] == float(raw)


def test_residency_rows_are_whole_pages():
    rec = wl.CONFIGS["cfg4"].scaled(S=64 * 100, N=2)
    rows = rec.residency_rows(1)
    assert len(rows) == 10 * 64
    assert np.all(np.diff(rows) > 0)
    pages = rows.reshape(-1, 64)
    assert np.all(pages % 64 == np.arange(64)[None, :])


def test_accepted_range():
    rec = wl.CONFIGS["cfg3"]
    a = rec.accepted(1)
    assert a.min() >= 0 and a.max() <= rec.K and len(np.unique(a)) == rec.K + 1


def _overlaps(rec, rnd_a, rnd_b, nreq):
    keys = rec.index_keys(0, nreq)
    qa, qb = rec.index_queries(rnd_a, 0, nreq), rec.index_queries(rnd_b, 0, nreq)
    sel = lambda q, r: set(oracle.topk_ordered(oracle.index_scores(q, keys[r], rec.S), rec.topk))
    cross, within = [], []
    for r in range(nreq):
        sb = [sel(qb[r, j], r) for j in range(rec.K)]
        for j in range(rec.K):
            cross.append(len(sel(qa[r, j], r) & sb[j]) / rec.topk)
            within += [len(sb[j] & sb[i]) / rec.topk for i in range(j)]
    return np.mean(cross), (np.mean(within) if within else None)


def test_cfg2_sharing_structure():
    cross, within = _overlaps(wl.CONFIGS["cfg2"], 0, 1, 4)
    assert 0.6 < cross < 0.8      # ~70% overlap with the previous selection
    assert 0.5 < within < 0.7     # queries of a request share ~60% of rows


def test_cfg1_previous_step_overlap():
    cross, _ = _overlaps(wl.CONFIGS["cfg1"], 0, 1, 1)
    assert 0.4 < cross < 0.6      # hot cache seeded with ~50% of the previous top-k
