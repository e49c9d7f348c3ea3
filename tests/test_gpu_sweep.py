"""The load-adaptive sweep's shapes (the DFlash2-style configuration: 128
requests, S = 102400, four indexer heads of 128, top-k 2048, GQA 16/1) at the
points where its behaviour changes, against the oracle on sampled requests
through the C ABI:

- 100% optional residency: every selected row resolves in step 1 of Fig. 2
  (ring tail or optional map), so nothing is fetched from the host and every
  request counts as direct-only;
- 25% residency with K = 1 (non-speculative decode on a partly resident
  history);
- per-query (independent) retrieval at K = 8, where each missing selection is
  fetched on its own.

One context at full size (optional pool for the whole history) serves all
three; each test binds every slot again first.
"""
import numpy as np
import pytest

import workload as wl
from harness import build_oracle, compare_round, compare_state, oracle_round

pytestmark = pytest.mark.gpu

SLOTS = [0, 61, 127]


@pytest.fixture(scope="module")
def full_run():
    import hierarchical_sparse_kv_int8_gb300 as dhs
    from hierarchical_sparse_kv_int8_gb300.runner import Runner
    dhs.build()
    rec = wl.sweep_recipe(1.0)
    run = Runner(rec)
    yield run
    run.ctx.close()


def _sweep_rounds(run, rec, rows_of, kr, shared, rounds=2):
    """Rounds 0 (the previous step) and 1 on the GPU and on the oracle for the
    sampled slots, compared element by element; returns the oracle and the
    library's counters."""
    run.rebind()
    run.ctx.reset_stats()
    o = build_oracle(rec, SLOTS, k_max=run.Km, opt_rows_max=run.cfg.opt_rows_max)
    # the LRU clock belongs to the source and keeps running across binds:
    # start the oracle's where the context's stands
    o.t = run.ctx.stats()["resolve_calls"]
    if rows_of is not None:
        run.set_residency(rows_of)
        for r in SLOTS:
            o.set_residency(r, rows_of(r))
    for rnd in range(rounds):
        acc = rec.accepted(rnd, kr)
        run.load_round(rnd)
        run.select(kr)
        run.resolve(shared)
        run.attend()
        ores = oracle_round(o, rec, rnd, SLOTS, kr, None, shared)
        compare_round(run, o, ores, SLOTS, kr, "%s round %d" % (rec.name, rnd))
        run.commit(acc)
        o.commit(acc)
        compare_state(run, o, SLOTS, "%s round %d" % (rec.name, rnd), full_host=False)
    st = run.ctx.stats()
    assert st["device_error"] == 0
    return o, st


def test_full_residency_every_lookup_direct(full_run):
    rec = wl.sweep_recipe(1.0)
    all_rows = np.arange(rec.S, dtype=np.int32)
    o, st = _sweep_rounds(full_run, rec, lambda r: all_rows, rec.k_per_req(), True)
    # Fig. 2: every request skips the hot scan and the host fetch, every round
    assert st["misses"] == 0 and st["host_rows_fetched"] == 0 and st["hot_hits"] == 0
    assert st["direct_only"] == 2 * rec.N
    assert o.stats.direct_only == 2 * len(SLOTS) and o.stats.misses == 0


def test_quarter_residency_single_query(full_run):
    rec25 = wl.sweep_recipe(0.25)
    kr = np.ones(rec25.N, np.int32)
    o, st = _sweep_rounds(full_run, rec25, rec25.residency_rows, kr, True)
    assert o.stats.opt_hits > 0 and o.stats.misses > 0 and o.stats.hot_hits > 0
    frac = st["host_rows_fetched"] / st["selections"]
    assert 0.3 < frac < 0.9, frac  # about three quarters of the first round miss


def test_per_query_retrieval_eight_queries(full_run):
    rec0 = wl.sweep_recipe(0.0)
    o, st = _sweep_rounds(full_run, rec0, None, rec0.k_per_req(), False)
    # each missing selection is fetched on its own: fetched = missing selections
    assert st["host_rows_fetched"] == st["miss_selections"] > st["misses"]
    assert o.stats.host_rows_fetched == o.stats.miss_selections
