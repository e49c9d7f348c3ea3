"""The residency policy ("Adaptive DHiSparse", section 3.1, eq. (3) and (4))
carried out on a GPU context: the library's dhs_policy_* calls decide how
many optional pages each admitted request holds (checked decision by
decision against the oracle's policy), the test turns each decision into
dhs_set_residency calls between verification rounds (a reclaimed request's
optional set is cleared before the new request's pages are written;
repopulated pages are added), and every round is compared with the oracle
run on the same optional sets: selections, locations, union and miss lists,
optional/hot/host counts, outputs and cache state.  Rows made optional are
attended from the pool, so a row published before its bytes had landed would
show as a wrong output; the pool rows are also compared with the host rows
directly.
"""
import numpy as np
import pytest

import workload as wl
from harness import build_oracle, compare_round, compare_state, oracle_round
from oracle.dhs_oracle import ResidencyPolicy

pytestmark = pytest.mark.gpu

# 4 slots, 40 pages of 16 rows of history each; hot cache 64 rows (4 pages)
# and ring 64 rows (4 pages) are each request's required pages.
REC = wl.Recipe("policy_driven", N=4, K=3, S=640, H_idx=1, d_idx=64, topk=64, Hq=8, Hkv=1,
                qk_dim=128, v_dim=128, kv_layout=0, B=64, rho_within=0.6, rho_cross=0.7,
                W=32, p=16, opt_frac=1.0, seed=17)
HIST_PAGES = REC.S // REC.p
REQUIRED = 8


def _rows(pages):
    return np.arange(pages * REC.p, dtype=np.int32)


def test_policy_decisions_carried_out_between_rounds():
    import torch
    import hierarchical_sparse_kv_int8_gb300 as dhs
    from hierarchical_sparse_kv_int8_gb300.runner import Runner

    dhs.build()
    run = Runner(REC)
    slots = list(range(REC.N))
    o = build_oracle(REC, slots)
    lib, ref = dhs.Policy(80, 8), ResidencyPolicy(80, 8)
    held = {}          # request -> optional pages it holds now
    active = set()
    rnd = [0]

    def apply(r, pages):
        held[r] = pages
        rows = _rows(pages)
        run.ctx.set_residency(r, rows)
        o.set_residency(r, rows)

    def admit(r):
        got = lib.admit(r, REQUIRED, HIST_PAGES)
        assert got == ref.admit(r, REQUIRED, HIST_PAGES)
        ok, opt, reclaimed = got
        assert ok
        for q in reclaimed:            # reclaim first: the pages go to r
            apply(q, 0)
        apply(r, opt)
        active.add(r)
        return reclaimed

    def round_():
        kr = np.array([REC.K if r in active else 0 for r in slots], np.int32)
        acc = REC.accepted(rnd[0], kr)
        run.ctx.reset_stats()
        before = vars(o.stats).copy()
        run.load_round(rnd[0])
        run.select(kr)
        run.resolve(True)
        run.attend()
        ores = oracle_round(o, REC, rnd[0], slots, kr, None, True)
        compare_round(run, o, ores, slots, kr, "policy round %d" % rnd[0])
        run.commit(acc)
        o.commit(acc)
        compare_state(run, o, slots, "policy round %d" % rnd[0])
        st = run.ctx.stats()
        delta = {k: v - before[k] for k, v in vars(o.stats).items()}
        for k in ("opt_hits", "hot_hits", "misses", "host_rows_fetched", "direct_only"):
            assert st[k] == delta[k], (k, st[k], delta[k])
        rnd[0] += 1
        return st

    admit(0)                                     # 40 optional pages: whole history
    assert held[0] == HIST_PAGES
    admit(1)                                     # the 16 pages left
    assert held[1] == 16
    st1 = round_()
    assert st1["opt_hits"] > 0
    assert admit(2) == [0]                       # deficit 8: request 0 is reclaimed
    assert held == {0: 0, 1: 16, 2: 32}
    st2 = round_()
    assert st2["misses"] > 0
    # request 0's rows now come from the hot cache or the host
    lib.complete(1)
    ref.complete(1)
    active.discard(1)
    apply(1, 0)
    given = lib.repopulate(20)
    assert given == ref.repopulate(20)
    assert given and sum(g for _, g in given) == 20
    for r, g in given:
        apply(r, held[r] + g)
    for r in active:
        assert lib.query(r)[1] == held[r]
    round_()
    # pool slot i of each request holds row i of its optional set
    pool = run.export("opt", torch.int16, (REC.N, REC.opt_rows_max, REC.row_elems)).cpu().numpy()
    for r in active:
        n = held[r] * REC.p
        assert np.array_equal(pool[r, :n].view(np.uint16), o.req[r].host[:n])
    assert run.ctx.stats()["device_error"] == 0
