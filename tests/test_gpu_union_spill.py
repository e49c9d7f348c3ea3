"""Union/probe slices whose union outgrows the slice's shared-memory area:
such a slice keeps its union rows, their locations and query masks in a
global scratch area of its own.  Crafted index keys make every query select
rows of one or two slices of the history, so that those slices hold several
thousand union rows; whole rounds (selections, union and miss lists,
locations, staged rows, outputs, cache state) equal the oracle's."""
import numpy as np
import pytest

import workload as wl
from harness import compare_round, compare_state, oracle_config, oracle_inputs

pytestmark = pytest.mark.gpu

SLICES = 7  # history slices of the union/probe (one per non-leader CTA of its cluster)


def _slice_rows(s_max):
    return (((s_max + SLICES - 1) // SLICES) + 31) & ~31


def _crafted(rec, rows_of):
    """Index keys and queries under which query j's top-k is exactly
    rows_of(j): key byte j of those rows is 1, query j's byte j is 100, every
    other byte 0 (score 100 for the chosen rows, 0 for the rest)."""
    keys = np.zeros((rec.N, rec.s_max, rec.idx_row), np.int8)
    qi = np.zeros((rec.N, rec.kmax, rec.idx_row), np.int8)
    for j in range(rec.K):
        rows = np.asarray(rows_of(j))
        assert len(rows) == rec.topk and rows.max() < rec.S
        keys[:, rows, j] = 1
        qi[:, j, j] = 100
    return keys, qi


@pytest.mark.parametrize("two_slices", [False, True], ids=["one_slice", "two_slices"])
def test_union_outgrowing_a_slice(two_slices):
    import torch
    import oracle.dhs_oracle as oracle
    from hierarchical_sparse_kv_int8_gb300.runner import Runner
    k = 1536 if two_slices else 1024
    rec = wl.Recipe("union_spill_%d" % k, N=2, K=8, S=65536, H_idx=1, d_idx=64, topk=k, Hq=8,
                    Hkv=1, qk_dim=128, v_dim=128, kv_layout=0, B=2048, rho_within=0.5,
                    rho_cross=0.6, W=16, p=8, seed=5)
    sl = _slice_rows(rec.s_max)
    if two_slices:  # queries 0-3 in slice 0, queries 4-7 in slice 1: 6144 union rows each
        rows_of = lambda j: (j % 4) * k + np.arange(k) + (sl if j >= 4 else 0)
    else:  # all eight queries in slice 0: 8192 union rows
        rows_of = lambda j: j * k + np.arange(k)
    keys, qi = _crafted(rec, rows_of)
    run = Runner(rec, keys=torch.from_numpy(keys).cuda())
    o = oracle.Oracle(oracle_config(rec))
    slots = list(range(rec.N))
    for r in slots:
        o.bind(r, rec.host_rows(r, r + 1)[0], keys[r], rec.S)
    kr = rec.k_per_req()
    for rnd in range(2):
        acc = rec.accepted(rnd, kr)
        run.load_round(rnd)
        run.q_idx.copy_(torch.from_numpy(qi).cuda())
        run.select(kr)
        run.resolve(True)
        run.attend()
        _, qa, bl = oracle_inputs(rec, rnd, slots, o.cfg.k_max)
        sel = o.select(qi, kr)
        o.resolve(sel, shared=True)
        o.check_placement()
        out, lse = o.attend(qa, bl)
        ores = dict(topk=sel.copy(), loc=o.loc.copy(), out=out, lse=lse,
                    union={r: o.union[r].copy() for r in slots},
                    misses={r: o.misses[r].copy() for r in slots},
                    staging={r: o.staging[r].copy() for r in slots})
        for r in slots:
            assert len(ores["union"][r]) == rec.K * k  # disjoint selections
        compare_round(run, o, ores, slots, kr, "union spill round %d" % rnd)
        run.commit(acc)
        o.commit(acc)
        compare_state(run, o, slots, "union spill round %d" % rnd)
    assert run.ctx.stats()["device_error"] == 0
