"""Physical-source sharing and layer groups ("Adaptive DHiSparse" 2.2, 3.2,
3.4) on the GPU through the C ABI, against the oracle run source by source.

- A GLM-style layer group: one index producer and three follower payload
  layers (each with its own host rows, hot cache and ring) take the
  producer's positions; they stage in chi = 2 shared arenas (layers 0 and 2
  on arena 0, 1 and 3 on arena 1), resolves (with their host gathers) are
  issued on a copy stream while attention runs on a compute stream, so the
  second pair's gathers wait on the GPU for the first pair's attention
  readers.  Several steps; every layer compared with its own oracle.
- A DeepSeek-style shared source: a Full layer, a Reuse layer (same location
  vector, its own queries), then a Reindex layer (a fresh selection over the
  same source and cache state) before the one commit of the step.
- The arena protocol's refusals (a resolve into an arena whose rows nobody
  has read yet; an attend after another source took the arena).
"""
import numpy as np
import pytest

import workload as wl
from harness import build_oracle, compare_round, compare_state, oracle_inputs

pytestmark = pytest.mark.gpu

BASE = wl.Recipe("group_tiny", N=3, K=3, S=700, H_idx=1, d_idx=64, topk=64, Hq=8, Hkv=1,
                 qk_dim=128, v_dim=128, kv_layout=0, B=48, rho_within=0.6, rho_cross=0.7,
                 W=40, p=8, seed=81)


def _layer_oracle_round(o, rec, rnd, slots, kr, sel, acc=None):
    """One round of a follower's oracle on the producer's selection."""
    Km = o.cfg.k_max
    _, qa, bl = oracle_inputs(rec, rnd, slots, Km)
    o.adopt(sel, kr)
    o.resolve(sel)
    o.check_placement()
    out, lse = o.attend(qa, bl)
    return dict(topk=sel.copy(), loc=o.loc.copy(), out=out, lse=lse,
                union={r: o.union[r].copy() for r in slots if r in o.union},
                misses={r: o.misses[r].copy() for r in slots if r in o.misses},
                staging={r: o.staging[r].copy() for r in slots if r in o.staging})


@pytest.mark.parametrize("attn_pass", [1, 2, 3], ids=["per_query", "union_tensor_cores", "union_mma_sync"])
def test_layer_group_followers_on_shared_arenas(attn_pass):
    import torch
    import hierarchical_sparse_kv_int8_gb300 as dhs
    from hierarchical_sparse_kv_int8_gb300.runner import Runner

    dhs.build()
    L, chi = 4, 2
    recs = [BASE.scaled(seed=BASE.seed + l) for l in range(L)]  # own payload per layer
    arenas = dhs.Arenas(chi, BASE.N, BASE.kmax, BASE.topk, BASE.row_elems)
    assert arenas.nbytes() == chi * BASE.N * BASE.kmax * BASE.topk * BASE.row_bytes
    runs = [Runner(recs[0], attn_pass=attn_pass, arenas=arenas, arena=0, role=dhs.ROLE_FULL)]
    for l in range(1, L):
        runs.append(Runner(recs[l], attn_pass=attn_pass, arenas=arenas, arena=l % chi,
                           role=dhs.ROLE_FOLLOWER, keys=runs[0].keys))
    slots = list(range(BASE.N))
    oracles = [build_oracle(rec, slots) for rec in recs]
    comp, copy = torch.cuda.Stream(), torch.cuda.Stream()
    for rnd in range(3):
        kr = BASE.k_per_req()
        acc = BASE.accepted(rnd, kr)
        for run in runs:
            run.load_round(rnd)
        torch.cuda.synchronize()
        p = runs[0]
        p.ctx.select(p.q_idx, kr, p.topk, None, comp)
        sel_done = torch.cuda.Event()
        sel_done.record(comp)
        copy.wait_event(sel_done)          # the followers read the producer's lists
        for l, run in enumerate(runs):
            if l > 0:
                run.topk = p.topk
                run.ctx.adopt(kr, None, copy)
            run.ctx.resolve(run.topk, run.loc, True, copy)
            if l >= 1:                      # attention trails the copies by one layer
                prev = runs[l - 1]
                prev.ctx.attend(prev.q, prev.block, prev.loc, prev.out, prev.lse, comp)
        last = runs[-1]
        last.ctx.attend(last.q, last.block, last.loc, last.out, last.lse, comp)
        torch.cuda.synchronize()
        sel = oracles[0].select(oracle_inputs(recs[0], rnd, slots, BASE.kmax)[0], kr)
        for l in range(L):
            if l == 0:
                oracles[0].resolve(sel)
                oracles[0].check_placement()
                _, qa, bl = oracle_inputs(recs[0], rnd, slots, BASE.kmax)
                out, lse = oracles[0].attend(qa, bl)
                ores = dict(topk=sel.copy(), loc=oracles[0].loc.copy(), out=out, lse=lse,
                            union={r: oracles[0].union[r].copy() for r in slots},
                            misses={r: oracles[0].misses[r].copy() for r in slots},
                            staging={r: oracles[0].staging[r].copy() for r in slots})
            else:
                ores = _layer_oracle_round(oracles[l], recs[l], rnd, slots, kr, sel)
            # layers 0 and 1's arenas were reused by layers 2 and 3
            compare_round(runs[l], oracles[l], ores, slots, kr, "layer %d round %d" % (l, rnd),
                          check_staging=l >= L - chi)
        for l, run in enumerate(runs):
            run.ctx.commit(acc, comp)
            oracles[l].commit(acc)
        torch.cuda.synchronize()
        for l in range(L):
            compare_state(runs[l], oracles[l], slots, "layer %d round %d" % (l, rnd))
    for run in runs:
        assert run.ctx.stats()["device_error"] == 0
        run.ctx.close()
    arenas.close()


@pytest.mark.parametrize("attn_pass", [1, 2, 3], ids=["per_query", "union_tensor_cores", "union_mma_sync"])
def test_reindex_and_reuse_on_one_source(attn_pass):
    import torch
    import hierarchical_sparse_kv_int8_gb300 as dhs
    from hierarchical_sparse_kv_int8_gb300.runner import Runner
    from harness import compare_outputs

    dhs.build()
    rec = BASE.scaled(opt_frac=0.1)
    run = Runner(rec, attn_pass=attn_pass)
    slots = list(range(rec.N))
    o = build_oracle(rec, slots)
    run.set_residency()
    for r in slots:
        o.set_residency(r, rec.residency_rows(r))
    for rnd in range(3):
        kr = rec.k_per_req()
        acc = rec.accepted(rnd, kr)
        qi, qa, bl = oracle_inputs(rec, rnd, slots, run.Km)
        _, qa_b, _ = oracle_inputs(rec, rnd + 50, slots, run.Km)   # the Reuse layer's queries
        qi_c, qa_c, _ = oracle_inputs(rec, rnd + 90, slots, run.Km)  # the Reindex layer's
        # Full layer
        run.load_round(rnd)
        run.select(kr)
        run.resolve(True)
        run.attend()
        sel = o.select(qi, kr)
        o.resolve(sel)
        o.check_placement()
        out, lse = o.attend(qa, bl)
        ores = dict(topk=sel.copy(), loc=o.loc.copy(), out=out, lse=lse,
                    union={r: o.union[r].copy() for r in slots},
                    misses={r: o.misses[r].copy() for r in slots},
                    staging={r: o.staging[r].copy() for r in slots})
        compare_round(run, o, ores, slots, kr, "full round %d" % rnd)
        # Reuse layer: same locations, its own queries
        run.q.copy_(torch.from_numpy(qa_b.view(np.int16)))
        run.attend()
        out_b, lse_b = o.attend(qa_b, bl)
        torch.cuda.synchronize()
        compare_outputs(run.out.float().cpu().numpy().astype(np.float64),
                        run.lse.cpu().numpy().astype(np.float64),
                        dict(out=out_b, lse=lse_b), slots, kr, "reuse round %d" % rnd)
        # Reindex layer: a fresh selection over the same source
        run.q_idx.copy_(torch.from_numpy(qi_c))
        run.q.copy_(torch.from_numpy(qa_c.view(np.int16)))
        run.select(kr)
        run.resolve(True)
        run.attend()
        sel_c = o.select(qi_c, kr)
        o.resolve(sel_c)
        o.check_placement()
        out_c, lse_c = o.attend(qa_c, bl)
        ores_c = dict(topk=sel_c.copy(), loc=o.loc.copy(), out=out_c, lse=lse_c,
                      union={r: o.union[r].copy() for r in slots},
                      misses={r: o.misses[r].copy() for r in slots},
                      staging={r: o.staging[r].copy() for r in slots})
        compare_round(run, o, ores_c, slots, kr, "reindex round %d" % rnd)
        run.commit(acc)
        o.commit(acc)
        compare_state(run, o, slots, "round %d" % rnd)
    st = run.ctx.stats()
    assert st["device_error"] == 0
    assert st["misses"] == o.stats.misses and st["hot_hits"] == o.stats.hot_hits
    assert st["resolve_calls"] == 6


def test_arena_protocol_refusals():
    import torch
    import hierarchical_sparse_kv_int8_gb300 as dhs
    from hierarchical_sparse_kv_int8_gb300.runner import Runner

    dhs.build()
    arenas = dhs.Arenas(1, BASE.N, BASE.kmax, BASE.topk, BASE.row_elems)
    a = Runner(BASE, arenas=arenas, arena=0)
    b = Runner(BASE.scaled(seed=99), arenas=arenas, arena=0, role=dhs.ROLE_FOLLOWER, keys=a.keys)
    kr = BASE.k_per_req()
    for run in (a, b):
        run.load_round(0)
    a.select(kr)
    a.resolve(True)
    b.adopt(kr, a.topk)
    with pytest.raises(dhs.DhsError) as e:      # a's rows in the arena are unread
        b.resolve(True)
    assert e.value.code == 1
    a.attend()
    b.resolve(True)                             # now b takes the arena
    with pytest.raises(dhs.DhsError) as e:      # a may not read it any more
        a.attend()
    assert e.value.code == 1
    with pytest.raises(dhs.DhsError):           # a follower does not score
        b.ctx.select(b.q_idx, kr, b.topk)
    b.attend()
    torch.cuda.synchronize()
    with pytest.raises(dhs.DhsError):           # contexts still stage in the arenas
        arenas.close()
    a.ctx.close()
    b.ctx.close()
    arenas.close()
