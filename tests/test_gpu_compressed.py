"""Sources that pack m token positions into each stored row ([ADHS] eq. (8)):
rounds of select, resolve, attend and dhs_commit_compressed equal the
oracle's -- selections over the complete rows only, the rows each commit
completes published with the compressor's payload and index keys, the
partial group kept out, no history row served by the ring -- and the calls
that assume one position per row refuse such a source."""
import numpy as np
import pytest

import workload as wl
from harness import build_oracle, compare_round, compare_state, oracle_round

pytestmark = pytest.mark.gpu

TINY_GQA = wl.Recipe("tiny_gqa", N=3, K=4, S=700, H_idx=2, d_idx=32, topk=64, Hq=8, Hkv=1,
                     qk_dim=128, v_dim=128, kv_layout=0, B=96, rho_within=0.5, rho_cross=0.6,
                     W=16, p=8, seed=3)


@pytest.mark.parametrize("m", [3, 4])
def test_compressed_source_rounds(m):
    from hierarchical_sparse_kv_int8_gb300.runner import Runner
    rec = TINY_GQA.scaled(name="tiny_m%d" % m, m=m)
    run = Runner(rec, attn_pass=2)
    slots = list(range(rec.N))
    o = build_oracle(rec, slots)
    for rnd in range(4):
        kr = rec.k_per_req()
        acc = rec.accepted(rnd, kr)
        pos = None
        if rnd == 2:  # queries placed inside the history: domains floor((pos + 1) / m)
            tok = np.array([o.req[r].tok for r in slots], np.int64)
            pos = np.stack([tok - 1 - 5 * j for j in range(rec.kmax)], axis=1)
            pos[0, 1] = 2 * m - 2  # one complete row short of 2 rows
        run.load_round(rnd)
        run.select(kr, pos)
        run.resolve(True)
        run.attend()
        run.commit_compressed(rnd, acc)
        ores = oracle_round(o, rec, rnd, slots, kr, None, True, pos)
        o.commit_compressed(acc, rec.compressed_rows(rnd, 0, rec.N),
                            rec.compressed_keys(rnd, 0, rec.N))
        compare_round(run, o, ores, slots, kr, "m=%d round %d" % (m, rnd))
        compare_state(run, o, slots, "m=%d round %d" % (m, rnd))
        keys = run.keys.cpu().numpy()
        for r in slots:
            assert np.array_equal(keys[r], o.req[r].keys), "key rows r=%d" % r
    st = run.ctx.stats()
    assert st["device_error"] == 0 and st["ring_hits"] == 0


def test_single_position_calls_refuse_compressed_sources():
    import torch
    from hierarchical_sparse_kv_int8_gb300 import DhsError
    from hierarchical_sparse_kv_int8_gb300.runner import Runner
    rec = TINY_GQA.scaled(name="tiny_m2", m=2)
    run = Runner(rec, attn_pass=2, round_groups=2)
    kr = rec.k_per_req()
    acc = rec.accepted(0, kr)
    run.load_round(0)
    with pytest.raises(DhsError):
        run.round_fused(kr, acc)
    bk = torch.zeros((rec.N, run.Km, rec.idx_row), dtype=torch.int8, device="cuda")
    with pytest.raises(DhsError):
        run.ctx.append_keys(acc, bk, run.stream)
    run.select(kr)
    run.resolve(True)
    run.attend()
    with pytest.raises(DhsError):
        run.commit(acc)
    run.commit_compressed(0, acc)  # the compressed commit still closes the round
    assert run.ctx.stats()["device_error"] == 0
