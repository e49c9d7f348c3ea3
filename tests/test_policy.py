"""Residency policy of optional history ("Adaptive DHiSparse", section 3.1,
eq. (3) and (4)): the oracle pinned to a hand-worked trace, to a library
formulation of eq. (4) and to the section's invariants, and the library's
dhs_policy_* calls (host logic, no device) equal to the oracle decision by
decision."""
import json
import os
import random

import numpy as np
import pytest

from oracle.dhs_oracle import ResidencyPolicy, reclaim_prefix

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "residency_policy_trace.json")


def _run(policy, step):
    if step["op"] == "admit":
        return policy.admit(step["request"], step["required"], step["history"])
    if step["op"] == "repopulate":
        return policy.repopulate(step["max_pages"])
    return policy.complete(step["request"])


def _check_golden(policy, free):
    g = json.load(open(GOLDEN))
    for step in g["steps"]:
        got = _run(policy, step)
        want = step["want"]
        if step["op"] == "admit":
            assert got == (want["admitted"], want["optional"], want["reclaimed"]), step["note"]
        elif step["op"] == "repopulate":
            assert [list(x) for x in got] == want["given"], step["note"]
        assert free(policy) == want["free"], step["note"]


def test_oracle_hand_worked_trace():
    g = json.load(open(GOLDEN))
    _check_golden(ResidencyPolicy(g["total_pages"], g["reserve_pages"]), lambda p: p.free())


def test_reclaim_prefix_against_searchsorted():
    """Eq. (4) as a library routine: with cumulative pages c, q' is one past
    the first index where c >= delta (numpy's left searchsorted)."""
    rng = np.random.default_rng(5)
    for _ in range(2000):
        a = rng.integers(0, 6, rng.integers(0, 7)).tolist()
        delta = int(rng.integers(1, 25))
        c = np.cumsum(a) if a else np.zeros(0, np.int64)
        i = int(np.searchsorted(c, delta, side="left"))
        want = i + 1 if i < len(a) else None
        assert reclaim_prefix(a, delta) == want, (a, delta)
    assert reclaim_prefix([4, 1], 0) == 0


def _random_ops(seed, n_ops=300):
    rng = random.Random(seed)
    live, nxt, ops = [], 0, []
    for _ in range(n_ops):
        u = rng.random()
        if u < 0.45 or not live:
            ops.append(dict(op="admit", request=nxt, required=rng.randint(0, 30),
                            history=rng.randint(0, 60)))
            live.append(nxt)
            nxt += 1
        elif u < 0.7:
            r = rng.choice(live)
            ops.append(dict(op="complete", request=r))
        else:
            ops.append(dict(op="repopulate", max_pages=rng.randint(0, 40)))
    return ops


@pytest.mark.parametrize("seed", range(6))
def test_oracle_invariants(seed):
    """Eq. (3) after every call; a reclaim takes the shortest covering prefix
    of the reclaim order and nothing else; waits change nothing;
    repopulation stays within its bound, the free pages and each history."""
    total, reserve = 200, 20
    p = ResidencyPolicy(total, reserve)
    admitted = set()
    for op in _random_ops(seed):
        before = {r["id"]: r["optional"] for r in p.reqs}
        order = [r["id"] for r in p.reqs]
        free0 = p.free()
        if op["op"] == "complete":
            if op["request"] not in admitted:
                continue
            p.complete(op["request"])
            admitted.discard(op["request"])
        elif op["op"] == "admit":
            ok, opt, rec = p.admit(op["request"], op["required"], op["history"])
            if not ok:
                assert {r["id"]: r["optional"] for r in p.reqs} == before
                assert sum(before.values()) < op["required"] - free0
                continue
            admitted.add(op["request"])
            deficit = op["required"] - free0
            if deficit > 0:
                holders = [i for i in order if before[i] > 0]
                assert rec == holders[:len(rec)]  # a prefix of the reclaim order
                assert sum(before[i] for i in rec) >= deficit
                assert sum(before[i] for i in rec[:-1]) < deficit  # shortest
                for i in order:
                    assert p.query(i)[1] == (0 if i in rec else before[i])
            else:
                assert rec == []
            assert 0 <= opt <= op["history"]
        else:
            got = p.repopulate(op["max_pages"])
            assert sum(g for _, g in got) <= min(op["max_pages"], free0)
            for rid, g in got:
                assert g > 0
                req, o, h = p.query(rid)
                assert o <= h and o == before[rid] + g
        assert p.free() >= 0  # eq. (3)
        assert sum(r["required"] + r["optional"] for r in p.reqs) + reserve <= total


def _lib_policy(total, reserve):
    import hierarchical_sparse_kv_int8_gb300 as dhs
    return dhs.Policy(total, reserve)


def test_library_hand_worked_trace():
    g = json.load(open(GOLDEN))
    _check_golden(_lib_policy(g["total_pages"], g["reserve_pages"]), lambda p: p.free_pages())


@pytest.mark.parametrize("seed", range(6))
def test_library_equals_oracle(seed):
    o, lib = ResidencyPolicy(150, 15), _lib_policy(150, 15)
    admitted = set()
    for op in _random_ops(100 + seed):
        if op["op"] == "complete":
            if op["request"] not in admitted:
                continue
            admitted.discard(op["request"])
        got, want = _run(lib, op), _run(o, op)
        assert got == want, op
        if op["op"] == "admit" and want[0]:
            admitted.add(op["request"])
        assert lib.free_pages() == o.free()
        for rid in admitted:
            assert lib.query(rid) == o.query(rid)


def test_library_argument_checks():
    import hierarchical_sparse_kv_int8_gb300 as dhs
    with pytest.raises(dhs.DhsError):
        dhs.Policy(10, 11)  # reserve above total
    p = _lib_policy(10, 0)
    p.admit(7, 2, 3)
    with pytest.raises(dhs.DhsError):
        p.admit(7, 1, 1)  # already admitted
    with pytest.raises(dhs.DhsError):
        p.admit(8, -1, 0)
    with pytest.raises(dhs.DhsError):
        p.complete(9)
    with pytest.raises(dhs.DhsError):
        p.query(9)
    assert p.free_pages() == 10 - 2 - 3


def test_request_larger_than_the_budget_is_refused():
    """A request whose required pages exceed total - reserve can never satisfy
    eq. (3), even alone, so it is refused (capacity) instead of waiting; the
    oracle and the library agree and nothing changes."""
    import hierarchical_sparse_kv_int8_gb300 as dhs
    o, lib = ResidencyPolicy(100, 10), _lib_policy(100, 10)
    for p in (o, lib):
        assert p.admit(1, 30, 50)[0]
    with pytest.raises(ValueError, match="capacity"):
        o.admit(2, 91, 0)
    with pytest.raises(dhs.DhsError) as e:
        lib.admit(2, 91, 0)
    assert e.value.code == 3
    assert o.free() == lib.free_pages() == 100 - 10 - 30 - 50
    # within the budget it waits while the optional pages cannot cover it ...
    assert o.admit(3, 90, 0) == lib.admit(3, 90, 0) == (False, 0, [])
    # ... and exactly the budget less the reserve is admitted once it fits
    for p in (o, lib):
        p.complete(1)
    assert o.admit(3, 90, 0) == lib.admit(3, 90, 0) == (True, 0, [])
    assert o.free() == lib.free_pages() == 0
