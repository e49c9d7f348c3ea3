"""The C-ABI library builds for sm_103a, loads, and exports every entry point
include/dhs.h declares; host-side argument checks that need no GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import hierarchical_sparse_kv_int8_gb300 as dhs
    dhs.build()
    return dhs.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "dhs.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dhs_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), "missing export %s" % n


def test_strerror_and_kernel_names(lib):
    for code in range(7):
        assert lib.dhs_strerror(code)
    n = lib.dhs_kernel_count()
    names = [lib.dhs_kernel_name(i).decode() for i in range(n)]
    assert "index_score" in names and "attn" in names and "gather" in names


def test_invalid_configs_rejected_before_any_cuda_call(lib):
    import hierarchical_sparse_kv_int8_gb300 as dhs
    good = dict(n_slots=8, k_max=4, topk=2048, s_max=32832, idx_heads=1, idx_dim=64, q_heads=8,
                kv_heads=1, qk_dim=128, v_dim=128, kv_layout=0, budget=4096, ring_window=2048,
                page_rows=64, opt_rows_max=0, softmax_scale=0.0)
    bad = [dict(n_slots=0), dict(k_max=9), dict(topk=100), dict(topk=8192), dict(idx_dim=63),
           dict(q_heads=12, kv_heads=8), dict(qk_dim=96, v_dim=96), dict(kv_layout=2),
           dict(kv_layout=1, qk_dim=576, v_dim=512, kv_heads=2), dict(budget=0),
           dict(opt_rows_max=40000), dict(q_heads=32)]
    for b in bad:
        cfg = dhs.make_config(**{**good, **b})
        h = ctypes.c_void_p()
        rc = lib.dhs_create(ctypes.byref(cfg), ctypes.byref(h))
        assert rc == 1, (b, rc)
        assert not h.value


def test_null_context_calls_are_rejected(lib):
    assert lib.dhs_select(None, None, None, None, None, None) == 1
    assert lib.dhs_commit(None, None, None) == 1
    assert lib.dhs_ring_rows(None) == 0
    lib.dhs_destroy(None)


def test_library_path_is_in_tree(lib):
    import hierarchical_sparse_kv_int8_gb300 as dhs
    assert dhs.library_path().startswith(os.path.join(ROOT, "hierarchical_sparse_kv_int8_gb300"))
