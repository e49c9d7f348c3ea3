"""Python binding of libdhs (speculative-verification sparse attention over a
two-tier KV cache on one GB300 GPU).

This module only marshals arguments to the C ABI declared in
``include/dhs.h``; every step of the hot path runs in the library's CUDA
kernels.  Device buffers are passed as CUDA tensors (or raw device
addresses), small per-request control arrays as host numpy arrays, and the
stream defaults to torch's current stream.  There is no CPU fallback: if the
library is not built, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import numpy as np

from . import _build

__all__ = ["Arenas", "Config", "Context", "DhsError", "build", "load", "LOC_RING", "LOC_OPT",
           "LOC_HOT", "LOC_STAGE", "BUF", "ROLE_FULL", "ROLE_FOLLOWER"]

LOC_RING, LOC_OPT, LOC_HOT, LOC_STAGE = 0, 1, 2, 3
LOC_TIER_SHIFT = 28
KV_SPLIT, KV_LATENT = 0, 1
BUF = dict(hot_row=0, hot_stamp=1, hot_data=2, ring=3, stage=4, opt=5, union=6, miss=7,
           counts=8, lru=9, frontier=10, hot_map=11, opt_map=12, scores=13)


class Config(ctypes.Structure):
    _fields_ = [("n_slots", ctypes.c_int32), ("k_max", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("s_max", ctypes.c_int64), ("idx_heads", ctypes.c_int32),
                ("idx_dim", ctypes.c_int32), ("q_heads", ctypes.c_int32),
                ("kv_heads", ctypes.c_int32), ("qk_dim", ctypes.c_int32),
                ("v_dim", ctypes.c_int32), ("kv_layout", ctypes.c_int32),
                ("budget", ctypes.c_int32), ("ring_window", ctypes.c_int32),
                ("page_rows", ctypes.c_int32), ("opt_rows_max", ctypes.c_int64),
                ("softmax_scale", ctypes.c_float), ("attn_pass", ctypes.c_int32),
                ("topk_pass", ctypes.c_int32), ("round_groups", ctypes.c_int32),
                ("tokens_per_row", ctypes.c_int32)]

ATTN_AUTO, ATTN_PER_QUERY, ATTN_UNION, ATTN_UNION_MMA = 0, 1, 2, 3
TOPK_AUTO, TOPK_CLUSTER, TOPK_ROW = 0, 1, 2


class Stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "resolve_calls", "selections", "union_rows", "ring_hits", "opt_hits", "hot_hits",
        "misses", "miss_selections", "host_rows_fetched", "host_bytes", "installs", "evictions",
        "direct_only")] + [("device_error", ctypes.c_int32), ("device_error_site", ctypes.c_int32),
                        ("topk_rescans", ctypes.c_int64)]


class DhsError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s: %s (code %d)" % (what, load().dhs_strerror(code).decode(), code))


_lib = None
_SIGS = {
    "dhs_create": ([ctypes.POINTER(Config), ctypes.POINTER(ctypes.c_void_p)], ctypes.c_int),
    "dhs_destroy": ([ctypes.c_void_p], None),
    "dhs_ring_rows": ([ctypes.c_void_p], ctypes.c_int64),
    "dhs_device_bytes": ([ctypes.c_void_p], ctypes.c_int64),
    "dhs_bind_request": ([ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                          ctypes.c_int64, ctypes.c_void_p], ctypes.c_int),
    "dhs_select": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                    ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "dhs_resolve": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                     ctypes.c_void_p], ctypes.c_int),
    "dhs_attend": ([ctypes.c_void_p] * 6 + [ctypes.c_void_p], ctypes.c_int),
    "dhs_commit": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "dhs_append_keys": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
                        ctypes.c_int),
    "dhs_commit_compressed": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                               ctypes.c_void_p], ctypes.c_int),
    "dhs_set_residency": ([ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                           ctypes.c_void_p], ctypes.c_int),
    "dhs_policy_create": ([ctypes.c_int64, ctypes.c_int64, ctypes.POINTER(ctypes.c_void_p)],
                          ctypes.c_int),
    "dhs_policy_destroy": ([ctypes.c_void_p], None),
    "dhs_policy_admit": ([ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                          ctypes.c_void_p], ctypes.c_int),
    "dhs_policy_complete": ([ctypes.c_void_p, ctypes.c_int32], ctypes.c_int),
    "dhs_policy_repopulate": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                              ctypes.c_int32, ctypes.c_void_p], ctypes.c_int),
    "dhs_policy_query": ([ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                         ctypes.c_void_p], ctypes.c_int),
    "dhs_policy_free_pages": ([ctypes.c_void_p], ctypes.c_int64),
    "dhs_get_stats": ([ctypes.c_void_p, ctypes.POINTER(Stats), ctypes.c_void_p], ctypes.c_int),
    "dhs_reset_stats": ([ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "dhs_buffer_bytes": ([ctypes.c_void_p, ctypes.c_int32], ctypes.c_int64),
    "dhs_export": ([ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                    ctypes.c_void_p], ctypes.c_int),
    "dhs_set_timing": ([ctypes.c_void_p, ctypes.c_int32], ctypes.c_int),
    "dhs_graph_begin": ([ctypes.c_void_p], ctypes.c_int),
    "dhs_graph_end": ([ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)], ctypes.c_int),
    "dhs_graph_launch": ([ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "dhs_graph_destroy": ([ctypes.c_void_p], None),
    "dhs_kernel_times": ([ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p],
                         ctypes.c_int),
    "dhs_kernel_name": ([ctypes.c_int32], ctypes.c_char_p),
    "dhs_kernel_count": ([], ctypes.c_int32),
    "dhs_timing_accumulate_graph": ([ctypes.c_void_p], ctypes.c_int),
    "dhs_snapshot": ([ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p],
                     ctypes.c_int),
    "dhs_restore": ([ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p], ctypes.c_int),
    "dhs_snapshot_free": ([ctypes.c_void_p, ctypes.c_int32], ctypes.c_int),
    "dhs_arenas_create": ([ctypes.c_int32] * 5 + [ctypes.POINTER(ctypes.c_void_p)], ctypes.c_int),
    "dhs_arenas_bytes": ([ctypes.c_void_p], ctypes.c_int64),
    "dhs_arenas_destroy": ([ctypes.c_void_p], ctypes.c_int),
    "dhs_create_on_arena": ([ctypes.POINTER(Config), ctypes.c_void_p, ctypes.c_int32,
                             ctypes.c_int32, ctypes.POINTER(ctypes.c_void_p)], ctypes.c_int),
    "dhs_adopt": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
                  ctypes.c_int),
    "dhs_round_host": ([ctypes.c_void_p] * 9, ctypes.c_int),
    "dhs_round": ([ctypes.c_void_p] * 11, ctypes.c_int),
    "dhs_strerror": ([ctypes.c_int], ctypes.c_char_p),
    "dhs_last_error": ([ctypes.c_void_p], ctypes.c_char_p),
    "dhs_select_noalloc": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                            ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p],
                           ctypes.c_int),
}


def build(force: bool = False) -> str:
    """Compile libdhs.so for sm_103a (nvcc; works without a GPU)."""
    return _build.build(force=force)


def library_path() -> str:
    return _build.LIB


def load():
    """Load libdhs.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError("libdhs.so is not built (%s); call "
                               "hierarchical_sparse_kv_int8_gb300.build() first" % _build.LIB)
        lib = ctypes.CDLL(_build.LIB)
        for name, (args, res) in _SIGS.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
    return _lib


def _dptr(x) -> Optional[int]:
    """Device (or pinned host) address of a tensor, or an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


_ptr_memo: dict = {}


def _host_ptr(a: np.ndarray) -> int:
    """Address of a host array; remembered per array object, since asking
    numpy for it costs about a microsecond per call."""
    hit = _ptr_memo.get(id(a))
    if hit is not None and hit[0] is a:
        return hit[1]
    ptr = a.ctypes.data
    if len(_ptr_memo) > 64:
        _ptr_memo.clear()
    _ptr_memo[id(a)] = (a, ptr)
    return ptr


def _host_i32(x, n) -> np.ndarray:
    if isinstance(x, np.ndarray) and x.dtype == np.int32 and x.flags.c_contiguous:
        a = x
    else:
        a = np.ascontiguousarray(np.asarray(x, dtype=np.int32))
    if a.size < n:
        raise ValueError("expected %d int32 values, got %d" % (n, a.size))
    return a


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def select_noalloc(q_idx, keys, n_queries, n_rows, idx_row_bytes, topk, topk_out, stream=None):
    """Indexer + top-k through dhs_select_noalloc, which allocates nothing.

    For callers that cannot allocate device memory at the call (graph capture,
    engines that own all device memory, decode loops that must not
    synchronise); see include/dhs.h for the limits and the shared scratch.
    """
    rc = load().dhs_select_noalloc(_dptr(q_idx), _dptr(keys), n_queries, n_rows, idx_row_bytes,
                                   topk, _dptr(topk_out), _stream(stream))
    if rc:
        raise DhsError(rc, "dhs_select_noalloc")


def make_config(**kw) -> Config:
    c = Config()
    for name, _ in Config._fields_:
        setattr(c, name, kw.get(name, 0))
    return c


class Graph:
    """A CUDA graph of library calls captured on one stream, instantiated with
    the launches' priorities honoured (dhs_graph_*).  Use as
    ``with Graph.capture(stream) as g: ...calls on stream...`` then
    ``g.replay()``."""

    def __init__(self):
        self._lib = load()
        self.h = None
        self._stream = None

    @classmethod
    def capture(cls, stream):
        g = cls()
        g._stream = stream
        return g

    def __enter__(self):
        rc = self._lib.dhs_graph_begin(_stream(self._stream))
        if rc:
            raise DhsError(rc, "dhs_graph_begin")
        return self

    def __exit__(self, exc_type, exc, tb):
        h = ctypes.c_void_p()
        rc = self._lib.dhs_graph_end(_stream(self._stream), ctypes.byref(h))
        if rc and exc_type is None:
            raise DhsError(rc, "dhs_graph_end")
        self.h = h.value
        return False

    def replay(self, stream=None):
        rc = self._lib.dhs_graph_launch(self.h, _stream(stream if stream is not None else self._stream))
        if rc:
            raise DhsError(rc, "dhs_graph_launch")

    def close(self):
        if self.h:
            self._lib.dhs_graph_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Policy:
    """Residency policy of optional history (dhs_policy_*): page accounting
    on the host, no device.  admit() returns (admitted, optional_pages,
    reclaimed request ids); repopulate() returns [(request, pages added)]."""

    def __init__(self, total_pages: int, reserve_pages: int = 0):
        self._lib = load()
        h = ctypes.c_void_p()
        rc = self._lib.dhs_policy_create(int(total_pages), int(reserve_pages), ctypes.byref(h))
        if rc:
            raise DhsError(rc, "dhs_policy_create")
        self.h = h.value
        self.requests = []  # admitted ids, admission order (sizes the output arrays)

    def close(self):
        if getattr(self, "h", None):
            self._lib.dhs_policy_destroy(self.h)
            self.h = None

    def __del__(self):
        self.close()

    def _check(self, rc, what):
        if rc:
            raise DhsError(rc, what)

    def admit(self, request: int, required_pages: int, history_pages: int):
        cap = max(1, len(self.requests))
        rec = np.zeros(cap, np.int32)
        ok, opt, n = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int32()
        self._check(self._lib.dhs_policy_admit(self.h, int(request), int(required_pages),
                                               int(history_pages), ctypes.byref(ok),
                                               ctypes.byref(opt), rec.ctypes.data, cap,
                                               ctypes.byref(n)), "dhs_policy_admit")
        if ok.value:
            self.requests.append(int(request))
        return bool(ok.value), int(opt.value), [int(x) for x in rec[:n.value]]

    def complete(self, request: int):
        self._check(self._lib.dhs_policy_complete(self.h, int(request)), "dhs_policy_complete")
        self.requests.remove(int(request))

    def repopulate(self, max_pages: int):
        cap = max(1, len(self.requests))
        req, pg = np.zeros(cap, np.int32), np.zeros(cap, np.int64)
        n = ctypes.c_int32()
        self._check(self._lib.dhs_policy_repopulate(self.h, int(max_pages), req.ctypes.data,
                                                    pg.ctypes.data, cap, ctypes.byref(n)),
                    "dhs_policy_repopulate")
        return [(int(req[i]), int(pg[i])) for i in range(n.value)]

    def query(self, request: int):
        r, o, h = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        self._check(self._lib.dhs_policy_query(self.h, int(request), ctypes.byref(r),
                                               ctypes.byref(o), ctypes.byref(h)),
                    "dhs_policy_query")
        return int(r.value), int(o.value), int(h.value)

    def free_pages(self) -> int:
        return int(self._lib.dhs_policy_free_pages(self.h))


ROLE_FULL, ROLE_FOLLOWER = 0, 1


class Arenas:
    """chi staging arenas shared by the sources of a layer group (dhs_arenas_*)."""

    def __init__(self, chi: int, n_slots: int, k_max: int, topk: int, row_elems: int):
        self._lib = load()
        h = ctypes.c_void_p()
        rc = self._lib.dhs_arenas_create(chi, n_slots, k_max, topk, row_elems, ctypes.byref(h))
        if rc:
            raise DhsError(rc, "dhs_arenas_create")
        self.h = h.value
        self.chi = chi

    def nbytes(self) -> int:
        return int(self._lib.dhs_arenas_bytes(self.h))

    def close(self):
        if getattr(self, "h", None):
            rc = self._lib.dhs_arenas_destroy(self.h)
            if rc:
                raise DhsError(rc, "dhs_arenas_destroy")
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Context:
    """One KV source (layer) with ``n_slots`` request slots; see include/dhs.h.
    With ``arenas`` the context stages in arena ``arena`` of that set
    (dhs_create_on_arena) and may be a follower (``role``)."""

    def __init__(self, cfg: Config, arenas: Optional[Arenas] = None, arena: int = 0,
                 role: int = ROLE_FULL):
        self.cfg = cfg
        self._lib = load()
        h = ctypes.c_void_p()
        if arenas is None:
            rc = self._lib.dhs_create(ctypes.byref(cfg), ctypes.byref(h))
        else:
            rc = self._lib.dhs_create_on_arena(ctypes.byref(cfg), arenas.h, arena, role,
                                               ctypes.byref(h))
        if rc:
            raise DhsError(rc, "dhs_create")
        self.h = h
        self.arenas = arenas  # kept alive while the context uses them

    def close(self):
        if getattr(self, "h", None):
            self._lib.dhs_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, rc, what):
        if rc:
            detail = self._lib.dhs_last_error(self.h).decode() if rc == 4 else ""
            raise DhsError(rc, what + (" [%s]" % detail if detail else ""))

    @property
    def ring_rows(self) -> int:
        return self._lib.dhs_ring_rows(self.h)

    def device_bytes(self) -> int:
        return self._lib.dhs_device_bytes(self.h)

    def bind(self, slot, host_kv, idx_keys, n_committed, stream=None):
        self._check(self._lib.dhs_bind_request(self.h, slot, _dptr(host_kv), _dptr(idx_keys),
                                               n_committed, _stream(stream)), "dhs_bind_request")

    def select(self, q_idx, k_per_req, topk_out, pos=None, stream=None):
        kr = _host_i32(k_per_req, self.cfg.n_slots)
        p = None
        if pos is not None:
            p = np.ascontiguousarray(np.asarray(pos, dtype=np.int64))
        self._check(self._lib.dhs_select(self.h, _dptr(q_idx), _host_ptr(kr),
                                         None if p is None else p.ctypes.data, _dptr(topk_out),
                                         _stream(stream)), "dhs_select")

    def adopt(self, k_per_req, pos=None, stream=None):
        kr = _host_i32(k_per_req, self.cfg.n_slots)
        p = None
        if pos is not None:
            p = np.ascontiguousarray(np.asarray(pos, dtype=np.int64))
        self._check(self._lib.dhs_adopt(self.h, _host_ptr(kr), None if p is None else p.ctypes.data,
                                        _stream(stream)), "dhs_adopt")

    def resolve(self, topk, loc_out, shared=True, stream=None):
        self._check(self._lib.dhs_resolve(self.h, _dptr(topk), _dptr(loc_out), 1 if shared else 0,
                                          _stream(stream)), "dhs_resolve")

    def attend(self, q, block_kv, loc, out, lse=None, stream=None):
        self._check(self._lib.dhs_attend(self.h, _dptr(q), _dptr(block_kv), _dptr(loc), _dptr(out),
                                         _dptr(lse), _stream(stream)), "dhs_attend")

    def commit(self, accepted_len, stream=None):
        a = _host_i32(accepted_len, self.cfg.n_slots)
        self._check(self._lib.dhs_commit(self.h, _host_ptr(a), _stream(stream)), "dhs_commit")

    def commit_compressed(self, accepted_len, rows_kv, rows_idx_keys=None, stream=None):
        """Commit for a source packing tokens_per_row positions into a row:
        the stored rows the kept positions complete, from the compressor's
        rows (device bf16 [n_slots][ceil(k_max/m)][row_elems]) and keys
        (device int8 [n_slots][ceil(k_max/m)][idx_row], or None)."""
        a = _host_i32(accepted_len, self.cfg.n_slots)
        self._check(self._lib.dhs_commit_compressed(self.h, _host_ptr(a), _dptr(rows_kv),
                                                    _dptr(rows_idx_keys), _stream(stream)),
                    "dhs_commit_compressed")

    def append_keys(self, accepted_len, block_idx_keys, stream=None):
        """Index keys of the rows the coming commit keeps (device int8
        [n_slots][k_max][idx_row]) into the bound key buffers."""
        a = _host_i32(accepted_len, self.cfg.n_slots)
        self._check(self._lib.dhs_append_keys(self.h, _host_ptr(a), _dptr(block_idx_keys),
                                              _stream(stream)), "dhs_append_keys")

    def set_residency(self, slot, rows, stream=None):
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        self._check(self._lib.dhs_set_residency(self.h, slot, rows.ctypes.data if rows.size else None,
                                                rows.size, _stream(stream)), "dhs_set_residency")

    def stats(self, stream=None, check=True) -> Dict[str, int]:
        st = Stats()
        rc = self._lib.dhs_get_stats(self.h, ctypes.byref(st), _stream(stream))
        if rc and (check or rc != 5):
            raise DhsError(rc, "dhs_get_stats")
        return {n: getattr(st, n) for n, _ in Stats._fields_}

    def reset_stats(self, stream=None):
        self._check(self._lib.dhs_reset_stats(self.h, _stream(stream)), "dhs_reset_stats")

    def buffer_bytes(self, which: str) -> int:
        return self._lib.dhs_buffer_bytes(self.h, BUF[which])

    def export(self, which: str, dst, stream=None):
        """Copy internal buffer ``which`` into the CUDA tensor ``dst`` (its nbytes)."""
        nbytes = dst.numel() * dst.element_size()
        self._check(self._lib.dhs_export(self.h, BUF[which], _dptr(dst), nbytes, _stream(stream)),
                    "dhs_export")

    def set_timing(self, enable: bool):
        self._check(self._lib.dhs_set_timing(self.h, 1 if enable else 0), "dhs_set_timing")

    def kernel_times(self) -> Dict[str, tuple]:
        n = self._lib.dhs_kernel_count()
        launches = np.zeros(n, np.int64)
        ms = np.zeros(n, np.float64)
        self._check(self._lib.dhs_kernel_times(self.h, n, launches.ctypes.data, ms.ctypes.data),
                    "dhs_kernel_times")
        return {self._lib.dhs_kernel_name(i).decode(): (int(launches[i]), float(ms[i]))
                for i in range(n)}

    def timing_accumulate_graph(self):
        self._check(self._lib.dhs_timing_accumulate_graph(self.h), "dhs_timing_accumulate_graph")

    def snapshot(self, stream=None) -> int:
        sid = ctypes.c_int32()
        self._check(self._lib.dhs_snapshot(self.h, ctypes.byref(sid), _stream(stream)),
                    "dhs_snapshot")
        return sid.value

    def restore(self, sid: int, stream=None):
        self._check(self._lib.dhs_restore(self.h, sid, _stream(stream)), "dhs_restore")

    def snapshot_free(self, sid: int):
        self._check(self._lib.dhs_snapshot_free(self.h, sid), "dhs_snapshot_free")

    def round(self, q_idx, k_per_req, q, block_kv, accepted_len, topk_out, loc_out, out, lse=None,
              stream=None):
        kr = _host_i32(k_per_req, self.cfg.n_slots)
        a = _host_i32(accepted_len, self.cfg.n_slots)
        self._check(self._lib.dhs_round(self.h, _dptr(q_idx), _host_ptr(kr), _dptr(q),
                                        _dptr(block_kv), _host_ptr(a), _dptr(topk_out),
                                        _dptr(loc_out), _dptr(out), _dptr(lse), _stream(stream)),
                    "dhs_round")

    def round_host(self, q_idx, k_per_req, q, block_kv, accepted_len, out, lse=None, stream=None):
        kr = _host_i32(k_per_req, self.cfg.n_slots)
        a = _host_i32(accepted_len, self.cfg.n_slots)
        self._check(self._lib.dhs_round_host(self.h, _dptr(q_idx), _host_ptr(kr), _dptr(q),
                                             _dptr(block_kv), _host_ptr(a), _dptr(out),
                                             _dptr(lse), _stream(stream)), "dhs_round_host")
