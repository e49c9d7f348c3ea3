"""Seeded synthetic workloads for the verification hot path.

This package is the only code shared by the CUDA path's tests, the benchmark
and the oracle.  It holds none of the method's arithmetic: it turns a recipe
(shapes and seed) into input tensors, element by element, through the
counter-based generator in ``gen.c``.  Because every element is a pure function
of (seed, stream, index), one request of a large batch can be regenerated on
its own, which is how the oracle checks sampled requests of the full-size
configurations.

Stand-in for the pages' serving benchmarks (closed-loop concurrency over
prepared prefixes of GLM-5.3 and DeepSeek-V4.1-Flash): none of those prompts,
models or traces are used; the tensors below only reproduce the shapes, value
ranges and sharing structure the configurations name.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field, replace
from typing import List, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "libwl.so")
_lib = None

NTHREADS = max(1, min(64, os.cpu_count() or 1))


def build(force: bool = False) -> str:
    """Compile gen.c into an in-tree shared library (plain gcc, any host)."""
    src = os.path.join(_HERE, "gen.c")
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(src)):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC",
                           "-pthread", src, "-o", tmp])
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, u64, vp, ci = ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int
        lib.wl_gen_i8.argtypes = [vp, i64, u64, u64, i64, ci, ci, ci]
        lib.wl_gen_bf16_normal.argtypes = [vp, i64, u64, u64, i64, ci]
        lib.wl_gen_u32.argtypes = [vp, i64, u64, u64, i64, ci]
        for f in (lib.wl_gen_i8, lib.wl_gen_bf16_normal, lib.wl_gen_u32):
            f.restype = None
        _lib = lib
    return _lib


def _ptr(a) -> int:
    """Address of a contiguous numpy array or CPU torch tensor."""
    if isinstance(a, np.ndarray):
        assert a.flags["C_CONTIGUOUS"]
        return a.ctypes.data
    assert a.is_contiguous() and a.device.type == "cpu"
    return a.data_ptr()


def fill_i8(dst, seed: int, stream: int, offset: int = 0, lo: int = -8, hi: int = 8):
    """Fill int8 ``dst`` with uniform integers in [lo, hi] (inclusive)."""
    n = dst.size if isinstance(dst, np.ndarray) else dst.numel()
    _load().wl_gen_i8(_ptr(dst), n, seed, stream, offset, lo, hi, NTHREADS)
    return dst


def fill_bf16_normal(dst, seed: int, stream: int, offset: int = 0):
    """Fill ``dst`` (uint16 / int16 / bfloat16 storage) with bf16 N(0,1)-like values."""
    n = dst.size if isinstance(dst, np.ndarray) else dst.numel()
    _load().wl_gen_bf16_normal(_ptr(dst), n, seed, stream, offset, NTHREADS)
    return dst


def fill_u32(dst, seed: int, stream: int, offset: int = 0):
    """Fill uint32 ``dst`` with uniform 32-bit words."""
    n = dst.size if isinstance(dst, np.ndarray) else dst.numel()
    _load().wl_gen_u32(_ptr(dst), n, seed, stream, offset, NTHREADS)
    return dst


def i8(n, seed, stream, offset=0, lo=-8, hi=8) -> np.ndarray:
    return fill_i8(np.empty(n, np.int8), seed, stream, offset, lo, hi)


def bf16_bits(n, seed, stream, offset=0) -> np.ndarray:
    return fill_bf16_normal(np.empty(n, np.uint16), seed, stream, offset)


def u32(n, seed, stream, offset=0) -> np.ndarray:
    return fill_u32(np.empty(n, np.uint32), seed, stream, offset)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bfloat16 bit patterns as float64."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# Stream ids: one per input tensor; per-round tensors add ROUND_STRIDE * round.
S_KEYS, S_HOST, S_QI_BASE, S_QI_FRESH, S_QI_SEL = 1, 2, 3, 4, 5
S_QI_XSEL, S_QI_XFRESH, S_QA, S_BLOCK, S_ACCEPT, S_RESID = 6, 7, 8, 9, 10, 11
S_QI_FSEL, S_QI_FFRESH = 12, 13
S_BLOCK_KEYS = 14
S_CROWS, S_CKEYS = 15, 16
ROUND_STRIDE = 1000


@dataclass(frozen=True)
class Recipe:
    """Shapes and seeds of one synthetic verification workload.

    N request slots, K verification queries per request (positions n..n+K-1),
    S committed history rows per request, an int8 indexer of H_idx heads of
    d_idx, top-k selections, GQA (Hq query heads per Hkv kv heads, head dim
    qk_dim / v_dim, row = K heads followed by V heads) or an MLA-like shared
    latent (kv_layout=1: one latent of qk_dim elements, values are its first
    v_dim elements), a hot cache of B rows per request, a draft ring window W
    with p rows per page, and optional residency of opt_frac of the history
    pages.

    Query correlation: within a round, query j of request r copies each
    element of the request's base query with probability rho_within and draws
    it fresh otherwise; from one round to the next the base query keeps each
    element with probability rho_cross.  Round 0 is the previous decode step
    that leaves the hot cache in the state the configuration describes.
    """
    name: str
    N: int
    K: int
    S: int
    H_idx: int
    d_idx: int
    topk: int
    Hq: int
    Hkv: int
    qk_dim: int
    v_dim: int
    kv_layout: int
    B: int
    rho_within: float
    rho_cross: float
    W: int = 2048
    p: int = 64
    K_max: int = 0
    opt_frac: float = 0.0
    seed: int = 0
    s_slack: int = 64
    i8_lo: int = -8      # indexer keys and queries are uniform over i8_lo..i8_hi
    i8_hi: int = 8
    m: int = 1           # token positions per stored row (eq. 8); S counts stored rows
    req0: int = 0        # request r of this recipe is request req0 + r of the workload

    @property
    def kmax(self) -> int:
        return self.K_max or self.K

    @property
    def row_elems(self) -> int:
        if self.kv_layout == 1:
            return self.qk_dim
        return self.Hkv * (self.qk_dim + self.v_dim)

    @property
    def row_bytes(self) -> int:
        return 2 * self.row_elems

    @property
    def s_max(self) -> int:
        return self.S + self.s_slack

    @property
    def idx_row(self) -> int:
        return self.H_idx * self.d_idx

    @property
    def opt_pages(self) -> int:
        return int(round(self.opt_frac * (self.S // self.p)))

    @property
    def opt_rows_max(self) -> int:
        return self.opt_pages * self.p

    def scaled(self, **kw) -> "Recipe":
        return replace(self, **kw)

    # ---- inputs -------------------------------------------------------
    def index_keys(self, r0: int, r1: int) -> np.ndarray:
        """int8 [r1-r0][s_max][H_idx*d_idx], uniform over i8_lo..i8_hi."""
        per = self.s_max * self.idx_row
        out = np.empty((r1 - r0, self.s_max, self.idx_row), np.int8)
        fill_i8(out, self.seed, S_KEYS, (self.req0 + r0) * per, self.i8_lo, self.i8_hi)
        return out

    def host_rows_into(self, dst, r0: int, r1: int):
        """Fill bf16 bits [r1-r0][s_max][row_elems] (numpy or pinned torch CPU)."""
        per = self.s_max * self.row_elems
        return fill_bf16_normal(dst, self.seed, S_HOST, (self.req0 + r0) * per)

    def host_rows(self, r0: int, r1: int) -> np.ndarray:
        out = np.empty((r1 - r0, self.s_max, self.row_elems), np.uint16)
        return self.host_rows_into(out, r0, r1)

    def _drift(self, x0: np.ndarray, rnd: int, s_sel: int, s_fresh: int, off: int) -> np.ndarray:
        """Round ``rnd`` version of x0: each round redraws each element with
        probability 1 - rho_cross and keeps it otherwise."""
        thr = np.uint64(int(self.rho_cross * 4294967296.0))
        x = x0
        for y in range(1, rnd + 1):
            sel = u32(x.size, self.seed, s_sel + ROUND_STRIDE * y, off)
            fresh = i8(x.size, self.seed, s_fresh + ROUND_STRIDE * y, off, self.i8_lo, self.i8_hi)
            keep = sel.astype(np.uint64).reshape(x.shape) < thr
            x = np.where(keep, x, fresh.reshape(x.shape))
        return x

    def index_queries(self, rnd: int, r0: int, r1: int) -> np.ndarray:
        """int8 [r1-r0][K_max][H_idx*d_idx] for round ``rnd``.

        Query j of request r takes each element from the request's base query
        with probability rho_within (a fixed choice per element) and from its
        own private draw otherwise; base and private draws drift from round to
        round as ``_drift`` describes, so a query keeps about rho_cross of its
        elements from the previous step.
        """
        E, Km, n = self.idx_row, self.kmax, r1 - r0
        r0 += self.req0
        lo, hi = self.i8_lo, self.i8_hi
        base = i8(n * E, self.seed, S_QI_BASE, r0 * E, lo, hi).reshape(n, 1, E)
        base = self._drift(base, rnd, S_QI_XSEL, S_QI_XFRESH, r0 * E)
        off = r0 * Km * E
        own = i8(n * Km * E, self.seed, S_QI_FRESH, off, lo, hi).reshape(n, Km, E)
        own = self._drift(own, rnd, S_QI_FSEL, S_QI_FFRESH, off)
        sel = u32(n * Km * E, self.seed, S_QI_SEL, off).reshape(n, Km, E)
        thr = np.uint64(int(self.rho_within * 4294967296.0))
        keep = sel.astype(np.uint64) < thr
        return np.where(keep, base, own).astype(np.int8)

    def attn_queries(self, rnd: int, r0: int, r1: int) -> np.ndarray:
        """bf16 bits [r1-r0][K_max][Hq][qk_dim]."""
        per = self.kmax * self.Hq * self.qk_dim
        out = np.empty((r1 - r0, self.kmax, self.Hq, self.qk_dim), np.uint16)
        return fill_bf16_normal(out, self.seed, S_QA + ROUND_STRIDE * rnd, (self.req0 + r0) * per)

    def block_rows(self, rnd: int, r0: int, r1: int) -> np.ndarray:
        """bf16 bits [r1-r0][K_max][row_elems]: K/V rows the target computes for the block."""
        per = self.kmax * self.row_elems
        out = np.empty((r1 - r0, self.kmax, self.row_elems), np.uint16)
        return fill_bf16_normal(out, self.seed, S_BLOCK + ROUND_STRIDE * rnd, (self.req0 + r0) * per)

    @property
    def cmax(self) -> int:
        """Stored rows one round can complete: ceil(K_max / m)."""
        return (self.kmax + self.m - 1) // self.m

    def compressed_rows(self, rnd: int, r0: int, r1: int) -> np.ndarray:
        """bf16 bits [r1-r0][cmax][row_elems]: stored rows a compressor gives
        the rows round ``rnd`` completes, N(0, 1)."""
        per = self.cmax * self.row_elems
        out = np.empty((r1 - r0, self.cmax, self.row_elems), np.uint16)
        return fill_bf16_normal(out, self.seed, S_CROWS + ROUND_STRIDE * rnd, (self.req0 + r0) * per)

    def compressed_keys(self, rnd: int, r0: int, r1: int) -> np.ndarray:
        """int8 [r1-r0][cmax][H_idx*d_idx]: index keys of those rows."""
        per = self.cmax * self.idx_row
        out = np.empty((r1 - r0, self.cmax, self.idx_row), np.int8)
        fill_i8(out, self.seed, S_CKEYS + ROUND_STRIDE * rnd, (self.req0 + r0) * per,
                self.i8_lo, self.i8_hi)
        return out

    def block_index_keys(self, rnd: int, r0: int, r1: int) -> np.ndarray:
        """int8 [r1-r0][K_max][H_idx*d_idx]: index keys the target computes for
        the block rows, uniform over i8_lo..i8_hi."""
        per = self.kmax * self.idx_row
        out = np.empty((r1 - r0, self.kmax, self.idx_row), np.int8)
        fill_i8(out, self.seed, S_BLOCK_KEYS + ROUND_STRIDE * rnd, (self.req0 + r0) * per,
                self.i8_lo, self.i8_hi)
        return out

    def k_per_req(self) -> np.ndarray:
        return np.full(self.N, self.K, np.int32)

    def accepted(self, rnd: int, k_per_req: Optional[np.ndarray] = None) -> np.ndarray:
        """int32 [N]: rows kept at commit, uniform over 0..K_r."""
        kr = self.k_per_req() if k_per_req is None else k_per_req
        w = u32(self.N, self.seed, S_ACCEPT + ROUND_STRIDE * rnd, self.req0).astype(np.uint64)
        return ((w * (kr.astype(np.uint64) + 1)) >> np.uint64(32)).astype(np.int32)

    def residency_rows(self, r: int) -> np.ndarray:
        """Ascending int32 rows of the whole pages made optional-resident for request r."""
        m = self.opt_pages
        if m == 0:
            return np.zeros(0, np.int32)
        n_pages = self.S // self.p
        keys = u32(n_pages, self.seed, S_RESID, (self.req0 + r) * n_pages)
        order = np.lexsort((np.arange(n_pages), keys))
        pages = np.sort(order[:m]).astype(np.int64)
        rows = (pages[:, None] * self.p + np.arange(self.p)[None, :]).reshape(-1)
        return rows.astype(np.int32)


# Query-correlation constants, chosen once by measuring with the oracle the
# top-k overlaps they produce on each shape (round 1 against round 0, and
# between the queries of one request); the workload tests re-measure them.
#   cfg1: ~48% of the previous step's top-k at seed 0 (rho_cross 0.90; the
#         single 256-row selection makes this ratio noisy across seeds)
#   cfg2: ~62% pairwise within a request, ~69% with the previous step
#   cfg3: ~60% pairwise within a request, ~49% with the previous step
#   cfg4: independent queries, ~50% with the previous step
CONFIGS = {
    # 1. Non-speculative single query, one request.
    "cfg1": Recipe("cfg1_single_query_S4096", N=1, K=1, S=4096, H_idx=1, d_idx=64,
                   topk=256, Hq=8, Hkv=1, qk_dim=128, v_dim=128, kv_layout=0,
                   B=512, rho_within=0.0, rho_cross=0.90),
    # 2. DSpark-style verification, K=4, batch 8, S=32768, ring window 2048.
    "cfg2": Recipe("cfg2_dspark_K4_N8_S32768", N=8, K=4, S=32768, H_idx=1, d_idx=64,
                   topk=2048, Hq=8, Hkv=1, qk_dim=128, v_dim=128, kv_layout=0,
                   B=4096, rho_within=0.93, rho_cross=0.92),
    # 3. DFlash2-style block of 8, batch 128, S=102400, 4 indexer heads summed.
    "cfg3": Recipe("cfg3_dflash2_K8_N128_S102400", N=128, K=8, S=102400, H_idx=4,
                   d_idx=128, topk=2048, Hq=16, Hkv=1, qk_dim=128, v_dim=128,
                   kv_layout=0, B=4096, rho_within=0.95, rho_cross=0.90),
    # 4. Long-context pressure: S=524288, MLA-like latent 576 (values = first 512).
    "cfg4": Recipe("cfg4_mla_K4_N64_S524288", N=64, K=4, S=524288, H_idx=1, d_idx=128,
                   topk=2048, Hq=16, Hkv=1, qk_dim=576, v_dim=512, kv_layout=1,
                   B=2048, opt_frac=0.10, rho_within=0.0, rho_cross=0.92),
}

# 5. Load-adaptive sweep on cfg3's shapes.
SWEEP_OPT = (0.0, 0.05, 0.25, 1.0)
SWEEP_K = (1, 2, 4, 8)


def sweep_recipe(opt_frac: float) -> Recipe:
    return replace(CONFIGS["cfg3"], name="cfg5_sweep_opt%g" % opt_frac,
                   opt_frac=opt_frac, K_max=8)
