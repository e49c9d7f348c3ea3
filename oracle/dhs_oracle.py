"""Oracle for the verification hot path of Adaptive DHiSparse.

TEST INFRASTRUCTURE ONLY.  This module is a plain, slow CPU restatement of
what the hot path computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import or call it; the library in
``hierarchical_sparse_kv_int8_gb300`` never does, and shares no code with it.
Inputs reach both sides only through the seeded generators of ``workload``.

Source: "Adaptive DHiSparse: Speculative Decoding over a Load-Adaptive KV
Hierarchy" (arXiv 2610.13708), cited below as [ADHS] with its section,
equation or figure; the blog "Adaptive DHiSparse: technical breakdown" is
cited as [blog] where it fills a detail the paper leaves open.

Arithmetic: index scores are exact int64; attention uses float64 for every
product, softmax and accumulation over the exact bfloat16 input values.

Parity pins (each checked by ``tests/test_oracle_*.py`` against something
other than this file):
  ring_rows, ring_address, staging_bytes   worked examples of [ADHS] 3.4
  index_scores                             naive triple loop on tiny inputs
  topk_ordered                             brute-force sort, ties, k >= |domain|
  union / miss set                         set algebra of [ADHS] eq. (6),
                                           Fig. 3 callout 2, |U| <= K k, D in H
  attention                                k = S equals dense causal attention
                                           (a library routine), closed forms
  commit / rollback                        Fig. 3 example, stage-K-then-commit-a
                                           equals stage-a-then-commit-a
  append_keys                              kept rows' key rows equal the block's,
                                           the rest untouched; the next round's
                                           hand-computed maximum score puts exactly
                                           the kept rows first
  source sharing (adopt, Reindex, Reuse)   a follower's attention equals attention
                                           over its own rows at the producer's
                                           positions; a Reindex selection misses
                                           exactly the rows absent after the first
                                           selection's update; a Reuse consumer's
                                           output is attention over the inherited
                                           rows (fp64 closed computation)
  residency policy                         eq. (4) against numpy searchsorted over
                                           the cumulative pages, a hand-worked
                                           trace (tests/golden), eq. (3) and the
                                           reclaim invariants on random sequences
  LRU replacement                          invariants of [ADHS] 3.2 and one
                                           hand-worked trace.  Beyond those the
                                           replacement order (one clock tick per
                                           resolve call, victims by (stamp,
                                           slot), overflow misses by ascending
                                           row) is this file's reading and is
                                           "parity unpinned" by the pages.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

# Location tags of [ADHS] eq. (12): tier in bits 29..28, index below.
RING, OPT, HOT, STAGE = 0, 1, 2, 3
TIER_SHIFT = 28
INDEX_MASK = (1 << TIER_SHIFT) - 1


def encode_loc(tier: int, index: int) -> int:
    return (tier << TIER_SHIFT) | index


def decode_loc(loc: int):
    return loc >> TIER_SHIFT, loc & INDEX_MASK


# ---------------------------------------------------------------------------
# Sizing formulas, [ADHS] 3.4
# ---------------------------------------------------------------------------
def ring_rows(W: int, p: int, K_max: int) -> int:
    """Draft ring rows per request: p * ceil((W + p - 1 + K_max) / p), [ADHS] eq. (9).

    A drafter that reads at most W prior positions needs the window plus its
    current block of at most K_max positions; page alignment adds at most p-1.
    """
    return p * ((W + p - 1 + K_max + p - 1) // p)


def ring_address(i: int, t: int, R_d: int) -> int:
    """Physical ring row of draft position t of request slot i, [ADHS] eq. (10)."""
    return i * R_d + (t % R_d)


def staging_bytes(chi: int, N: int, K_max: int, k: int, d_kv: int) -> int:
    """Verification staging reservation M_stage = chi N K_max k d_KV, [ADHS] 3.4."""
    return chi * N * K_max * k * d_kv


# ---------------------------------------------------------------------------
# Selection, [ADHS] 2.1 eq. (1) and 3.3 eq. (5)
# ---------------------------------------------------------------------------
def domain_length(n: int, pos: Optional[int], m: int = 1) -> int:
    """Selectable history rows of a query at position ``pos``.

    [ADHS] eq. (5) splits the visible set of query j into the committed
    history v < n (served through the hierarchy, hence selectable) and the
    current block, which is read from the tail and not selected.  A query
    placed inside the history (pos < n) sees rows v <= pos only.  For a
    source packing m token positions into a row (eq. 8), n counts complete
    rows and row s holds positions s m .. s m + m - 1, so a query at ``pos``
    sees the complete rows whose last position is at most pos: s < (pos+1)//m.
    """
    if pos is None:
        return n
    return max(0, min(n, (pos + 1) // m))


def completed_rows(n_tok: int, a: int, m: int) -> range:
    """Source rows a round completes, [ADHS] eq. (8): committing a of the
    block's positions moves the token frontier from n_tok to n_tok + a, and
    the rows floor(n_tok / m) <= s < floor((n_tok + a) / m) become complete
    (the bracket of the equation's upper bound is garbled on the page; the
    floor is the reading under which a partial group stays in the tail)."""
    return range(n_tok // m, (n_tok + a) // m)


def index_scores(q: np.ndarray, keys: np.ndarray, dom: int) -> np.ndarray:
    """I[s] = sum over indexer heads h and dims d of q[h,d] * K[s,h,d], [ADHS] eq. (1).

    ``q`` is int8 [H_idx*d_idx], ``keys`` int8 [rows][H_idx*d_idx]; the head
    sum follows the multi-head indexer of [blog] (per-head scores added).
    Exact int64 arithmetic over the first ``dom`` rows.
    """
    return keys[:dom].astype(np.int64) @ q.astype(np.int64)


def topk_ordered(scores: np.ndarray, k: int) -> np.ndarray:
    """The model's ordered top-k list, [ADHS] 2.1 eq. (1).

    Rows are ordered by score descending and, among equal scores, by row
    index ascending (the lower index wins a tie); the first min(k, |domain|)
    are kept and the list is padded with -1 to length k.
    """
    dom = scores.shape[0]
    order = np.lexsort((np.arange(dom), -scores))
    out = np.full(k, -1, np.int64)
    m = min(k, dom)
    out[:m] = order[:m]
    return out


def union_rows(selections: List[np.ndarray]) -> np.ndarray:
    """Retrieval union U_r of the K_r selections, ascending, [ADHS] eq. (6)."""
    vals = [s[s >= 0] for s in selections]
    if not vals:
        return np.zeros(0, np.int64)
    return np.unique(np.concatenate(vals)).astype(np.int64)


# ---------------------------------------------------------------------------
# Attention, [ADHS] eq. (1) with the visible set of eq. (5)
# ---------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def split_row(row: np.ndarray, kvh: int, cfg: "Config"):
    """Key and value vectors of kv head ``kvh`` in a stored row (float64)."""
    if cfg.kv_layout == 1:  # shared latent: keys are the latent, values its prefix
        return row[..., :cfg.qk_dim], row[..., :cfg.v_dim]
    k0 = kvh * cfg.qk_dim
    v0 = cfg.Hkv * cfg.qk_dim + kvh * cfg.v_dim
    return row[..., k0:k0 + cfg.qk_dim], row[..., v0:v0 + cfg.v_dim]


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """softmax(scale * K q) V and its log-sum-exp, all float64."""
    logits = scale * (K @ q)
    m = logits.max()
    w = np.exp(logits - m)
    z = w.sum()
    return (w @ V) / z, m + math.log(z)


# ---------------------------------------------------------------------------
# The per-source state machine: select, resolve, attend, commit, residency
# ---------------------------------------------------------------------------
@dataclass
class Config:
    n_slots: int
    k_max: int
    topk: int
    s_max: int
    idx_heads: int
    idx_dim: int
    q_heads: int
    Hkv: int
    qk_dim: int
    v_dim: int
    kv_layout: int
    budget: int
    ring_window: int = 2048
    page_rows: int = 64
    opt_rows_max: int = 0
    softmax_scale: float = 0.0
    tokens_per_row: int = 1    # m of [ADHS] eq. (8); 1 = uncompressed

    @property
    def m(self) -> int:
        return max(1, self.tokens_per_row)

    @property
    def row_elems(self) -> int:
        return self.qk_dim if self.kv_layout == 1 else self.Hkv * (self.qk_dim + self.v_dim)

    @property
    def R_d(self) -> int:
        return ring_rows(self.ring_window, self.page_rows, self.k_max)

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale > 0 else 1.0 / math.sqrt(self.qk_dim)


@dataclass
class Request:
    host: np.ndarray           # bf16 bits [s_max][row_elems]: host backing H_r
    keys: np.ndarray           # int8 [s_max][H_idx*d_idx]: GPU index state
    n: int                     # committed history rows (n_r when m = 1)
    ring_first: int            # first position ever committed through the ring
    hot_row: np.ndarray        # int64 [B], -1 = empty
    hot_stamp: np.ndarray      # int64 [B], -1 = never used
    hot_payload: np.ndarray    # bf16 bits [B][row_elems]
    ring: np.ndarray           # bf16 bits [R_d][row_elems]
    opt_slot: Dict[int, int] = field(default_factory=dict)
    opt_pool: Optional[np.ndarray] = None
    K: int = 0
    tok: int = 0               # committed token positions n_r (= n when m = 1)


@dataclass
class Stats:
    selections: int = 0
    union_rows: int = 0
    ring_hits: int = 0
    opt_hits: int = 0
    hot_hits: int = 0
    misses: int = 0
    miss_selections: int = 0
    host_rows_fetched: int = 0
    installs: int = 0
    evictions: int = 0
    direct_only: int = 0


class Oracle:
    """One KV source (layer) with N request slots, [ADHS] 3.1-3.5."""

    def __init__(self, cfg: Config):
        self.cfg = cfg
        self.t = 0
        self.req: Dict[int, Request] = {}
        self.stats = Stats()
        self.topk: Optional[np.ndarray] = None
        self.union: Dict[int, np.ndarray] = {}
        self.misses: Dict[int, np.ndarray] = {}
        self.uloc: Dict[int, np.ndarray] = {}
        self.promote: Dict[int, list] = {}
        self.staging: Dict[int, np.ndarray] = {}
        self.loc: Optional[np.ndarray] = None

    # -- binding ---------------------------------------------------------
    def bind(self, slot: int, host: np.ndarray, keys: np.ndarray, n: int):
        """``n``: committed token positions; the history holds n // m rows."""
        c = self.cfg
        self.req[slot] = Request(
            host=host, keys=keys, n=n // c.m, ring_first=n // c.m, tok=n,
            hot_row=np.full(c.budget, -1, np.int64),
            hot_stamp=np.full(c.budget, -1, np.int64),
            hot_payload=np.zeros((c.budget, c.row_elems), np.uint16),
            ring=np.zeros((c.R_d, c.row_elems), np.uint16),
            opt_pool=np.zeros((c.opt_rows_max, c.row_elems), np.uint16))

    def hot_map(self, r: int) -> Dict[int, int]:
        q = self.req[r]
        return {int(row): v for v, row in enumerate(q.hot_row) if row >= 0}

    # -- residency, [ADHS] 3.1 -------------------------------------------
    def set_residency(self, r: int, rows: np.ndarray):
        """Make ``rows`` the ready optional history of request r.

        Whole pages of imported history become optional ([ADHS] 3.1); the
        bytes are copied first and the ready locations published after the
        copy ("reserve, copy, publish").  Row i of the list occupies pool
        slot i.  Rows of the previous optional set become not ready.
        """
        c, q = self.cfg, self.req[r]
        rows = np.asarray(rows, np.int64)
        if len(rows) > c.opt_rows_max:
            raise ValueError("capacity")
        if len(np.unique(rows)) != len(rows) or (len(rows) and (rows.min() < 0 or rows.max() >= q.n)):
            raise ValueError("invalid")
        for i, s in enumerate(rows):
            q.opt_pool[i] = q.host[s]
        q.opt_slot = {int(s): i for i, s in enumerate(rows)}

    # -- step 1: select, [ADHS] eq. (1) ------------------------------------
    def select(self, q_idx: np.ndarray, k_per_req: np.ndarray, pos: Optional[np.ndarray] = None):
        """Top-k per verification query over its causal history domain."""
        c = self.cfg
        out = np.full((c.n_slots, c.k_max, c.topk), -1, np.int64)
        for r, q in self.req.items():
            q.K = int(k_per_req[r])
            for j in range(q.K):
                p = None if pos is None else int(pos[r][j])
                dom = domain_length(q.n, p, c.m)
                sc = index_scores(q_idx[r][j].reshape(-1), q.keys, dom)
                out[r, j] = topk_ordered(sc, c.topk)
        self.topk = out
        return out

    # -- a follower source takes another source's positions, [ADHS] 3.2 ----
    def adopt(self, topk: np.ndarray, k_per_req: np.ndarray):
        """A layer with its own payload takes the ordered selections another
        source's indexer announced (GLM-style index sharing: producers
        announce positions for several follower payload layers).  Nothing is
        scored; ``resolve`` then maps the same positions to this source's
        own cache and host rows, and ``attend`` reads this source's rows."""
        for r, q in self.req.items():
            q.K = int(k_per_req[r])
        self.topk = np.asarray(topk, np.int64).copy()
        return self.topk

    # -- steps 2-4: union, probe, compact, shared gather, [ADHS] 3.2-3.3 ---
    def resolve(self, topk: np.ndarray, shared: bool = True):
        """Turn the selected rows into device locations.

        Per request: the union U_r of the K_r selections (eq. 6) is probed in
        ascending row order: rows in the live tail of the draft ring first,
        then the ready optional map, then the hot cache (Fig. 2 callouts 1
        and 2; a row held in two places gets the first of these, 3.5).  The
        rest form D_r = U_r minus R_r; each distinct missing row is copied
        from host once into the staging arena and its location is returned to
        every query that selected it (3.3, Fig. 3 callout 2).

        Replacement (3.2): hot rows in U_r are protected; a hot hit refreshes
        its stamp to the call's tick t; victims are unprotected slots in
        order of (stamp, slot), empty slots first; the first min(|D_r|,
        #victims) missing rows, in ascending row order, take the victims in
        that order and are copied from staging into the hot cache after
        attention (3.4).

        ``shared=False`` is the per-query baseline: every selection of a
        missing row is fetched on its own into staging slot j*k + i; the
        cache state evolves exactly as in shared mode.
        """
        c = self.cfg
        self.t += 1
        t = self.t
        k = c.topk
        self.topk = topk
        loc = np.full((c.n_slots, c.k_max, k), -1, np.int64)
        st = self.stats
        for r, q in self.req.items():
            if q.K == 0:
                continue
            sel = [topk[r][j] for j in range(q.K)]
            U = union_rows(sel)
            ring_lo = max(q.ring_first, q.n - c.ring_window)
            hmap = self.hot_map(r)
            protected = set()
            uloc = np.zeros(len(U), np.int64)
            misses = []
            hits_here = 0
            for qi, u in enumerate(U):
                u = int(u)
                if u in hmap:
                    protected.add(hmap[u])
                if ring_lo <= u < q.n:
                    uloc[qi] = encode_loc(RING, u % c.R_d)
                    st.ring_hits += 1
                elif u in q.opt_slot:
                    uloc[qi] = encode_loc(OPT, q.opt_slot[u])
                    st.opt_hits += 1
                elif u in hmap:
                    uloc[qi] = encode_loc(HOT, hmap[u])
                    q.hot_stamp[hmap[u]] = t
                    hits_here += 1
                else:
                    uloc[qi] = encode_loc(STAGE, len(misses))
                    misses.append(u)
            st.union_rows += len(U)
            st.hot_hits += hits_here
            st.misses += len(misses)
            if not misses and hits_here == 0:
                st.direct_only += 1  # Fig. 2: steps 2 and 3 skipped

            # replacement: victims in (stamp, slot) order among unprotected slots
            cand = [v for v in range(c.budget) if v not in protected]
            cand.sort(key=lambda v: (int(q.hot_stamp[v]), v))
            P = min(len(misses), len(cand))
            promote = []
            for p in range(P):
                v = cand[p]
                if q.hot_row[v] >= 0:
                    st.evictions += 1
                q.hot_row[v] = misses[p]
                q.hot_stamp[v] = t
                promote.append([p, v])
            st.installs += P

            # locations, in each query's selection order ([ADHS] eq. 12)
            pos_in_u = {int(u): qi for qi, u in enumerate(U)}
            staging = np.zeros((c.k_max * k, c.row_elems), np.uint16)
            first_occ = {}
            for j in range(q.K):
                for i in range(k):
                    s = int(sel[j][i])
                    if s < 0:
                        continue
                    st.selections += 1
                    l = int(uloc[pos_in_u[s]])
                    tier, idx = decode_loc(l)
                    if tier == STAGE:
                        st.miss_selections += 1
                        if not shared:
                            l = encode_loc(STAGE, j * k + i)
                            staging[j * k + i] = q.host[s]
                            first_occ.setdefault(idx, j * k + i)
                    loc[r, j, i] = l
            if shared:
                for m, u in enumerate(misses):
                    staging[m] = q.host[u]
                st.host_rows_fetched += len(misses)
            else:
                for pr in promote:
                    pr[0] = first_occ[pr[0]]
                st.host_rows_fetched += sum(
                    1 for j in range(q.K) for i in range(k)
                    if loc[r, j, i] >= 0 and decode_loc(int(loc[r, j, i]))[0] == STAGE)
            self.union[r] = U
            self.misses[r] = np.asarray(misses, np.int64)
            self.uloc[r] = uloc
            self.promote[r] = promote
            self.staging[r] = staging
        self.loc = loc
        return loc

    def payload_at(self, r: int, loc: int) -> np.ndarray:
        """GPU payload KV[loc] of request r as the oracle's state holds it."""
        q = self.req[r]
        tier, idx = decode_loc(loc)
        if tier == RING:
            return q.ring[idx]
        if tier == OPT:
            return q.opt_pool[idx]
        if tier == HOT:
            return q.hot_payload[idx]
        return self.staging[r][idx]

    def check_placement(self):
        """[ADHS] eq. (11): KV[l_{r,j,i}] equals the original row c_{r, s_{r,j,i}}."""
        for r, q in self.req.items():
            for j in range(q.K):
                for i, s in enumerate(self.topk[r][j]):
                    if s < 0:
                        continue
                    got = self.payload_at(r, int(self.loc[r, j, i]))
                    if not np.array_equal(got, q.host[int(s)]):
                        raise AssertionError("placement broken at r=%d j=%d i=%d" % (r, j, i))

    # -- step 5: attend, then install promoted rows ------------------------
    def attend(self, q_attn: np.ndarray, block: np.ndarray):
        """Attention of every query over its own selection plus the block rows
        up to itself ([ADHS] eq. 5), reading the ORIGINAL rows c_{r,s}
        (eq. 11).  The block rows are staged in the draft ring at phi(r, n+u)
        (eq. 10).  Afterwards promoted rows move from staging to their hot
        slots (3.4).  Returns (out [N][K_max][Hq][v_dim], lse [N][K_max][Hq])
        in float64; entries of idle queries are NaN.
        """
        c = self.cfg
        out = np.full((c.n_slots, c.k_max, c.q_heads, c.v_dim), np.nan)
        lse = np.full((c.n_slots, c.k_max, c.q_heads), np.nan)
        group = c.q_heads // c.Hkv
        for r, q in self.req.items():
            if q.K == 0:
                continue
            for u in range(q.K):
                q.ring[(q.n + u) % c.R_d] = block[r][u]
            for j in range(q.K):
                sel = [int(s) for s in self.topk[r][j] if s >= 0]
                rows = [q.host[s] for s in sel] + [block[r][u] for u in range(j + 1)]
                R = bf16_to_f64(np.stack(rows))
                for h in range(c.q_heads):
                    Kh, Vh = split_row(R, h // group, c)
                    o, l = attention(bf16_to_f64(q_attn[r][j][h]), Kh, Vh, c.scale)
                    out[r, j, h] = o
                    lse[r, j, h] = l
            for src, v in self.promote.get(r, []):
                q.hot_payload[v] = self.staging[r][src]
        self.promote = {}
        return out, lse

    # -- commit / rollback, [ADHS] eq. (7) ---------------------------------
    def commit(self, accepted: np.ndarray):
        """Keep the first a_r block rows of every active request.

        a_r counts the rows kept: the anchor plus the accepted drafts, 1 + A_r
        in eq. (7); 0 rolls the whole block back.  Kept rows join the history
        (n_r <- n_r + a_r) and are written to the host backing, so every row
        not ready on the GPU keeps a host copy (eq. 6, D in H).  Rejected rows
        are never published: the frontier simply does not pass them.
        """
        c = self.cfg
        if c.m > 1:
            raise ValueError("invalid")  # compressed rows come from commit_compressed
        for r, q in self.req.items():
            a = int(accepted[r])
            if q.K and not (0 <= a <= q.K):
                raise ValueError("invalid")
            if q.K and q.n + a > c.s_max:
                raise ValueError("capacity")
        for r, q in self.req.items():
            if q.K == 0:
                continue
            a = int(accepted[r])
            for u in range(a):
                q.host[q.n + u] = q.ring[(q.n + u) % c.R_d]
            q.n += a
            q.tok += a
            q.K = 0

    def commit_compressed(self, accepted: np.ndarray, rows: np.ndarray,
                          row_keys: Optional[np.ndarray] = None):
        """Commit for a source packing m positions into a row, [ADHS] eq. (8).

        Keeping a_r positions moves the token frontier by a_r; the rows the
        round completes (``completed_rows``) join the immutable history with
        the payload and index keys the model's compressor gave them (rows[r][i]
        and row_keys[r][i] for the i-th completed row), written to the host
        backing as every committed row is.  A partial group stays in the
        tail: its positions count, no row of it is published.  Such rows
        never come from the draft ring (it holds the block's token rows), so
        the ring serves no history row of a compressed source.
        """
        c = self.cfg
        for r, q in self.req.items():
            a = int(accepted[r])
            if q.K and not (0 <= a <= q.K):
                raise ValueError("invalid")
            if q.K and (q.tok + a) // c.m > c.s_max:
                raise ValueError("capacity")
        for r, q in self.req.items():
            if q.K == 0:
                continue
            a = int(accepted[r])
            done = completed_rows(q.tok, a, c.m)
            for i, s in enumerate(done):
                q.host[s] = rows[r, i]
                if row_keys is not None:
                    q.keys[s] = row_keys[r, i]
            q.tok += a
            q.n = q.tok // c.m
            q.ring_first = q.n
            q.K = 0

    # -- index keys of kept rows, [ADHS] 3.3 with 2.2 ----------------------
    def append_keys(self, accepted: np.ndarray, block_keys: np.ndarray):
        """Rows a commit keeps join the history with their index keys.

        Called before that commit: key row n_r + u of request r becomes
        block_keys[r][u] for u < a_r (n_r the committed history at the
        call).  Later rounds score those rows like every other history row;
        the current round's domains end below n_r.
        """
        c = self.cfg
        if c.m > 1:
            raise ValueError("invalid")  # compressed rows bring their keys at commit
        for r in range(len(accepted)):
            a = int(accepted[r])
            if a < 0 or a > c.k_max or (a > 0 and r not in self.req):
                raise ValueError("invalid")
            if a and self.req[r].n + a > c.s_max:
                raise ValueError("capacity")
        for r, q in self.req.items():
            a = int(accepted[r])
            if a:
                q.keys[q.n:q.n + a] = block_keys[r, :a]

    def ring_live(self, r: int) -> Dict[int, np.ndarray]:
        """Live ring positions [max(first, n - W), n) and their rows."""
        c, q = self.cfg, self.req[r]
        lo = max(q.ring_first, q.n - c.ring_window)
        return {t: q.ring[t % c.R_d].copy() for t in range(lo, q.n)}


# ---------------------------------------------------------------------------
# Residency policy of optional history, [ADHS] 3.1, eq. (3) and (4)
# ---------------------------------------------------------------------------
def reclaim_prefix(a: List[int], delta: int) -> Optional[int]:
    """Eq. (4): the least q with a_1 + ... + a_q >= delta, walking the reclaim
    order; None when even all of them fall short (the admission waits)."""
    if delta <= 0:
        return 0
    s = 0
    for q, pages in enumerate(a, start=1):
        s += pages
        if s >= delta:
            return q
    return None


class ResidencyPolicy:
    """Page accounting of [ADHS] 3.1 under the budget of eq. (3):
    required + optional + reserve <= total.  Readings where the section
    leaves a choice: the reclaim order is the admission order; an admitted
    request keeps min(history, free pages) optional pages (resident-first
    admission; after a reclaim the new request takes the freed pages); a
    repopulation attempt walks the admitted requests cyclically from just
    after the last one the previous attempt served, giving each up to its
    unmet history until the attempt's bound or the free pages run out."""

    def __init__(self, total: int, reserve: int):
        self.total, self.reserve = total, reserve
        self.reqs: List[dict] = []  # admission order
        self.cursor = 0

    def free(self) -> int:
        return self.total - self.reserve - sum(r["required"] + r["optional"] for r in self.reqs)

    def admit(self, rid: int, required: int, history: int):
        # eq. (3) cannot hold a request whose required pages exceed the whole
        # budget less the reserve, even with no other request admitted: it
        # could only wait forever, so it is refused
        if required > self.total - self.reserve:
            raise ValueError("capacity")
        free = self.free()
        freed, reclaimed = 0, []
        if required > free:
            q = reclaim_prefix([r["optional"] for r in self.reqs], required - free)
            if q is None:
                return False, 0, []
            for r in self.reqs[:q]:
                if r["optional"] > 0:
                    reclaimed.append(r["id"])
                    freed += r["optional"]
                    r["optional"] = 0
        opt = min(history, free + freed - required)
        self.reqs.append(dict(id=rid, required=required, history=history, optional=opt))
        return True, opt, reclaimed

    def complete(self, rid: int):
        i = [r["id"] for r in self.reqs].index(rid)
        del self.reqs[i]
        if i < self.cursor:
            self.cursor -= 1
        if self.cursor >= len(self.reqs):
            self.cursor = 0

    def repopulate(self, max_pages: int):
        budget = min(max_pages, self.free())
        n, out, nxt = len(self.reqs), [], self.cursor
        for k in range(n):
            if budget <= 0:
                break
            i = (self.cursor + k) % n
            r = self.reqs[i]
            give = min(r["history"] - r["optional"], budget)
            if give <= 0:
                continue
            r["optional"] += give
            budget -= give
            out.append((r["id"], give))
            nxt = (i + 1) % n
        self.cursor = nxt
        return out

    def query(self, rid: int):
        r = next(x for x in self.reqs if x["id"] == rid)
        return r["required"], r["optional"], r["history"]
