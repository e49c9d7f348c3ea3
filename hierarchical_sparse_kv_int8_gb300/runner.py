"""Drive one KV source of the library over a synthetic workload recipe.

Plumbing only: allocates the pinned host tier and the device buffers with
torch, fills them from the seeded generators of ``workload``, binds every
request slot and issues the C-ABI calls of one verification round.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from . import Context, make_config


def config_for(rec, k_max: Optional[int] = None, opt_rows_max: Optional[int] = None,
               attn_pass: int = 0, topk_pass: int = 0, round_groups: int = 0):
    return make_config(
        n_slots=rec.N, k_max=k_max or rec.kmax, topk=rec.topk, s_max=rec.s_max,
        idx_heads=rec.H_idx, idx_dim=rec.d_idx, q_heads=rec.Hq, kv_heads=rec.Hkv,
        qk_dim=rec.qk_dim, v_dim=rec.v_dim, kv_layout=rec.kv_layout, budget=rec.B,
        ring_window=rec.W, page_rows=rec.p,
        opt_rows_max=rec.opt_rows_max if opt_rows_max is None else opt_rows_max,
        softmax_scale=0.0, attn_pass=attn_pass, topk_pass=topk_pass, round_groups=round_groups,
        tokens_per_row=rec.m)


class Runner:
    def __init__(self, rec, k_max: Optional[int] = None, opt_rows_max: Optional[int] = None,
                 stream=None, attn_pass: int = 0, topk_pass: int = 0, arenas=None, arena: int = 0,
                 role: int = 0, keys=None, round_groups: int = 0):
        """``arenas``/``arena``/``role``: a source of a layer group staging in a
        shared arena (a follower takes positions from a producer).  ``keys``:
        device index keys to bind instead of generating them (a follower
        never reads them)."""
        import torch
        self.torch = torch
        self.rec = rec
        self.cfg = config_for(rec, k_max, opt_rows_max, attn_pass, topk_pass, round_groups)
        self.Km = self.cfg.k_max
        self.ctx = Context(self.cfg, arenas, arena, role)
        self.stream = stream
        N, Sm, row = rec.N, rec.s_max, rec.row_elems
        self.host = torch.empty((N, Sm, row), dtype=torch.int16, pin_memory=True)
        rec.host_rows_into(self.host, 0, N)
        dev = torch.device("cuda")
        if keys is not None:
            self.keys = keys
        else:
            self.keys = torch.empty((N, Sm, rec.idx_row), dtype=torch.int8, device=dev)
            chunk = max(1, (1 << 30) // max(1, Sm * rec.idx_row))
            for r0 in range(0, N, chunk):
                r1 = min(N, r0 + chunk)
                self.keys[r0:r1].copy_(torch.from_numpy(rec.index_keys(r0, r1)))
        Km = self.Km
        self.q_idx = torch.zeros((N, Km, rec.idx_row), dtype=torch.int8, device=dev)
        self.q = torch.zeros((N, Km, rec.Hq, rec.qk_dim), dtype=torch.int16, device=dev)
        self.block = torch.zeros((N, Km, row), dtype=torch.int16, device=dev)
        self.topk = torch.full((N, Km, rec.topk), -1, dtype=torch.int32, device=dev)
        self.loc = torch.full((N, Km, rec.topk), -1, dtype=torch.int32, device=dev)
        self.out = torch.zeros((N, Km, rec.Hq, rec.v_dim), dtype=torch.bfloat16, device=dev)
        self.lse = torch.zeros((N, Km, rec.Hq), dtype=torch.float32, device=dev)
        for r in range(N):
            self.ctx.bind(r, self.host[r], self.keys[r], rec.S * rec.m, stream)

    def rebind(self):
        """Bind every slot again at the recipe's history length: empty hot
        cache, no optional rows, no live ring rows (rows the previous rounds
        committed past the history stay in the host tier, unused)."""
        for r in range(self.rec.N):
            self.ctx.bind(r, self.host[r], self.keys[r], self.rec.S * self.rec.m, self.stream)

    def set_residency(self, frac_rows=None):
        for r in range(self.rec.N):
            rows = self.rec.residency_rows(r) if frac_rows is None else frac_rows(r)
            self.ctx.set_residency(r, rows, self.stream)

    def load_round(self, rnd: int):
        """Copy round ``rnd``'s query and block inputs to the device buffers."""
        torch, rec, Km = self.torch, self.rec, self.Km
        qi = rec.index_queries(rnd, 0, rec.N)
        qa = rec.attn_queries(rnd, 0, rec.N)
        bl = rec.block_rows(rnd, 0, rec.N)
        self.q_idx[:, :qi.shape[1]].copy_(torch.from_numpy(qi))
        self.q[:, :qa.shape[1]].copy_(torch.from_numpy(qa.view(np.int16)))
        self.block[:, :bl.shape[1]].copy_(torch.from_numpy(bl.view(np.int16)))

    def select(self, k_per_req, pos=None):
        self.ctx.select(self.q_idx, k_per_req, self.topk, pos, self.stream)

    def adopt(self, k_per_req, topk, pos=None):
        """Take a producer's selection (its top-k tensor) for this round."""
        self.topk = topk
        self.ctx.adopt(k_per_req, pos, self.stream)

    def resolve(self, shared=True):
        self.ctx.resolve(self.topk, self.loc, shared, self.stream)

    def attend(self):
        self.ctx.attend(self.q, self.block, self.loc, self.out, self.lse, self.stream)

    def commit(self, accepted):
        self.ctx.commit(accepted, self.stream)

    def commit_compressed(self, rnd: int, accepted):
        """Commit of a compressed source (rec.m > 1) with round ``rnd``'s
        compressor rows and keys from the recipe."""
        torch, rec = self.torch, self.rec
        if not hasattr(self, "crows"):
            cm = rec.cmax
            self.crows = torch.zeros((rec.N, cm, rec.row_elems), dtype=torch.int16, device="cuda")
            self.ckeys = torch.zeros((rec.N, cm, rec.idx_row), dtype=torch.int8, device="cuda")
        self.crows.copy_(torch.from_numpy(rec.compressed_rows(rnd, 0, rec.N).view(np.int16)))
        self.ckeys.copy_(torch.from_numpy(rec.compressed_keys(rnd, 0, rec.N)))
        self.ctx.commit_compressed(accepted, self.crows, self.ckeys, self.stream)

    def round_fused(self, k_per_req, accepted):
        """The whole round in one dhs_round call (request groups on internal
        streams when the config asks for them)."""
        self.ctx.round(self.q_idx, k_per_req, self.q, self.block, accepted, self.topk, self.loc,
                       self.out, self.lse, self.stream)

    def round(self, k_per_req, accepted, shared=True):
        self.select(k_per_req)
        self.resolve(shared)
        self.attend()
        self.commit(accepted)

    def export(self, which, dtype, shape):
        t = self.torch.empty(shape, dtype=dtype, device="cuda")
        self.ctx.export(which, t, self.stream)
        return t
