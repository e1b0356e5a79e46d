"""Decode context parallelism with every rank's shard in one GPU's memory.

A layer whose index-key and latent caches are sharded by token over `world`
ranks (turns of `interleave` tokens go round the ranks), run through one
rank's calls per rank (include/dsa.h, DCP): each rank scores its own keys and
offers its local top-k as packed candidates, the selector merges the lists in
place into the global top-k, each rank compacts the slots it owns and attends
over them, and the partial outputs are LSE-combined ("Day 0 support for
Mistral Large 4", Long context: decode and prefill context parallelism).

Setup builds each rank's view of a workload with dsa_dcp_shard_seqs: its
local token counts, the local causal bound of every query (the last token it
owns at or before the query's position) with the query's absolute position
for RoPE and SSMax, and, when the interleave is a whole number of pages, its
page table (its tokens are then whole pages of the shared caches); otherwise
its rows are gathered into contiguous shard caches, as a rank that holds only
its own tokens would have them.  Only
marshalling and that setup happen here; every step of the layer runs in the
library's kernels.
"""

from __future__ import annotations

from typing import List, Optional

import numpy as np
import torch

from . import _binding as B


def owner(t, world: int, interleave: int):
    return (t // interleave) % world


def local_pos(t, world: int, interleave: int):
    return (t // (interleave * world)) * interleave + t % interleave


class RankView:
    """One rank's shard: its dsa_seqs view and its caches."""

    def __init__(self, seqs: B.Seqs, k_idx, k_scale, latent, latent2, max_ctx: int):
        self.seqs, self.k_idx, self.k_scale, self.latent, self.latent2 = seqs, k_idx, k_scale, latent, latent2
        self.max_ctx = max_ctx


class ShardedLayer:
    """Owns the per-rank views, buffers and workspace; ``run()`` enqueues one
    sharded layer (and the shared-indexer layer when the workload has one,
    reusing the merged selection)."""

    def __init__(self, d: dict, queries_per_seq: int, k: int, world: int, interleave: int, device="cuda"):
        lay = d["layout"]
        self.d, self.k, self.world, self.interleave = d, int(k), int(world), int(interleave)
        self.num_q = Q = len(lay.q_pos)
        self.k_fp8 = d["k_idx"].dtype == torch.uint8
        self.lat_fp8 = d["latent"].dtype == torch.uint8
        self.shared = "q_mla2" in d
        q_pos = np.asarray(lay.q_pos, np.int64)
        q_seq = np.asarray(lay.q_seq, np.int64)
        ps = lay.page_size
        by_pages = lay.page_table is not None and interleave % ps == 0
        self.views: List[RankView] = []
        self.shards = [B.DcpShard(world, r, interleave) for r in range(world)]
        rope_pos = d["q_pos"]  # absolute positions
        full = B.Seqs(d["ctx_len"], d["q_start"], d["q_pos"], max_ctx=max(lay.ctx_len),
                      max_q_per_seq=queries_per_seq, num_rows=lay.num_rows, page_table=d.get("page_table"),
                      page_size=ps, seq_base=d.get("seq_base"))
        for r in range(world):
            shard = self.shards[r]
            # the rank's view from the library: local lengths, causal bounds and,
            # for page-aligned turns, its page table
            ctx_t = torch.empty(len(lay.ctx_len), dtype=torch.int32, device=device)
            bound_t = torch.empty(Q, dtype=torch.int32, device=device)
            lmaxp = (lay.max_pages + world - 1) // world + 1 if by_pages else 0
            table = torch.empty(len(lay.ctx_len), max(lmaxp, 1), dtype=torch.int32, device=device) if by_pages else None
            status = torch.zeros(1, dtype=torch.int32, device=device)
            lmax = B.dsa_dcp_shard_seqs(full, Q, shard, ctx_t, bound_t, table, lmaxp, status)
            ctx_r = ctx_t.cpu().tolist()
            if int(status.item()) != 0 or min(ctx_r) < 1:
                raise ValueError(f"rank {r} owns no token at or before some query's position; use longer contexts "
                                 "or fewer ranks")
            if by_pages:
                seqs = B.Seqs(ctx_t, d["q_start"], bound_t, max_ctx=lmax, max_q_per_seq=queries_per_seq,
                              num_rows=lay.num_rows, page_table=table, page_size=ps, q_rope_pos=rope_pos)
                view = RankView(seqs, d["k_idx"], d.get("k_scale"), d["latent"], d.get("latent2"), lmax)
            else:
                # a contiguous shard cache of the rank's own rows (what a rank
                # holds in a real deployment; here gathered from the full cache)
                rows_r = []
                for b, c in enumerate(lay.ctx_len):
                    t = np.arange(c, dtype=np.int64)
                    mine = owner(t, world, interleave) == r
                    rows_r.append(lay.phys_rows(b)[torch.from_numpy(np.flatnonzero(mine))])
                rows = torch.cat(rows_r).to(device)
                base = torch.tensor(np.concatenate([[0], np.cumsum(ctx_r)[:-1]]), dtype=torch.int64, device=device)
                seqs = B.Seqs(ctx_t, d["q_start"], bound_t, max_ctx=lmax, max_q_per_seq=queries_per_seq,
                              num_rows=int(rows.shape[0]), seq_base=base, q_rope_pos=rope_pos)
                ks = d["k_scale"].index_select(0, rows) if self.k_fp8 else None
                lat2 = d["latent2"].index_select(0, rows) if self.shared else None
                view = RankView(seqs, d["k_idx"].index_select(0, rows), ks, d["latent"].index_select(0, rows), lat2,
                                lmax)
            view.bound = bound_t
            self.views.append(view)
        # buffers
        kk = self.k
        self.ws_bytes = max(B.dsa_workspace_size(v.seqs, Q, kk) for v in self.views)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)
        for v in self.views:
            v.ld = (v.max_ctx + 3) // 4 * 4
            v.scores = torch.empty(Q, v.ld, dtype=torch.float32, device=device)
            v.idx = torch.empty(Q, kk, dtype=torch.int32, device=device)
            v.len = torch.empty(Q, dtype=torch.int32, device=device)
            v.cand = torch.empty(Q, kk, dtype=torch.int64, device=device)
            v.lidx = torch.empty(Q, kk, dtype=torch.int32, device=device)
            v.llen = torch.empty(Q, dtype=torch.int32, device=device)
            v.out = torch.empty(Q, 64, 512, dtype=torch.bfloat16, device=device)
            v.lse = torch.empty(Q, 64, dtype=torch.float32, device=device)
            if self.shared:
                v.out2, v.lse2 = torch.empty_like(v.out), torch.empty_like(v.lse)
        self.idx = torch.empty(Q, kk, dtype=torch.int32, device=device)
        self.topk_len = torch.empty(Q, dtype=torch.int32, device=device)
        self.out = torch.empty(Q, 64, 512, dtype=torch.bfloat16, device=device)
        self.lse = torch.empty(Q, 64, dtype=torch.float32, device=device)
        if self.shared:
            self.out2, self.lse2 = torch.empty_like(self.out), torch.empty_like(self.lse)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def run(self, stream=None, marks: Optional[list] = None):
        """One sharded layer.  ``marks``: optional list of 5 CUDA events,
        recorded before the ranks' indexers and after the candidates, the merge,
        the ranks' compaction + attention and the combine."""
        d, Q, kk = self.d, self.num_q, self.k
        kd = B.DSA_FP8_E4M3_ROWSCALE if self.k_fp8 else B.DSA_BF16
        ld_ = B.DSA_FP8_DS_MLA if self.lat_fp8 else B.DSA_BF16
        st = self.status

        def mark(i):
            if marks is not None:
                marks[i].record(stream if stream is not None else torch.cuda.current_stream())

        mark(0)
        for v, sh in zip(self.views, self.shards):
            B.dsa_index_scores(d["q_idx"], d["w"], d["ssmax_s"], d["ssmax_b"], d["inv_freq"], v.k_idx, v.k_scale, kd,
                               v.seqs, Q, v.scores, v.ld, self.ws, self.ws_bytes, st, stream)
            B.dsa_topk_candidates(v.scores, v.ld, v.seqs, Q, kk, sh, v.idx, v.len, v.cand, self.ws, self.ws_bytes, st,
                                  stream)
        mark(1)
        B.dsa_topk_merge([v.cand for v in self.views], kk, Q, kk, self.idx, self.topk_len, st, stream)
        mark(2)
        for v, sh in zip(self.views, self.shards):
            B.dsa_topk_compact(self.idx, self.topk_len, Q, kk, sh, v.lidx, v.llen, st, stream)
            B.sparse_mla_decode(d["q_mla"], v.latent, ld_, v.seqs, Q, v.lidx, v.llen, kk, d["sm_scale"], v.out, v.lse,
                                self.ws, self.ws_bytes, st, stream)
            if self.shared:
                B.sparse_mla_decode(d["q_mla2"], v.latent2, ld_, v.seqs, Q, v.lidx, v.llen, kk, d["sm_scale"], v.out2,
                                    v.lse2, self.ws, self.ws_bytes, st, stream)
        mark(3)
        B.dsa_lse_combine([v.out for v in self.views], [v.lse for v in self.views], Q, self.out, self.lse, stream)
        if self.shared:
            B.dsa_lse_combine([v.out2 for v in self.views], [v.lse2 for v in self.views], Q, self.out2, self.lse2,
                              stream)
        mark(4)

    def device_status(self) -> int:
        return int(self.status.item())
