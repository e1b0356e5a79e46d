"""Every rank's view of a workload (dsa_dcp_shard_seqs, through
dcp.ShardedLayer) against the oracle's ownership rule.  Each rank
holds exactly the tokens it owns, numbered in token order; each query's local
causal bound is its last owned token at or before its position; a rank's
local token l reads the same cache row as global token global(l), through a
page-table slice (interleave a whole number of pages) or a gathered shard."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from dsa_sparse_mla_query_gb300 import inputs as I
from dsa_sparse_mla_query_gb300.dcp import ShardedLayer
import oracle

pytestmark = pytest.mark.gpu
W = I.WORKLOADS
DEV = "cuda"


def _local_rows(view, b, n):
    """Physical rows of a rank's first n local tokens of sequence b."""
    s = view.seqs
    j = torch.arange(n, dtype=torch.int64)
    if s.page_table is not None:
        return s.page_table[b].cpu().to(torch.int64)[j // s.page_size] * s.page_size + j % s.page_size
    return s.seq_base[b].cpu() + j


@pytest.mark.parametrize("name,world,inter", [
    ("paged", 4, 64), ("paged", 3, 128), ("paged", 2, 1), ("tiny", 3, 5), ("specv", 2, 64),
])
def test_rank_views_follow_the_ownership_rule(name, world, inter):
    ctx = {"paged": (700, 1500, 4163), "tiny": None, "specv": None}[name]
    wl = W[name]
    if ctx:
        wl = I.scaled(wl, num_seqs=len(ctx), ctx=None, ctx_list=ctx)
    elif name == "specv":
        wl = I.scaled(wl, num_seqs=3, ctx_range=(2100, 3000))
    d = I.make_inputs(wl, DEV)
    lay = d["layout"]
    sh = ShardedLayer(d, wl.queries_per_seq, wl.topk, world, inter, device=DEV)
    by_pages = lay.page_table is not None and inter % lay.page_size == 0
    keys = d["k_idx"].cpu()
    for r, v in enumerate(sh.views):
        ctx_r = v.seqs.ctx_len.tolist()
        bound = v.bound.tolist()
        assert (v.seqs.page_table is not None) == by_pages
        for b, c in enumerate(lay.ctx_len):
            owned = [t for t in range(c) if oracle.dcp_owner(t, world, inter) == r]
            assert ctx_r[b] == len(owned)
            assert [oracle.dcp_local(t, world, inter) for t in owned] == list(range(len(owned)))
            glob_rows = lay.phys_rows(b)[torch.tensor(owned, dtype=torch.int64)]
            loc = _local_rows(v, b, len(owned))
            if by_pages:
                assert torch.equal(loc, glob_rows), f"rank {r} seq {b}: page slice maps the wrong rows"
            else:
                assert torch.equal(v.k_idx.cpu()[loc], keys[glob_rows]), f"rank {r} seq {b}: gathered rows differ"
        for t, (b, pos) in enumerate(zip(lay.q_seq, lay.q_pos)):
            last = max(u for u in range(pos + 1) if oracle.dcp_owner(u, world, inter) == r)
            assert bound[t] == oracle.dcp_local(last, world, inter)
        assert torch.equal(v.seqs.q_rope_pos.cpu(), d["q_pos"].cpu())


def test_a_rank_without_tokens_is_refused():
    """A query before any token of some rank: the view cannot be built."""
    wl = I.scaled(W["tiny"], num_seqs=1, ctx=300, queries_per_seq=1)
    d = I.make_inputs(wl, DEV)
    with pytest.raises(ValueError, match="owns no token"):
        ShardedLayer(d, 1, wl.topk, 4, 128, device=DEV)
