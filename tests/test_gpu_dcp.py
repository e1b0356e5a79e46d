"""Parity of one rank's DCP calls (through the C ABI) with the CPU oracle on a
GB300, and of a whole layer sharded over several ranks on one GPU with the
oracle's unsharded layer ("Day 0 support for Mistral Large 4", Long context:
decode and prefill context parallelism).

Candidates, the selector and compaction are integer work: bit-exact against
the oracle.  The LSE combine rounds an fp32 sum to bf16: within one bf16
rounding plus fp32 noise.  The sharded layer must select what the unsharded
oracle selects (boundary ties within the top-k tolerance) and attend like the
oracle over that selection.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import dsa_sparse_mla_query_gb300 as dsa
from dsa_sparse_mla_query_gb300 import inputs as I
from dsa_sparse_mla_query_gb300.dcp import ShardedLayer
from dsa_sparse_mla_query_gb300.runner import DecodeStep
import oracle
import parity as P

pytestmark = pytest.mark.gpu

DEV = "cuda"
W = I.WORKLOADS


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    dsa.load()
    yield
    torch.cuda.synchronize()


def _u64(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint64)


def _tied_scores(seed, tid, n):
    """Seeded scores on a 0.25 grid (exact in fp32, many ties)."""
    x = I.normal(I.stream_key(seed, tid), I._counters(0, n, DEV)).to(torch.float32)
    return torch.round(x * 8) / 4


def _contig_seqs(ctx, qpos, qps):
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device=DEV)
    qs = torch.tensor([i * qps for i in range(len(ctx) + 1)], dtype=torch.int32, device=DEV)
    qp = torch.tensor(qpos, dtype=torch.int32, device=DEV)
    base = torch.tensor(np.concatenate([[0], np.cumsum(ctx)[:-1]]), dtype=torch.int64, device=DEV)
    return dsa.Seqs(ctx_t, qs, qp, max_ctx=max(ctx), max_q_per_seq=qps, num_rows=sum(ctx), seq_base=base)


@pytest.mark.parametrize("world,rank,inter", [(3, 1, 7), (4, 0, 1), (1, 0, 1), (8, 7, 64)])
def test_topk_candidates(world, rank, inter):
    """The local top-k and its packed candidates, global ids by the ownership
    rule; contexts below, at and above k; two queries per sequence."""
    ctx = [700, 2048, 5000, 9]
    qps, k = 2, 2048
    qpos = [c - qps + i for c in ctx for i in range(qps)]
    qpos[-2] = 3  # a query far before the end of its sequence
    seqs = _contig_seqs(ctx, qpos, qps)
    Q = len(qpos)
    ld = (max(ctx) + 3) // 4 * 4
    scores = _tied_scores(11, 50, Q * ld).view(Q, ld).contiguous()
    idx = torch.empty(Q, k, dtype=torch.int32, device=DEV)
    tlen = torch.empty(Q, dtype=torch.int32, device=DEV)
    cand = torch.empty(Q, k, dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    shard = dsa.DcpShard(world, rank, inter)
    dsa.dsa_topk_candidates(scores, ld, seqs, Q, k, shard, idx, tlen, cand, None, 0, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    sc, ih, lh, ch = scores.cpu().numpy(), idx.cpu().numpy(), tlen.cpu().numpy(), _u64(cand)
    for t in range(Q):
        row = sc[t, :qpos[t] + 1].astype(np.float64)
        ri, m = oracle.topk(row, k)
        sel = np.sort(ri[:m])
        assert lh[t] == m and np.array_equal(ih[t, :m], sel) and np.all(ih[t, m:] == -1)
        glob = [oracle.dcp_global(int(l), rank, world, inter) for l in sel]
        want = oracle.dcp_pack(sc[t, sel], glob)
        assert np.array_equal(ch[t, :m], want), f"query {t}: packed candidates differ"
        assert np.all(ch[t, m:] == 0)


def _oracle_lists(seed, R, Q, n, k, fill=1.0):
    """R lists [Q, n] of packed candidates made by the oracle from seeded tied
    scores and distinct ids (ranks' disjoint shards); a fraction 1 - fill of
    the slots empty."""
    rng = np.random.default_rng(seed)
    lists = np.zeros((R, Q, n), np.uint64)
    for q in range(Q):
        ids = rng.permutation(10 ** 6)[:R * n]
        sc = (rng.integers(-12, 13, R * n) * 0.25).astype(np.float32)
        keep = rng.random(R * n) < fill
        packed = np.where(keep, oracle.dcp_pack(sc, ids), 0).astype(np.uint64)
        lists[:, q, :] = packed.reshape(R, n)
    return lists


@pytest.mark.parametrize("R,n,k,fill", [(4, 2048, 2048, 1.0), (8, 2048, 2048, 0.7), (16, 1024, 2048, 0.9),
                                        (3, 100, 64, 0.5), (2, 50, 2048, 0.8), (1, 2048, 2048, 1.0),
                                        (5, 7, 3, 1.0)])
def test_topk_merge(R, n, k, fill):
    """The selector against the oracle's, bit for bit: the k best by (score
    desc, id asc), ids ascending; fewer candidates than k; one list."""
    Q = 6
    lists = _oracle_lists(100 + R + n, R, Q, n, k, fill)
    dl = [torch.from_numpy(lists[r].view(np.int64)).to(DEV) for r in range(R)]
    idx = torch.empty(Q, k, dtype=torch.int32, device=DEV)
    tlen = torch.empty(Q, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.dsa_topk_merge(dl, n, Q, k, idx, tlen, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want, wlen = oracle.topk_merge(lists, k)
    assert np.array_equal(tlen.cpu().numpy(), wlen)
    assert np.array_equal(idx.cpu().numpy(), want)


def test_topk_merge_all_empty_and_all_tied():
    """No candidates: an empty row; every score equal: the k smallest ids."""
    R, Q, n, k = 4, 2, 512, 300
    lists = np.zeros((R, Q, n), np.uint64)
    ids = np.random.default_rng(5).permutation(50000)[:R * n]
    lists[:, 1, :] = oracle.dcp_pack(np.full(R * n, 1.5, np.float32), ids).reshape(R, n)
    dl = [torch.from_numpy(lists[r].view(np.int64)).to(DEV) for r in range(R)]
    idx = torch.empty(Q, k, dtype=torch.int32, device=DEV)
    tlen = torch.empty(Q, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.dsa_topk_merge(dl, n, Q, k, idx, tlen, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ih = idx.cpu().numpy()
    assert int(tlen[0]) == 0 and np.all(ih[0] == -1)
    assert int(tlen[1]) == k and np.array_equal(ih[1], np.sort(ids)[:k])


def test_topk_merge_reports_a_repeated_id():
    """The same id from two lists among the selected: the query's row empty and
    DSA_ERR_BAD_INPUT; the other query is merged."""
    R, Q, n, k = 2, 2, 64, 32
    lists = _oracle_lists(7, R, Q, n, k)
    lists[1, 0, 5] = oracle.dcp_pack(np.float32([1000.0]), [oracle.dcp_unpack(int(lists[0, 0, 3]))[1]])[0]
    lists[0, 0, 3] = oracle.dcp_pack(np.float32([999.0]), [oracle.dcp_unpack(int(lists[0, 0, 3]))[1]])[0]
    dl = [torch.from_numpy(lists[r].view(np.int64)).to(DEV) for r in range(R)]
    idx = torch.empty(Q, k, dtype=torch.int32, device=DEV)
    tlen = torch.empty(Q, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.dsa_topk_merge(dl, n, Q, k, idx, tlen, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 6
    assert int(tlen[0]) == 0 and torch.all(idx[0] == -1)
    want, wlen = oracle.topk_merge(lists[:, 1:2, :], k)
    assert int(tlen[1]) == wlen[0] and np.array_equal(idx[1].cpu().numpy(), want[0])


@pytest.mark.parametrize("world,inter", [(4, 1), (3, 64), (8, 16), (2, 100000)])
@pytest.mark.parametrize("in_place", [False, True])
def test_topk_compact(world, inter, in_place):
    """Each rank's compaction against the oracle's, bit for bit, with holes
    (-1 inside the selection), entries past topk_len and empty rows."""
    Q, k = 7, 2048
    rng = np.random.default_rng(world * 31 + inter)
    idx = np.full((Q, k), -1, np.int32)
    lens = np.array([2048, 1500, 0, 1, 37, 2048, 900], np.int32)
    for q in range(Q):
        idx[q, :lens[q]] = np.sort(rng.permutation(500000)[:lens[q]])
        if lens[q] > 10:
            idx[q, 5] = -1
        idx[q, lens[q]:lens[q] + 3] = 12345  # past topk_len: ignored
    idx[:, k - 3:] = np.where(lens[:, None] == k, idx[:, k - 3:], 7)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for r in range(world):
        di = torch.from_numpy(idx).to(DEV)
        dl = torch.from_numpy(lens).to(DEV)
        li, ll = (di, dl) if in_place else (torch.empty_like(di), torch.empty_like(dl))
        dsa.dsa_topk_compact(di, dl, Q, k, dsa.DcpShard(world, r, inter), li, ll, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        want, wlen = oracle.topk_compact(idx, lens, r, world, inter)
        assert np.array_equal(ll.cpu().numpy(), wlen)
        assert np.array_equal(li.cpu().numpy(), want)


def test_lse_combine():
    """Against the oracle on the bf16 parts: parts at -inf, a row with every
    part at -inf, lse far apart; lse within fp32 noise; out within one bf16
    rounding plus fp32 noise on the weighted terms (the weights exp(lse_r -
    lse) carry about one fp32 ulp of lse, 8e-6 at lse ~ 75)."""
    R, Q = 5, 9
    o = [I.to_bf16(I.normal(I.stream_key(9, 60 + r), I._counters(0, Q * 64 * 512, DEV))).view(Q, 64, 512)
         for r in range(R)]
    lse = [(I.normal(I.stream_key(9, 80 + r), I._counters(0, Q * 64, DEV)) * 4).to(torch.float32).view(Q, 64)
           for r in range(R)]
    lse[1][:, :7] = float("-inf")
    o[1][:, :7] = 0
    for r in range(R):
        lse[r][3] = float("-inf")
        o[r][3] = 0
    lse[2][5] += 60.0  # one part dominates
    out = torch.empty(Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    lo = torch.empty(Q, 64, dtype=torch.float32, device=DEV)
    dsa.dsa_lse_combine(o, lse, Q, out, lo)
    torch.cuda.synchronize()
    ro, rl = oracle.lse_combine(np.stack([x.float().cpu().numpy() for x in o]),
                                np.stack([x.cpu().numpy() for x in lse]))
    got = out.float().cpu().numpy()
    assert np.all(got[3] == 0) and np.all(np.isneginf(lo[3].cpu().numpy()))
    fin = np.isfinite(rl)
    gl = lo.cpu().numpy()
    assert np.array_equal(np.isfinite(gl), fin)
    assert np.max(np.abs(gl[fin] - rl[fin]) / np.maximum(1.0, np.abs(rl[fin]))) <= 2e-6
    quantum = np.exp2(np.floor(np.log2(np.maximum(np.abs(ro), 2.0 ** -126))) - 7)
    mag, _ = oracle.lse_combine(np.stack([np.abs(x.float().cpu().numpy()) for x in o]),
                                np.stack([x.cpu().numpy() for x in lse]))  # sum_r w_r |o_r|
    bound = 0.5 * quantum * (1 + 1e-9) + 3e-5 * mag
    assert np.all(np.abs(got - ro) <= bound), f"worst excess {np.max(np.abs(got - ro) - bound):.3e}"


DCP_CASES = {
    "paged_small": (I.scaled(W["paged"], num_seqs=3, ctx=None, ctx_list=(1500, 4163, 700)), 4, 64),
    "paged_tokens": (I.scaled(W["paged"], num_seqs=2, ctx=None, ctx_list=(3000, 2222)), 3, 1),
    "fp8_small": (I.scaled(W["long_fp8"], num_seqs=2, ctx=None, ctx_list=(9000, 5000)), 4, 16),
    "specv_small": (I.scaled(W["specv"], num_seqs=2, ctx_range=(3000, 5000)), 2, 128),
}


@pytest.mark.parametrize("name", list(DCP_CASES))
def test_sharded_layer_matches_unsharded_oracle(name):
    """A layer sharded over `world` ranks on one GPU: the merged selection is
    the oracle's global top-k (boundary ties within the tolerance) and equals
    the unsharded library's bit for bit; the combined output and lse match the
    oracle's attention over that selection (and the shared-indexer layer's)."""
    wl, world, inter = DCP_CASES[name]
    d = P.to_device(I.make_inputs(wl, "cpu"), DEV)
    sh = ShardedLayer(d, wl.queries_per_seq, wl.topk, world, inter)
    sh.run()
    step = DecodeStep(d, wl.queries_per_seq, wl.topk)
    step.run()
    torch.cuda.synchronize()
    assert sh.device_status() == 0 and step.device_status() == 0
    idx, tlen = sh.idx.cpu().numpy(), sh.topk_len.cpu().numpy()
    assert np.array_equal(idx, step.idx.cpu().numpy()) and np.array_equal(tlen, step.topk_len.cpu().numpy())
    lay = d["layout"]
    out, lse = sh.out.float().cpu().numpy(), sh.lse.cpu().numpy()
    for t in range(sh.num_q):
        pos = lay.q_pos[t]
        ref = P.oracle_scores_for_query(d, t)
        P.check_topk(idx[t], int(tlen[t]), ref[:pos + 1], wl.topk)
        sel = idx[t][:tlen[t]]
        ro, rl = P.oracle_mla_for_query(d, t, sel)
        P.check_mla(out[t], lse[t], ro, rl)
        if sh.shared:
            ro2, rl2 = P.oracle_mla_for_query(d, t, sel, shared=True)
            P.check_mla(sh.out2[t].float().cpu().numpy(), sh.lse2[t].cpu().numpy(), ro2, rl2)


def test_sharded_layer_at_benchmark_size_sampled():
    """The sharded benchmark configuration (64 sequences x 32768 keys in
    64-token pages, four ranks in turns of one page), checked on sampled
    queries."""
    wl = W["paged"]
    d = I.make_inputs(wl, DEV)
    sh = ShardedLayer(d, wl.queries_per_seq, wl.topk, 4, 64)
    sh.run()
    torch.cuda.synchronize()
    assert sh.device_status() == 0
    idx, tlen = sh.idx.cpu().numpy(), sh.topk_len.cpu().numpy()
    out, lse = sh.out.float().cpu().numpy(), sh.lse.cpu().numpy()
    lay = d["layout"]
    for t in P.sample_queries(sh.num_q, 4):
        ref = P.oracle_scores_for_query(d, t)
        P.check_topk(idx[t], int(tlen[t]), ref[:lay.q_pos[t] + 1], wl.topk)
        ro, rl = P.oracle_mla_for_query(d, t, idx[t][:tlen[t]])
        P.check_mla(out[t], lse[t], ro, rl)
