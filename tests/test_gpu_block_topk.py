"""Block-sparse selection on a GB300 through the C ABI ("vLLM adds NVFP4 serving
for MiniMax M3.1 Flash", MiniMax Sparse Attention: 128-token blocks, 16
selected with the most recent kept, exact attention over their keys).

dsa_block_topk is compared bit for bit with the oracle's block selection on
the same seeded scores (many equal scores, so block maxima tie); the fused
layer in block mode (indexer -> block selection -> attention) is compared with
the separate calls, with the oracle's selection on the oracle's scores (block
ties allowed within the tolerance of tests/parity.py) and with the oracle's
attention over the selection it made.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import dsa_sparse_mla_query_gb300 as dsa
import oracle
from dsa_sparse_mla_query_gb300 import inputs as I
from dsa_sparse_mla_query_gb300.runner import DecodeStep
import parity as P

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    dsa.load()
    yield
    torch.cuda.synchronize()


def _seqs(ctx, qpos, qps):
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device=DEV)
    qs = torch.tensor([i * qps for i in range(len(ctx) + 1)], dtype=torch.int32, device=DEV)
    qp = torch.tensor(qpos, dtype=torch.int32, device=DEV)
    base = torch.tensor(np.concatenate([[0], np.cumsum(ctx)[:-1]]), dtype=torch.int64, device=DEV)
    return dsa.Seqs(ctx_t, qs, qp, max_ctx=max(ctx), max_q_per_seq=qps, num_rows=sum(ctx), seq_base=base)


def _scores(Q, ld, key, nan_row=None):
    """Seeded scores rounded to quarter steps, so block maxima tie often."""
    x = I.normal(I.stream_key(21, key), I._counters(0, Q * ld, DEV)).to(torch.float32)
    sc = (torch.round(x * 4) / 4).view(Q, ld).contiguous()
    if nan_row is not None:  # NaN scores in the early blocks of one row
        sc[nan_row, : ld // 3 : 3] = float("nan")
    return sc


# contexts: several full blocks with a ragged own block, a context of exactly
# 2048, one where the blocks are fewer than nsel, a five-key context, and a
# long row
CTX = [9000, 2048, 130, 40000, 5]


@pytest.mark.parametrize("block,nsel", [(128, 16), (64, 32), (32, 1), (100, 20), (1, 64), (1, 1), (2048, 1)])
def test_block_topk_matches_oracle(block, nsel):
    qps = 2
    qpos = [c - qps + i if c >= qps else c - 1 for c in CTX for i in range(qps)]
    qpos[0] = 4000  # a query well inside its context
    s = _seqs(CTX, qpos, qps)
    Q = len(qpos)
    ld = P.ld_of(max(CTX))
    scores = _scores(Q, ld, 3, nan_row=6)
    k = nsel * block
    idx = torch.full((Q, k), -7, dtype=torch.int32, device=DEV)
    tlen = torch.full((Q,), -7, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.dsa_block_topk(scores, ld, s, Q, block, nsel, idx, tlen, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    sc, idx_h, len_h = scores.cpu().numpy(), idx.cpu().numpy(), tlen.cpu().numpy()
    for t in range(Q):
        want, m = oracle.block_topk(sc[t, :qpos[t] + 1].astype(np.float64), block, nsel)
        assert int(len_h[t]) == m, (t, len_h[t], m)
        assert np.array_equal(idx_h[t], want[:k]), f"query {t}: selection differs"


def test_block_topk_one_key_blocks_reduce_to_topk_plus_own_key():
    """block = 1: the query's own key, then the nsel - 1 best other keys; where
    the own key is already among the top nsel this is the top-nsel itself."""
    ctx = [3000]
    s = _seqs(ctx, [2999], 1)
    ld = P.ld_of(3000)
    sc = _scores(1, ld, 5)
    sc[0, 2999] = 100.0  # the own key is the largest
    idx = torch.empty(1, 64, dtype=torch.int32, device=DEV)
    tlen = torch.empty(1, dtype=torch.int32, device=DEV)
    dsa.dsa_block_topk(sc, ld, s, 1, 1, 64, idx, tlen)
    torch.cuda.synchronize()
    ref, m = oracle.topk(sc[0, :3000].cpu().numpy().astype(np.float64), 64)
    assert int(tlen[0]) == m == 64
    assert np.array_equal(idx[0].cpu().numpy(), np.sort(ref[:m]))


# the fused layer in block mode: e4m3 index keys and fp8_ds_mla latent rows as
# the long-context block workload, at sizes the oracle finishes in seconds
BLOCK_SMALL = I.scaled(I.WORKLOADS["block_fp8"], num_seqs=4, ctx=None, ctx_list=(9000, 20000, 2049, 130))
BLOCK_SMALL_BF16 = I.scaled(BLOCK_SMALL, index_fp8=False, latent_fp8=False, page_size=64,
                            ctx_list=(5000, 12345, 300, 64))


@pytest.mark.parametrize("wl", [BLOCK_SMALL, BLOCK_SMALL_BF16], ids=["fp8", "bf16_paged"])
def test_block_sparse_layer(wl):
    d = P.to_device(I.make_inputs(wl, "cpu"), DEV)
    blk, k = wl.select_block, wl.topk
    nsel = k // blk
    step = DecodeStep(d, wl.queries_per_seq, k, select_block=blk)
    step.run()
    torch.cuda.synchronize()
    assert step.device_status() == 0, step.device_status()
    # separate calls: the indexer's scores, then dsa_block_topk on them
    ld = P.ld_of(step.seqs.max_ctx)
    scores = torch.full((step.num_q, ld), float("nan"), dtype=torch.float32, device=DEV)
    dsa.dsa_index_scores(d["q_idx"], d["w"], d["ssmax_s"], d["ssmax_b"], d["inv_freq"], d["k_idx"], d.get("k_scale"),
                         dsa.DSA_FP8_E4M3_ROWSCALE if step.k_fp8 else dsa.DSA_BF16, step.seqs, step.num_q, scores,
                         ld, step.ws, step.ws_bytes, step.status)
    idx = torch.empty(step.num_q, k, dtype=torch.int32, device=DEV)
    tlen = torch.empty(step.num_q, dtype=torch.int32, device=DEV)
    dsa.dsa_block_topk(scores, ld, step.seqs, step.num_q, blk, nsel, idx, tlen, step.status)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    assert torch.equal(idx, step.idx) and torch.equal(tlen, step.topk_len), "fused and separate selections differ"
    lay = d["layout"]
    fidx, flen = step.idx.cpu().numpy(), step.topk_len.cpu().numpy()
    out, lse = step.out.float().cpu().numpy(), step.lse.cpu().numpy()
    for t in range(step.num_q):
        ref = P.oracle_scores_for_query(d, t)
        pos = lay.q_pos[t]
        P.check_block_select(fidx[t], int(flen[t]), ref[:pos + 1], blk, nsel)
        sel = fidx[t, :flen[t]]
        ro, rl = P.oracle_mla_for_query(d, t, sel)
        P.check_mla(out[t], lse[t], ro, rl)


def test_block_mode_launch_count_and_refusals():
    wl = BLOCK_SMALL
    d = P.to_device(I.make_inputs(wl, "cpu"), DEV)
    step = DecodeStep(d, wl.queries_per_seq, wl.topk, select_block=wl.select_block)
    a = step.layer_args()
    # query prep, scores, block selection, attention (+ combine)
    n = dsa.dsa_decode_layer_launches_for(a, step.seqs, step.num_q)
    assert n in (4, 5)
    bad = dict(a, select_block=3000)  # k = 2048 is not a multiple
    assert dsa.dsa_decode_layer_launches_for(bad, step.seqs, step.num_q) == 0
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_decode_layer(bad, step.seqs, step.num_q, step.ws, step.ws_bytes, step.status)
    assert "select_block" in str(e.value)
