"""NVFP4 caches on a GB300 ("vLLM adds NVFP4 serving for MiniMax M3.1 Flash":
NVFP4 attention and indexer caches, 4.5 bits per value with their block
scales, converted inside the decode kernels).

Latent rows: the seeded bf16 rows quantised by the oracle's NVFP4 encoder (E2M1
codes, one E4M3 scale per 16 values, one fp32 tensor scale).  Index keys: the
workloads' own NVFP4 keys (inputs.quantize_nvfp4, which a CPU test holds byte
for byte to the oracle's encoder).  Both sides read the same bytes.  Scores are
compared element by element with the oracle's scores over the decoded keys,
the selections with the oracle's exact top-k of those scores, and the
attention with the oracle's attention over the decoded rows, at the
tolerances of tests/parity.py.
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


def _nvfp4_latent(lat_bf16: torch.Tensor):
    """(codes uint8 [rows,288], scales uint8 [rows,36], g) from bf16 rows, by
    the oracle's encoder; g = max|v| / (6 x 448) so every block scale fits E4M3."""
    v = lat_bf16.float().cpu().numpy().astype(np.float64)
    g = float(np.max(np.abs(v))) / (6.0 * 448.0)
    codes, scales = oracle.nvfp4_quantize(v, g)
    return torch.from_numpy(codes).to(DEV), torch.from_numpy(scales).to(DEV), g


def _oracle_att(d, codes_h, scales_h, g, t, sel):
    """Oracle attention of query t over logical positions sel (NVFP4 rows)."""
    lay = d["layout"]
    rows = P.seq_rows_host(d, lay.q_seq[t])[torch.from_numpy(np.asarray(sel, np.int64))].numpy()
    n = len(sel)
    olay = oracle.Layout(np.array([max(n, 1)], np.int32), max(n, 1), seq_base=np.zeros(1, np.int64))
    return oracle.sparse_mla_nvfp4(d["q_mla"][t].cpu(), codes_h[rows], scales_h[rows], g, olay, 0,
                                   np.arange(n, dtype=np.int32), n, d["sm_scale"])


WLS = {
    "paged": I.scaled(I.WORKLOADS["paged"], num_seqs=3, ctx=None, ctx_list=(1500, 4163, 130)),
    "contig": I.scaled(I.WORKLOADS["tiny"], num_seqs=2, ctx=None, ctx_list=(3000, 2049), queries_per_seq=2),
}


@pytest.mark.parametrize("name", list(WLS))
def test_nvfp4_attention_matches_oracle(name):
    wl = WLS[name]
    d = P.to_device(I.make_inputs(wl, "cpu"), DEV)
    codes, scales, g = _nvfp4_latent(d["latent"])
    codes_h, scales_h = codes.cpu().numpy(), scales.cpu().numpy()
    step = DecodeStep(d, wl.queries_per_seq, wl.topk)
    lay = d["layout"]
    Q, k = step.num_q, wl.topk
    # selections: the oracle's own top-k of each query (some rows shorter)
    idx = torch.full((Q, k), -1, dtype=torch.int32)
    tlen = torch.zeros(Q, dtype=torch.int32)
    sels = []
    for t in range(Q):
        ref = P.oracle_scores_for_query(d, t)
        sel, m = oracle.topk(ref[:lay.q_pos[t] + 1], k)
        sel = np.sort(sel[:m])
        if t == 1:
            sel = sel[: m // 3]  # a compacted row
        sels.append(sel)
        idx[t, :len(sel)] = torch.from_numpy(sel.astype(np.int32))
        tlen[t] = len(sel)
    out = torch.empty(Q, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(Q, 64, dtype=torch.float32, device=DEV)
    dsa.sparse_mla_decode_nvfp4(d["q_mla"], codes, scales, g, step.seqs, Q, idx.to(DEV), tlen.to(DEV), k,
                                d["sm_scale"], out, lse, step.ws, step.ws_bytes, step.status)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    for t in range(Q):
        ro, rl = _oracle_att(d, codes_h, scales_h, g, t, sels[t])
        P.check_mla(o[t], l[t], ro, rl)


def test_nvfp4_latent_in_the_fused_layer():
    wl = WLS["paged"]
    d = P.to_device(I.make_inputs(wl, "cpu"), DEV)
    codes, scales, g = _nvfp4_latent(d["latent"])
    codes_h, scales_h = codes.cpu().numpy(), scales.cpu().numpy()
    step = DecodeStep(d, wl.queries_per_seq, wl.topk)
    a = step.layer_args()
    a.update(latent=codes, latent_dtype=dsa.DSA_NVFP4, latent_scales=scales, latent_global=g)
    dsa.dsa_decode_layer(a, step.seqs, step.num_q, step.ws, step.ws_bytes, step.status)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    lay = d["layout"]
    fidx, flen = step.idx.cpu().numpy(), step.topk_len.cpu().numpy()
    o, l = step.out.float().cpu().numpy(), step.lse.cpu().numpy()
    for t in range(step.num_q):
        ref = P.oracle_scores_for_query(d, t)
        P.check_topk(fidx[t], int(flen[t]), ref[:lay.q_pos[t] + 1], wl.topk)
        ro, rl = _oracle_att(d, codes_h, scales_h, g, t, fidx[t, :flen[t]])
        P.check_mla(o[t], l[t], ro, rl)


def test_nvfp4_refusals():
    wl = WLS["contig"]
    d = P.to_device(I.make_inputs(wl, "cpu"), DEV)
    step = DecodeStep(d, wl.queries_per_seq, wl.topk)
    out = torch.empty(step.num_q, 64, 512, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(dsa.DsaError, match="sparse_mla_decode_nvfp4"):
        dsa.sparse_mla_decode(d["q_mla"], d["latent"], dsa.DSA_NVFP4, step.seqs, step.num_q, step.idx,
                              step.topk_len, wl.topk, d["sm_scale"], out, None, step.ws, step.ws_bytes, step.status)
    with pytest.raises(dsa.DsaError, match="tensor scale"):
        dsa.sparse_mla_decode_nvfp4(d["q_mla"], d["latent"], d["latent"], 0.0, step.seqs, step.num_q, step.idx,
                                    step.topk_len, wl.topk, d["sm_scale"], out, None, step.ws, step.ws_bytes,
                                    step.status)


# NVFP4 index keys: one, two, four (+ a ragged second chunk) queries per
# sequence, paged and contiguous, RoPE and NoPE
IDX_WLS = {
    "paged_q1": I.scaled(I.WORKLOADS["paged"], num_seqs=3, ctx=None, ctx_list=(1500, 4163, 130), index_nvfp4=True),
    "contig_q2": I.scaled(I.WORKLOADS["tiny"], num_seqs=2, ctx=None, ctx_list=(3000, 2049), queries_per_seq=2,
                          index_nvfp4=True),
    "contig_q5": I.scaled(I.WORKLOADS["tiny"], num_seqs=2, ctx=None, ctx_list=(2500, 700), queries_per_seq=5,
                          index_nvfp4=True),
    "nope_q4": I.scaled(I.WORKLOADS["specv"], num_seqs=2, ctx=None, ctx_range=None, ctx_list=(2000, 1100),
                        shared_layer=False, index_nvfp4=True),
}


@pytest.mark.parametrize("name", list(IDX_WLS))
def test_nvfp4_index_scores_match_oracle(name):
    wl = IDX_WLS[name]
    d = P.to_device(I.make_inputs(wl, "cpu"), DEV)
    step = DecodeStep(d, wl.queries_per_seq, wl.topk)
    lay = d["layout"]
    Q = step.num_q
    ld = P.ld_of(max(lay.ctx_len))
    scores = torch.full((Q, ld), float("nan"), dtype=torch.float32, device=DEV)
    dsa.dsa_index_scores_nvfp4(d["q_idx"], d["w"], d["ssmax_s"], d["ssmax_b"], d["inv_freq"], d["k_idx"],
                               d["k_bscale"], d["k_global"], step.seqs, Q, scores, ld, step.ws, step.ws_bytes,
                               step.status)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    sc = scores.cpu().numpy()
    worst = 0.0
    for t in range(Q):
        b = lay.q_seq[t]
        ref = P.oracle_scores_for_query(d, t)
        worst = max(worst, P.check_scores(sc[t], ref, lay.q_pos[t], lay.ctx_len[b]))
        # exact selection from these scores (ties within the band are free)
        sel, m = oracle.topk(sc[t, :lay.q_pos[t] + 1].astype(np.float64), wl.topk)
        P.check_topk(np.sort(sel[:m]), m, ref[:lay.q_pos[t] + 1], wl.topk)
    # the keys are exact in f16 and q' keeps ~2^-22: far inside the tolerance
    assert worst < 1e-4, worst


def test_nvfp4_index_refusals():
    wl = IDX_WLS["contig_q2"]
    d = P.to_device(I.make_inputs(wl, "cpu"), DEV)
    step = DecodeStep(d, wl.queries_per_seq, wl.topk)
    ld = P.ld_of(max(d["layout"].ctx_len))
    scores = torch.empty(step.num_q, ld, dtype=torch.float32, device=DEV)
    with pytest.raises(dsa.DsaError, match="dsa_index_scores_nvfp4"):
        dsa.dsa_index_scores(d["q_idx"], d["w"], d["ssmax_s"], d["ssmax_b"], d["inv_freq"], d["k_idx"], None,
                             dsa.DSA_NVFP4, step.seqs, step.num_q, scores, ld, step.ws, step.ws_bytes, step.status)
    for g in (0.0, float("inf")):
        with pytest.raises(dsa.DsaError, match="tensor scale"):
            dsa.dsa_index_scores_nvfp4(d["q_idx"], d["w"], d["ssmax_s"], d["ssmax_b"], d["inv_freq"], d["k_idx"],
                                       d["k_bscale"], g, step.seqs, step.num_q, scores, ld, step.ws, step.ws_bytes,
                                       step.status)


# the whole layer over NVFP4 caches: keys and latent, top-k and block selection
LAYER_WLS = {
    "topk": I.scaled(I.WORKLOADS["long_nvfp4"], num_seqs=3, ctx=None, ctx_list=(5000, 2300, 700)),
    "paged_topk": I.scaled(I.WORKLOADS["long_nvfp4"], num_seqs=2, ctx=None, ctx_list=(4100, 3000), page_size=64),
    "blocks": I.scaled(I.WORKLOADS["long_nvfp4"], num_seqs=2, ctx=None, ctx_list=(9000, 2100), select_block=128),
}


@pytest.mark.parametrize("name", list(LAYER_WLS))
def test_nvfp4_caches_in_the_fused_layer(name):
    wl = LAYER_WLS[name]
    d = P.to_device(I.make_inputs(wl, "cpu"), DEV)
    step = DecodeStep(d, wl.queries_per_seq, wl.topk, select_block=wl.select_block)
    step.run()
    torch.cuda.synchronize()
    assert step.device_status() == 0
    lay = d["layout"]
    fidx, flen = step.idx.cpu().numpy(), step.topk_len.cpu().numpy()
    o, l = step.out.float().cpu().numpy(), step.lse.cpu().numpy()
    for t in range(step.num_q):
        ref = P.oracle_scores_for_query(d, t)
        causal = ref[:lay.q_pos[t] + 1]
        if wl.select_block:
            P.check_block_select(fidx[t], int(flen[t]), causal, wl.select_block, wl.topk // wl.select_block)
        else:
            P.check_topk(fidx[t], int(flen[t]), causal, wl.topk)
        ro, rl = P.oracle_mla_for_query(d, t, fidx[t, :flen[t]])
        P.check_mla(o[t], l[t], ro, rl)
