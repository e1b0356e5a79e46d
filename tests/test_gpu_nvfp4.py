"""NVFP4 latent caches on a GB300 ("vLLM adds NVFP4 serving for MiniMax M3.1
Flash": NVFP4 attention caches, 4.5 bits per value with their block scales,
converted inside the decode kernel).

The seeded bf16 latent rows are quantised by the oracle's NVFP4 encoder
(E2M1 codes, one E4M3 scale per 16 values, one fp32 tensor scale); the CUDA
path and the oracle both read those bytes.  sparse_mla_decode_nvfp4 and the
fused layer with an NVFP4 latent are compared with the oracle's attention
over the decoded values, at the tolerances of tests/parity.py.
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
