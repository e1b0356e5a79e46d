"""Parity of the CUDA path (through the C ABI) with the CPU oracle on a GB300.

Small workloads span several key tiles, ragged tails, pages, several queries
per sequence, NoPE + a shared-indexer layer, fp8 and NVFP4 caches and a prefill chunk;
every query is checked.  The full-size workloads run in the launch
configuration the benchmark times and are checked on sampled queries.
Tolerances are in tests/parity.py.
"""

from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import dsa_sparse_mla_query_gb300 as dsa
from dsa_sparse_mla_query_gb300 import inputs as I
from dsa_sparse_mla_query_gb300.runner import DecodeStep
import parity as P

pytestmark = pytest.mark.gpu

DEV = "cuda"
W = I.WORKLOADS
SMALL = {
    "tiny": W["tiny"],
    "paged_small": I.scaled(W["paged"], num_seqs=3, ctx=None, ctx_list=(1500, 4163, 130)),
    "specv_small": I.scaled(W["specv"], num_seqs=4, ctx_range=(2100, 6000)),
    "fp8_small": I.scaled(W["long_fp8"], num_seqs=3, ctx=None, ctx_list=(2000, 9000, 2049)),
    "nvfp4_small": I.scaled(W["long_nvfp4"], num_seqs=3, ctx=None, ctx_list=(2000, 9000, 2049)),
    "prefill_small": I.scaled(W["prefill"], ctx=3000, queries_per_seq=40),
}


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    dsa.load()
    yield
    torch.cuda.synchronize()


def _inputs_cpu_then_gpu(wl):
    d = I.make_inputs(wl, "cpu")
    return P.to_device(d, DEV), d


def _separate_scores(d, wl, step):
    """dsa_index_scores into a [Q, ld] buffer (NaN-poisoned, so unwritten
    entries inside the context would show)."""
    ld = P.ld_of(step.seqs.max_ctx)
    scores = torch.full((step.num_q, ld), float("nan"), dtype=torch.float32, device=DEV)
    if "k_bscale" in d:  # NVFP4 keys
        dsa.dsa_index_scores_nvfp4(d["q_idx"], d["w"], d["ssmax_s"], d["ssmax_b"], d["inv_freq"], d["k_idx"],
                                   d["k_bscale"], d["k_global"], step.seqs, step.num_q, scores, ld, step.ws,
                                   step.ws_bytes, step.status)
    else:
        dsa.dsa_index_scores(d["q_idx"], d["w"], d["ssmax_s"], d["ssmax_b"], d["inv_freq"], d["k_idx"],
                             d.get("k_scale"), dsa.DSA_FP8_E4M3_ROWSCALE if step.k_fp8 else dsa.DSA_BF16, step.seqs,
                             step.num_q, scores, ld, step.ws, step.ws_bytes, step.status)
    return scores, ld


def _check_workload(d, wl, queries, threads=8):
    """Runs the separate calls and the fused layer; checks queries against the
    oracle.  Returns a small report."""
    step = DecodeStep(d, wl.queries_per_seq, wl.topk)
    k = wl.topk
    scores, ld = _separate_scores(d, wl, step)
    idx = torch.empty(step.num_q, k, dtype=torch.int32, device=DEV)
    tlen = torch.empty(step.num_q, dtype=torch.int32, device=DEV)
    dsa.dsa_topk(scores, ld, step.seqs, step.num_q, k, idx, tlen, step.ws, step.ws_bytes, step.status)
    step.run()  # fused layer(s), the launch configuration the benchmark times
    torch.cuda.synchronize()
    assert step.device_status() == 0, f"device status {step.device_status()}"
    lay = d["layout"]
    sc_h, idx_h, len_h = scores.cpu().numpy(), idx.cpu().numpy(), tlen.cpu().numpy()
    fidx_h, flen_h = step.idx.cpu().numpy(), step.topk_len.cpu().numpy()
    assert np.array_equal(fidx_h, idx_h) and np.array_equal(flen_h, len_h), "fused and separate selections differ"

    def one(t):
        b = lay.q_seq[t]
        pos, ctx = lay.q_pos[t], lay.ctx_len[b]
        ref = P.oracle_scores_for_query(d, t)
        rep = {"t": t}
        rep["score_rel_err"] = P.check_scores(sc_h[t], ref, pos, ctx)
        rep["boundary_diff"] = P.check_topk(idx_h[t], int(len_h[t]), ref[:pos + 1], k)
        ref_idx, m = __import__("oracle").topk(ref[:pos + 1], k)
        rep["oracle_sel"] = np.sort(ref_idx[:m])
        return rep

    with ThreadPoolExecutor(max_workers=threads) as ex:
        reps = list(ex.map(one, queries))

    # attention on the oracle's own selection through sparse_mla_decode
    oidx = torch.full((step.num_q, k), -1, dtype=torch.int32)
    olen = torch.zeros(step.num_q, dtype=torch.int32)
    for r in reps:
        oidx[r["t"], :len(r["oracle_sel"])] = torch.from_numpy(r["oracle_sel"].astype(np.int32))
        olen[r["t"]] = len(r["oracle_sel"])
    oidx_d, olen_d = oidx.to(DEV), olen.to(DEV)
    layers = [("latent", "q_mla", False)] + ([("latent2", "q_mla2", True)] if step.shared else [])
    for lat_key, q_key, shared in layers:
        out = torch.empty(step.num_q, 64, 512, dtype=torch.bfloat16, device=DEV)
        lse = torch.empty(step.num_q, 64, dtype=torch.float32, device=DEV)
        if "lat_bscale" in d and not shared:  # NVFP4 latent rows
            dsa.sparse_mla_decode_nvfp4(d[q_key], d[lat_key], d["lat_bscale"], d["lat_global"], step.seqs,
                                        step.num_q, oidx_d, olen_d, k, d["sm_scale"], out, lse, step.ws,
                                        step.ws_bytes, step.status)
        else:
            dsa.sparse_mla_decode(d[q_key], d[lat_key], dsa.DSA_FP8_DS_MLA if step.lat_fp8 else dsa.DSA_BF16,
                                  step.seqs, step.num_q, oidx_d, olen_d, k, d["sm_scale"], out, lse, step.ws,
                                  step.ws_bytes, step.status)
        torch.cuda.synchronize()
        assert step.device_status() == 0
        out_h, lse_h = out.float().cpu().numpy(), lse.cpu().numpy()
        fout = (step.out2 if shared else step.out).float().cpu().numpy()
        flse = (step.lse2 if shared else step.lse).cpu().numpy()

        def att(r):
            t = r["t"]
            ro, rl = P.oracle_mla_for_query(d, t, r["oracle_sel"], shared)
            e = P.check_mla(out_h[t], lse_h[t], ro, rl)
            # fused layer: its own selection; where it equals the oracle's the
            # output must match; where boundary ties were resolved the other
            # way the output must be attention over the selection it made
            fsel = fidx_h[t][:flen_h[t]]
            if np.array_equal(np.sort(fsel), r["oracle_sel"]):
                P.check_mla(fout[t], flse[t], ro, rl)
            else:
                vo, vl = P.oracle_mla_for_query(d, t, fsel, shared)
                P.check_mla(fout[t], flse[t], vo, vl)
            return e

        with ThreadPoolExecutor(max_workers=threads) as ex:
            errs = list(ex.map(att, reps))
        for r, e in zip(reps, errs):
            r["out_rel_err_" + lat_key] = e
    return reps


@pytest.mark.parametrize("name", list(SMALL))
def test_small_workload_all_queries(name):
    wl = SMALL[name]
    d, _ = _inputs_cpu_then_gpu(wl)
    reps = _check_workload(d, wl, list(range(wl.num_queries)))
    worst = max(r["score_rel_err"] for r in reps)
    assert worst < 1e-4, f"scores should be near fp32 accuracy, got {worst:.2e}"


@pytest.mark.parametrize("ctx_list", [(1,), (2047,), (2048,), (2049,), (4096 + 37,)])
def test_context_around_k(ctx_list):
    """Context shorter than, equal to and just above k; one key; a ragged tail."""
    wl = I.scaled(W["tiny"], num_seqs=len(ctx_list), ctx=None, ctx_list=ctx_list, queries_per_seq=1)
    d, _ = _inputs_cpu_then_gpu(wl)
    _check_workload(d, wl, list(range(wl.num_queries)))


@pytest.mark.parametrize("k", [1, 7, 100, 2047])
def test_small_k(k):
    wl = I.scaled(W["paged"], num_seqs=2, ctx=None, ctx_list=(3000, 777), topk=k)
    d, _ = _inputs_cpu_then_gpu(wl)
    _check_workload(d, wl, list(range(wl.num_queries)))


def test_two_splits_combine_in_cluster():
    """70 queries give two splits per query, whose pair combines in-kernel
    (thread-block cluster); contexts leave the second split empty (1, 500,
    1000 keys), split at the boundary (1024, 1025) or fill both (2048, 2049,
    3000, 6000)."""
    ctx_cycle = (1, 500, 1000, 1024, 1025, 2048, 2049, 3000, 6000, 4163)
    ctx_list = tuple(ctx_cycle[i % len(ctx_cycle)] for i in range(70))
    wl = I.scaled(W["tiny"], num_seqs=70, ctx=None, ctx_list=ctx_list, queries_per_seq=1)
    d, _ = _inputs_cpu_then_gpu(wl)
    step = DecodeStep(d, wl.queries_per_seq, wl.topk)
    assert step.launches_per_step() == 4, "bf16 with two splits runs without a combine launch"
    _check_workload(d, wl, list(range(wl.num_queries)))


def test_long_rows_streamed_topk():
    """Rows longer than 32,768 keys take the streamed top-k: ragged last
    blocks (32769, 40001), a longer row (70000) and, in the same launch, a row
    of at most k keys (1000)."""
    wl = I.scaled(W["tiny"], num_seqs=4, ctx=None, ctx_list=(40001, 1000, 70000, 32769), queries_per_seq=1)
    d, _ = _inputs_cpu_then_gpu(wl)
    step = DecodeStep(d, wl.queries_per_seq, wl.topk)
    # query prep, scores, top-k, attention in 16 splits + their combine
    assert step.launches_per_step() == 2 + 1 + 2
    _check_workload(d, wl, list(range(wl.num_queries)), threads=4)


def test_long_rows_all_equal_scores():
    """w = 0 makes every score 0: every key of a long row falls into one
    first digit, more than the list of that digit's keys holds, so the finer
    digits are found by passes over the row; the selection is positions
    0..k-1."""
    wl = I.scaled(W["tiny"], num_seqs=2, ctx=None, ctx_list=(40000, 50000), queries_per_seq=1)
    d, _ = _inputs_cpu_then_gpu(wl)
    d["w"].zero_()
    step = DecodeStep(d, wl.queries_per_seq, wl.topk)
    step.run()
    torch.cuda.synchronize()
    assert step.device_status() == 0
    idx, tlen = step.idx.cpu().numpy(), step.topk_len.cpu().numpy()
    for t in range(2):
        assert tlen[t] == 2048
        assert np.array_equal(idx[t], np.arange(2048))


def test_long_rows_sampled_threshold():
    """Rows of 4 blocks (65,536 keys) or more per CTA of their cluster: each
    CTA samples 1024 evenly spaced keys, lists the keys at or above the
    sample's threshold digit in one pass and selects from the lists; the
    selection falls back to two passes over the row when a list overflows or
    the lists hold fewer than k keys.  Three rows of one launch (clusters of 8
    CTAs): normal scores with a ragged last block (1,100,000 keys); equal
    scores (every key listed: overflow); and 300 scores near 8 planted at
    multiples of 128, where the evenly spaced sample of a 1,048,576-key row
    lands, above normal scores (the sample's threshold passes 300 keys, fewer
    than k).  Each row's selection is the oracle's."""
    ctx = [1100000, 1048576, 1048576]
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device=DEV)
    qs = torch.arange(len(ctx) + 1, dtype=torch.int32, device=DEV)
    qp = torch.tensor([c - 1 for c in ctx], dtype=torch.int32, device=DEV)
    base = torch.tensor(np.concatenate([[0], np.cumsum(ctx)[:-1]]), dtype=torch.int64, device=DEV)
    seqs = dsa.Seqs(ctx_t, qs, qp, max_ctx=max(ctx), max_q_per_seq=1, num_rows=sum(ctx), seq_base=base)
    k, Q, ld = 2048, len(ctx), P.ld_of(max(ctx))
    g = torch.Generator().manual_seed(17)
    sc = torch.full((Q, ld), float("nan"), dtype=torch.float32)
    sc[0, : ctx[0]] = torch.randn(ctx[0], generator=g)
    sc[1, : ctx[1]] = 0.25
    v = torch.randn(ctx[2], generator=g)
    planted = 128 * torch.randperm(ctx[2] // 128, generator=g)[:300]
    v[planted] = 8.0 + torch.rand(300, generator=g)
    sc[2, : ctx[2]] = v
    idx = torch.empty(Q, k, dtype=torch.int32, device=DEV)
    tlen = torch.empty(Q, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.dsa_topk(sc.to(DEV), ld, seqs, Q, k, idx, tlen, None, 0, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    idx, tlen = idx.cpu().numpy(), tlen.cpu().numpy()
    oracle = __import__("oracle")
    for t, n in enumerate(ctx):
        ref, m = oracle.topk(sc[t, :n].double().numpy(), k)
        assert tlen[t] == m == k
        assert np.array_equal(idx[t], np.sort(ref[:m])), f"row {t}"


@pytest.mark.parametrize("seed", [0, 1])
def test_topk_rows_in_shared_memory(seed):
    """Rows of 16,385 to 32,768 keys (one CTA per row, the row in shared
    memory) on crafted scores against the oracle's exact top-k: ties at the
    boundary (8 distinct values), one first digit holding more keys than the
    candidate buffer (values within 2^-10 of 1), signed values with -0.0 and
    +0.0 mixed, and all scores equal (positions 0..k-1)."""
    ctx_list = (16385, 32768, 25000, 20001)
    wl = I.scaled(W["tiny"], num_seqs=4, ctx=None, ctx_list=ctx_list, queries_per_seq=1)
    d, _ = _inputs_cpu_then_gpu(wl)
    step = DecodeStep(d, wl.queries_per_seq, wl.topk)
    ld = P.ld_of(step.seqs.max_ctx)
    g = torch.Generator().manual_seed(100 + seed)
    sc = torch.full((4, ld), float("nan"), dtype=torch.float32)
    n0, n1, n2, n3 = ctx_list
    sc[0, :n0] = torch.randint(0, 8, (n0,), generator=g).float() * 0.5
    sc[1, :n1] = 1.0 + torch.rand(n1, generator=g) * 2.0 ** -10
    v = torch.randn(n2, generator=g)
    v[torch.randint(0, n2, (3000,), generator=g)] = 0.0
    v[torch.randint(0, n2, (3000,), generator=g)] = -0.0
    sc[2, :n2] = v
    sc[3, :n3] = 0.25
    dsa.dsa_topk(sc.to(DEV), ld, step.seqs, 4, wl.topk, step.idx, step.topk_len, step.ws, step.ws_bytes, step.status)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    idx, tlen = step.idx.cpu().numpy(), step.topk_len.cpu().numpy()
    oracle = __import__("oracle")
    for t, n in enumerate(ctx_list):
        ref, m = oracle.topk(sc[t, :n].double().numpy(), wl.topk)
        assert tlen[t] == m == wl.topk
        assert np.array_equal(idx[t], np.sort(ref[:m])), f"row {t}"


def test_topk_rows_narrow_key_range():
    """Rows whose scores span a few ulps (the digits of the selection then
    have 1 to 3 significant bits): two adjacent floats, five adjacent floats
    with ties across the boundary, and one key above a row of equal keys."""
    ctx_list = (20000, 30000, 17000)
    wl = I.scaled(W["tiny"], num_seqs=3, ctx=None, ctx_list=ctx_list, queries_per_seq=1)
    d, _ = _inputs_cpu_then_gpu(wl)
    step = DecodeStep(d, wl.queries_per_seq, wl.topk)
    ld = P.ld_of(step.seqs.max_ctx)
    g = torch.Generator().manual_seed(5)
    sc = torch.full((3, ld), float("nan"), dtype=torch.float32)
    ulp = np.nextafter(np.float32(1.0), np.float32(2.0)) - np.float32(1.0)
    n0, n1, n2 = ctx_list
    sc[0, :n0] = 1.0 + float(ulp) * torch.randint(0, 2, (n0,), generator=g).float()
    sc[1, :n1] = -3.0 + 2 * float(ulp) * torch.randint(0, 5, (n1,), generator=g).float()
    sc[2, :n2] = 0.5
    sc[2, 12345] = float(np.nextafter(np.float32(0.5), np.float32(1.0)))
    dsa.dsa_topk(sc.to(DEV), ld, step.seqs, 3, wl.topk, step.idx, step.topk_len, step.ws, step.ws_bytes, step.status)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    idx, tlen = step.idx.cpu().numpy(), step.topk_len.cpu().numpy()
    oracle = __import__("oracle")
    for t, n in enumerate(ctx_list):
        ref, m = oracle.topk(sc[t, :n].double().numpy(), wl.topk)
        assert tlen[t] == m == wl.topk
        assert np.array_equal(idx[t], np.sort(ref[:m])), f"row {t}"


def test_topk_rows_top_keys_on_a_sparse_lattice():
    """Rows of 16,385 to 32,768 keys whose largest scores sit on a sparse,
    irregular lattice of positions (one key in 32: 1024 w + 4 l + 128 (l mod
    8), w and l < 32), fewer than k of them, with a quarter of the row tied
    just below: the oracle's exact top-k, ties to the smaller position."""
    ctx_list = (32768, 20001)
    wl = I.scaled(W["tiny"], num_seqs=2, ctx=None, ctx_list=ctx_list, queries_per_seq=1)
    d, _ = _inputs_cpu_then_gpu(wl)
    step = DecodeStep(d, wl.queries_per_seq, wl.topk)
    ld = P.ld_of(step.seqs.max_ctx)
    g = torch.Generator().manual_seed(11)
    sc = torch.full((2, ld), float("nan"), dtype=torch.float32)
    for r, n in enumerate(ctx_list):
        v = torch.randn(n, generator=g)
        v[torch.randint(0, n, (n // 4,), generator=g)] = 1.5  # ties below the sampled keys
        sp = [1024 * w + 4 * l + 128 * (l % 8) for w in range(32) for l in range(32)]
        sp = torch.tensor([q for q in sp if q < n])
        v[sp] = 8.0 + torch.rand(len(sp), generator=g)
        sc[r, :n] = v
    dsa.dsa_topk(sc.to(DEV), ld, step.seqs, 2, wl.topk, step.idx, step.topk_len, step.ws, step.ws_bytes, step.status)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    idx, tlen = step.idx.cpu().numpy(), step.topk_len.cpu().numpy()
    oracle = __import__("oracle")
    for t, n in enumerate(ctx_list):
        ref, m = oracle.topk(sc[t, :n].double().numpy(), wl.topk)
        assert tlen[t] == m == wl.topk
        assert np.array_equal(idx[t], np.sort(ref[:m])), f"row {t}"


def test_fp8_index_keys_every_code_class():
    """e4m3 index keys of one sequence drawn from the subnormal codes (and
    zero) alone, of the other from every finite code: scores, selection and
    attention match the oracle for each, so a decode that flushed subnormals
    or misplaced a sign, exponent or mantissa bit fails."""
    wl = I.scaled(W["long_fp8"], num_seqs=2, ctx=None, ctx_list=(3000, 2100))
    d, _ = _inputs_cpu_then_gpu(wl)
    g = torch.Generator().manual_seed(7)
    sub = torch.tensor(list(range(8)) + [0x80 + c for c in range(8)], dtype=torch.uint8)
    fin = torch.tensor([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=torch.uint8)
    codes = d["k_idx"].cpu()
    for b, pool in enumerate((sub, fin)):
        rows = P.seq_rows_host(d, b)
        codes[rows] = pool[torch.randint(0, len(pool), (len(rows), 128), generator=g)]
    d["k_idx"].copy_(codes.to(DEV))
    reps = _check_workload(d, wl, list(range(wl.num_queries)))
    worst = max(r["score_rel_err"] for r in reps)
    assert worst < 1e-4, f"scores should be near fp32 accuracy, got {worst:.2e}"


def test_fp8_rows_at_odd_bases():
    """e4m3 keys of sequences whose first rows are not multiples of four
    (contexts 2001, 4163, 130): their row scales cannot be copied in 16-byte
    blocks and take the per-row path; the last tile runs past the cache."""
    wl = I.scaled(W["long_fp8"], num_seqs=3, ctx=None, ctx_list=(2001, 4163, 130))
    d, _ = _inputs_cpu_then_gpu(wl)
    assert int(P.seq_rows_host(d, 1)[0]) % 4 != 0
    reps = _check_workload(d, wl, list(range(wl.num_queries)))
    worst = max(r["score_rel_err"] for r in reps)
    assert worst < 1e-4, f"scores should be near fp32 accuracy, got {worst:.2e}"


def test_all_equal_scores_take_smallest_indices():
    """w = 0 makes every score 0: the selection is positions 0..k-1."""
    wl = I.scaled(W["tiny"], num_seqs=1, ctx=5000, queries_per_seq=2)
    d, _ = _inputs_cpu_then_gpu(wl)
    d["w"].zero_()
    step = DecodeStep(d, wl.queries_per_seq, wl.topk)
    step.run()
    torch.cuda.synchronize()
    idx = step.idx.cpu().numpy()
    for t in range(2):
        assert np.array_equal(idx[t], np.arange(2048))
    _check_workload(d, wl, [0, 1])


def test_empty_selection_and_holes():
    """topk_len = 0 gives zeros and -inf; -1 slots inside the selection are skipped."""
    wl = I.scaled(W["tiny"], num_seqs=1, ctx=3000, queries_per_seq=3)
    d, _ = _inputs_cpu_then_gpu(wl)
    step = DecodeStep(d, wl.queries_per_seq, wl.topk)
    k = wl.topk
    idx = torch.full((3, k), -1, dtype=torch.int32)
    sel = np.array([5, 17, 2999, 0, 1024, 1500], np.int32)
    idx[1, :6] = torch.from_numpy(sel)
    idx[1, 2] = -1                     # a hole
    idx[2, :6] = torch.from_numpy(sel)
    tlen = torch.tensor([0, 6, 6], dtype=torch.int32)
    out = torch.empty(3, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(3, 64, dtype=torch.float32, device=DEV)
    dsa.sparse_mla_decode(d["q_mla"], d["latent"], dsa.DSA_BF16, step.seqs, 3, idx.to(DEV), tlen.to(DEV), k,
                          d["sm_scale"], out, lse, step.ws, step.ws_bytes, step.status)
    torch.cuda.synchronize()
    assert step.device_status() == 0
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    assert np.all(o[0] == 0) and np.all(np.isneginf(l[0]))
    r1 = P.oracle_mla_for_query(d, 1, np.delete(sel, 2))
    P.check_mla(o[1], l[1], *r1)
    r2 = P.oracle_mla_for_query(d, 2, sel)
    P.check_mla(o[2], l[2], *r2)


def test_bad_position_sets_device_status():
    """A query position outside its context is reported in d_status and its
    row is skipped; the other queries are unaffected; nothing traps."""
    wl = I.scaled(W["tiny"], num_seqs=2, ctx=None, ctx_list=(3000, 2500), queries_per_seq=1)
    d, _ = _inputs_cpu_then_gpu(wl)
    d["q_pos"][1] = 2500  # == ctx_len[1]
    step = DecodeStep(d, 1, wl.topk)
    step.run()
    torch.cuda.synchronize()
    assert step.device_status() == 6  # DSA_ERR_BAD_INPUT
    assert int(step.topk_len[1].item()) == 0
    assert int(step.topk_len[0].item()) == 2048
    torch.cuda.synchronize()


FULL = ["paged", "specv", "long_fp8", "prefill", "long_nvfp4"]
SAMPLES = {"paged": 6, "specv": 6, "long_fp8": 3, "prefill": 4, "long_nvfp4": 3}


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    """Full-size workload in the benchmark's launch configuration; sampled
    queries against the oracle."""
    wl = W[name]
    d = I.make_inputs(wl, DEV)
    try:
        qs = P.sample_queries(wl.num_queries, SAMPLES[name])
        reps = _check_workload(d, wl, qs, threads=8)
        print(name, [(r["t"], round(r["score_rel_err"], 9), r["boundary_diff"]) for r in reps])
    finally:
        del d
        torch.cuda.empty_cache()
