"""Parity of the cache-write side (through the C ABI) with the CPU oracle on a
GB300: new indexer keys and latent rows into their caches, and the attention
query's RoPE + SSMax.

A stored value must be a nearest bf16 / e4m3 rounding of the oracle's exact
value (the kernel rounds an fp32 result, so where the exact value sits within
fp32 noise of a midpoint either neighbour is accepted), every scale must match
the oracle's amax / 448, untouched rows must stay untouched, and the rows the
inserts write must read back through the decode path like the oracle reads
the same bytes.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import dsa_sparse_mla_query_gb300 as dsa
from dsa_sparse_mla_query_gb300 import inputs as I
import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda"
SENTINEL = 0x5A
REL = 2e-6      # fp32 evaluation slack relative to the value (rotation, scaling)
REL_ROW = 1e-6  # and relative to its row's largest magnitude (LayerNorm's cancellation near zero)


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    dsa.load()
    yield
    torch.cuda.synchronize()


_E4M3 = np.array([oracle.e4m3_value(c) for c in range(256)], np.float64)


def _bf16(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def _bf16_quantum(v):
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 7)


def _e4m3_quantum(t):
    a = np.maximum(np.abs(t), 2.0 ** -6)
    return np.exp2(np.floor(np.log2(a)) - 3)


def _nearest(got, exact, quantum, what):
    """got is a nearest rounding of exact, up to the fp32 evaluation's slack:
    REL of the value plus REL_ROW of the largest magnitude in its last axis."""
    err = np.abs(got - exact)
    row = np.max(np.abs(exact), axis=-1, keepdims=True)
    bound = 0.5 * quantum * (1 + 1e-9) + REL * np.abs(exact) + REL_ROW * row
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} values not a nearest rounding; worst excess " \
                          f"{np.max(err - bound):.3e}"


def _check_bf16_store(got_bits_t, exact, what):
    got = _bf16(got_bits_t)
    _nearest(got, exact, _bf16_quantum(exact), what)
    enc = np.vectorize(oracle.bf16_encode, otypes=[np.uint16])(exact)
    same = (got_bits_t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16) == enc).mean()
    assert same > 0.995, f"{what}: only {same:.4f} of the values equal the oracle's rounding"


def _check_e4m3_store(codes_t, scale_gpu, exact, group, what, agree_rows=None):
    """codes [n, d] uint8, scale_gpu fp64 [n, d / group], exact fp64 [n, d];
    agreement with the oracle's own codes on agree_rows (all rows by default)."""
    codes = codes_t.cpu().numpy()
    n, d = exact.shape
    amax = np.abs(exact.reshape(n, d // group, group)).max(axis=2)
    scale_o = np.where(amax > 0, amax / 448.0, 1.0)
    assert np.allclose(scale_gpu, scale_o, rtol=1e-6, atol=0), f"{what}: scales differ"
    t = exact.reshape(n, d // group, group) / scale_gpu[:, :, None]
    dec = _E4M3[codes].reshape(n, d // group, group)
    _nearest(dec, np.clip(t, -448.0, 448.0), _e4m3_quantum(t), what)
    rows = np.arange(n) if agree_rows is None else np.asarray(agree_rows)
    enc_codes, _ = oracle.quantize_rows_e4m3(exact[rows], group)
    same = (codes[rows] == enc_codes).mean()
    assert same > 0.995, f"{what}: only {same:.4f} of the codes equal the oracle's"


def _inputs(n, nq, num_rows, rope=True, seed=0, page_size=0):
    d = I.make_insert_inputs(n, nq, num_rows, DEV, seed=seed, rope=rope, page_size=page_size)
    return d, {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in d.items()}


def _insert_fp8(d, n, rows, pos=None):
    keys = torch.full((rows, 128), SENTINEL, dtype=torch.uint8, device=DEV)
    k_scale = torch.zeros(rows, dtype=torch.float32, device=DEV)
    latent = torch.full((rows, I.DS_MLA_ROW_BYTES), SENTINEL, dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pos = d["pos"] if pos is None else pos
    dsa.dsa_index_k_insert(d["x"], d["gamma"], d["beta"], 1e-6, pos, d["inv_freq"], d["slot"], n, keys, k_scale,
                           dsa.DSA_FP8_E4M3_ROWSCALE, rows, st)
    dsa.dsa_latent_insert(d["c_kv"], d["k_pe"], pos, d["inv_freq"], d["slot"], n, latent, dsa.DSA_FP8_DS_MLA, rows,
                          st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return keys, k_scale, latent


def _check_fp8_tokens(d, keys, k_scale, latent, pick, pos=None):
    """The e4m3 key and fp8_ds_mla latent rows of the tokens in pick against the oracle."""
    pk = torch.as_tensor(pick, dtype=torch.long).to(DEV)
    sl = d["slot"][pk]
    hp = (d["pos"] if pos is None else pos)[pk].cpu()
    ek = oracle.index_k(d["x"][pk].cpu(), d["gamma"].cpu(), d["beta"].cpu(), 1e-6, hp, d["inv_freq"].cpu())
    _check_e4m3_store(keys[sl], k_scale[sl].cpu().numpy().astype(np.float64)[:, None], ek, 128, "index keys")
    el = oracle.latent_k(d["c_kv"][pk].cpu(), d["k_pe"][pk].cpu(), hp, d["inv_freq"].cpu())
    got = latent[sl]
    scales = got[:, 512:528].contiguous().view(torch.float32).cpu().numpy().astype(np.float64)
    _check_e4m3_store(got[:, :512], scales, el[:, :512], 128, "latent codes")
    _check_bf16_store(got[:, 528:].contiguous().view(torch.bfloat16), el[:, 512:], "latent RoPE dims")


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("rope", [True, False])
def test_index_k_insert(fp8, rope):
    n, rows = 301, 1000  # a ragged last CTA; rows not written must stay untouched
    d, h = _inputs(n, 1, rows, rope=rope, seed=1)
    width = 128 if fp8 else 256
    cache = torch.full((rows, width), SENTINEL, dtype=torch.uint8, device=DEV)
    k_scale = torch.full((rows,), -7.0, dtype=torch.float32, device=DEV) if fp8 else None
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.dsa_index_k_insert(d["x"], d["gamma"], d["beta"], 1e-6, d["pos"], d["inv_freq"], d["slot"], n, cache, k_scale,
                           dsa.DSA_FP8_E4M3_ROWSCALE if fp8 else dsa.DSA_BF16, rows, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    exact = oracle.index_k(h["x"], h["gamma"], h["beta"], 1e-6, h["pos"], h["inv_freq"])
    slot = h["slot"].numpy()
    got = cache[d["slot"]]
    if fp8:
        _check_e4m3_store(got, k_scale[d["slot"]].cpu().numpy().astype(np.float64)[:, None], exact, 128, "index keys")
    else:
        _check_bf16_store(got.view(torch.bfloat16), exact, "index keys")
    untouched = np.setdiff1d(np.arange(rows), slot)
    assert torch.all(cache[torch.from_numpy(untouched).to(DEV)] == SENTINEL)


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("rope", [True, False])
def test_latent_insert(fp8, rope):
    n, rows = 203, 640
    d, h = _inputs(n, 1, rows, rope=rope, seed=2)
    width = I.DS_MLA_ROW_BYTES if fp8 else 2 * I.MLA_DIM
    latent = torch.full((rows, width), SENTINEL, dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.dsa_latent_insert(d["c_kv"], d["k_pe"], d["pos"], d["inv_freq"], d["slot"], n, latent,
                          dsa.DSA_FP8_DS_MLA if fp8 else dsa.DSA_BF16, rows, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    exact = oracle.latent_k(h["c_kv"], h["k_pe"], h["pos"], h["inv_freq"])
    got = latent[d["slot"]]
    if fp8:
        scales = got[:, 512:528].contiguous().view(torch.float32).cpu().numpy().astype(np.float64)
        _check_e4m3_store(got[:, :512], scales, exact[:, :512], 128, "latent codes")
        _check_bf16_store(got[:, 528:].contiguous().view(torch.bfloat16), exact[:, 512:], "latent RoPE dims")
    else:
        vals = got.contiguous().view(torch.bfloat16)
        assert torch.equal(vals[:, :512].cpu(), h["c_kv"]), "latent dims must be stored as given"
        _check_bf16_store(vals[:, 512:], exact[:, 512:], "latent RoPE dims")
    untouched = np.setdiff1d(np.arange(rows), h["slot"].numpy())
    assert torch.all(latent[torch.from_numpy(untouched).to(DEV)] == SENTINEL)


@pytest.mark.parametrize("rope", [True, False])
@pytest.mark.parametrize("in_place", [False, True])
def test_mla_q_prep(rope, in_place):
    d, h = _inputs(9001, 5, 9001, rope=rope, seed=3)  # positions up to 9000
    q = d["q"].clone()
    out = q if in_place else torch.empty_like(q)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.dsa_mla_q_prep(q, d["ssmax_s"], d["ssmax_b"], d["inv_freq"], d["q_pos"], 5, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    exact = oracle.mla_q(h["q"], h["ssmax_s"], h["ssmax_b"], h["q_pos"], h["inv_freq"])
    _check_bf16_store(out.reshape(5, -1), exact.reshape(5, -1), "attention query")


def test_insert_skips_and_reports():
    """slot -1 skips the token; a slot past the cache or a negative position is
    reported in the device status and skipped; the other tokens are written."""
    n, rows = 40, 64
    d, h = _inputs(n, 1, rows, seed=4)
    slot = d["slot"].clone()
    slot[3] = -1
    slot[7] = rows          # past the cache
    pos = d["pos"].clone()
    pos[11] = -5            # a negative position
    cache = torch.full((rows, 128), SENTINEL, dtype=torch.uint8, device=DEV)
    k_scale = torch.zeros(rows, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.dsa_index_k_insert(d["x"], d["gamma"], d["beta"], 1e-6, pos, d["inv_freq"], slot, n, cache, k_scale,
                           dsa.DSA_FP8_E4M3_ROWSCALE, rows, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 6  # DSA_ERR_BAD_INPUT
    for t in (3, 7, 11):
        r = int(h["slot"][t])
        assert torch.all(cache[r] == SENTINEL), f"token {t} must not be written"
    ok = [t for t in range(n) if t not in (3, 7, 11)]
    assert not torch.any(torch.all(cache[d["slot"][ok]] == SENTINEL, dim=1))
    with pytest.raises(dsa.DsaError):
        dsa.dsa_latent_insert(d["c_kv"], d["k_pe"], d["pos"], None, d["slot"], n, cache, 99, rows, st)


def test_inserted_rows_read_back_through_the_decode_path():
    """Keys and latent rows written by the inserts (e4m3 keys, fp8_ds_mla
    latent) are read by dsa_index_scores and sparse_mla_decode like the oracle
    reads the same bytes: the writer and the readers share one layout."""
    ctx, rows = 3000, 3000
    d, h = _inputs(ctx, 1, rows, seed=5)
    keys = torch.zeros((rows, 128), dtype=torch.uint8, device=DEV)
    k_scale = torch.zeros(rows, dtype=torch.float32, device=DEV)
    latent = torch.zeros((rows, I.DS_MLA_ROW_BYTES), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.dsa_index_k_insert(d["x"], d["gamma"], d["beta"], 1e-6, d["pos"], d["inv_freq"], d["slot"], ctx, keys, k_scale,
                           dsa.DSA_FP8_E4M3_ROWSCALE, rows, st)
    dsa.dsa_latent_insert(d["c_kv"], d["k_pe"], d["pos"], d["inv_freq"], d["slot"], ctx, latent, dsa.DSA_FP8_DS_MLA,
                          rows, st)
    # one query at the last position; the sequence's token j lives at row slot[j] (a page table of 1-token pages
    # is not allowed, so the rows are gathered into a contiguous copy for the query's view)
    order = d["slot"]
    keys_c, scale_c, lat_c = keys[order].contiguous(), k_scale[order].contiguous(), latent[order].contiguous()
    q_idx = I.to_bf16(I.normal(I.stream_key(5, 40), I._counters(0, 32 * 128, DEV))).view(1, 32, 128)
    w = I.normal(I.stream_key(5, 41), I._counters(0, 32, DEV)).to(torch.float32).view(1, 32)
    ss = torch.full((32,), 0.1, dtype=torch.float32, device=DEV)
    sb = torch.ones(32, dtype=torch.float32, device=DEV)
    ctx_len = torch.tensor([ctx], dtype=torch.int32, device=DEV)
    q_start = torch.tensor([0, 1], dtype=torch.int32, device=DEV)
    q_pos = torch.tensor([ctx - 1], dtype=torch.int32, device=DEV)
    seqs = dsa.Seqs(ctx_len, q_start, q_pos, max_ctx=ctx, max_q_per_seq=1, num_rows=rows,
                    seq_base=torch.zeros(1, dtype=torch.int64, device=DEV))
    ws_bytes = dsa.dsa_workspace_size(seqs, 1, 2048)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    ld = (ctx + 3) // 4 * 4
    scores = torch.empty(1, ld, dtype=torch.float32, device=DEV)
    dsa.dsa_index_scores(q_idx, w, ss, sb, d["inv_freq"], keys_c, scale_c, dsa.DSA_FP8_E4M3_ROWSCALE, seqs, 1, scores,
                         ld, ws, ws_bytes, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    layout = oracle.Layout(np.array([ctx], np.int32), rows, seq_base=np.zeros(1, np.int64))
    ref = oracle.index_scores(q_idx.cpu(), w.cpu(), ss.cpu(), sb.cpu(), h["inv_freq"], np.zeros(1, np.int32),
                              np.array([ctx - 1], np.int32), keys_c.cpu(), layout, key_scale=scale_c.cpu())[0]
    g = scores[0, :ctx].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(g - ref[:ctx])) <= 1e-4 * np.max(np.abs(ref[:ctx]))
    # attention over the inserted latent rows, positions 0..2047
    q = I.to_bf16(I.normal(I.stream_key(5, 42), I._counters(0, 64 * 576, DEV))).view(1, 64, 576)
    idx = torch.arange(2048, dtype=torch.int32, device=DEV).view(1, 2048)
    tlen = torch.tensor([2048], dtype=torch.int32, device=DEV)
    out = torch.empty(1, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(1, 64, dtype=torch.float32, device=DEV)
    dsa.sparse_mla_decode(q, lat_c, dsa.DSA_FP8_DS_MLA, seqs, 1, idx, tlen, 2048, 192 ** -0.5, out, lse, ws, ws_bytes,
                          st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ro, rl, _ = oracle.sparse_mla(q[0].cpu(), lat_c.cpu(), layout, 0, np.arange(2048, dtype=np.int32), 2048,
                                  192 ** -0.5, fp8=True)
    o = out[0].float().cpu().numpy()
    assert np.max(np.abs(o - ro)) <= 1e-2 * np.max(np.abs(ro))
    assert np.max(np.abs(lse[0].cpu().numpy() - rl)) <= 1e-3 * max(1.0, np.max(np.abs(rl)))


def test_insert_many_tokens_per_warp():
    """45001 new tokens: more than two grid passes of both kernels, so every
    warp takes several keys and rows, two loads ahead, with a ragged end.  Every
    key row is checked (against the oracle's own codes on a sample), the latent
    rows on a sample spread over the range and its last 300 tokens; no row
    outside the slots is written."""
    n, rows = 45001, 46000
    d, h = _inputs(n, 1, rows, seed=7)
    keys, k_scale, latent = _insert_fp8(d, n, rows)
    ek = oracle.index_k(h["x"], h["gamma"], h["beta"], 1e-6, h["pos"], h["inv_freq"])
    pick = np.unique(np.concatenate([np.linspace(0, n - 1, 700).astype(np.int64), np.arange(n - 300, n)]))
    _check_e4m3_store(keys[d["slot"]], k_scale[d["slot"]].cpu().numpy().astype(np.float64)[:, None], ek, 128,
                      "index keys", agree_rows=pick)
    _check_fp8_tokens(d, keys, k_scale, latent, pick)
    untouched = torch.from_numpy(np.setdiff1d(np.arange(rows), h["slot"].numpy())).to(DEV)
    assert torch.all(keys[untouched] == SENTINEL) and torch.all(latent[untouched] == SENTINEL)


def test_insert_positions_past_2_24():
    """RoPE angles on both sides of 2^24 radians-per-unit positions (the kernels
    change how they reduce the angle there) and near the largest position."""
    n, rows = 600, 600
    d, h = _inputs(n, 5, rows, seed=8)  # 5 attention queries
    pos = d["pos"].clone()
    pos[:300] += (1 << 24) - 150        # 2^24 - 150 .. 2^24 + 149
    pos[300:] += (1 << 31) - 1 - n      # up to 2^31 - 2
    keys, k_scale, latent = _insert_fp8(d, n, rows, pos=pos)
    _check_fp8_tokens(d, keys, k_scale, latent, np.arange(n), pos=pos)
    q = d["q"].clone()
    assert q.shape == (5, 64, 576)
    qp = torch.tensor([(1 << 24) - 1, 1 << 24, (1 << 24) + 1, (1 << 30) + 7, (1 << 31) - 2],
                      dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.dsa_mla_q_prep(q, d["ssmax_s"], d["ssmax_b"], d["inv_freq"], qp, 5, q, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    exact = oracle.mla_q(h["q"], h["ssmax_s"], h["ssmax_b"], qp.cpu(), h["inv_freq"])
    _check_bf16_store(q.reshape(5, -1), exact.reshape(5, -1), "attention query")


def test_insert_bench_size_sampled():
    """The benchmark's step (2^20 new tokens in 64-token pages taken in a random
    order, e4m3 keys, fp8_ds_mla latent), checked on 257 sampled tokens."""
    n = rows = 1 << 20
    d, _ = _inputs(n, 1, rows, seed=6, page_size=64)
    keys, k_scale, latent = _insert_fp8(d, n, rows)
    _check_fp8_tokens(d, keys, k_scale, latent, np.linspace(0, n - 1, 257).astype(np.int64))
    assert not torch.any(torch.all(keys == SENTINEL, dim=1)), "every row is some token's"
