"""Pins of the CPU oracle to facts other than itself.

Each ``pin_*`` takes a handle on a build of the oracle (``oracle.lib()`` or a
deliberately broken copy) and raises AssertionError when the build disagrees
with a closed form, an invariant, a library routine on a special case, or a
byte count printed on the pages.  ``tests/test_oracle.py`` runs them on the
real oracle; ``tests/test_oracle_mutants.py`` checks that every planted
mistake fails at least one of them.

Sources: "Day 0 support for Mistral Large 4" (vLLM blog) and the colibri
"Mistral-Large-4" doc (What differs from GLM-5.2).
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# helpers
def bf16_bits(x) -> np.ndarray:
    """Round fp64/fp32 values to bf16 bit patterns (nearest even) with numpy."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def contiguous(ctx_len, rows):
    base = np.concatenate([[0], np.cumsum(ctx_len)[:-1]]).astype(np.int64)
    return oracle.Layout(np.asarray(ctx_len, np.int32), rows, seq_base=base)


def index_case(n=16, pos=None, rope=False, seed=1):
    """Random small indexer inputs: one query in one sequence of n keys."""
    rng = np.random.default_rng(seed)
    q = bf16_bits(rng.standard_normal((1, 32, 128)))
    w = rng.standard_normal((1, 32)).astype(np.float32)
    s = np.full(32, 0.0, np.float32)
    b = np.full(32, 1.0, np.float32)
    inv = (0.5 ** np.arange(32)).astype(np.float32) if rope else None
    keys = bf16_bits(rng.standard_normal((n, 128)))
    pos = n - 1 if pos is None else pos
    return dict(q=q, w=w, ssmax_s=s, ssmax_b=b, inv_freq=inv, q_seq=np.array([0], np.int32),
                q_pos=np.array([pos], np.int32), keys=keys)


def scores_of(L, c, layout=None, **over):
    d = dict(c)
    d.update(over)
    lay = layout or contiguous([d["keys"].shape[0]], d["keys"].shape[0])
    return oracle.index_scores(d["q"], d["w"], d["ssmax_s"], d["ssmax_b"], d["inv_freq"], d["q_seq"], d["q_pos"],
                               d["keys"], lay, key_scale=d.get("key_scale"), L=L)[0]


def close(a, b, tol=1e-12):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), "finite pattern differs"
    assert np.array_equal(a[~fin], b[~fin]), "non-finite values differ"
    err = np.max(np.abs(a[fin] - b[fin]), initial=0.0)
    assert err <= tol * max(1.0, np.max(np.abs(b[fin]), initial=0.0)), f"max err {err}"


# ---------------------------------------------------------------------------
# formats
def pin_bf16_decode(L):
    """bf16 = top half of binary32: every 16-bit pattern against torch."""
    import torch
    codes = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_value(int(c), L=L) for c in codes[::97]] + [oracle.bf16_value(0x3F80, L=L)])
    want = np.concatenate([ref[::97], [1.0]])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    m = ~np.isnan(want)
    assert np.array_equal(got[m], want[m])


def pin_e4m3_decode(L):
    """OCP E4M3: all 256 codes against torch.float8_e4m3fn, plus the format's
    landmarks (1.0 = 0x38, max 448 = 0x7E, min subnormal 2^-9 = 0x01, NaN = 0x7F)."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(int(c), L=L) for c in codes])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m])
    assert oracle.e4m3_value(0x38, L=L) == 1.0 and oracle.e4m3_value(0x7E, L=L) == 448.0
    assert oracle.e4m3_value(0x01, L=L) == 2.0 ** -9 and oracle.e4m3_value(0x80 | 0x38, L=L) == -1.0
    assert math.isnan(oracle.e4m3_value(0x7F, L=L)) and math.isnan(oracle.e4m3_value(0xFF, L=L))


def pin_kv_bytes(L):
    """Per-token cache bytes printed on the pages (tests/golden/kv_bytes.json)."""
    with open(os.path.join(GOLDEN, "kv_bytes.json")) as f:
        g = json.load(f)
    lat8 = oracle.latent_row_bytes(oracle.LATENT_DS_MLA, L=L)
    lat16 = oracle.latent_row_bytes(oracle.LATENT_BF16, L=L)
    idx8 = oracle.index_row_bytes(oracle.KEYS_E4M3_ROW, L=L)
    n_lat, n_idx = g["cache_owning_layers"], g["indexer_layers"]
    assert n_lat * lat8 == g["latent_bytes_fp8_ds_mla"]
    assert n_idx * idx8 == g["indexer_bytes_fp8"]
    assert n_lat * lat8 + n_idx * idx8 == g["total_bytes_fp8"]
    assert lat8 == g["fp8_ds_mla_row"] and lat16 == g["bf16_row"] and idx8 == g["indexer_row"]
    assert n_lat * lat16 + n_idx * idx8 == g["total_bytes_bf16"]
    assert n_lat * g["plain_e4m3_row"] + n_idx * idx8 == g["total_bytes_plain_e4m3"]


def pin_ds_mla_row(L):
    """fp8_ds_mla row decode: group g of 128 latent dims uses scale g; RoPE
    dims are bf16 after the 16 scale bytes."""
    row = np.zeros(656, np.uint8)
    row[:512] = 0x38                                   # e4m3 1.0 everywhere
    row[5] = 0xB8                                      # -1.0
    row[300] = 0x40                                    # 2.0
    scales = np.array([1.0, 2.0, 4.0, 0.5], np.float32)
    row[512:528] = np.frombuffer(scales.tobytes(), np.uint8)
    rope = np.arange(64, dtype=np.float32) - 31.5      # exact in bf16
    row[528:656] = np.frombuffer(bf16_bits(rope).tobytes(), np.uint8)
    got = oracle.ds_mla_row(row, L=L)
    want = np.concatenate([np.repeat(scales.astype(np.float64), 128), rope.astype(np.float64)])
    want[5] = -1.0
    want[300] = 2.0 * 4.0
    assert np.array_equal(got, want)


# ---------------------------------------------------------------------------
# indexer score
def _one_head_case(n=8, head=3, weight=2.0, pos=None):
    rng = np.random.default_rng(7)
    c = index_case(n=n, pos=pos)
    q = bf16_bits(rng.standard_normal((1, 32, 128)))
    q[0, head, :] = 0
    q[0, head, :8] = bf16_bits(np.ones(8))            # q_h = 1 on dims 0..7
    w = np.zeros((1, 32), np.float32)
    w[0, head] = weight
    keys = np.zeros((n, 128), np.float32)
    keys[:, :8] = (np.arange(n) - 2.0)[:, None]        # k_j = j-2 on dims 0..7
    keys[:, 8:] = rng.standard_normal((n, 120))        # q_h is 0 there
    c.update(q=q, w=w, keys=bf16_bits(keys))
    return c


def pin_score_single_head(L):
    """One head weighted 2, f = 1, q.k = 8(j-2): score = 2 relu(8(j-2)/sqrt(128))/sqrt(32) = max(j-2,0)/4."""
    c = _one_head_case()
    got = scores_of(L, c)
    want = np.maximum(np.arange(8) - 2.0, 0.0) / 4.0
    close(got, want, 1e-14)


def pin_score_negative_weight(L):
    """The weight multiplies relu(...), it is not inside it: w = -2 gives -max(j-2,0)/4."""
    c = _one_head_case(weight=-2.0)
    close(scores_of(L, c), -np.maximum(np.arange(8) - 2.0, 0.0) / 4.0, 1e-14)


def pin_ssmax_scale(L):
    """SSMax f = s*ln(pos+1) + b multiplies the query before relu:
    f > 0 scales the score, f < 0 mirrors the relu."""
    c = _one_head_case(pos=7)
    s = np.zeros(32, np.float32)
    b = np.zeros(32, np.float32)
    s[3], b[3] = 0.5, -0.25
    f = float(np.float32(0.5)) * math.log(8.0) + float(np.float32(-0.25))
    base = np.maximum(np.arange(8) - 2.0, 0.0) / 4.0
    close(scores_of(L, c, ssmax_s=s, ssmax_b=b), f * base, 1e-13)
    # negative f: relu(f x) = |f| relu(-x): keys 0,1 (q.k < 0) now count
    s[3], b[3] = 0.0, -1.0
    close(scores_of(L, c, ssmax_s=s, ssmax_b=b), np.maximum(2.0 - np.arange(8), 0.0) / 4.0, 1e-14)
    # position 0: ln 1 = 0 so f = b whatever s is
    c0 = _one_head_case(pos=0)
    s[3], b[3] = 100.0, 3.0
    got = scores_of(L, c0, ssmax_s=s, ssmax_b=b)
    assert got[0] == 0.0 and np.all(np.isneginf(got[1:]))


def pin_causal_mask(L):
    """Keys after the query position are -inf; the position itself scores."""
    c = _one_head_case(n=8, pos=4)
    got = scores_of(L, c)
    assert np.all(np.isneginf(got[5:])) and np.all(np.isfinite(got[:5]))
    assert abs(got[4] - 0.5) < 1e-14


def pin_rope_interleaved(L):
    """Interleaved pairs: q with pair i = (1, 0) rotated by theta = pos*inv_freq_i
    becomes (cos, sin); against a key (0, 1) on that pair the dot is sin(theta).
    A half-split rotation or the opposite direction gives 0 here."""
    n, pos, pair, head = 6, 3, 5, 0
    c = index_case(n=n, pos=pos, rope=True)
    inv = (0.1 * (np.arange(32) + 1)).astype(np.float32)
    inv[pair] = 0.5
    q = np.zeros((1, 32, 128), np.uint16)
    q[0, head, 2 * pair] = bf16_bits(1.0)
    w = np.zeros((1, 32), np.float32)
    w[0, head] = 64.0                                  # cancels 1/(sqrt(128) sqrt(32))
    keys = np.zeros((n, 128), np.float32)
    keys[:, 2 * pair + 1] = 1.0
    got = scores_of(L, c, q=q, w=w, keys=bf16_bits(keys), inv_freq=inv)
    th = pos * float(inv[pair])
    want = np.full(n, -np.inf)
    want[:pos + 1] = max(math.sin(th), 0.0)
    assert math.sin(th) > 0.5
    close(got, want, 1e-14)
    # the cosine component lands on dim 2*pair
    keys = np.zeros((n, 128), np.float32)
    keys[:, 2 * pair] = 1.0
    got = scores_of(L, c, q=q, w=w, keys=bf16_bits(keys), inv_freq=inv)
    want[:pos + 1] = max(math.cos(th), 0.0)
    close(got, want, 1e-14)


def pin_rope_first_64_only(L):
    """Dims 64..127 are never rotated: a query and key on dim 100 only give
    the same score at any position and frequency."""
    n = 5
    q = np.zeros((1, 32, 128), np.uint16)
    q[0, 9, 100] = bf16_bits(1.5)
    w = np.zeros((1, 32), np.float32)
    w[0, 9] = 64.0
    keys = np.zeros((n, 128), np.float32)
    keys[:, 100] = np.arange(n) + 1.0
    inv = np.full(32, 0.7, np.float32)
    for pos in (0, 4):
        c = index_case(n=n, pos=pos, rope=True)
        got = scores_of(L, c, q=q, w=w, keys=bf16_bits(keys), inv_freq=inv)
        want = np.full(n, -np.inf)
        want[:pos + 1] = 1.5 * (np.arange(pos + 1) + 1.0)
        close(got, want, 1e-14)


def pin_nope_is_zero_frequency(L):
    """NoPE equals RoPE with every frequency 0 (angle 0), on random data."""
    c = index_case(n=40, rope=True, seed=3)
    a = scores_of(L, c, inv_freq=None)
    b = scores_of(L, c, inv_freq=np.zeros(32, np.float32))
    close(a, b, 0.0)


def pin_rope_rotation_invariance(L):
    """Rotating the key by the query's own angles (same pairs) leaves the
    unrotated score: R(theta) q . R(theta) k = q . k.  Checked with exact
    rotations by multiples of pi/2 (cos, sin in {0, +-1})."""
    c = index_case(n=12, pos=11, rope=False, seed=5)
    base = scores_of(L, c)
    # theta_i = pos * inv_freq_i = 11 * (pi/2 * m_i / 11) -> quarter turns m_i
    m = np.arange(32) % 4
    inv = (np.pi / 2 * m / 11.0).astype(np.float32)
    th = 11.0 * inv.astype(np.float64)
    cs, sn = np.round(np.cos(th)), np.round(np.sin(th))
    assert np.allclose(np.cos(th), cs, atol=1e-6)
    k = np.array([oracle.bf16_value(int(v), L=L) for v in c["keys"].ravel()]).reshape(12, 128)
    kr = k.copy()
    kr[:, 0:64:2] = k[:, 0:64:2] * cs - k[:, 1:64:2] * sn
    kr[:, 1:64:2] = k[:, 0:64:2] * sn + k[:, 1:64:2] * cs
    got = scores_of(L, c, inv_freq=inv, keys=bf16_bits(kr))
    # the fp32 angle is not exactly a quarter turn: allow its tiny residue
    close(got, base, 1e-5)


def pin_linear_in_weights(L):
    """The score is linear in the head weights."""
    c = index_case(n=30, rope=True, seed=11)
    rng = np.random.default_rng(2)
    w1 = rng.standard_normal((1, 32)).astype(np.float32)
    w2 = rng.standard_normal((1, 32)).astype(np.float32)
    a = scores_of(L, c, w=w1)
    b = scores_of(L, c, w=w2)
    ab = scores_of(L, c, w=(w1.astype(np.float64) + w2).astype(np.float32))
    close(ab[np.isfinite(ab)], (a + b)[np.isfinite(ab)], 1e-6)


def pin_paged_equals_contiguous(L):
    """A page table gives the same scores as the rows gathered in order."""
    rng = np.random.default_rng(4)
    ps, n = 4, 22
    pages = (n + ps - 1) // ps
    perm = rng.permutation(pages + 3)[:pages].astype(np.int32)
    phys = rng.standard_normal(((pages + 3) * ps, 128))
    keys_phys = bf16_bits(phys)
    logical = np.concatenate([keys_phys[p * ps:(p + 1) * ps] for p in perm])[:n]
    c = index_case(n=n, rope=True, seed=9)
    paged = oracle.Layout(np.array([n], np.int32), keys_phys.shape[0], page_table=perm[None, :], page_size=ps)
    a = scores_of(L, c, keys=keys_phys, layout=paged)
    b = scores_of(L, c, keys=logical)
    close(a, b, 0.0)


def pin_fp8_keys_equal_their_values(L):
    """e4m3 keys times a power-of-two row scale score like bf16 keys holding
    the same values (all exact in bf16)."""
    rng = np.random.default_rng(6)
    n = 17
    codes = rng.integers(0, 256, (n, 128)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C               # no NaN codes
    scale = (2.0 ** rng.integers(-6, 3, n)).astype(np.float32)
    vals = np.array([[oracle.e4m3_value(int(x), L=L) for x in r] for r in codes]) * scale[:, None]
    c = index_case(n=n, rope=True, seed=12)
    a = scores_of(L, c, keys=codes, key_scale=scale)
    b = scores_of(L, c, keys=bf16_bits(vals))
    close(a, b, 0.0)


def pin_multi_query_sequences(L):
    """Two sequences, two queries each: each query reads only its own
    sequence's keys up to its own position."""
    rng = np.random.default_rng(13)
    ctx = [9, 6]
    keys = bf16_bits(rng.standard_normal((15, 128)))
    lay = contiguous(ctx, 15)
    q = bf16_bits(rng.standard_normal((4, 32, 128)))
    w = rng.standard_normal((4, 32)).astype(np.float32)
    s = (0.1 * np.ones(32)).astype(np.float32)
    b = np.ones(32, np.float32)
    inv = (0.3 ** np.arange(32)).astype(np.float32)
    qseq = np.array([0, 0, 1, 1], np.int32)
    qpos = np.array([7, 8, 4, 5], np.int32)
    allq = oracle.index_scores(q, w, s, b, inv, qseq, qpos, keys, lay, L=L)
    for t in range(4):
        bb = int(qseq[t])
        sub = keys[sum(ctx[:bb]):sum(ctx[:bb]) + ctx[bb]]
        one = oracle.index_scores(q[t:t + 1], w[t:t + 1], s, b, inv, np.array([0], np.int32), qpos[t:t + 1], sub,
                                  contiguous([ctx[bb]], ctx[bb]), ld=9, L=L)[0]
        close(allq[t], one, 0.0)


# ---------------------------------------------------------------------------
# top-k
def pin_topk_library(L):
    """Exact top-k against numpy's lexsort (score descending, index
    ascending) on scores with many ties."""
    rng = np.random.default_rng(21)
    for n, k in ((50, 8), (300, 64), (64, 64), (10, 30), (1, 1), (5, 0)):
        s = rng.integers(-5, 6, n).astype(np.float64) * 0.25
        idx, m = oracle.topk(s, k, L=L)
        order = np.lexsort((np.arange(n), -s))
        assert m == min(n, k)
        assert np.array_equal(idx[:m], order[:m].astype(np.int32))
        assert np.all(idx[m:] == -1)


def pin_topk_properties(L):
    """Every selected score >= every unselected one; among scores equal to
    the k-th, the selected indices are the smallest."""
    rng = np.random.default_rng(22)
    n, k = 1000, 100
    s = np.round(rng.standard_normal(n), 1)
    idx, m = oracle.topk(s, k, L=L)
    sel = np.zeros(n, bool)
    sel[idx[:m]] = True
    assert sel.sum() == k
    assert s[sel].min() >= s[~sel].max()
    kth = s[sel].min()
    eq = np.flatnonzero(s == kth)
    assert np.array_equal(np.flatnonzero(sel & (s == kth)), eq[:np.count_nonzero(sel & (s == kth))])


def pin_topk_short_context(L):
    """Context <= k: the selection is every causal key; the other slots -1."""
    s = np.random.default_rng(23).standard_normal(37)
    idx, m = oracle.topk(s, 2048, L=L)
    assert m == 37 and sorted(idx[:m].tolist()) == list(range(37)) and np.all(idx[m:] == -1)


# ---------------------------------------------------------------------------
# sparse MLA
def mla_case(n=12, seed=31):
    rng = np.random.default_rng(seed)
    q = bf16_bits(rng.standard_normal((64, 576)))
    lat = bf16_bits(rng.standard_normal((n, 576)))
    return q, lat, contiguous([n], n)


def _vals(L, bits):
    return np.array([oracle.bf16_value(int(v), L=L) for v in np.asarray(bits).ravel()]).reshape(np.shape(bits))


def pin_mla_one_key(L):
    """One selected key: every head outputs that key's 512 latent dims and
    LSE = sm_scale * q_h . c_j over all 576 dims."""
    q, lat, lay = mla_case()
    qv, lv = _vals(L, q), _vals(L, lat)
    idx = np.array([7, -1, -1], np.int32)
    out, lse, _ = oracle.sparse_mla(q, lat, lay, 0, idx, 3, 0.125, L=L)
    close(out, np.tile(lv[7, :512], (64, 1)), 0.0)
    close(lse, 0.125 * (qv @ lv[7]), 1e-12)


def pin_mla_two_keys_rope_dims(L):
    """Two keys that differ only in the 64 RoPE dims: the score uses all 576
    dims, softmax is over keys, LSE = log(e^s1 + e^s2) (natural log)."""
    q = np.zeros((64, 576), np.uint16)
    lat = np.zeros((2, 576), np.float32)
    lat[0, :512] = 1.0
    lat[1, :512] = -1.0
    lat[0, 512:] = 0.25
    lat[1, 512:] = -0.5
    h = np.arange(64)
    qf = np.zeros((64, 576), np.float32)
    qf[:, 512:] = ((h % 7) - 3.0)[:, None] / 8.0
    q = bf16_bits(qf)
    lay = contiguous([2], 2)
    out, lse, p = oracle.sparse_mla(q, bf16_bits(lat), lay, 0, np.array([0, 1], np.int32), 2, 0.5,
                                    want_probs=True, L=L)
    a = 0.5 * 64 * 0.25 * ((h % 7) - 3.0) / 8.0
    b = 0.5 * 64 * -0.5 * ((h % 7) - 3.0) / 8.0
    p0 = 1.0 / (1.0 + np.exp(b - a))
    close(out, np.repeat((p0 * 1.0 + (1 - p0) * -1.0)[:, None], 512, 1), 1e-13)
    close(lse, np.logaddexp(a, b), 1e-13)
    close(p[:, 0], p0, 1e-13)


def pin_mla_uniform_scores(L):
    """q = 0: equal weights, O = mean of the selected rows, LSE = ln n."""
    _, lat, lay = mla_case(n=20)
    lv = _vals(L, lat)
    idx = np.array([3, 9, 4, 17, -1, 0], np.int32)
    out, lse, p = oracle.sparse_mla(np.zeros((64, 576), np.uint16), lat, lay, 0, idx, 6, 1.0, want_probs=True, L=L)
    sel = [3, 9, 4, 17, 0]
    close(out, np.tile(lv[sel, :512].mean(0), (64, 1)), 1e-14)
    close(lse, np.full(64, math.log(5.0)), 1e-14)
    assert np.all(p[:, 4] == 0.0)


def pin_mla_softmax_sums_to_one(L):
    """Softmax weights of every head sum to 1 (|sum - 1| <= 1e-12)."""
    q, lat, lay = mla_case(n=300, seed=33)
    idx = np.random.default_rng(1).permutation(300)[:257].astype(np.int32)
    _, _, p = oracle.sparse_mla(q, lat, lay, 0, idx, 257, 1.0 / math.sqrt(192), want_probs=True, L=L)
    assert np.max(np.abs(p.sum(1) - 1.0)) <= 1e-12
    assert np.all(p >= 0)


def pin_mla_empty(L):
    """No selected key: O = 0, LSE = -inf (an empty row is neutral)."""
    q, lat, lay = mla_case()
    out, lse, _ = oracle.sparse_mla(q, lat, lay, 0, np.full(4, -1, np.int32), 4, 1.0, L=L)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    out, lse, _ = oracle.sparse_mla(q, lat, lay, 0, np.full(4, 2, np.int32), 0, 1.0, L=L)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def pin_mla_library_softmax(L):
    """Against scipy.special.softmax/logsumexp with numpy matmuls (library
    routines on a small random case)."""
    from scipy.special import logsumexp, softmax
    q, lat, lay = mla_case(n=40, seed=34)
    qv, lv = _vals(L, q), _vals(L, lat)
    idx = np.arange(0, 40, 3, dtype=np.int32)
    sc = 1.0 / math.sqrt(192)
    out, lse, _ = oracle.sparse_mla(q, lat, lay, 0, idx, len(idx), sc, L=L)
    s = sc * qv @ lv[idx].T
    close(out, softmax(s, axis=1) @ lv[idx, :512], 1e-12)
    close(lse, logsumexp(s, axis=1), 1e-12)


def pin_mla_sparse_equals_dense(L):
    """Context <= k: top-k selects every causal key, so sparse attention over
    the selection equals dense attention over all keys (order-free)."""
    q, lat, lay = mla_case(n=50, seed=35)
    s = np.random.default_rng(3).standard_normal(50)
    idx, m = oracle.topk(s, 2048, L=L)
    a, la, _ = oracle.sparse_mla(q, lat, lay, 0, idx, 2048, 0.07, L=L)
    b, lb, _ = oracle.sparse_mla(q, lat, lay, 0, np.arange(50, dtype=np.int32), 50, 0.07, L=L)
    close(a, b, 1e-12)
    close(la, lb, 1e-12)


def pin_mla_fp8_equals_values(L):
    """fp8_ds_mla rows score and average like bf16 rows holding the same
    dequantised values (power-of-two scales keep them exact)."""
    rng = np.random.default_rng(36)
    n = 24
    rows = np.zeros((n, 656), np.uint8)
    codes = rng.integers(0, 256, (n, 512)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x30
    rows[:, :512] = codes
    sc = (2.0 ** rng.integers(-4, 2, (n, 4))).astype(np.float32)
    rows[:, 512:528] = np.frombuffer(sc.tobytes(), np.uint8).reshape(n, 16)
    rope = bf16_bits(rng.standard_normal((n, 64)))
    rows[:, 528:] = np.frombuffer(rope.tobytes(), np.uint8).reshape(n, 128)
    vals = np.stack([oracle.ds_mla_row(r, L=L) for r in rows])
    q = bf16_bits(rng.standard_normal((64, 576)))
    lay = contiguous([n], n)
    idx = rng.permutation(n)[:15].astype(np.int32)
    a, la, _ = oracle.sparse_mla(q, rows, lay, 0, idx, 15, 0.1, fp8=True, L=L)
    b, lb, _ = oracle.sparse_mla(q, bf16_bits(vals), lay, 0, idx, 15, 0.1, L=L)
    close(a, b, 0.0)
    close(la, lb, 0.0)


def pin_mla_paged(L):
    """Selected tokens go through the page table."""
    rng = np.random.default_rng(37)
    ps, n = 8, 30
    pages = 4
    perm = np.array([5, 0, 3, 1], np.int32)
    phys = bf16_bits(rng.standard_normal((6 * ps, 576)))
    logical = np.concatenate([phys[p * ps:(p + 1) * ps] for p in perm])[:n]
    q = bf16_bits(rng.standard_normal((64, 576)))
    idx = np.array([29, 0, 8, 17, 25, 3], np.int32)
    paged = oracle.Layout(np.array([n], np.int32), phys.shape[0], page_table=perm[None, :pages], page_size=ps)
    a, la, _ = oracle.sparse_mla(q, phys, paged, 0, idx, 6, 0.1, L=L)
    b, lb, _ = oracle.sparse_mla(q, logical, contiguous([n], n), 0, idx, 6, 0.1, L=L)
    close(a, b, 0.0)
    close(la, lb, 0.0)


# ---------------------------------------------------------------------------
# the cache-write side: encoders, indexer key, latent row, attention query
def pin_e4m3_encode_roundtrip(L):
    """Every finite e4m3 code encodes back from its own value (both zeros)."""
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert oracle.e4m3_encode(oracle.e4m3_value(c, L), L) == c, hex(c)


def pin_e4m3_encode_ties_and_range(L):
    """Midpoints between neighbouring codes go to the even code; past 448 the
    code saturates; below half the smallest subnormal it is zero."""
    for c in range(0, 0x7E):
        lo, hi = oracle.e4m3_value(c, L), oracle.e4m3_value(c + 1, L)
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode((lo + hi) / 2, L) == want, hex(c)
        assert oracle.e4m3_encode(lo + (hi - lo) * 0.49, L) == c
        assert oracle.e4m3_encode(-(lo + (hi - lo) * 0.51), L) == 0x80 | (c + 1)
    assert oracle.e4m3_encode(449.0, L) == 0x7E and oracle.e4m3_encode(-1e9, L) == 0xFE
    assert oracle.e4m3_encode(2.0 ** -11, L) == 0 and oracle.e4m3_encode(2.0 ** -10 * 1.01, L) == 1


def pin_bf16_encode(L):
    """Every finite bf16 pattern encodes back from its value; values exact in
    fp32 round like numpy's nearest-even bit rounding; ties to even."""
    for b in range(0, 1 << 16, 7):
        if (b & 0x7F80) == 0x7F80:
            continue
        assert oracle.bf16_encode(oracle.bf16_value(b, L), L) == b, hex(b)
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(500) * np.exp(rng.uniform(-20, 20, 500))).astype(np.float32)
    want = bf16_bits(x)
    got = np.array([oracle.bf16_encode(float(v), L) for v in x], np.uint16)
    assert np.array_equal(got, want)
    assert oracle.bf16_encode(1.0 + 2.0 ** -8, L) == 0x3F80 and oracle.bf16_encode(1.0 + 3 * 2.0 ** -8, L) == 0x3F82


def _insert_rows(n, d, seed):
    rng = np.random.default_rng(seed)
    return bf16_bits(rng.standard_normal((n, d)) * 2.0 + 0.3)


def pin_index_k_layer_norm_library(L):
    """NoPE: the key is torch's fp64 layer_norm of the bf16 inputs."""
    import torch
    x = _insert_rows(6, 128, 11)
    rng = np.random.default_rng(12)
    g = rng.uniform(0.5, 1.5, 128).astype(np.float32)
    b = rng.uniform(-0.2, 0.2, 128).astype(np.float32)
    got = oracle.index_k(x, g, b, 1e-6, np.arange(6, dtype=np.int32), None, L=L)
    xv = torch.from_numpy(np.array([[oracle.bf16_value(int(v), L) for v in row] for row in x]))
    want = torch.nn.functional.layer_norm(xv, (128,), torch.from_numpy(g).double(), torch.from_numpy(b).double(),
                                          eps=1e-6).numpy()
    close(got, want, 1e-11)


def pin_index_k_constant_row_is_beta(L):
    """A constant input row normalises to zero, leaving beta (rotated on RoPE layers)."""
    x = np.full((1, 128), bf16_bits(np.array([3.0]))[0], np.uint16)
    g = np.full(128, 2.0, np.float32)
    b = (np.arange(128) / 128.0).astype(np.float32)
    got = oracle.index_k(x, g, b, 1e-6, np.array([0], np.int32), None, L=L)
    close(got[0], b.astype(np.float64), 1e-12)


def pin_index_k_rope_complex(L):
    """RoPE layers: dims 0..63 as complex pairs x0 + i x1 times exp(i pos f);
    dims 64..127 as without rotation."""
    x = _insert_rows(4, 128, 13)
    g = np.ones(128, np.float32)
    b = np.zeros(128, np.float32)
    fr = (1.0 / 10000.0 ** (np.arange(32) / 32.0)).astype(np.float32)
    pos = np.array([0, 5, 1000, 77777], np.int32)
    plain = oracle.index_k(x, g, b, 1e-6, pos, None, L=L)
    rot = oracle.index_k(x, g, b, 1e-6, pos, fr, L=L)
    z = (plain[:, 0:64:2] + 1j * plain[:, 1:64:2]) * np.exp(1j * pos[:, None].astype(np.float64) * fr.astype(np.float64))
    close(rot[:, 0:64:2], z.real, 1e-10)
    close(rot[:, 1:64:2], z.imag, 1e-10)
    close(rot[:, 64:], plain[:, 64:], 0.0)


def pin_latent_k(L):
    """The 512 latent dims are the inputs' values; the 64 RoPE dims are the
    k_pe values rotated as complex pairs (unrotated without a frequency table)."""
    c = _insert_rows(3, 512, 14)
    k = _insert_rows(3, 64, 15)
    fr = (0.5 / 10000.0 ** (np.arange(32) / 32.0)).astype(np.float32)
    pos = np.array([1, 33, 4095], np.int32)
    got = oracle.latent_k(c, k, pos, fr, L=L)
    cv = np.array([[oracle.bf16_value(int(v), L) for v in row] for row in c])
    kv = np.array([[oracle.bf16_value(int(v), L) for v in row] for row in k])
    close(got[:, :512], cv, 0.0)
    z = (kv[:, 0::2] + 1j * kv[:, 1::2]) * np.exp(1j * pos[:, None].astype(np.float64) * fr.astype(np.float64))
    close(got[:, 512::2], z.real, 1e-10)
    close(got[:, 513::2], z.imag, 1e-10)
    close(oracle.latent_k(c, k, pos, None, L=L)[:, 512:], kv, 0.0)


def pin_mla_q(L):
    """Every dim of head h times s_h ln(pos+1) + b_h; RoPE dims rotated first
    (complex pairs); position 0 gives the factor b_h."""
    rng = np.random.default_rng(16)
    q = _insert_rows(2 * 64, 576, 17).reshape(2, 64, 576)
    ss = rng.uniform(0.05, 0.15, 64).astype(np.float32)
    sb = rng.uniform(0.9, 1.1, 64).astype(np.float32)
    fr = (1.0 / 10000.0 ** (np.arange(32) / 32.0)).astype(np.float32)
    pos = np.array([0, 9000], np.int32)
    got = oracle.mla_q(q, ss, sb, pos, fr, L=L)
    qv = np.vectorize(lambda b: oracle.bf16_value(int(b), L))(q)
    f = ss[None, :].astype(np.float64) * np.log(pos[:, None] + 1.0) + sb[None, :].astype(np.float64)
    close(got[:, :, :512], qv[:, :, :512] * f[:, :, None], 1e-12)
    z = (qv[:, :, 512::2] + 1j * qv[:, :, 513::2]) * np.exp(1j * pos[:, None, None] * fr.astype(np.float64))
    close(got[:, :, 512::2], z.real * f[:, :, None], 1e-10)
    close(got[:, :, 513::2], z.imag * f[:, :, None], 1e-10)
    close(got[0, :, :512], qv[0, :, :512] * sb[:, None].astype(np.float64), 1e-12)


def pin_quantize_rows_e4m3(L):
    """Per-group quantisation: the largest magnitude of a group maps to +-448,
    and every value is recovered within half an e4m3 step of its scaled self."""
    rng = np.random.default_rng(18)
    v = rng.standard_normal((5, 512)) * np.exp(rng.uniform(-3, 3, (5, 1)))
    codes, scale = oracle.quantize_rows_e4m3(v, 128, L=L)
    dec = np.vectorize(lambda c: oracle.e4m3_value(int(c), L))(codes).reshape(5, 4, 128) * scale[:, :, None]
    g = v.reshape(5, 4, 128)
    assert np.all(np.abs(np.abs(dec).max(axis=2) - np.abs(g).max(axis=2)) <= 1e-12 * np.abs(g).max(axis=2))
    step = np.exp2(np.floor(np.log2(np.maximum(np.abs(g / scale[:, :, None]), 2.0 ** -6))) - 3) * scale[:, :, None]
    assert np.all(np.abs(dec - g) <= 0.5 * step * (1 + 1e-12))


# ---------------------------------------------------------------------------
# DCP: the per-rank steps of decode context parallelism ([vLLM-ML4] Long
# context: decode and prefill context parallelism)
def _owner(t, world, interleave):
    """Ownership restated here: turns of `interleave` tokens go round the ranks."""
    return (t // interleave) % world


def pin_dcp_ownership_partitions_tokens(L):
    """Every token has one owner; each rank numbers the tokens it owns 0, 1, 2,
    ... in token order; global(local(t)) = t.  Hand case: two ranks, turns of
    three: tokens 0-2 and 6-8 on rank 0 (local 0-5), 3-5 on rank 1 (local 0-2)."""
    assert [oracle.dcp_owner(t, 2, 3, L=L) for t in range(9)] == [0, 0, 0, 1, 1, 1, 0, 0, 0]
    assert [oracle.dcp_local(t, 2, 3, L=L) for t in range(9)] == [0, 1, 2, 0, 1, 2, 3, 4, 5]
    for world, inter in ((1, 1), (4, 1), (3, 64), (8, 16), (5, 7), (2, 1000)):
        seen = [0] * world
        for t in range(1200):
            r = oracle.dcp_owner(t, world, inter, L=L)
            assert r == _owner(t, world, inter)
            loc = oracle.dcp_local(t, world, inter, L=L)
            assert loc == seen[r], (world, inter, t)
            seen[r] += 1
            assert oracle.dcp_global(loc, r, world, inter, L=L) == t


_SPECIAL = [0.0, -0.0, 1.0, -1.0, 0.5, -0.5, 2.0, 1.0000001, float("inf"), float("-inf"), 1e-45, -1e-45,
            1.1754942e-38, 3.4028235e38, -3.4028235e38, 7.25, -7.25]


def pin_dcp_pack_orders_like_score_then_id(L):
    """Packed candidates sorted as unsigned 64-bit integers (descending) come in
    the order of Python's own sort by (score descending, id ascending), -0 equal
    to +0, over infinities, subnormals, the extremes and ties; every candidate
    unpacks to its (score, id) and none packs to the empty value 0."""
    ids = [0, 1, 2, 5, 12345, 2 ** 31 - 1]
    cand = [(float(np.float32(v)), i) for v in _SPECIAL for i in ids]
    packed = [int(oracle.dcp_pack(np.float32([sc]), [i], L=L)[0]) for sc, i in cand]
    assert all(p != 0 for p in packed)
    by_packed = sorted(range(len(cand)), key=lambda j: -packed[j])
    by_ref = sorted(range(len(cand)), key=lambda j: (-(cand[j][0] + 0.0), cand[j][1]))
    assert [cand[j][0] + 0.0 for j in by_packed] == [cand[j][0] + 0.0 for j in by_ref]
    assert [cand[j][1] for j in by_packed] == [cand[j][1] for j in by_ref]
    for (sc, i), p in zip(cand, packed):
        got = oracle.dcp_unpack(p, L=L)
        assert got is not None and got[1] == i and got[0] == sc + 0.0 and math.copysign(1, got[0]) == \
            math.copysign(1, sc + 0.0)
    assert oracle.dcp_unpack(0, L=L) is None


def _shard_lists(L, s, k, world, inter):
    """Each rank's candidates: the pinned top-k of the scores it owns, ids global."""
    n = len(s)
    lists = np.zeros((world, 1, k), np.uint64)
    for r in range(world):
        owned = [t for t in range(n) if _owner(t, world, inter) == r]
        if not owned:
            continue
        ls = s[owned]
        li, lm = oracle.topk(ls, k, L=L)
        glob = [owned[j] for j in li[:lm]]
        lists[r, 0, :lm] = oracle.dcp_pack(ls[li[:lm]].astype(np.float32), glob, L=L)
    return lists


def pin_topk_merge_of_shards_is_global_topk(L):
    """The DCP identity: a row's global top-k lies within the union of its
    shards' local top-ks, so merging the shards' candidates gives exactly the
    global top-k of the pinned oracle.topk (ids ascending, then -1), for
    several world sizes, interleaves and k, on scores with many ties."""
    rng = np.random.default_rng(41)
    for n, k, world, inter in ((1000, 64, 4, 1), (1000, 64, 3, 64), (777, 100, 8, 16), (50, 64, 4, 8),
                               (4096, 2048, 2, 64), (300, 7, 5, 300), (9, 4, 16, 1)):
        s = rng.integers(-20, 21, n).astype(np.float64) * 0.25  # exact in fp32, many ties
        gi, gm = oracle.topk(s, k, L=L)
        ids, lens = oracle.topk_merge(_shard_lists(L, s, k, world, inter), k, L=L)
        assert lens[0] == gm
        assert np.array_equal(ids[0, :gm], np.sort(gi[:gm]))
        assert np.all(ids[0, gm:] == -1)


def pin_topk_merge_library(L):
    """The selector against numpy's lexsort on lists of distinct random ids with
    tied scores and empty slots; fewer candidates than k: all of them."""
    rng = np.random.default_rng(42)
    for R, n, k in ((4, 16, 8), (3, 50, 64), (8, 32, 32), (1, 10, 3), (2, 5, 0)):
        ids_all = rng.permutation(10 ** 6)[:R * n].astype(np.int64)
        sc = (rng.integers(-6, 7, R * n) * 0.5).astype(np.float32)
        keep = rng.random(R * n) < 0.8
        lists = np.where(keep, oracle.dcp_pack(sc, ids_all, L=L), 0).astype(np.uint64).reshape(R, 1, n)
        got, lens = oracle.topk_merge(lists, k, L=L)
        cs, ci = sc[keep].astype(np.float64), ids_all[keep]
        order = np.lexsort((ci, -cs))[:k]
        m = min(k, int(keep.sum()))
        assert lens[0] == m
        assert np.array_equal(got[0, :m], np.sort(ci[order]).astype(np.int32))
        assert np.all(got[0, m:] == -1)


def pin_topk_merge_refuses_duplicate_ids(L):
    """An id offered by two lists cannot come from disjoint shards: refused."""
    lists = np.zeros((2, 1, 4), np.uint64)
    lists[0, 0, 0] = oracle.dcp_pack(np.float32([1.0]), [7], L=L)[0]
    lists[1, 0, 0] = oracle.dcp_pack(np.float32([2.0]), [7], L=L)[0]
    try:
        oracle.topk_merge(lists, 4, L=L)
    except ValueError:
        return
    raise AssertionError("a duplicate id was accepted")


def pin_topk_compact_partitions_selection(L):
    """Over the ranks, the compacted local slots mapped back by the ownership
    rule are exactly the selection's valid slots, each on the rank that owns it
    and in the selection's order; the lengths add up; slots past topk_len and
    -1 slots are ignored; the rest of each row is -1."""
    rng = np.random.default_rng(43)
    k = 64
    for world, inter in ((4, 1), (3, 64), (8, 16), (1, 1)):
        sel = rng.permutation(5000)[:50].astype(np.int32)
        idx = np.full((1, k), -1, np.int32)
        idx[0, :50] = sel
        idx[0, 7] = -1          # a hole inside the valid range
        idx[0, 55] = 4321       # past topk_len: ignored
        valid = [int(t) for t in idx[0, :50] if t >= 0]
        total = 0
        for r in range(world):
            li, ll = oracle.topk_compact(idx, np.array([50], np.int32), r, world, inter, L=L)
            mine = [t for t in valid if _owner(t, world, inter) == r]
            assert ll[0] == len(mine)
            back = [oracle.dcp_global(int(x), r, world, inter, L=L) for x in li[0, :ll[0]]]
            assert back == mine
            assert np.all(li[0, ll[0]:] == -1)
            total += int(ll[0])
        assert total == len(valid)


def pin_lse_combine_of_split_attention(L):
    """Attention over a selection equals the LSE combine of the attentions over
    disjoint parts of it (each by the pinned oracle.sparse_mla), an empty part
    (out 0, lse -inf) included; in parts of 1, 2 and 5."""
    q, lat, lay = mla_case(n=40, seed=44)
    sel = np.random.default_rng(44).permutation(40)[:29].astype(np.int32)
    ref_o, ref_l, _ = oracle.sparse_mla(q, lat, lay, 0, sel, 29, 0.07, L=L)
    for parts in (1, 2, 5):
        chunks = np.array_split(sel, parts) + [np.zeros(0, np.int32)]
        os_, ls_ = [], []
        for c in chunks:
            o, l, _ = oracle.sparse_mla(q, lat, lay, 0, np.ascontiguousarray(c), len(c), 0.07, L=L)
            os_.append(o)
            ls_.append(l)
        out, lse = oracle.lse_combine(np.stack(os_), np.stack(ls_), L=L)
        close(out, ref_o, 1e-12)
        close(lse, ref_l, 1e-12)


def pin_lse_combine_closed_forms(L):
    """Two parts: lse = logaddexp(a, b) (numpy), out = e^(a-lse) x + e^(b-lse) y;
    one part: itself; every part at -inf: out 0, lse -inf."""
    rng = np.random.default_rng(45)
    a, b = rng.standard_normal(6) * 3, rng.standard_normal(6) * 3
    x, y = rng.standard_normal((6, 5)), rng.standard_normal((6, 5))
    out, lse = oracle.lse_combine(np.stack([x, y]), np.stack([a, b]), L=L)
    ref = np.logaddexp(a, b)
    close(lse, ref)
    close(out, np.exp(a - ref)[:, None] * x + np.exp(b - ref)[:, None] * y)
    out, lse = oracle.lse_combine(x[None], a[None], L=L)
    close(out, x)
    close(lse, a)
    ninf = np.full((3, 6), -np.inf)
    out, lse = oracle.lse_combine(np.zeros((3, 6, 5)), ninf, L=L)
    assert np.all(out == 0) and np.all(lse == -np.inf)


# ---------------------------------------------------------------------------
# NVFP4 ("vLLM adds NVFP4 serving for MiniMax M3.1 Flash": 4.5-bit cache values)
# The E2M1 element values, written out: magnitudes of codes 0..7.
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _nearest_e2m1(x):
    """Brute force on the table: nearest magnitude, a tie to the even code."""
    a = abs(x)
    d = [abs(a - t) for t in E2M1_TABLE]
    best = [i for i in range(8) if d[i] == min(d)]
    c = best[0] if len(best) == 1 else next(i for i in best if i % 2 == 0)
    return (8 if math.copysign(1.0, x) < 0 else 0) | c


def pin_e2m1_table(L):
    """The 16 E2M1 codes decode to the format's table, the sign bit negating."""
    for c in range(16):
        v = oracle.e2m1_value(c, L=L)
        want = E2M1_TABLE[c & 7] * (-1.0 if c & 8 else 1.0)
        assert v == want and math.copysign(1.0, v) == math.copysign(1.0, want), (c, v)


def pin_e2m1_encode_nearest(L):
    """Encoding is the nearest table value (ties to the even code, 6 past the
    top, sign kept, zeros included) on a grid through every midpoint, and
    decoding then encoding returns every code."""
    grid = [i / 16.0 for i in range(-130, 131)] + [6.5, 7.0, 100.0, -9.0, 1e-300, -1e-300, 0.25, 0.75, 1.25,
                                                      1.75, 2.5, 3.5, 5.0, -5.0]
    for x in grid:
        assert oracle.e2m1_encode(x, L=L) == _nearest_e2m1(x), x
    for c in range(16):
        assert oracle.e2m1_encode(oracle.e2m1_value(c, L=L), L=L) == c


def pin_nvfp4_hand_block(L):
    """A block whose values sit on the grid: scale and codes by hand.  Max
    |v| = 12 with g = 1 gives the E4M3 block scale 2.0 (code 0x40), so each
    v / 2 is an exact E2M1 value; the even element goes to the low nibble
    (1.0 and -6.0 -> 0x2 | 0xF << 4)."""
    v = np.array([2.0, -12.0, 1.0, 3.0, 0.0, 8.0, -4.0, 6.0, 0.5 * 2, 1.5 * 2, -0.0, 2.0, 4.0, -1.0, 12.0, 0.0])
    codes, scales = oracle.nvfp4_quantize(v, 1.0, L=L)
    assert scales.tolist() == [0x40]
    assert codes[0] == 0xF2  # 2/2 = 1.0 -> 0x2 (low), -12/2 = -6.0 -> 0xF (high)
    assert codes[1] == 0x31  # 1/2 = 0.5 -> 0x1 (low), 3/2 = 1.5 -> 0x3 (high)
    back = oracle.nvfp4_dequantize(codes, scales, 1.0, L=L)
    assert np.array_equal(back, v)


def pin_nvfp4_quantize_properties(L):
    """Random blocks and tensor scales (powers of two and not): each block
    scale is the pinned E4M3 encoding of max|v| / (6 g); each code is the
    table's nearest value of v / (g s); dequantisation is g * s * value; a
    block of zeros has scale 0 and codes 0."""
    rng = np.random.default_rng(47)
    for g in (1.0, 0.25, 3.0e-3, 17.0):
        v = rng.standard_normal((5, 64)) * rng.choice([1e-3, 1.0, 50.0], size=(5, 1))
        v[2, 16:32] = 0.0
        codes, scales = oracle.nvfp4_quantize(v, g, L=L)
        back = oracle.nvfp4_dequantize(codes, scales, g, L=L)
        for r in range(5):
            for b in range(4):
                blk = v[r, 16 * b:16 * b + 16]
                sc = int(scales[r, b])
                assert sc == oracle.e4m3_encode(np.max(np.abs(blk)) / (6.0 * g), L=L)
                s_val = oracle.e4m3_value(sc, L=L)
                for i in range(16):
                    byte = int(codes[r, 8 * b + i // 2])
                    nib = (byte >> 4) if i % 2 else (byte & 15)
                    want = _nearest_e2m1(blk[i] / (g * s_val)) if s_val > 0 else 0
                    assert nib == want, (g, r, b, i)
                    assert back[r, 16 * b + i] == g * s_val * E2M1_TABLE[nib & 7] * (-1 if nib & 8 else 1)
        assert np.all(scales[2, 1] == 0) and np.all(codes[2, 8:16] == 0)


def pin_nvfp4_bits_per_value(L):
    """4-bit values plus their block scales cost 4.5 bits per value, the
    pages' figure, and 4.5 / 8 is the pages' FP8 -> NVFP4 byte ratio
    (tests/golden/nvfp4.json)."""
    with open(os.path.join(GOLDEN, "nvfp4.json")) as f:
        g = json.load(f)
    n = 4096
    codes, scales = oracle.nvfp4_quantize(np.ones(n), 1.0, L=L)
    bits = 8.0 * (codes.size + scales.size) / n
    assert bits == g["bits_per_value"]
    assert g["kv_bytes_per_token_fp8"] * bits / 8.0 == g["kv_bytes_per_token_nvfp4"]
    assert 100.0 * (1.0 - bits / 8.0) == g["reduction_percent"]
    # the NVFP4 cache rows: 128 index dims and 576 latent dims at 4.5 bits
    assert oracle.index_row_bytes(oracle.KEYS_NVFP4, L=L) * 8 == 128 * g["bits_per_value"]
    assert oracle.latent_row_bytes(oracle.LATENT_NVFP4, L=L) * 8 == 576 * g["bits_per_value"]


def _nvfp4_rows(rng, n, dims):
    """Random NVFP4 rows: any E2M1 codes, positive finite E4M3 block scales."""
    codes = rng.integers(0, 256, (n, dims // 2)).astype(np.uint8)
    scales = rng.integers(0, 0x7F, (n, dims // 16)).astype(np.uint8)  # 0x7F is NaN
    return codes, scales


def pin_nvfp4_keys_equal_their_values(L):
    """NVFP4 index keys (a power-of-two tensor scale) score like bf16 keys
    holding their decoded values: E2M1 x E4M3 has at most 6 significant bits,
    so the values are exact in bf16."""
    rng = np.random.default_rng(50)
    n, g = 19, 0.25
    codes, scales = _nvfp4_rows(rng, n, 128)
    vals = oracle.nvfp4_dequantize(codes, scales, g, L=L)
    assert np.array_equal(oracle.e2m1_value(int(codes[3, 5]) >> 4, L=L) * oracle.e4m3_value(int(scales[3, 0]), L=L)
                          * g, vals[3, 11])
    c = index_case(n=n, rope=True, seed=13)
    a = oracle.index_scores_nvfp4(c["q"], c["w"], c["ssmax_s"], c["ssmax_b"], c["inv_freq"], c["q_seq"], c["q_pos"],
                                  codes, scales, g, contiguous([n], n), L=L)
    b = scores_of(L, c, keys=bf16_bits(vals))
    close(a[0], b, 0.0)


def pin_mla_nvfp4_equals_values(L):
    """NVFP4 latent rows (all 576 dims) score and average like bf16 rows
    holding their decoded values."""
    rng = np.random.default_rng(51)
    n, g = 22, 0.5
    codes, scales = _nvfp4_rows(rng, n, 576)
    vals = oracle.nvfp4_dequantize(codes, scales, g, L=L)
    q = bf16_bits(rng.standard_normal((64, 576)) * 1e-3)
    lay = contiguous([n], n)
    idx = rng.permutation(n)[:13].astype(np.int32)
    a, la = oracle.sparse_mla_nvfp4(q, codes, scales, g, lay, 0, idx, 13, 0.1, L=L)
    b, lb, _ = oracle.sparse_mla(q, bf16_bits(vals), lay, 0, idx, 13, 0.1, L=L)
    close(a, b, 0.0)
    close(la, lb, 0.0)


# ---------------------------------------------------------------------------
# block-sparse selection (MiniMax Sparse Attention)
def pin_block_topk_closed_forms(L):
    """Scores rising with position select the 16 most recent blocks; falling
    scores select blocks 0..14 and the query's own block; a context of at most
    16 blocks is selected whole."""
    n = 5000  # 40 blocks, the last holding keys 4992..4999
    idx, m = oracle.block_topk(np.arange(n, dtype=np.float64), L=L)
    assert m == 15 * 128 + 8 and np.array_equal(idx[:m], np.arange(24 * 128, n)) and np.all(idx[m:] == -1)
    idx, m = oracle.block_topk(np.arange(n, dtype=np.float64)[::-1].copy(), L=L)
    assert np.array_equal(idx[:m], np.concatenate([np.arange(15 * 128), np.arange(4992, n)]))
    for n in (1, 127, 128, 129, 2047, 2048):
        idx, m = oracle.block_topk(np.random.default_rng(n).standard_normal(n), L=L)
        assert m == n and np.array_equal(idx[:m], np.arange(n))


def pin_block_topk_library(L):
    """Against numpy: block maxima (np.maximum.reduceat), blocks ordered by
    (max descending, block ascending) with numpy's lexsort, the query's block
    forced; many ties, ragged last blocks, other block sizes and counts."""
    rng = np.random.default_rng(48)
    for n, block, nsel in ((9000, 128, 16), (2049, 128, 16), (3000, 64, 5), (777, 7, 16), (40000, 128, 16),
                           (5, 2, 1), (300, 128, 2)):
        s = rng.integers(-8, 9, n).astype(np.float64) * 0.5
        idx, m = oracle.block_topk(s, block, nsel, L=L)
        starts = np.arange(0, n, block)
        bmax = np.maximum.reduceat(s, starts)
        nb, last = len(starts), len(starts) - 1
        order = [b for b in np.lexsort((np.arange(nb), -bmax)) if b != last][:nsel - 1]
        chosen = sorted(order + [last])
        want = np.concatenate([np.arange(b * block, min(n, (b + 1) * block)) for b in chosen])
        assert m == len(want) and np.array_equal(idx[:m], want), (n, block, nsel)
        assert np.all(idx[m:] == -1)


def pin_block_topk_block_one_is_topk(L):
    """With blocks of one key, nsel = k, and the query's own key scoring
    highest, the selection is the pinned top-k's (as a sorted set)."""
    rng = np.random.default_rng(49)
    for n, k in ((500, 64), (3000, 2048), (40, 64)):
        s = np.round(rng.standard_normal(n), 1)
        s[-1] = 100.0
        idx, m = oracle.block_topk(s, 1, k, L=L)
        ti, tm = oracle.topk(s, k, L=L)
        assert m == tm and np.array_equal(idx[:m], np.sort(ti[:tm]))


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
