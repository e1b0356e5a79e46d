"""The seeded input generator (dsa_sparse_mla_query_gb300/inputs.py), the one
module the CUDA path and the oracle share: counter-based streams (element i
of tensor T under seed s depends on (s, T, i) only), the distributions and
structures the workloads state, and the storage recipe of the generated fp8
data.  CPU only."""

from __future__ import annotations

import numpy as np
import torch

from dsa_sparse_mla_query_gb300 import inputs as I
import oracle


def test_splitmix64_first_output_of_seed_zero():
    """SplitMix64 seeded with 0 first returns its finaliser of the golden
    gamma: the published first output 0xE220A8397B1DCDAF."""
    assert I.mix64_int(0x9E3779B97F4A7C15) == 0xE220A8397B1DCDAF


def test_tensor_stream_matches_the_integer_form():
    """The int64 tensor form (arithmetic shifts masked to logical ones) gives
    the same 64-bit values as the Python-int form, large counters included."""
    key = I.stream_key(7, 3)
    counters = torch.tensor([0, 1, 2, 12345, 2 ** 31 + 5, 2 ** 40 + 17, 2 ** 62 + 3], dtype=torch.int64)
    got = I.bits(key, counters).numpy().view(np.uint64)
    want = np.array([I.bits_int(key, int(c)) for c in counters], dtype=np.uint64)
    assert np.array_equal(got, want)


def test_streams_depend_on_seed_tensor_and_counter_only():
    a = I.bits(I.stream_key(0, 5), I._counters(0, 1000, "cpu"))
    b = I.bits(I.stream_key(0, 5), I._counters(0, 1000, "cpu"))
    assert torch.equal(a, b)
    assert not torch.equal(a, I.bits(I.stream_key(0, 6), I._counters(0, 1000, "cpu")))
    assert not torch.equal(a, I.bits(I.stream_key(1, 5), I._counters(0, 1000, "cpu")))
    # a window of the stream is the same window of the whole
    assert torch.equal(I.bits(I.stream_key(0, 5), I._counters(400, 100, "cpu")), a[400:500])


def test_rows_do_not_depend_on_which_rows_are_generated():
    """Cache rows are a function of their physical row id: a scattered subset
    equals the same rows of the whole cache (the oracle regenerates only the
    rows it needs)."""
    key = I.stream_key(0, I.T_LATENT)
    full = I.gen_bf16_rows(key, torch.arange(300, dtype=torch.int64), 576, "cpu")
    pick = torch.tensor([299, 0, 37, 150, 151], dtype=torch.int64)
    part = I.gen_bf16_rows(key, pick, 576, "cpu")
    assert torch.equal(part, full[pick])
    codes, scale = I.gen_e4m3_rowscale_rows(I.stream_key(0, I.T_K_IDX), torch.arange(64, dtype=torch.int64), "cpu")
    c2, s2 = I.gen_e4m3_rowscale_rows(I.stream_key(0, I.T_K_IDX), torch.tensor([63, 5]), "cpu")
    assert torch.equal(c2, codes[[63, 5]]) and torch.equal(s2, scale[[63, 5]])


def test_distributions():
    """Uniforms in [0, 1) with mean 1/2 and variance 1/12; normals with mean 0
    and variance 1 (2^20 samples each, 5-sigma bounds)."""
    n = 1 << 20
    u = I.uniform(I.stream_key(3, 1), I._counters(0, n, "cpu")).numpy()
    assert u.min() >= 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 5 * np.sqrt(1 / 12 / n)
    assert abs(u.var() - 1 / 12) < 5 * np.sqrt(1 / 180 / n)
    z = I.normal(I.stream_key(3, 2), I._counters(0, n, "cpu")).numpy()
    assert abs(z.mean()) < 5 / np.sqrt(n)
    assert abs(z.var() - 1.0) < 5 * np.sqrt(2.0 / n)
    assert abs(np.mean(z ** 3)) < 5 * np.sqrt(15.0 / n)  # symmetric


def test_page_table_is_a_permutation_of_all_pages():
    wl = I.scaled(I.WORKLOADS["paged"], num_seqs=5, ctx=None, ctx_list=(1500, 64, 4163, 65, 3000))
    lay = I.make_layout(wl)
    pages = [(c + lay.page_size - 1) // lay.page_size for c in lay.ctx_len]
    used = torch.cat([lay.page_table[b, :pages[b]] for b in range(len(pages))])
    assert sorted(used.tolist()) == list(range(sum(pages)))
    assert lay.num_rows == sum(pages) * lay.page_size


def test_insert_rows_are_distinct():
    d = I.make_insert_inputs(1000, 2, 1500, "cpu", seed=3)
    sl = d["slot"]
    assert len(set(sl.tolist())) == 1000 and int(sl.min()) >= 0 and int(sl.max()) < 1500
    d = I.make_insert_inputs(640, 1, 1024, "cpu", seed=3, page_size=64)
    sl = d["slot"].view(10, 64)
    assert torch.equal(sl - sl[:, :1], torch.arange(64).expand(10, 64))  # a page's tokens are contiguous
    assert torch.all(sl[:, 0] % 64 == 0) and len(set(sl[:, 0].tolist())) == 10


def test_generated_fp8_follows_the_recipe():
    """The generator's e4m3 groups (scale amax / 448, codes rounded to nearest
    even) agree with the oracle's quantiser, except where the fp32 and fp64
    divisions straddle a rounding midpoint."""
    v = I.normal(I.stream_key(4, 9), I._counters(0, 64 * 512, "cpu")).to(torch.float32).view(64, 512)
    codes, scale = I.quantize_e4m3_groups(v, 128)
    oc, os_ = oracle.quantize_rows_e4m3(v.double().numpy(), 128)
    assert np.allclose(scale.double().numpy(), os_, rtol=1e-6, atol=0)
    assert (codes.numpy() == oc).mean() > 0.999


def test_nvfp4_encoding_matches_the_oracles_encoder():
    """The NVFP4 storage encoding that both sides read is byte for byte the
    oracle's own encoder ("vLLM adds NVFP4 serving for MiniMax M3.1 Flash":
    E2M1 codes, one E4M3 scale per 16 values, one tensor scale): on bf16
    N(0,1) rows, on the E2M1 ties and past 6, and on an all-zero block."""
    g = 2.0 ** -9  # a power of two, so that the ties below stay exact ties
    x = I.gen_bf16_rows(I.stream_key(5, I.T_K_IDX), torch.arange(300), 128, "cpu").to(torch.float64) * (g / I.NVFP4_GLOBAL)
    # one block at scale 1.5 (its largest value 6 x 1.5 g) holding every E2M1
    # tie, and one whose scale saturates at 448 so that values pass 6
    ties = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -2.5, -5.0, 6.0, -0.75, 0.0, 4.9, 1.0, 3.0])
    x[0, :16] = ties * g * 1.5
    x[2, :16] = torch.linspace(-4000.0, 5000.0, 16, dtype=torch.float64) * g
    x[1, 16:32] = 0.0
    codes, scales = I.quantize_nvfp4(x, g)
    oc, os_ = oracle.nvfp4_quantize(x.numpy(), g)
    assert np.array_equal(scales.numpy(), os_)
    assert np.array_equal(codes.numpy(), oc)
    assert scales[0, 0] == 0x3C and scales[2, 0] == 0x7E  # 1.5, 448
    assert scales[1, 1] == 0 and np.all(codes[1, 8:16].numpy() == 0)
    lo, hi = codes[0, :8] & 15, codes[0, :8] >> 4
    assert [int(v) for v in torch.stack([lo, hi], 1).reshape(-1)] == [0, 2, 2, 4, 4, 6, 6, 8, 12, 14, 7, 10, 0, 6, 2, 5]
    assert int(codes[2, 7] >> 4) == 7 and int(codes[2, 0] & 15) == 15


def test_generated_nvfp4_follows_the_recipe():
    wl = I.scaled(I.WORKLOADS["long_nvfp4"], num_seqs=2, ctx=300)
    d = I.make_inputs(wl, "cpu")
    assert d["k_idx"].shape == (600, 64) and d["k_bscale"].shape == (600, 8)
    assert d["latent"].shape == (600, 288) and d["lat_bscale"].shape == (600, 36)
    assert d["k_global"] == d["lat_global"] == I.NVFP4_GLOBAL
    ref = I.gen_bf16_rows(I.stream_key(wl.seed, I.T_K_IDX), torch.arange(600), 128, "cpu")
    back = oracle.nvfp4_dequantize(d["k_idx"].numpy(), d["k_bscale"].numpy(), I.NVFP4_GLOBAL)
    # E2M1 rounds to within half its widest step (2, between 4 and 6) of g s,
    # and s = amax / (6 g) rounds to E4M3 within 1/16
    err = np.abs(back - ref.double().numpy()).reshape(600, 8, 16).max(-1)
    amax = np.abs(ref.double().numpy()).reshape(600, 8, 16).max(-1)
    assert np.all(err <= amax / 6.0 * (1 + 1 / 16) + 1e-12)
