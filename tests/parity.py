"""Parity checks of the CUDA path against the CPU oracle.

Tolerances (written here, used by every GPU test):
  * indexer scores: |gpu - oracle| <= 1e-2 * max_j |oracle(t, j)| over the
    causal keys of the row; the -inf pattern after the position matches exactly;
  * top-k: same count, positions ascending and unique, -1 after; the set
    equals the oracle's except keys whose oracle score lies within 1e-3
    (relative) of the k-th largest oracle score -- several sets are correct
    when scores tie at the boundary;
  * attention: max |out_gpu - out_oracle| <= 1e-2 * max |out_oracle| (fp8
    caches: the oracle runs on the dequantised values, which is what it reads);
    LSE within 1e-3 absolute, -inf where the selection is empty.
"""

from __future__ import annotations

import math
from typing import Dict, List

import numpy as np
import torch

import oracle
from dsa_sparse_mla_query_gb300 import inputs as I

SCORE_RTOL = 1e-2
TIE_RTOL = 1e-3
OUT_RTOL = 1e-2
LSE_ATOL = 1e-3


def check_scores(gpu_row: np.ndarray, ref_row: np.ndarray, pos: int, ctx: int) -> float:
    g = np.asarray(gpu_row[:ctx], np.float64)
    r = np.asarray(ref_row[:ctx], np.float64)
    assert np.all(np.isneginf(g[pos + 1:])), "keys after the position must be -inf"
    assert np.all(np.isfinite(g[:pos + 1])), "causal scores must be finite"
    scale = max(float(np.max(np.abs(r[:pos + 1]))), 1e-30)
    err = float(np.max(np.abs(g[:pos + 1] - r[:pos + 1])))
    assert err <= SCORE_RTOL * scale, f"score error {err:.3e} > {SCORE_RTOL} * {scale:.3e}"
    return err / scale


def check_topk(gpu_idx: np.ndarray, gpu_len: int, ref_causal: np.ndarray, k: int) -> int:
    """Returns the number of exempt boundary keys on which the sets differ."""
    n = ref_causal.shape[0]
    m = min(k, n)
    assert gpu_len == m, f"topk_len {gpu_len} != {m}"
    sel = np.asarray(gpu_idx[:m], np.int64)
    assert np.all(np.asarray(gpu_idx[m:]) == -1), "slots after topk_len must be -1"
    assert np.all(np.diff(sel) > 0), "selected positions must be ascending and unique"
    assert m == 0 or (sel[0] >= 0 and sel[-1] < n), "selected position outside the causal range"
    ref_idx, ref_m = oracle.topk(ref_causal, k)
    assert ref_m == m
    diff = set(sel.tolist()) ^ set(ref_idx[:m].tolist())
    if diff:
        kth = ref_causal[ref_idx[m - 1]]
        bad = [j for j in diff if abs(ref_causal[j] - kth) > TIE_RTOL * abs(kth)]
        assert not bad, f"{len(bad)} keys differ outside the tie band, e.g. {bad[:5]}"
    return len(diff)


def check_block_select(gpu_idx: np.ndarray, gpu_len: int, ref_causal: np.ndarray, block: int, nsel: int) -> int:
    """Block-sparse selection against the oracle's on the oracle's scores:
    the output is the selected blocks' causal keys ascending, then -1; the
    query's own block is always in; the other chosen blocks equal the
    oracle's except blocks whose oracle maximum lies within 1e-3 (relative)
    of the last chosen block's maximum.  Returns the number of such blocks."""
    n = ref_causal.shape[0]
    k = nsel * block
    sel = np.asarray(gpu_idx[:gpu_len], np.int64)
    assert np.all(np.asarray(gpu_idx[gpu_len:k]) == -1), "slots after topk_len must be -1"
    assert np.all(np.diff(sel) > 0) and (gpu_len == 0 or (sel[0] >= 0 and sel[-1] < n))
    blocks = np.unique(sel // block)
    # whole blocks (the own block up to the query)
    for b in blocks:
        want = np.arange(b * block, min(n, (b + 1) * block))
        assert np.array_equal(sel[(sel >= b * block) & (sel < (b + 1) * block)], want), f"block {b} not whole"
    nb = (n + block - 1) // block
    assert nb - 1 in blocks, "the query's own block must be selected"
    assert len(blocks) == min(nsel, nb)
    ref_idx, ref_m = oracle.block_topk(ref_causal, block, nsel)
    ref_blocks = np.unique(ref_idx[:ref_m] // block)
    diff = set(blocks.tolist()) ^ set(ref_blocks.tolist())
    if diff:
        bmax = np.array([np.max(ref_causal[b * block:min(n, (b + 1) * block)]) for b in range(nb)])
        last = min(bmax[b] for b in ref_blocks if b != nb - 1)
        bad = [b for b in diff if abs(bmax[b] - last) > TIE_RTOL * abs(last)]
        assert not bad, f"blocks {bad[:5]} differ outside the tie band"
    return len(diff)


def check_mla(out_gpu, lse_gpu, out_ref: np.ndarray, lse_ref: np.ndarray) -> float:
    o = np.asarray(out_gpu, np.float64)
    scale = float(np.max(np.abs(out_ref)))
    err = float(np.max(np.abs(o - out_ref)))
    if scale == 0.0:
        assert err == 0.0, f"empty selection must give zeros, max {err}"
    else:
        assert err <= OUT_RTOL * scale, f"attention error {err:.3e} > {OUT_RTOL} * {scale:.3e}"
    if lse_gpu is not None:
        lg = np.asarray(lse_gpu, np.float64)
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lg), fin), "LSE finite pattern differs"
        assert np.all(np.isneginf(lg[~fin]))
        if fin.any():
            le = float(np.max(np.abs(lg[fin] - lse_ref[fin])))
            assert le <= LSE_ATOL, f"LSE error {le:.3e}"
    return err / scale if scale else 0.0


# ---------------------------------------------------------------------------
# host views of a sequence for the oracle (inputs only; nothing from the kernels)
def seq_rows_host(d: Dict, b: int) -> torch.Tensor:
    return d["layout"].phys_rows(b)


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy()


def oracle_scores_for_query(d: Dict, t: int) -> np.ndarray:
    """fp64 oracle scores of query row t over its sequence (length ctx)."""
    lay = d["layout"]
    b = lay.q_seq[t]
    ctx = lay.ctx_len[b]
    rows = seq_rows_host(d, b).to(d["k_idx"].device)
    keys = d["k_idx"].index_select(0, rows)
    ks = d["k_scale"].index_select(0, rows) if "k_scale" in d else None
    olay = oracle.Layout(np.array([ctx], np.int32), ctx, seq_base=np.zeros(1, np.int64))
    if "k_bscale" in d:  # NVFP4 keys
        return oracle.index_scores_nvfp4(d["q_idx"][t:t + 1], d["w"][t:t + 1], d["ssmax_s"], d["ssmax_b"],
                                         d["inv_freq"], np.zeros(1, np.int32), np.array([lay.q_pos[t]], np.int32),
                                         keys, d["k_bscale"].index_select(0, rows), d["k_global"], olay)[0]
    return oracle.index_scores(d["q_idx"][t:t + 1], d["w"][t:t + 1], d["ssmax_s"], d["ssmax_b"], d["inv_freq"],
                               np.zeros(1, np.int32), np.array([lay.q_pos[t]], np.int32), keys, olay,
                               key_scale=ks)[0]


def oracle_mla_for_query(d: Dict, t: int, sel: np.ndarray, shared: bool = False):
    """Oracle attention of query t over logical positions ``sel``."""
    lay = d["layout"]
    b = lay.q_seq[t]
    rows = seq_rows_host(d, b)[torch.from_numpy(np.asarray(sel, np.int64))].to(d["latent"].device)
    lat = (d["latent2"] if shared else d["latent"]).index_select(0, rows)
    q = d["q_mla2" if shared else "q_mla"][t]
    n = len(sel)
    olay = oracle.Layout(np.array([max(n, 1)], np.int32), max(n, 1), seq_base=np.zeros(1, np.int64))
    if "lat_bscale" in d and not shared:  # NVFP4 latent rows
        return oracle.sparse_mla_nvfp4(q, lat, d["lat_bscale"].index_select(0, rows), d["lat_global"], olay, 0,
                                       np.arange(n, dtype=np.int32), n, d["sm_scale"])
    out, lse, _ = oracle.sparse_mla(q, lat, olay, 0, np.arange(n, dtype=np.int32), n, d["sm_scale"],
                                    fp8=lat.dtype == torch.uint8)
    return out, lse


def sample_queries(num_q: int, n: int) -> List[int]:
    if num_q <= n:
        return list(range(num_q))
    return sorted(set([0, num_q - 1] + [int(round(x)) for x in np.linspace(0, num_q - 1, n)]))


def to_device(d: Dict, device) -> Dict:
    out = {}
    for k, v in d.items():
        out[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    return out


def ld_of(max_ctx: int) -> int:
    return (max_ctx + 3) // 4 * 4
