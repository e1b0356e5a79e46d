"""sparse_mla_decode_noalloc: the attention entry point for callers that cannot
allocate device memory (their GPU memory belongs to another allocator, so they
cannot pass a workspace).  Its split-K partials live in a static device array
inside the library.  Checked through the C ABI against sparse_mla_decode (the
workspace entry point) on two calls in a row, within the tolerances of the
other parity tests, and on sampled queries against the oracle.  Collected
last on purpose."""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import dsa_sparse_mla_query_gb300 as dsa
from dsa_sparse_mla_query_gb300 import _binding as B
from dsa_sparse_mla_query_gb300 import inputs as I
from dsa_sparse_mla_query_gb300.runner import seqs_from_inputs
import parity as P


def _case(wl):
    d = P.to_device(I.make_inputs(wl, "cpu"), "cuda")
    seqs = seqs_from_inputs(d, wl.queries_per_seq)
    lay = d["layout"]
    k = wl.topk
    g = torch.Generator().manual_seed(5)
    idx = torch.full((wl.num_queries, k), -1, dtype=torch.int32)
    tlen = torch.empty(wl.num_queries, dtype=torch.int32)
    for t in range(wl.num_queries):
        n = min(k, lay.q_pos[t] + 1)
        sel = torch.randperm(lay.q_pos[t] + 1, generator=g)[:n].to(torch.int32)
        idx[t, :n] = sel
        tlen[t] = n - (t % 3)       # some rows shorter than their selection
    return d, seqs, idx.cuda(), tlen.cuda()


CASES = {
    # a few queries: many splits per query, partials in the static array
    "paged6": ("paged", False, (3000, 2049, 700, 5000, 4100, 2048)),
    "fp8_6": ("long_fp8", True, (3000, 2049, 700, 5000, 4100, 2048)),
    # 64 queries: the batched-decode batch size (its own split policy)
    "paged64": ("paged", False, tuple(2100 + 37 * i for i in range(64))),
}


@pytest.mark.gpu
@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_matches_workspace_entry_point(case):
    name, fp8, ctx = CASES[case]
    wl = I.scaled(I.WORKLOADS[name], num_seqs=len(ctx), ctx=None, ctx_list=ctx)
    d, seqs, idx, tlen = _case(wl)
    Q, k = wl.num_queries, wl.topk
    dt = dsa.DSA_FP8_DS_MLA if fp8 else dsa.DSA_BF16
    assert B.load().sparse_mla_decode_noalloc is not None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws_bytes = dsa.dsa_workspace_size(seqs, Q, k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.empty(Q, 64, 512, dtype=torch.bfloat16, device="cuda")
    ref_lse = torch.empty(Q, 64, dtype=torch.float32, device="cuda")
    dsa.sparse_mla_decode(d["q_mla"], d["latent"], dt, seqs, Q, idx, tlen, k, d["sm_scale"], ref, ref_lse, ws,
                          ws_bytes, status)
    torch.cuda.synchronize()
    r_out, r_lse = ref.float().cpu().numpy(), ref_lse.cpu().numpy()
    for call in range(2):
        out = torch.full((Q, 64, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((Q, 64), float("nan"), dtype=torch.float32, device="cuda")
        dsa.sparse_mla_decode_noalloc(d["q_mla"], d["latent"], dt, seqs, Q, idx, tlen, k, d["sm_scale"], out, lse,
                                      status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        o, l = out.float().cpu().numpy(), lse.cpu().numpy()
        for t in range(Q):
            P.check_mla(o[t], l[t], r_out[t].astype(np.float64), r_lse[t].astype(np.float64))
    # and against the oracle on sampled queries (the selection as passed)
    idx_h, len_h = idx.cpu().numpy(), tlen.cpu().numpy()
    for t in P.sample_queries(Q, 3):
        sel = idx_h[t, :len_h[t]]
        ro, rl = P.oracle_mla_for_query(d, t, sel[sel >= 0])
        P.check_mla(o[t], l[t], ro, rl)


@pytest.mark.parametrize("num_q", [1, 10, 64, 4096, 20000])
def test_noalloc_batch_sizes(num_q):
    """Where the splits' partials would not fit the static array (10 queries
    take 15 splits in sparse_mla_decode: 10 x 15 x 131,584 bytes > 16 MiB),
    the call takes fewer splits, so no batch size is refused (host check
    only: the pointers are fake, so without a GPU an accepted call stops at
    the device query with DSA_ERR_CUDA)."""
    lib = B.load() if B._lib is not None else None
    if lib is None:
        from dsa_sparse_mla_query_gb300 import build
        build.build()
        lib = B.load()
    if torch.cuda.is_available():
        pytest.skip("host-only check: with a GPU the fake pointers would be launched")
    s = B.DsaSeqsC(num_seqs=num_q, max_ctx=4096, max_q_per_seq=1, page_size=0, max_pages=0, reserved=0,
                   num_rows=num_q * 4096, ctx_len=0x1000, q_start=0x2000, q_pos=0x3000, page_table=None,
                   seq_base=0x4000)
    rc = lib.sparse_mla_decode_noalloc(0x100, 0x100, 0, ctypes.byref(s), num_q, 0x100, 0x100, 2048,
                                       ctypes.c_float(0.07), 0x100, None, None, None)
    assert rc == B.DSA_ERR_CUDA, (rc, lib.dsa_last_error_string().decode())
