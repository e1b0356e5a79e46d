"""Decode context parallelism across processes ("Day 0 support for Mistral
Large 4", Long context: DCP): two processes on the one GPU each own one shard
of the paged caches (turns of one 64-token page), build their view of the
sequences with dsa_dcp_shard_seqs, score their keys and offer their local
top-k as packed candidates, exchange the candidate lists through
torch.distributed (gloo: host copies, no peer loads), merge them into the
exact global top-k, compact the slots they own, attend over their shard,
exchange the partial (out, lse) and LSE-combine them.  Rank 0 checks the
merged selection against the oracle's top-k of the unsharded scores and the
combined attention against the oracle over that selection.  No kernel of one
process waits on the other's: the exchange is on the host between launches.
"""

from __future__ import annotations

import datetime
import os
import socket
import sys
import traceback

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
WORLD = 2


def _free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    for p in (ROOT, HERE):
        if p not in sys.path:
            sys.path.insert(0, p)
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        import torch.distributed as dist
        dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=180))
        import dsa_sparse_mla_query_gb300 as dsa
        from dsa_sparse_mla_query_gb300 import inputs as I
        from dsa_sparse_mla_query_gb300.runner import seqs_from_inputs
        import parity as P

        torch.cuda.set_device(0)
        dev = torch.device("cuda", 0)
        dsa.load()
        wl = I.scaled(I.WORKLOADS["paged"], num_seqs=3, ctx=None, ctx_list=(1500, 4163, 2100))
        d = P.to_device(I.make_inputs(wl, "cpu"), dev)
        lay = d["layout"]
        full = seqs_from_inputs(d, wl.queries_per_seq)
        Q, k = wl.num_queries, wl.topk
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        shard = dsa.DcpShard(world, rank, lay.page_size)  # turns of one page
        # this rank's view: local lengths, causal bounds and page table
        lmaxp = lay.max_pages // world + 1
        lctx = torch.empty(len(lay.ctx_len), dtype=torch.int32, device=dev)
        lpos = torch.empty(Q, dtype=torch.int32, device=dev)
        ltab = torch.empty(len(lay.ctx_len), lmaxp, dtype=torch.int32, device=dev)
        lmax = dsa.dsa_dcp_shard_seqs(full, Q, shard, lctx, lpos, ltab, lmaxp, st)
        seqs = dsa.Seqs(lctx, d["q_start"], lpos, max_ctx=lmax, max_q_per_seq=wl.queries_per_seq,
                        num_rows=lay.num_rows, page_table=ltab, page_size=lay.page_size, q_rope_pos=d["q_pos"])
        ws_bytes = dsa.dsa_workspace_size(seqs, Q, k)
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
        ld = (lmax + 3) // 4 * 4
        scores = torch.empty(Q, ld, dtype=torch.float32, device=dev)
        idx = torch.empty(Q, k, dtype=torch.int32, device=dev)
        tlen = torch.empty(Q, dtype=torch.int32, device=dev)
        cand = torch.empty(Q, k, dtype=torch.int64, device=dev)
        dsa.dsa_index_scores(d["q_idx"], d["w"], d["ssmax_s"], d["ssmax_b"], d["inv_freq"], d["k_idx"], None,
                             dsa.DSA_BF16, seqs, Q, scores, ld, ws, ws_bytes, st)
        dsa.dsa_topk_candidates(scores, ld, seqs, Q, k, shard, idx, tlen, cand, ws, ws_bytes, st)
        torch.cuda.synchronize()
        # exchange 1: every rank's candidate list (host copies through gloo)
        lists = [torch.empty(Q, k, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(lists, cand.cpu())
        lists_d = [x.to(dev) for x in lists]
        gidx = torch.empty(Q, k, dtype=torch.int32, device=dev)
        glen = torch.empty(Q, dtype=torch.int32, device=dev)
        dsa.dsa_topk_merge(lists_d, k, Q, k, gidx, glen, st)
        lidx = torch.empty(Q, k, dtype=torch.int32, device=dev)
        llen = torch.empty(Q, dtype=torch.int32, device=dev)
        dsa.dsa_topk_compact(gidx, glen, Q, k, shard, lidx, llen, st)
        out = torch.empty(Q, 64, 512, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(Q, 64, dtype=torch.float32, device=dev)
        dsa.sparse_mla_decode(d["q_mla"], d["latent"], dsa.DSA_BF16, seqs, Q, lidx, llen, k, d["sm_scale"], out, lse,
                              ws, ws_bytes, st)
        torch.cuda.synchronize()
        # exchange 2: the partial outputs and their LSE
        outs = [torch.empty(Q, 64, 512, dtype=torch.bfloat16) for _ in range(world)]
        lses = [torch.empty(Q, 64, dtype=torch.float32) for _ in range(world)]
        dist.all_gather(outs, out.cpu())
        dist.all_gather(lses, lse.cpu())
        fout = torch.empty(Q, 64, 512, dtype=torch.bfloat16, device=dev)
        flse = torch.empty(Q, 64, dtype=torch.float32, device=dev)
        dsa.dsa_lse_combine([x.to(dev) for x in outs], [x.to(dev) for x in lses], Q, fout, flse)
        torch.cuda.synchronize()
        status = int(st.item())
        assert status == 0, f"rank {rank}: device status {status}"
        # the view the library built, against the ownership rule written out
        lc, lp = lctx.cpu().numpy(), lpos.cpu().numpy()
        for b, c in enumerate(lay.ctx_len):
            t = np.arange(c)
            mine = (t // lay.page_size) % world == rank
            assert lc[b] == mine.sum()
            for qi in range(lay.q_start[b], lay.q_start[b + 1]):
                assert lp[qi] == np.cumsum(mine)[lay.q_pos[qi]] - 1
        if rank == 0:
            gi, gl = gidx.cpu().numpy(), glen.cpu().numpy()
            o, l = fout.float().cpu().numpy(), flse.cpu().numpy()
            for t in range(Q):
                ref = P.oracle_scores_for_query(d, t)
                pos = lay.q_pos[t]
                P.check_topk(gi[t], int(gl[t]), ref[:pos + 1], k)
                ro, rl = P.oracle_mla_for_query(d, t, gi[t, :gl[t]])
                P.check_mla(o[t], l[t], ro, rl)
        dist.barrier()
        dist.destroy_process_group()
        with open(os.path.join(out_dir, f"rank{rank}.ok"), "w") as f:
            f.write("ok")
    except Exception:
        with open(os.path.join(out_dir, f"rank{rank}.err"), "w") as f:
            f.write(traceback.format_exc())
        raise


def test_dcp_two_processes_one_shard_each(tmp_path):
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import torch.multiprocessing as mp
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, WORLD, port, str(tmp_path))) for r in range(WORLD)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=600)
    for p in procs:
        if p.is_alive():
            p.kill()
            p.join()
    errs = [open(tmp_path / f"rank{r}.err").read() for r in range(WORLD) if (tmp_path / f"rank{r}.err").exists()]
    assert not errs, "\n".join(errs)
    for r in range(WORLD):
        assert (tmp_path / f"rank{r}.ok").exists(), f"rank {r} did not finish (exit code {procs[r].exitcode})"
