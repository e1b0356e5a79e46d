"""Wiring of one decode step over device-resident inputs: holds the dsa_seqs
view, the caller workspace and the outputs, and issues the C-ABI calls.

A step is one indexer-owning layer (dsa_decode_layer) and, for workloads with
a shared-indexer layer, a second call that reuses the selection over that
layer's own query and latent cache.  Only marshalling happens here.
"""

from __future__ import annotations

import torch

from . import _binding as B


def seqs_from_inputs(d: dict, queries_per_seq: int) -> B.Seqs:
    lay = d["layout"]
    return B.Seqs(d["ctx_len"], d["q_start"], d["q_pos"], max_ctx=max(lay.ctx_len), max_q_per_seq=queries_per_seq,
                  num_rows=lay.num_rows, page_table=d.get("page_table"), page_size=lay.page_size,
                  seq_base=d.get("seq_base"))


class DecodeStep:
    """Owns workspace and outputs for one workload; ``run()`` enqueues a step."""

    def __init__(self, d: dict, queries_per_seq: int, k: int, device="cuda", select_block: int = 0):
        self.d = d
        self.select_block = int(select_block)  # 0: exact top-k; > 0: block-sparse selection
        self.seqs = seqs_from_inputs(d, queries_per_seq)
        self.num_q = int(d["q_pos"].shape[0])
        self.k = int(k)
        self.ws_bytes = B.dsa_workspace_size(self.seqs, self.num_q, self.k)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)
        Q = self.num_q
        self.idx = torch.empty(Q, self.k, dtype=torch.int32, device=device)
        self.topk_len = torch.empty(Q, dtype=torch.int32, device=device)
        self.out = torch.empty(Q, 64, 512, dtype=torch.bfloat16, device=device)
        self.lse = torch.empty(Q, 64, dtype=torch.float32, device=device)
        self.shared = "q_mla2" in d
        if self.shared:
            self.out2 = torch.empty_like(self.out)
            self.lse2 = torch.empty_like(self.lse)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.k_fp8 = d["k_idx"].dtype == torch.uint8
        self.lat_fp8 = d["latent"].dtype == torch.uint8
        self.launches = 0

    def layer_args(self, shared: bool = False, queries: dict = None) -> dict:
        """dsa_layer_args fields; ``queries`` (q_idx, w, q_mla, q_mla2) replaces
        the workload's own query tensors (same shapes)."""
        d = dict(self.d, **queries) if queries else self.d
        k_nv4, lat_nv4 = "k_bscale" in d, "lat_bscale" in d  # NVFP4 caches
        a = dict(q_idx=d["q_idx"], w=d["w"], ssmax_s=d["ssmax_s"], ssmax_b=d["ssmax_b"], inv_freq=d["inv_freq"],
                 k_idx=d["k_idx"], k_scale=d.get("k_scale"),
                 k_dtype=B.DSA_NVFP4 if k_nv4 else B.DSA_FP8_E4M3_ROWSCALE if self.k_fp8 else B.DSA_BF16,
                 k_block_scales=d.get("k_bscale"), k_global=d.get("k_global", 0.0),
                 reuse_idx=0, k=self.k, select_block=self.select_block,
                 idx=self.idx, topk_len=self.topk_len, q_mla=d["q_mla"], latent=d["latent"],
                 latent_dtype=B.DSA_NVFP4 if lat_nv4 else B.DSA_FP8_DS_MLA if self.lat_fp8 else B.DSA_BF16,
                 latent_scales=d.get("lat_bscale"), latent_global=d.get("lat_global", 0.0),
                 sm_scale=d["sm_scale"], out=self.out, lse=self.lse)
        if shared:
            a.update(reuse_idx=1, q_mla=d["q_mla2"], latent=d["latent2"], out=self.out2, lse=self.lse2)
        return a

    def launches_per_step(self) -> int:
        n = B.dsa_decode_layer_launches_for(self.layer_args(False), self.seqs, self.num_q)
        if self.shared:
            n += B.dsa_decode_layer_launches_for(self.layer_args(True), self.seqs, self.num_q)
        return n

    def run(self, stream=None, events=None, events2=None, queries=None):
        """One step; ``events``/``events2``: optional 4 recorded CUDA events per
        layer (before the indexer, after the indexer, top-k, attention);
        ``queries``: another set of query tensors for this step."""
        a = self.layer_args(False, queries)
        a["events"] = events
        B.dsa_decode_layer(a, self.seqs, self.num_q, self.ws, self.ws_bytes, self.status, stream)
        if self.shared:
            a = self.layer_args(True, queries)
            a["events"] = events2
            B.dsa_decode_layer(a, self.seqs, self.num_q, self.ws, self.ws_bytes, self.status, stream)

    def device_status(self) -> int:
        return int(self.status.item())
