"""GB300 (sm_103a) DSA decode path: lightning indexer -> exact top-k -> sparse
absorbed-MLA attention, as hand-written CUDA behind a C ABI (include/dsa.h),
plus the cache-write side (new indexer keys and latent rows into the caches,
the attention query's RoPE + SSMax) and one rank's compute steps of decode
context parallelism (top-k candidates, their merge, compaction, LSE combine).

The Python names mirror the C entry points; they only marshal arguments.
Importing the package loads nothing; the first call loads ``libdsa.so`` and
raises if it is not built.
"""

from ._binding import (  # noqa: F401
    DSA_BF16,
    DSA_FP8_DS_MLA,
    DSA_FP8_E4M3_ROWSCALE,
    DSA_NVFP4,
    DcpShard,
    DsaError,
    Seqs,
    dsa_block_topk,
    dsa_decode_layer,
    dsa_decode_layer_launches,
    dsa_decode_layer_launches_for,
    dsa_dcp_shard_seqs,
    dsa_index_k_insert,
    dsa_index_scores,
    dsa_index_scores_nvfp4,
    dsa_latent_insert,
    dsa_lse_combine,
    dsa_mla_q_prep,
    dsa_topk,
    dsa_topk_candidates,
    dsa_topk_compact,
    dsa_topk_merge,
    dsa_workspace_size,
    load,
    sparse_mla_decode,
    sparse_mla_decode_noalloc,
    sparse_mla_decode_nvfp4,
    version,
)

__all__ = ["Seqs", "DsaError", "dsa_workspace_size", "dsa_index_scores", "dsa_index_scores_nvfp4", "dsa_topk", "sparse_mla_decode", "sparse_mla_decode_noalloc", "sparse_mla_decode_nvfp4",
           "dsa_decode_layer", "dsa_decode_layer_launches", "dsa_decode_layer_launches_for", "dsa_index_k_insert", "dsa_latent_insert", "dsa_mla_q_prep",
           "DcpShard", "dsa_topk_candidates", "dsa_topk_merge", "dsa_topk_compact", "dsa_lse_combine",
           "dsa_block_topk", "dsa_dcp_shard_seqs",
           "load", "version", "DSA_BF16", "DSA_FP8_E4M3_ROWSCALE", "DSA_FP8_DS_MLA"]
