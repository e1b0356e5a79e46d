/* dsa.h -- C ABI of the GB300 (sm_103a) DSA decode path.
 *
 * One decode layer of a Mistral-Large-4-style DeepSeek Sparse Attention stack:
 *   1. lightning indexer: SSMax-scaled, interleaved-RoPE index queries scored
 *      against every causal key (dsa_index_scores),
 *   2. exact top-k selection per query (dsa_topk),
 *   3. absorbed-MLA attention of 64 heads over only the selected latent rows
 *      (sparse_mla_decode),
 * and the three chained on one stream (dsa_decode_layer), including the
 * shared-indexer variant that reuses an earlier layer's selection.  Around it:
 * the cache-write side (new indexer keys and latent rows into their caches,
 * the attention query's RoPE + SSMax) and one rank's compute steps of decode
 * context parallelism (top-k candidates, their merge, compaction, LSE combine).
 *
 * Sources (web pages, cited by title and section):
 *   [vLLM-ML4] "Day 0 support for Mistral Large 4" (vLLM blog), Implementation
 *              details: Model architecture; Sparse MLA + DSA indexer; NoPE,
 *              SSMax and LeRoPE; Long context: DCP (LSE combine, top-k
 *              compaction with topk_length, slots of -1); ROCm implementation
 *              details: Sparse MLA on AITER (top-k positions mapped to cache
 *              slots), DSA indexer on AITER (132-byte FP8 indexer rows), FP8
 *              latent cache (656-byte fp8_ds_mla rows, 1,152-byte bf16 rows).
 *   [colibri]  "Mistral-Large-4 (c/colibri.c)", What differs from GLM-5.2:
 *              NoPE layers; SSMax; The indexer; RoPE and the rest.
 *   [vLLM-ML4] Long context: decode and prefill context parallelism (the DCP
 *              calls); Implementation details, fusions (the indexer K path
 *              written straight into the FP8 cache; MLA RoPE + SSMax).
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE memory owned by the caller unless marked "host".  The
 *     library never allocates; scratch comes from a caller workspace sized by
 *     dsa_workspace_size.
 *   - Work is enqueued on `stream` and returns without synchronising.  Calls are
 *     deterministic: the same inputs give the same bits.
 *   - The return value reports what the host can see: a NULL or misaligned
 *     pointer, an unsupported size or dtype, a too-small workspace, a launch
 *     error.  Nothing is enqueued when it is not DSA_OK.  dsa_last_error_string()
 *     gives the reason (thread-local).
 *   - What only the device can see (a position outside its context, a page or
 *     row outside the cache, an out-of-range selected index, a malformed
 *     q_start) is written to *d_status (device int32; first error wins, the
 *     caller clears it) and the affected work item is skipped.  No kernel traps
 *     or asserts.  The status code is in bits 0-7; for DSA_ERR_TIMEOUT (a
 *     bounded in-kernel wait that gave up after 1 s) bits 8-15 name the kernel
 *     (1 indexer scan, 2 attention, 3 attention over fp8_ds_mla, 4 attention
 *     over NVFP4 latent rows, 5 indexer scan over NVFP4 keys) and bits
 *     16-30 the wait (its mbarrier's shared-memory offset / 8, or 0x7FFF for
 *     the attention's issue loop).
 *   - Indices are logical token positions within a sequence.  The page table or
 *     seq_base maps them to physical cache rows.
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_INDEX_HEADS 32   /* index heads ([vLLM-ML4] Model architecture: 32 index heads) */
#define DSA_INDEX_DIM 128    /* per index head; first 64 dims rotate on RoPE layers ([colibri] The indexer) */
#define DSA_MLA_HEADS 64     /* attention heads ([vLLM-ML4] Model architecture) */
#define DSA_MLA_DIM 576      /* latent row: 512 KV-LoRA dims + 64 RoPE dims */
#define DSA_MLA_VDIM 512     /* value / output width in latent space */
#define DSA_DS_MLA_ROW 656   /* fp8_ds_mla bytes per token */
#define DSA_MAX_TOPK 2048    /* largest k served ([vLLM-ML4] top-k 2048) */

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1,  /* NULL/misaligned pointer, bad size or stride */
    DSA_ERR_UNSUPPORTED = 2,  /* valid but not served (dtype, k, shape) */
    DSA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    DSA_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than dsa_workspace_size */
    DSA_ERR_TIMEOUT = 5,      /* device: a bounded wait gave up */
    DSA_ERR_BAD_INPUT = 6     /* device: position, page, row or index out of range */
} dsa_status;

typedef enum {
    DSA_BF16 = 0,               /* bf16 rows: index keys [rows,128], latent [rows,576] */
    DSA_FP8_E4M3_ROWSCALE = 1,  /* index keys: [rows,128] OCP e4m3 codes + k_scale fp32 [rows]
                                   (132 B/token, [vLLM-ML4] DSA indexer on AITER) */
    DSA_FP8_DS_MLA = 2,         /* latent: [rows,656] bytes = [0,512) e4m3 latent codes,
                                   [512,528) 4 fp32 scales (one per 128 latent dims),
                                   [528,656) 64 bf16 RoPE dims ([vLLM-ML4] FP8 latent cache) */
    DSA_NVFP4 = 3               /* latent: codes [rows,288] bytes (576 E2M1 values, value 2i in the low
                                   nibble of byte i) + E4M3 block scales [rows,36] (one per 16 values) +
                                   one fp32 tensor scale g: value = g * scale * code, 4.5 bits/value;
                                   index keys: codes [rows,64] + scales [rows,8] + g (72 B/token)
                                   ("vLLM adds NVFP4 serving for MiniMax M3.1 Flash": NVFP4 caches) */
} dsa_dtype;

/* Where tokens live.  Sequence b holds ctx_len[b] tokens; its queries are rows
 * q_start[b] .. q_start[b+1]-1 of every per-query tensor, at absolute
 * positions q_pos[row] < ctx_len[b] (a query sees keys 0..q_pos).  Token j of
 * sequence b is physical row page_table[b*max_pages + j/page_size]*page_size +
 * j%page_size when page_table is non-NULL, else seq_base[b] + j. */
typedef struct {
    int32_t num_seqs;         /* host: B >= 1 */
    int32_t max_ctx;          /* host: >= every ctx_len[b]; sizes the grids */
    int32_t max_q_per_seq;    /* host: >= every q_start[b+1]-q_start[b] */
    int32_t page_size;        /* host: tokens per page (page_table only), a power of two >= 16 */
    int32_t max_pages;        /* host: columns of page_table */
    int32_t reserved;
    int64_t num_rows;         /* host: physical rows in every cache, for bounds checks */
    const int32_t* ctx_len;   /* [B] */
    const int32_t* q_start;   /* [B+1], q_start[0] = 0, q_start[B] = num_q */
    const int32_t* q_pos;     /* [num_q] */
    const int32_t* page_table;/* [B, max_pages] or NULL */
    const int64_t* seq_base;  /* [B] when page_table is NULL */
    const int32_t* q_rope_pos;/* [num_q] or NULL: the queries' absolute positions for the index query's
                                 SSMax and RoPE when q_pos holds a shard's local causal bounds (DCP);
                                 NULL: q_pos */
} dsa_seqs;

/* Bytes of workspace the calls below need for these sizes (host only; no
 * device access).  One workspace sized for the largest call serves all. */
dsa_status dsa_workspace_size(const dsa_seqs* seqs, int32_t num_q, int32_t k, size_t* bytes);

/* Lightning-indexer scores ([colibri] SSMax, The indexer, RoPE and the rest;
 * [vLLM-ML4] Model architecture, NoPE, SSMax and LeRoPE):
 *   f_h = ssmax_s[h]*ln(pos+1) + ssmax_b[h];  q_h <- f_h * q_h;
 *   RoPE layers (inv_freq != NULL): pairs (2i, 2i+1), i < 32, of q_h rotated by
 *   pos*inv_freq[i] (inv_freq already holds the YaRN frequency divided by the
 *   LeRoPE factor exp(alpha_i)); NoPE layers (inv_freq == NULL): no rotation;
 *   score[t][j] = sum_h w[t][h] * relu(q_h . k_j / sqrt(128)) / sqrt(32)
 *   for 0 <= j <= pos_t, and -inf for pos_t < j < ctx_len.  Entries at
 *   j >= ctx_len are not written.  Cached keys are stored already rotated.
 *   q_idx   bf16 [num_q, 32, 128]          w        fp32 [num_q, 32]
 *   ssmax_s, ssmax_b fp32 [32]              inv_freq fp32 [32] or NULL
 *   k_idx   k_dtype DSA_BF16 ([rows,128] bf16) or DSA_FP8_E4M3_ROWSCALE
 *           ([rows,128] e4m3 + k_scale fp32 [rows]; k_scale NULL for bf16)
 *   scores  fp32 [num_q, ld], ld >= max_ctx, ld % 4 == 0
 * Alignment: every pointer 16-byte aligned. */
dsa_status dsa_index_scores(const void* q_idx, const float* w, const float* ssmax_s, const float* ssmax_b,
                            const float* inv_freq, const void* k_idx, const float* k_scale, dsa_dtype k_dtype,
                            const dsa_seqs* seqs, int32_t num_q, float* scores, int64_t ld, void* workspace,
                            size_t workspace_bytes, int32_t* d_status, cudaStream_t stream);

/* dsa_index_scores over NVFP4 index keys ("vLLM adds NVFP4 serving for
 * MiniMax M3.1 Flash": NVFP4 indexer caches at 4.5 bits per value, converted
 * inside the kernel).  Key j is k_j = k_global * scale * code:
 *   k_codes        [rows, 64] bytes: 128 E2M1 values, value 2i in the low
 *                  nibble of byte i (16-byte aligned)
 *   k_block_scales [rows, 8] E4M3 codes, one per 16 values (16-byte aligned)
 *   k_global       fp32 tensor scale, > 0 and finite
 * The kernel decodes each key exactly to f16 (an E2M1 value times its E4M3
 * scale) and folds k_global into the head weight.  Scores, layout and errors
 * otherwise as dsa_index_scores (which refuses DSA_NVFP4). */
dsa_status dsa_index_scores_nvfp4(const void* q_idx, const float* w, const float* ssmax_s, const float* ssmax_b,
                                  const float* inv_freq, const void* k_codes, const void* k_block_scales,
                                  float k_global, const dsa_seqs* seqs, int32_t num_q, float* scores, int64_t ld,
                                  void* workspace, size_t workspace_bytes, int32_t* d_status, cudaStream_t stream);

/* Exact top-k per query ([vLLM-ML4] Model architecture: top-k 2048; DCP: an
 * exact top-k, top-k compaction with topk_length, unused slots -1):
 * the min(k, pos+1) keys j <= pos_t with the largest scores; at the boundary
 * equal scores go to the smaller index (-0.0 counts as +0.0).
 *   scores   fp32 [num_q, ld] (as written by dsa_index_scores)
 *   idx      int32 [num_q, k]: selected positions in ascending order, then -1
 *   topk_len int32 [num_q]: number of selected positions
 *   workspace, workspace_bytes: unused (may be NULL and 0): the selection
 *            needs no scratch at any row length
 * 1 <= k <= 2048. */
dsa_status dsa_topk(const float* scores, int64_t ld, const dsa_seqs* seqs, int32_t num_q, int32_t k, int32_t* idx,
                    int32_t* topk_len, void* workspace, size_t workspace_bytes, int32_t* d_status,
                    cudaStream_t stream);

/* Block-sparse selection ("vLLM adds NVFP4 serving for MiniMax M3.1 Flash",
 * MiniMax Sparse Attention: 128-token KV blocks, 16 selected by scanning the
 * index keys with the most recent block always kept, exact attention over the
 * selected blocks' keys).  Over the causal scores j <= pos_t of each query:
 * block i holds keys [i*block, (i+1)*block) and scores the maximum of its
 * causal keys' scores; the query's own block is always selected, then the
 * nsel-1 other blocks with the largest scores (ties to the smaller block).
 *   scores   fp32 [num_q, ld] (as written by dsa_index_scores)
 *   idx      int32 [num_q, nsel*block]: the selected blocks' causal keys in
 *            ascending order, then -1;  topk_len int32 [num_q]
 * As dsa_topk's output, for sparse_mla_decode with k = nsel*block.
 * 1 <= nsel <= DSA_BLOCK_TOPK_MAX_NSEL, nsel*block <= 2048, and
 * ceil(max_ctx / block) blocks must fit one CTA's shared memory (4 bytes each,
 * DSA_BLOCK_TOPK_MAX_SMEM in all). */
#define DSA_BLOCK_TOPK_MAX_NSEL 64
#define DSA_BLOCK_TOPK_MAX_SMEM (200u << 10)
dsa_status dsa_block_topk(const float* scores, int64_t ld, const dsa_seqs* seqs, int32_t num_q, int32_t block,
                          int32_t nsel, int32_t* idx, int32_t* topk_len, int32_t* d_status, cudaStream_t stream);

/* Absorbed-MLA attention over selected latent rows ([vLLM-ML4] Model
 * architecture: 64 heads, KV LoRA rank 512, RoPE dim 64; Sparse MLA + DSA
 * indexer; NoPE, SSMax and LeRoPE: NoPE layers are MLA with zero RoPE dims):
 *   for query t, head h, over slots i < topk_len[t] with idx[t][i] >= 0:
 *   s_i = sm_scale * q[t][h] . c_{idx[t][i]} (576 dims), p = softmax(s),
 *   out[t][h] = sum_i p_i c_{idx[t][i]}[0:512],  lse[t][h] = ln sum_i exp(s_i).
 *   An empty selection gives out = 0 and lse = -inf.
 *   q      bf16 [num_q, 64, 576] (SSMax and RoPE already applied)
 *   latent DSA_BF16 [rows, 576] bf16 or DSA_FP8_DS_MLA [rows, 656] bytes
 *   idx    int32 [num_q, k], topk_len int32 [num_q] (0..k)
 *   out    bf16 [num_q, 64, 512]; lse fp32 [num_q, 64] or NULL
 * 1 <= k <= 2048. */
dsa_status sparse_mla_decode(const void* q, const void* latent, dsa_dtype latent_dtype, const dsa_seqs* seqs,
                             int32_t num_q, const int32_t* idx, const int32_t* topk_len, int32_t k, float sm_scale,
                             void* out, float* lse, void* workspace, size_t workspace_bytes, int32_t* d_status,
                             cudaStream_t stream);

/* sparse_mla_decode over an NVFP4 latent cache (DSA_NVFP4: codes [rows,288],
 * block_scales [rows,36], tensor scale g > 0; "vLLM adds NVFP4 serving for
 * MiniMax M3.1 Flash": NVFP4 caches, converted inside the decode kernel).
 * The gather decodes each row to f16, exactly (an E2M1 value times its E4M3
 * block scale), and g folds into the score scale and the output:
 * s_i = sm_scale g q . c~_i, out = g sum_i p_i c~_i[0:512].  Arguments and
 * results otherwise as sparse_mla_decode.  Alignment: codes 16 bytes,
 * block_scales 4 bytes. */
dsa_status sparse_mla_decode_nvfp4(const void* q, const void* codes, const void* block_scales, float g,
                                   const dsa_seqs* seqs, int32_t num_q, const int32_t* idx, const int32_t* topk_len,
                                   int32_t k, float sm_scale, void* out, float* lse, void* workspace,
                                   size_t workspace_bytes, int32_t* d_status, cudaStream_t stream);

/* ---- the cache-write side: the kernels on either side of the decode path ----
 * Each writes new tokens' rows at the physical rows slot[i] (slot < 0: the
 * token is skipped; slot >= num_rows or pos < 0: DSA_ERR_BAD_INPUT in
 * *d_status, the token skipped).  Storage rounding: bf16 to nearest even;
 * e4m3 (OCP) to nearest even of value / scale, saturating at 448, with
 * scale = max |value| / 448 over the scale's values (1 when they are all 0). */

/* Indexer keys of n new tokens into the indexer cache ([colibri] The indexer:
 * k = LayerNorm(wk(x)), rotated on its first 64 dims on RoPE layers;
 * [vLLM-ML4] Implementation details: the indexer K path written straight
 * into the FP8 cache; DSA indexer on AITER: one FP8 scale per key):
 *   k = (x - mean) / sqrt(var + ln_eps) * ln_gamma + ln_beta over the 128 dims
 *   (biased variance); RoPE layers (inv_freq != NULL): pairs (2i, 2i+1), i < 32,
 *   rotated by pos*inv_freq[i]; stored as k_dtype DSA_BF16 ([rows,128] bf16) or
 *   DSA_FP8_E4M3_ROWSCALE ([rows,128] e4m3 codes + k_scale fp32 [rows]).
 *   x bf16 [n,128] (the projection's output); ln_gamma, ln_beta fp32 [128];
 *   pos int32 [n]; inv_freq fp32 [32] or NULL; slot int64 [n].
 * The rows dsa_index_scores reads.  Alignment: every pointer 16-byte aligned
 * (pos, slot, k_scale: their element size). */
dsa_status dsa_index_k_insert(const void* x, const float* ln_gamma, const float* ln_beta, float ln_eps,
                              const int32_t* pos, const float* inv_freq, const int64_t* slot, int32_t n,
                              void* k_cache, float* k_scale, dsa_dtype k_dtype, int64_t num_rows, int32_t* d_status,
                              cudaStream_t stream);

/* Latent rows of n new tokens ([vLLM-ML4] Model architecture: KV LoRA rank
 * 512, RoPE dim 64; Sparse MLA + DSA indexer: the fp8_ds_mla cache, 656
 * bytes per token): c_kv bf16 [n,512] stored as is (DSA_BF16) or as e4m3 with
 * one fp32 scale per 128 values (DSA_FP8_DS_MLA: [0,512) codes, [512,528) the
 * four scales, [528,656) the RoPE dims bf16); k_pe bf16 [n,64] rotated as
 * interleaved pairs by pos*inv_freq on RoPE layers (NULL: stored as given).
 * latent: [rows,576] bf16 or [rows,656] bytes; the rows sparse_mla_decode
 * reads. */
dsa_status dsa_latent_insert(const void* c_kv, const void* k_pe, const int32_t* pos, const float* inv_freq,
                             const int64_t* slot, int32_t n, void* latent, dsa_dtype latent_dtype, int64_t num_rows,
                             int32_t* d_status, cudaStream_t stream);

/* The attention query ([colibri] SSMax: every head's query times
 * s_h ln(pos+1) + b_h; [vLLM-ML4] Implementation details: MLA RoPE + SSMax):
 *   q_out[t][h] = f_h(pos_t) * (q[t][h] with dims 512..575 rotated as
 *   interleaved pairs by pos_t*inv_freq on RoPE layers), rounded to bf16.
 *   q, q_out bf16 [num_q, 64, 576] (may be the same buffer); ssmax_s, ssmax_b
 *   fp32 [64]; q_pos int32 [num_q]; inv_freq fp32 [32] or NULL.
 * The query sparse_mla_decode takes.  A negative position: DSA_ERR_BAD_INPUT,
 * that query's row left unwritten. */
dsa_status dsa_mla_q_prep(const void* q, const float* ssmax_s, const float* ssmax_b, const float* inv_freq,
                          const int32_t* q_pos, int32_t num_q, void* q_out, int32_t* d_status, cudaStream_t stream);

/* ---- DCP: one rank's compute steps of decode context parallelism ----
 * ([vLLM-ML4] Long context: decode and prefill context parallelism.)  The
 * latent and index caches are sharded by token over `world` ranks.  Each rank
 * scores its own keys and offers its local top-k as packed (score, id)
 * candidates (dsa_topk_candidates); the candidate lists are exchanged (peer
 * inboxes, NCCL: the caller's) and the selector merges them in place into the
 * exact global top-k (dsa_topk_merge); each rank keeps the selected slots it
 * owns as local positions with their count (dsa_topk_compact), attends over
 * them with sparse_mla_decode on its shard (a rank owning none of a query's
 * slots gets out = 0, lse = -inf), and the partial outputs are merged
 * (dsa_lse_combine).  On one GPU the ranks' shards can live in one memory and
 * the same calls run the sharded layer.
 *
 * Ownership: turns of `interleave` tokens go round the ranks: token t of a
 * sequence lives on rank (t / interleave) % world at local position
 * (t / (interleave * world)) * interleave + t % interleave. */
#define DSA_DCP_MAX_RANKS 16          /* ranks, candidate lists and combine parts per call */
#define DSA_DCP_MAX_CANDIDATES 16384  /* num_lists x list_len per query in the selector */

typedef struct {
    int32_t world;       /* ranks sharing a sequence's tokens, 1..DSA_DCP_MAX_RANKS */
    int32_t rank;        /* this rank, 0..world-1 */
    int32_t interleave;  /* tokens per turn, >= 1 (a contiguous shard of S tokens: S) */
} dsa_dcp_shard;

/* Packed candidate (uint64): the high 32 bits the score's order-preserving
 * code (its fp32 bits with the sign bit set when positive, all bits inverted
 * when negative; -0 coded as +0), the low 32 bits 0xFFFFFFFF - id.  A larger
 * packed value is a larger score or, at equal scores, a smaller id, so the
 * exact top-k of any set of candidates is the k largest packed values; 0 is
 * an empty slot. */

/* A rank's top-k candidates: dsa_topk over the rank's local scores (seqs,
 * scores and the causal bounds q_pos in the rank's local positions), then
 * each selected local position l packed with its score and its global id
 * (l / interleave * world + rank) * interleave + l % interleave.
 *   idx, topk_len, workspace: as dsa_topk (the local selection)
 *   cand uint64 [num_q, k], 8-byte aligned: slot i < topk_len[t] the packed
 *        candidate of idx[t][i], the rest 0.
 * Scores must not be NaN.  A global id past INT32_MAX: DSA_ERR_BAD_INPUT in
 * *d_status and an empty slot. */
dsa_status dsa_topk_candidates(const float* scores, int64_t ld, const dsa_seqs* seqs, int32_t num_q, int32_t k,
                               const dsa_dcp_shard* shard, int32_t* idx, int32_t* topk_len, uint64_t* cand,
                               void* workspace, size_t workspace_bytes, int32_t* d_status, cudaStream_t stream);

/* The selector: the exact top-k of num_lists candidate lists per query,
 * read in place (one list per rank).
 *   lists    host array of num_lists (1..16) device pointers, each uint64
 *            [num_q, list_len], 8-byte aligned; num_lists * list_len <= 16384
 *   idx      int32 [num_q, k]: the min(k, #candidates) candidates with the
 *            largest scores (ties to the smaller id), their ids ascending,
 *            then -1;  topk_len int32 [num_q]
 * Ids must be distinct across a query's lists (the shards are disjoint).  A
 * repeated id among the selected: DSA_ERR_BAD_INPUT in *d_status and that
 * query's row empty (topk_len 0, all -1).  1 <= k <= 2048. */
dsa_status dsa_topk_merge(const uint64_t* const* lists, int32_t num_lists, int32_t list_len, int32_t num_q,
                          int32_t k, int32_t* idx, int32_t* topk_len, int32_t* d_status, cudaStream_t stream);

/* Top-k compaction for one rank: the slots i < topk_len[t] of idx holding a
 * global id >= 0 that shard->rank owns, in their order, as local positions;
 * local_len[t] their number; the rest of local_idx[t] -1.  With local_idx and
 * local_len as idx and topk_len, sparse_mla_decode on the rank's shard reads
 * only the rank's share of the selection, its loop bounded by local_len.
 *   idx int32 [num_q, k], topk_len int32 [num_q] (0..k; outside: clamped and
 *   DSA_ERR_BAD_INPUT); local_idx int32 [num_q, k], local_len int32 [num_q].
 * The outputs may be the inputs (in place). */
dsa_status dsa_topk_compact(const int32_t* idx, const int32_t* topk_len, int32_t num_q, int32_t k,
                            const dsa_dcp_shard* shard, int32_t* local_idx, int32_t* local_len, int32_t* d_status,
                            cudaStream_t stream);

/* One rank's view of the sequences, for its calls on its own shard (the
 * shard's tokens at local positions, by the ownership rule above):
 *   local_ctx_len int32 [B]: the tokens the rank owns of each sequence;
 *   local_q_pos   int32 [num_q]: each query's local causal bound, the number
 *                 of tokens the rank owns at or before the query's position
 *                 minus one (-1 and DSA_ERR_BAD_INPUT when it owns none);
 *   local_page_table int32 [B, local_max_pages] or NULL: the rank's pages in
 *                 local order (-1 past the table); needs seqs->page_table and
 *                 an interleave that is a whole number of pages;
 *   local_max_ctx (host out): the most tokens the rank owns of a sequence of
 *                 max_ctx tokens.
 * The rank's dsa_seqs is then seqs with max_ctx = *local_max_ctx, ctx_len =
 * local_ctx_len, q_pos = local_q_pos, q_rope_pos = seqs->q_pos, and either
 * page_table = local_page_table with max_pages = local_max_pages, or (a
 * contiguous shard cache) the shard's own seq_base and num_rows.  The same
 * positions are what dsa_topk_candidates packs and dsa_topk_compact returns. */
dsa_status dsa_dcp_shard_seqs(const dsa_seqs* seqs, int32_t num_q, const dsa_dcp_shard* shard,
                              int32_t* local_ctx_len, int32_t* local_q_pos, int32_t* local_page_table,
                              int32_t local_max_pages, int32_t* local_max_ctx, int32_t* d_status,
                              cudaStream_t stream);

/* LSE combine of num_parts partial attention results (one per rank), per
 * query and head: lse = ln sum_r exp(lse_r), out = sum_r exp(lse_r - lse) o_r;
 * parts at -inf (empty rows) add nothing; all at -inf give out = 0, lse = -inf.
 *   o_parts   host array of num_parts (1..16) device pointers, each bf16
 *             [num_q, 64, 512] (16-byte aligned), as sparse_mla_decode writes
 *   lse_parts host array of num_parts device pointers, each fp32 [num_q, 64]
 *   out bf16 [num_q, 64, 512]; lse fp32 [num_q, 64] or NULL
 * Weights and sums in fp32, out rounded to bf16 (nearest even). */
dsa_status dsa_lse_combine(const void* const* o_parts, const float* const* lse_parts, int32_t num_parts,
                           int32_t num_q, void* out, float* lse, cudaStream_t stream);

/* One decode layer: dsa_index_scores -> dsa_topk -> sparse_mla_decode on one
 * stream, with the scores kept in the workspace.  reuse_idx != 0 is a
 * shared-indexer layer ([vLLM-ML4] Model architecture: 28 layers reuse the
 * top-k of the nearest earlier indexer layer; [colibri] The indexer): idx and
 * topk_len are inputs and only the attention runs; otherwise they are outputs.
 * select_block > 0 selects by blocks instead of keys ("vLLM adds NVFP4 serving
 * for MiniMax M3.1 Flash", MiniMax Sparse Attention): dsa_block_topk with
 * blocks of select_block keys and nsel = k / select_block blocks takes the
 * place of dsa_topk (k a multiple of select_block, and dsa_block_topk's
 * limits); select_block = 0 is the exact top-k. */
typedef struct {
    /* indexer (ignored when reuse_idx != 0) */
    const void* q_idx;
    const float* w;
    const float* ssmax_s;
    const float* ssmax_b;
    const float* inv_freq;
    const void* k_idx;
    const float* k_scale;
    dsa_dtype k_dtype;
    int32_t reuse_idx;
    /* selection */
    int32_t k;
    int32_t select_block;  /* 0: exact top-k; > 0: block-sparse selection, blocks of this many keys */
    int32_t* idx;
    int32_t* topk_len;
    /* attention */
    const void* q_mla;
    const void* latent;
    dsa_dtype latent_dtype;
    float sm_scale;
    void* out;
    float* lse;
    /* optional: NULL, or 4 events recorded on `stream` before the indexer and
       after the indexer, the top-k and the attention (a shared-indexer layer
       records the first three back to back), for per-stage timing */
    cudaEvent_t* events;
    /* latent_dtype == DSA_NVFP4: E4M3 block scales [rows,36] and the tensor
       scale of the latent cache (latent holds the codes [rows,288]) */
    const void* latent_scales;
    float latent_global;
    /* k_dtype == DSA_NVFP4: E4M3 block scales [rows,8] and the tensor scale of
       the index keys (k_idx holds the codes [rows,64]) */
    float k_global;
    const void* k_block_scales;
} dsa_layer_args;

dsa_status dsa_decode_layer(const dsa_layer_args* args, const dsa_seqs* seqs, int32_t num_q, void* workspace,
                            size_t workspace_bytes, int32_t* d_status, cudaStream_t stream);

/* sparse_mla_decode without a workspace, for callers that cannot allocate
 * device memory at all: code embedded in a host process whose GPU memory is
 * owned by another allocator (a serving engine that reserves the whole pool at
 * start-up, a plugin ABI that hands over only input and output buffers), so it
 * has no way to provide the workspace the other entry points take.  The pages
 * have no counterpart of this call; it is a deployment convenience.
 *   Same arguments, semantics and results (within rounding: the split of the
 *   work may differ) as sparse_mla_decode, minus the workspace.  The partial
 *   results of a query's splits go to a static device array of
 *   DSA_NOALLOC_SCRATCH_BYTES owned by the library: every GPU that loads the
 *   library holds it until the process exits.  Where sparse_mla_decode's
 *   splits would need more than the array holds, this call takes fewer splits
 *   per query (down to two, which combine on chip and need none), so no batch
 *   size is refused; such batches run somewhat slower.
 *   The first call on each device looks up the array's device address with
 *   that device current (a runtime query, no allocation); make that first call
 *   before any stream capture on the device.  Every call shares the one array
 *   and each call writes every partial it later reads, so nothing needs
 *   clearing between calls; calls that overlap on the GPU (other streams, other
 *   host threads) race on it and must be serialised by the caller.  No call
 *   allocates or frees memory. */
#define DSA_NOALLOC_SCRATCH_BYTES (16u << 20)
dsa_status sparse_mla_decode_noalloc(const void* q, const void* latent, dsa_dtype latent_dtype,
                                     const dsa_seqs* seqs, int32_t num_q, const int32_t* idx,
                                     const int32_t* topk_len, int32_t k, float sm_scale, void* out, float* lse,
                                     int32_t* d_status, cudaStream_t stream);

/* Number of kernels dsa_decode_layer enqueues for these sizes (reuse_idx and
 * latent_dtype as in dsa_layer_args); 0 when the sizes or the dtype are
 * refused.  For callers that count or capture launches.  (The attention adds
 * its combine kernel when three or more CTAs share a query's selection; the
 * split count is planned for GB300's 152 SMs.) */
int32_t dsa_decode_layer_launches(const dsa_seqs* seqs, int32_t num_q, int32_t k, int32_t reuse_idx,
                                  dsa_dtype latent_dtype);
/* The same count for a full argument set (it also reads select_block); 0 when
 * dsa_decode_layer would refuse the sizes, the selection mode or the dtypes.
 * Host only: no pointer in args is read. */
int32_t dsa_decode_layer_launches_for(const dsa_layer_args* args, const dsa_seqs* seqs, int32_t num_q);

/* Text of the last non-OK status returned on this thread ("" if none). */
const char* dsa_last_error_string(void);
/* Name of a status code. */
const char* dsa_status_string(dsa_status s);
/* Library version, "major.minor.patch". */
const char* dsa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H */
