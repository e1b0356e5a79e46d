/* dsa_oracle.h -- CPU oracle for the DSA decode path (TEST INFRASTRUCTURE ONLY).
 *
 * A plain, slow, single-threaded fp64 statement of what one decode layer of a
 * Mistral-Large-4-style DeepSeek Sparse Attention stack computes: the
 * lightning-indexer scores, the exact top-k selection and absorbed-MLA
 * attention over the selected latent rows.  Only the test suite, the package
 * smoke check and the CPU-baseline leg of the benchmark may load it.  It shares
 * no code, header, table or helper with the CUDA library.
 *
 * Sources (web pages; cited by title and section):
 *   [vLLM-ML4]  "Day 0 support for Mistral Large 4" (vLLM blog),
 *               Implementation details: Model architecture table; Sparse MLA +
 *               DSA indexer; NoPE, SSMax and LeRoPE; DCP (top-k compaction);
 *               ROCm implementation details: FP8 latent cache.
 *   [colibri]   "Mistral-Large-4 (c/colibri.c)" (colibri docs,
 *               mistral-large4.md), What differs from GLM-5.2: NoPE layers;
 *               SSMax; The indexer; RoPE and the rest.
 *
 * Every pointer is host memory owned by the caller.  Functions return 0 on
 * success and a negative code on a bad argument (nothing is written then).
 */
#ifndef DSA_ORACLE_H
#define DSA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* key storage kinds */
#define ORACLE_KEYS_BF16 0        /* [rows,128] bf16 bits                          */
#define ORACLE_KEYS_E4M3_ROW 1    /* [rows,128] e4m3 codes + [rows] fp32 scale      */
#define ORACLE_KEYS_NVFP4 2       /* [rows,64] E2M1 pairs + [rows,8] E4M3, x tensor scale (72 B) */
/* latent storage kinds */
#define ORACLE_LATENT_BF16 0      /* [rows,576] bf16 bits                           */
#define ORACLE_LATENT_DS_MLA 2    /* [rows,656] bytes: 512 e4m3, 4 fp32, 64 bf16    */
#define ORACLE_LATENT_NVFP4 3     /* [rows,288] E2M1 pairs + [rows,36] E4M3, x tensor scale (324 B) */

#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_POS (-2)       /* query position outside [0, ctx_len)            */
#define ORACLE_ERR_PAGE (-3)      /* page id / row outside the cache                */
#define ORACLE_ERR_INDEX (-4)     /* selected index outside [0, ctx_len)            */
#define ORACLE_ERR_NOMEM (-5)

/* Where each sequence's tokens live.  Token j of sequence b is physical row
 * page_table[b*max_pages + j/page_size]*page_size + j%page_size when
 * page_table is non-NULL, else seq_base[b] + j. */
typedef struct {
    int32_t num_seqs;
    const int32_t* ctx_len;     /* [num_seqs] */
    const int32_t* page_table;  /* [num_seqs*max_pages] or NULL */
    int32_t page_size;
    int32_t max_pages;
    const int64_t* seq_base;    /* [num_seqs], used when page_table == NULL */
    int64_t num_rows;           /* rows in every cache, for bounds checks */
} oracle_seqs;

double oracle_bf16_value(uint16_t bits);
double oracle_e4m3_value(uint8_t code);
int oracle_ds_mla_row(const uint8_t* row656, double* out576);

/* Indexer scores of nq queries.  scores[t*ld + j] for j <= q_pos[t]; the rest
 * of the row up to ctx_len is set to -INFINITY. */
int oracle_index_scores(int32_t nq, const uint16_t* q /*[nq,32,128]*/, const float* w /*[nq,32]*/,
                        const float* ssmax_s, const float* ssmax_b /*[32]*/,
                        const float* inv_freq /*[32] or NULL = NoPE*/,
                        const int32_t* q_seq, const int32_t* q_pos /*[nq]*/,
                        int32_t key_kind, const void* keys, const float* key_scale,
                        const oracle_seqs* seqs, double* scores, int64_t ld);

/* Exact top-k of n scores: the min(k, n) largest, ties to the smaller index.
 * idx[0..len) in selection order (score descending, index ascending), the
 * rest of idx[0..k) set to -1. */
int oracle_topk(const double* scores, int32_t n, int32_t k, int32_t* idx, int32_t* len);

/* Absorbed-MLA attention of one query over the selected tokens of its
 * sequence: slots idx[0..topk_len) that are >= 0.  out [64,512], lse [64]
 * (natural log); probs [64, topk_len] (per slot, 0 for skipped slots) or NULL. */
int oracle_sparse_mla(const uint16_t* q /*[64,576]*/, int32_t latent_kind, const void* latent,
                      const oracle_seqs* seqs, int32_t seq, const int32_t* idx, int32_t topk_len,
                      double sm_scale, double* out, double* lse, double* probs);

/* Row sizes in bytes of the stored formats, per token per layer. */
int64_t oracle_latent_row_bytes(int32_t latent_kind);
int64_t oracle_index_row_bytes(int32_t key_kind);

/* ---- the cache-write side (the kernels on either side of the decode path) ----
 *
 * Round-to-nearest-even encoders (the decoders above are their inverses):
 * bf16 (8 significant bits, subnormals kept) and OCP e4m3 (4 significant
 * bits, subnormals 2^-9 apart, saturating at +-448; NaN -> 0x7F). */
uint16_t oracle_bf16_encode(double v);
uint8_t oracle_e4m3_encode(double v);

/* Indexer key of n new tokens ([colibri] The indexer: k = LayerNorm(wk(x)),
 * rotated on its first 64 dims on RoPE layers): x [n,128] bf16 bits (the
 * projection's output), LayerNorm over the 128 dims with biased variance,
 * (x - mean) / sqrt(var + eps) * gamma + beta, then on RoPE layers the pairs
 * (2i, 2i+1), i < 32, rotated by pos[t] * inv_freq[i].  out [n,128], exact
 * values before storage rounding. */
int oracle_index_k(int32_t n, const uint16_t* x, const float* gamma, const float* beta, double eps,
                   const int32_t* pos, const float* inv_freq /*[32] or NULL = NoPE*/, double* out);

/* Latent row of n new tokens ([vLLM-ML4] Model architecture: KV LoRA rank
 * 512 + RoPE dim 64): c_kv [n,512] bf16 bits copied, k_pe [n,64] bf16 bits
 * rotated as interleaved pairs by pos[t] * inv_freq[i] on RoPE layers.
 * out [n,576], exact values before storage rounding. */
int oracle_latent_k(int32_t n, const uint16_t* c_kv, const uint16_t* k_pe, const int32_t* pos,
                    const float* inv_freq /*[32] or NULL*/, double* out);

/* Attention query of nq queries ([colibri] SSMax: every head's query times
 * s_h ln(pos+1) + b_h; [vLLM-ML4] fusions "MLA RoPE + SSMax"): q [nq,64,576]
 * bf16 bits (absorbed: 512 latent dims + 64 RoPE dims), the RoPE dims
 * rotated as interleaved pairs by pos * inv_freq on RoPE layers, every dim
 * of head h times f_h.  out [nq,64,576], exact values before rounding. */
int oracle_mla_q(int32_t nq, const uint16_t* q, const float* ssmax_s, const float* ssmax_b /*[64]*/,
                 const float* inv_freq /*[32] or NULL*/, const int32_t* pos, double* out);

/* ---- DCP: the per-rank steps of decode context parallelism ----
 *
 * [vLLM-ML4] Long context: decode and prefill context parallelism: the latent
 * cache is sharded by token; each rank pushes its packed (score, id) top-k
 * candidates to its peers and a selector merges them; each rank compacts the
 * global top-k slots it owns and bounds its attention with topk_length (a
 * rank owning none of a query's slots gets an empty row); the ranks' partial
 * outputs are merged by an LSE combine.
 *
 * Ownership: `world` ranks take a sequence's tokens in turns of `interleave`:
 * token t lives on rank (t / interleave) mod world, at local position
 * (t / (interleave * world)) * interleave + t mod interleave. */
int32_t oracle_dcp_owner(int32_t t, int32_t world, int32_t interleave);
int32_t oracle_dcp_local(int32_t t, int32_t world, int32_t interleave);
int32_t oracle_dcp_global(int32_t local, int32_t rank, int32_t world, int32_t interleave);

/* Packed candidate: the high 32 bits an order-preserving code of the fp32
 * score (its bits with the sign bit set when positive, all bits inverted when
 * negative; -0 coded as +0), the low 32 bits 0xFFFFFFFF - id (0 <= id).  A
 * larger packed value is a larger score or, at equal scores, a smaller id;
 * 0 is an empty slot.  unpack returns 1 for a candidate, 0 for an empty slot. */
uint64_t oracle_dcp_pack(float score, int32_t id);
int oracle_dcp_unpack(uint64_t c, float* score, int32_t* id);

/* The selector: the min(k, #candidates) candidates of num_lists lists of
 * list_len packed slots (lists[r*list_len + i]; empty slots skipped) with the
 * largest scores, ties to the smaller id; their ids ascending in ids[0..len),
 * the rest of ids[0..k) -1.  An id present twice: ORACLE_ERR_INDEX. */
int oracle_topk_merge(int32_t num_lists, int32_t list_len, const uint64_t* lists, int32_t k, int32_t* ids,
                      int32_t* len);

/* Top-k compaction for one rank: the slots i < len of idx holding an id >= 0
 * that `rank` owns, in their order, as local positions; *local_len their
 * number, the rest of local_idx[0..k) -1. */
int oracle_topk_compact(int32_t k, const int32_t* idx, int32_t len, int32_t rank, int32_t world,
                        int32_t interleave, int32_t* local_idx, int32_t* local_len);

/* LSE combine of num_parts partial results for `rows` (query, head) rows:
 * lse[i] = ln sum_r exp(lse_parts[r*rows + i]), out[i] = sum_r
 * exp(lse_parts[r*rows + i] - lse[i]) * o_parts[(r*rows + i)*dim + d]; parts
 * at -inf add nothing; all at -inf give out = 0 and lse = -inf. */
int oracle_lse_combine(int32_t num_parts, int64_t rows, int32_t dim, const double* o_parts,
                       const double* lse_parts, double* out, double* lse);

/* ---- NVFP4: 4.5-bit cache values ("vLLM adds NVFP4 serving for MiniMax
 * M3.1 Flash": NVFP4 attention and indexer caches, 4-bit values costing 4.5
 * bits with their block scales) ----
 * Elements are E2M1 (sign, 2 exponent bits with bias 1, 1 mantissa bit:
 * magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), two per byte with the even element
 * in the low nibble; every 16 consecutive elements share one E4M3 block scale
 * (4 + 8/16 = 4.5 bits per value) and a tensor shares one fp32 scale g:
 * value = g * e4m3(block scale) * e2m1(code). */
double oracle_e2m1_value(uint8_t nibble);
/* nearest E2M1 (ties to the even mantissa), saturating at +-6; the sign of
 * v (also of a zero) in the sign bit; NaN -> +0 */
uint8_t oracle_e2m1_encode(double v);
/* n values (n % 16 == 0), tensor scale g > 0: block b's scale s_b =
 * e4m3_encode(max |v| over the block / (6 g)); its codes e2m1_encode(v /
 * (g * e4m3(s_b))), all +0 when the scale is 0.  codes [n/2], scales [n/16]. */
int oracle_nvfp4_quantize(int32_t n, const double* v, double g, uint8_t* codes, uint8_t* scales);
int oracle_nvfp4_dequantize(int32_t n, const uint8_t* codes, const uint8_t* scales, double g, double* out);

/* NVFP4 caches: the indexer scores and the attention of oracle_index_scores
 * and oracle_sparse_mla over keys and latent rows stored as NVFP4 planes: index
 * keys codes [rows,64] with E4M3 scales [rows,8]; latent rows (all 576 dims)
 * codes [rows,288] with scales [rows,36]; g the cache's tensor scale. */
int oracle_index_scores_nvfp4(int32_t nq, const uint16_t* q, const float* w, const float* ssmax_s,
                              const float* ssmax_b, const float* inv_freq, const int32_t* q_seq,
                              const int32_t* q_pos, const uint8_t* codes, const uint8_t* block_scales, double g,
                              const oracle_seqs* seqs, double* scores, int64_t ld);
int oracle_sparse_mla_nvfp4(const uint16_t* q, const uint8_t* codes, const uint8_t* block_scales, double g,
                            const oracle_seqs* seqs, int32_t seq, const int32_t* idx, int32_t topk_len,
                            double sm_scale, double* out, double* lse, double* probs);

/* ---- block-sparse selection ("vLLM adds NVFP4 serving for MiniMax M3.1
 * Flash", MiniMax Sparse Attention: 128-token KV blocks, 16 blocks selected by
 * scanning the index keys with the most recent block always kept, exact
 * attention over the selected blocks' 2,048 keys) ----
 * Over the n causal scores of a query (keys 0..n-1, the query at n-1): block
 * b holds keys [b*block, (b+1)*block) and scores the maximum of its keys'
 * scores; the query's own block (the most recent) is always selected, then the
 * nsel-1 other blocks with the largest scores (ties to the smaller block).
 * idx[0..len) are the selected blocks' causal keys in ascending order, the
 * rest of idx[0..nsel*block) -1. */
int oracle_block_topk(const double* scores, int32_t n, int32_t block, int32_t nsel, int32_t* idx, int32_t* len);

#ifdef __cplusplus
}
#endif
#endif
