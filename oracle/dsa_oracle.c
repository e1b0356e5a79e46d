/* dsa_oracle.c -- CPU oracle for the DSA decode path (TEST INFRASTRUCTURE ONLY).
 *
 * Plain fp64, single-threaded, no blocking, fusion or reordering beyond the
 * definitions on the pages.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg use it.  See dsa_oracle.h for the sources.
 *
 * Its pins are defined in tests/oracle_pins.py and run by tests/test_oracle.py
 * (closed forms, invariants, special cases, brute force on tiny inputs);
 * tests/test_oracle_mutants.py plants mistakes in a copy and checks each is
 * caught.
 *
 * Plain C rather than C++: every operation is written out where it happens
 * (no overloads, templates or library algorithms between a formula and the
 * code), the same gcc build with -ffp-contract=off rounds alike on x86 and
 * Arm, and the unmangled symbols load directly through ctypes.
 */
#include "dsa_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

enum { IH = 32, ID = 128, RP = 32, MH = 64, MD = 576, MV = 512 };

/* bf16 is the upper 16 bits of an IEEE-754 binary32. */
double oracle_bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa
 * bits; exponent 0 is subnormal (2^-6 * m/8); no infinities; S.1111.111 is
 * NaN; largest finite 448.  The fp8 caches store this format
 * ([vLLM-ML4] Sparse MLA + DSA indexer; FP8 latent cache). */
double oracle_e4m3_value(uint8_t code) {
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, 1 - 7);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* fp8_ds_mla row, 656 bytes per token per layer ([vLLM-ML4] Sparse MLA + DSA
 * indexer: 41,328 latent bytes per token = 63 cache-owning layers x 656; FP8
 * latent cache: 656 for fp8_ds_mla).  Byte order taken here: [0,512) e4m3
 * latent codes, [512,528) four little-endian fp32 scales, one per 128 latent
 * dims, [528,656) the 64 RoPE dims as bf16. */
int oracle_ds_mla_row(const uint8_t* row, double* out) {
    float scale[4];
    for (int g = 0; g < 4; ++g) memcpy(&scale[g], row + MV + 4 * g, 4);
    for (int d = 0; d < MV; ++d) out[d] = oracle_e4m3_value(row[d]) * (double)scale[d / 128];
    for (int r = 0; r < MD - MV; ++r) {
        uint16_t b;
        memcpy(&b, row + MV + 16 + 2 * r, 2);
        out[MV + r] = oracle_bf16_value(b);
    }
    return 0;
}

int64_t oracle_latent_row_bytes(int32_t kind) {
    if (kind == ORACLE_LATENT_BF16) return 2 * MD; /* 1,152 */
    if (kind == ORACLE_LATENT_DS_MLA) return MV + 4 * 4 + 2 * (MD - MV); /* 656 */
    if (kind == ORACLE_LATENT_NVFP4) return MD / 2 + MD / 16;           /* 324: 288 code bytes, 36 scales */
    return -1;
}

int64_t oracle_index_row_bytes(int32_t kind) {
    if (kind == ORACLE_KEYS_BF16) return 2 * ID;        /* 256 */
    if (kind == ORACLE_KEYS_E4M3_ROW) return ID + 4;    /* 132 */
    if (kind == ORACLE_KEYS_NVFP4) return ID / 2 + ID / 16; /* 72: 64 code bytes, 8 scales */
    return -1;
}

/* Physical row of token j of sequence b, or -1. */
static int64_t phys_row(const oracle_seqs* s, int32_t b, int64_t j) {
    int64_t row;
    if (s->page_table) {
        int64_t p = j / s->page_size;
        if (p >= s->max_pages) return -1;
        int64_t page = s->page_table[(int64_t)b * s->max_pages + p];
        if (page < 0) return -1;
        row = page * s->page_size + j % s->page_size;
    } else {
        row = s->seq_base[b] + j;
    }
    if (row < 0 || row >= s->num_rows) return -1;
    return row;
}

/* where and how the index keys are stored */
typedef struct {
    int32_t kind;
    const void* keys;            /* bf16 or e4m3 [rows,128]; NVFP4: codes [rows,64] */
    const float* row_scale;      /* e4m3: [rows] */
    const uint8_t* block_scale;  /* NVFP4: E4M3 [rows,8] */
    double global;               /* NVFP4: tensor scale */
} key_store;

static void decode_key(const key_store* ks, int64_t row, double* k) {
    if (ks->kind == ORACLE_KEYS_BF16) {
        const uint16_t* p = (const uint16_t*)ks->keys + row * ID;
        for (int d = 0; d < ID; ++d) k[d] = oracle_bf16_value(p[d]);
    } else if (ks->kind == ORACLE_KEYS_E4M3_ROW) {
        const uint8_t* p = (const uint8_t*)ks->keys + row * ID;
        double sc = (double)ks->row_scale[row];
        for (int d = 0; d < ID; ++d) k[d] = oracle_e4m3_value(p[d]) * sc;
    } else {
        oracle_nvfp4_dequantize(ID, (const uint8_t*)ks->keys + row * (ID / 2), ks->block_scale + row * (ID / 16),
                                ks->global, k);
    }
}

/* Lightning-indexer score of one query against every causal key.
 *
 * [colibri] What differs from GLM-5.2 -- SSMax: every head's query is
 * multiplied by s*log(position+1)+b with the head's own s and b, in the
 * indexer too (natural log, 0-based absolute position).  The indexer: q and k
 * are rotated on their first 64 dims on RoPE layers (the cached keys are
 * stored already rotated at their own positions, so only q rotates here); the
 * score is relu(q.k/sqrt(128)) weighted by w/sqrt(32), summed over the 32
 * index heads ([vLLM-ML4] Model architecture: 32 index heads).  RoPE and the
 * rest: interleaved pairs (2i, 2i+1), i < 32, rotated by pos*inv_freq_i where
 * inv_freq already holds the YaRN frequency divided by the pair's learned
 * LeRoPE factor ([vLLM-ML4] NoPE, SSMax and LeRoPE: LeRoPE is folded into the
 * YaRN frequencies).  NoPE layers: no rotation (inv_freq == NULL). */
static int score_query(const uint16_t* q, const float* w, const float* ss, const float* sb,
                       const float* inv_freq, int32_t b, int32_t pos, const key_store* ks,
                       const oracle_seqs* seqs, double* out) {
    double qh[IH][ID];
    double k[ID];
    for (int h = 0; h < IH; ++h) {
        double f = (double)ss[h] * log((double)pos + 1.0) + (double)sb[h];
        for (int d = 0; d < ID; ++d) qh[h][d] = f * oracle_bf16_value(q[h * ID + d]);
        if (inv_freq) {
            for (int i = 0; i < RP; ++i) {
                double th = (double)pos * (double)inv_freq[i];
                double c = cos(th), s = sin(th);
                double x0 = qh[h][2 * i], x1 = qh[h][2 * i + 1];
                qh[h][2 * i] = x0 * c - x1 * s;
                qh[h][2 * i + 1] = x0 * s + x1 * c;
            }
        }
    }
    for (int64_t j = 0; j <= pos; ++j) {
        int64_t row = phys_row(seqs, b, j);
        if (row < 0) return ORACLE_ERR_PAGE;
        decode_key(ks, row, k);
        double total = 0.0;
        for (int h = 0; h < IH; ++h) {
            double dot = 0.0;
            for (int d = 0; d < ID; ++d) dot += qh[h][d] * k[d];
            double r = dot / sqrt(128.0);
            if (r < 0.0) r = 0.0;
            total += (double)w[h] * r / sqrt(32.0);
        }
        out[j] = total;
    }
    return 0;
}

static int index_scores(int32_t nq, const uint16_t* q, const float* w, const float* ssmax_s,
                        const float* ssmax_b, const float* inv_freq, const int32_t* q_seq, const int32_t* q_pos,
                        const key_store* ks, const oracle_seqs* seqs, double* scores, int64_t ld) {
    if (nq < 0 || !q || !w || !ssmax_s || !ssmax_b || !q_seq || !q_pos || !ks->keys || !seqs || !scores)
        return ORACLE_ERR_ARG;
    for (int32_t t = 0; t < nq; ++t) {
        int32_t b = q_seq[t], pos = q_pos[t];
        if (b < 0 || b >= seqs->num_seqs) return ORACLE_ERR_ARG;
        if (pos < 0 || pos >= seqs->ctx_len[b] || seqs->ctx_len[b] > ld) return ORACLE_ERR_POS;
    }
    for (int32_t t = 0; t < nq; ++t) {
        int32_t b = q_seq[t], pos = q_pos[t];
        double* row = scores + (int64_t)t * ld;
        int rc = score_query(q + (int64_t)t * IH * ID, w + (int64_t)t * IH, ssmax_s, ssmax_b, inv_freq, b, pos,
                             ks, seqs, row);
        if (rc) return rc;
        for (int64_t j = (int64_t)pos + 1; j < seqs->ctx_len[b]; ++j) row[j] = -INFINITY;
    }
    return 0;
}

int oracle_index_scores(int32_t nq, const uint16_t* q, const float* w, const float* ssmax_s,
                        const float* ssmax_b, const float* inv_freq, const int32_t* q_seq,
                        const int32_t* q_pos, int32_t key_kind, const void* keys, const float* key_scale,
                        const oracle_seqs* seqs, double* scores, int64_t ld) {
    if (key_kind != ORACLE_KEYS_BF16 && key_kind != ORACLE_KEYS_E4M3_ROW) return ORACLE_ERR_ARG;
    if (key_kind == ORACLE_KEYS_E4M3_ROW && !key_scale) return ORACLE_ERR_ARG;
    key_store ks = {key_kind, keys, key_scale, NULL, 1.0};
    return index_scores(nq, q, w, ssmax_s, ssmax_b, inv_freq, q_seq, q_pos, &ks, seqs, scores, ld);
}

int oracle_index_scores_nvfp4(int32_t nq, const uint16_t* q, const float* w, const float* ssmax_s,
                              const float* ssmax_b, const float* inv_freq, const int32_t* q_seq,
                              const int32_t* q_pos, const uint8_t* codes, const uint8_t* block_scales, double g,
                              const oracle_seqs* seqs, double* scores, int64_t ld) {
    if (!codes || !block_scales || !(g > 0.0)) return ORACLE_ERR_ARG;
    key_store ks = {ORACLE_KEYS_NVFP4, codes, NULL, block_scales, g};
    return index_scores(nq, q, w, ssmax_s, ssmax_b, inv_freq, q_seq, q_pos, &ks, seqs, scores, ld);
}

typedef struct {
    double s;
    int32_t j;
} scored;

/* score descending, then index ascending */
static int by_score(const void* a, const void* b) {
    const scored* x = (const scored*)a;
    const scored* y = (const scored*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j > y->j) - (x->j < y->j);
}

/* Exact top-k: the keys with the k largest scores ([vLLM-ML4] Highlights and
 * Model architecture: top-k 2048 keys per query; Specialized decode: an exact
 * top-2048).  Ties at the boundary go to the smaller index (a reading; the
 * pages name no rule).  Fewer than k causal keys: all of them, the rest of
 * the slots -1 ([vLLM-ML4] DCP: top-k compaction, topk_length and slots full
 * of -1). */
int oracle_topk(const double* scores, int32_t n, int32_t k, int32_t* idx, int32_t* len) {
    if (n < 0 || k < 0 || (!scores && n) || (!idx && k) || !len) return ORACLE_ERR_ARG;
    scored* v = (scored*)malloc(sizeof(scored) * (size_t)(n ? n : 1));
    if (!v) return ORACLE_ERR_NOMEM;
    for (int32_t j = 0; j < n; ++j) {
        v[j].s = scores[j];
        v[j].j = j;
    }
    qsort(v, (size_t)n, sizeof(scored), by_score);
    int32_t m = n < k ? n : k;
    for (int32_t i = 0; i < k; ++i) idx[i] = i < m ? v[i].j : -1;
    *len = m;
    free(v);
    return 0;
}

/* Absorbed-MLA attention over the selected latent rows.
 *
 * [vLLM-ML4] Model architecture: 64 heads, MLA with KV LoRA rank 512 and RoPE
 * dim 64, so each token holds one shared 576-dim latent row (512 latent + 64
 * RoPE) that serves as the key of every head; in absorbed form the value is
 * the 512 latent dims and the output stays in latent space.  Sparse MLA + DSA
 * indexer: attention reads only the indexer's selected tokens.  For head h:
 * s_j = sm_scale * q_h . c_j over the 576 dims, p = softmax(s) over the
 * selected j, O_h = sum_j p_j c_j[0:512], LSE_h = log sum_j exp(s_j).  An
 * empty selection gives O = 0 and LSE = -inf ([vLLM-ML4] DCP: a fused kernel
 * neutralises empty rows).  NoPE layers are MLA with zero RoPE dims ([vLLM-ML4]
 * NoPE, SSMax and LeRoPE): their inputs carry zeros in dims 512..575. */
/* where and how the latent rows are stored */
typedef struct {
    int32_t kind;
    const void* latent;          /* bf16 [rows,576] or fp8_ds_mla [rows,656]; NVFP4: codes [rows,288] */
    const uint8_t* block_scale;  /* NVFP4: E4M3 [rows,36] */
    double global;               /* NVFP4: tensor scale */
} latent_store;

static int sparse_mla(const uint16_t* q, const latent_store* ls, const oracle_seqs* seqs, int32_t seq,
                      const int32_t* idx, int32_t topk_len, double sm_scale, double* out, double* lse,
                      double* probs) {
    const int32_t latent_kind = ls->kind;
    const void* latent = ls->latent;
    if (!q || !latent || !seqs || !out || !lse || topk_len < 0 || (topk_len && !idx)) return ORACLE_ERR_ARG;
    if (seq < 0 || seq >= seqs->num_seqs) return ORACLE_ERR_ARG;
    int64_t row_bytes = oracle_latent_row_bytes(latent_kind);
    double* c = (double*)malloc(sizeof(double) * MD * (size_t)(topk_len ? topk_len : 1));
    int32_t* slot = (int32_t*)malloc(sizeof(int32_t) * (size_t)(topk_len ? topk_len : 1));
    double* s = (double*)malloc(sizeof(double) * (size_t)(topk_len ? topk_len : 1));
    if (!c || !slot || !s) {
        free(c); free(slot); free(s);
        return ORACLE_ERR_NOMEM;
    }
    int32_t n = 0;
    for (int32_t i = 0; i < topk_len; ++i) {
        int32_t j = idx[i];
        if (j < 0) continue;
        if (j >= seqs->ctx_len[seq]) {
            free(c); free(slot); free(s);
            return ORACLE_ERR_INDEX;
        }
        int64_t row = phys_row(seqs, seq, j);
        if (row < 0) {
            free(c); free(slot); free(s);
            return ORACLE_ERR_PAGE;
        }
        double* cj = c + (int64_t)n * MD;
        if (latent_kind == ORACLE_LATENT_BF16) {
            const uint16_t* p = (const uint16_t*)latent + row * MD;
            for (int d = 0; d < MD; ++d) cj[d] = oracle_bf16_value(p[d]);
        } else if (latent_kind == ORACLE_LATENT_DS_MLA) {
            oracle_ds_mla_row((const uint8_t*)latent + row * row_bytes, cj);
        } else {
            oracle_nvfp4_dequantize(MD, (const uint8_t*)latent + row * (MD / 2), ls->block_scale + row * (MD / 16),
                                    ls->global, cj);
        }
        slot[n++] = i;
    }
    double qd[MD];
    if (probs) memset(probs, 0, sizeof(double) * (size_t)MH * (size_t)topk_len);
    for (int h = 0; h < MH; ++h) {
        for (int d = 0; d < MD; ++d) qd[d] = oracle_bf16_value(q[h * MD + d]);
        double* oh = out + (int64_t)h * MV;
        for (int d = 0; d < MV; ++d) oh[d] = 0.0;
        if (n == 0) {
            lse[h] = -INFINITY;
            continue;
        }
        double mx = -INFINITY;
        for (int32_t j = 0; j < n; ++j) {
            double dot = 0.0;
            for (int d = 0; d < MD; ++d) dot += qd[d] * c[(int64_t)j * MD + d];
            s[j] = sm_scale * dot;
            if (s[j] > mx) mx = s[j];
        }
        double l = 0.0;
        for (int32_t j = 0; j < n; ++j) l += exp(s[j] - mx);
        for (int32_t j = 0; j < n; ++j) {
            double p = exp(s[j] - mx) / l;
            if (probs) probs[(int64_t)h * topk_len + slot[j]] = p;
            const double* cj = c + (int64_t)j * MD;
            for (int d = 0; d < MV; ++d) oh[d] += p * cj[d];
        }
        lse[h] = mx + log(l);
    }
    free(c);
    free(slot);
    free(s);
    return 0;
}

int oracle_sparse_mla(const uint16_t* q, int32_t latent_kind, const void* latent, const oracle_seqs* seqs,
                      int32_t seq, const int32_t* idx, int32_t topk_len, double sm_scale, double* out,
                      double* lse, double* probs) {
    if (latent_kind != ORACLE_LATENT_BF16 && latent_kind != ORACLE_LATENT_DS_MLA) return ORACLE_ERR_ARG;
    latent_store ls = {latent_kind, latent, NULL, 1.0};
    return sparse_mla(q, &ls, seqs, seq, idx, topk_len, sm_scale, out, lse, probs);
}

int oracle_sparse_mla_nvfp4(const uint16_t* q, const uint8_t* codes, const uint8_t* block_scales, double g,
                            const oracle_seqs* seqs, int32_t seq, const int32_t* idx, int32_t topk_len,
                            double sm_scale, double* out, double* lse, double* probs) {
    if (!codes || !block_scales || !(g > 0.0)) return ORACLE_ERR_ARG;
    latent_store ls = {ORACLE_LATENT_NVFP4, codes, block_scales, g};
    return sparse_mla(q, &ls, seqs, seq, idx, topk_len, sm_scale, out, lse, probs);
}

/* ---------------------------------------------------------------------------
 * The cache-write side.  Encoders: round to nearest, ties to the even
 * significand, written out from the two formats' definitions. */
uint16_t oracle_bf16_encode(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                 /* a = m 2^e, m in [0.5, 1): the leading bit is 2^(e-1) */
    int lead = e - 1;
    if (lead < -126) lead = -126; /* subnormals: the quantum stays 2^-133 */
    double q = ldexp(1.0, lead - 7);
    double r = rint(a / q);       /* exact division by a power of two; rint ties to even */
    double val = r * q;
    if (val >= ldexp(2.0, 127)) return sign | 0x7F80;  /* past the largest finite: infinity */
    int be;
    frexp(val, &be);
    if (be - 1 < -126) return sign | (uint16_t)r;      /* subnormal: the significand is the code */
    uint16_t ebits = (uint16_t)(be - 1 + 127);
    uint16_t mbits = (uint16_t)((int64_t)rint(ldexp(val, -(be - 1) + 7)) - 128);
    return sign | (uint16_t)(ebits << 7) | mbits;
}

uint8_t oracle_e4m3_encode(double v) {
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);
    int lead = e - 1;
    if (lead < -6) lead = -6;     /* subnormals: the quantum stays 2^-9 */
    double q = ldexp(1.0, lead - 3);
    double val = rint(a / q) * q;
    if (val > 448.0) val = 448.0; /* saturate */
    if (val == 0.0) return sign;
    int be;
    frexp(val, &be);
    if (be - 1 < -6) return sign | (uint8_t)rint(val / ldexp(1.0, -9));  /* subnormal */
    uint8_t ebits = (uint8_t)(be - 1 + 7);
    uint8_t mbits = (uint8_t)((int64_t)rint(ldexp(val, -(be - 1) + 3)) - 8);
    return sign | (uint8_t)(ebits << 3) | mbits;
}

/* rotate 32 interleaved pairs of v by pos * inv_freq_i ([colibri] RoPE and the rest) */
static void rope32(double* v, int32_t pos, const float* inv_freq) {
    for (int i = 0; i < RP; ++i) {
        double ang = (double)inv_freq[i] * (double)pos;
        double c = cos(ang), s = sin(ang);
        double x0 = v[2 * i], x1 = v[2 * i + 1];
        v[2 * i] = x0 * c - x1 * s;
        v[2 * i + 1] = x0 * s + x1 * c;
    }
}

int oracle_index_k(int32_t n, const uint16_t* x, const float* gamma, const float* beta, double eps,
                   const int32_t* pos, const float* inv_freq, double* out) {
    if (n < 0 || !x || !gamma || !beta || !pos || !out || !(eps >= 0.0)) return ORACLE_ERR_ARG;
    for (int32_t t = 0; t < n; ++t) {
        double v[ID], mean = 0.0, var = 0.0;
        for (int d = 0; d < ID; ++d) mean += (v[d] = oracle_bf16_value(x[(int64_t)t * ID + d]));
        mean /= ID;
        for (int d = 0; d < ID; ++d) var += (v[d] - mean) * (v[d] - mean);
        var /= ID;
        double inv = 1.0 / sqrt(var + eps);
        for (int d = 0; d < ID; ++d) v[d] = (v[d] - mean) * inv * (double)gamma[d] + (double)beta[d];
        if (inv_freq) rope32(v, pos[t], inv_freq);
        for (int d = 0; d < ID; ++d) out[(int64_t)t * ID + d] = v[d];
    }
    return 0;
}

int oracle_latent_k(int32_t n, const uint16_t* c_kv, const uint16_t* k_pe, const int32_t* pos,
                    const float* inv_freq, double* out) {
    if (n < 0 || !c_kv || !k_pe || !pos || !out) return ORACLE_ERR_ARG;
    for (int32_t t = 0; t < n; ++t) {
        double* o = out + (int64_t)t * MD;
        for (int d = 0; d < MV; ++d) o[d] = oracle_bf16_value(c_kv[(int64_t)t * MV + d]);
        for (int d = 0; d < MD - MV; ++d) o[MV + d] = oracle_bf16_value(k_pe[(int64_t)t * (MD - MV) + d]);
        if (inv_freq) rope32(o + MV, pos[t], inv_freq);
    }
    return 0;
}

int oracle_mla_q(int32_t nq, const uint16_t* q, const float* ssmax_s, const float* ssmax_b,
                 const float* inv_freq, const int32_t* pos, double* out) {
    if (nq < 0 || !q || !ssmax_s || !ssmax_b || !pos || !out) return ORACLE_ERR_ARG;
    for (int32_t t = 0; t < nq; ++t) {
        if (pos[t] < 0) return ORACLE_ERR_POS;
        for (int h = 0; h < MH; ++h) {
            const uint16_t* qi = q + ((int64_t)t * MH + h) * MD;
            double* o = out + ((int64_t)t * MH + h) * MD;
            double f = (double)ssmax_s[h] * log((double)pos[t] + 1.0) + (double)ssmax_b[h];
            for (int d = 0; d < MD; ++d) o[d] = oracle_bf16_value(qi[d]);
            if (inv_freq) rope32(o + MV, pos[t], inv_freq);
            for (int d = 0; d < MD; ++d) o[d] *= f;
        }
    }
    return 0;
}

/* ---- DCP: the per-rank steps of decode context parallelism ([vLLM-ML4] Long
 * context: decode and prefill context parallelism) ---- */

/* The cache is sharded by token; token t's turn is t / interleave, and turns go
 * round the ranks in order. */
int32_t oracle_dcp_owner(int32_t t, int32_t world, int32_t interleave) {
    return (t / interleave) % world;
}

int32_t oracle_dcp_local(int32_t t, int32_t world, int32_t interleave) {
    int32_t turn = t / interleave;
    return (turn / world) * interleave + t % interleave;
}

int32_t oracle_dcp_global(int32_t local, int32_t rank, int32_t world, int32_t interleave) {
    int32_t own_turn = local / interleave;
    return (own_turn * world + rank) * interleave + local % interleave;
}

/* Order-preserving code of a float: negative values map below positive ones
 * and, among negatives, a larger magnitude maps lower. */
static uint32_t score_code(float score) {
    uint32_t b;
    if (score == 0.0f) score = 0.0f; /* -0 as +0 */
    memcpy(&b, &score, 4);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

uint64_t oracle_dcp_pack(float score, int32_t id) {
    return ((uint64_t)score_code(score) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)id);
}

int oracle_dcp_unpack(uint64_t c, float* score, int32_t* id) {
    if (c == 0) return 0;
    uint32_t code = (uint32_t)(c >> 32);
    uint32_t b = (code & 0x80000000u) ? (code & 0x7FFFFFFFu) : ~code;
    memcpy(score, &b, 4);
    *id = (int32_t)(0xFFFFFFFFu - (uint32_t)(c & 0xFFFFFFFFu));
    return 1;
}

static int by_id(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* The selector: every candidate of every list, sorted by score descending and
 * id ascending (the same rule as oracle_topk, the id in the index's place);
 * the first k taken and returned in id order. */
int oracle_topk_merge(int32_t num_lists, int32_t list_len, const uint64_t* lists, int32_t k, int32_t* ids,
                      int32_t* len) {
    if (num_lists < 0 || list_len < 0 || k < 0 || (!lists && num_lists && list_len) || (!ids && k) || !len)
        return ORACLE_ERR_ARG;
    int64_t total = (int64_t)num_lists * list_len;
    scored* v = (scored*)malloc(sizeof(scored) * (size_t)(total ? total : 1));
    if (!v) return ORACLE_ERR_NOMEM;
    int64_t n = 0;
    for (int64_t i = 0; i < total; ++i) {
        float sc;
        int32_t id;
        if (oracle_dcp_unpack(lists[i], &sc, &id)) {
            v[n].s = (double)sc;
            v[n].j = id;
            ++n;
        }
    }
    qsort(v, (size_t)n, sizeof(scored), by_score);
    int32_t m = n < k ? (int32_t)n : k;
    for (int32_t i = 0; i < m; ++i) ids[i] = v[i].j;
    qsort(ids, (size_t)m, sizeof(int32_t), by_id);
    for (int32_t i = m; i < k; ++i) ids[i] = -1;
    /* an id seen twice among all candidates */
    int32_t* all = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n ? n : 1));
    if (!all) {
        free(v);
        return ORACLE_ERR_NOMEM;
    }
    for (int64_t i = 0; i < n; ++i) all[i] = v[i].j;
    qsort(all, (size_t)n, sizeof(int32_t), by_id);
    int dup = 0;
    for (int64_t i = 1; i < n; ++i) dup |= all[i] == all[i - 1];
    free(all);
    free(v);
    *len = m;
    return dup ? ORACLE_ERR_INDEX : 0;
}

int oracle_topk_compact(int32_t k, const int32_t* idx, int32_t len, int32_t rank, int32_t world,
                        int32_t interleave, int32_t* local_idx, int32_t* local_len) {
    if (k < 0 || len < 0 || len > k || world < 1 || interleave < 1 || rank < 0 || rank >= world ||
        (!idx && len) || (!local_idx && k) || !local_len)
        return ORACLE_ERR_ARG;
    int32_t m = 0;
    for (int32_t i = 0; i < len; ++i) {
        int32_t t = idx[i];
        if (t >= 0 && oracle_dcp_owner(t, world, interleave) == rank)
            local_idx[m++] = oracle_dcp_local(t, world, interleave);
    }
    for (int32_t i = m; i < k; ++i) local_idx[i] = -1;
    *local_len = m;
    return 0;
}

int oracle_lse_combine(int32_t num_parts, int64_t rows, int32_t dim, const double* o_parts,
                       const double* lse_parts, double* out, double* lse) {
    if (num_parts < 1 || rows < 0 || dim < 0 || !o_parts || !lse_parts || !out || !lse) return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < rows; ++i) {
        double m = -INFINITY;
        for (int32_t r = 0; r < num_parts; ++r) m = fmax(m, lse_parts[(int64_t)r * rows + i]);
        double* o = out + i * dim;
        for (int32_t d = 0; d < dim; ++d) o[d] = 0.0;
        if (m == -INFINITY) {
            lse[i] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int32_t r = 0; r < num_parts; ++r) sum += exp(lse_parts[(int64_t)r * rows + i] - m);
        double L = m + log(sum);
        for (int32_t r = 0; r < num_parts; ++r) {
            double wgt = exp(lse_parts[(int64_t)r * rows + i] - L);
            const double* op = o_parts + ((int64_t)r * rows + i) * dim;
            for (int32_t d = 0; d < dim; ++d) o[d] += wgt * op[d];
        }
        lse[i] = L;
    }
    return 0;
}

/* ---- NVFP4 ("vLLM adds NVFP4 serving for MiniMax M3.1 Flash": NVFP4
 * attention and indexer caches at 4.5 bits per value) ---- */

/* E2M1: exponent field 0 is subnormal (m / 2), otherwise (1 + m / 2) 2^(e - 1). */
double oracle_e2m1_value(uint8_t nibble) {
    int sgn = (nibble >> 3) & 1, e = (nibble >> 1) & 3, m = nibble & 1;
    double v = e == 0 ? m * 0.5 : ldexp(1.0 + m * 0.5, e - 1);
    return sgn ? -v : v;
}

/* the magnitude codes 0..7 in increasing order; nearest by distance, a tie
 * to the code with mantissa bit 0, past 6 the largest */
uint8_t oracle_e2m1_encode(double v) {
    if (isnan(v)) return 0;
    uint8_t sgn = signbit(v) ? 8 : 0;
    double a = fabs(v);
    uint8_t best = 0;
    double best_d = INFINITY;
    for (uint8_t c = 0; c < 8; ++c) {
        double d = fabs(a - oracle_e2m1_value(c));
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sgn | best);
}

int oracle_nvfp4_quantize(int32_t n, const double* v, double g, uint8_t* codes, uint8_t* scales) {
    if (n < 0 || n % 16 || !(g > 0.0) || (n && (!v || !codes || !scales))) return ORACLE_ERR_ARG;
    for (int32_t b = 0; b < n / 16; ++b) {
        const double* x = v + 16 * b;
        double amax = 0.0;
        for (int i = 0; i < 16; ++i) amax = fmax(amax, fabs(x[i]));
        scales[b] = oracle_e4m3_encode(amax / (6.0 * g));
        double s = oracle_e4m3_value(scales[b]);
        for (int i = 0; i < 16; i += 2) {
            uint8_t lo = s > 0.0 ? oracle_e2m1_encode(x[i] / (g * s)) : 0;
            uint8_t hi = s > 0.0 ? oracle_e2m1_encode(x[i + 1] / (g * s)) : 0;
            codes[8 * b + i / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
    return 0;
}

int oracle_nvfp4_dequantize(int32_t n, const uint8_t* codes, const uint8_t* scales, double g, double* out) {
    if (n < 0 || n % 16 || (n && (!codes || !scales || !out))) return ORACLE_ERR_ARG;
    for (int32_t i = 0; i < n; ++i) {
        uint8_t byte = codes[i / 2];
        uint8_t nib = (i % 2) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
        out[i] = g * oracle_e4m3_value(scales[i / 16]) * oracle_e2m1_value(nib);
    }
    return 0;
}

/* ---- block-sparse selection ("vLLM adds NVFP4 serving for MiniMax M3.1
 * Flash", MiniMax Sparse Attention) ---- */
int oracle_block_topk(const double* scores, int32_t n, int32_t block, int32_t nsel, int32_t* idx, int32_t* len) {
    if (n < 1 || block < 1 || nsel < 1 || !scores || !idx || !len) return ORACLE_ERR_ARG;
    const int32_t nb = (n + block - 1) / block; /* blocks holding causal keys */
    const int32_t last = nb - 1;                /* the query's own block */
    scored* v = (scored*)malloc(sizeof(scored) * (size_t)nb);
    char* chosen = (char*)calloc((size_t)nb, 1);
    if (!v || !chosen) {
        free(v);
        free(chosen);
        return ORACLE_ERR_NOMEM;
    }
    for (int32_t b = 0; b < nb; ++b) {
        double m = -INFINITY;
        for (int32_t j = b * block; j < n && j < (b + 1) * block; ++j) m = fmax(m, scores[j]);
        v[b].s = m;
        v[b].j = b;
    }
    chosen[last] = 1;
    /* the other blocks by score descending, block ascending */
    qsort(v, (size_t)nb, sizeof(scored), by_score);
    int32_t taken = 1;
    for (int32_t i = 0; i < nb && taken < nsel; ++i) {
        if (v[i].j == last) continue;
        chosen[v[i].j] = 1;
        ++taken;
    }
    int32_t m = 0;
    for (int32_t b = 0; b < nb; ++b)
        if (chosen[b])
            for (int32_t j = b * block; j < n && j < (b + 1) * block; ++j) idx[m++] = j;
    for (int32_t i = m; i < nsel * block; ++i) idx[i] = -1;
    *len = m;
    free(v);
    free(chosen);
    return 0;
}
