// api.cu -- the C ABI of include/dsa.h: host-side validation (default-deny,
// every reason listed), workspace carving and the launch sequence.  No entry
// point allocates, synchronises or reads device memory on the host.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <string>

#include "dsa_internal.cuh"

namespace dsa {
namespace {

thread_local char g_err[1024] = "";

dsa_status fail(dsa_status st, const std::string& why) {
    snprintf(g_err, sizeof g_err, "%s", why.c_str());
    return st;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Collects every reason a call is refused, so one message lists them all.
struct Check {
    std::string why;
    dsa_status st = DSA_OK;
    void need(bool ok, dsa_status code, const char* fmt, ...) {
        if (ok) return;
        char buf[256];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        if (!why.empty()) why += "; ";
        why += buf;
        if (st == DSA_OK || (st == DSA_ERR_UNSUPPORTED && code == DSA_ERR_INVALID_ARG)) st = code;
    }
    void ptr(const void* p, const char* name, size_t align = 16) {
        need(p != nullptr, DSA_ERR_INVALID_ARG, "%s is NULL", name);
        if (p) need(aligned(p, align), DSA_ERR_INVALID_ARG, "%s is not %zu-byte aligned", name, align);
    }
    dsa_status done() {
        if (st != DSA_OK) return fail(st, why);
        g_err[0] = 0;
        return DSA_OK;
    }
};

void check_seqs(Check& c, const dsa_seqs* s, int32_t num_q) {
    c.need(s != nullptr, DSA_ERR_INVALID_ARG, "seqs is NULL");
    if (!s) return;
    c.need(s->num_seqs >= 1, DSA_ERR_INVALID_ARG, "num_seqs %d < 1", s->num_seqs);
    c.need(s->max_ctx >= 1 && s->max_ctx <= (1 << 30), DSA_ERR_INVALID_ARG, "max_ctx %d outside [1, 2^30]",
           s->max_ctx);
    c.need(s->max_q_per_seq >= 1, DSA_ERR_INVALID_ARG, "max_q_per_seq %d < 1", s->max_q_per_seq);
    c.need(num_q >= 0, DSA_ERR_INVALID_ARG, "num_q %d < 0", num_q);
    c.need(s->num_rows >= 1, DSA_ERR_INVALID_ARG, "num_rows %lld < 1", (long long)s->num_rows);
    c.ptr(s->ctx_len, "seqs.ctx_len", 4);
    c.ptr(s->q_start, "seqs.q_start", 4);
    c.ptr(s->q_pos, "seqs.q_pos", 4);
    if (s->q_rope_pos) c.ptr(s->q_rope_pos, "seqs.q_rope_pos", 4);
    if (s->page_table) {
        c.ptr(s->page_table, "seqs.page_table", 4);
        c.need(s->page_size >= 16 && (s->page_size & (s->page_size - 1)) == 0, DSA_ERR_UNSUPPORTED,
               "page_size %d is not a power of two >= 16", s->page_size);
        c.need(s->max_pages >= 1, DSA_ERR_INVALID_ARG, "max_pages %d < 1", s->max_pages);
    } else {
        c.ptr(s->seq_base, "seqs.seq_base (page_table is NULL)", 8);
    }
}

void check_workspace(Check& c, const dsa_seqs* s, int32_t num_q, int32_t k, const void* ws, size_t bytes) {
    if (!s || c.st != DSA_OK) return;
    int64_t ld;
    const size_t need = workspace_bytes(*s, num_q, k, &ld);
    c.need(ws != nullptr || need == 0, DSA_ERR_WORKSPACE, "workspace is NULL");
    c.need(ws == nullptr || aligned(ws, 256), DSA_ERR_WORKSPACE, "workspace is not 256-byte aligned");
    c.need(bytes >= need, DSA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", bytes, need);
}

dsa_status cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) {
        g_err[0] = 0;
        return DSA_OK;
    }
    return fail(DSA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

}  // namespace

size_t workspace_bytes(const dsa_seqs& s, int num_q, int k, int64_t* scores_ld) {
    const int64_t ld = ((int64_t)s.max_ctx + 3) / 4 * 4;
    if (scores_ld) *scores_ld = ld;
    const int kk = k < 1 ? 1 : (k > DSA_MAX_TOPK ? DSA_MAX_TOPK : k);
    const int nq = num_q > 0 ? num_q : 1;
    size_t b = 0;
    b += up256((size_t)num_q * kQprepBytes);                         // q'
    b += up256((size_t)num_q * kIH * 4);                             // w'
    b += up256(mla_part_bytes(nq, kk));                              // partial outputs
    b += up256(mla_ml_bytes(nq, kk));                                // partial (max, sum)
    b += up256((size_t)num_q * ld * 4);                              // scores (fused layer)
    return b;
}

Workspace carve_workspace(void* base, const dsa_seqs& s, int num_q, int k) {
    Workspace w{};
    int64_t ld;
    workspace_bytes(s, num_q, k, &ld);
    const int kk = k < 1 ? 1 : (k > DSA_MAX_TOPK ? DSA_MAX_TOPK : k);
    const int nq = num_q > 0 ? num_q : 1;
    uint8_t* p = reinterpret_cast<uint8_t*>(base);
    w.qprep = p;
    p += up256((size_t)num_q * kQprepBytes);
    w.wprep = reinterpret_cast<float*>(p);
    p += up256((size_t)num_q * kIH * 4);
    w.mla_part = reinterpret_cast<float*>(p);
    p += up256(mla_part_bytes(nq, kk));
    w.mla_ml = reinterpret_cast<float*>(p);
    p += up256(mla_ml_bytes(nq, kk));
    w.scores = reinterpret_cast<float*>(p);
    w.scores_ld = ld;
    p += up256((size_t)num_q * ld * 4);
    return w;
}

}  // namespace dsa

namespace dsa {
cudaError_t launch_index_k_insert(const void* x, const float* gamma, const float* beta, float eps, const int32_t* pos,
                                  const float* inv_freq, const int64_t* slot, int32_t n, void* cache, float* k_scale,
                                  bool fp8, int64_t num_rows, int32_t* d_status, cudaStream_t stream);
cudaError_t launch_latent_insert(const void* c_kv, const void* k_pe, const int32_t* pos, const float* inv_freq,
                                 const int64_t* slot, int32_t n, void* latent, bool fp8, int64_t num_rows,
                                 int32_t* d_status, cudaStream_t stream);
cudaError_t launch_mla_q_prep(const void* q, const float* ssmax_s, const float* ssmax_b, const float* inv_freq,
                              const int32_t* q_pos, int32_t num_q, void* q_out, int32_t* d_status,
                              cudaStream_t stream);
cudaError_t launch_cand_pack(const float* scores, int64_t ld, const int32_t* idx, const int32_t* topk_len, int num_q,
                             int k, int world, int rank, int inter, uint64_t* cand, int32_t* d_status,
                             cudaStream_t stream);
cudaError_t launch_topk_merge(const uint64_t* const* lists, int num_lists, int list_len, int num_q, int k,
                              int32_t* idx, int32_t* topk_len, int32_t* d_status, cudaStream_t stream);
cudaError_t launch_topk_compact(const int32_t* idx, const int32_t* topk_len, int num_q, int k, int world, int rank,
                                int inter, int32_t* local_idx, int32_t* local_len, int32_t* d_status,
                                cudaStream_t stream);
cudaError_t launch_lse_combine(const void* const* o_parts, const float* const* lse_parts, int num_parts, int num_q,
                               void* out, float* lse, cudaStream_t stream);
int64_t dcp_owned_tokens(int64_t n, int world, int rank, int inter);
cudaError_t launch_dcp_shard_seqs(const dsa_seqs& s, int num_q, int world, int rank, int inter, int32_t* lctx,
                                  int32_t* lpos, int32_t* ltable, int lmax_pages, int32_t* d_status,
                                  cudaStream_t stream);
size_t block_topk_smem(int max_ctx, int block, int nsel);
cudaError_t launch_block_topk(const float* scores, int64_t ld, const dsa_seqs& s, int num_q, int block, int nsel,
                              int32_t* idx, int32_t* topk_len, int32_t* d_status, cudaStream_t stream,
                              bool from_groups = false);
}  // namespace dsa


using namespace dsa;

// kernels one dsa_decode_layer call enqueues
static int32_t layer_launches(const dsa_seqs& s, int num_q, int k, bool reuse, int select_block) {
    // attention, plus the LSE combine unless every query's splits combine in-kernel
    const int mla = mla_launches(num_q, k);
    (void)s;
    (void)select_block;
    return (reuse ? 0 : 3) + mla;  // query prep, scores, selection (top-k or blocks: one kernel)
}

static void check_shard(Check& c, const dsa_dcp_shard* sh) {
    c.need(sh != nullptr, DSA_ERR_INVALID_ARG, "shard is NULL");
    if (!sh) return;
    c.need(sh->world >= 1 && sh->world <= DSA_DCP_MAX_RANKS, DSA_ERR_UNSUPPORTED, "shard world %d outside [1, %d]",
           sh->world, DSA_DCP_MAX_RANKS);
    c.need(sh->rank >= 0 && sh->rank < sh->world, DSA_ERR_INVALID_ARG, "shard rank %d outside [0, world)", sh->rank);
    c.need(sh->interleave >= 1, DSA_ERR_INVALID_ARG, "shard interleave %d < 1", sh->interleave);
}

extern "C" {

const char* dsa_last_error_string(void) { return g_err; }

const char* dsa_status_string(dsa_status s) {
    switch (s) {
        case DSA_OK: return "DSA_OK";
        case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
        case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
        case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
        case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
        case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
        case DSA_ERR_BAD_INPUT: return "DSA_ERR_BAD_INPUT";
    }
    return "unknown dsa_status";
}

const char* dsa_version(void) { return "0.1.0"; }

dsa_status dsa_workspace_size(const dsa_seqs* seqs, int32_t num_q, int32_t k, size_t* bytes) {
    Check c;
    check_seqs(c, seqs, num_q);
    c.need(bytes != nullptr, DSA_ERR_INVALID_ARG, "bytes is NULL");
    c.need(k >= 1 && k <= DSA_MAX_TOPK, DSA_ERR_UNSUPPORTED, "k %d outside [1, %d]", k, DSA_MAX_TOPK);
    dsa_status st = c.done();
    if (st != DSA_OK) return st;
    *bytes = workspace_bytes(*seqs, num_q, k, nullptr);
    return DSA_OK;
}

static void check_index_args(Check& c, const void* q_idx, const float* w, const float* ssmax_s, const float* ssmax_b,
                             const float* inv_freq, const void* k_idx, const float* k_scale, dsa_dtype k_dtype,
                             const void* k_block_scales = nullptr, float k_global = 0.f) {
    c.ptr(q_idx, "q_idx");
    c.ptr(w, "w", 4);
    c.ptr(ssmax_s, "ssmax_s", 4);
    c.ptr(ssmax_b, "ssmax_b", 4);
    if (inv_freq) c.ptr(inv_freq, "inv_freq", 4);
    c.ptr(k_idx, "k_idx");
    c.need(k_dtype == DSA_BF16 || k_dtype == DSA_FP8_E4M3_ROWSCALE || k_dtype == DSA_NVFP4, DSA_ERR_UNSUPPORTED,
           "index key dtype %d is not DSA_BF16, DSA_FP8_E4M3_ROWSCALE or DSA_NVFP4", (int)k_dtype);
    if (k_dtype == DSA_FP8_E4M3_ROWSCALE) c.ptr(k_scale, "k_scale", 4);
    if (k_dtype == DSA_NVFP4) {
        c.ptr(k_block_scales, "NVFP4 index key block scales", 16);
        c.need(k_global > 0.f && k_global < INFINITY, DSA_ERR_INVALID_ARG,
               "NVFP4 index key tensor scale must be positive and finite");
    }
}

static dsa_status index_scores_common(const char* name, const void* q_idx, const float* w, const float* ssmax_s,
                                      const float* ssmax_b, const float* inv_freq, const void* k_idx,
                                      const float* k_scale, dsa_dtype k_dtype, const void* k_block_scales,
                                      float k_global, const dsa_seqs* seqs, int32_t num_q, float* scores, int64_t ld,
                                      void* workspace, size_t workspace_bytes, int32_t* d_status,
                                      cudaStream_t stream) {
    Check c;
    check_seqs(c, seqs, num_q);
    check_index_args(c, q_idx, w, ssmax_s, ssmax_b, inv_freq, k_idx, k_scale, k_dtype, k_block_scales, k_global);
    c.ptr(scores, "scores");
    if (seqs) c.need(ld >= seqs->max_ctx && ld % 4 == 0, DSA_ERR_INVALID_ARG, "ld %lld must be >= max_ctx and a multiple of 4", (long long)ld);
    check_workspace(c, seqs, num_q, 1, workspace, workspace_bytes);
    dsa_status st = c.done();
    if (st != DSA_OK || num_q == 0) return st;
    Workspace ws = carve_workspace(workspace, *seqs, num_q, 1);
    return cuda_status(launch_index_scores(q_idx, w, ssmax_s, ssmax_b, inv_freq, k_idx, k_scale, k_dtype, *seqs,
                                           num_q, scores, ld, nullptr, 0, ws, d_status, stream, k_block_scales,
                                           k_global),
                       name);
}

dsa_status dsa_index_scores(const void* q_idx, const float* w, const float* ssmax_s, const float* ssmax_b,
                            const float* inv_freq, const void* k_idx, const float* k_scale, dsa_dtype k_dtype,
                            const dsa_seqs* seqs, int32_t num_q, float* scores, int64_t ld, void* workspace,
                            size_t workspace_bytes, int32_t* d_status, cudaStream_t stream) {
    if (k_dtype == DSA_NVFP4) {
        Check c;
        c.need(false, DSA_ERR_UNSUPPORTED, "NVFP4 index keys take dsa_index_scores_nvfp4");
        return c.done();
    }
    return index_scores_common("dsa_index_scores launch", q_idx, w, ssmax_s, ssmax_b, inv_freq, k_idx, k_scale,
                               k_dtype, nullptr, 0.f, seqs, num_q, scores, ld, workspace, workspace_bytes, d_status,
                               stream);
}

dsa_status dsa_index_scores_nvfp4(const void* q_idx, const float* w, const float* ssmax_s, const float* ssmax_b,
                                  const float* inv_freq, const void* k_codes, const void* k_block_scales,
                                  float k_global, const dsa_seqs* seqs, int32_t num_q, float* scores, int64_t ld,
                                  void* workspace, size_t workspace_bytes, int32_t* d_status, cudaStream_t stream) {
    return index_scores_common("dsa_index_scores_nvfp4 launch", q_idx, w, ssmax_s, ssmax_b, inv_freq, k_codes,
                               nullptr, DSA_NVFP4, k_block_scales, k_global, seqs, num_q, scores, ld, workspace,
                               workspace_bytes, d_status, stream);
}

dsa_status dsa_index_k_insert(const void* x, const float* ln_gamma, const float* ln_beta, float ln_eps,
                              const int32_t* pos, const float* inv_freq, const int64_t* slot, int32_t n,
                              void* k_cache, float* k_scale, dsa_dtype k_dtype, int64_t num_rows, int32_t* d_status,
                              cudaStream_t stream) {
    Check c;
    c.need(n >= 0, DSA_ERR_INVALID_ARG, "n %d < 0", n);
    c.need(num_rows >= 1, DSA_ERR_INVALID_ARG, "num_rows %lld < 1", (long long)num_rows);
    c.need(k_dtype == DSA_BF16 || k_dtype == DSA_FP8_E4M3_ROWSCALE, DSA_ERR_UNSUPPORTED,
           "k_dtype %d is neither DSA_BF16 nor DSA_FP8_E4M3_ROWSCALE", (int)k_dtype);
    c.need(ln_eps >= 0.f, DSA_ERR_INVALID_ARG, "ln_eps must be >= 0");
    if (n > 0) {
        c.ptr(x, "x");
        c.ptr(ln_gamma, "ln_gamma");
        c.ptr(ln_beta, "ln_beta");
        c.ptr(pos, "pos", 4);
        c.ptr(slot, "slot", 8);
        c.ptr(k_cache, "k_cache");
        if (inv_freq) c.ptr(inv_freq, "inv_freq");  // read as float4
        if (k_dtype == DSA_FP8_E4M3_ROWSCALE) c.ptr(k_scale, "k_scale", 4);
    }
    dsa_status st = c.done();
    if (st != DSA_OK || n == 0) return st;
    return cuda_status(launch_index_k_insert(x, ln_gamma, ln_beta, ln_eps, pos, inv_freq, slot, n, k_cache, k_scale,
                                             k_dtype == DSA_FP8_E4M3_ROWSCALE, num_rows, d_status, stream),
                       "dsa_index_k_insert launch");
}

dsa_status dsa_latent_insert(const void* c_kv, const void* k_pe, const int32_t* pos, const float* inv_freq,
                             const int64_t* slot, int32_t n, void* latent, dsa_dtype latent_dtype, int64_t num_rows,
                             int32_t* d_status, cudaStream_t stream) {
    Check c;
    c.need(n >= 0, DSA_ERR_INVALID_ARG, "n %d < 0", n);
    c.need(num_rows >= 1, DSA_ERR_INVALID_ARG, "num_rows %lld < 1", (long long)num_rows);
    c.need(latent_dtype == DSA_BF16 || latent_dtype == DSA_FP8_DS_MLA, DSA_ERR_UNSUPPORTED,
           "latent_dtype %d is neither DSA_BF16 nor DSA_FP8_DS_MLA", (int)latent_dtype);
    if (n > 0) {
        c.ptr(c_kv, "c_kv");
        c.ptr(k_pe, "k_pe");
        c.ptr(pos, "pos", 4);
        c.ptr(slot, "slot", 8);
        c.ptr(latent, "latent");
        if (inv_freq) c.ptr(inv_freq, "inv_freq", 4);
    }
    dsa_status st = c.done();
    if (st != DSA_OK || n == 0) return st;
    return cuda_status(launch_latent_insert(c_kv, k_pe, pos, inv_freq, slot, n, latent,
                                            latent_dtype == DSA_FP8_DS_MLA, num_rows, d_status, stream),
                       "dsa_latent_insert launch");
}

dsa_status dsa_mla_q_prep(const void* q, const float* ssmax_s, const float* ssmax_b, const float* inv_freq,
                          const int32_t* q_pos, int32_t num_q, void* q_out, int32_t* d_status, cudaStream_t stream) {
    Check c;
    c.need(num_q >= 0, DSA_ERR_INVALID_ARG, "num_q %d < 0", num_q);
    if (num_q > 0) {
        c.ptr(q, "q");
        c.ptr(ssmax_s, "ssmax_s", 4);
        c.ptr(ssmax_b, "ssmax_b", 4);
        c.ptr(q_pos, "q_pos", 4);
        c.ptr(q_out, "q_out");
        if (inv_freq) c.ptr(inv_freq, "inv_freq", 4);
    }
    dsa_status st = c.done();
    if (st != DSA_OK || num_q == 0) return st;
    return cuda_status(launch_mla_q_prep(q, ssmax_s, ssmax_b, inv_freq, q_pos, num_q, q_out, d_status, stream),
                       "dsa_mla_q_prep launch");
}

dsa_status dsa_topk(const float* scores, int64_t ld, const dsa_seqs* seqs, int32_t num_q, int32_t k, int32_t* idx,
                    int32_t* topk_len, void* workspace, size_t workspace_bytes, int32_t* d_status,
                    cudaStream_t stream) {
    Check c;
    check_seqs(c, seqs, num_q);
    c.ptr(scores, "scores");
    c.ptr(idx, "idx", 4);
    c.ptr(topk_len, "topk_len", 4);
    c.need(k >= 1 && k <= DSA_MAX_TOPK, DSA_ERR_UNSUPPORTED, "k %d outside [1, %d]", k, DSA_MAX_TOPK);
    if (seqs) c.need(ld >= seqs->max_ctx && ld % 4 == 0, DSA_ERR_INVALID_ARG, "ld %lld must be >= max_ctx and a multiple of 4", (long long)ld);
    (void)workspace;  // no scratch at any row length
    (void)workspace_bytes;
    dsa_status st = c.done();
    if (st != DSA_OK || num_q == 0) return st;
    return cuda_status(launch_topk(scores, ld, *seqs, num_q, k, idx, topk_len, Workspace{}, d_status, stream),
                       "dsa_topk launch");
}

dsa_status dsa_topk_candidates(const float* scores, int64_t ld, const dsa_seqs* seqs, int32_t num_q, int32_t k,
                               const dsa_dcp_shard* shard, int32_t* idx, int32_t* topk_len, uint64_t* cand,
                               void* workspace, size_t workspace_bytes, int32_t* d_status, cudaStream_t stream) {
    Check c;
    check_seqs(c, seqs, num_q);
    check_shard(c, shard);
    c.ptr(scores, "scores");
    c.ptr(idx, "idx", 4);
    c.ptr(topk_len, "topk_len", 4);
    c.ptr(cand, "cand", 8);
    c.need(k >= 1 && k <= DSA_MAX_TOPK, DSA_ERR_UNSUPPORTED, "k %d outside [1, %d]", k, DSA_MAX_TOPK);
    if (seqs) c.need(ld >= seqs->max_ctx && ld % 4 == 0, DSA_ERR_INVALID_ARG, "ld %lld must be >= max_ctx and a multiple of 4", (long long)ld);
    (void)workspace;  // no scratch at any row length
    (void)workspace_bytes;
    dsa_status st = c.done();
    if (st != DSA_OK || num_q == 0) return st;
    cudaError_t e = launch_topk(scores, ld, *seqs, num_q, k, idx, topk_len, Workspace{}, d_status, stream);
    if (e == cudaSuccess)
        e = launch_cand_pack(scores, ld, idx, topk_len, num_q, k, shard->world, shard->rank, shard->interleave, cand,
                             d_status, stream);
    return cuda_status(e, "dsa_topk_candidates launch");
}

dsa_status dsa_topk_merge(const uint64_t* const* lists, int32_t num_lists, int32_t list_len, int32_t num_q,
                          int32_t k, int32_t* idx, int32_t* topk_len, int32_t* d_status, cudaStream_t stream) {
    Check c;
    c.need(num_q >= 0, DSA_ERR_INVALID_ARG, "num_q %d < 0", num_q);
    c.need(lists != nullptr, DSA_ERR_INVALID_ARG, "lists (host array) is NULL");
    c.need(num_lists >= 1 && num_lists <= DSA_DCP_MAX_RANKS, DSA_ERR_UNSUPPORTED, "num_lists %d outside [1, %d]",
           num_lists, DSA_DCP_MAX_RANKS);
    c.need(list_len >= 1, DSA_ERR_INVALID_ARG, "list_len %d < 1", list_len);
    c.need((int64_t)num_lists * list_len <= DSA_DCP_MAX_CANDIDATES, DSA_ERR_UNSUPPORTED,
           "num_lists x list_len = %lld exceeds %d", (long long)num_lists * list_len, DSA_DCP_MAX_CANDIDATES);
    c.need(k >= 1 && k <= DSA_MAX_TOPK, DSA_ERR_UNSUPPORTED, "k %d outside [1, %d]", k, DSA_MAX_TOPK);
    if (num_q > 0) {
        if (lists && num_lists >= 1 && num_lists <= DSA_DCP_MAX_RANKS)
            for (int r = 0; r < num_lists; ++r) c.ptr(lists[r], "lists[r]", 8);
        c.ptr(idx, "idx", 4);
        c.ptr(topk_len, "topk_len", 4);
    }
    dsa_status st = c.done();
    if (st != DSA_OK || num_q == 0) return st;
    return cuda_status(launch_topk_merge(lists, num_lists, list_len, num_q, k, idx, topk_len, d_status, stream),
                       "dsa_topk_merge launch");
}

dsa_status dsa_topk_compact(const int32_t* idx, const int32_t* topk_len, int32_t num_q, int32_t k,
                            const dsa_dcp_shard* shard, int32_t* local_idx, int32_t* local_len, int32_t* d_status,
                            cudaStream_t stream) {
    Check c;
    c.need(num_q >= 0, DSA_ERR_INVALID_ARG, "num_q %d < 0", num_q);
    c.need(k >= 1 && k <= DSA_MAX_TOPK, DSA_ERR_UNSUPPORTED, "k %d outside [1, %d]", k, DSA_MAX_TOPK);
    check_shard(c, shard);
    if (num_q > 0) {
        c.ptr(idx, "idx", 4);
        c.ptr(topk_len, "topk_len", 4);
        c.ptr(local_idx, "local_idx", 4);
        c.ptr(local_len, "local_len", 4);
    }
    dsa_status st = c.done();
    if (st != DSA_OK || num_q == 0) return st;
    return cuda_status(launch_topk_compact(idx, topk_len, num_q, k, shard->world, shard->rank, shard->interleave,
                                           local_idx, local_len, d_status, stream),
                       "dsa_topk_compact launch");
}

dsa_status dsa_dcp_shard_seqs(const dsa_seqs* seqs, int32_t num_q, const dsa_dcp_shard* shard,
                              int32_t* local_ctx_len, int32_t* local_q_pos, int32_t* local_page_table,
                              int32_t local_max_pages, int32_t* local_max_ctx, int32_t* d_status,
                              cudaStream_t stream) {
    Check c;
    check_seqs(c, seqs, num_q);
    check_shard(c, shard);
    c.ptr(local_ctx_len, "local_ctx_len", 4);
    if (num_q > 0) c.ptr(local_q_pos, "local_q_pos", 4);
    c.need(local_max_ctx != nullptr, DSA_ERR_INVALID_ARG, "local_max_ctx (host) is NULL");
    int64_t lmax = 0;
    if (seqs && c.st == DSA_OK) lmax = dcp_owned_tokens(seqs->max_ctx, shard->world, shard->rank, shard->interleave);
    if (local_page_table && seqs && c.st == DSA_OK) {
        c.ptr(local_page_table, "local_page_table", 4);
        c.need(seqs->page_table != nullptr, DSA_ERR_INVALID_ARG, "local_page_table needs seqs.page_table");
        c.need(seqs->page_size >= 1 && shard->interleave % seqs->page_size == 0, DSA_ERR_UNSUPPORTED,
               "interleave %d is not a whole number of %d-token pages", shard->interleave, seqs->page_size);
        if (seqs->page_size >= 1)
            c.need((int64_t)local_max_pages * seqs->page_size >= lmax, DSA_ERR_INVALID_ARG,
                   "local_max_pages %d x page_size %d < %lld local tokens", local_max_pages, seqs->page_size,
                   (long long)lmax);
    }
    dsa_status st = c.done();
    if (st != DSA_OK) return st;
    *local_max_ctx = (int32_t)(lmax < 1 ? 1 : lmax);
    return cuda_status(launch_dcp_shard_seqs(*seqs, num_q, shard->world, shard->rank, shard->interleave,
                                             local_ctx_len, local_q_pos, local_page_table, local_max_pages, d_status,
                                             stream),
                       "dsa_dcp_shard_seqs launch");
}

dsa_status dsa_lse_combine(const void* const* o_parts, const float* const* lse_parts, int32_t num_parts,
                           int32_t num_q, void* out, float* lse, cudaStream_t stream) {
    Check c;
    c.need(num_q >= 0, DSA_ERR_INVALID_ARG, "num_q %d < 0", num_q);
    c.need(o_parts != nullptr && lse_parts != nullptr, DSA_ERR_INVALID_ARG, "o_parts / lse_parts (host arrays) NULL");
    c.need(num_parts >= 1 && num_parts <= DSA_DCP_MAX_RANKS, DSA_ERR_UNSUPPORTED, "num_parts %d outside [1, %d]",
           num_parts, DSA_DCP_MAX_RANKS);
    if (num_q > 0) {
        if (o_parts && lse_parts && num_parts >= 1 && num_parts <= DSA_DCP_MAX_RANKS)
            for (int r = 0; r < num_parts; ++r) {
                c.ptr(o_parts[r], "o_parts[r]");
                c.ptr(lse_parts[r], "lse_parts[r]", 4);
            }
        c.ptr(out, "out");
        if (lse) c.ptr(lse, "lse", 4);
    }
    dsa_status st = c.done();
    if (st != DSA_OK || num_q == 0) return st;
    return cuda_status(launch_lse_combine(o_parts, lse_parts, num_parts, num_q, out, lse, stream),
                       "dsa_lse_combine launch");
}

dsa_status dsa_block_topk(const float* scores, int64_t ld, const dsa_seqs* seqs, int32_t num_q, int32_t block,
                          int32_t nsel, int32_t* idx, int32_t* topk_len, int32_t* d_status, cudaStream_t stream) {
    Check c;
    check_seqs(c, seqs, num_q);
    c.ptr(scores, "scores");
    c.ptr(idx, "idx", 4);
    c.ptr(topk_len, "topk_len", 4);
    c.need(block >= 1 && nsel >= 1 && nsel <= DSA_BLOCK_TOPK_MAX_NSEL, DSA_ERR_UNSUPPORTED,
           "block %d must be >= 1 and nsel %d in [1, %d]", block, nsel, DSA_BLOCK_TOPK_MAX_NSEL);
    c.need((int64_t)block * nsel <= DSA_MAX_TOPK, DSA_ERR_UNSUPPORTED, "nsel x block = %lld exceeds %d",
           (long long)block * nsel, DSA_MAX_TOPK);
    if (seqs) {
        c.need(ld >= seqs->max_ctx && ld % 4 == 0, DSA_ERR_INVALID_ARG, "ld %lld must be >= max_ctx and a multiple of 4",
               (long long)ld);
        if (block >= 1 && nsel >= 1 && seqs->max_ctx >= 1)
            c.need(block_topk_smem(seqs->max_ctx, block, nsel) <= DSA_BLOCK_TOPK_MAX_SMEM, DSA_ERR_UNSUPPORTED,
                   "max_ctx %d / block %d: too many blocks for one CTA's shared memory", seqs->max_ctx, block);
    }
    dsa_status st = c.done();
    if (st != DSA_OK || num_q == 0) return st;
    return cuda_status(launch_block_topk(scores, ld, *seqs, num_q, block, nsel, idx, topk_len, d_status, stream),
                       "dsa_block_topk launch");
}

static void check_mla_args(Check& c, const void* q, const void* latent, dsa_dtype latent_dtype, const int32_t* idx,
                           const int32_t* topk_len, int32_t k, float sm_scale, const void* out, const float* lse,
                           const void* lat_scales = nullptr, float lat_global = 0.f) {
    c.ptr(q, "q");
    c.ptr(latent, "latent");
    c.need(latent_dtype == DSA_BF16 || latent_dtype == DSA_FP8_DS_MLA || latent_dtype == DSA_NVFP4,
           DSA_ERR_UNSUPPORTED, "latent dtype %d is not DSA_BF16, DSA_FP8_DS_MLA or DSA_NVFP4", (int)latent_dtype);
    if (latent_dtype == DSA_NVFP4) {
        c.ptr(lat_scales, "NVFP4 latent block scales", 4);
        c.need(lat_global > 0.f && lat_global < 1e30f, DSA_ERR_INVALID_ARG,
               "NVFP4 latent tensor scale must be positive and finite");
    }
    c.ptr(idx, "idx", 4);
    c.ptr(topk_len, "topk_len", 4);
    c.need(k >= 1 && k <= DSA_MAX_TOPK, DSA_ERR_UNSUPPORTED, "k %d outside [1, %d]", k, DSA_MAX_TOPK);
    c.need(sm_scale > 0.f && sm_scale < 1e30f, DSA_ERR_INVALID_ARG, "sm_scale must be positive and finite");
    c.ptr(out, "out");
    if (lse) c.ptr(lse, "lse", 4);
}

dsa_status sparse_mla_decode(const void* q, const void* latent, dsa_dtype latent_dtype, const dsa_seqs* seqs,
                             int32_t num_q, const int32_t* idx, const int32_t* topk_len, int32_t k, float sm_scale,
                             void* out, float* lse, void* workspace, size_t workspace_bytes, int32_t* d_status,
                             cudaStream_t stream) {
    Check c;
    check_seqs(c, seqs, num_q);
    c.need(latent_dtype != DSA_NVFP4, DSA_ERR_UNSUPPORTED, "an NVFP4 latent cache takes sparse_mla_decode_nvfp4");
    check_mla_args(c, q, latent, latent_dtype, idx, topk_len, k, sm_scale, out, lse);
    check_workspace(c, seqs, num_q, k, workspace, workspace_bytes);
    dsa_status st = c.done();
    if (st != DSA_OK || num_q == 0) return st;
    Workspace ws = carve_workspace(workspace, *seqs, num_q, k);
    return cuda_status(launch_sparse_mla(q, latent, latent_dtype, *seqs, num_q, idx, topk_len, k, sm_scale, out, lse,
                                         ws, d_status, stream),
                       "sparse_mla_decode launch");
}

// the block-sparse selection mode of dsa_decode_layer: k / select_block
// blocks, within dsa_block_topk's limits
static void check_block_select(Check& c, const dsa_seqs* seqs, int32_t k, int32_t block) {
    c.need(block >= 0, DSA_ERR_INVALID_ARG, "select_block %d < 0", block);
    if (block <= 0) return;
    c.need(k % block == 0, DSA_ERR_UNSUPPORTED, "k %d is not a multiple of select_block %d", k, block);
    const int nsel = k / block;
    c.need(nsel >= 1 && nsel <= DSA_BLOCK_TOPK_MAX_NSEL, DSA_ERR_UNSUPPORTED,
           "k / select_block = %d blocks outside [1, %d]", nsel, DSA_BLOCK_TOPK_MAX_NSEL);
    if (seqs && seqs->max_ctx >= 1 && nsel >= 1)
        c.need(block_topk_smem(seqs->max_ctx, block, nsel) <= DSA_BLOCK_TOPK_MAX_SMEM, DSA_ERR_UNSUPPORTED,
               "max_ctx %d / select_block %d: too many blocks for one CTA's shared memory", seqs->max_ctx, block);
}

static void check_layer(Check& c, const dsa_layer_args* a, const dsa_seqs* seqs, int32_t num_q) {
    check_seqs(c, seqs, num_q);
    if (!a->reuse_idx) {
        check_index_args(c, a->q_idx, a->w, a->ssmax_s, a->ssmax_b, a->inv_freq, a->k_idx, a->k_scale, a->k_dtype,
                         a->k_block_scales, a->k_global);
        check_block_select(c, seqs, a->k, a->select_block);
    }
    check_mla_args(c, a->q_mla, a->latent, a->latent_dtype, a->idx, a->topk_len, a->k, a->sm_scale, a->out, a->lse,
                   a->latent_scales, a->latent_global);
}

dsa_status sparse_mla_decode_nvfp4(const void* q, const void* codes, const void* block_scales, float g,
                                   const dsa_seqs* seqs, int32_t num_q, const int32_t* idx, const int32_t* topk_len,
                                   int32_t k, float sm_scale, void* out, float* lse, void* workspace,
                                   size_t workspace_bytes, int32_t* d_status, cudaStream_t stream) {
    Check c;
    check_seqs(c, seqs, num_q);
    check_mla_args(c, q, codes, DSA_NVFP4, idx, topk_len, k, sm_scale, out, lse, block_scales, g);
    check_workspace(c, seqs, num_q, k, workspace, workspace_bytes);
    dsa_status st = c.done();
    if (st != DSA_OK || num_q == 0) return st;
    Workspace ws = carve_workspace(workspace, *seqs, num_q, k);
    return cuda_status(launch_sparse_mla(q, codes, DSA_NVFP4, *seqs, num_q, idx, topk_len, k, sm_scale, out, lse, ws,
                                         d_status, stream, kNoCap, block_scales, g),
                       "sparse_mla_decode_nvfp4 launch");
}

dsa_status dsa_decode_layer(const dsa_layer_args* a, const dsa_seqs* seqs, int32_t num_q, void* workspace,
                            size_t workspace_bytes, int32_t* d_status, cudaStream_t stream) {
    Check c;
    c.need(a != nullptr, DSA_ERR_INVALID_ARG, "args is NULL");
    if (!a) return c.done();
    check_layer(c, a, seqs, num_q);
    check_workspace(c, seqs, num_q, a->k, workspace, workspace_bytes);
    dsa_status st = c.done();
    if (st != DSA_OK || num_q == 0) return st;
    Workspace ws = carve_workspace(workspace, *seqs, num_q, a->k);
    cudaError_t e = cudaSuccess;
    auto mark = [&](int i) {
        if (a->events && e == cudaSuccess) e = cudaEventRecord(a->events[i], stream);
    };
    mark(0);
    if (!a->reuse_idx) {
        // block selection with blocks of whole 32-key groups needs only the
        // groups' maxima: the indexer writes those (1/32 of the row) in place
        // of the scores
        const bool groups = a->select_block > 0 && a->select_block % 32 == 0;
        const int64_t ldg = (((int64_t)seqs->max_ctx + 31) / 32 + 3) / 4 * 4;
        if (e == cudaSuccess)
            e = launch_index_scores(a->q_idx, a->w, a->ssmax_s, a->ssmax_b, a->inv_freq, a->k_idx, a->k_scale,
                                    a->k_dtype, *seqs, num_q, groups ? nullptr : ws.scores, ws.scores_ld,
                                    groups ? ws.scores : nullptr, ldg, ws, d_status, stream, a->k_block_scales,
                                    a->k_global);
        mark(1);
        if (e == cudaSuccess) {
            if (a->select_block > 0)
                e = launch_block_topk(ws.scores, groups ? ldg : ws.scores_ld, *seqs, num_q, a->select_block,
                                      a->k / a->select_block, a->idx, a->topk_len, d_status, stream, groups);
            else
                e = launch_topk(ws.scores, ws.scores_ld, *seqs, num_q, a->k, a->idx, a->topk_len, ws, d_status,
                                stream);
        }
        mark(2);
    } else {
        mark(1);
        mark(2);
    }
    if (e == cudaSuccess)
        e = launch_sparse_mla(a->q_mla, a->latent, a->latent_dtype, *seqs, num_q, a->idx, a->topk_len, a->k,
                              a->sm_scale, a->out, a->lse, ws, d_status, stream, kNoCap, a->latent_scales,
                              a->latent_global);
    mark(3);
    return cuda_status(e, "dsa_decode_layer launch");
}

int32_t dsa_decode_layer_launches(const dsa_seqs* seqs, int32_t num_q, int32_t k, int32_t reuse_idx,
                                  dsa_dtype latent_dtype) {
    Check c;
    check_seqs(c, seqs, num_q);
    c.need(k >= 1 && k <= DSA_MAX_TOPK, DSA_ERR_UNSUPPORTED, "k %d outside [1, %d]", k, DSA_MAX_TOPK);
    c.need(latent_dtype == DSA_BF16 || latent_dtype == DSA_FP8_DS_MLA, DSA_ERR_INVALID_ARG, "latent_dtype %d",
           (int)latent_dtype);
    if (c.done() != DSA_OK || num_q == 0) return 0;
    return layer_launches(*seqs, num_q, k, reuse_idx != 0, 0);
}

int32_t dsa_decode_layer_launches_for(const dsa_layer_args* a, const dsa_seqs* seqs, int32_t num_q) {
    Check c;
    c.need(a != nullptr, DSA_ERR_INVALID_ARG, "args is NULL");
    if (!a) return 0;
    check_seqs(c, seqs, num_q);
    c.need(a->k >= 1 && a->k <= DSA_MAX_TOPK, DSA_ERR_UNSUPPORTED, "k %d outside [1, %d]", a->k, DSA_MAX_TOPK);
    c.need(a->latent_dtype == DSA_BF16 || a->latent_dtype == DSA_FP8_DS_MLA || a->latent_dtype == DSA_NVFP4,
           DSA_ERR_INVALID_ARG, "latent_dtype %d", (int)a->latent_dtype);
    if (!a->reuse_idx) check_block_select(c, seqs, a->k, a->select_block);
    if (c.done() != DSA_OK || num_q == 0) return 0;
    return layer_launches(*seqs, num_q, a->k, a->reuse_idx != 0, a->reuse_idx ? 0 : a->select_block);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// sparse_mla_decode_noalloc: the attention's split-K partials in a
// library-owned static device array instead of a caller workspace.
namespace dsa {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the static array on the current device, looked up once
// per device with that device current.
cudaError_t noalloc_scratch(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status sparse_mla_decode_noalloc(const void* q, const void* latent, dsa_dtype latent_dtype,
                                                const dsa_seqs* seqs, int32_t num_q, const int32_t* idx,
                                                const int32_t* topk_len, int32_t k, float sm_scale, void* out,
                                                float* lse, int32_t* d_status, cudaStream_t stream) {
    Check c;
    check_seqs(c, seqs, num_q);
    c.need(latent_dtype != DSA_NVFP4, DSA_ERR_UNSUPPORTED, "no no-workspace entry point for an NVFP4 latent cache");
    check_mla_args(c, q, latent, latent_dtype, idx, topk_len, k, sm_scale, out, lse);
    // the split count is held so that the partials fit the static array
    // (fewer splits than sparse_mla_decode on some batches; no size refused:
    // one split or a two-split cluster pair needs no scratch)
    const size_t cap = DSA_NOALLOC_SCRATCH_BYTES;
    size_t part_bytes = 0, ml_bytes = 0;
    if (c.st == DSA_OK && num_q > 0) {
        part_bytes = up256(mla_part_bytes(num_q, k, cap));
        ml_bytes = up256(mla_ml_bytes(num_q, k, cap));
        c.need(part_bytes + ml_bytes <= cap, DSA_ERR_UNSUPPORTED,
               "%d queries need %zu bytes of scratch; the static scratch holds %zu", num_q, part_bytes + ml_bytes,
               cap);
    }
    dsa_status st = c.done();
    if (st != DSA_OK || num_q == 0) return st;
    void* base = nullptr;
    cudaError_t e = noalloc_scratch(&base);
    if (e != cudaSuccess) return cuda_status(e, "sparse_mla_decode_noalloc scratch address");
    Workspace ws{};
    ws.mla_part = reinterpret_cast<float*>(base);
    ws.mla_ml = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(base) + part_bytes);
    return cuda_status(launch_sparse_mla(q, latent, latent_dtype, *seqs, num_q, idx, topk_len, k, sm_scale, out, lse,
                                         ws, d_status, stream, cap),
                       "sparse_mla_decode_noalloc launch");
}
