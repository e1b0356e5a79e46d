// dcp.cu -- one rank's compute steps of decode context parallelism (sm_103a).
//
// [vLLM-ML4] "Day 0 support for Mistral Large 4", Long context: decode and
// prefill context parallelism.  The latent cache is sharded by token; each
// rank pushes its packed (score, id) top-k candidates to its peers and a
// selector merges them in place; each rank compacts the global top-k slots it
// owns and bounds its attention with topk_length (a rank owning none of a
// query's slots gets an empty row: out 0, lse -inf); the ranks' partial
// outputs are merged by an LSE combine.  The exchange itself belongs to the
// caller; these are the kernels on either side of it.
//
// Ownership: turns of `interleave` tokens go round the ranks, so token t lives
// on rank (t / I) mod R at local position (t / (I R)) I + t mod I.
#include <mutex>

#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kMaxLists = 16;         // ranks (lists, parts) per call
constexpr int kMergeMaxCand = 16384;  // candidates per query in the selector (128 KB of shared memory)
constexpr int kMergeThreads = 512;

struct ListPtrs {
    const uint64_t* p[kMaxLists];
};

struct PartPtrs {
    const __nv_bfloat16* o[kMaxLists];
    const float* l[kMaxLists];
};

// order-preserving code of a score: negative values below positive ones, and
// among negatives the larger magnitude lower; -0 coded as +0
__device__ __forceinline__ uint32_t score_code(float s) {
    const uint32_t b = __float_as_uint(s == 0.f ? 0.f : s);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// a larger packed value: a larger score, or at equal scores a smaller id
__device__ __forceinline__ uint64_t pack_cand(float s, uint32_t id) {
    return ((uint64_t)score_code(s) << 32) | (uint64_t)(0xFFFFFFFFu - id);
}

__device__ __forceinline__ int32_t cand_id(uint64_t c) { return (int32_t)(0xFFFFFFFFu - (uint32_t)c); }

// ---------------------------------------------------------------------------
// A rank's candidates: slot i < topk_len of its local top-k packed with its
// score and its global id.  Grid: (queries, ceil(k / 256)).
__global__ void __launch_bounds__(256) cand_pack_kernel(const float* __restrict__ scores, int64_t ld,
                                                        const int32_t* __restrict__ idx,
                                                        const int32_t* __restrict__ topk_len, int k, int world,
                                                        int rank, int inter, uint64_t* __restrict__ cand,
                                                        int32_t* d_status) {
    pdl_enter();
    const int t = blockIdx.x;
    const int i = blockIdx.y * 256 + threadIdx.x;
    if (i >= k) return;
    const int len = __ldg(topk_len + t);
    uint64_t c = 0;
    if (i < len) {
        const int l = __ldg(idx + (int64_t)t * k + i);
        if (l >= 0) {
            const int64_t g = ((int64_t)(l / inter) * world + rank) * inter + l % inter;
            if (g <= INT32_MAX) {
                c = pack_cand(__ldg(scores + (int64_t)t * ld + l), (uint32_t)g);
            } else {
                report(d_status, DSA_ERR_BAD_INPUT);
            }
        }
    }
    cand[(int64_t)t * k + i] = c;
}

// ---------------------------------------------------------------------------
// The selector: one CTA per query.  Every candidate of the query's lists goes
// to shared memory; an MSB-first radix select over the 64-bit packed values
// (eight 8-bit digits) finds the kk-th largest, kk = min(k, candidates); the
// ids of the values at or above it are sorted ascending (bitonic).  Distinct
// ids make distinct packed values, so exactly kk are selected; a duplicate
// among them is reported and the query's row left empty.
__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(ListPtrs lists, int num_lists, int list_len,
                                                                   int k, int32_t* __restrict__ idx,
                                                                   int32_t* __restrict__ topk_len,
                                                                   int32_t* d_status) {
    extern __shared__ __align__(16) uint64_t vals[];  // [num_lists * list_len], then the selected ids
    __shared__ int hist[256];
    __shared__ int s_count, s_digit, s_rem, s_dup;
    const int total = num_lists * list_len;
    int* sel = reinterpret_cast<int*>(vals + total);
    const int t = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_enter();
    if (tid == 0) {
        s_count = 0;
        s_dup = 0;
    }
    __syncthreads();
    int nz = 0;
    for (int j = tid; j < total; j += kMergeThreads) {
        const int r = j / list_len, i = j - r * list_len;
        const uint64_t v = __ldg(lists.p[r] + (int64_t)t * list_len + i);
        vals[j] = v;
        nz += v != 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nz += __shfl_xor_sync(0xffffffffu, nz, o);
    if (lane == 0) atomicAdd(&s_count, nz);
    __syncthreads();
    const int kk = min(k, s_count);
    __syncthreads();
    uint64_t prefix = 0, mask = 0;
    int rem = kk;
    for (int pass = 0; pass < 8 && kk > 0; ++pass) {
        const int shift = 56 - 8 * pass;
        if (tid < 256) hist[tid] = 0;
        __syncthreads();
        for (int j = tid; j < total; j += kMergeThreads) {
            const uint64_t v = vals[j];
            if (v != 0 && (v & mask) == prefix) atomicAdd(&hist[(int)(v >> shift) & 0xFF], 1);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l holds digits 255 - 8l .. 248 - 8l (descending)
            int c[8], sum = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                c[e] = hist[255 - 8 * lane - e];
                sum += c[e];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            const int above = incl - sum;  // values in higher digits
            if (above < rem && rem <= incl) {
                int cum = above;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (cum + c[e] >= rem) {
                        s_digit = 255 - 8 * lane - e;
                        s_rem = rem - cum;
                        break;
                    }
                    cum += c[e];
                }
            }
        }
        __syncthreads();
        prefix |= (uint64_t)s_digit << shift;
        mask |= (uint64_t)0xFF << shift;
        rem = s_rem;
        __syncthreads();
    }
    // collect the ids at or above the kk-th largest value
    if (tid == 0) s_count = 0;
    __syncthreads();
    if (kk > 0) {
        for (int j = tid; j < total; j += kMergeThreads) {
            const uint64_t v = vals[j];
            if (v != 0 && v >= prefix) {
                const int p = atomicAdd(&s_count, 1);
                if (p < k) sel[p] = cand_id(v);
            }
        }
    }
    __syncthreads();
    const int got = s_count;
    bool bad = got != kk;  // more than kk: a repeated value, so a repeated id
    int P = 1;
    while (P < kk) P <<= 1;
    if (!bad) {
        for (int j = kk + tid; j < P; j += kMergeThreads) sel[j] = INT32_MAX;
        __syncthreads();
        for (int size = 2; size <= P; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int j = tid; j < P / 2; j += kMergeThreads) {
                    const int a = 2 * j - (j & (stride - 1));
                    const int b = a + stride;
                    const bool up = (a & size) == 0;
                    const int x = sel[a], y = sel[b];
                    if ((x > y) == up) {
                        sel[a] = y;
                        sel[b] = x;
                    }
                }
                __syncthreads();
            }
        }
        for (int j = tid + 1; j < kk; j += kMergeThreads)
            if (sel[j] == sel[j - 1]) s_dup = 1;
        __syncthreads();
        bad = s_dup != 0;
    }
    if (bad && tid == 0) report(d_status, DSA_ERR_BAD_INPUT);
    const int len = bad ? 0 : kk;
    for (int j = tid; j < k; j += kMergeThreads) idx[(int64_t)t * k + j] = j < len ? sel[j] : -1;
    if (tid == 0) topk_len[t] = len;
}

// ---------------------------------------------------------------------------
// Top-k compaction for one rank: the slots i < topk_len holding an id >= 0
// that the rank owns, in order, as local positions; the rest of the row -1.
// One CTA of 256 threads per query, thread i holding the 8 consecutive slots
// 8i .. 8i + 7 (k <= 2048): every slot is read before the block's prefix sum
// and written after it, so the output may be the input.
constexpr int kCompactThreads = 256;
constexpr int kCompactPer = DSA_MAX_TOPK / kCompactThreads;  // 8

__global__ void __launch_bounds__(kCompactThreads) topk_compact_kernel(const int32_t* idx, const int32_t* topk_len,
                                                                       int num_q, int k, int world, int rank,
                                                                       int inter, int32_t* local_idx,
                                                                       int32_t* local_len, int32_t* d_status) {
    pdl_enter();
    __shared__ int wsum[kCompactThreads / 32];
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int len = topk_len[t];
    if (len < 0 || len > k) {
        if (tid == 0) report(d_status, DSA_ERR_BAD_INPUT);
        len = len < 0 ? 0 : k;
    }
    const int32_t* in = idx + (int64_t)t * k;
    int32_t* out = local_idx + (int64_t)t * k;
    int loc[kCompactPer];
    int c = 0;
#pragma unroll
    for (int u = 0; u < kCompactPer; ++u) {
        const int i = tid * kCompactPer + u;
        const int id = i < len ? in[i] : -1;
        const bool own = id >= 0 && (id / inter) % world == rank;
        loc[u] = own ? (id / inter / world) * inter + id % inter : -1;
        c += own;
    }
    // exclusive prefix of the owned counts over the block
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();  // every slot has been read
    int before = x - c, total = 0;
#pragma unroll
    for (int w = 0; w < kCompactThreads / 32; ++w) {
        before += w < warp ? wsum[w] : 0;
        total += wsum[w];
    }
#pragma unroll
    for (int u = 0; u < kCompactPer; ++u)
        if (loc[u] >= 0) out[before++] = loc[u];
    for (int i = total + tid; i < k; i += kCompactThreads) out[i] = -1;
    if (tid == 0) local_len[t] = total;
}

// ---------------------------------------------------------------------------
// LSE combine: one warp per (query, head).  Lane r < R holds part r's lse;
// weights exp(lse_r - L), L = ln sum_r exp(lse_r); parts at -inf are skipped.
// Lane l sums dims 16l..16l+15 over the parts.
__global__ void __launch_bounds__(128) lse_combine_kernel(PartPtrs parts, int num_parts, int num_q,
                                                          __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int64_t wi = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (wi >= (int64_t)num_q * kMH) return;
    const float lr = lane < num_parts ? __ldg(parts.l[lane] + wi) : -INFINITY;
    float m = lr;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
    float L = -INFINITY;
    if (m != -INFINITY) {
        float e = lr == -INFINITY ? 0.f : expf(lr - m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
        L = m + logf(e);
        const float wr = lr == -INFINITY ? 0.f : expf(lr - L);
        for (int r = 0; r < num_parts; ++r) {
            const float w = __shfl_sync(0xffffffffu, wr, r);
            if (w == 0.f) continue;  // a part at -inf (an empty row) adds nothing
            const uint4* src = reinterpret_cast<const uint4*>(parts.o[r] + wi * kMV) + 2 * lane;
            const uint4 a = __ldg(src), b = __ldg(src + 1);
            const uint32_t wd[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                acc[2 * i] = fmaf(w, __uint_as_float(wd[i] << 16), acc[2 * i]);
                acc[2 * i + 1] = fmaf(w, __uint_as_float(wd[i] & 0xFFFF0000u), acc[2 * i + 1]);
            }
        }
    }
    uint4* dst = reinterpret_cast<uint4*>(out + wi * kMV) + 2 * lane;
    dst[0] = make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]), pack_bf16(acc[4], acc[5]),
                        pack_bf16(acc[6], acc[7]));
    dst[1] = make_uint4(pack_bf16(acc[8], acc[9]), pack_bf16(acc[10], acc[11]), pack_bf16(acc[12], acc[13]),
                        pack_bf16(acc[14], acc[15]));
    if (lse && lane == 0) lse[wi] = L;
}

// ---------------------------------------------------------------------------
// One rank's view of the sequences: the tokens of a sequence of n tokens the
// rank owns are f I + clamp(n mod (I R) - r I, 0, I) with f = n / (I R) (whole
// turns, then the rank's part of the last); a query at position p sees its
// owned tokens <= p, so its local causal bound is owned(p + 1) - 1 (-1: the
// rank owns none, DSA_ERR_BAD_INPUT); with a page table and I a whole number
// m of pages, local page l is global page ((l / m) R + r) m + l mod m.
__host__ __device__ __forceinline__ int64_t dcp_owned(int64_t n, int world, int rank, int inter) {
    const int64_t turn = (int64_t)inter * world;
    const int64_t f = n / turn, rem = n - f * turn - (int64_t)rank * inter;
    return f * inter + (rem < 0 ? 0 : (rem > inter ? inter : rem));
}

__global__ void __launch_bounds__(128) dcp_shard_seqs_kernel(dsa_seqs s, int num_q, int world, int rank, int inter,
                                                             int32_t* __restrict__ lctx, int32_t* __restrict__ lpos,
                                                             int32_t* __restrict__ ltable, int lmax_pages,
                                                             int32_t* d_status) {
    pdl_enter();
    const int i = blockIdx.x * 128 + threadIdx.x;
    if (i < s.num_seqs) {
        const int c = __ldg(s.ctx_len + i);
        if (c < 0 || c > s.max_ctx) report(d_status, DSA_ERR_BAD_INPUT);
        lctx[i] = (int32_t)dcp_owned(c < 0 ? 0 : c, world, rank, inter);
    }
    if (i < num_q) {
        const int b = seq_of(s.q_start, s.num_seqs, i);
        const int c = __ldg(s.ctx_len + b), p = __ldg(s.q_pos + i);
        int64_t bound = -1;
        if (p >= 0 && p < c) bound = dcp_owned((int64_t)p + 1, world, rank, inter) - 1;
        if (bound < 0) report(d_status, DSA_ERR_BAD_INPUT);
        lpos[i] = (int32_t)bound;
    }
    if (ltable) {
        const int m = inter / s.page_size;  // pages per turn
        const int64_t cells = (int64_t)s.num_seqs * lmax_pages;
        for (int64_t e = (int64_t)blockIdx.x * 128 + threadIdx.x; e < cells; e += (int64_t)gridDim.x * 128) {
            const int b = (int)(e / lmax_pages), l = (int)(e - (int64_t)b * lmax_pages);
            const int64_t gp = ((int64_t)(l / m) * world + rank) * m + l % m;
            ltable[e] = gp < s.max_pages ? __ldg(s.page_table + (int64_t)b * s.max_pages + gp) : -1;
        }
    }
}

}  // namespace

int64_t dcp_owned_tokens(int64_t n, int world, int rank, int inter) { return dcp_owned(n, world, rank, inter); }

cudaError_t launch_dcp_shard_seqs(const dsa_seqs& s, int num_q, int world, int rank, int inter, int32_t* lctx,
                                  int32_t* lpos, int32_t* ltable, int lmax_pages, int32_t* d_status,
                                  cudaStream_t stream) {
    const int n = num_q > s.num_seqs ? num_q : s.num_seqs;
    int blocks = (n + 127) / 128;
    if (ltable) {
        const int64_t cells = (int64_t)s.num_seqs * lmax_pages;
        const int64_t tb = (cells + 127) / 128;
        if (tb > blocks) blocks = (int)(tb < 4096 ? tb : 4096);
    }
    return launch_pdl(dcp_shard_seqs_kernel, dim3(blocks < 1 ? 1 : blocks), dim3(128), 0, stream, 1, s, num_q, world,
                      rank, inter, lctx, lpos, ltable, lmax_pages, d_status);
}

cudaError_t launch_cand_pack(const float* scores, int64_t ld, const int32_t* idx, const int32_t* topk_len, int num_q,
                             int k, int world, int rank, int inter, uint64_t* cand, int32_t* d_status,
                             cudaStream_t stream) {
    if (num_q <= 0) return cudaSuccess;
    return launch_pdl(cand_pack_kernel, dim3((unsigned)num_q, (unsigned)((k + 255) / 256)), dim3(256), 0, stream, 1,
                      scores, ld, idx, topk_len, k, world, rank, inter, cand, d_status);
}

cudaError_t launch_topk_merge(const uint64_t* const* lists, int num_lists, int list_len, int num_q, int k,
                              int32_t* idx, int32_t* topk_len, int32_t* d_status, cudaStream_t stream) {
    if (num_q <= 0) return cudaSuccess;
    ListPtrs lp{};
    for (int r = 0; r < num_lists; ++r) lp.p[r] = lists[r];
    // sel holds up to the next power of two of k ids (the bitonic sort's padding)
    int P = 1;
    while (P < k) P <<= 1;
    const size_t smem = (size_t)num_lists * list_len * sizeof(uint64_t) + (size_t)P * sizeof(int32_t);
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)(kMergeMaxCand * sizeof(uint64_t) + DSA_MAX_TOPK * sizeof(int32_t)));
    });
    if (attr != cudaSuccess) return attr;
    return launch_pdl(topk_merge_kernel, dim3((unsigned)num_q), dim3(kMergeThreads), smem, stream, 1, lp, num_lists,
                      list_len, k, idx, topk_len, d_status);
}

cudaError_t launch_topk_compact(const int32_t* idx, const int32_t* topk_len, int num_q, int k, int world, int rank,
                                int inter, int32_t* local_idx, int32_t* local_len, int32_t* d_status,
                                cudaStream_t stream) {
    if (num_q <= 0) return cudaSuccess;
    return launch_pdl(topk_compact_kernel, dim3((unsigned)num_q), dim3(kCompactThreads), 0, stream, 1, idx, topk_len,
                      num_q, k, world, rank, inter, local_idx, local_len, d_status);
}

cudaError_t launch_lse_combine(const void* const* o_parts, const float* const* lse_parts, int num_parts, int num_q,
                               void* out, float* lse, cudaStream_t stream) {
    if (num_q <= 0) return cudaSuccess;
    PartPtrs pp{};
    for (int r = 0; r < num_parts; ++r) {
        pp.o[r] = static_cast<const __nv_bfloat16*>(o_parts[r]);
        pp.l[r] = lse_parts[r];
    }
    const int64_t warps = (int64_t)num_q * kMH;
    return launch_pdl(lse_combine_kernel, dim3((unsigned)((warps + 3) / 4)), dim3(128), 0, stream, 1, pp, num_parts,
                      num_q, static_cast<__nv_bfloat16*>(out), lse);
}

}  // namespace dsa
