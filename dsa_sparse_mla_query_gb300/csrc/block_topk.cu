// block_topk.cu -- block-sparse selection (sm_103a).
//
// "vLLM adds NVFP4 serving for MiniMax M3.1 Flash", MiniMax Sparse Attention:
// the KV cache is divided into 128-token blocks, the index keys are scanned
// over the context and 16 blocks are selected, the most recent always kept,
// and exact attention runs over the selected blocks' keys.  A block scores the
// maximum of its causal keys' indexer scores; the query's own block is always
// selected, then the nsel - 1 best other blocks, ties to the smaller block.
// The selection leaves as dsa_topk's does (ascending positions, then -1, and
// topk_len), so sparse_mla_decode reads it with k = nsel * block.
//
// One CTA per query.  Block maxima go to shared memory (a warp per block,
// coalesced reads of its scores, or, in the fused layer, a thread per block
// over the 32-key group maxima the indexer wrote in place of the scores); nsel rounds of a block-wide argmax over
// packed (order-preserving score code, inverted block id) values pick the
// blocks; the chosen ids are sorted and their keys written in order.
#include <mutex>

#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kBtThreads = 512;
constexpr int kBtWarps = kBtThreads / 32;

__device__ __forceinline__ uint32_t bt_code(float s) {
    const uint32_t b = __float_as_uint(s == 0.f ? 0.f : s);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// FromGroups: `scores` holds, per query, the maxima of the 32-key groups of
// its score row (group i: keys [32 i, 32 i + 32), -inf past the query's
// position), which the indexer writes in place of the row; block must then be
// a multiple of 32, and a block's maximum is the maximum of its groups.
template <bool FromGroups>
__global__ void __launch_bounds__(kBtThreads) block_topk_kernel(const float* __restrict__ scores, int64_t ld,
                                                                dsa_seqs s, int block, int nsel,
                                                                int32_t* __restrict__ idx,
                                                                int32_t* __restrict__ topk_len, int32_t* d_status) {
    extern __shared__ __align__(16) float bmax[];  // [max blocks], then chosen ids [nsel]
    __shared__ unsigned long long wbest[kBtWarps];
    __shared__ int s_pick;
    const int t = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = nsel * block;
    const int max_blocks = (s.max_ctx + block - 1) / block;
    int* chosen = reinterpret_cast<int*>(bmax + max_blocks);
    pdl_enter();
    const int b = seq_of(s.q_start, s.num_seqs, t);
    const int pos = __ldg(s.q_pos + t);
    const int ctx = __ldg(s.ctx_len + b);
    int32_t* out = idx + (int64_t)t * k;
    if (pos < 0 || pos >= ctx || ctx > s.max_ctx) {
        if (tid == 0) {
            report(d_status, DSA_ERR_BAD_INPUT);
            topk_len[t] = 0;
        }
        for (int i = tid; i < k; i += kBtThreads) out[i] = -1;
        return;
    }
    const int n = pos + 1;                    // causal keys
    const int nb = (n + block - 1) / block;   // blocks holding them
    const float* row = scores + (int64_t)t * ld;
    // block maxima; fmaxf skips NaN scores, so a maximum is never NaN and NaN
    // below marks a block already chosen
    if constexpr (FromGroups) {
        // a thread per block over its groups (keys past the position are -inf)
        const int gpb = block >> 5, ng = (n + 31) >> 5;
        for (int bi = tid; bi < nb; bi += kBtThreads) {
            float m = -INFINITY;
            const int g1 = min(ng, (bi + 1) * gpb);
            for (int gi = bi * gpb; gi < g1; ++gi) m = fmaxf(m, __ldg(row + gi));
            bmax[bi] = bi == nb - 1 ? __int_as_float(0x7FC00000) : m;  // own block: taken first
        }
    } else {
        // a warp per block, coalesced reads of its scores
        for (int bi = warp; bi < nb; bi += kBtWarps) {
            float m = -INFINITY;
            const int j1 = min(n, (bi + 1) * block);
            for (int j = bi * block + lane; j < j1; j += 32) m = fmaxf(m, __ldg(row + j));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) bmax[bi] = bi == nb - 1 ? __int_as_float(0x7FC00000) : m;  // own block: taken first
        }
    }
    if (tid == 0) {
        chosen[0] = nb - 1;
        s_pick = 1;
    }
    __syncthreads();
    // nsel - 1 rounds of argmax over the other blocks: larger packed value =
    // larger score, then smaller block
    const int rounds = min(nsel, nb);
    for (int r = 1; r < rounds; ++r) {
        unsigned long long best = 0;
        for (int bi = tid; bi < nb; bi += kBtThreads) {
            const float v = bmax[bi];
            if (v != v) continue;  // NaN marks a block already chosen
            const unsigned long long c = ((unsigned long long)bt_code(v) << 32) | (0xFFFFFFFFu - (uint32_t)bi);
            best = c > best ? c : best;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long u = __shfl_xor_sync(0xffffffffu, best, o);
            best = u > best ? u : best;
        }
        if (lane == 0) wbest[warp] = best;
        __syncthreads();
        if (tid == 0) {
            unsigned long long m = 0;
            for (int w = 0; w < kBtWarps; ++w) m = wbest[w] > m ? wbest[w] : m;
            // m == 0 would mean no block left: impossible while r < nb, but
            // never index with it
            const int bi = m ? (int)(0xFFFFFFFFu - (uint32_t)m) : -1;
            if (bi >= 0 && bi < nb) {
                chosen[r] = bi;
                bmax[bi] = __int_as_float(0x7FC00000);  // NaN: taken
                s_pick = r + 1;
            } else {
                report(d_status, DSA_ERR_BAD_INPUT);
            }
        }
        __syncthreads();
        if (s_pick != r + 1) break;
    }
    // the chosen ids in ascending order (at most a few dozen: one thread)
    if (tid == 0) {
        for (int i = 1; i < s_pick; ++i) {
            const int x = chosen[i];
            int j = i - 1;
            while (j >= 0 && chosen[j] > x) {
                chosen[j + 1] = chosen[j];
                --j;
            }
            chosen[j + 1] = x;
        }
    }
    __syncthreads();
    // the own block is the highest chosen id and the only partial one, so
    // chosen block i starts at slot i * block
    int len = 0;
    for (int i = 0; i < s_pick; ++i) len += min(n, (chosen[i] + 1) * block) - chosen[i] * block;
    for (int sl = tid; sl < k; sl += kBtThreads) {
        const int i = sl / block, jj = sl - i * block;
        int v = -1;
        if (i < s_pick) {
            const int j = chosen[i] * block + jj;
            if (j < n) v = j;
        }
        out[sl] = v;
    }
    if (tid == 0) topk_len[t] = len;
}

}  // namespace

size_t block_topk_smem(int max_ctx, int block, int nsel) {
    const int max_blocks = (max_ctx + block - 1) / block;
    return (size_t)max_blocks * sizeof(float) + (size_t)nsel * sizeof(int);
}

cudaError_t launch_block_topk(const float* scores, int64_t ld, const dsa_seqs& s, int num_q, int block, int nsel,
                              int32_t* idx, int32_t* topk_len, int32_t* d_status, cudaStream_t stream,
                              bool from_groups) {
    if (num_q <= 0) return cudaSuccess;
    const size_t smem = block_topk_smem(s.max_ctx, block, nsel);  // <= DSA_BLOCK_TOPK_MAX_SMEM (checked)
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(block_topk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)DSA_BLOCK_TOPK_MAX_SMEM);
        if (attr == cudaSuccess)
            attr = cudaFuncSetAttribute(block_topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)DSA_BLOCK_TOPK_MAX_SMEM);
    });
    if (attr != cudaSuccess) return attr;
    return launch_pdl(from_groups ? block_topk_kernel<true> : block_topk_kernel<false>, dim3((unsigned)num_q),
                      dim3(kBtThreads), smem, stream, 1, scores, ld, s, block, nsel, idx, topk_len, d_status);
}

}  // namespace dsa
