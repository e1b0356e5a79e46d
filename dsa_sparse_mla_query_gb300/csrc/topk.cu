// topk.cu -- exact top-k per query by radix select (sm_103a).
//
// "Day 0 support for Mistral Large 4" (vLLM blog): Model architecture (top-k
// 2048 keys per query), Specialized decode (an exact top-2048), DCP (a radix
// select; top-k compaction with topk_length instead of slots full of -1).
//
// The selection never sorts the context.  Scores map to order-preserving
// 32-bit keys (-0.0 folded onto +0.0); four 8-bit digit passes, each a shared-
// memory histogram of the keys that still match the selected prefix, pin the
// exact k-th largest key T and how many keys equal to T are needed.  A final
// pass in index order writes every key > T and the first needed keys == T
// (ties to the smaller index) with block-wide prefix sums, so the output is
// the selected positions in ascending order: deterministic and compacted.
#include "dsa_internal.cuh"

namespace dsa {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;  // -0.0 ranks as +0.0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// exclusive block prefix sum of v over kTopkThreads threads; *total = sum
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_buf, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_buf[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kTopkWarps ? warp_buf[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_buf[32 + lane] = w;  // inclusive warp totals
    }
    __syncthreads();
    const int before = (warp ? warp_buf[32 + warp - 1] : 0) + x - v;
    *total = warp_buf[32 + kTopkWarps - 1];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ scores, int64_t ld, dsa_seqs s,
                                                             int k, int32_t* __restrict__ idx,
                                                             int32_t* __restrict__ topk_len, int32_t* d_status) {
    __shared__ int hist[256];
    __shared__ int scan_buf[64];
    __shared__ int sel_digit, sel_above;
    const int t = blockIdx.x;
    const int tid = threadIdx.x;
    const int b = seq_of(s.q_start, s.num_seqs, t);
    const int pos = __ldg(s.q_pos + t);
    const int ctx = __ldg(s.ctx_len + b);
    int32_t* out = idx + (int64_t)t * k;
    if (pos < 0 || pos >= ctx || ctx > s.max_ctx) {
        if (tid == 0) {
            report(d_status, DSA_ERR_BAD_INPUT);
            topk_len[t] = 0;
        }
        for (int i = tid; i < k; i += kTopkThreads) out[i] = -1;
        return;
    }
    const int n = pos + 1;
    const float* row = scores + (int64_t)t * ld;
    if (n <= k) {  // every causal key
        for (int i = tid; i < k; i += kTopkThreads) out[i] = i < n ? i : -1;
        if (tid == 0) topk_len[t] = n;
        return;
    }

    // ---- radix select of the k-th largest order key
    uint32_t prefix = 0, mask = 0;
    int remaining = k;  // keys still to take among those matching prefix
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        if (tid < 256) hist[tid] = 0;
        __syncthreads();
        for (int i = tid; i < n; i += kTopkThreads) {
            const uint32_t u = order_key(__ldg(row + i));
            if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255], 1);
        }
        __syncthreads();
        // digits in descending order: thread i <-> digit 255 - i
        int c = tid < 256 ? hist[255 - tid] : 0;
        int tot;
        const int before = block_exclusive_scan(c, scan_buf, &tot);
        if (tid < 256 && before < remaining && before + c >= remaining) {
            sel_digit = 255 - tid;
            sel_above = before;
        }
        __syncthreads();
        prefix |= (uint32_t)sel_digit << shift;
        mask |= 255u << shift;
        remaining -= sel_above;
        __syncthreads();
    }
    const uint32_t T = prefix;  // exact key of the k-th largest score
    const int need_eq = remaining;

    // ---- compaction in index order (4 consecutive scores per thread)
    int base_out = 0, base_eq = 0;
    for (int start = 0; start < n; start += 4 * kTopkThreads) {
        const int i0 = start + 4 * tid;
        uint32_t u[4];
        int n_eq = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            u[e] = (i0 + e < n) ? order_key(__ldg(row + i0 + e)) : 0u;
            n_eq += (i0 + e < n && u[e] == T);
        }
        int tot_eq;
        int eq_rank = base_eq + block_exclusive_scan(n_eq, scan_buf, &tot_eq);
        bool take[4];
        int n_sel = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const bool valid = i0 + e < n;
            bool tk = valid && u[e] > T;
            if (valid && u[e] == T) {
                tk = eq_rank < need_eq;
                ++eq_rank;
            }
            take[e] = tk;
            n_sel += tk;
        }
        int tot_sel;
        int o = base_out + block_exclusive_scan(n_sel, scan_buf, &tot_sel);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (take[e] && o < k) out[o++] = i0 + e;
        base_out += tot_sel;
        base_eq += tot_eq;
    }
    for (int i = base_out + tid; i < k; i += kTopkThreads) out[i] = -1;
    if (tid == 0) topk_len[t] = min(base_out, k);
}

cudaError_t launch_topk(const float* scores, int64_t ld, const dsa_seqs& s, int num_q, int k, int32_t* idx,
                        int32_t* topk_len, int32_t* d_status, cudaStream_t stream) {
    topk_kernel<<<num_q, kTopkThreads, 0, stream>>>(scores, ld, s, k, idx, topk_len, d_status);
    return cudaGetLastError();
}

}  // namespace dsa
