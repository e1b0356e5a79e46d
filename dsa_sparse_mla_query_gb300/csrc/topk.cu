// topk.cu -- exact top-k per query by radix select (sm_103a).
//
// "Day 0 support for Mistral Large 4" (vLLM blog): Model architecture (top-k
// 2048 keys per query), Specialized decode (an exact top-2048), DCP (a radix
// select; top-k compaction with topk_length instead of slots full of -1).
//
// The selection never sorts the context.  Scores map to order-preserving
// 32-bit keys (-0.0 folded onto +0.0); digit passes, each a shared-memory
// histogram of the keys that still match the selected prefix, pin the exact
// k-th largest key T and how many keys equal to T are needed.  A final pass in
// index order writes every key > T and the first needed keys == T (ties to the
// smaller index) with block-wide prefix sums, so the output is the selected
// positions in ascending order: deterministic and compacted.
//
// Three kernels share that scheme: rows up to 32,768 keys take one CTA each
// with the row in registers (three passes of 11 + 11 + 10 bits); longer rows
// up to 16 x 32,768 keys a thread-block cluster per row; anything longer one
// CTA per row with four 8-bit passes over memory.

#include <algorithm>
#include <climits>
#include <cstdint>
#include <mutex>

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
    pdl_enter();
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

// exclusive prefix sum over the THREADS threads of a block; *total = sum
template <int THREADS>
__device__ __forceinline__ int scan_threads(int v, int* buf, int* total) {
    constexpr int W = THREADS / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) buf[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < W ? buf[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        buf[32 + lane] = w;
    }
    __syncthreads();
    const int before = (warp ? buf[32 + warp - 1] : 0) + x - v;
    *total = buf[32 + W - 1];
    __syncthreads();
    return before;
}

// ---------------------------------------------------------------------------
// One CTA per row, the row held in registers (THREADS threads x EPT
// consecutive scores, rows up to 32,768 keys).  Three digit passes (11 + 11 + 10 bits)
// with __syncthreads only.  Scores of a row crowd into few bins of the first
// digit, so that histogram is counted into eight private copies (four warps
// each) to spread the same-address atomics; the keys of the chosen bin are
// then compacted into shared memory and the two finer passes run over them.
constexpr int kRowBins = 2048;
constexpr int kRowSub = 8;             // private copies of the first histogram
constexpr int kRowCandCap = 4096;
constexpr size_t kRowSmem = (size_t)kRowSub * kRowBins * 4 + kRowCandCap * 4;

template <int THREADS, int EPT>
__global__ void __launch_bounds__(THREADS, 1) topk_row_kernel(const float* __restrict__ scores, int64_t ld,
                                                                dsa_seqs s, int k, int32_t* __restrict__ idx,
                                                                int32_t* __restrict__ topk_len, int32_t* d_status) {
    pdl_enter();
    extern __shared__ __align__(16) int row_smem[];
    int* sub = row_smem;                                                   // [kRowSub][kRowBins]
    uint32_t* cand = reinterpret_cast<uint32_t*>(row_smem + kRowSub * kRowBins);  // [kRowCandCap]
    __shared__ int scan_buf[64];
    __shared__ int sel_digit, sel_above, ncand;
    const int t = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int b = seq_of(s.q_start, s.num_seqs, t);
    const int pos = __ldg(s.q_pos + t);
    const int ctx = __ldg(s.ctx_len + b);
    int32_t* out = idx + (int64_t)t * k;
    if (pos < 0 || pos >= ctx || ctx > s.max_ctx || pos + 1 > THREADS * EPT) {
        if (tid == 0) {
            report(d_status, DSA_ERR_BAD_INPUT);
            topk_len[t] = 0;
        }
        for (int i = tid; i < k; i += THREADS) out[i] = -1;
        return;
    }
    const int n = pos + 1;
    if (n <= k) {
        for (int i = tid; i < k; i += THREADS) out[i] = i < n ? i : -1;
        if (tid == 0) topk_len[t] = n;
        return;
    }
    // ---- this thread's EPT consecutive keys: every load issued before any is
    // used (indexes clamped into the row, so no load waits on a bounds branch)
    const float* row = scores + (int64_t)t * ld;
    const int base = tid * EPT;
    const int last4 = (int)((ld - 4) & ~(int64_t)3);  // the row holds ld >= n floats, ld a multiple of 4
    uint32_t u[EPT];  // raw bits first, order keys after
    if (base + EPT <= ld) {  // the whole run lies in the row: offsets from one pointer
        const uint4* p = reinterpret_cast<const uint4*>(row + base);
#pragma unroll
        for (int v = 0; v < EPT / 4; ++v) {
            const uint4 r = __ldg(p + v);
            u[4 * v] = r.x;
            u[4 * v + 1] = r.y;
            u[4 * v + 2] = r.z;
            u[4 * v + 3] = r.w;
        }
    } else {
#pragma unroll
        for (int v = 0; v < EPT / 4; ++v) {
            const uint4 r = __ldg(reinterpret_cast<const uint4*>(row + min(base + 4 * v, last4)));
            u[4 * v] = r.x;
            u[4 * v + 1] = r.y;
            u[4 * v + 2] = r.z;
            u[4 * v + 3] = r.w;
        }
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) u[e] = order_key(__uint_as_float(u[e]));
    const int nv = min(max(n - base, 0), EPT);  // this thread's keys inside the row: u[0 .. nv)
    uint32_t prefix = 0, mask = 0;
    int remaining = k;
    bool use_cand = false;
    if (tid == 0) ncand = 0;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nb = pass == 2 ? 1024 : 2048;
        const int copies = use_cand ? 1 : kRowSub;
        for (int i = tid; i < copies * kRowBins; i += THREADS) sub[i] = 0;
        __syncthreads();
        if (use_cand) {
            for (int i = tid; i < ncand; i += THREADS) {
                const uint32_t c = cand[i];
                if ((c & mask) == prefix) atomicAdd(sub + ((c >> shift) & (nb - 1)), 1);
            }
        } else {
            int* h = sub + (warp % kRowSub) * kRowBins;
#pragma unroll
            for (int e = 0; e < EPT; ++e)
                if ((e < nv) && (u[e] & mask) == prefix) atomicAdd(h + ((u[e] >> shift) & (nb - 1)), 1);
        }
        __syncthreads();
        // digits in descending order, nb / 1024 per thread, summed over the copies
        constexpr int kMaxPer = kRowBins / THREADS;
        const int per = nb / THREADS;
        static_assert(kRowBins % THREADS == 0 && 1024 % THREADS == 0, "bins per thread");
        int c[kMaxPer], csum = 0;
#pragma unroll
        for (int q = 0; q < kMaxPer; ++q) {
            int v = 0;
            if (q < per) {
                const int d = nb - 1 - per * tid - q;
                for (int cp = 0; cp < copies; ++cp) v += sub[cp * kRowBins + d];
            }
            c[q] = v;
            csum += v;
        }
        int tot;
        int before = scan_threads<THREADS>(csum, scan_buf, &tot);
#pragma unroll
        for (int q = 0; q < kMaxPer; ++q) {
            if (q < per && before < remaining && before + c[q] >= remaining) {
                sel_digit = nb - 1 - per * tid - q;
                sel_above = before;
            }
            before += c[q];
        }
        __syncthreads();
        prefix |= (uint32_t)sel_digit << shift;
        mask |= (uint32_t)(nb - 1) << shift;
        remaining -= sel_above;
        if (pass == 0) {
            // keep the keys of the chosen bin for the next two passes (prefix-sum slots)
            int mine = 0;
#pragma unroll
            for (int e = 0; e < EPT; ++e) mine += (e < nv) && (u[e] & mask) == prefix;
            int nc;
            int sl = scan_threads<THREADS>(mine, scan_buf, &nc);
            if (nc <= kRowCandCap) {
#pragma unroll
                for (int e = 0; e < EPT; ++e)
                    if ((e < nv) && (u[e] & mask) == prefix) cand[sl++] = u[e];
            }
            if (tid == 0) ncand = nc;
            __syncthreads();
            use_cand = nc <= kRowCandCap;
        } else {
            __syncthreads();  // the next pass clears the histogram this one read
        }
    }
    const uint32_t T = prefix;
    const int need_eq = remaining;
    // ---- ranks in index order: every key > T, the first need_eq keys == T
    int n_gt = 0, n_eq = 0;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        const bool vld = e < nv;
        n_gt += vld && u[e] > T;
        n_eq += vld && u[e] == T;
    }
    int tot_eq;
    int eq_rank = scan_threads<THREADS>(n_eq, scan_buf, &tot_eq);
    const int n_sel = n_gt + max(0, min(need_eq - eq_rank, n_eq));
    int tot_sel;
    int o = scan_threads<THREADS>(n_sel, scan_buf, &tot_sel);
    // positions staged in shared memory (the candidate buffer, k <= its size),
    // then written out with coalesced stores
    int* stage_out = reinterpret_cast<int*>(cand);
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        if (!(e < nv)) continue;
        bool take = u[e] > T;
        if (u[e] == T) take = eq_rank++ < need_eq;
        if (take && o < k) stage_out[o++] = base + e;
    }
    __syncthreads();
    for (int i = tid; i < k; i += THREADS) out[i] = stage_out[i];
    if (tid == 0) topk_len[t] = k;
}

// ---------------------------------------------------------------------------
// The same selection with the row in shared memory: loops stay rolled, so the
// code is small (the register-resident version is instruction-fetch bound)
// and nothing spills.  1024 threads; thread t owns keys t*EPT .. t*EPT+EPT-1,
// key i stored at (i mod 32) * 1025 + i / 32.  The row is read with coalesced
// 16-byte loads (a warp reads 512 contiguous bytes); with the padded stride
// both those stores and a thread's reads of its own keys are free of bank
// conflicts.
// The list of keys from the chosen first digit up (key and 16-bit position)
// lives after the first histogram copy, over the other copies, which are free
// once that digit is chosen.
constexpr int kSmemCand = 12288;
constexpr size_t kSmemListBytes = (size_t)kSmemCand * (4 + 2);
template <int EPT>
constexpr size_t smem_row_bytes() {
    return (size_t)32 * (EPT * 1024 / 32 + 1) * 4 + (size_t)kRowBins * 4 +
           std::max(kSmemListBytes, (size_t)(kRowSub - 1) * kRowBins * 4);
}

template <int EPT>
__global__ void __launch_bounds__(1024, 1) topk_smem_kernel(const float* __restrict__ scores, int64_t ld, dsa_seqs s,
                                                             int k, int32_t* __restrict__ idx,
                                                             int32_t* __restrict__ topk_len, int32_t* d_status) {
    constexpr int NT = 1024;
    pdl_enter();
    extern __shared__ __align__(16) int sm_smem[];
    constexpr int KS = EPT * NT / 32 + 1;                                     // padded stride
    uint32_t* keys = reinterpret_cast<uint32_t*>(sm_smem);                    // key i at (i % 32) * KS + i / 32
    int* sub = sm_smem + 32 * KS;                                             // [kRowSub][kRowBins]
    uint32_t* cand = reinterpret_cast<uint32_t*>(sub + kRowBins);  // [kSmemCand] keys, over copies 1..
    uint16_t* cpos = reinterpret_cast<uint16_t*>(cand + kSmemCand);  // [kSmemCand] their positions
    __shared__ int scan_buf[64];
    __shared__ int sel_digit, sel_above, ncand;
    const int t = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int b = seq_of(s.q_start, s.num_seqs, t);
    const int pos = __ldg(s.q_pos + t);
    const int ctx = __ldg(s.ctx_len + b);
    int32_t* out = idx + (int64_t)t * k;
    if (pos < 0 || pos >= ctx || ctx > s.max_ctx || pos + 1 > NT * EPT) {
        if (tid == 0) {
            report(d_status, DSA_ERR_BAD_INPUT);
            topk_len[t] = 0;
        }
        for (int i = tid; i < k; i += NT) out[i] = -1;
        return;
    }
    const int n = pos + 1;
    if (n <= k) {
        for (int i = tid; i < k; i += NT) out[i] = i < n ? i : -1;
        if (tid == 0) topk_len[t] = n;
        return;
    }
    // ---- the row into shared memory: coalesced loads, all in flight first
    const float* row = scores + (int64_t)t * ld;
    const int last4 = (int)((ld - 4) & ~(int64_t)3);
    {
        uint4 r[EPT / 4];
#pragma unroll
        for (int v = 0; v < EPT / 4; ++v)
            r[v] = __ldg(reinterpret_cast<const uint4*>(row + min((v * NT + tid) * 4, last4)));
#pragma unroll
        for (int v = 0; v < EPT / 4; ++v) {
            const int i0 = (v * NT + tid) * 4;
            const uint32_t w4[4] = {r[v].x, r[v].y, r[v].z, r[v].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) keys[((i0 + c) & 31) * KS + ((i0 + c) >> 5)] = order_key(__uint_as_float(w4[c]));
        }
    }
    __syncthreads();
    const int base = tid * EPT;
    const int nv = min(max(n - base, 0), EPT);  // this thread's keys inside the row
    uint32_t prefix = 0, mask = 0;
    int remaining = k;
    bool use_cand = false;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nb = pass == 2 ? 1024 : 2048;
        const int copies = use_cand ? 1 : kRowSub;
        for (int i = tid; i < copies * kRowBins; i += NT) sub[i] = 0;
        __syncthreads();
        if (use_cand) {
            for (int i = tid; i < ncand; i += NT) {
                const uint32_t c = cand[i];
                if ((c & mask) == prefix) atomicAdd(sub + ((c >> shift) & (nb - 1)), 1);
            }
        } else {
            int* h = sub + (warp % kRowSub) * kRowBins;
#pragma unroll 8
            for (int e = 0; e < nv; ++e) {
                const uint32_t u = keys[e * KS + tid];
                if ((u & mask) == prefix) atomicAdd(h + ((u >> shift) & (nb - 1)), 1);
            }
        }
        __syncthreads();
        // digits in descending order, 2 (or 1) per thread, summed over the copies
        const int per = nb / NT;
        int c0 = 0, c1 = 0;
        {
            const int d0 = nb - 1 - per * tid;
            for (int cp = 0; cp < copies; ++cp) c0 += sub[cp * kRowBins + d0];
            if (per == 2)
                for (int cp = 0; cp < copies; ++cp) c1 += sub[cp * kRowBins + d0 - 1];
        }
        int tot;
        const int before = scan_threads<NT>(c0 + c1, scan_buf, &tot);
        if (before < remaining && before + c0 >= remaining) {
            sel_digit = nb - 1 - per * tid;
            sel_above = before;
        } else if (per == 2 && before + c0 < remaining && before + c0 + c1 >= remaining) {
            sel_digit = nb - 2 - per * tid;
            sel_above = before + c0;
        }
        __syncthreads();
        prefix |= (uint32_t)sel_digit << shift;
        mask |= (uint32_t)(nb - 1) << shift;
        remaining -= sel_above;
        if (pass == 0) {
            // every key of the chosen first digit or above -- the selection
            // lies among them -- with its position, in ascending position
            // (prefix-sum slots; thread t holds positions t EPT ..): the two
            // finer passes and the final selection then walk this list alone
            int mine = 0;
#pragma unroll 8
            for (int e = 0; e < nv; ++e) mine += keys[e * KS + tid] >= prefix;
            int nc;
            int sl = scan_threads<NT>(mine, scan_buf, &nc);
            if (nc <= kSmemCand)
#pragma unroll 8
                for (int e = 0; e < nv; ++e) {
                    const uint32_t u = keys[e * KS + tid];
                    if (u >= prefix) {
                        cand[sl] = u;
                        cpos[sl++] = (uint16_t)(base + e);
                    }
                }
            if (tid == 0) ncand = nc;
            __syncthreads();
            use_cand = nc <= kSmemCand;
        } else {
            __syncthreads();  // the next pass clears the histogram this one read
        }
    }
    const uint32_t T = prefix;
    const int need_eq = remaining;
    if (use_cand) {
        // ---- from the list: every key > T, the first need_eq keys == T,
        // consecutive entries per thread, written in ascending position
        const int nc = ncand, per_t = (nc + NT - 1) / NT;
        const int j0 = min(tid * per_t, nc), j1 = min(j0 + per_t, nc);
        int n_gt = 0, n_eq = 0;
        for (int j = j0; j < j1; ++j) {
            n_gt += cand[j] > T;
            n_eq += cand[j] == T;
        }
        int tot_eq;
        int eq_rank = scan_threads<NT>(n_eq, scan_buf, &tot_eq);
        const int n_sel = n_gt + max(0, min(need_eq - eq_rank, n_eq));
        int tot_sel;
        int o = scan_threads<NT>(n_sel, scan_buf, &tot_sel);
        for (int j = j0; j < j1; ++j) {
            const uint32_t c = cand[j];
            bool take = c > T;
            if (c == T) take = eq_rank++ < need_eq;
            if (take && o < k) out[o++] = cpos[j];
        }
        if (tid == 0) topk_len[t] = k;
        return;
    }
    // ---- ranks in index order: every key > T, the first need_eq keys == T
    int n_gt = 0, n_eq = 0;
#pragma unroll 8
    for (int e = 0; e < nv; ++e) {
        const uint32_t u = keys[e * KS + tid];
        n_gt += u > T;
        n_eq += u == T;
    }
    int tot_eq;
    int eq_rank = scan_threads<NT>(n_eq, scan_buf, &tot_eq);
    const int n_sel = n_gt + max(0, min(need_eq - eq_rank, n_eq));
    int tot_sel;
    int o = scan_threads<NT>(n_sel, scan_buf, &tot_sel);
    int* stage_out = reinterpret_cast<int*>(cand);  // k <= kSmemCand
#pragma unroll 8
    for (int e = 0; e < nv; ++e) {
        const uint32_t u = keys[e * KS + tid];
        bool take = u > T;
        if (u == T) take = eq_rank++ < need_eq;
        if (take && o < k) stage_out[o++] = base + e;
    }
    __syncthreads();
    for (int i = tid; i < k; i += NT) out[i] = stage_out[i];
    if (tid == 0) topk_len[t] = k;
}

// ---------------------------------------------------------------------------
// Rows longer than 32,768 keys: a chunked pipeline over every SM (no kernel
// needs the CTAs of a row to be co-resident).  Chunks of kLongChunk keys.
//   1. topk_hist_kernel  (chunk x row): histogram of the first digit (top 11
//      bits of the order key) of each chunk, added into the row's histogram;
//   2. topk_cand_kernel  (chunk x row): the digit d0 of the k-th key from the
//      row's histogram; the positions of the chunk's keys above d0 (fewer than
//      k in the row) and the keys of d0 (key, position) are appended to the
//      row's lists, one reservation per CTA;
//   3. topk_final_kernel (row): the exact k-th key T among the keys of d0
//      (11 + 10 more bits; by passes over the row in memory when they
//      overflowed their list), then the selected positions -- every key above
//      d0, the keys of d0 above T and the smallest positions of the keys equal
//      to T that are needed -- sorted ascending in shared memory.
constexpr int kLongThreads = 1024;
constexpr int kLongEPT = kLongChunk / kLongThreads;  // 16: four rounds of one float4 per thread
constexpr int kFinalThreads = 1024;
constexpr size_t kFinalSmem = (size_t)kLongCand * 8 + (size_t)kLongCand * 4 + 2048 * 4 + DSA_MAX_TOPK * 4;

// false: nothing for the chunk kernels to do on row t (a bad row is reported
// by the final kernel; a row of at most k keys is written by it)
__device__ __forceinline__ bool long_row(const dsa_seqs& s, int t, int k, int* n_out) {
    const int b = seq_of(s.q_start, s.num_seqs, t);
    const int pos = __ldg(s.q_pos + t);
    const int ctx = __ldg(s.ctx_len + b);
    if (pos < 0 || pos >= ctx || ctx > s.max_ctx) return false;
    *n_out = pos + 1;
    return pos + 1 > k;
}

// position of this thread's key e in the chunk starting at j0: round e / 4 of
// coalesced float4 loads (a warp reads 512 contiguous bytes), component e % 4
__device__ __forceinline__ int chunk_pos(int j0, int e) {
    return j0 + ((e >> 2) * kLongThreads + (int)threadIdx.x) * 4 + (e & 3);
}

__device__ __forceinline__ void chunk_keys(const float* row, int64_t ld, int j0, uint32_t* u) {
    const int last4 = (int)((ld - 4) & ~(int64_t)3);
    uint4 r[kLongEPT / 4];
#pragma unroll
    for (int v = 0; v < kLongEPT / 4; ++v)
        r[v] = __ldg(reinterpret_cast<const uint4*>(row + min(j0 + (v * kLongThreads + (int)threadIdx.x) * 4, last4)));
#pragma unroll
    for (int v = 0; v < kLongEPT / 4; ++v) {
        u[4 * v] = order_key(__uint_as_float(r[v].x));
        u[4 * v + 1] = order_key(__uint_as_float(r[v].y));
        u[4 * v + 2] = order_key(__uint_as_float(r[v].z));
        u[4 * v + 3] = order_key(__uint_as_float(r[v].w));
    }
}

// The first digit of the k-th largest key of a row from its histogram, and
// the number of keys in higher digits; the same result in every thread.
template <int THREADS>
__device__ __forceinline__ void first_digit(const int* hr, int k, int* buf, int* sh, int& d0, int& above) {
    constexpr int PER = 2048 / THREADS;
    int c[PER], csum = 0;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        c[q] = __ldcg(hr + 2047 - PER * (int)threadIdx.x - q);
        csum += c[q];
    }
    int tot;
    int before = scan_threads<THREADS>(csum, buf, &tot);
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        if (before < k && before + c[q] >= k) {
            sh[0] = 2047 - PER * (int)threadIdx.x - q;
            sh[1] = before;
        }
        before += c[q];
    }
    __syncthreads();
    d0 = sh[0];
    above = sh[1];
    __syncthreads();
}

__global__ void __launch_bounds__(kLongThreads) topk_hist_kernel(const float* __restrict__ scores, int64_t ld,
                                                                  dsa_seqs s, int k, int* __restrict__ hist) {
    pdl_enter();
    __shared__ int h[4][2048];
    const int t = blockIdx.y, j0 = blockIdx.x * kLongChunk;
    int n = 0;
    if (!long_row(s, t, k, &n) || j0 >= n) return;  // uniform over the CTA
    for (int i = threadIdx.x; i < 4 * 2048; i += kLongThreads) (&h[0][0])[i] = 0;
    __syncthreads();
    uint32_t u[kLongEPT];
    chunk_keys(scores + (int64_t)t * ld, ld, j0, u);
    int* hw = h[(threadIdx.x >> 5) & 3];  // four copies spread the same-address atomics
#pragma unroll
    for (int e = 0; e < kLongEPT; ++e)
        if (chunk_pos(j0, e) < n) atomicAdd(hw + (u[e] >> 21), 1);
    __syncthreads();
    int* hr = hist + (int64_t)t * 2048;
    for (int b = threadIdx.x; b < 2048; b += kLongThreads) {
        const int v = h[0][b] + h[1][b] + h[2][b] + h[3][b];
        if (v) atomicAdd(hr + b, v);
    }
}

__global__ void __launch_bounds__(kLongThreads) topk_cand_kernel(const float* __restrict__ scores, int64_t ld,
                                                                  dsa_seqs s, int k, const int* __restrict__ hist,
                                                                  int* __restrict__ ncand, int* __restrict__ nabove,
                                                                  uint2* __restrict__ cand, int* __restrict__ above_pos) {
    pdl_enter();
    __shared__ int buf[64], sh[2];
    const int t = blockIdx.y, j0 = blockIdx.x * kLongChunk;
    int n = 0;
    if (!long_row(s, t, k, &n) || j0 >= n) return;
    uint32_t u[kLongEPT];
    chunk_keys(scores + (int64_t)t * ld, ld, j0, u);  // in flight while the digit is found
    int d0, above;
    first_digit<kLongThreads>(hist + (int64_t)t * 2048, k, buf, sh, d0, above);
    int na = 0, nc = 0;
#pragma unroll
    for (int e = 0; e < kLongEPT; ++e) {
        const int dg = chunk_pos(j0, e) < n ? (int)(u[e] >> 21) : -1;
        na += dg > d0;
        nc += dg == d0;
    }
    // one reservation per CTA and list (the chunks of a row share the counters)
    int tot_a, tot_c;
    int sa = scan_threads<kLongThreads>(na, buf, &tot_a);
    int sc = scan_threads<kLongThreads>(nc, buf, &tot_c);
    if (threadIdx.x == 0) {
        sh[0] = tot_a > 0 ? atomicAdd(nabove + t, tot_a) : 0;
        sh[1] = tot_c > 0 ? atomicAdd(ncand + t, tot_c) : 0;
    }
    __syncthreads();
    sa += sh[0];
    sc += sh[1];
    int* ar = above_pos + (int64_t)t * DSA_MAX_TOPK;
    uint2* cr = cand + (int64_t)t * kLongCand;
#pragma unroll
    for (int e = 0; e < kLongEPT; ++e) {
        const int p = chunk_pos(j0, e);
        const int dg = p < n ? (int)(u[e] >> 21) : -1;
        if (dg > d0) {
            if (sa < DSA_MAX_TOPK) ar[sa] = p;
            ++sa;
        } else if (dg == d0) {
            if (sc < kLongCand) cr[sc] = make_uint2(u[e], (uint32_t)p);
            ++sc;
        }
    }
}

// ascending bitonic sort of a[0 .. N), N a power of two, by the whole block
template <int THREADS>
__device__ void bitonic_sort(int* a, int N) {
    for (int size = 2; size <= N; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < N / 2; i += THREADS) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const bool up = (lo & size) == 0;
                const int x = a[lo], y = a[hi];
                if ((x > y) == up) {
                    a[lo] = y;
                    a[hi] = x;
                }
            }
            __syncthreads();
        }
}

__global__ void __launch_bounds__(kFinalThreads) topk_final_kernel(
    const float* __restrict__ scores, int64_t ld, dsa_seqs s, int k, int32_t* __restrict__ idx,
    int32_t* __restrict__ topk_len, const int* __restrict__ hist, const int* __restrict__ ncand,
    const int* __restrict__ nabove, const uint2* __restrict__ cand, const int* __restrict__ above_pos,
    int32_t* d_status) {
    constexpr int NT = kFinalThreads;
    pdl_enter();
    extern __shared__ __align__(16) int fn_smem[];
    uint32_t* ck = reinterpret_cast<uint32_t*>(fn_smem);  // [kLongCand] keys of d0
    int* cp = fn_smem + kLongCand;                        // [kLongCand] their positions
    int* tie = cp + kLongCand;                            // [kLongCand] positions of keys == T
    int* hs = tie + kLongCand;                            // [2048] digit histogram
    int* sel = hs + 2048;                                 // [DSA_MAX_TOPK] selected positions
    __shared__ int buf[64], sh[4];
    const int t = blockIdx.x, tid = threadIdx.x;
    const int b = seq_of(s.q_start, s.num_seqs, t);
    const int pos = __ldg(s.q_pos + t);
    const int ctx = __ldg(s.ctx_len + b);
    int32_t* out = idx + (int64_t)t * k;
    if (pos < 0 || pos >= ctx || ctx > s.max_ctx) {
        if (tid == 0) {
            report(d_status, DSA_ERR_BAD_INPUT);
            topk_len[t] = 0;
        }
        for (int i = tid; i < k; i += NT) out[i] = -1;
        return;
    }
    const int n = pos + 1;
    if (n <= k) {
        for (int i = tid; i < k; i += NT) out[i] = i < n ? i : -1;
        if (tid == 0) topk_len[t] = n;
        return;
    }
    int d0, above;
    first_digit<NT>(hist + (int64_t)t * 2048, k, buf, sh, d0, above);
    const uint32_t dpre = (uint32_t)d0 << 21, dmask = 0x7FFu << 21;
    uint32_t prefix = dpre, mask = dmask;
    int remaining = k - above;
    const int nc = __ldcg(ncand + t);
    const bool in_smem = nc <= kLongCand;
    const float* row = scores + (int64_t)t * ld;
    if (in_smem)
        for (int i = tid; i < nc; i += NT) {
            const uint2 e = __ldcg(cand + (int64_t)t * kLongCand + i);
            ck[i] = e.x;
            cp[i] = (int)e.y;
        }
    // two more digit passes (11 then 10 bits) over the keys of d0
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        const int shift = pass == 0 ? 10 : 0;
        const int nb = pass == 0 ? 2048 : 1024;
        for (int i = tid; i < 2048; i += NT) hs[i] = 0;
        __syncthreads();
        if (in_smem) {
            for (int i = tid; i < nc; i += NT)
                if ((ck[i] & mask) == prefix) atomicAdd(hs + ((ck[i] >> shift) & (nb - 1)), 1);
        } else {
            for (int j = tid; j < n; j += NT) {
                const uint32_t u = order_key(__ldg(row + j));
                if ((u & mask) == prefix) atomicAdd(hs + ((u >> shift) & (nb - 1)), 1);
            }
        }
        __syncthreads();
        const int per = nb / NT;  // 2 or 1 digits per thread, descending
        const int dA = nb - 1 - per * tid;
        const int cA = hs[dA], cB = per == 2 ? hs[dA - 1] : 0;
        int tot;
        const int before = scan_threads<NT>(cA + cB, buf, &tot);
        if (before < remaining && before + cA >= remaining) {
            sh[0] = dA;
            sh[1] = before;
        } else if (per == 2 && before + cA < remaining && before + cA + cB >= remaining) {
            sh[0] = dA - 1;
            sh[1] = before + cA;
        }
        __syncthreads();
        prefix |= (uint32_t)sh[0] << shift;
        mask |= (uint32_t)(nb - 1) << shift;
        remaining -= sh[1];
        __syncthreads();
    }
    const uint32_t T = prefix;
    const int need_eq = remaining;  // keys == T to take, >= 1
    // the selection: every key above d0, the keys of d0 above T, then the
    // need_eq smallest positions among the keys equal to T
    const int na = min(__ldcg(nabove + t), DSA_MAX_TOPK);  // == above
    for (int i = tid; i < na; i += NT) sel[i] = __ldcg(above_pos + (int64_t)t * DSA_MAX_TOPK + i);
    if (tid == 0) {
        sh[2] = na;  // next free slot of sel
        sh[3] = 0;   // ties found
    }
    __syncthreads();
    if (in_smem) {
        // compaction by prefix sums: thread tid takes candidates [i0, i1)
        const int per = (nc + NT - 1) / NT;
        const int i0 = min(tid * per, nc), i1 = min(i0 + per, nc);
        int ng = 0, nq = 0;
        for (int i = i0; i < i1; ++i) {
            ng += ck[i] > T;
            nq += ck[i] == T;
        }
        int tg, tq;
        int og = na + scan_threads<NT>(ng, buf, &tg);
        int oq = scan_threads<NT>(nq, buf, &tq);
        for (int i = i0; i < i1; ++i) {
            if (ck[i] > T) sel[og++] = cp[i];
            else if (ck[i] == T) tie[oq++] = cp[i];
        }
        if (tid == 0) {
            sh[2] = na + tg;
            sh[3] = tq;
        }
        __syncthreads();
        const int ne = sh[3];
        if (ne > need_eq) {  // keep the smallest positions
            int N = 1;
            while (N < ne) N <<= 1;
            for (int i = ne + tid; i < N; i += NT) tie[i] = INT_MAX;
            __syncthreads();
            bitonic_sort<NT>(tie, N);
        }
        const int base = sh[2];
        for (int i = tid; i < need_eq; i += NT) sel[base + i] = tie[i];
    } else {
        // keys of d0 above T from the row; ties in position order, block by block
        for (int j = tid; j < n; j += NT) {
            const uint32_t u = order_key(__ldg(row + j));
            if ((u & dmask) == dpre && u > T) sel[atomicAdd(sh + 2, 1)] = j;
        }
        __syncthreads();
        int taken = 0;
        const int base = sh[2];
        for (int j0 = 0; j0 < n && taken < need_eq; j0 += NT) {
            const int j = j0 + tid;
            const bool eq = j < n && order_key(__ldg(row + j)) == T;
            int tot;
            const int r = scan_threads<NT>(eq ? 1 : 0, buf, &tot);
            if (eq && taken + r < need_eq) sel[base + taken + r] = j;
            taken += tot;
        }
    }
    __syncthreads();
    // k positions, ascending (k <= 2048 slots, padded to a power of two)
    int N = 1;
    while (N < k) N <<= 1;
    for (int i = k + tid; i < N; i += NT) sel[i] = INT_MAX;
    __syncthreads();
    bitonic_sort<NT>(sel, N);
    for (int i = tid; i < k; i += NT) out[i] = sel[i];
    if (tid == 0) topk_len[t] = k;
}

namespace {

template <int THREADS, int EPT>
cudaError_t launch_row(const float* scores, int64_t ld, const dsa_seqs& s, int num_q, int k, int32_t* idx,
                       int32_t* topk_len, int32_t* d_status, cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(topk_row_kernel<THREADS, EPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kRowSmem);
    });
    if (attr != cudaSuccess) return attr;
    return launch_pdl(topk_row_kernel<THREADS, EPT>, dim3(num_q), dim3(THREADS), kRowSmem, stream, 1, scores, ld, s, k,
                      idx, topk_len, d_status);
}

template <int EPT>
cudaError_t launch_smem_row(const float* scores, int64_t ld, const dsa_seqs& s, int num_q, int k, int32_t* idx,
                            int32_t* topk_len, int32_t* d_status, cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(topk_smem_kernel<EPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem_row_bytes<EPT>());
    });
    if (attr != cudaSuccess) return attr;
    return launch_pdl(topk_smem_kernel<EPT>, dim3(num_q), dim3(1024), smem_row_bytes<EPT>(), stream, 1, scores, ld, s,
                      k, idx, topk_len, d_status);
}

}  // namespace

cudaError_t launch_topk(const float* scores, int64_t ld, const dsa_seqs& s, int num_q, int k, int32_t* idx,
                        int32_t* topk_len, const Workspace& ws, int32_t* d_status, cudaStream_t stream) {
    // rows up to 32,768 keys: one CTA per row
    if (s.max_ctx <= 1024 * 8)
        return launch_row<1024, 8>(scores, ld, s, num_q, k, idx, topk_len, d_status, stream);
    if (s.max_ctx <= 1024 * 16)
        return launch_row<1024, 16>(scores, ld, s, num_q, k, idx, topk_len, d_status, stream);
    if (s.max_ctx <= 1024 * 32)
        return launch_smem_row<32>(scores, ld, s, num_q, k, idx, topk_len, d_status, stream);
    const int C = topk_chunks(s.max_ctx);
    if (topk_chunked(s.max_ctx) && ws.tk_hist) {
        static std::once_flag once;
        static cudaError_t attr = cudaSuccess;
        std::call_once(once, [] {
            attr = cudaFuncSetAttribute(topk_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kFinalSmem);
        });
        if (attr != cudaSuccess) return attr;
        cudaError_t e = cudaMemsetAsync(ws.tk_hist, 0, (size_t)num_q * (2048 + 2) * 4, stream);
        if (e == cudaSuccess)
            e = launch_pdl(topk_hist_kernel, dim3(C, num_q), dim3(kLongThreads), 0, stream, 1, scores, ld, s, k,
                           ws.tk_hist);
        if (e == cudaSuccess)
            e = launch_pdl(topk_cand_kernel, dim3(C, num_q), dim3(kLongThreads), 0, stream, 1, scores, ld, s, k,
                           (const int*)ws.tk_hist, ws.tk_ncand, ws.tk_nabove, ws.tk_cand, ws.tk_above);
        if (e == cudaSuccess)
            e = launch_pdl(topk_final_kernel, dim3(num_q), dim3(kFinalThreads), kFinalSmem, stream, 1, scores, ld, s,
                           k, idx, topk_len, (const int*)ws.tk_hist, (const int*)ws.tk_ncand,
                           (const int*)ws.tk_nabove, (const uint2*)ws.tk_cand, (const int*)ws.tk_above, d_status);
        return e;
    }
    // rows longer than 16M keys: one CTA per row, passes over memory
    return launch_pdl(topk_kernel, dim3(num_q), dim3(kTopkThreads), 0, stream, 1, scores, ld, s, k, idx, topk_len,
                      d_status);
}

}  // namespace dsa
