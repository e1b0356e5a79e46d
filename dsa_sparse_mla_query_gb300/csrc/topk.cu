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
// Three kernels share that scheme, one CTA per row each: rows up to 16,384
// keys with the row in registers, up to 32,768 keys with the row in shared
// memory (three passes of 11 + 11 + 10 bits), longer rows streamed from
// memory in blocks (the first digit over the row, the finer two over the
// keys of the chosen first digit).

#include <cooperative_groups.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <mutex>

#include "dsa_internal.cuh"


namespace dsa {

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;  // -0.0 ranks as +0.0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
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
// Rows longer than 32,768 keys (any length): a thread-block cluster of P CTAs
// per row (P = 1 when the rows alone fill the GPU, up to 8 for a few long
// rows); CTA r streams its contiguous share of the row's 16,384-key blocks,
// thread t holding 16 consecutive positions of a block (four float4 from one
// 64-byte run), so that thread order is position order:
//   1. the first digit's histogram over the row (the row from HBM), summed
//      over the cluster in distributed shared memory: the digit d0 of the
//      k-th key and the number of keys above it;
//   2. the positions above d0 (fewer than k) and the keys of d0 with their
//      positions, each list ascending (the row again, mostly from L2);
//   3. two finer digits (11 + 10 bits) over the lists of the cluster (over
//      the row when a list overflowed): the k-th key T and how many keys == T
//      to take;
//   4. each CTA's count of selected keys (and of keys == T) through the
//      cluster: its slice of the output, where it merges its two ascending
//      lists.
// No global atomics, no scratch, no sort; every barrier is over the cluster,
// whose CTAs run together.
constexpr int kStreamThreads = 1024;
constexpr int kStreamEPT = 16;
constexpr int kStreamBlock = kStreamThreads * kStreamEPT;  // 16384 keys
constexpr int kStreamCand = 8192;                           // keys of d0 a CTA lists
constexpr int kSampleBlocks = 4;                            // blocks a CTA needs for the sampled pass
constexpr int kStreamMaxP = 8;
// h [4][2048], hs [2048], ck/cp [kStreamCand], ap [2048], sel [2048]
constexpr size_t kStreamSmem = (size_t)(5 * 2048 + 2 * kStreamCand + 2 * DSA_MAX_TOPK) * 4;

__device__ __forceinline__ int stream_pos(int j0, int e) { return j0 + (int)threadIdx.x * kStreamEPT + e; }

// this thread's 16 positions of the block at j0 as order keys (loads clamped into the row)
__device__ __forceinline__ void stream_block(const float* row, int last4, int j0, uint32_t (&u)[kStreamEPT]) {
    uint4 r[kStreamEPT / 4];
#pragma unroll
    for (int v = 0; v < kStreamEPT / 4; ++v)
        r[v] = __ldg(reinterpret_cast<const uint4*>(row + min(stream_pos(j0, 4 * v), last4)));
#pragma unroll
    for (int v = 0; v < kStreamEPT / 4; ++v) {
        u[4 * v] = order_key(__uint_as_float(r[v].x));
        u[4 * v + 1] = order_key(__uint_as_float(r[v].y));
        u[4 * v + 2] = order_key(__uint_as_float(r[v].z));
        u[4 * v + 3] = order_key(__uint_as_float(r[v].w));
    }
}

// the digit (of nb, descending, 1 or 2 per thread) holding the remaining-th
// key in the histogram hs, and the keys in higher digits; every thread
template <int NT>
__device__ __forceinline__ void select_digit(const int* hs, int nb, int remaining, int* buf, int* sh, int& digit,
                                             int& above) {
    const int per = nb / NT;
    const int dA = nb - 1 - per * (int)threadIdx.x;
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
    digit = sh[0];
    above = sh[1];
    __syncthreads();
}

// hs = the sum over the cluster's CTAs of their local histograms h (after a
// cluster barrier that makes them complete)
__device__ __forceinline__ void cluster_hist_sum(cooperative_groups::cluster_group& cl, int* h, int* hs, int P) {
    for (int i = threadIdx.x; i < 2048; i += kStreamThreads) {
        int v = 0;
        for (int r = 0; r < P; ++r) v += cl.map_shared_rank(h, r)[i];
        hs[i] = v;
    }
}

// first index i of a[0 .. n) (ascending) with a[i] > v
__device__ __forceinline__ int upper_idx(const int* a, int n, int v) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] <= v) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(kStreamThreads, 1) topk_stream_kernel(const float* __restrict__ scores, int64_t ld,
                                                                         dsa_seqs s, int k, int32_t* __restrict__ idx,
                                                                         int32_t* __restrict__ topk_len,
                                                                         int32_t* d_status) {
    constexpr int NT = kStreamThreads;
    pdl_enter();
    cooperative_groups::cluster_group cl = cooperative_groups::this_cluster();
    const int P = (int)cl.num_blocks(), me = (int)cl.block_rank();
    extern __shared__ __align__(16) int st_smem[];
    int* h = st_smem;                                        // [4][2048] local histograms (h[0..2048): their sum)
    int* hs = h + 4 * 2048;                                  // [2048] the cluster's histogram
    uint32_t* ck = reinterpret_cast<uint32_t*>(hs + 2048);  // [kStreamCand] keys of d0 in this CTA's range
    int* cp = reinterpret_cast<int*>(ck + kStreamCand);     // [kStreamCand] their positions
    int* ap = cp + kStreamCand;                              // [DSA_MAX_TOPK] positions above d0 (this range)
    int* sel = ap + DSA_MAX_TOPK;                            // [DSA_MAX_TOPK] selected positions of d0 (this range)
    __shared__ int buf[64], sh[2], xch[4];
    const int t = blockIdx.x / P, tid = threadIdx.x, warp = tid >> 5;
    const int b = seq_of(s.q_start, s.num_seqs, t);
    const int pos = __ldg(s.q_pos + t);
    const int ctx = __ldg(s.ctx_len + b);
    int32_t* out = idx + (int64_t)t * k;
    // (the same row for every CTA of the cluster: these exits are uniform)
    if (pos < 0 || pos >= ctx || ctx > s.max_ctx) {
        if (me == 0) {
            if (tid == 0) {
                report(d_status, DSA_ERR_BAD_INPUT);
                topk_len[t] = 0;
            }
            for (int i = tid; i < k; i += NT) out[i] = -1;
        }
        return;
    }
    const int n = pos + 1;
    if (n <= k) {
        if (me == 0) {
            for (int i = tid; i < k; i += NT) out[i] = i < n ? i : -1;
            if (tid == 0) topk_len[t] = n;
        }
        return;
    }
    const float* row = scores + (int64_t)t * ld;
    const int last4 = (int)((ld - 4) & ~(int64_t)3);
    const int nblk = (n + kStreamBlock - 1) / kStreamBlock;
    const int b0 = (int)((int64_t)nblk * me / P), b1 = (int)((int64_t)nblk * (me + 1) / P);  // this CTA's blocks
    uint32_t u[kStreamEPT];
    int d0 = 0, na = 0, nc = 0, remaining = k;  // na, nc: this CTA's so far (the same in every thread)
    uint32_t prefix = 0, mask = 0;
    bool over = false;

    // ---- 0: one pass, when a sample allows: every CTA samples one key per
    // thread over its range; the cluster's sample histogram gives the first
    // digit holding its (mu + 4 sqrt(mu) + 2)-th largest key, mu = the number
    // of sampled keys expected among the top k; each CTA then lists every key
    // of that digit or above, with its position, in position order.  When the
    // lists fit and hold at least k keys (the row's k-th key is then theirs),
    // three digit passes over them pin the k-th key; otherwise steps 1-2 run.
    // Only CTAs with kSampleBlocks blocks or more sample: over fewer, the
    // second pass of steps 1-2 reads blocks still in L2, and the sample's
    // fixed costs (scattered loads, a digit selection, one more pass over a
    // longer list) outweigh it.  (nblk and P are the cluster's: uniform.)
    bool sampled = false;
    if (nblk >= kSampleBlocks * P) {
        for (int i = tid; i < 2048; i += NT) h[i] = 0;
        const int j_lo = b0 * kStreamBlock, j_hi = min(b1 * kStreamBlock, n);
        const bool has = j_hi > j_lo;
        const int sp = has ? j_lo + (int)((int64_t)(j_hi - j_lo) * tid / NT) : 0;
        const uint32_t sk = has ? order_key(__ldg(row + sp)) : 0u;
        __syncthreads();
        if (has) atomicAdd(h + (sk >> 21), 1);
        const int ns_me = __syncthreads_count(has);
        if (tid == 0) xch[0] = ns_me;
        cl.sync();  // every CTA's sample histogram and count
        cluster_hist_sum(cl, h, hs, P);
        int ns = 0;
        for (int r = 0; r < P; ++r) ns += cl.map_shared_rank(xch, r)[0];
        __syncthreads();
        const float mu = (float)ns * (float)k / (float)n;
        const int target = (int)ceilf(mu + 4.f * sqrtf(mu) + 2.f);
        const bool try_list = ns >= target;  // the same in every CTA of the cluster
        if (try_list) {
            int dth, abv;
            select_digit<NT>(hs, 2048, target, buf, sh, dth, abv);
            const uint32_t thr = (uint32_t)dth << 21;
            for (int blk = b0; blk < b1; ++blk) {
                const int j0 = blk * kStreamBlock;
                stream_block(row, last4, j0, u);
                int cc = 0;
#pragma unroll
                for (int e = 0; e < kStreamEPT; ++e) cc += stream_pos(j0, e) < n && u[e] >= thr;
                int tot;
                int oc = nc + scan_threads<NT>(cc, buf, &tot);
#pragma unroll
                for (int e = 0; e < kStreamEPT; ++e) {
                    const int p = stream_pos(j0, e);
                    if (p < n && u[e] >= thr) {
                        if (oc < kStreamCand) {
                            ck[oc] = u[e];
                            cp[oc] = p;
                        }
                        ++oc;
                    }
                }
                nc += tot;
            }
        }
        // (also: every CTA is done with the others' sample histograms)
        if (tid == 0) {
            xch[1] = nc;
            xch[2] = nc > kStreamCand;
        }
        cl.sync();
        int total = 0;
        bool ovf = false;
        for (int r = 0; r < P; ++r) {
            const int* x = cl.map_shared_rank(xch, r);
            total += x[1];
            ovf |= x[2] != 0;
        }
        sampled = try_list && !ovf && total >= k;
    }
    if (!sampled) {
        nc = 0;
        // ---- 1: the first digit over the row
        for (int i = tid; i < 4 * 2048; i += NT) h[i] = 0;
        __syncthreads();
        {
            int* hw = h + (warp & 3) * 2048;  // four copies spread the same-address atomics
            for (int blk = b0; blk < b1; ++blk) {
                const int j0 = blk * kStreamBlock;
                stream_block(row, last4, j0, u);
    #pragma unroll
                for (int e = 0; e < kStreamEPT; ++e)
                    if (stream_pos(j0, e) < n) atomicAdd(hw + (u[e] >> 21), 1);
            }
        }
        __syncthreads();
        for (int i = tid; i < 2048; i += NT) h[i] += h[2048 + i] + h[4096 + i] + h[6144 + i];
        cl.sync();
        cluster_hist_sum(cl, h, hs, P);
        __syncthreads();
        int above;
        select_digit<NT>(hs, 2048, k, buf, sh, d0, above);
        prefix = (uint32_t)d0 << 21;
        mask = 0x7FFu << 21;
        remaining = k - above;

        // ---- 2: the positions above d0 and the keys of d0, ascending
        na = 0;
        nc = 0;  // this CTA's so far (the same in every thread)
        for (int blk = b0; blk < b1; ++blk) {
            const int j0 = blk * kStreamBlock;
            stream_block(row, last4, j0, u);
            int ca = 0, cc = 0;
    #pragma unroll
            for (int e = 0; e < kStreamEPT; ++e) {
                const int dg = stream_pos(j0, e) < n ? (int)(u[e] >> 21) : -1;
                ca += dg > d0;
                cc += dg == d0;
            }
            int tot;
            const int pk = scan_threads<NT>((ca << 16) | cc, buf, &tot);  // each at most 16384 per block
            int oa = na + (pk >> 16), oc = nc + (pk & 0xFFFF);
    #pragma unroll
            for (int e = 0; e < kStreamEPT; ++e) {
                const int p = stream_pos(j0, e);
                const int dg = p < n ? (int)(u[e] >> 21) : -1;
                if (dg > d0) {
                    if (oa < DSA_MAX_TOPK) ap[oa] = p;
                    ++oa;
                } else if (dg == d0) {
                    if (oc < kStreamCand) {
                        ck[oc] = u[e];
                        cp[oc] = p;
                    }
                    ++oc;
                }
            }
            na += tot >> 16;
            nc += tot & 0xFFFF;
        }
        if (tid == 0) xch[0] = nc > kStreamCand;
        cl.sync();  // also: every CTA has summed the others' first histograms
        over = false;  // some CTA's list of d0 overflowed: the finer digits come from the row
        for (int r = 0; r < P; ++r) over |= cl.map_shared_rank(xch, r)[0] != 0;
    }

    // ---- 3: the digits not yet pinned (the two finer ones after steps 1-2,
    // all three over the sampled lists), over the cluster's lists
#pragma unroll 1
    for (int pass = sampled ? 0 : 1; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nb = pass == 2 ? 1024 : 2048;
        for (int i = tid; i < 2048; i += NT) h[i] = 0;
        __syncthreads();
        if (!over) {
            for (int i = tid; i < nc; i += NT)
                if ((ck[i] & mask) == prefix) atomicAdd(h + ((ck[i] >> shift) & (nb - 1)), 1);
        } else {
            for (int blk = b0; blk < b1; ++blk) {
                const int j0 = blk * kStreamBlock;
                stream_block(row, last4, j0, u);
#pragma unroll
                for (int e = 0; e < kStreamEPT; ++e)
                    if (stream_pos(j0, e) < n && (u[e] & mask) == prefix)
                        atomicAdd(h + ((u[e] >> shift) & (nb - 1)), 1);
            }
        }
        cl.sync();
        cluster_hist_sum(cl, h, hs, P);
        cl.sync();  // every CTA has read the others' histograms before they change
        int dg, ab;
        select_digit<NT>(hs, nb, remaining, buf, sh, dg, ab);
        prefix |= (uint32_t)dg << shift;
        mask |= (uint32_t)(nb - 1) << shift;
        remaining -= ab;
    }
    const uint32_t T = prefix;
    const int need_eq = remaining;  // keys == T to take over the row, >= 1

    // ---- 4: this CTA's keys of d0 above T and equal to T; through the
    // cluster, its slice of the output and its share of the keys == T
    int g_me, e_me;
    {
        int gt = 0, eq = 0;
        if (!over) {
            for (int i = tid; i < nc; i += NT) {
                gt += ck[i] > T;
                eq += ck[i] == T;
            }
        } else {
            for (int blk = b0; blk < b1; ++blk) {
                const int j0 = blk * kStreamBlock;
                stream_block(row, last4, j0, u);
#pragma unroll
                for (int e = 0; e < kStreamEPT; ++e)
                    if (stream_pos(j0, e) < n && (int)(u[e] >> 21) == d0) {
                        gt += u[e] > T;
                        eq += u[e] == T;
                    }
            }
        }
        scan_threads<NT>(gt, buf, &g_me);
        scan_threads<NT>(eq, buf, &e_me);
    }
    if (tid == 0) {
        xch[1] = na;
        xch[2] = g_me;
        xch[3] = e_me;
    }
    cl.sync();
    int eq_before = 0, out_before = 0;  // over the cluster's earlier CTAs (earlier positions)
    for (int r = 0; r < me; ++r) {
        const int* x = cl.map_shared_rank(xch, r);
        out_before += x[1] + x[2] + max(0, min(need_eq - eq_before, x[3]));
        eq_before += x[3];
    }
    const int quota = max(0, min(need_eq - eq_before, e_me));  // keys == T this CTA takes
    const int m = min(g_me + quota, DSA_MAX_TOPK);

    // ---- 5: this CTA's selected keys of d0, ascending, merged with its
    // positions above d0 into its slice of the output
    if (!over) {
        const int per = (nc + NT - 1) / NT;  // consecutive list entries per thread
        const int i0 = min(tid * per, nc), i1 = min(i0 + per, nc);
        int ng = 0, nq = 0;
        for (int i = i0; i < i1; ++i) {
            ng += ck[i] > T;
            nq += ck[i] == T;
        }
        int tq;
        int er = scan_threads<NT>(nq, buf, &tq);
        const int ns = ng + max(0, min(quota - er, nq));
        int tb;
        int o = scan_threads<NT>(ns, buf, &tb);
        for (int i = i0; i < i1; ++i) {
            bool take = ck[i] > T;
            if (ck[i] == T) take = er++ < quota;
            if (take && o < DSA_MAX_TOPK) sel[o++] = cp[i];
        }
    } else {
        int o_base = 0, er_base = 0;
        for (int blk = b0; blk < b1 && o_base < m; ++blk) {
            const int j0 = blk * kStreamBlock;
            stream_block(row, last4, j0, u);
            int ng = 0, nq = 0;
#pragma unroll
            for (int e = 0; e < kStreamEPT; ++e)
                if (stream_pos(j0, e) < n && (int)(u[e] >> 21) == d0) {
                    ng += u[e] > T;
                    nq += u[e] == T;
                }
            int tot;
            const int pk = scan_threads<NT>((ng << 16) | nq, buf, &tot);  // each at most 16384 per block
            const int left = max(quota - er_base, 0);                     // keys == T still to take
            int er = er_base + (pk & 0xFFFF);
            int o = o_base + (pk >> 16) + min(left, pk & 0xFFFF);
#pragma unroll
            for (int e = 0; e < kStreamEPT; ++e) {
                const int p = stream_pos(j0, e);
                if (p >= n || (int)(u[e] >> 21) != d0) continue;
                bool take = u[e] > T;
                if (u[e] == T) take = er++ < quota;
                if (take && o < DSA_MAX_TOPK) sel[o++] = p;
            }
            o_base += (tot >> 16) + min(left, tot & 0xFFFF);
            er_base += tot & 0xFFFF;
        }
    }
    __syncthreads();
    const int nna = min(na, DSA_MAX_TOPK);
    for (int i = tid; i < nna; i += NT) {
        const int v = ap[i];
        const int at = out_before + i + upper_idx(sel, m, v);
        if (at < k) out[at] = v;
    }
    for (int j = tid; j < m; j += NT) {
        const int v = sel[j];
        const int at = out_before + j + upper_idx(ap, nna, v);
        if (at < k) out[at] = v;
    }
    if (me == 0 && tid == 0) topk_len[t] = k;
    cl.sync();  // no CTA leaves while another may still read its shared memory
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
    (void)ws;  // no scratch
    // rows up to 32,768 keys: one CTA per row
    if (s.max_ctx <= 1024 * 8)
        return launch_row<1024, 8>(scores, ld, s, num_q, k, idx, topk_len, d_status, stream);
    if (s.max_ctx <= 1024 * 16)
        return launch_row<1024, 16>(scores, ld, s, num_q, k, idx, topk_len, d_status, stream);
    if (s.max_ctx <= 1024 * 32)
        return launch_smem_row<32>(scores, ld, s, num_q, k, idx, topk_len, d_status, stream);
    // longer rows: a cluster of P CTAs per row streams the row; P fills the
    // GPU's SMs when the rows are few (a power of two, at most 8, and no more
    // than the longest row's blocks)
    int P = 1;
    while (P < kStreamMaxP && (int64_t)num_q * P * 2 <= 152 && P * kStreamBlock < s.max_ctx) P *= 2;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(topk_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStreamSmem);
    });
    if (attr != cudaSuccess) return attr;
    return launch_pdl(topk_stream_kernel, dim3((unsigned)num_q * P), dim3(kStreamThreads), kStreamSmem, stream, P,
                      scores, ld, s, k, idx, topk_len, d_status);
}

}  // namespace dsa
