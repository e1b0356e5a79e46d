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
#include <cooperative_groups.h>

#include <mutex>

#include "dsa_internal.cuh"

namespace cg = cooperative_groups;

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
template <int EPT>
constexpr size_t smem_row_bytes() {
    return (size_t)32 * (EPT * 1024 / 32 + 1) * 4 + (size_t)kRowSub * kRowBins * 4 + kRowCandCap * 4;
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
    uint32_t* cand = reinterpret_cast<uint32_t*>(sub + kRowSub * kRowBins);   // [kRowCandCap]
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
            // keep the keys of the chosen bin for the next two passes (prefix-sum slots)
            int mine = 0;
#pragma unroll 8
            for (int e = 0; e < nv; ++e) mine += (keys[e * KS + tid] & mask) == prefix;
            int nc;
            int sl = scan_threads<NT>(mine, scan_buf, &nc);
            if (nc <= kRowCandCap)
#pragma unroll 8
                for (int e = 0; e < nv; ++e) {
                    const uint32_t u = keys[e * KS + tid];
                    if ((u & mask) == prefix) cand[sl++] = u;
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
    int* stage_out = reinterpret_cast<int*>(cand);  // k <= kRowCandCap
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
// Register-resident variant: a thread-block cluster of CL CTAs per query row,
// each CTA holding 512 x EPT scores in registers, so the row is read from
// memory exactly once.  Three digit passes (11 + 11 + 10 bits): each CTA
// histograms its keys in shared memory (lanes of a warp that hit the same bin
// add with one atomic), CTA r of the cluster sums slice r of the CL histograms
// through distributed shared memory, and every CTA reads the merged slices
// and finds the same digit.  After the first pass only the keys of the chosen
// bin take part, compacted into shared memory when they fit.  The compaction
// ranks ties and positions across the cluster with prefix sums of per-CTA
// counts, so the output is the same as the one-CTA kernel's.
constexpr int kCT = 512;                 // threads per CTA
constexpr int kCBins = 2048;
constexpr int kCandCap = 4096;           // keys of the chosen bin kept in shared memory

// exclusive prefix sum over the kCT threads of a CTA
__device__ __forceinline__ int cta_exclusive_scan(int v, int* buf, int* total) {
    constexpr int W = kCT / 32;
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

__device__ __forceinline__ void hist_add(int* hist, bool act, int bin) {
    const unsigned am = __ballot_sync(0xffffffffu, act);
    if (act) {
        const unsigned peers = __match_any_sync(am, bin);
        if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(hist + bin, __popc(peers));
    }
}

template <int EPT>
__global__ void __launch_bounds__(kCT, EPT <= 16 ? 2 : 1)
    topk_cluster_kernel(const float* __restrict__ scores, int64_t ld, dsa_seqs s, int k, int32_t* __restrict__ idx,
                        int32_t* __restrict__ topk_len, int32_t* d_status) {
    pdl_enter();
    constexpr int kChunk = kCT * EPT;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int CL = (int)cluster.num_blocks();
    __shared__ int hist[kCBins];     // this CTA's histogram
    __shared__ int mhist[kCBins];    // merged counts of the bins this CTA owns
    __shared__ uint32_t cand[kCandCap];
    __shared__ int scan_buf[64];
    __shared__ int sel_digit, sel_above, ncand;
    __shared__ int cnt[2];
    const int t = blockIdx.y;
    const int tid = threadIdx.x;
    const int b = seq_of(s.q_start, s.num_seqs, t);
    const int pos = __ldg(s.q_pos + t);
    const int ctx = __ldg(s.ctx_len + b);
    int32_t* out = idx + (int64_t)t * k;
    // uniform per row: every CTA of the cluster takes the same branch
    if (pos < 0 || pos >= ctx || ctx > s.max_ctx || pos + 1 > CL * kChunk) {
        if (rank == 0) {
            if (tid == 0) {
                report(d_status, DSA_ERR_BAD_INPUT);
                topk_len[t] = 0;
            }
            for (int i = tid; i < k; i += kCT) out[i] = -1;
        }
        return;
    }
    const int n = pos + 1;
    if (n <= k) {
        if (rank == 0) {
            for (int i = tid; i < k; i += kCT) out[i] = i < n ? i : -1;
            if (tid == 0) topk_len[t] = n;
        }
        return;
    }
    // ---- this thread's EPT consecutive keys
    const float* row = scores + (int64_t)t * ld;
    const int base = rank * kChunk + tid * EPT;
    uint32_t u[EPT];
    uint64_t valid = 0;
#pragma unroll
    for (int v = 0; v < EPT / 4; ++v) {
        const int i0 = base + 4 * v;
        float4 f;
        if (i0 + 3 < n) {
            f = __ldg(reinterpret_cast<const float4*>(row + i0));
        } else {
            f.x = i0 < n ? __ldg(row + i0) : 0.f;
            f.y = i0 + 1 < n ? __ldg(row + i0 + 1) : 0.f;
            f.z = i0 + 2 < n ? __ldg(row + i0 + 2) : 0.f;
            f.w = i0 + 3 < n ? __ldg(row + i0 + 3) : 0.f;
        }
        u[4 * v] = order_key(f.x);
        u[4 * v + 1] = order_key(f.y);
        u[4 * v + 2] = order_key(f.z);
        u[4 * v + 3] = order_key(f.w);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (i0 + e < n) valid |= 1ull << (4 * v + e);
    }
    // ---- three digit passes
    uint32_t prefix = 0, mask = 0;
    int remaining = k;
    bool use_cand = false;
    if (tid == 0) ncand = 0;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nb = pass == 2 ? 1024 : 2048;
        for (int i = tid; i < kCBins; i += kCT) hist[i] = 0;
        __syncthreads();
        if (use_cand) {
            const int nc = ncand, nc_r = (nc + 31) & ~31;  // whole warps take part in hist_add
            for (int i = tid; i < nc_r; i += kCT) {
                const bool act = i < nc && (cand[i < nc ? i : 0] & mask) == prefix;
                hist_add(hist, act, act ? (cand[i] >> shift) & (nb - 1) : 0);
            }
        } else {
#pragma unroll
            for (int e = 0; e < EPT; ++e) {
                const bool act = ((valid >> e) & 1) && (u[e] & mask) == prefix;
                hist_add(hist, act, (u[e] >> shift) & (nb - 1));
            }
        }
        cluster.sync();  // A: every CTA's histogram is final
        // merge slice `rank` of the bins over the cluster
        const int slice = nb / CL;
        for (int i = tid; i < slice; i += kCT) {
            const int bin = rank * slice + i;
            int v = 0;
            for (int r = 0; r < CL; ++r) v += cluster.map_shared_rank(hist, r)[bin];
            mhist[bin] = v;
        }
        cluster.sync();  // B: merged slices final
        // digits in descending order, 4 per thread, read from their owners
        int c[4], csum = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int d = nb - 1 - 4 * tid - q;
            const int v = d >= 0 ? cluster.map_shared_rank(mhist, d / slice)[d] : 0;
            c[q] = v;
            csum += v;
        }
        int tot;
        int before = cta_exclusive_scan(csum, scan_buf, &tot);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (before < remaining && before + c[q] >= remaining) {
                sel_digit = nb - 1 - 4 * tid - q;
                sel_above = before;
            }
            before += c[q];
        }
        cluster.sync();  // C: every CTA is done reading histograms; the digit is visible
        prefix |= (uint32_t)sel_digit << shift;
        mask |= (uint32_t)(nb - 1) << shift;
        remaining -= sel_above;
        if (pass == 0) {
            // keep the keys of the chosen bin for the next two passes
            const int lane = tid & 31;
#pragma unroll
            for (int e = 0; e < EPT; ++e) {
                const bool act = ((valid >> e) & 1) && (u[e] & mask) == prefix;
                const unsigned am = __ballot_sync(0xffffffffu, act);
                int slot0 = 0;
                if (lane == 0 && am) slot0 = atomicAdd(&ncand, __popc(am));
                slot0 = __shfl_sync(0xffffffffu, slot0, 0);
                const int sl = slot0 + __popc(am & ((1u << lane) - 1));
                if (act && sl < kCandCap) cand[sl] = u[e];
            }
            __syncthreads();
            use_cand = ncand <= kCandCap;
        }
    }
    const uint32_t T = prefix;
    const int need_eq = remaining;
    // ---- cluster-wide ranks: keys > T and keys == T, in index order
    int n_gt = 0, n_eq = 0;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        const bool vld = (valid >> e) & 1;
        n_gt += vld && u[e] > T;
        n_eq += vld && u[e] == T;
    }
    int gt_cta, eq_cta;
    cta_exclusive_scan(n_gt, scan_buf, &gt_cta);
    const int eq_before = cta_exclusive_scan(n_eq, scan_buf, &eq_cta);
    if (tid == 0) {
        cnt[0] = gt_cta;
        cnt[1] = eq_cta;
    }
    cluster.sync();
    int gt_prefix = 0, eq_prefix = 0;
    for (int r = 0; r < rank; ++r) {
        const int* rc = cluster.map_shared_rank(cnt, r);
        gt_prefix += rc[0];
        eq_prefix += rc[1];
    }
    int eq_rank = eq_prefix + eq_before;
    const int n_sel = n_gt + max(0, min(need_eq - eq_rank, n_eq));
    int sel_cta;
    int o = gt_prefix + min(need_eq, eq_prefix) + cta_exclusive_scan(n_sel, scan_buf, &sel_cta);
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        if (!((valid >> e) & 1)) continue;
        bool take = u[e] > T;
        if (u[e] == T) take = eq_rank++ < need_eq;
        if (take && o < k) out[o++] = base + e;
    }
    if (rank == 0 && tid == 0) topk_len[t] = k;
    cluster.sync();  // no CTA leaves while another may still read its counts
}

namespace {

struct ClusterPlan {
    int cl, ept;
};

// CTAs per row and keys per thread: enough capacity for the longest row, then
// more CTAs per row (down to 16 keys per thread) until the launch fills the GPU.
ClusterPlan topk_plan(int max_ctx, int num_q) {
    ClusterPlan p{1, 64};
    while (p.cl * kCT * 64 < max_ctx) p.cl *= 2;
    while (p.cl < 16 && p.cl * num_q < 256 && (p.cl * 2) * kCT * 16 <= max_ctx * 2) p.cl *= 2;
    p.ept = 16;
    while (p.cl * kCT * p.ept < max_ctx) p.ept *= 2;
    return p;
}

template <int EPT>
int max_cluster() {
    static std::once_flag once;
    static int max_ok = 0;
    std::call_once(once, [] {
        cudaFuncSetAttribute(topk_cluster_kernel<EPT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        for (int c = 1; c <= 16; c *= 2) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(c, 1, 1);
            cfg.blockDim = dim3(kCT, 1, 1);
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = c;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, topk_cluster_kernel<EPT>, &cfg) == cudaSuccess && n > 0) max_ok = c;
            else break;
        }
        cudaGetLastError();
    });
    return max_ok;
}

template <int EPT>
cudaError_t launch_cluster(int cl, const float* scores, int64_t ld, const dsa_seqs& s, int num_q, int k,
                           int32_t* idx, int32_t* topk_len, int32_t* d_status, cudaStream_t stream) {
    return launch_pdl(topk_cluster_kernel<EPT>, dim3(cl, num_q), dim3(kCT), 0, stream, cl, scores, ld, s, k, idx,
                      topk_len, d_status);
}


}  // namespace

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

cudaError_t launch_topk(const float* scores, int64_t ld, const dsa_seqs& s, int num_q, int k, int32_t* idx,
                        int32_t* topk_len, int32_t* d_status, cudaStream_t stream) {
    // rows up to 32,768 keys: one CTA per row
    if (s.max_ctx <= 1024 * 8)
        return launch_row<1024, 8>(scores, ld, s, num_q, k, idx, topk_len, d_status, stream);
    if (s.max_ctx <= 1024 * 16)
        return launch_row<1024, 16>(scores, ld, s, num_q, k, idx, topk_len, d_status, stream);
    if (s.max_ctx <= 1024 * 32)
        return launch_smem_row<32>(scores, ld, s, num_q, k, idx, topk_len, d_status, stream);
    const ClusterPlan p = topk_plan(s.max_ctx, num_q);
    if (p.cl <= 16 && p.ept <= 64) {
        if (p.ept == 16 && p.cl <= max_cluster<16>())
            return launch_cluster<16>(p.cl, scores, ld, s, num_q, k, idx, topk_len, d_status, stream);
        if (p.ept == 32 && p.cl <= max_cluster<32>())
            return launch_cluster<32>(p.cl, scores, ld, s, num_q, k, idx, topk_len, d_status, stream);
        if (p.ept == 64 && p.cl <= max_cluster<64>())
            return launch_cluster<64>(p.cl, scores, ld, s, num_q, k, idx, topk_len, d_status, stream);
    }
    // rows longer than 16 x 32,768 keys: one CTA per row, passes over memory
    return launch_pdl(topk_kernel, dim3(num_q), dim3(kTopkThreads), 0, stream, 1, scores, ld, s, k, idx, topk_len,
                      d_status);
}

}  // namespace dsa
