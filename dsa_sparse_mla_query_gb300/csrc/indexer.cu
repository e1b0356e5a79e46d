// indexer.cu -- query preparation and lightning-indexer scores (sm_103a).
//
// Definition ([colibri] "Mistral-Large-4 (c/colibri.c)", What differs from
// GLM-5.2: SSMax, The indexer, RoPE and the rest; "Day 0 support for Mistral
// Large 4", Model architecture and NoPE, SSMax and LeRoPE):
//   f_h = s_h ln(pos+1) + b_h,  q_h <- f_h q_h,  RoPE layers rotate the pairs
//   (2i, 2i+1), i < 32, by pos*inv_freq_i;
//   score(t, j) = sum_h w_h relu(q_h . k_j / sqrt(128)) / sqrt(32).
//
// Exact refolding used here (same value, fewer roundings on the device):
//   relu(f x) = |f| relu(sgn(f) x), and sqrt(128) sqrt(32) = 64, so
//   score = sum_h w'_h relu(q'_h . k_j) with w'_h = w_h |f_h| / 64 and
//   q'_h = sgn(f_h) rot(q_h).  The unrotated dims of q' stay exact bf16; the 64
//   rotated dims (exact fp64 angle, fp32 rotation) are split into hi + lo 16-bit
//   parts, so the contraction runs over K = 192 columns [hi | lo | unrotated]
//   against key dims [0..63 | 0..63 | 64..127] and reproduces the fp64 query to
//   ~2^-17 relative.  That keeps the top-k boundary exact (see dsa_topk).
//   e4m3 keys decode exactly to f16, so the fp8 path runs the same contraction
//   in f16 and multiplies the per-row scale after the relu-weighted sum
//   (scale >= 0).
#include "indexer_common.cuh"

namespace dsa {

// ---------------------------------------------------------------------------
// query preparation: q' [Q, 32, KP] (KP = 192 RoPE, 128 NoPE), w' [Q, 32]
//
// The 32 rotation angles of a query are formed in fp64, where pos*inv_freq is
// exact (it reaches ~5e5 rad at 512K context, where an fp32 angle would lose
// the phase), reduced by 2 pi in fp64 and passed to fp32 sincos; the 32 SSMax
// factors s log(pos + 1) + b are fp32.  The rotation of the exact bf16 inputs
// runs in fp32 with fused multiply-adds (relative error ~2^-22, below the
// 2^-17 of the hi + lo split).  GB300's fp64 rate is tiny: only the angle and
// its reduction stay in fp64.
template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }
template <typename T>
__device__ __forceinline__ float to_float(T x);
template <>
__device__ __forceinline__ float to_float<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <>
__device__ __forceinline__ float to_float<__half>(__half x) { return __half2float(x); }

template <typename T>
__global__ void __launch_bounds__(kIH * 16) qprep_kernel(const __nv_bfloat16* __restrict__ q, const float* __restrict__ w,
                                                    const float* __restrict__ ss, const float* __restrict__ sb,
                                                    const float* __restrict__ inv_freq, dsa_seqs s, int num_q,
                                                    T* __restrict__ qp, float* __restrict__ wp,
                                                    int32_t* d_status) {
    pdl_enter();
    const int t = blockIdx.x;
    const bool rope = inv_freq != nullptr;
    const int KP = rope ? 192 : 128;
    __shared__ float cs[32], sn[32], sgn[32], wsc[32];
    __shared__ int ok;
    // one thread = 4 consecutive pairs (8 dims) of one head, its load in
    // flight during the per-query setup
    const __nv_bfloat16* qt = q + (int64_t)t * kIH * kID;
    T* out = qp + (int64_t)t * kIH * KP;
    const int h = threadIdx.x >> 4, c8 = threadIdx.x & 15;  // dims 8*c8 .. 8*c8+7
    const uint4 raw = *reinterpret_cast<const uint4*>(qt + h * kID + c8 * 8);
    qprep_setup(w, ss, sb, inv_freq, s, t, cs, sn, sgn, wsc, &ok, d_status);
    if (threadIdx.x < 32) wp[(int64_t)t * kIH + threadIdx.x] = wsc[threadIdx.x];
    {
        const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&raw);
        const float g = ok ? sgn[h] : 0.f;
        T* o = out + h * KP;
        alignas(16) T hi[8];
        alignas(16) T lo[8];
        if (rope && c8 < 8) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int p = c8 * 4 + u;
                const float x0 = __bfloat162float(x[2 * u]), x1 = __bfloat162float(x[2 * u + 1]);
                const float y0 = g * fmaf(x0, cs[p], -x1 * sn[p]);
                const float y1 = g * fmaf(x0, sn[p], x1 * cs[p]);
                hi[2 * u] = from_float<T>(y0);
                hi[2 * u + 1] = from_float<T>(y1);
                lo[2 * u] = from_float<T>(y0 - to_float<T>(hi[2 * u]));
                lo[2 * u + 1] = from_float<T>(y1 - to_float<T>(hi[2 * u + 1]));
            }
            *reinterpret_cast<uint4*>(o + c8 * 8) = *reinterpret_cast<const uint4*>(hi);
            *reinterpret_cast<uint4*>(o + 64 + c8 * 8) = *reinterpret_cast<const uint4*>(lo);
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) hi[u] = from_float<T>(g * __bfloat162float(x[u]));
            *reinterpret_cast<uint4*>(o + (rope ? 64 : 0) + c8 * 8) = *reinterpret_cast<const uint4*>(hi);
        }
    }
}

// e4m3 index keys: the tensor cores take both operands in e4m3
// (kind::f8f6f4), straight from the key tiles in shared memory.  q' (fp32,
// sign-folded and rotated as above) is split per head into three e4m3 parts,
//   q' = s (c_0 + 2^-4 c_1 + 2^-8 c_2),
// with s the smallest power of two that keeps max |q'| / s <= 448 (e4m3's
// largest value): each part rounds the remaining residual to 4 significant
// bits, so q' is kept to ~2^-12 relative (measured: scores within 2e-5 of
// the row maximum of those from four parts), and every residual fits its
// part's range (it is at most half an e4m3 ulp of the previous part, <= 16
// units).  Each step (scaling by a power of two, the residual's subtraction)
// is exact.  s is folded into the head weight, since relu(s x) = s relu(x):
// w'' = w |f| s / 64.  Layout: [Q][3 parts][32 heads][128] e4m3 codes, one
// 128-byte row per (query, part, head): the MMA's N rows.
constexpr int kQParts = 3;  // e4m3 parts of q' (e4m3 index keys)

__global__ void __launch_bounds__(kIH * 32) qprep_e4m3_kernel(const __nv_bfloat16* __restrict__ q,
                                                         const float* __restrict__ w, const float* __restrict__ ss,
                                                         const float* __restrict__ sb,
                                                         const float* __restrict__ inv_freq, dsa_seqs s, int num_q,
                                                         uint8_t* __restrict__ qp, float* __restrict__ wp,
                                                         int32_t* d_status) {
    pdl_enter();
    const int t = blockIdx.x;
    const bool rope = inv_freq != nullptr;
    __shared__ float cs[32], sn[32], sgn[32], wsc[32];
    __shared__ int ok;
    // warp h: head h; lane: dims 4 lane .. 4 lane + 3, i.e. rotation pairs 2
    // lane and 2 lane + 1 (the load in flight during the per-query setup)
    const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint2 raw = *reinterpret_cast<const uint2*>(q + ((int64_t)t * kIH + h) * kID + 4 * lane);
    qprep_setup(w, ss, sb, inv_freq, s, t, cs, sn, sgn, wsc, &ok, d_status);
    {
        const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&raw);
        const float g = ok ? sgn[h] : 0.f;
        float y[4];
        if (rope && lane < 16) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int p = 2 * lane + u;
                const float x0 = __bfloat162float(x[2 * u]), x1 = __bfloat162float(x[2 * u + 1]);
                y[2 * u] = g * fmaf(x0, cs[p], -x1 * sn[p]);
                y[2 * u + 1] = g * fmaf(x0, sn[p], x1 * cs[p]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) y[i] = g * __bfloat162float(x[i]);
        }
        float m = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        int e = 0;
        if (m > 0.f) frexpf(m * (1.f / 448.f), &e);  // m / 448 <= 2^e
        uint8_t* out = qp + (((int64_t)t * kQParts) * kIH + h) * kID + 4 * lane;
#pragma unroll
        for (int part = 0; part < kQParts; ++part) {
            const int pe = e - 4 * part;  // this part's scale is 2^pe
            uint32_t word = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(ldexpf(y[i], -pe), __NV_SATFINITE, __NV_E4M3);
                const __half_raw hv = __nv_cvt_fp8_to_halfraw(c, __NV_E4M3);
                y[i] -= ldexpf(__half2float(__half(hv)), pe);
                word |= (uint32_t)c << (8 * i);
            }
            *reinterpret_cast<uint32_t*>(out + (int64_t)part * kIH * kID) = word;
        }
        if (lane == 0) wp[(int64_t)t * kIH + h] = ldexpf(wsc[h], e);
    }
}

// ---------------------------------------------------------------------------
// scores on the 5th-generation tensor cores.
//
// Work: tiles of 128 keys of one sequence x one chunk of NQ <= 8 queries of
// that sequence (N = NQ*32 accumulator columns).  The tile space
// (sequence, chunk, tile) is cut into one contiguous range per CTA; CTAs are
// persistent (one per SM) and stream their range through a ring of shared-
// memory stages:
//   warp 0     TMA producer: key tiles (128-byte swizzled, K-major) and, at
//              each new (sequence, chunk), the chunk's q' (same layout);
//   warp 1     allocates TMEM and issues tcgen05.mma: M = 128 keys, N = NQ*32
//              heads, K = 192 (hi | lo | unrotated) or 128 (NoPE), fp32
//              accumulators double-buffered in TMEM;
//   warps 2-5  epilogue: one key row per thread straight from TMEM, relu and
//              head weights, causal mask, fp8 row scale, coalesced stores
//              (warps 2-9 for bf16 shapes of four or more queries at one CTA
//              per SM).
// e4m3 keys: the MMA runs kind::f8f6f4 on the staged codes themselves (K =
// 128 bytes, one 128-byte swizzled row per key) against q' split into three
// e4m3 parts (qprep_e4m3_kernel): N = NQ x 3 x 32 accumulator columns, which
// the epilogue recombines per head with exact power-of-two scalings.
// Keys past the context are never stored; pages are read through the page
// table one TMA box (R rows, R | page size) at a time.

// Per contracted tile, the producer hands the epilogue, through a ring of
// shared-memory slots, the physical row of each TMA box (-1: not loaded) and,
// for e4m3 keys, the 128 row scales, copied asynchronously (cp.async, tracked
// by the slot's barrier).  The epilogue then makes no global load per tile:
// under a saturated HBM a dependent load takes longer than a tile.
constexpr int kInfoSlots = 16;  // > stages + key operand buffers + accumulators: never the bottleneck
template <bool FP8>
struct TileInfo {
    static constexpr int bytes = 64 + (FP8 ? kTileKeys * 4 : 0);  // int64 box_base[8]; float scale[128]
};

template <int NQ, int KP, bool FP8>
struct IdxCfg {
    static constexpr int N = NQ * kIH;
    static_assert(!FP8 || NQ <= 2, "e4m3 keys take at most two queries per chunk (TMEM)");
    static constexpr int NM = FP8 ? kQParts * N : N;  // MMA N = accumulator columns per buffer
    static constexpr int KM = FP8 ? kID : KP;    // contraction length in elements
    // bf16: KP/64 blocks of N x 128 B; e4m3: NM rows of 128 B
    static constexpr int q_bytes = FP8 ? NM * kID : N * KP * 2;
    // bf16: two 128-byte swizzled 64-dim blocks; e4m3: the codes, one
    // 128-byte (swizzled) row per key
    static constexpr int stage_bytes = FP8 ? kTileKeys * kID : kTileKeys * kID * 2;
    static constexpr int info_bytes = kInfoSlots * TileInfo<FP8>::bytes;
    // epilogue warps: bf16 with several queries and one CTA per SM has warp
    // slots to spare, so two warps per TMEM lane quarter each reduce half of
    // the queries (the epilogue, not the MMA, bounds those shapes otherwise)
    static constexpr int ew_max = (!FP8 && NQ >= 4) ? 8 : 4;
    static constexpr int tail_raw =
        (2 * 8 + 6 + 2 * kInfoSlots) * 8 + 16 + ew_max * NQ * kIH * 4 + ew_max * NQ * 4;
    static constexpr int tail = (tail_raw + 1023) / 1024 * 1024;  // barriers, TMEM slot, per-warp weights
    // Decode shapes (small q') run two persistent CTAs per SM, so two
    // producer / MMA-issuer pairs overlap their per-tile issue work: when two
    // CTAs' stages and double-buffered accumulators fit.
    // (110 KB per CTA: two fit an SM's 228 KB; the full 113 KB gives the
    // paged bf16 shape a third stage, measured slower than two)
    static constexpr bool two_fit =
        (110 * 1024 - q_bytes - info_bytes - 1024 - tail) / stage_bytes >= 2 && 2 * NM <= 256;
    static constexpr int ctas_per_sm = two_fit ? 2 : 1;
    static constexpr int budget = (ctas_per_sm == 2 ? 110 : 220) * 1024;
    static constexpr int stages_fit = (budget - q_bytes - info_bytes - 1024 - tail) / stage_bytes;
    static constexpr int S = stages_fit > 8 ? 8 : stages_fit;
    static constexpr int EW = (ew_max == 8 && ctas_per_sm == 1) ? 8 : 4;
    static constexpr int QPW = NQ * 4 / EW;  // queries per epilogue warp
    static constexpr int threads = EW == 8 ? 320 : 192;
    // two accumulator buffers; tcgen05.alloc takes a power of two >= 32 columns
    static constexpr int tmem_cols = 2 * NM <= 32 ? 32 : 2 * NM <= 64 ? 64 : 2 * NM <= 128 ? 128 : 2 * NM <= 256 ? 256 : 512;
    static constexpr int nacc = 2;
    static constexpr size_t smem = 1024 + (size_t)S * stage_bytes + q_bytes + info_bytes + tail;  // + alignment slack
    static_assert(S >= 2, "too little shared memory for two stages");
    static_assert(2 * NM <= 512, "accumulators exceed TMEM");
    static_assert(ctas_per_sm * tmem_cols <= 512, "the CTAs of an SM must fit its TMEM together");
};

template <int NQ, int KP, bool FP8>
__global__ void __launch_bounds__(IdxCfg<NQ, KP, FP8>::threads, IdxCfg<NQ, KP, FP8>::ctas_per_sm)
    index_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                    const float* __restrict__ wp, const float* __restrict__ k_scale, dsa_seqs s,
                    float* __restrict__ scores, int64_t ld, float* __restrict__ gmax, int64_t ldg,
                    int tiles_per_seq, int chunks, int64_t total_tiles, int box_rows, int32_t* d_status) {
    pdl_enter();
    using C = IdxCfg<NQ, KP, FP8>;
    constexpr int S = C::S, N = C::N;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = base;
    uint8_t* qs = base + S * C::stage_bytes;  // 1024-aligned (stage bytes are multiples of 1024)
    uint8_t* info = qs + C::q_bytes;  // [kInfoSlots] TileInfo
    uint64_t* bars = reinterpret_cast<uint64_t*>(info + C::info_bytes);
    uint64_t* full = bars;               // [S] TMA landed
    uint64_t* empty = bars + S;          // [S] stage read by the MMA
    uint64_t* tfull = bars + 2 * S;      // [2] accumulator ready
    uint64_t* tempty = bars + 2 * S + 2; // [2] accumulator drained
    uint64_t* qfull = bars + 2 * S + 4;
    uint64_t* qempty = bars + 2 * S + 5;
    uint64_t* ifull = bars + 2 * S + 6;                // [kInfoSlots] tile info written (and scales landed)
    uint64_t* iempty = bars + 2 * S + 6 + kInfoSlots;  // [kInfoSlots] tile info read
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 6 + 2 * kInfoSlots);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);  // and the kernel tag at +1
    float* sw_all = reinterpret_cast<float*>(tmem_slot + 4);  // [EW][NQ*32] head weights, one copy per epilogue warp
    int* spos_all = reinterpret_cast<int*>(sw_all + C::EW * NQ * kIH);  // [EW][NQ] query positions

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int64_t t_begin, t_end;  // every warp computes the same range
    balanced_range<NQ>(s, chunks, tiles_per_seq, &t_begin, &t_end);
    (void)total_tiles;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            ptx::mbar_init(full + i, 1);
            ptx::mbar_init(empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(tfull + i, 1);
            ptx::mbar_init(tempty + i, C::EW);
        }
        for (int i = 0; i < kInfoSlots; ++i) {
            ptx::mbar_init(ifull + i, FP8 ? 33 : 1);  // lane 0, plus each lane's scale copies (e4m3)
            ptx::mbar_init(iempty + i, C::EW);
        }
        ptx::mbar_init(qfull, 1);
        ptx::mbar_init(qempty, 1);
        *abort_flag = 0;
        abort_flag[1] = kTagIndexer;  // names this kernel in a timeout's status
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, C::tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The whole warp walks the tiles; lanes fetch 32 page-table entries at
        // a time, lane 0 waits on the ring and issues the TMA copies.
        if (lane == 0) {
            ptx::prefetch_tmap(&kmap);
            ptx::prefetch_tmap(&qmap);
        }
        TileWalker<NQ> wk(t_begin, t_end, tiles_per_seq, chunks);
        int seg, j0, kind, q_seg = -1, qloads = 0;
        int64_t issued = 0;
        int win_b = -1, win_p0 = 0, win_entry = -1;
        const int ps_log2 = s.page_table ? __ffs(s.page_size) - 1 : 7;  // page size is a power of two
        const int ps_mask = (1 << ps_log2) - 1;
        const int nb = kTileKeys / box_rows;  // row blocks per tile (<= 8, so <= 16 boxes <= 32 lanes)
        while (wk.next(s, 2, d_status, false, seg, j0, kind)) {
            const IdxSeg& g = wk.g;
            bool ok = true;
            if (seg != q_seg) {
                if (lane == 0) {
                    ok = qloads == 0 || ptx::mbar_wait(qempty, (qloads - 1) & 1, abort_flag, d_status);
                    if (ok) {
                        ptx::mbar_expect_tx(qfull, C::q_bytes);
                        if (FP8)
                            ptx::tma_load_2d(qs, &qmap, 0, g.q0 * kQParts * kIH, qfull);
                        else
                            for (int kb = 0; kb < KP / 64; ++kb)
                                ptx::tma_load_2d(qs + kb * N * 128, &qmap, kb * 64, g.q0 * kIH, qfull);
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                q_seg = seg;
                ++qloads;
            }
            // One TMA box per lane: lane L takes row block L >> 1 (L for e4m3)
            // and, for bf16, K-half L & 1.  Blocks past the context or behind an
            // invalid page are not loaded (the epilogue masks and reports them);
            // rows of a block past the end of the cache read as zeros.
            const int jn = min(kTileKeys, g.ctx - j0);
            const int rb = FP8 ? lane : (lane >> 1), half = FP8 ? 0 : (lane & 1);
            const int j = j0 + rb * box_rows;
            int64_t row = -1;
            if (s.page_table) {
                const int p_first = j0 >> ps_log2, p_last = (j0 + jn - 1) >> ps_log2;
                if (g.b != win_b || p_first < win_p0 || p_last >= win_p0 + 32) {
                    win_b = g.b;
                    win_p0 = p_first;
                    const int p = win_p0 + lane;
                    win_entry = p < s.max_pages ? __ldg(s.page_table + (int64_t)g.b * s.max_pages + p) : -1;
                }
                const int entry = __shfl_sync(0xffffffffu, win_entry, ((j >> ps_log2) - win_p0) & 31);
                const int64_t r = ((int64_t)entry << ps_log2) + (j & ps_mask);
                if (rb < nb && rb * box_rows < jn && entry >= 0 && r < s.num_rows) row = r;
            } else {
                const int64_t r = g.base + j;
                if (rb < nb && rb * box_rows < jn && r >= 0 && r < s.num_rows) row = r;
            }
            const uint32_t loads = __ballot_sync(0xffffffffu, row >= 0);
            const int st = (int)(issued % S);
            const int is = (int)(issued % kInfoSlots);
            if (lane == 0) {
                const uint32_t use = (uint32_t)(issued / S);
                ok = issued < S || ptx::mbar_wait(empty + st, (use - 1) & 1, abort_flag, d_status);
                if (ok && issued >= kInfoSlots)
                    ok = ptx::mbar_wait(iempty + is, ((uint32_t)(issued / kInfoSlots) - 1) & 1, abort_flag, d_status);
                if (ok) ptx::mbar_expect_tx(full + st, (uint32_t)__popc(loads) * box_rows * 128);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (row >= 0) {
                uint8_t* dst = stages + st * C::stage_bytes + half * (kTileKeys * 128) + rb * box_rows * 128;
                ptx::tma_load_2d(dst, &kmap, half * 64, (int)row, full + st);
            }
            uint8_t* ti = info + is * TileInfo<FP8>::bytes;
            if (half == 0 && rb < 8) reinterpret_cast<int64_t*>(ti)[rb] = row;
            if (FP8) {
                float* sc = reinterpret_cast<float*>(ti + 64);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int r = lane + 32 * u;  // key row of the tile
                    const int64_t bb = __shfl_sync(0xffffffffu, row, r / box_rows);
                    const int64_t pr = bb + (r & (box_rows - 1));
                    if (bb >= 0 && pr < s.num_rows) ptx::cp_async4(sc + r, k_scale + pr);
                }
                ptx::cp_async_arrive_noinc(ifull + is);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ifull + is);
            ++issued;
        }
        // drain: every issued copy has landed and every MMA reading a stage is done
        if (lane == 0) {
            for (int64_t i = issued > S ? issued - S : 0; i < issued; ++i) {
                const int st = (int)(i % S);
                const uint32_t ph = (uint32_t)(i / S) & 1;
                if (!ptx::mbar_drain(empty + st, ph)) ptx::mbar_drain(full + st, ph);
            }
            if (qloads > 0) ptx::mbar_drain(qempty, (qloads - 1) & 1);
        }
        ptx::cp_async_wait_all();
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        // e4m3 x e4m3 (kind::f8f6f4) encodes like f16 x f16: both type fields 0
        constexpr uint32_t idesc = ptx::idesc_f16_m128(C::NM, !FP8);
        TileWalker<NQ> wk(t_begin, t_end, tiles_per_seq, chunks);
        int seg, j0, kind, nseg, nj0, nkind;
        bool have = wk.next(s, 2, d_status, false, seg, j0, kind);
        int q_seg = -1, qloads = 0;
        int64_t consumed = 0;
        int st = 0, a = 0;     // ring stage, accumulator
        uint32_t use = 0, au = 0;  // and how often each has come round
        while (have) {
            const bool have_next = wk.next(s, 2, d_status, false, nseg, nj0, nkind);
            if (seg != q_seg) {
                if (!ptx::mbar_wait(qfull, qloads & 1, abort_flag, d_status)) break;
                ++qloads;
                q_seg = seg;
            }
            if (!ptx::mbar_wait(full + st, use & 1, abort_flag, d_status)) break;
            if (consumed >= C::nacc && !ptx::mbar_wait(tempty + a, (au - 1) & 1, abort_flag, d_status)) break;
            ptx::tc_fence_after();
            const uint32_t kbase = smem_u32(stages + st * C::stage_bytes);
            const uint32_t qbase = smem_u32(qs);
            if (FP8) {
                // 4 k-steps of 32 codes (32 bytes) within the 128-byte rows
#pragma unroll
                for (int ks = 0; ks < C::KM / 32; ++ks)
                    ptx::mma_ss_f8(tmem_base + a * C::NM, ptx::sdesc_sw128(kbase + ks * 32),
                                   ptx::sdesc_sw128(qbase + ks * 32), idesc, ks > 0 ? 1u : 0u);
            } else {
#pragma unroll
                for (int ks = 0; ks < KP / 16; ++ks) {
                    int kd;  // key dim of this k-step: [hi | lo | unrotated] read dims 0..63, 0..63, 64..127
                    if (KP == 192) kd = ks < 4 ? ks * 16 : (ks < 8 ? (ks - 4) * 16 : 64 + (ks - 8) * 16);
                    else kd = ks * 16;
                    const uint64_t bd =
                        ptx::sdesc_sw128(qbase + ((ks * 16) >> 6) * (N * 128) + ((ks * 16) & 63) * 2);
                    const uint64_t ad = ptx::sdesc_sw128(kbase + (kd >> 6) * (kTileKeys * 128) + (kd & 63) * 2);
                    ptx::mma_ss(tmem_base + a * N, ad, bd, idesc, ks > 0 ? 1u : 0u);
                }
            }
            ptx::mma_commit(empty + st);
            ptx::mma_commit(tfull + a);
            if (++st == S) { st = 0; ++use; }
            if (++a == C::nacc) { a = 0; ++au; }
            if (!have_next || nseg != seg) ptx::mma_commit(qempty);
            ++consumed;
            have = have_next;
            seg = nseg;
            j0 = nj0;
            kind = nkind;
        }
    } else if (warp >= 2 && warp < 2 + C::EW) {
        // ------------------------------------------------------------ epilogue
        // each epilogue warp keeps its own copy of the chunk's weights and
        // positions, so the warps never wait on each other; with eight, the
        // second four take the upper half of the queries
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int q_lo = ((warp - 2) >> 2) * C::QPW;
        float* sw = sw_all + (warp - 2) * NQ * kIH;
        int* spos = spos_all + (warp - 2) * NQ;
        TileWalker<NQ> wk(t_begin, t_end, tiles_per_seq, chunks);
        int seg, j0, kind, cur = -1;
        int64_t consumed = 0;
        while (wk.next(s, 1, d_status, true, seg, j0, kind)) {
            const IdxSeg& g = wk.g;
            if (seg != cur) {
                __syncwarp();
                for (int e = lane; e < NQ * kIH; e += 32)
                    sw[e] = (e / kIH) < g.nq ? __ldg(wp + (int64_t)g.q0 * kIH + e) : 0.f;
                if (lane < NQ) {
                    int p = lane < g.nq ? __ldg(s.q_pos + g.q0 + lane) : -1;
                    if (lane < g.nq && (p < 0 || p >= g.ctx)) {
                        report(d_status, DSA_ERR_BAD_INPUT);
                        p = -1;
                    }
                    spos[lane] = p;
                }
                __syncwarp();
                cur = seg;
            }
            const int j = j0 + row;
            const bool in_ctx = j < g.ctx;
            // this warp's 32 keys are group grp of the row (gmax: their maximum)
            const int grp = (j0 >> 5) + quarter;
            const bool grp_live = j0 + quarter * 32 < g.ctx;
            if (kind == 1) {
                for (int q = q_lo; q < min(g.nq, q_lo + C::QPW); ++q) {
                    if (scores && in_ctx) scores[(int64_t)(g.q0 + q) * ld + j] = -INFINITY;
                    if (gmax && lane == 0 && grp_live) gmax[(int64_t)(g.q0 + q) * ldg + grp] = -INFINITY;
                }
                continue;
            }
            // this row's physical location and scale, from the producer
            const int is = (int)(consumed % kInfoSlots);
            if (!__all_sync(0xffffffffu,
                            ptx::mbar_wait(ifull + is, (uint32_t)(consumed / kInfoSlots) & 1, abort_flag, d_status)))
                break;
            const uint8_t* ti = info + is * TileInfo<FP8>::bytes;
            const int64_t bb = reinterpret_cast<const int64_t*>(ti)[row / box_rows];
            int64_t prow = bb >= 0 ? bb + (row & (box_rows - 1)) : -1;
            if (prow >= s.num_rows) prow = -1;
            float sigma = FP8 ? reinterpret_cast<const float*>(ti + 64)[row] : 1.f;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(iempty + is);
            if (in_ctx && prow < 0) report(d_status, DSA_ERR_BAD_INPUT);
            if (FP8 && prow >= 0 && sigma < 0.f) {
                report(d_status, DSA_ERR_BAD_INPUT);
                sigma = 0.f;
            }
            const int a = (int)(consumed % C::nacc);
            const uint32_t au = (uint32_t)(consumed / C::nacc);
            // warp-uniform outcome: a lane that sees an abort takes the whole warp out
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(tfull + a, au & 1, abort_flag, d_status))) break;
            ptx::tc_fence_after();
            const uint32_t tcol = tmem_base + ((uint32_t)(quarter * 32) << 16) + a * C::NM;
            // relu-weighted sum over the 32 heads of query q (four partial
            // sums, so the FMA chain is 8 deep rather than 32)
            auto relu_sum = [&](const uint32_t (&v)[32], int q) -> float {
                const float4* w4 = reinterpret_cast<const float4*>(sw + q * kIH);
                float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
#pragma unroll
                for (int h = 0; h < 32; h += 4) {
                    const float4 w = w4[h >> 2];
                    r0 = fmaf(w.x, fmaxf(__uint_as_float(v[h]), 0.f), r0);
                    r1 = fmaf(w.y, fmaxf(__uint_as_float(v[h + 1]), 0.f), r1);
                    r2 = fmaf(w.z, fmaxf(__uint_as_float(v[h + 2]), 0.f), r2);
                    r3 = fmaf(w.w, fmaxf(__uint_as_float(v[h + 3]), 0.f), r3);
                }
                return (r0 + r1) + (r2 + r3);
            };
            auto reduce = [&](int q) -> float {
                if (FP8) {
                    // head h of query q: parts at columns q 96 + p 32 + h,
                    // q'.k / s = D0 + 2^-4 (D1 + 2^-4 D2), exact scalings
                    const float4* w4 = reinterpret_cast<const float4*>(sw + q * kIH);
                    float r0 = 0.f, r1 = 0.f;
#pragma unroll 1
                    for (int h0 = 0; h0 < 32; h0 += 16) {
                        float d[kQParts][16];
#pragma unroll
                        for (int p = 0; p < kQParts; ++p) ptx::tmem_ld16(tcol + (q * kQParts + p) * kIH + h0, d[p]);
#pragma unroll
                        for (int h = 0; h < 16; h += 4) {
                            const float4 w = w4[(h0 + h) >> 2];
                            const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                float x = fmaf(d[2][h + u], 0.0625f, d[1][h + u]);
                                x = fmaf(x, 0.0625f, d[0][h + u]);
                                if (u & 1) r1 = fmaf(wv[u], fmaxf(x, 0.f), r1);
                                else r0 = fmaf(wv[u], fmaxf(x, 0.f), r0);
                            }
                        }
                    }
                    return r0 + r1;
                }
                uint32_t v[32];
                ptx::tmem_ld32_async(tcol + q * 32, v);
                ptx::tmem_wait_ld32(v);
                return relu_sum(v, q);
            };
            // the row's score (-inf past the query's position); with gmax, the
            // maximum of the warp's 32 keys too (called by the whole warp)
            auto store = [&](int q, float r) {
                if (q >= g.nq) return;
                const float v = (in_ctx && prow >= 0 && j <= spos[q]) ? r * sigma : -INFINITY;
                if (scores && in_ctx) scores[(int64_t)(g.q0 + q) * ld + j] = v;
                if (gmax) {
                    const float m = ptx::warp_max(v);
                    if (lane == 0 && grp_live) gmax[(int64_t)(g.q0 + q) * ldg + grp] = m;
                }
            };
            auto release = [&] {
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(tempty + a);
            };
            // One or two queries: the accumulator goes back to the MMA before
            // the stores.
            if constexpr (FP8 && NQ == 1) {
                // all 96 columns (3 parts x 32 heads) into registers, then the
                // release: the recombination and head sum run off the MMA's path
                uint32_t d[kQParts][32];
#pragma unroll
                for (int p = 0; p < kQParts; ++p) ptx::tmem_ld32_async(tcol + p * kIH, d[p]);
#pragma unroll
                for (int p = 0; p < kQParts; ++p) ptx::tmem_wait_ld32(d[p]);
                release();
                const float4* w4 = reinterpret_cast<const float4*>(sw);
                float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
#pragma unroll
                for (int h = 0; h < 32; h += 4) {
                    const float4 w = w4[h >> 2];
                    const float wv[4] = {w.x, w.y, w.z, w.w};
                    float x[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        // q'.k / s = D0 + 2^-4 (D1 + 2^-4 D2), exact scalings
                        const float v = fmaf(__uint_as_float(d[2][h + u]), 0.0625f, __uint_as_float(d[1][h + u]));
                        x[u] = fmaxf(fmaf(v, 0.0625f, __uint_as_float(d[0][h + u])), 0.f);
                    }
                    r0 = fmaf(wv[0], x[0], r0);
                    r1 = fmaf(wv[1], x[1], r1);
                    r2 = fmaf(wv[2], x[2], r2);
                    r3 = fmaf(wv[3], x[3], r3);
                }
                store(0, (r0 + r1) + (r2 + r3));
            } else if constexpr (NQ <= 2) {
                float acc[NQ];
#pragma unroll
                for (int q = 0; q < NQ; ++q) acc[q] = reduce(q);
                release();
#pragma unroll
                for (int q = 0; q < NQ; ++q) store(q, acc[q]);
            } else {
                // this warp's queries; the next one's columns load while this
                // one's are summed
                uint32_t v[2][32];
                ptx::tmem_ld32_async(tcol + q_lo * 32, v[0]);
                ptx::tmem_wait_ld32(v[0]);
#pragma unroll
                for (int i = 0; i < C::QPW; ++i) {
                    if (i + 1 < C::QPW) ptx::tmem_ld32_async(tcol + (q_lo + i + 1) * 32, v[(i + 1) & 1]);
                    const float r = relu_sum(v[i & 1], q_lo + i);
                    if (i + 1 < C::QPW) ptx::tmem_wait_ld32(v[(i + 1) & 1]);
                    store(q_lo + i, r);
                }
                release();
            }
            ++consumed;
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::tmem_cols);
    }
}

// ---------------------------------------------------------------------------
// host side
namespace {

template <int NQ, int KP, bool FP8>
cudaError_t launch_tc(const void* qp, int num_q, const float* wp, const void* k_idx, const float* k_scale,
                      const dsa_seqs& s, float* scores, int64_t ld, float* gmax, int64_t ldg, int32_t* d_status,
                      cudaStream_t stream) {
    using C = IdxCfg<NQ, KP, FP8>;
    const int box_rows = s.page_table ? std::min(64, s.page_size & -s.page_size) : kTileKeys;
    CUtensorMap kmap, qmap;
    cudaError_t e;
    if (FP8)
        e = make_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, k_idx, kID, (uint64_t)s.num_rows, kID, kID, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
    else
        e = make_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k_idx, kID, (uint64_t)s.num_rows, kID * 2, 64,
                     box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    if (FP8)  // [Q x 3 parts x 32 heads] rows of 128 codes; one box = a chunk's NM rows
        e = make_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, qp, kID, (uint64_t)num_q * kQParts * kIH, kID, kID, C::NM,
                     CU_TENSOR_MAP_SWIZZLE_128B);
    else
        e = make_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, qp, KP, (uint64_t)num_q * kIH, KP * 2, 64, C::N,
                     CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    auto kern = index_tc_kernel<NQ, KP, FP8>;
    static std::once_flag once;  // one per instantiation
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [kern] {
        attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::smem);
    });
    if (attr != cudaSuccess) return attr;
    const int tiles_per_seq = (s.max_ctx + kTileKeys - 1) / kTileKeys;
    const int chunks = (s.max_q_per_seq + NQ - 1) / NQ;
    const int64_t total = (int64_t)s.num_seqs * chunks * tiles_per_seq;
    const int grid = (int)std::min<int64_t>((int64_t)C::ctas_per_sm * num_sms(), total);
    return launch_pdl(kern, dim3(grid), dim3(C::threads), C::smem, stream, 1, kmap, qmap, wp, k_scale, s, scores, ld,
                      gmax, ldg, tiles_per_seq, chunks, total, box_rows, d_status);
}

template <int NQ>
cudaError_t launch_tc_nq(bool rope, bool fp8, const void* qp, int num_q, const float* wp, const void* k_idx,
                         const float* k_scale, const dsa_seqs& s, float* scores, int64_t ld, float* gmax, int64_t ldg,
                         int32_t* d_status, cudaStream_t stream) {
    if (fp8) {  // q' parts hold the rotated (or unrotated) 128 dims either way
        if constexpr (NQ <= 2)
            return launch_tc<NQ, 128, true>(qp, num_q, wp, k_idx, k_scale, s, scores, ld, gmax, ldg, d_status, stream);
        else
            return cudaErrorInvalidValue;
    }
    return rope ? launch_tc<NQ, 192, false>(qp, num_q, wp, k_idx, k_scale, s, scores, ld, gmax, ldg, d_status, stream)
                : launch_tc<NQ, 128, false>(qp, num_q, wp, k_idx, k_scale, s, scores, ld, gmax, ldg, d_status, stream);
}

}  // namespace

cudaError_t launch_index_scores(const void* q_idx, const float* w, const float* ssmax_s, const float* ssmax_b,
                                const float* inv_freq, const void* k_idx, const float* k_scale, dsa_dtype k_dtype,
                                const dsa_seqs& s, int num_q, float* scores, int64_t ld, float* gmax, int64_t ldg,
                                const Workspace& ws, int32_t* d_status, cudaStream_t stream,
                                const void* k_block_scales, float k_global) {
    if (k_dtype == DSA_NVFP4)
        return launch_index_scores_nvfp4(q_idx, w, ssmax_s, ssmax_b, inv_freq, k_idx, k_block_scales, k_global, s,
                                         num_q, scores, ld, gmax, ldg, ws, d_status, stream);
    const bool fp8 = k_dtype == DSA_FP8_E4M3_ROWSCALE;
    const bool rope = inv_freq != nullptr;
    const __nv_bfloat16* qi = reinterpret_cast<const __nv_bfloat16*>(q_idx);
    cudaError_t e =
        fp8 ? launch_pdl(qprep_e4m3_kernel, dim3(num_q), dim3(kIH * 32), 0, stream, 1, qi, w, ssmax_s, ssmax_b, inv_freq, s,
                         num_q, reinterpret_cast<uint8_t*>(ws.qprep), ws.wprep, d_status)
            : launch_pdl(qprep_kernel<__nv_bfloat16>, dim3(num_q), dim3(kIH * 16), 0, stream, 1, qi, w, ssmax_s, ssmax_b,
                         inv_freq, s, num_q, reinterpret_cast<__nv_bfloat16*>(ws.qprep), ws.wprep, d_status);
    if (e != cudaSuccess) return e;
    const int mq = s.max_q_per_seq;
    if (fp8)  // e4m3 keys: chunks of at most two queries (four parts each fill the TMEM)
        return mq <= 1 ? launch_tc_nq<1>(rope, fp8, ws.qprep, num_q, ws.wprep, k_idx, k_scale, s, scores, ld, gmax, ldg, d_status,
                                         stream)
                       : launch_tc_nq<2>(rope, fp8, ws.qprep, num_q, ws.wprep, k_idx, k_scale, s, scores, ld, gmax, ldg, d_status,
                                         stream);
    if (mq <= 1) return launch_tc_nq<1>(rope, fp8, ws.qprep, num_q, ws.wprep, k_idx, k_scale, s, scores, ld, gmax, ldg, d_status, stream);
    if (mq <= 2) return launch_tc_nq<2>(rope, fp8, ws.qprep, num_q, ws.wprep, k_idx, k_scale, s, scores, ld, gmax, ldg, d_status, stream);
    if (mq <= 4) return launch_tc_nq<4>(rope, fp8, ws.qprep, num_q, ws.wprep, k_idx, k_scale, s, scores, ld, gmax, ldg, d_status, stream);
    return launch_tc_nq<8>(rope, fp8, ws.qprep, num_q, ws.wprep, k_idx, k_scale, s, scores, ld, gmax, ldg, d_status, stream);
}

}  // namespace dsa
