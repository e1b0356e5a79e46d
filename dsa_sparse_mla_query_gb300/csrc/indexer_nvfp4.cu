// indexer_nvfp4.cu -- lightning-indexer scores over NVFP4 index keys (sm_103a).
//
// Key format ("vLLM adds NVFP4 serving for MiniMax M3.1 Flash": NVFP4
// indexer caches at 4.5 bits per value): per cached row 64 code bytes (128
// E2M1 values, value 2i in the low nibble of byte i), 8 E4M3 block scales
// (one per 16 values) and one fp32 tensor scale g for the whole cache;
// k = g * scale * code.  The scores are those of the bf16 path (indexer.cu):
//   score(t, j) = sum_h w'_h relu(q'_h . k_j),  w'_h = w_h |f_h| / 64.
//
// Conversion inside the kernel.  An E2M1 value times an E4M3 scale has at
// most 6 significant bits and lies in [2^-10, 2688], so it is exact in f16:
// the key tile is decoded to f16 with no rounding at all, and g (> 0) folds
// into the head weight.  The decoded tile goes straight into tensor memory,
// where tcgen05.mma reads it as its A operand (kind::f16, A from TMEM), so
// the decode costs no shared-memory round trip and the MMA reads no key bytes
// from shared memory.  The query is split into f16 hi + lo parts like the bf16
// path's q' (K = 192 on RoPE layers, 128 on NoPE layers), after a per-head
// power-of-two scaling that keeps it clear of f16's range limits; that power
// of two folds into the head weight as well.
//
// Work split and roles (one CTA per SM for four-query chunks, two otherwise):
//   warp 0     TMA producer: code tiles (128 keys x 64 bytes, 64-byte
//              swizzle), the rows' block scales beside them (a map of 8-byte
//              elements, one per row: each box starts at the even row at or
//              below its first row, 16-byte aligned, and takes two more), and the
//              chunk's q' at each new (sequence, chunk);
//   warp 1     allocates TMEM and issues the MMAs: M = 128 keys from TMEM,
//              N = NQ x 32 heads, fp32 accumulators double-buffered;
//   warps 2-5  epilogue (as the bf16 path's): relu, head weights, mask, stores;
//   warps 6-9  decoders: one key row per thread, codes and scales from shared
//              memory, E2M1 -> f16 times the block scale, tcgen05.st into one
//              of two A buffers in TMEM.
#include <cuda_fp4.h>

#include "indexer_common.cuh"

namespace dsa {

// ---------------------------------------------------------------------------
// query preparation, f16, scaled per head by 2^-e so that max |q'| lies in
// [2^14, 2^15); w'' = w |f| g 2^e / 64.  The rotated dims keep ~2^-22 of their
// value through an f16 hi + lo pair; the unrotated dims are bf16 values times
// a power of two, exact in f16 down to 2^-29 of the head's largest value.
// Layouts:
//   split_n = 0: q' [Q, 32, KP] as the bf16 path's ([hi(0..63) | lo(0..63) |
//                dims 64..127] on RoPE layers, dims 0..127 on NoPE layers):
//                the lo part extends K (K = 192);
//   split_n = 1: q' [Q, 64, 128], rows 0..31 the heads' hi parts over all 128
//                dims, rows 32..63 their lo parts (zero on dims 64..127): the
//                lo part extends N instead (RoPE layers, one query per chunk).
__global__ void __launch_bounds__(kIH * 32) qprep_f16_kernel(const __nv_bfloat16* __restrict__ q,
                                                        const float* __restrict__ w, const float* __restrict__ ss,
                                                        const float* __restrict__ sb,
                                                        const float* __restrict__ inv_freq, dsa_seqs s, int num_q,
                                                        float g, int split_n, __half* __restrict__ qp,
                                                        float* __restrict__ wp, int32_t* d_status) {
    pdl_enter();
    const int t = blockIdx.x;
    const bool rope = inv_freq != nullptr;
    const int KP = rope ? 192 : 128;
    __shared__ float cs[32], sn[32], sgn[32], wsc[32];
    __shared__ int ok;
    // warp h: head h; lane: dims 4 lane .. 4 lane + 3 (rotation pairs 2 lane,
    // 2 lane + 1; the load in flight during the per-query setup)
    const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint2 raw = *reinterpret_cast<const uint2*>(q + ((int64_t)t * kIH + h) * kID + 4 * lane);
    qprep_setup(w, ss, sb, inv_freq, s, t, cs, sn, sgn, wsc, &ok, d_status);
    {
        const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&raw);
        const float sg = ok ? sgn[h] : 0.f;
        const bool rot = rope && lane < 16;
        float y[4];
        if (rot) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int p = 2 * lane + u;
                const float x0 = __bfloat162float(x[2 * u]), x1 = __bfloat162float(x[2 * u + 1]);
                y[2 * u] = sg * fmaf(x0, cs[p], -x1 * sn[p]);
                y[2 * u + 1] = sg * fmaf(x0, sn[p], x1 * cs[p]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) y[i] = sg * __bfloat162float(x[i]);
        }
        float m = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        int e = 0;
        if (m > 0.f) {
            int E;
            frexpf(m, &E);  // m < 2^E
            e = E - 15;
        }
        alignas(8) __half hi[4];
        alignas(8) __half lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float v = ldexpf(y[i], -e);
            hi[i] = __float2half_rn(v);
            lo[i] = __float2half_rn(v - __half2float(hi[i]));
        }
        if (split_n) {
            __half* o = qp + ((int64_t)t * 2 * kIH + h) * kID + 4 * lane;
            *reinterpret_cast<uint2*>(o) = *reinterpret_cast<const uint2*>(hi);
            *reinterpret_cast<uint2*>(o + kIH * kID) = rot ? *reinterpret_cast<const uint2*>(lo) : make_uint2(0, 0);
            if (lane == 0) wp[(int64_t)t * kIH + h] = ldexpf(wsc[h] * g, e);
            return;
        }
        __half* o = qp + ((int64_t)t * kIH + h) * KP;
        if (rot) {
            *reinterpret_cast<uint2*>(o + 4 * lane) = *reinterpret_cast<const uint2*>(hi);
            *reinterpret_cast<uint2*>(o + 64 + 4 * lane) = *reinterpret_cast<const uint2*>(lo);
        } else {
            *reinterpret_cast<uint2*>(o + (rope ? 64 : 0) + 4 * lane) = *reinterpret_cast<const uint2*>(hi);
        }
        if (lane == 0) wp[(int64_t)t * kIH + h] = ldexpf(wsc[h] * g, e);
    }
}

// ---------------------------------------------------------------------------
// E2M1 codes x E4M3 block scale -> f16, exact.  A 32-bit word holds 8 codes
// (value 2i in the low nibble of byte i); its four bytes are unpacked into
// byte registers and each converted as is (cvt.rn.f16x2.e2m1x2, low nibble to
// the low half), so no shift or mask per pair; s2 = the block scale in both
// halves.
__device__ __forceinline__ void nv4_word(uint32_t w, __half2 s2, uint32_t* out) {
    uint32_t o[4];
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&o[i]), s2);
        out[i] = *reinterpret_cast<const uint32_t*>(&v);
    }
}

// Decodes 16 code bytes (32 values of two blocks, scales s01 = the blocks'
// two E4M3 scale codes) into 16 f16x2 words.
__device__ __forceinline__ void nv4_chunk(const uint4& c, uint32_t s01, uint32_t* out) {
    const __half2_raw sr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(s01 & 0xFFFFu), __NV_E4M3);
    __half2 sp;
    reinterpret_cast<__half2_raw&>(sp) = sr;
    const __half2 s0 = __low2half2(sp), s1 = __high2half2(sp);
    nv4_word(c.x, s0, out);
    nv4_word(c.y, s0, out + 4);
    nv4_word(c.z, s1, out + 8);
    nv4_word(c.w, s1, out + 12);
}

constexpr int kNvCodeBytes = kID / 2;   // 64 code bytes per key
constexpr int kNvScaleBytes = kID / 16; // 8 E4M3 block scales per key
constexpr int kNvInfoSlots = 16;        // box bases handed to the epilogue (> stages in flight)

// MMA cost on GB300 is close to a fixed ~50 cycles per M = 128 x K = 16
// instruction for N up to 64, so a RoPE chunk of one query (N = 32) takes its
// lo part in N (N = 64, K = 128: 8 instructions per tile) rather than in K
// (N = 32, K = 192: 12); wider chunks keep it in K, where N is already large.
template <int NQ, int KP>
struct Nv4Cfg {
    static constexpr int N = NQ * kIH;                  // heads of the chunk (score columns)
    static constexpr bool split_n = NQ == 1 && KP == 192;
    static constexpr int NM = split_n ? 2 * N : N;      // MMA N: accumulator columns per buffer
    static constexpr int KM = split_n ? kID : KP;       // MMA K
    static constexpr int q_bytes = NM * KM * 2;
    // codes (64-byte swizzled rows) then the boxes' block scales, one slot of
    // round_up((box rows + 2) x 8, 128) bytes per box: at most 2 KB
    static constexpr int codes_bytes = kTileKeys * kNvCodeBytes;
    static constexpr int scale_region = 2048;
    static constexpr int stage_bytes = codes_bytes + scale_region;  // 10 KB, 1024-aligned
    static constexpr int info_bytes = kNvInfoSlots * 64;                         // int64 box_base[8]
    static constexpr int a_cols = kID / 2;  // one decoded tile: 128 lanes x 64 columns
    static constexpr int tmem_need = 2 * NM + 2 * a_cols;
    static constexpr int tmem_cols = tmem_need <= 256 ? 256 : 512;
    static constexpr int ctas_per_sm = tmem_cols <= 256 ? 2 : 1;
    // barriers, TMEM slot and flag, weights, positions, box parities [8][8]
    static constexpr int tail_raw = (2 * 8 + 4 + 4 + 2 + 2 * kNvInfoSlots) * 8 + 16 + 4 * N * 4 + 4 * NQ * 4 + 64;
    static constexpr int tail = (tail_raw + 1023) / 1024 * 1024;
    static constexpr int budget = (ctas_per_sm == 2 ? 110 : 220) * 1024;
    static constexpr int stages_fit = (budget - q_bytes - info_bytes - 1024 - tail) / stage_bytes;
    static constexpr int S = stages_fit > 8 ? 8 : stages_fit;
    static constexpr int threads = 320;
    static constexpr size_t smem = 1024 + (size_t)S * stage_bytes + q_bytes + info_bytes + tail;
    static_assert(stage_bytes % 1024 == 0, "stages must stay 1024-byte aligned");
    static_assert(S >= 2, "too little shared memory for two stages");
    static_assert(tmem_need <= 512, "accumulators and A buffers exceed TMEM");
};

template <int NQ, int KP>
__global__ void __launch_bounds__(320, Nv4Cfg<NQ, KP>::ctas_per_sm)
    index_nv4_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap smap, const float* __restrict__ wp, dsa_seqs s,
                     float* __restrict__ scores, int64_t ld, float* __restrict__ gmax, int64_t ldg,
                     int tiles_per_seq, int chunks, int64_t total_tiles, int box_rows, int32_t* d_status) {
    pdl_enter();
    using C = Nv4Cfg<NQ, KP>;
    constexpr int S = C::S, N = C::N, NM = C::NM, KM = C::KM;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = base;
    uint8_t* qs = base + S * C::stage_bytes;
    uint8_t* info = qs + C::q_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(info + C::info_bytes);
    uint64_t* full = bars;               // [S] codes landed (TMA) and scales copied (cp.async)
    uint64_t* empty = bars + S;          // [S] stage read by the decoders
    uint64_t* afull = bars + 2 * S;      // [2] decoded tile in TMEM
    uint64_t* aempty = bars + 2 * S + 2; // [2] decoded tile read by the MMA
    uint64_t* tfull = bars + 2 * S + 4;  // [2] accumulator ready
    uint64_t* tempty = bars + 2 * S + 6; // [2] accumulator drained
    uint64_t* qfull = bars + 2 * S + 8;
    uint64_t* qempty = bars + 2 * S + 9;
    uint64_t* ifull = bars + 2 * S + 10;                  // [kNvInfoSlots]
    uint64_t* iempty = bars + 2 * S + 10 + kNvInfoSlots;  // [kNvInfoSlots]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 10 + 2 * kNvInfoSlots);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* sw_all = reinterpret_cast<float*>(tmem_slot + 4);  // [4][N] head weights, one copy per epilogue warp
    int* spos_all = reinterpret_cast<int*>(sw_all + 4 * N);   // [4][NQ] query positions
    uint8_t* bpar = reinterpret_cast<uint8_t*>(spos_all + 4 * NQ);  // [S][8] first row & 1 of each scale box

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int64_t t_begin, t_end;  // every warp computes the same range
    balanced_range<NQ>(s, chunks, tiles_per_seq, &t_begin, &t_end);
    (void)total_tiles;
    const int sc_slot = ((box_rows + 2) * kNvScaleBytes + 127) & ~127;  // bytes per box of scales

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            ptx::mbar_init(full + i, 1);  // lane 0's expect_tx
            ptx::mbar_init(empty + i, 4);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(afull + i, 4);
            ptx::mbar_init(aempty + i, 1);
            ptx::mbar_init(tfull + i, 1);
            ptx::mbar_init(tempty + i, 4);
        }
        for (int i = 0; i < kNvInfoSlots; ++i) {
            ptx::mbar_init(ifull + i, 1);
            ptx::mbar_init(iempty + i, 4);
        }
        ptx::mbar_init(qfull, 1);
        ptx::mbar_init(qempty, 1);
        *abort_flag = 0;
        abort_flag[1] = kTagIndexerNvfp4;
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
    const uint32_t acol0 = 2 * NM;  // A buffers after the two accumulators

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            ptx::prefetch_tmap(&kmap);
            ptx::prefetch_tmap(&qmap);
            ptx::prefetch_tmap(&smap);
        }
        TileWalker<NQ> wk(t_begin, t_end, tiles_per_seq, chunks);
        int seg, j0, kind, q_seg = -1, qloads = 0;
        int64_t issued = 0;
        int win_b = -1, win_p0 = 0, win_entry = -1;
        const int ps_log2 = s.page_table ? __ffs(s.page_size) - 1 : 7;
        const int ps_mask = (1 << ps_log2) - 1;
        const int nb = kTileKeys / box_rows;  // row blocks per tile (<= 8)
        while (wk.next(s, 2, d_status, false, seg, j0, kind)) {
            const IdxSeg& g = wk.g;
            bool ok = true;
            if (seg != q_seg) {
                if (lane == 0) {
                    ok = qloads == 0 || ptx::mbar_wait(qempty, (qloads - 1) & 1, abort_flag, d_status);
                    if (ok) {
                        ptx::mbar_expect_tx(qfull, C::q_bytes);
                        for (int kb = 0; kb < KM / 64; ++kb)
                            ptx::tma_load_2d(qs + kb * NM * 128, &qmap, kb * 64, g.q0 * (NM / NQ), qfull);
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                q_seg = seg;
                ++qloads;
            }
            // lane L < nb: TMA box of row block L (box_rows rows of 64 code bytes)
            const int jn = min(kTileKeys, g.ctx - j0);
            const int rb = lane, j = j0 + rb * box_rows;
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
            const int is = (int)(issued % kNvInfoSlots);
            if (lane == 0) {
                const uint32_t use = (uint32_t)(issued / S);
                ok = issued < S || ptx::mbar_wait(empty + st, (use - 1) & 1, abort_flag, d_status);
                if (ok && issued >= kNvInfoSlots)
                    ok = ptx::mbar_wait(iempty + is, ((uint32_t)(issued / kNvInfoSlots) - 1) & 1, abort_flag,
                                        d_status);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            // the stage is free: the boxes' parities, then (ordered by the warp
            // barrier and lane 0's arrival) the copies
            if (row >= 0) bpar[st * 8 + rb] = (uint8_t)(row & 1);
            __syncwarp();
            if (lane == 0)
                ptx::mbar_expect_tx(full + st, (uint32_t)__popc(loads) *
                                                   (box_rows * kNvCodeBytes + (box_rows + 2) * kNvScaleBytes));
            __syncwarp();
            uint8_t* stg = stages + st * C::stage_bytes;
            if (row >= 0) {
                ptx::tma_load_2d(stg + rb * box_rows * kNvCodeBytes, &kmap, 0, (int)row, full + st);
                ptx::tma_load_2d(stg + C::codes_bytes + rb * sc_slot, &smap, (int)(row & ~int64_t(1)), 0, full + st);
            }
            int64_t* ti = reinterpret_cast<int64_t*>(info + is * 64);
            if (rb < 8) ti[rb] = row;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ifull + is);
            ++issued;
        }
        if (lane == 0) {
            for (int64_t i = issued > S ? issued - S : 0; i < issued; ++i) {
                const int st = (int)(i % S);
                const uint32_t ph = (uint32_t)(i / S) & 1;
                if (!ptx::mbar_drain(empty + st, ph)) ptx::mbar_drain(full + st, ph);
            }
            if (qloads > 0) ptx::mbar_drain(qempty, (qloads - 1) & 1);
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = ptx::idesc_f16_m128(NM, false);  // f16 x f16
        TileWalker<NQ> wk(t_begin, t_end, tiles_per_seq, chunks);
        int seg, j0, kind, nseg, nj0, nkind;
        bool have = wk.next(s, 2, d_status, false, seg, j0, kind);
        int q_seg = -1, qloads = 0;
        int64_t c = 0;
        while (have) {
            const bool have_next = wk.next(s, 2, d_status, false, nseg, nj0, nkind);
            if (seg != q_seg) {
                if (!ptx::mbar_wait(qfull, qloads & 1, abort_flag, d_status)) break;
                ++qloads;
                q_seg = seg;
            }
            const int b = (int)(c & 1);
            const uint32_t bu = (uint32_t)(c >> 1);
            if (!ptx::mbar_wait(afull + b, bu & 1, abort_flag, d_status)) break;
            if (c >= 2 && !ptx::mbar_wait(tempty + b, (bu - 1) & 1, abort_flag, d_status)) break;
            ptx::tc_fence_after();
            const uint32_t qbase = smem_u32(qs);
            const uint32_t abuf = tmem_base + acol0 + b * C::a_cols;
#pragma unroll
            for (int ks = 0; ks < KM / 16; ++ks) {
                int kd;  // key dim of this k-step: [hi | lo | unrotated] read dims 0..63, 0..63, 64..127
                if (KM == 192) kd = ks < 4 ? ks * 16 : (ks < 8 ? (ks - 4) * 16 : 64 + (ks - 8) * 16);
                else kd = ks * 16;
                const uint64_t bd = ptx::sdesc_sw128(qbase + ((ks * 16) >> 6) * (NM * 128) + ((ks * 16) & 63) * 2);
                ptx::mma_ts(tmem_base + b * NM, abuf + kd / 2, bd, idesc, ks > 0 ? 1u : 0u);
            }
            ptx::mma_commit(aempty + b);
            ptx::mma_commit(tfull + b);
            if (!have_next || nseg != seg) ptx::mma_commit(qempty);
            ++c;
            have = have_next;
            seg = nseg;
            j0 = nj0;
            kind = nkind;
        }
    } else if (warp >= 6) {
        // ------------------------------------------------------------ decoders
        // TMEM lanes of this warp's quarter: key rows quarter*32 .. +31
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const int swz = (row >> 1) & 3;  // 64-byte swizzle: 16-byte chunk c sits at c ^ swz
        const int rbx = row / box_rows, rin = row & (box_rows - 1);
        TileWalker<NQ> wk(t_begin, t_end, tiles_per_seq, chunks);
        int seg, j0, kind;
        int64_t c = 0;
        while (wk.next(s, 2, d_status, false, seg, j0, kind)) {
            const int st = (int)(c % S);
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(full + st, (uint32_t)(c / S) & 1, abort_flag, d_status)))
                break;
            const uint8_t* stg = stages + st * C::stage_bytes;
            uint4 cw[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                cw[k] = *reinterpret_cast<const uint4*>(stg + row * kNvCodeBytes + ((k ^ swz) << 4));
            const uint2 sc = *reinterpret_cast<const uint2*>(stg + C::codes_bytes + rbx * sc_slot +
                                                             (rin + bpar[st * 8 + rbx]) * kNvScaleBytes);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty + st);  // codes in registers: the stage may refill
            const int b = (int)(c & 1);
            const uint32_t bu = (uint32_t)(c >> 1);
            if (!__all_sync(0xffffffffu, c < 2 || ptx::mbar_wait(aempty + b, (bu - 1) & 1, abort_flag, d_status)))
                break;
            ptx::tc_fence_after();
            const uint32_t dst = tmem_base + lane_addr + acol0 + b * C::a_cols;
            uint32_t v[32];
            nv4_chunk(cw[0], sc.x, v);
            nv4_chunk(cw[1], sc.x >> 16, v + 16);
            ptx::tmem_st32_nowait(dst, v);
            nv4_chunk(cw[2], sc.y, v);
            nv4_chunk(cw[3], sc.y >> 16, v + 16);
            ptx::tmem_st32_nowait(dst + 32, v);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(afull + b);
            ++c;
        }
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        float* sw = sw_all + (warp - 2) * N;
        int* spos = spos_all + (warp - 2) * NQ;
        TileWalker<NQ> wk(t_begin, t_end, tiles_per_seq, chunks);
        int seg, j0, kind, cur = -1;
        int64_t consumed = 0;
        while (wk.next(s, 1, d_status, true, seg, j0, kind)) {
            const IdxSeg& g = wk.g;
            if (seg != cur) {
                __syncwarp();
                for (int e = lane; e < N; e += 32)
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
            const int grp = (j0 >> 5) + quarter;
            const bool grp_live = j0 + quarter * 32 < g.ctx;
            if (kind == 1) {
                for (int q = 0; q < g.nq; ++q) {
                    if (scores && in_ctx) scores[(int64_t)(g.q0 + q) * ld + j] = -INFINITY;
                    if (gmax && lane == 0 && grp_live) gmax[(int64_t)(g.q0 + q) * ldg + grp] = -INFINITY;
                }
                continue;
            }
            const int is = (int)(consumed % kNvInfoSlots);
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(ifull + is, (uint32_t)(consumed / kNvInfoSlots) & 1,
                                                        abort_flag, d_status)))
                break;
            const int64_t bb = reinterpret_cast<const int64_t*>(info + is * 64)[row / box_rows];
            int64_t prow = bb >= 0 ? bb + (row & (box_rows - 1)) : -1;
            if (prow >= s.num_rows) prow = -1;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(iempty + is);
            if (in_ctx && prow < 0) report(d_status, DSA_ERR_BAD_INPUT);
            const int a = (int)(consumed & 1);
            const uint32_t au = (uint32_t)(consumed >> 1);
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(tfull + a, au & 1, abort_flag, d_status))) break;
            ptx::tc_fence_after();
            const uint32_t tcol = tmem_base + ((uint32_t)(quarter * 32) << 16) + a * NM;
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
            auto store = [&](int q, float r) {
                if (q >= g.nq) return;
                const float v = (in_ctx && prow >= 0 && j <= spos[q]) ? r : -INFINITY;
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
            if constexpr (C::split_n) {
                // hi and lo columns into registers, the accumulator back, their sums
                uint32_t v[2][32];
                ptx::tmem_ld32_async(tcol, v[0]);
                ptx::tmem_ld32_async(tcol + 32, v[1]);
                ptx::tmem_wait_ld32(v[0]);
                ptx::tmem_wait_ld32(v[1]);
                release();
#pragma unroll
                for (int h = 0; h < 32; ++h)
                    v[0][h] = __float_as_uint(__uint_as_float(v[0][h]) + __uint_as_float(v[1][h]));
                store(0, relu_sum(v[0], 0));
            } else if constexpr (NQ == 1) {
                // every column into registers, then the accumulator goes back
                uint32_t v[NQ][32];
#pragma unroll
                for (int q = 0; q < NQ; ++q) ptx::tmem_ld32_async(tcol + q * 32, v[q]);
#pragma unroll
                for (int q = 0; q < NQ; ++q) ptx::tmem_wait_ld32(v[q]);
                release();
#pragma unroll
                for (int q = 0; q < NQ; ++q) store(q, relu_sum(v[q], q));
            } else {
                // the next query's columns load while this one's are summed
                uint32_t v[2][32];
                ptx::tmem_ld32_async(tcol, v[0]);
                ptx::tmem_wait_ld32(v[0]);
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    if (q + 1 < NQ) ptx::tmem_ld32_async(tcol + (q + 1) * 32, v[(q + 1) & 1]);
                    const float r = relu_sum(v[q & 1], q);
                    if (q + 1 < NQ) ptx::tmem_wait_ld32(v[(q + 1) & 1]);
                    if (q + 1 == NQ) release();
                    store(q, r);
                }
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

template <int NQ, int KP>
cudaError_t launch_nv4(const void* qp, int num_q, const float* wp, const void* codes, const void* kscales,
                       const dsa_seqs& s, float* scores, int64_t ld, float* gmax, int64_t ldg, int32_t* d_status,
                       cudaStream_t stream) {
    using C = Nv4Cfg<NQ, KP>;
    const int box_rows = s.page_table ? std::min(64, s.page_size & -s.page_size) : kTileKeys;
    CUtensorMap kmap, qmap, smap;
    cudaError_t e = make_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, kNvCodeBytes, (uint64_t)s.num_rows,
                             kNvCodeBytes, kNvCodeBytes, box_rows, CU_TENSOR_MAP_SWIZZLE_64B);
    if (e != cudaSuccess) return e;
    // the block scales as one 8-byte element per row (a single outer row); a
    // box covers its rows plus two
    e = make_map(&smap, CU_TENSOR_MAP_DATA_TYPE_UINT64, kscales, (uint64_t)s.num_rows, 1,
                 ((uint64_t)s.num_rows * kNvScaleBytes + 15) / 16 * 16, (uint32_t)box_rows + 2, 1,
                 CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    e = make_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qp, C::KM, (uint64_t)num_q * (C::NM / NQ), C::KM * 2, 64,
                 C::NM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    auto kern = index_nv4_kernel<NQ, KP>;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [kern] {
        attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::smem);
    });
    if (attr != cudaSuccess) return attr;
    const int tiles_per_seq = (s.max_ctx + kTileKeys - 1) / kTileKeys;
    const int chunks = (s.max_q_per_seq + NQ - 1) / NQ;
    const int64_t total = (int64_t)s.num_seqs * chunks * tiles_per_seq;
    const int grid = (int)std::min<int64_t>((int64_t)C::ctas_per_sm * num_sms(), total);
    return launch_pdl(kern, dim3(grid), dim3(C::threads), C::smem, stream, 1, kmap, qmap, smap, wp, s, scores, ld,
                      gmax, ldg, tiles_per_seq, chunks, total, box_rows, d_status);
}

template <int NQ>
cudaError_t launch_nv4_nq(bool rope, const void* qp, int num_q, const float* wp, const void* codes,
                          const void* kscales, const dsa_seqs& s, float* scores, int64_t ld, float* gmax, int64_t ldg,
                          int32_t* d_status, cudaStream_t stream) {
    return rope ? launch_nv4<NQ, 192>(qp, num_q, wp, codes, kscales, s, scores, ld, gmax, ldg, d_status, stream)
                : launch_nv4<NQ, 128>(qp, num_q, wp, codes, kscales, s, scores, ld, gmax, ldg, d_status, stream);
}

}  // namespace

cudaError_t launch_index_scores_nvfp4(const void* q_idx, const float* w, const float* ssmax_s, const float* ssmax_b,
                                      const float* inv_freq, const void* k_codes, const void* k_block_scales,
                                      float k_global, const dsa_seqs& s, int num_q, float* scores, int64_t ld,
                                      float* gmax, int64_t ldg, const Workspace& ws, int32_t* d_status,
                                      cudaStream_t stream) {
    const bool rope = inv_freq != nullptr;
    __half* qp = reinterpret_cast<__half*>(ws.qprep);
    const int mq = s.max_q_per_seq;
    const int split_n = Nv4Cfg<1, 192>::split_n && rope && mq <= 1;  // the layout the kernel below reads
    cudaError_t e = launch_pdl(qprep_f16_kernel, dim3(num_q), dim3(kIH * 32), 0, stream, 1,
                               reinterpret_cast<const __nv_bfloat16*>(q_idx), w, ssmax_s, ssmax_b, inv_freq, s, num_q,
                               k_global, split_n, qp, ws.wprep, d_status);
    if (e != cudaSuccess) return e;
    if (mq <= 1)
        return launch_nv4_nq<1>(rope, qp, num_q, ws.wprep, k_codes, k_block_scales, s, scores, ld, gmax, ldg, d_status,
                                stream);
    if (mq <= 2)
        return launch_nv4_nq<2>(rope, qp, num_q, ws.wprep, k_codes, k_block_scales, s, scores, ld, gmax, ldg, d_status,
                                stream);
    return launch_nv4_nq<4>(rope, qp, num_q, ws.wprep, k_codes, k_block_scales, s, scores, ld, gmax, ldg, d_status,
                            stream);
}

}  // namespace dsa
