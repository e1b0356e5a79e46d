// mla.cu -- sparse absorbed-MLA attention over selected latent rows (sm_103a).
//
// "Day 0 support for Mistral Large 4" (vLLM blog), Model architecture (64
// heads, MLA with KV LoRA rank 512 and RoPE dim 64), Sparse MLA + DSA indexer
// (attention reads only the selected tokens), NoPE, SSMax and LeRoPE (NoPE
// layers are MLA with zero RoPE dims), DCP (partial results merged by an LSE
// combine; an empty row is neutral), FP8 latent cache (656-byte fp8_ds_mla
// rows).
//
// For query t and head h over the selected rows c_j (576 dims):
//   s_j = sm_scale q_h . c_j,  out_h = sum_j softmax(s)_j c_j[0:512],
//   lse_h = ln sum_j exp(s_j).
// One CTA takes one query and one split of its selected slots; the kernel is
// described above mla_tc_kernel.  Splits combine in-kernel when there are two
// (a thread-block cluster), else they write unnormalised partial outputs with
// their (max, sum), merged by the LSE combine kernel.  fp8_ds_mla rows are
// dequantised by the gather (code x group scale, one rounding to f16).
#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include <mutex>

#include <cuda_fp4.h>

#include "tc_ptx.cuh"

namespace dsa {

static size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Split count of each query's selected slots: as many splits as fill one wave
// of 152 SMs (one resident CTA per SM), at least two 64-row tiles per split,
// at most 16 (the combine's weights per head).  Two splits run as a cluster
// pair and combine in distributed shared memory; more write fp32 partials
// that the combine kernel merges, which must fit `cap` bytes of scratch
// (fewer splits otherwise; one or two always fit).
// One CTA per SM at a time: a query split s ways is num_q * s CTAs of
// ceil(tiles / s) tiles, which run in ceil(num_q * s / 152) waves.  The split
// count minimises waves x (tiles per split + a CTA's fixed cost), in tenths
// of a tile: the query's load and the pipeline's fill (about one tile), the
// pair's exchange in distributed shared memory (two splits, 0.3), or the fp32
// partials of three or more splits and their combine (128 KB per split and
// query, about two tiles more).  At least two tiles per split, at most 16.
int mla_splits(int num_q, int k, size_t cap) {
    const int tiles = (k + 63) / 64;
    const int64_t nq = num_q > 0 ? num_q : 1;
    int max_sp = tiles / 2 > 0 ? tiles / 2 : 1;  // at least two 64-row tiles per split
    if (max_sp > 16) max_sp = 16;                  // the combine holds 16 weights per head
    int sp = 1;
    int64_t best = -1;
    for (int c = 1; c <= max_sp; ++c) {
        const int64_t waves = (nq * c + 151) / 152;
        const int64_t fixed = 10 + (c > 2 ? 20 : c == 2 ? 3 : 0);
        const int64_t cost = waves * (10 * ((tiles + c - 1) / c) + fixed);
        if (best < 0 || cost < best) {
            best = cost;
            sp = c;
        }
    }
    while (sp > 2 && up256((size_t)nq * sp * kMH * kMV * 4) + up256((size_t)nq * sp * kMH * 2 * 4) > cap) --sp;
    return sp;
}

static bool mla_pair(int splits) { return splits == 2; }

size_t mla_part_bytes(int num_q, int k, size_t cap) {
    const int sp = mla_splits(num_q, k, cap);
    return sp > 1 && !mla_pair(sp) ? (size_t)num_q * sp * kMH * kMV * 4 : 0;
}

size_t mla_ml_bytes(int num_q, int k, size_t cap) {
    const int sp = mla_splits(num_q, k, cap);
    return sp > 1 && !mla_pair(sp) ? (size_t)num_q * sp * kMH * 2 * 4 : 0;
}

int mla_launches(int num_q, int k, size_t cap) {
    const int sp = mla_splits(num_q, k, cap);
    return sp > 1 && !mla_pair(sp) ? 2 : 1;
}

// LSE combine of the splits of one query ([vLLM-ML4] DCP: LSE combine):
//   M = max_s m_s, out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
// One block per (query, 4 heads), one thread per 4 output dims, every
// split's load of them in flight together.
constexpr int kCombineHeads = 4;
constexpr int kCombineThreads = kCombineHeads * kMV / 4;  // 512
__global__ void __launch_bounds__(kCombineThreads) mla_combine_kernel(const float* __restrict__ part_o,
                                                          const float* __restrict__ part_ml, int splits,
                                                          __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
    pdl_enter();
    __shared__ float wgt[kCombineHeads * 16];
    __shared__ float inv_l[kCombineHeads];
    const int t = blockIdx.x, h0 = blockIdx.y * kCombineHeads;
    const float* ml = part_ml + (int64_t)t * splits * kMH * 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < kCombineHeads) {  // warp hh: the weights of head h0 + hh, lane s those of split s
        const int h = h0 + warp;
        const bool has = lane < splits;
        const float m = has ? ml[(lane * kMH + h) * 2] : -INFINITY;
        const float l = has ? ml[(lane * kMH + h) * 2 + 1] : 0.f;
        float M = m;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float wv = (!has || M == -INFINITY) ? 0.f : exp2f(m - M);
        float L = wv * l;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (has) wgt[warp * 16 + lane] = wv;
        if (lane == 0) {
            inv_l[warp] = L > 0.f ? 1.f / L : 0.f;
            if (lse) lse[(int64_t)t * kMH + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
        }
    }
    __syncthreads();
    const float* po = part_o + (int64_t)t * splits * kMH * kMV + (int64_t)h0 * kMV;
    __nv_bfloat16* ot = out + (int64_t)t * kMH * kMV + (int64_t)h0 * kMV;
    {
        const int e = threadIdx.x;
        const int hh = (e * 4) / kMV;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int sp = 0; sp < splits; ++sp) {
            const float wv = wgt[hh * 16 + sp];
            const float4 v = *reinterpret_cast<const float4*>(po + (int64_t)sp * kMH * kMV + e * 4);
            acc.x += wv * v.x;
            acc.y += wv * v.y;
            acc.z += wv * v.z;
            acc.w += wv * v.w;
        }
        const float il = inv_l[hh];
        uint2 o;
        o.x = pack_bf16(acc.x * il, acc.y * il);
        o.y = pack_bf16(acc.z * il, acc.w * il);
        *reinterpret_cast<uint2*>(ot + e * 4) = o;
    }
}

// 16-byte read-only load that does not allocate in L1: gathered rows are used
// once, and skipping the L1 fill leaves the shared-memory banks (the same SRAM)
// to the tensor-core operand reads.
__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ldg_stream8(const void* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// 8 e4m3 codes x their group scale -> 8 f16 (one rounding, from fp32); sets
// `over` when a value leaves the f16 range
__device__ __forceinline__ uint4 dequant8_f16(uint2 codes, float scale, bool& over) {
    const uint32_t w[4] = {codes.x & 0xFFFFu, codes.x >> 16, codes.y & 0xFFFFu, codes.y >> 16};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t h2 = e4m3x2_to_f16x2((uint16_t)w[i]);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
        const float a = f.x * scale, b = f.y * scale;
        over |= fabsf(a) >= 65520.f || fabsf(b) >= 65520.f;
        o[i] = pack_f16(a, b);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// 8 E2M1 values (4 bytes, the even value in each low nibble) x their E4M3
// group scale -> 8 f16.  Exact: a product of a 2-bit and a 4-bit significand
// within f16's range (at most 6 x 448).
__device__ __forceinline__ uint4 nvfp4x8_to_f16x8(uint32_t codes, uint32_t scale_code) {
    const __half2_raw sr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(scale_code | (scale_code << 8)),
                                                      __NV_E4M3);
    const __half2 sc = *reinterpret_cast<const __half2*>(&sr);
    // the four code bytes unpacked into byte registers, each converted as is
    uint32_t h[4], o[4];
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(codes));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 pr = __hmul2(*reinterpret_cast<const __half2*>(&h[i]), sc);
        o[i] = *reinterpret_cast<const uint32_t*>(&pr);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// 8 bf16 -> 8 f16 (exact inside the f16 range)
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v, bool& over) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = __uint_as_float(w[i] << 16), b = __uint_as_float(w[i] & 0xFFFF0000u);
        over |= fabsf(a) >= 65520.f || fabsf(b) >= 65520.f;
        o[i] = pack_f16(a, b);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// ---------------------------------------------------------------------------
// Latent cache on the 5th-generation tensor cores: bf16 rows, or fp8_ds_mla
// rows dequantised to f16 by the gather (the query is then converted to f16
// in shared memory, exact inside the f16 range, and the products run in f16).
//
// One CTA = one query x one split of its selected slots, tiles of 64 rows:
//   warp 0      loads the 64 query heads (TMA) and resolves each tile's slots
//               to physical rows (page table) up to three tiles ahead;
//   warps 10-17 gather the tile's rows: 16-byte loads, 18 per thread in flight,
//               stored into the 128-byte-swizzled K-major layout (two stages);
//               random 1,152-byte rows stream fastest this way on GB300;
//   warp 1      issues S^T = K Q^T on the tensor cores (M = 64 keys, N = 64
//               heads, K = 576; key r lands in TMEM lane 32 (r / 16) + r % 16);
//   warp 18     issues O^T += V^T P^T (M = 128 value dims per block, N = 64
//               heads, K = 64 keys; V^T is the same gathered tile read
//               MN-major), each product as soon as its P^T is written;
//   warps 2-9   softmax, two warps per TMEM lane quarter (16 keys), each with
//               32 of the heads, straight from TMEM: exact per-head maxima of
//               the first tile set the running max; later tiles only check
//               that no score exceeds it by more than 2^64 (one flag per warp
//               exchanged) and raise it, each warp rescaling its own part of
//               O^T, only when one does; exp2, row sums kept in TMEM, P^T
//               written over the tile's rope block (64 keys x 64 heads, bf16,
//               exactly its size), which the scores no longer need; then the
//               output or the split partial.
namespace tcmla {
constexpr int TK = 64;                     // selected rows per tile
constexpr int KB = kMD / 64;               // 9 blocks of 64 dims
constexpr int kKBlock = TK * 128;          // bytes of one 64-dim block of a tile
constexpr int kStage = KB * kKBlock;       // 73728
constexpr int kQBytes = KB * kMH * 128;    // 73728
constexpr int kMisc = 4608;
constexpr size_t kSmem = 2 * (size_t)kStage + kQBytes + kMisc;
constexpr float kRescale = 64.f;           // log2 headroom before O^T is rescaled (bf16 P, fp32 O)
constexpr uint32_t kOCol = 0;              // O^T: 4 blocks x 64 heads
constexpr uint32_t kSCol = 256;            // S^T: 2 buffers x 64 heads
constexpr uint32_t kLCol = 384;            // row sums: lanes = keys, columns = heads
constexpr uint32_t kTmemCols = 512;
constexpr int kThreads = 608;              // 19 warps
constexpr int kGatherWarps = 8;
constexpr int kSoftWarps = 8;
constexpr int kPvWarp = 2 + kSoftWarps + kGatherWarps;  // 18: issues O^T += V^T P^T
constexpr int kRing = 3;                   // resolved-row ring depth
constexpr int kBf16Rows = 0, kDsMlaRows = 1, kNvfp4Rows = 2;  // latent cache kinds
constexpr int kNvRow = kMD / 2;            // NVFP4 code bytes per row (288)
constexpr int kNvScales = kMD / 16;        // NVFP4 E4M3 scales per row (36)
static_assert(kKBlock == TK * kMH * 2, "P^T must fit the rope block of its tile");
}  // namespace tcmla

// KIND: the latent cache (kBf16Rows, kDsMlaRows, kNvfp4Rows); out_scale
// multiplies every output (an NVFP4 cache's tensor scale, else 1).
template <int KIND>
__global__ void __launch_bounds__(tcmla::kThreads, 1)
    mla_tc_kernel(const __grid_constant__ CUtensorMap qmap, const uint8_t* __restrict__ latent,
                  const uint8_t* __restrict__ lat_scales, dsa_seqs s, const int32_t* __restrict__ idx,
                  const int32_t* __restrict__ topk_len, int k, float scale_log2, float out_scale, int splits, int pair,
                  __nv_bfloat16* __restrict__ out, float* __restrict__ lse, float* __restrict__ part_o,
                  float* __restrict__ part_ml, int32_t* d_status) {
    pdl_enter();
    using namespace tcmla;
    constexpr bool FP8 = KIND == kDsMlaRows;
    constexpr bool NV4 = KIND == kNvfp4Rows;
    constexpr bool F16 = FP8 || NV4;  // products in f16 (the gather decodes to f16)
    extern __shared__ __align__(1024) uint8_t tc_smem[];   // 1024-aligned for the 128-byte swizzle atoms
    uint8_t* const smem = tc_smem;
    uint8_t* stage = smem;                                  // [2][KB][TK rows x 128 B]; block 8 later holds P^T
    uint8_t* qs = smem + 2 * kStage;                        // [KB][64 heads x 128 B]
    uint8_t* misc = qs + kQBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
    uint64_t* qfull = bars + 0;
    // A tile is stored and released in two halves: blocks 0-3 (value dims
    // 0-255) and blocks 4-8 (value dims 256-511, the rope block, later P^T).
    uint64_t* kfull = bars + 1;   // [2 halves][2 stages] half of a gathered tile stored (8 gather warps)
    uint64_t* kempty = bars + 5;  // [2 halves][2 stages] half of a tile no longer read by the MMA
    uint64_t* sfull = bars + 9;   // [2] S^T ready
    uint64_t* sempty = bars + 11; // [2] S^T read by the softmax warps
    uint64_t* xch = bars + 13;    // [2] growth flags of the softmax warps written
    uint64_t* pfull = bars + 27;  // [2] P^T written (and O^T rescaled) by the softmax warps
    uint64_t* pvdone = bars + 16; // O^T += V^T P^T of the tile complete
    uint64_t* ofull = bars + 17;  // last product complete
    uint64_t* lready = bars + 18; // row sums of the softmax warps written
    uint64_t* rfull = bars + 19;  // [3] rows of a tile resolved
    uint64_t* rfree = bars + 22;  // [3] rows of a tile no longer read (gather + softmax warps)
    uint64_t* xmax = bars + 25;   // per-head maxima of the softmax warps written (first tile, growth)
    uint64_t* qconv = bars + 26;  // fp8 cache: the query converted to f16 (softmax warps)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 256);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 260);  // and the kernel tag at +264
    int* srow = reinterpret_cast<int*>(misc + 512);          // [3][TK] physical row (-1 = masked)
    float* wmax = reinterpret_cast<float*>(misc + 1280);     // [4 lane quarters][64] per-head maxima
    float* mu = reinterpret_cast<float*>(misc + 2304);       // [8 warps][32 heads] running max (log2 units)
    float* lsum = reinterpret_cast<float*>(misc + 3328);     // [4 lane quarters][64] row sums
    int* wflag = reinterpret_cast<int*>(misc + 4352);        // [2 parity][8 warps] growth flags

    const int t = blockIdx.y, sp = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = seq_of(s.q_start, s.num_seqs, t);
    const int ctx = __ldg(s.ctx_len + b);
    int len = __ldg(topk_len + t);
    if (len < 0 || len > k || ctx > s.max_ctx) {
        if (threadIdx.x == 0 && sp == 0) report(d_status, DSA_ERR_BAD_INPUT);
        len = 0;
    }
    // the query's live slots [0, len) in equal whole tiles per split (a
    // compacted selection, len << k, keeps every split busy)
    const int per = ((len + splits - 1) / splits + TK - 1) / TK * TK;
    const int slot0 = sp * per;
    const int slot1 = min(slot0 + per, len);
    const int ntiles = slot1 > slot0 ? (slot1 - slot0 + TK - 1) / TK : 0;
    const int32_t* tidx = idx + (int64_t)t * k;

    if (threadIdx.x == 0) {
        ptx::mbar_init(qfull, 1);
        for (int i = 0; i < 4; ++i) {
            ptx::mbar_init(kfull + i, kGatherWarps);
            ptx::mbar_init(kempty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(sfull + i, 1);
            ptx::mbar_init(sempty + i, kSoftWarps);
            ptx::mbar_init(xch + i, kSoftWarps);
        }
        for (int i = 0; i < kRing; ++i) {
            ptx::mbar_init(rfull + i, 1);
            ptx::mbar_init(rfree + i, kGatherWarps + kSoftWarps);
        }
        ptx::mbar_init(pfull, kSoftWarps);
        ptx::mbar_init(pfull + 1, kSoftWarps);
        ptx::mbar_init(pvdone, 1);
        ptx::mbar_init(ofull, 1);
        ptx::mbar_init(lready, kSoftWarps);
        ptx::mbar_init(xmax, kSoftWarps);
        ptx::mbar_init(qconv, kSoftWarps);
        *abort_flag = 0;
        abort_flag[1] = FP8 ? kTagMlaFp8 : NV4 ? kTagMlaNvfp4 : kTagMla;  // names this kernel in a timeout's status
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ query load, row resolution
        if (lane == 0 && ntiles > 0) {
            ptx::prefetch_tmap(&qmap);
            ptx::mbar_expect_tx(qfull, kQBytes);
            for (int kb = 0; kb < KB; ++kb) ptx::tma_load_2d(qs + kb * kMH * 128, &qmap, kb * 64, t * kMH, qfull);
        }
        for (int i = 0; i < ntiles; ++i) {
            const int r = i % kRing;
            int rows2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int slot = slot0 + i * TK + 2 * lane + u;
                int row = -1;
                if (slot < slot1) {
                    const int j = __ldg(tidx + slot);
                    if (j >= ctx || j < -1) {
                        report(d_status, DSA_ERR_BAD_INPUT);
                    } else if (j >= 0) {
                        const int64_t pr = phys_row(s, b, j);
                        if (pr < 0) report(d_status, DSA_ERR_BAD_INPUT);
                        else row = (int)pr;
                    }
                }
                rows2[u] = row;
            }
            bool ok = true;
            if (lane == 0 && i >= kRing) ok = ptx::mbar_wait(rfree + r, ((i / kRing) - 1) & 1, abort_flag, d_status);
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            srow[r * TK + 2 * lane] = rows2[0];
            srow[r * TK + 2 * lane + 1] = rows2[1];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(rfull + r);
        }
    } else if (warp == 1 || warp == kPvWarp) {
        // ------------------------------------------------------------ MMA issuers
        // Two threads issue the tensor-core work, each in its own order: warp
        // 1 the scores S^T of every tile, warp 18 the products O^T += V^T P^T.
        // A thread issuing MMAs is held ~60 cycles per instruction whatever
        // its size, while a 64 x 64 x 16 MMA keeps the pipe only a fraction of
        // that: with two issuers the product of tile i goes in as soon as its
        // P^T is written, not behind S^T of tile i+1, and the stage it frees
        // reaches the gather of tile i+2 that much sooner.  Each thread's
        // commits track its own MMAs; the product of tile i follows S^T of tile
        // i (its P^T needs those scores), so its commits release the stage.
        if (lane == 0 && ntiles > 0 && warp == 1) {
            constexpr uint32_t idesc_s = ptx::idesc_f16(64, kMH, !F16);
            const uint32_t qb = smem_u32(qs);
            // S^T of a tile in two parts, blocks 0-3 then 4-8, each as soon as
            // that half of the tile is stored
            auto issue_s = [&](int st, int kb0, int kb1) {
                ptx::tc_fence_after();
                const uint32_t kbase = smem_u32(stage + st * kStage);
#pragma unroll
                for (int kb = kb0; kb < kb1; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t ad = ptx::sdesc_sw128(kbase + kb * kKBlock + ks * 32);
                        const uint64_t bd = ptx::sdesc_sw128(qb + kb * kMH * 128 + ks * 32);
                        ptx::mma_ss(tmem + kSCol + st * kMH, ad, bd, idesc_s, (kb > 0 || ks > 0) ? 1u : 0u);
                    }
            };
            bool ok = ptx::mbar_wait(F16 ? qconv : qfull, 0, abort_flag, d_status);
            for (int i = 0; ok && i < ntiles; ++i) {
                const int st = i & 1;
                const uint32_t ph = (i >> 1) & 1;
                // the S^T buffer read by the softmax two tiles back, then each half stored
                ok = (i < 2 || ptx::mbar_wait(sempty + st, ph ^ 1, abort_flag, d_status)) &&
                     ptx::mbar_wait(kfull + st, ph, abort_flag, d_status);
                if (!ok) break;
                issue_s(st, 0, 4);
                if (!(ok = ptx::mbar_wait(kfull + 2 + st, ph, abort_flag, d_status))) break;
                issue_s(st, 4, KB);
                ptx::mma_commit(sfull + st);
            }
        } else if (lane == 0 && ntiles > 0) {
            constexpr uint32_t idesc_pv = ptx::idesc_f16(128, kMH, !F16, true, true);
            bool ok = true;
            for (int i = 0; ok && i < ntiles; ++i) {
                if (!(ok = ptx::mbar_wait(pfull + (i & 1), (i >> 1) & 1, abort_flag, d_status))) break;
                ptx::tc_fence_after();
                const uint32_t kbase = smem_u32(stage + (i & 1) * kStage);
                const uint32_t pb = kbase + 8 * kKBlock;
#pragma unroll
                for (int db = 0; db < 4; ++db) {
#pragma unroll
                    for (int kk = 0; kk < TK / 16; ++kk) {
                        const uint64_t ad = ptx::sdesc_sw128_mn(kbase + 2 * db * kKBlock + kk * 2048, kKBlock, 1024);
                        const uint64_t bd = ptx::sdesc_sw128_mn(pb + kk * 2048, kKBlock, 1024);
                        ptx::mma_ss(tmem + kOCol + db * kMH, ad, bd, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
                    }
                    if (db == 1) ptx::mma_commit(kempty + (i & 1));  // blocks 0-3 read
                }
                ptx::mma_commit(kempty + 2 + (i & 1));              // blocks 4-8 (with P^T) read
                ptx::mma_commit(pvdone);
            }
            if (ok) ptx::mma_commit(ofull);  // every product complete (the last follows every S^T)
        }
    } else if (warp >= 2 + kSoftWarps) {
        // ------------------------------------------------------------ gather
        // thread gt: 16-byte chunk c8 of rows r0 and r0 + 32 in every 64-dim
        // block (eight threads read one row's 128 contiguous bytes of a block)
        const int gt = threadIdx.x - (2 + kSoftWarps) * 32;  // 0..255
        const int c8 = gt & 7, r0 = gt >> 3;
        const uint32_t soff = (uint32_t)r0 * 128 + ((c8 ^ (r0 & 7)) << 4);  // same swizzle for r0 + 32
        for (int i = 0; i < ntiles; ++i) {
            const int st = i & 1, r = i % kRing;
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(rfull + r, (i / kRing) & 1, abort_flag, d_status))) break;
            uint4 v[18];  // v[2 kb + h]: block kb of row r0 + 32 h, 16-bit values as stored in the stage
            if constexpr (FP8) {
                // fp8_ds_mla row: [0,512) e4m3 codes, [512,528) four fp32 scales
                // (one per 128 dims), [528,656) 64 bf16 rope dims.  Thread (c8, r0):
                // codes 8 c8 .. 8 c8 + 7 of every 64-dim block of rows r0, r0 + 32.
                const uint8_t* b0 = latent + (size_t)max(srow[r * TK + r0], 0) * kDsRow;
                const uint8_t* b1 = latent + (size_t)max(srow[r * TK + r0 + 32], 0) * kDsRow;
                uint2 cv[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) cv[u] = ldg_stream8(((u & 1) ? b1 : b0) + (u >> 1) * 64 + c8 * 8);
                const float4 sc0 = __ldg(reinterpret_cast<const float4*>(b0 + kMV));
                const float4 sc1 = __ldg(reinterpret_cast<const float4*>(b1 + kMV));
                const uint4 rp0 = ldg_stream(reinterpret_cast<const uint4*>(b0 + kMV + 16) + c8);
                const uint4 rp1 = ldg_stream(reinterpret_cast<const uint4*>(b1 + kMV + 16) + c8);
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(rfree + r);
                bool over = false;
                const float s0[4] = {sc0.x, sc0.y, sc0.z, sc0.w}, s1[4] = {sc1.x, sc1.y, sc1.z, sc1.w};
#pragma unroll
                for (int u = 0; u < 16; ++u) v[u] = dequant8_f16(cv[u], (u & 1) ? s1[u >> 2] : s0[u >> 2], over);
                v[16] = bf16x8_to_f16x8(rp0, over);
                v[17] = bf16x8_to_f16x8(rp1, over);
                if (over) report(d_status, DSA_ERR_UNSUPPORTED);
            } else if constexpr (NV4) {
                // NVFP4 row: codes [288] (value 2i in the low nibble of byte i,
                // 2i + 1 in the high one) and E4M3 scales [36] (one per 16
                // values).  Thread (c8, r0): values 8 c8 .. 8 c8 + 7 of every
                // 64-dim block of rows r0, r0 + 32 -- 4 code bytes and the
                // scale of their 16-value group (byte c8 / 2 of the block's 4)
                const int row0 = max(srow[r * TK + r0], 0), row1 = max(srow[r * TK + r0 + 32], 0);
                const uint8_t* b0 = latent + (size_t)row0 * kNvRow;
                const uint8_t* b1 = latent + (size_t)row1 * kNvRow;
                const uint8_t* q0 = lat_scales + (size_t)row0 * kNvScales;
                const uint8_t* q1 = lat_scales + (size_t)row1 * kNvScales;
                uint32_t cw[18], sw4[18];
#pragma unroll
                for (int u = 0; u < 18; ++u) {
                    cw[u] = __ldg(reinterpret_cast<const uint32_t*>(((u & 1) ? b1 : b0) + (u >> 1) * 32 + c8 * 4));
                    sw4[u] = __ldg(reinterpret_cast<const uint32_t*>(((u & 1) ? q1 : q0) + (u >> 1) * 4));
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(rfree + r);
#pragma unroll
                for (int u = 0; u < 18; ++u) v[u] = nvfp4x8_to_f16x8(cw[u], (sw4[u] >> (8 * (c8 >> 1))) & 0xFFu);
            } else {
                const uint4* g0 = reinterpret_cast<const uint4*>(latent + (size_t)max(srow[r * TK + r0], 0) * (kMD * 2)) + c8;
                const uint4* g1 = reinterpret_cast<const uint4*>(latent + (size_t)max(srow[r * TK + r0 + 32], 0) * (kMD * 2)) + c8;
#pragma unroll
                for (int u = 0; u < 18; ++u) v[u] = ldg_stream(((u & 1) ? g1 : g0) + (u >> 1) * 8);
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(rfree + r);
            }
            uint8_t* dst = stage + st * kStage + soff;
            bool ok = true;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                // blocks 0-3 once the product two tiles back has read them, then blocks 4-8
                if (i >= 2 && !__all_sync(0xffffffffu, ptx::mbar_wait(kempty + 2 * half + st, ((i >> 1) - 1) & 1,
                                                                      abort_flag, d_status))) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int u = half ? 8 : 0; u < (half ? 18 : 8); ++u)
                    *reinterpret_cast<uint4*>(dst + (u >> 1) * kKBlock + (u & 1) * 32 * 128) = v[u];
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(kfull + 2 * half + st);
            }
            if (!ok) break;
        }
    } else {
        // ------------------------------------------------------------ softmax and output (warps 2-9)
        const int quarter = warp & 3;                       // TMEM lanes 32*quarter ..
        const int sw = warp - 2;                            // softmax warp index 0..7
        const int hb = (sw >> 2) * 32;                      // this warp's heads hb .. hb+31
        const bool mine = lane < 16;                        // lanes holding a key of the tile
        const int key = quarter * 16 + (lane & 15);         // key row of the tile
        const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);  // this warp's TMEM lanes
        float* my_mu = mu + sw * 32;                        // running max of heads hb .. hb+31
        if constexpr (F16) {
            // the query to f16 in place (its 16-bit elements keep their positions)
            if (ntiles > 0) {
                const bool got = __all_sync(0xffffffffu, ptx::mbar_wait(qfull, 0, abort_flag, d_status));
                bool over = false;
                if (got) {
                    uint4* q4 = reinterpret_cast<uint4*>(qs);
                    for (int e = sw * 32 + lane; e < kQBytes / 16; e += kSoftWarps * 32) q4[e] = bf16x8_to_f16x8(q4[e], over);
                }
                if (over) report(d_status, DSA_ERR_UNSUPPORTED);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(qconv);
            }
        }
        my_mu[lane] = -INFINITY;
        {
            float z[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) z[j] = 0.f;
            ptx::tmem_st32(tl + kLCol + hb, z);
        }
        __syncwarp();
        bool alive = true;
        int n_grow = 0;  // exact-maxima exchanges so far (same count in every softmax warp)
        for (int i = 0; alive && i < ntiles; ++i) {
            const int st = i & 1, r = i % kRing;
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(rfull + r, (i / kRing) & 1, abort_flag, d_status) &&
                                             ptx::mbar_wait(sfull + st, (i >> 1) & 1, abort_flag, d_status))) {
                alive = false;
                break;
            }
            const bool valid = mine && srow[r * TK + key] >= 0;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(rfree + r);
            ptx::tc_fence_after();
            const uint32_t s_addr = tl + kSCol + st * kMH + hb;
            // does any score of this tile rise more than 2^64 above the running max?
            bool grow = i == 0;
            if (i > 0) {
                float sv[32];
                ptx::tmem_ld32(s_addr, sv);
                float over = -INFINITY;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 m4 = reinterpret_cast<const float4*>(my_mu)[q];
                    over = fmaxf(over, fmaxf(fmaxf(sv[4 * q] * scale_log2 - m4.x, sv[4 * q + 1] * scale_log2 - m4.y),
                                             fmaxf(sv[4 * q + 2] * scale_log2 - m4.z, sv[4 * q + 3] * scale_log2 - m4.w)));
                }
                const bool g = __any_sync(0xffffffffu, valid && over > kRescale);
                if (lane == 0) wflag[st * kSoftWarps + sw] = g ? 1 : 0;
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(xch + st);
                // xch[st] serves tiles 1, 2, 3, ... (not 0): use u of it is tile 2u+1 or 2u+2
                if (!__all_sync(0xffffffffu, ptx::mbar_wait(xch + st, ((i - 1) >> 1) & 1, abort_flag, d_status))) {
                    alive = false;
                    break;
                }
                int any = 0;
#pragma unroll
                for (int w = 0; w < kSoftWarps; ++w) any |= wflag[st * kSoftWarps + w];
                grow = any != 0;
            }
            float alpha = 1.f;  // lane j: rescale factor of head hb + j
            if (grow) {
                // exact per-head maxima of this tile (first tile, or a growth)
                float sv[32];
                ptx::tmem_ld32(s_addr, sv);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float m = ptx::warp_max(valid ? sv[j] * scale_log2 : -INFINITY);
                    if (lane == j) wmax[quarter * kMH + hb + j] = m;
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(xmax);
                if (!__all_sync(0xffffffffu, ptx::mbar_wait(xmax, n_grow & 1, abort_flag, d_status))) {
                    alive = false;
                    break;
                }
                ++n_grow;
                const int h = hb + lane;
                const float mt = fmaxf(fmaxf(wmax[h], wmax[kMH + h]), fmaxf(wmax[2 * kMH + h], wmax[3 * kMH + h]));
                const float mo = my_mu[lane];
                const float mn = fmaxf(mo, mt);
                alpha = (mo == -INFINITY || mn == mo) ? (mo == mn ? 1.f : 0.f) : exp2f(mo - mn);
                __syncwarp();
                my_mu[lane] = mn;
                __syncwarp();
            }
            const bool rescale = grow && i > 0;
            if (rescale) {
                // O^T holds the products of tiles 0 .. i-1 once the previous one completes
                if (!__all_sync(0xffffffffu, ptx::mbar_wait(pvdone, (i - 1) & 1, abort_flag, d_status))) {
                    alive = false;
                    break;
                }
                ptx::tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 10; ++c) {  // 4 value blocks x 2 halves of this warp's heads, then the row sums
                    const uint32_t col = c < 8 ? kOCol + (c >> 1) * kMH + hb + (c & 1) * 16 : kLCol + hb + (c & 1) * 16;
                    float o[16];
                    ptx::tmem_ld16(tl + col, o);
#pragma unroll
                    for (int j = 0; j < 16; ++j) o[j] *= __shfl_sync(0xffffffffu, alpha, (c & 1) * 16 + j);
                    ptx::tmem_st16(tl + col, o);
                }
            }
            // probabilities, row sums (TMEM), this warp's half of the P^T row over the rope block
            uint8_t* prow = stage + st * kStage + 8 * kKBlock + key * 128;
#pragma unroll
            for (int g = 0; g < 2; ++g) {  // 16 heads at a time
                float sv[16], lv[16];
                ptx::tmem_ld16(s_addr + g * 16, sv);
                ptx::tmem_ld16(tl + kLCol + hb + g * 16, lv);
                uint32_t pk[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 m4 = reinterpret_cast<const float4*>(my_mu)[g * 4 + q];
                    const float mq[4] = {m4.x, m4.y, m4.z, m4.w};
                    float p[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        p[e] = (!valid || mq[e] == -INFINITY) ? 0.f : fast_exp2(sv[4 * q + e] * scale_log2 - mq[e]);
                        lv[4 * q + e] += p[e];
                    }
                    pk[2 * q] = F16 ? pack_f16(p[0], p[1]) : pack_bf16(p[0], p[1]);
                    pk[2 * q + 1] = F16 ? pack_f16(p[2], p[3]) : pack_bf16(p[2], p[3]);
                }
                ptx::tmem_st16(tl + kLCol + hb + g * 16, lv);
                if (mine) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int cc = (hb >> 3) + g * 2 + c;
                        *reinterpret_cast<uint4*>(prow + ((cc ^ (key & 7)) << 4)) =
                            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(sempty + st);
                ptx::mbar_arrive(pfull + (i & 1));
            }
        }
        // ---- row sums of this warp's 16 keys -> lsum[quarter][hb .. hb+31]
        if (alive && ntiles > 0) {
            ptx::tc_fence_after();
            float lv[32];
            ptx::tmem_ld32(tl + kLCol + hb, lv);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                float v = lv[j];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);  // lanes 16-31 add zeros
                if (lane == j) lsum[quarter * kMH + hb + j] = v;
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(lready);
        }
        // ---- output: value dim quarter*32 + lane of each 128-dim block, heads hb .. hb+31
        const int dim = quarter * 32 + lane;
        bool have = alive && ntiles > 0;
        if (have) have = __all_sync(0xffffffffu, ptx::mbar_wait(lready, 0, abort_flag, d_status));
        if (have) have = __all_sync(0xffffffffu, ptx::mbar_wait(ofull, 0, abort_flag, d_status));
        if (have) ptx::tc_fence_after();
        auto total_l = [&](int h) { return lsum[h] + lsum[kMH + h] + lsum[2 * kMH + h] + lsum[3 * kMH + h]; };
        auto run_max = [&](int h) { return mu[(h >> 5) * 4 * 32 + (h & 31)]; };  // copy of warp sw = 4 (h / 32)
        if (splits == 1) {
            __nv_bfloat16* ot = out + (int64_t)t * kMH * kMV;
#pragma unroll 1
            for (int db = 0; db < 4; ++db) {  // 32 columns = heads hb .. hb+31 of one 128-dim block
                float o[32];
                if (have) ptx::tmem_ld32(tl + kOCol + db * kMH + hb, o);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int h = hb + j;
                    const float L = have ? total_l(h) : 0.f;
                    const float v = L > 0.f ? (o[j] * out_scale) / L : 0.f;
                    ot[(int64_t)h * kMV + db * 128 + dim] = __float2bfloat16_rn(v);
                }
            }
            if (lse && sw == 0) {
                for (int h = lane; h < kMH; h += 32) {
                    const float L = have ? total_l(h) : 0.f;
                    lse[(int64_t)t * kMH + h] = L > 0.f ? (run_max(h) + log2f(L)) * 0.69314718055994531f : -INFINITY;
                }
            }
        } else if (!pair) {
            float* po = part_o + ((int64_t)t * splits + sp) * kMH * kMV;
#pragma unroll 1
            for (int db = 0; db < 4; ++db) {
                float o[32];
                if (have) ptx::tmem_ld32(tl + kOCol + db * kMH + hb, o);
#pragma unroll
                for (int j = 0; j < 32; ++j) po[(int64_t)(hb + j) * kMV + db * 128 + dim] = have ? o[j] * out_scale : 0.f;
            }
            if (sw == 0) {
                for (int h = lane; h < kMH; h += 32) {
                    float* ml = part_ml + (((int64_t)t * splits + sp) * kMH + h) * 2;
                    const float L = have ? total_l(h) : 0.f;
                    ml[0] = L > 0.f ? run_max(h) : -INFINITY;
                    ml[1] = L;
                }
            }
        } else {
            // Two splits of this query form a cluster: CTA r keeps heads 32r ..
            // 32r+31 and sends the other half of its unnormalised O^T, with the
            // running max and row sum of those heads, into the partner's
            // stages (free once every product of both CTAs is complete: the
            // first cluster barrier), then combines its half after the second.
            cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
            const int me = (int)cluster.block_rank();
            float* xo = reinterpret_cast<float*>(stage);   // [32 heads][512] partner's partial of my heads
            float* xml = xo + 32 * kMV;                     // [32 heads][2] partner's (max, sum)
            const float m_own = have ? run_max(hb + lane) : -INFINITY;
            const float l_own = have ? total_l(hb + lane) : 0.f;
            cluster.sync();  // 1: stages of both CTAs free
            if (hb != me * 32) {
                float* rxo = cluster.map_shared_rank(xo, me ^ 1);
                float* rml = cluster.map_shared_rank(xml, me ^ 1);
#pragma unroll 1
                for (int db = 0; db < 4; ++db) {
                    float o[32];
                    if (have) ptx::tmem_ld32(tl + kOCol + db * kMH + hb, o);
#pragma unroll
                    for (int j = 0; j < 32; ++j) rxo[j * kMV + db * 128 + dim] = have ? o[j] : 0.f;
                }
                if (quarter == 0) {
                    rml[lane * 2] = l_own > 0.f ? m_own : -INFINITY;
                    rml[lane * 2 + 1] = l_own;
                }
            }
            cluster.sync();  // 2: the partner's half is in my stages
            if (hb == me * 32) {
                // lane j: weights of head hb + j
                const float m1 = xml[lane * 2], l1 = xml[lane * 2 + 1];
                const float m0 = l_own > 0.f ? m_own : -INFINITY;
                const float mx = fmaxf(m0, m1);
                const float w0 = l_own > 0.f ? exp2f(m0 - mx) : 0.f;
                const float w1 = l1 > 0.f ? exp2f(m1 - mx) : 0.f;
                const float L = w0 * l_own + w1 * l1;
                const float inv = L > 0.f ? 1.f / L : 0.f;
                const float a0 = w0 * inv * out_scale, a1 = w1 * inv * out_scale;
                __nv_bfloat16* ot = out + (int64_t)t * kMH * kMV;
#pragma unroll 1
                for (int db = 0; db < 4; ++db) {
                    float o[32];
                    if (have) ptx::tmem_ld32(tl + kOCol + db * kMH + hb, o);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float x = xo[j * kMV + db * 128 + dim];
                        const float v = __shfl_sync(0xffffffffu, a0, j) * (have ? o[j] : 0.f) +
                                        __shfl_sync(0xffffffffu, a1, j) * x;
                        ot[(int64_t)(hb + j) * kMV + db * 128 + dim] = __float2bfloat16_rn(v);
                    }
                }
                if (lse && quarter == 0)
                    lse[(int64_t)t * kMH + hb + lane] = L > 0.f ? (mx + log2f(L)) * 0.69314718055994531f : -INFINITY;
            }
        }
    }
    if (pair && (warp < 2 || warp >= 2 + kSoftWarps)) {
        // the other roles take part in the two cluster barriers of the epilogue
        cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
        cluster.sync();
        cluster.sync();
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 mla_tmap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

cudaError_t bf16_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
    auto enc = mla_tmap_encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)kMD, rows};
    cuuint64_t strides[1] = {(cuuint64_t)kMD * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_sparse_mla(const void* q, const void* latent, dsa_dtype latent_dtype, const dsa_seqs& s,
                              int num_q, const int32_t* idx, const int32_t* topk_len, int k, float sm_scale,
                              void* out, float* lse, const Workspace& ws, int32_t* d_status, cudaStream_t stream,
                              size_t scratch_cap, const void* lat_scales, float lat_global) {
    const int kind = latent_dtype == DSA_FP8_DS_MLA ? tcmla::kDsMlaRows
                     : latent_dtype == DSA_NVFP4    ? tcmla::kNvfp4Rows
                                                    : tcmla::kBf16Rows;
    const int splits = mla_splits(num_q, k, scratch_cap);
    // an NVFP4 cache's tensor scale g: s_j = sm_scale g q.c~_j and out = g sum p c~
    const float g = kind == tcmla::kNvfp4Rows ? lat_global : 1.f;
    const float scale_log2 = sm_scale * g * 1.4426950408889634f;
    CUtensorMap qmap;
    cudaError_t e = bf16_map(&qmap, q, (uint64_t)num_q * kMH, 64);
    if (e != cudaSuccess) return e;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(mla_tc_kernel<tcmla::kBf16Rows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)tcmla::kSmem);
        if (attr == cudaSuccess)
            attr = cudaFuncSetAttribute(mla_tc_kernel<tcmla::kDsMlaRows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)tcmla::kSmem);
        if (attr == cudaSuccess)
            attr = cudaFuncSetAttribute(mla_tc_kernel<tcmla::kNvfp4Rows>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)tcmla::kSmem);
    });
    if (attr != cudaSuccess) return attr;
    // with two splits, the pair runs as a cluster and combines through
    // distributed shared memory: no partials, no combine launch
    const int pair = mla_pair(splits) ? 1 : 0;
    auto kern = kind == tcmla::kDsMlaRows   ? mla_tc_kernel<tcmla::kDsMlaRows>
                : kind == tcmla::kNvfp4Rows ? mla_tc_kernel<tcmla::kNvfp4Rows>
                                            : mla_tc_kernel<tcmla::kBf16Rows>;
    e = launch_pdl(kern, dim3(splits, num_q), dim3(tcmla::kThreads), tcmla::kSmem, stream, pair ? 2 : 1, qmap,
                   reinterpret_cast<const uint8_t*>(latent), reinterpret_cast<const uint8_t*>(lat_scales), s, idx,
                   topk_len, k, scale_log2, g, splits, pair, reinterpret_cast<__nv_bfloat16*>(out), lse, ws.mla_part,
                   ws.mla_ml, d_status);
    if (e != cudaSuccess || splits == 1 || pair) return e;
    return launch_pdl(mla_combine_kernel, dim3(num_q, kMH / kCombineHeads), dim3(kCombineThreads), 0, stream, 1, ws.mla_part,
                      ws.mla_ml, splits, reinterpret_cast<__nv_bfloat16*>(out), lse);
}

}  // namespace dsa
