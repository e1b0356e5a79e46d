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
//
// Work plan.  A query's k slots are T = ceil(k / 64) tiles of 64 slots.  The
// num_q x T tiles, query after query, are cut into G equal contiguous ranges,
// one per CTA (one resident CTA per SM, G at most the SM count), so every SM
// gets the same number of tiles whatever the batch.  A CTA's range is walked
// as segments, each the piece of one query that falls in it.  A segment
// holding a whole query writes that query's output; the pieces of a query cut
// between CTAs write normalised fp32 partial outputs with their (max, sum) -- the
// first segment of CTA c to partial slot 2c, its last to slot 2c + 1 -- and
// the combine kernel merges them with their LSE weights.  When a query's live
// slots [0, topk_len) are fewer than k, each piece's nominal tiles map
// proportionally onto the live tiles, so every CTA keeps an equal share.
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_ptx.cuh"

namespace dsa {

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

namespace tcmla {
constexpr int TK = 64;                     // selected rows per tile
constexpr int KB = kMD / 64;               // 9 blocks of 64 dims
constexpr int kKBlock = TK * 128;          // bytes of one 64-dim block of a tile
constexpr int kStage = KB * kKBlock;       // 73728
constexpr int kQBytes = KB * kMH * 128;    // 73728
constexpr int kMisc = 9728;
constexpr size_t kSmem = 2 * (size_t)kStage + kQBytes + kMisc;
static_assert(kSmem <= 232448, "one CTA per SM within the 227 KB of shared memory a CTA may use");
constexpr float kRescale = 64.f;           // log2 headroom before O^T is rescaled (bf16 P, fp32 O)
constexpr uint32_t kOCol = 0;              // O^T: 4 blocks x 64 heads
constexpr uint32_t kSCol = 256;            // S^T: 2 buffers x 64 heads
constexpr uint32_t kLCol = 384;            // row sums: lanes = keys, columns = heads
constexpr uint32_t kTmemCols = 512;
constexpr int kThreads = 576;              // 18 warps
constexpr int kGatherWarps = 8;
constexpr int kSoftWarps = 8;
constexpr int kRing = 4;                   // resolved-row ring: rows resolved and prefetched to L2 ahead
constexpr int kMinTiles = 2;               // fewest tiles a CTA is given
constexpr int kMaxParts = 64;              // pieces of one query the combine merges
constexpr int kMaxSegs = 128;              // segments of one CTA (its table in shared memory)
constexpr int kSlotBytes = kMH * kMV * 4;  // one partial output, fp32
constexpr int kSlotMl = kMH * 2 * 4;       // its (max, sum) per head
static_assert(kKBlock == TK * kMH * 2, "P^T must fit the rope block of its tile");
static_assert((DSA_MAX_TOPK + TK - 1) / TK + 1 <= kMaxParts, "a query's pieces fit the combine");
}  // namespace tcmla

// ---------------------------------------------------------------------------
// The work plan (host and device agree on it from these three numbers).
struct MlaPlan {
    int T;          // tiles per query: ceil(k / 64)
    int G;          // CTAs
    int64_t total;  // num_q * T
};

__host__ __device__ __forceinline__ int64_t plan_start(const MlaPlan& p, int c) {
    return (int64_t)c * p.total / p.G;
}
// the CTA whose range holds tile g: the largest c with plan_start(c) <= g
__host__ __device__ __forceinline__ int plan_cta_of(const MlaPlan& p, int64_t g) {
    return (int)(((g + 1) * p.G + p.total - 1) / p.total) - 1;
}

static MlaPlan mla_plan(int num_q, int k, int max_ctas) {
    MlaPlan p;
    p.T = (k + tcmla::TK - 1) / tcmla::TK;
    p.total = (int64_t)(num_q > 0 ? num_q : 1) * p.T;
    int64_t g = (p.total + tcmla::kMinTiles - 1) / tcmla::kMinTiles;
    if (g > max_ctas) g = max_ctas;
    // a range of at most (kMaxSegs - 2) T tiles touches at most kMaxSegs - 1
    // queries: very large batches take more CTAs (several waves)
    const int64_t per = (int64_t)(tcmla::kMaxSegs - 2) * p.T;
    const int64_t g_min = (p.total + per - 1) / per;
    if (g < g_min) g = g_min;
    p.G = g < 1 ? 1 : (int)g;
    return p;
}

// true when a CTA boundary falls inside a query: partials and the combine
static bool plan_splits(const MlaPlan& p) {
    for (int c = 1; c < p.G; ++c)
        if (plan_start(p, c) % p.T != 0) return true;
    return false;
}

static int device_sms() {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kMlaMaxCtas;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return kMlaMaxCtas;
        cache[dev] = n;
    }
    return cache[dev];
}

static int launch_ctas(int max_ctas) {
    const int sms = device_sms();
    return sms < max_ctas ? sms : max_ctas;
}

size_t mla_part_bytes(int num_q, int k, int max_ctas) {
    return (size_t)2 * mla_plan(num_q, k, max_ctas).G * tcmla::kSlotBytes;
}

size_t mla_ml_bytes(int num_q, int k, int max_ctas) {
    return (size_t)2 * mla_plan(num_q, k, max_ctas).G * tcmla::kSlotMl;
}

int mla_launches(int num_q, int k, int max_ctas) {
    return plan_splits(mla_plan(num_q, k, launch_ctas(max_ctas))) ? 2 : 1;
}

int mla_max_ctas_for_scratch(size_t bytes) {
    const size_t per = (size_t)2 * (tcmla::kSlotBytes + tcmla::kSlotMl);
    const size_t n = bytes / per;
    return (int)(n < (size_t)kMlaMaxCtas ? n : kMlaMaxCtas);
}

// A CTA's range as segments: the pieces of one query each.  Segment j of CTA
// c is query start(c) / T + j clipped to the range (no state to carry).
struct Seg {
    int q, a0, a1;  // query, nominal tiles [a0, a1) of its T
    bool first;     // the CTA's first segment
};
__device__ __forceinline__ int plan_nseg(const MlaPlan& p, int c) {
    const int64_t g0 = plan_start(p, c), e = plan_start(p, c + 1);
    return e > g0 ? (int)((e - 1) / p.T - g0 / p.T) + 1 : 0;
}
__device__ __forceinline__ Seg plan_seg(const MlaPlan& p, int c, int j) {
    const int64_t g0 = plan_start(p, c), e = plan_start(p, c + 1);
    Seg sg;
    sg.q = (int)(g0 / p.T) + j;
    const int64_t qs = (int64_t)sg.q * p.T;
    sg.a0 = (int)(max(g0, qs) - qs);
    sg.a1 = (int)(min(e, qs + p.T) - qs);
    sg.first = j == 0;
    return sg;
}
// A segment's live tiles: the query's slots [0, len) fill L = ceil(len / 64)
// tiles; its nominal tiles [a0, a1) of T take the live tiles [a0 L / T, a1 L / T).
struct Live {
    int b, ctx, len, l0, l1;
};
__device__ __forceinline__ Live seg_live(const Seg& sg, const dsa_seqs& s, const int32_t* topk_len, int k, int T,
                                        int32_t* d_status) {
    Live v;
    v.b = seq_of(s.q_start, s.num_seqs, sg.q);
    v.ctx = __ldg(s.ctx_len + v.b);
    v.len = __ldg(topk_len + sg.q);
    if (v.len < 0 || v.len > k || v.ctx > s.max_ctx) {
        if (d_status) report(d_status, DSA_ERR_BAD_INPUT);
        v.len = 0;
    }
    const int L = (v.len + tcmla::TK - 1) / tcmla::TK;
    v.l0 = (int)((int64_t)sg.a0 * L / T);
    v.l1 = (int)((int64_t)sg.a1 * L / T);
    return v;
}
// A CTA's segments, resolved once at the start into shared memory (their
// query lengths and sequences are global loads the roles' loops must not wait
// on).
struct SegEntry {
    int q, l0, l1, len;  // query, live tiles [l0, l1), live slots
    int b, ctx, flags, pad;  // its sequence and context; kWhole | kFirst
};
constexpr int kWhole = 1, kFirst = 2;

// The tiles of a CTA's non-empty segments, in order.
struct TileCursor {
    int j;                // next table entry to look at
    int seg, q, n, i, g;  // non-empty segment index, its query, its tiles, tile in it, tile in the CTA
    bool done;
    __device__ __forceinline__ TileCursor() : j(0), seg(-1), q(0), n(0), i(0), g(0), done(false) {}
    __device__ __forceinline__ void next_segment(const SegEntry* tab, int nseg) {
        while (j < nseg) {
            const SegEntry e = tab[j++];
            if (e.l1 > e.l0) {
                ++seg;
                q = e.q;
                n = e.l1 - e.l0;
                i = 0;
                return;
            }
        }
        done = true;
    }
    __device__ __forceinline__ void advance(const SegEntry* tab, int nseg) {
        ++g;
        if (++i == n) next_segment(tab, nseg);
    }
};

// LSE combine of the pieces of the queries cut between CTAs ([vLLM-ML4] DCP:
// LSE combine): with m_p in log2 units and l_p the pieces' row sums,
// w_p = l_p 2^(m_p - M) / sum_p l_p 2^(m_p - M), out = sum_p w_p o_p (o_p the
// normalised partial outputs).  One block per (query, 4 heads); queries held
// whole by one CTA were written by the attention kernel.
constexpr int kCombineHeads = 4;
__global__ void __launch_bounds__(128) mla_combine_kernel(const float* __restrict__ part_o,
                                                          const float* __restrict__ part_ml, MlaPlan plan,
                                                          __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
    using namespace tcmla;
    pdl_enter();
    __shared__ float wgt[kCombineHeads][kMaxParts];
    __shared__ int slot_of[kMaxParts];
    const int q = blockIdx.x, h0 = blockIdx.y * kCombineHeads;
    const int c_lo = plan_cta_of(plan, (int64_t)q * plan.T);
    const int c_hi = plan_cta_of(plan, (int64_t)(q + 1) * plan.T - 1);
    if (c_lo == c_hi) return;
    const int parts = min(c_hi - c_lo + 1, kMaxParts);
    for (int p = threadIdx.x; p < parts; p += blockDim.x) {
        const int cc = c_lo + p;
        const int first_q = (int)(plan_start(plan, cc) / plan.T);
        slot_of[p] = 2 * cc + (first_q == q ? 0 : 1);
    }
    __syncthreads();
    if (threadIdx.x < kCombineHeads) {
        const int h = h0 + threadIdx.x;
        float M = -INFINITY;
        for (int p = 0; p < parts; ++p) {
            const float* ml = part_ml + ((int64_t)slot_of[p] * kMH + h) * 2;
            if (ml[1] > 0.f) M = fmaxf(M, ml[0]);
        }
        float L = 0.f;
        for (int p = 0; p < parts; ++p) {
            const float* ml = part_ml + ((int64_t)slot_of[p] * kMH + h) * 2;
            const float wv = (ml[1] > 0.f && M != -INFINITY) ? ml[1] * exp2f(ml[0] - M) : 0.f;
            wgt[threadIdx.x][p] = wv;
            L += wv;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int p = 0; p < parts; ++p) wgt[threadIdx.x][p] *= inv;
        if (lse) lse[(int64_t)q * kMH + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
    }
    __syncthreads();
    __nv_bfloat16* ot = out + ((int64_t)q * kMH + h0) * kMV;
    for (int e = threadIdx.x; e < kCombineHeads * kMV / 4; e += blockDim.x) {
        const int hh = (e * 4) / kMV;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p = 0; p < parts; ++p) {
            const float wv = wgt[hh][p];
            if (wv == 0.f) continue;
            const float4 v = *reinterpret_cast<const float4*>(part_o + ((int64_t)slot_of[p] * kMH + h0) * kMV + e * 4);
            acc.x += wv * v.x;
            acc.y += wv * v.y;
            acc.z += wv * v.z;
            acc.w += wv * v.w;
        }
        uint2 o;
        o.x = pack_bf16(acc.x, acc.y);
        o.y = pack_bf16(acc.z, acc.w);
        *reinterpret_cast<uint2*>(ot + e * 4) = o;
    }
}

// ---------------------------------------------------------------------------
// Latent cache on the 5th-generation tensor cores: bf16 rows, or fp8_ds_mla
// rows dequantised to f16 by the gather (the query is then converted to f16
// in shared memory, exact inside the f16 range, and the products run in f16).
//
// One CTA walks its range of the plan, tiles of 64 selected rows:
//   warp 0      resolves each tile's slots to physical rows (page table) up to
//               kRing tiles ahead and prefetches those rows into L2 (one bulk
//               prefetch per row), so the gather's loads find them there;
//   warp 1      loads each segment's 64 query heads (TMA, once the previous
//               segment's scores are complete) and issues tcgen05.mma:
//               S^T = K Q^T (M = 64 keys, N = 64 heads, K = 576; key r lands in
//               TMEM lane 32 (r / 16) + r % 16) and O^T += V^T P^T (M = 128
//               value dims per block, N = 64 heads, K = 64 keys; V^T is the
//               same gathered tile read MN-major);
//   warps 10-17 gather the tile's rows: 16-byte loads, 18 per thread in flight,
//               stored into the 128-byte-swizzled K-major layout (two stages);
//   warps 2-9   softmax, two warps per TMEM lane quarter (16 keys), each with
//               32 of the heads, straight from TMEM: exact per-head maxima of
//               a segment's first tile set the running max; later tiles only
//               check that no score exceeds it by more than 2^64 (one flag per
//               warp exchanged) and raise it, each warp rescaling its own part
//               of O^T, only when one does; exp2, row sums kept in TMEM, P^T
//               written over the tile's rope block (64 keys x 64 heads, bf16,
//               exactly its size), which the scores no longer need; at a
//               segment's end the output or the partial.
template <bool FP8>
__global__ void __launch_bounds__(tcmla::kThreads, 1)
    mla_tc_kernel(const __grid_constant__ CUtensorMap qmap, const uint8_t* __restrict__ latent, dsa_seqs s,
                  const int32_t* __restrict__ idx, const int32_t* __restrict__ topk_len, int k, float scale_log2,
                  MlaPlan plan, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                  float* __restrict__ part_o, float* __restrict__ part_ml, int32_t* d_status) {
    pdl_enter();
    using namespace tcmla;
    extern __shared__ __align__(1024) uint8_t tc_smem[];   // 1024-aligned for the 128-byte swizzle atoms
    uint8_t* const smem = tc_smem;
    uint8_t* stage = smem;                                  // [2][KB][TK rows x 128 B]; block 8 later holds P^T
    uint8_t* qs = smem + 2 * kStage;                        // [KB][64 heads x 128 B]
    uint8_t* misc = qs + kQBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
    uint64_t* qfull = bars + 0;   // the segment's query loaded (TMA)
    // A tile is stored and released in two halves: blocks 0-3 (value dims
    // 0-255) and blocks 4-8 (value dims 256-511, the rope block, later P^T).
    uint64_t* kfull = bars + 1;   // [2 halves][2 stages] half of a gathered tile stored (8 gather warps)
    uint64_t* kempty = bars + 5;  // [2 halves][2 stages] half of a tile no longer read by the MMA
    uint64_t* sfull = bars + 9;   // [2] S^T ready
    uint64_t* sempty = bars + 11; // [2] S^T read by the softmax warps
    uint64_t* xch = bars + 13;    // [2] growth flags of the softmax warps written
    uint64_t* pfull = bars + 15;  // [2] P^T written (and O^T rescaled) by the softmax warps
    uint64_t* pvdone = bars + 17; // O^T += V^T P^T of the tile complete
    uint64_t* ofull = bars + 18;  // last product of a segment complete
    uint64_t* lready = bars + 19; // row sums of the softmax warps written
    uint64_t* xmax = bars + 20;   // per-head maxima of the softmax warps written (first tile, growth)
    uint64_t* qconv = bars + 21;  // fp8 cache: the query converted to f16 (softmax warps)
    uint64_t* qfree = bars + 22;  // every S^T of a segment complete: the query buffer may be reloaded
    uint64_t* oempty = bars + 23; // O^T of a segment read by the softmax warps
    uint64_t* mdone = bars + 24;  // every tensor-core operation of the CTA complete (exit)
    uint64_t* rfull = bars + 25;  // [kRing] rows of a tile resolved
    uint64_t* rfree = rfull + kRing;  // [kRing] rows of a tile no longer read (gather + softmax warps)
    static_assert(25 + 2 * kRing <= 64, "barriers fit their 512 bytes");
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 512);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 516);  // and the kernel tag at +520
    int* srow = reinterpret_cast<int*>(misc + 1024);                 // [kRing][TK] physical row (-1 = masked)
    float* wmax = reinterpret_cast<float*>(misc + 1024 + kRing * TK * 4);  // [4 lane quarters][64] maxima
    float* mu = wmax + 4 * kMH;                                      // [8 warps][32 heads] running max (log2)
    float* lsum = mu + kSoftWarps * 32;                              // [4 lane quarters][64] row sums
    int* wflag = reinterpret_cast<int*>(lsum + 4 * kMH);             // [2][8 warps] growth flags
    SegEntry* segtab = reinterpret_cast<SegEntry*>(misc + 5632);     // [kMaxSegs] the CTA's segments
    static_assert(1024 + kRing * TK * 4 + (4 * kMH + kSoftWarps * 32 + 4 * kMH) * 4 + 2 * kSoftWarps * 4 <= 5632,
                  "misc fits below the segment table");
    static_assert(5632 + kMaxSegs * sizeof(SegEntry) <= (size_t)kMisc, "segment table fits");

    const int c = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the CTA's segments, all resolved at once (the plan keeps them <= kMaxSegs)
    const int nseg = min(plan_nseg(plan, c), kMaxSegs);
    for (int j = threadIdx.x; j < nseg; j += kThreads) {
        const Seg sg = plan_seg(plan, c, j);
        // the CTA holding a query's first tile reports its bad length
        const Live lv = seg_live(sg, s, topk_len, k, plan.T, sg.a0 == 0 ? d_status : nullptr);
        SegEntry e;
        e.q = sg.q;
        e.l0 = lv.l0;
        e.l1 = lv.l1;
        e.len = lv.len;
        e.b = lv.b;
        e.ctx = lv.ctx;
        e.flags = (sg.a0 == 0 && sg.a1 == plan.T ? kWhole : 0) | (sg.first ? kFirst : 0);
        e.pad = 0;
        segtab[j] = e;
    }

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
            ptx::mbar_init(pfull + i, kSoftWarps);
        }
        for (int i = 0; i < kRing; ++i) {
            ptx::mbar_init(rfull + i, 1);
            ptx::mbar_init(rfree + i, kGatherWarps + kSoftWarps);
        }
        ptx::mbar_init(pvdone, 1);
        ptx::mbar_init(ofull, 1);
        ptx::mbar_init(lready, kSoftWarps);
        ptx::mbar_init(xmax, kSoftWarps);
        ptx::mbar_init(qconv, kSoftWarps);
        ptx::mbar_init(qfree, 1);
        ptx::mbar_init(oempty, kSoftWarps);
        ptx::mbar_init(mdone, 1);
        *abort_flag = 0;
        abort_flag[1] = FP8 ? kTagMlaFp8 : kTagMla;  // names this kernel in a timeout's status
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
        // ------------------------------------------------------------ row resolution, L2 prefetch
        // Tiles go in groups of kRing: the slot loads of the whole group are
        // issued together, then its page-table loads, so a group costs two
        // dependent load latencies rather than two per tile.  Lane l takes
        // slots 2l and 2l + 1 of each tile.
        const uint32_t row_bytes = FP8 ? (uint32_t)kDsRow : (uint32_t)(kMD * 2);
        int j = 0, lt = 0;  // cursor: segment, live tile within it
        if (nseg > 0) lt = segtab[0].l0;
        int gi = 0;
        bool ok = true;
        while (ok) {
            int tj[kRing], tlt[kRing], n = 0;  // the group's tiles: segment entry, live tile
#pragma unroll
            for (int u = 0; u < kRing; ++u) {
                while (j < nseg && lt >= segtab[j].l1)
                    if (++j < nseg) lt = segtab[j].l0;
                tj[u] = j < nseg ? j : 0;
                tlt[u] = j < nseg ? lt++ : 0;
                if (j < nseg) n = u + 1;
            }
            if (n == 0) break;
            int jv[kRing][2];
#pragma unroll
            for (int u = 0; u < kRing; ++u)
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    jv[u][v] = -2;  // no slot
                    if (u < n) {
                        const SegEntry& e = segtab[tj[u]];
                        const int slot = tlt[u] * TK + 2 * lane + v;
                        if (slot < e.len) jv[u][v] = __ldg(idx + (int64_t)e.q * k + slot);
                    }
                }
            int rows[kRing][2];
#pragma unroll
            for (int u = 0; u < kRing; ++u)
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    int row = -1;
                    if (u < n && jv[u][v] != -2) {
                        const SegEntry& e = segtab[tj[u]];
                        const int jj = jv[u][v];
                        if (jj >= e.ctx || jj < -1) {
                            report(d_status, DSA_ERR_BAD_INPUT);
                        } else if (jj >= 0) {
                            const int64_t pr = phys_row(s, e.b, jj);
                            if (pr < 0) report(d_status, DSA_ERR_BAD_INPUT);
                            else row = (int)pr;
                        }
                    }
                    rows[u][v] = row;
                }
#pragma unroll
            for (int u = 0; u < kRing; ++u)
#pragma unroll
                for (int v = 0; v < 2; ++v)
                    if (rows[u][v] >= 0) ptx::prefetch_l2_bulk(latent + (size_t)rows[u][v] * row_bytes, row_bytes);
#pragma unroll
            for (int u = 0; u < kRing; ++u) {
                if (u >= n) break;
                const int r = gi % kRing;
                if (lane == 0 && gi >= kRing) ok = ptx::mbar_wait(rfree + r, ((gi / kRing) - 1) & 1, abort_flag, d_status);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    ok = false;
                    break;
                }
                srow[r * TK + 2 * lane] = rows[u][0];
                srow[r * TK + 2 * lane + 1] = rows[u][1];
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(rfull + r);
                ++gi;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ query loads and the MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = ptx::idesc_f16(64, kMH, !FP8);
            constexpr uint32_t idesc_pv = ptx::idesc_f16(128, kMH, !FP8, true, true);
            const uint32_t qb = smem_u32(qs);
            ptx::prefetch_tmap(&qmap);
            TileCursor sc, pc;  // the S^T stream and the O^T stream
            sc.next_segment(segtab, nseg);
            pc.next_segment(segtab, nseg);
            int q_loaded = -1;  // last segment whose query load was issued
            int q_ready = -1;   // last segment whose query is known loaded (and converted)
            bool issued = false;
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
            auto issue_pv = [&](int g, bool first) {  // O^T (+)= V^T P^T for tile g
                ptx::tc_fence_after();
                const uint32_t kbase = smem_u32(stage + (g & 1) * kStage);
                const uint32_t pb = kbase + 8 * kKBlock;
#pragma unroll
                for (int db = 0; db < 4; ++db) {
#pragma unroll
                    for (int kk = 0; kk < TK / 16; ++kk) {
                        const uint64_t ad = ptx::sdesc_sw128_mn(kbase + 2 * db * kKBlock + kk * 2048, kKBlock, 1024);
                        const uint64_t bd = ptx::sdesc_sw128_mn(pb + kk * 2048, kKBlock, 1024);
                        ptx::mma_ss(tmem + kOCol + db * kMH, ad, bd, idesc_pv, (!first || kk > 0) ? 1u : 0u);
                    }
                    if (db == 1) ptx::mma_commit(kempty + (g & 1));  // blocks 0-3 read
                }
                ptx::mma_commit(kempty + 2 + (g & 1));              // blocks 4-8 (with P^T) read
                ptx::mma_commit(pvdone);
            };
            // The streams interleave: the scores of tile i+1 are computed while
            // the softmax of tile i runs, and a segment's query is loaded as soon
            // as the previous segment's scores are complete.  Every barrier is
            // probed without blocking: a blocking wait on one would miss another
            // completing.  S^T of a tile goes in two parts, blocks 0-3 then 4-8,
            // each as soon as that half of the tile is stored.
            int s_half = 0;
            bool ok = true;
            ptx::WaitClock idle;  // time without progress
            while (ok && !pc.done) {
                bool progressed = false;
                if (!sc.done && q_loaded < sc.seg &&
                    (sc.seg == 0 || ptx::mbar_test_wait(qfree, (sc.seg - 1) & 1))) {
                    ptx::mbar_expect_tx(qfull, kQBytes);
                    for (int kb = 0; kb < KB; ++kb)
                        ptx::tma_load_2d(qs + kb * kMH * 128, &qmap, kb * 64, sc.q * kMH, qfull);
                    q_loaded = sc.seg;
                    progressed = true;
                }
                if (!sc.done && q_ready < sc.seg && q_loaded == sc.seg &&
                    ptx::mbar_test_wait(FP8 ? qconv : qfull, sc.seg & 1))
                    q_ready = sc.seg;
                if (!sc.done && q_ready == sc.seg) {
                    const int st = sc.g & 1;
                    const uint32_t ph = (sc.g >> 1) & 1;
                    if (s_half == 0 && ptx::mbar_test_wait(kfull + st, ph) &&
                        (sc.g < 2 || ptx::mbar_test_wait(sempty + st, ph ^ 1))) {
                        issue_s(st, 0, 4);
                        issued = true;
                        s_half = 1;
                        progressed = true;
                    }
                    if (s_half == 1 && ptx::mbar_test_wait(kfull + 2 + st, ph)) {
                        issue_s(st, 4, KB);
                        ptx::mma_commit(sfull + st);
                        if (sc.i + 1 == sc.n) ptx::mma_commit(qfree);  // the segment's last S^T
                        s_half = 0;
                        sc.advance(segtab, nseg);
                        progressed = true;
                    }
                }
                if (pc.g < sc.g && ptx::mbar_test_wait(pfull + (pc.g & 1), (pc.g >> 1) & 1) &&
                    (pc.i > 0 || pc.seg == 0 || ptx::mbar_test_wait(oempty, (pc.seg - 1) & 1))) {
                    issue_pv(pc.g, pc.i == 0);
                    if (pc.i + 1 == pc.n) ptx::mma_commit(ofull);  // the segment's O^T complete
                    pc.advance(segtab, nseg);
                    progressed = true;
                }
                if (progressed) {
                    idle.reset();
                } else {
                    // bounded idle: give up after the wait limit like every other wait
                    if (idle.expired(ptx::kWaitTimeoutNs) || *abort_flag) {
                        if (!*abort_flag) {
                            *abort_flag = 1;
                            report(d_status, ptx::timeout_code(abort_flag, ptx::kLoopSite));
                        }
                        ok = false;
                    }
                    __nanosleep(32);
                }
            }
            // before the CTA exits: every tensor-core operation and the last
            // query load complete (immediate on the normal path)
            if (issued) {
                ptx::mma_commit(mdone);
                ptx::mbar_drain(mdone, 0);
            }
            if (q_loaded >= 0) ptx::mbar_drain(qfull, q_loaded & 1);
        }
    } else if (warp >= 2 + kSoftWarps) {
        // ------------------------------------------------------------ gather
        // thread gt: 16-byte chunk c8 of rows r0 and r0 + 32 in every 64-dim
        // block (eight threads read one row's 128 contiguous bytes of a block)
        const int gt = threadIdx.x - (2 + kSoftWarps) * 32;  // 0..255
        const int c8 = gt & 7, r0 = gt >> 3;
        const uint32_t soff = (uint32_t)r0 * 128 + ((c8 ^ (r0 & 7)) << 4);  // same swizzle for r0 + 32
        int gi = 0;
        bool alive = true;
        for (int j = 0; alive && j < nseg; ++j) {
            const SegEntry lv = segtab[j];
            for (int lt = lv.l0; lt < lv.l1; ++lt, ++gi) {
                const int st = gi & 1, r = gi % kRing;
                if (!__all_sync(0xffffffffu, ptx::mbar_wait(rfull + r, (gi / kRing) & 1, abort_flag, d_status))) {
                    alive = false;
                    break;
                }
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
                } else {
                    const uint4* g0 =
                        reinterpret_cast<const uint4*>(latent + (size_t)max(srow[r * TK + r0], 0) * (kMD * 2)) + c8;
                    const uint4* g1 =
                        reinterpret_cast<const uint4*>(latent + (size_t)max(srow[r * TK + r0 + 32], 0) * (kMD * 2)) + c8;
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
                    if (gi >= 2 && !__all_sync(0xffffffffu, ptx::mbar_wait(kempty + 2 * half + st, ((gi >> 1) - 1) & 1,
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
                if (!ok) {
                    alive = false;
                    break;
                }
            }
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
        const int dim = quarter * 32 + lane;                // output: value dim of each 128-dim block
        auto total_l = [&](int h) { return lsum[h] + lsum[kMH + h] + lsum[2 * kMH + h] + lsum[3 * kMH + h]; };
        auto run_max = [&](int h) { return mu[(h >> 5) * 4 * 32 + (h & 31)]; };  // copy of warp sw = 4 (h / 32)
        bool alive = true;
        int gi = 0, sn = 0;
        int n_grow = 0;  // exact-maxima exchanges so far (same count in every softmax warp)
        int n_xch = 0;   // growth-flag exchanges so far
        for (int j = 0; j < nseg; ++j) {
            const int ntl = alive ? segtab[j].l1 - segtab[j].l0 : 0;
            bool have = false;
            if (ntl > 0) {
                if constexpr (FP8) {
                    // the query to f16 in place (its 16-bit elements keep their positions)
                    const bool got = __all_sync(0xffffffffu, ptx::mbar_wait(qfull, sn & 1, abort_flag, d_status));
                    bool over = false;
                    if (got) {
                        uint4* q4 = reinterpret_cast<uint4*>(qs);
                        for (int e = sw * 32 + lane; e < kQBytes / 16; e += kSoftWarps * 32)
                            q4[e] = bf16x8_to_f16x8(q4[e], over);
                    }
                    if (over) report(d_status, DSA_ERR_UNSUPPORTED);
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(qconv);
                }
                my_mu[lane] = -INFINITY;
                {
                    float z[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) z[jj] = 0.f;
                    ptx::tmem_st16(tl + kLCol + hb, z);
                    ptx::tmem_st16(tl + kLCol + hb + 16, z);
                }
                __syncwarp();
                for (int i = 0; i < ntl; ++i, ++gi) {
                    const int st = gi & 1, r = gi % kRing;
                    if (!__all_sync(0xffffffffu,
                                    ptx::mbar_wait(rfull + r, (gi / kRing) & 1, abort_flag, d_status) &&
                                        ptx::mbar_wait(sfull + st, (gi >> 1) & 1, abort_flag, d_status))) {
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
                        float over = -INFINITY;
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {  // 16 heads at a time
                            float sv[16];
                            ptx::tmem_ld16(s_addr + hh * 16, sv);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const float4 m4 = reinterpret_cast<const float4*>(my_mu)[hh * 4 + q];
                                over = fmaxf(over, fmaxf(fmaxf(sv[4 * q] * scale_log2 - m4.x, sv[4 * q + 1] * scale_log2 - m4.y),
                                                         fmaxf(sv[4 * q + 2] * scale_log2 - m4.z, sv[4 * q + 3] * scale_log2 - m4.w)));
                            }
                        }
                        const bool g = __any_sync(0xffffffffu, valid && over > kRescale);
                        const int xb = n_xch & 1;  // flags buffer and barrier of this exchange
                        if (lane == 0) wflag[xb * kSoftWarps + sw] = g ? 1 : 0;
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(xch + xb);
                        if (!__all_sync(0xffffffffu, ptx::mbar_wait(xch + xb, (n_xch >> 1) & 1, abort_flag, d_status))) {
                            alive = false;
                            break;
                        }
                        ++n_xch;
                        int any = 0;
#pragma unroll
                        for (int w = 0; w < kSoftWarps; ++w) any |= wflag[xb * kSoftWarps + w];
                        grow = any != 0;
                    }
                    float alpha = 1.f;  // lane j: rescale factor of head hb + j
                    if (grow) {
                        // exact per-head maxima of this tile (a segment's first tile, or a growth)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {  // 16 heads at a time
                            float sv[16];
                            ptx::tmem_ld16(s_addr + hh * 16, sv);
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) {
                                const float m = ptx::warp_max(valid ? sv[jj] * scale_log2 : -INFINITY);
                                if (lane == hh * 16 + jj) wmax[quarter * kMH + hb + hh * 16 + jj] = m;
                            }
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
                    if (grow && i > 0) {
                        // O^T holds the products of the segment's tiles before this
                        // one once the previous one completes
                        if (!__all_sync(0xffffffffu, ptx::mbar_wait(pvdone, (gi - 1) & 1, abort_flag, d_status))) {
                            alive = false;
                            break;
                        }
                        ptx::tc_fence_after();
#pragma unroll 1
                        for (int cc = 0; cc < 10; ++cc) {  // 4 value blocks x 2 halves of this warp's heads, then the row sums
                            const uint32_t col =
                                cc < 8 ? kOCol + (cc >> 1) * kMH + hb + (cc & 1) * 16 : kLCol + hb + (cc & 1) * 16;
                            float o[16];
                            ptx::tmem_ld16(tl + col, o);
#pragma unroll
                            for (int j = 0; j < 16; ++j) o[j] *= __shfl_sync(0xffffffffu, alpha, (cc & 1) * 16 + j);
                            ptx::tmem_st16(tl + col, o);
                        }
                    }
                    // probabilities, row sums (TMEM), this warp's half of the P^T row over the rope block
                    uint8_t* prow = stage + st * kStage + 8 * kKBlock + key * 128;
#pragma unroll
                    for (int g = 0; g < 2; ++g) {  // 16 heads at a time
                        float sv[16], lvv[16];
                        ptx::tmem_ld16(s_addr + g * 16, sv);
                        ptx::tmem_ld16(tl + kLCol + hb + g * 16, lvv);
                        uint32_t pk[8];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float4 m4 = reinterpret_cast<const float4*>(my_mu)[g * 4 + q];
                            const float mq[4] = {m4.x, m4.y, m4.z, m4.w};
                            float p[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                p[e] = (!valid || mq[e] == -INFINITY) ? 0.f : fast_exp2(sv[4 * q + e] * scale_log2 - mq[e]);
                                lvv[4 * q + e] += p[e];
                            }
                            pk[2 * q] = FP8 ? pack_f16(p[0], p[1]) : pack_bf16(p[0], p[1]);
                            pk[2 * q + 1] = FP8 ? pack_f16(p[2], p[3]) : pack_bf16(p[2], p[3]);
                        }
                        ptx::tmem_st16(tl + kLCol + hb + g * 16, lvv);
                        if (mine) {
#pragma unroll
                            for (int cc = 0; cc < 2; ++cc) {
                                const int col = (hb >> 3) + g * 2 + cc;
                                *reinterpret_cast<uint4*>(prow + ((col ^ (key & 7)) << 4)) =
                                    make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
                            }
                        }
                    }
                    ptx::tc_fence_before();
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::mbar_arrive(sempty + st);
                        ptx::mbar_arrive(pfull + st);
                    }
                }
                // ---- row sums of this warp's 16 keys -> lsum[quarter][hb .. hb+31]
                have = alive;
                if (have) {
                    ptx::tc_fence_after();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {  // 16 heads at a time
                        float lvv[16];
                        ptx::tmem_ld16(tl + kLCol + hb + hh * 16, lvv);
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            float v = lvv[jj];
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);  // lanes 16-31 add zeros
                            if (lane == hh * 16 + jj) lsum[quarter * kMH + hb + hh * 16 + jj] = v;
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(lready);
                if (have) have = __all_sync(0xffffffffu, ptx::mbar_wait(lready, sn & 1, abort_flag, d_status));
                if (have) have = __all_sync(0xffffffffu, ptx::mbar_wait(ofull, sn & 1, abort_flag, d_status));
                if (have) ptx::tc_fence_after();
            }
            // ---- output of the segment: value dim `dim` of each 128-dim block, heads hb .. hb+31
            // lane jj: 1 / (row sum) of head hb + jj, shared by shuffle
            const float my_l = have ? total_l(hb + lane) : 0.f;
            const float my_inv = my_l > 0.f ? 1.f / my_l : 0.f;
            const int sq = segtab[j].q, sflags = segtab[j].flags;
            const bool whole = (sflags & kWhole) != 0;
            const int slot = 2 * c + ((sflags & kFirst) ? 0 : 1);
            if (whole) {
                __nv_bfloat16* ot = out + (int64_t)sq * kMH * kMV;
#pragma unroll 1
                for (int cb = 0; cb < 8; ++cb) {  // 16 columns = heads of one 128-dim block at a time
                    const int db = cb >> 1, h0 = hb + (cb & 1) * 16;
                    float o[16];
                    if (have) ptx::tmem_ld16(tl + kOCol + db * kMH + h0, o);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const float inv = __shfl_sync(0xffffffffu, my_inv, (cb & 1) * 16 + jj);
                        ot[(int64_t)(h0 + jj) * kMV + db * 128 + dim] = __float2bfloat16_rn(have ? o[jj] * inv : 0.f);
                    }
                }
                if (lse && sw == 0) {
                    for (int h = lane; h < kMH; h += 32) {
                        const float L = have ? total_l(h) : 0.f;
                        lse[(int64_t)sq * kMH + h] = L > 0.f ? (run_max(h) + log2f(L)) * 0.69314718055994531f : -INFINITY;
                    }
                }
            } else {
                // a piece of a query cut between CTAs: normalised output + (max, sum)
                float* po = part_o + (int64_t)slot * kMH * kMV;
#pragma unroll 1
                for (int cb = 0; cb < 8; ++cb) {  // 16 columns = heads of one 128-dim block at a time
                    const int db = cb >> 1, h0 = hb + (cb & 1) * 16;
                    float o[16];
                    if (have) ptx::tmem_ld16(tl + kOCol + db * kMH + h0, o);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const float inv = __shfl_sync(0xffffffffu, my_inv, (cb & 1) * 16 + jj);
                        po[(int64_t)(h0 + jj) * kMV + db * 128 + dim] = have ? o[jj] * inv : 0.f;
                    }
                }
                if (sw == 0) {
                    for (int h = lane; h < kMH; h += 32) {
                        float* ml = part_ml + ((int64_t)slot * kMH + h) * 2;
                        const float L = have ? total_l(h) : 0.f;
                        ml[0] = L > 0.f ? run_max(h) : -INFINITY;
                        ml[1] = L;
                    }
                }
            }
            if (ntl > 0) {
                ptx::tc_fence_before();  // this segment's TMEM reads before the release
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(oempty);
                ++sn;
            }
            // every softmax warp has read the shared maxima and sums of this
            // segment before any resets them (one barrier per segment in every
            // warp, on every path)
            ptx::named_sync(1, kSoftWarps * 32);
        }
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
                              int max_ctas) {
    const bool fp8 = latent_dtype == DSA_FP8_DS_MLA;
    const MlaPlan plan = mla_plan(num_q, k, launch_ctas(max_ctas));
    const float scale_log2 = sm_scale * 1.4426950408889634f;
    CUtensorMap qmap;
    cudaError_t e = bf16_map(&qmap, q, (uint64_t)num_q * kMH, 64);
    if (e != cudaSuccess) return e;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(mla_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tcmla::kSmem);
        if (attr == cudaSuccess)
            attr = cudaFuncSetAttribute(mla_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)tcmla::kSmem);
    });
    if (attr != cudaSuccess) return attr;
    auto* part_o = reinterpret_cast<float*>(ws.mla_part);
    e = launch_pdl(fp8 ? mla_tc_kernel<true> : mla_tc_kernel<false>, dim3(plan.G), dim3(tcmla::kThreads), tcmla::kSmem,
                   stream, 1, qmap, reinterpret_cast<const uint8_t*>(latent), s, idx, topk_len, k, scale_log2, plan,
                   reinterpret_cast<__nv_bfloat16*>(out), lse, part_o, ws.mla_ml, d_status);
    if (e != cudaSuccess || !plan_splits(plan)) return e;
    return launch_pdl(mla_combine_kernel, dim3(num_q, kMH / kCombineHeads), dim3(128), 0, stream, 1,
                      (const float*)part_o, (const float*)ws.mla_ml, plan,
                      reinterpret_cast<__nv_bfloat16*>(out), lse);
}

}  // namespace dsa
