// indexer_common.cuh -- pieces shared by the index-score kernels (bf16 and
// e4m3 keys in indexer.cu, NVFP4 keys in indexer_nvfp4.cu): the per-query
// setup of the query preparation, the walk over (sequence, query chunk, key
// tile) work, and the host's tensor-map and SM-count helpers.
#pragma once

#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "tc_ptx.cuh"

namespace dsa {

// 2 pi = kTwoPi1 + kTwoPi2 + kTwoPi3 (within 1e-33 relative); the first two
// have 26 significant bits each
constexpr double kTwoPi1 = 0x1.921fb58p+2;
constexpr double kTwoPi2 = -0x1.dde974p-25;
constexpr double kTwoPi3 = 0x1.1a62633145c07p-52;
constexpr double kInvTwoPi = 0x1.45f306dc9c883p-3;

// Per query, shared by the query preparations: the position check, the SSMax
// factor's sign and |f| w / 64 per head, and cos / sin of the 32 angles.
__device__ __forceinline__ void qprep_setup(const float* __restrict__ w, const float* __restrict__ ss,
                                            const float* __restrict__ sb, const float* __restrict__ inv_freq,
                                            const dsa_seqs& s, int t, float* cs, float* sn, float* sgn, float* wsc,
                                            int* ok, int32_t* d_status) {
    const bool rope = inv_freq != nullptr;
    const int b = seq_of(s.q_start, s.num_seqs, t);
    const int bound = __ldg(s.q_pos + t);                           // causal bound
    const int pos = s.q_rope_pos ? __ldg(s.q_rope_pos + t) : bound;  // SSMax and RoPE position
    if (threadIdx.x == 0) {
        const int ctx = __ldg(s.ctx_len + b);
        *ok = (bound >= 0 && bound < ctx && ctx <= s.max_ctx && pos >= 0);
        if (!*ok) report(d_status, DSA_ERR_BAD_INPUT);
    }
    if (threadIdx.x < 32) {
        const int h = threadIdx.x;
        const float f = fmaf(__ldg(ss + h), logf((float)pos + 1.f), __ldg(sb + h));
        sgn[h] = f < 0.f ? -1.f : 1.f;
        wsc[h] = __ldg(w + (int64_t)t * kIH + h) * fabsf(f) * (1.f / 64.f);
    } else if (threadIdx.x < 64 && rope) {
        const int i = threadIdx.x - 32;  // rotation pair
        // The angle pos * inv_freq is exact in fp64 (a 31-bit integer times a
        // float).  Cody & Waite's reduction by 2 pi, split into two 26-bit
        // parts and an fp64 remainder, keeps that accuracy for |k| < 2^27
        // (k * C1 and k * C2 are exact); cos and sin of the reduced angle in
        // fp32.  Larger angles take the fp64 library sincos.
        const double th = (double)pos * (double)__ldg(inv_freq + i);
        const double kq = rint(th * kInvTwoPi);
        float sf, cf;
        if (fabs(kq) < 134217728.0) {
            double r = fma(-kq, kTwoPi1, th);
            r = fma(-kq, kTwoPi2, r);
            r = fma(-kq, kTwoPi3, r);
            sincosf((float)r, &sf, &cf);
        } else {
            double sd, cd;
            sincos(th, &sd, &cd);
            sf = (float)sd;
            cf = (float)cd;
        }
        cs[i] = cf;
        sn[i] = sf;
    }
    __syncthreads();
}

constexpr int kTileKeys = 128;

struct IdxSeg {
    int b, ctx, q0, nq, maxpos;
    bool ok;
    int64_t base;  // first physical row (contiguous caches)
};

template <int NQ>
__device__ __forceinline__ IdxSeg load_seg(const dsa_seqs& s, int seg, int chunks, int32_t* d_status,
                                           bool report_errors) {
    IdxSeg g;
    g.b = seg / chunks;
    const int c = seg - g.b * chunks;
    g.ctx = __ldg(s.ctx_len + g.b);
    const int qs = __ldg(s.q_start + g.b), qe = __ldg(s.q_start + g.b + 1);
    g.ok = g.ctx >= 0 && g.ctx <= s.max_ctx && qe >= qs && qe - qs <= s.max_q_per_seq;
    g.q0 = qs + c * NQ;
    g.nq = g.ok ? max(0, min(NQ, qe - g.q0)) : 0;
    g.maxpos = -1;
    g.base = s.page_table ? 0 : __ldg(s.seq_base + g.b);
    if (!g.ok && report_errors && c == 0) report(d_status, DSA_ERR_BAD_INPUT);
    for (int i = 0; i < g.nq; ++i) {
        const int p = __ldg(s.q_pos + g.q0 + i);
        if (p >= 0 && p < g.ctx) g.maxpos = max(g.maxpos, p);
    }
    return g;
}

// 0 = nothing to do, 1 = only -inf to write (after every query position), 2 = contract
__device__ __forceinline__ int tile_kind(const IdxSeg& g, int j0) {
    if (!g.ok || g.nq == 0 || j0 >= g.ctx) return 0;
    return j0 > g.maxpos ? 1 : 2;
}

// Walks the CTA's tile range in order (no division per tile); next() returns
// the next tile of kind >= min_kind and skips the rest of a segment once no
// later tile of it can qualify.
template <int NQ>
struct TileWalker {
    int64_t t, t_end;
    int seg, tile, tiles_per_seq, chunks, cur_seg;
    IdxSeg g;
    __device__ TileWalker(int64_t t0, int64_t t1, int tps, int ch)
        : t(t0), t_end(t1), seg((int)(t0 / tps)), tile((int)(t0 - (t0 / tps) * tps)), tiles_per_seq(tps), chunks(ch),
          cur_seg(-1) {}
    __device__ bool next(const dsa_seqs& s, int min_kind, int32_t* d_status, bool report_errors, int& seg_out,
                         int& j0_out, int& kind_out) {
        while (t < t_end) {
            if (seg != cur_seg) {
                g = load_seg<NQ>(s, seg, chunks, d_status, report_errors);
                cur_seg = seg;
            }
            const int j0 = tile * kTileKeys;
            const int kind = tile_kind(g, j0);
            if (kind >= min_kind) {
                seg_out = seg;
                j0_out = j0;
                kind_out = kind;
                ++t;
                if (++tile == tiles_per_seq) {
                    tile = 0;
                    ++seg;
                }
                return true;
            }
            // every later tile of this segment is of this kind or lower
            t += tiles_per_seq - tile;
            tile = 0;
            ++seg;
        }
        return false;
    }
};

// This CTA's contiguous range [*t0, *t1) of the tile space (segment g =
// sequence x query chunk, tile i: index g * tiles_per_seq + i), balanced over
// the tiles that exist -- tile i of segment g when i * 128 < ctx and the chunk
// has queries -- rather than over the space padded to the longest context, so
// that contexts of very different lengths still give every CTA the same work.
// Called by a whole warp (every lane gets the result).
template <int NQ>
__device__ __forceinline__ void balanced_range(const dsa_seqs& s, int chunks, int tiles_per_seq, int64_t* t0,
                                               int64_t* t1) {
    const int lane = threadIdx.x & 31;
    const int nseg = s.num_seqs * chunks;
    auto real = [&](int g) -> int {
        if (g >= nseg) return 0;
        const int b = g / chunks, c = g - b * chunks;
        const int ctx = __ldg(s.ctx_len + b);
        const int nq = __ldg(s.q_start + b + 1) - __ldg(s.q_start + b);
        if (ctx <= 0 || ctx > s.max_ctx || nq <= c * NQ) return 0;
        return (ctx + kTileKeys - 1) / kTileKeys;
    };
    // the first 128 segments' counts are loaded together and kept; the rest
    // (more than 128 segments) are recomputed on the second walk
    constexpr int kKept = 4;
    int kept[kKept];
#pragma unroll
    for (int i = 0; i < kKept; ++i) kept[i] = real(32 * i + lane);
    auto count = [&](int g0) -> int {
        int v = g0 >= 32 * kKept ? real(g0 + lane) : 0;
#pragma unroll
        for (int i = 0; i < kKept; ++i)
            if (g0 == 32 * i) v = kept[i];
        return v;
    };
    int64_t total = 0;
    for (int g0 = 0; g0 < nseg; g0 += 32) {
        int v = count(g0);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        total += v;
    }
    const int64_t r0 = total * blockIdx.x / gridDim.x, r1 = total * (blockIdx.x + 1) / gridDim.x;
    // full-space index of compact index r (r == total: the end of the space)
    int64_t f0 = (int64_t)nseg * tiles_per_seq, f1 = f0;
    int64_t before = 0;  // real tiles of the segments before this group of 32
    for (int g0 = 0; g0 < nseg && before <= r1; g0 += 32) {
        const int v = count(g0);
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int64_t lo = before + incl - v, hi = before + incl;  // this lane's segment: [lo, hi)
        const uint32_t h0 = __ballot_sync(0xffffffffu, v > 0 && r0 >= lo && r0 < hi);
        const uint32_t h1 = __ballot_sync(0xffffffffu, v > 0 && r1 >= lo && r1 < hi);
        if (h0 && f0 == (int64_t)nseg * tiles_per_seq) {
            const int l = __ffs(h0) - 1;
            const int64_t off = r0 - __shfl_sync(0xffffffffu, lo, l);
            f0 = (int64_t)(g0 + l) * tiles_per_seq + off;
        }
        if (h1 && f1 == (int64_t)nseg * tiles_per_seq) {
            const int l = __ffs(h1) - 1;
            const int64_t off = r1 - __shfl_sync(0xffffffffu, lo, l);
            f1 = (int64_t)(g0 + l) * tiles_per_seq + off;
        }
        before += __shfl_sync(0xffffffffu, incl, 31);
    }
    *t0 = r0 < r1 ? f0 : 0;
    *t1 = r0 < r1 ? f1 : 0;
}

// ---------------------------------------------------------------------------
// host side
inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
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

inline cudaError_t make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    auto enc = tmap_encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

inline int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

}  // namespace dsa
