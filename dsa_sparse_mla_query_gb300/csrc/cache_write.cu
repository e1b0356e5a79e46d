// cache_write.cu -- the kernels on either side of the decode path (sm_103a):
// new tokens into the indexer-key and latent caches, and the attention query's
// RoPE + SSMax.
//
// Definitions ([colibri] "Mistral-Large-4 (c/colibri.c)", What differs from
// GLM-5.2: The indexer (k = LayerNorm(wk(x)), rotated on its first 64 dims on
// RoPE layers), SSMax, RoPE and the rest; "Day 0 support for Mistral Large 4",
// Model architecture (KV LoRA rank 512, RoPE dim 64), Implementation details
// (the indexer K path written straight into the FP8 cache; MLA RoPE + SSMax),
// DSA indexer on AITER (one FP8 scale per key, 132 bytes per token)).
//
// All three are HBM-bound elementwise passes: one warp per token (or per query
// head), lanes over contiguous dims, so every load and store is coalesced and
// the per-row reductions (LayerNorm moments, the quantisation maxima) are warp
// shuffles.  Storage rounding is to nearest even: bf16 by __float2bfloat16_rn,
// e4m3 by the saturating conversion of value / scale with scale = amax / 448.
#include <cuda_fp8.h>

#include <algorithm>
#include <mutex>

#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr float kTwoPi1 = 0x1.921fb6p+2f;  // 2 pi = kTwoPi1 + kTwoPi2 + kTwoPi3, fp32 parts
constexpr float kTwoPi2 = -0x1.777a5cp-23f;
constexpr float kTwoPi3 = -0x1.ee59dap-48f;
constexpr float kInvTwoPiF = 0x1.45f306p-3f;
constexpr double kTwoPiHi = 0x1.921fb58p+2;  // 2 pi = hi + mid + lo, the first two 26 bits each
constexpr double kTwoPiMid = -0x1.dde974p-25;
constexpr double kTwoPiLo = 0x1.1a62633145c07p-52;
constexpr double kInvTwoPiD = 0x1.45f306dc9c883p-3;

// cos and sin of pos * inv_freq, reduced by 2 pi the Cody & Waite way.  Below
// 2^24 (position and angle) the angle is held exactly as hi + lo, the fp32
// product and its FMA residual, and reduced with a three-part fp32 2 pi: the
// first step is exact (|hi - k c1| < 8 and both are multiples of 2^-21), so the
// reduced angle is off by under 3e-7.  Larger angles are reduced in fp64, which
// runs at a small fraction of the fp32 rate on this part.
__device__ __forceinline__ void rope_cs(int pos, float inv_freq, float& c, float& s) {
    const float pf = (float)pos;
    const float hi = pf * inv_freq;
    if (pos < (1 << 24) && fabsf(hi) < 16777216.f) {
        const float lo = fmaf(pf, inv_freq, -hi);
        const float k = rintf(hi * kInvTwoPiF);
        float r = fmaf(-k, kTwoPi1, hi);
        r = fmaf(-k, kTwoPi2, r);
        r = fmaf(-k, kTwoPi3, r) + lo;
        sincosf(r, &s, &c);
        return;
    }
    const double th = (double)pos * (double)inv_freq;
    const double kq = rint(th * kInvTwoPiD);
    if (fabs(kq) < 134217728.0) {
        double r = fma(-kq, kTwoPiHi, th);
        r = fma(-kq, kTwoPiMid, r);
        r = fma(-kq, kTwoPiLo, r);
        sincosf((float)r, &s, &c);
    } else {
        double sd, cd;
        sincos(th, &sd, &cd);
        s = (float)sd;
        c = (float)cd;
    }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// the physical row of a new token, or -1 (skipped: a negative slot; reported:
// a slot past the cache or a negative position)
__device__ __forceinline__ int64_t insert_row(int64_t r, int p, int64_t num_rows, int32_t* d_status) {
    if (r < 0) return -1;
    if (r >= num_rows || p < 0) {
        if ((threadIdx.x & 31) == 0) report(d_status, DSA_ERR_BAD_INPUT);
        return -1;
    }
    return r;
}

// A warp takes one token at a time (one query head for the query kernel);
// the token kernels walk the tokens with a grid stride and load kUnroll tokens
// before working on any, so a warp keeps that many rows of loads in flight.
constexpr int kWarpsPerCta = 4;
constexpr int kUnroll = 2;

// ---------------------------------------------------------------------------
// indexer key: LayerNorm over the 128 dims (biased variance), RoPE on dims
// 0..63, then bf16 or e4m3 with one fp32 scale per row.  Eight lanes per key,
// four keys per warp: lane j of a group holds dims 8j..8j+7 (RoPE pairs
// 4j..4j+3) and 64+8j..64+8j+7, so each load covers 128 contiguous bytes of a
// key and every lane has the same RoPE work.
constexpr int kKeyLanes = 8;
constexpr int kKeysPerWarp = 32 / kKeyLanes;

__device__ __forceinline__ float group_sum8(float x) {
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ void unpack_bf16x8(uint4 w, float* v) {
    v[0] = bf16_lo(w.x), v[1] = bf16_hi(w.x), v[2] = bf16_lo(w.y), v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z), v[5] = bf16_hi(w.z), v[6] = bf16_lo(w.w), v[7] = bf16_hi(w.w);
}

// row < 0: the group's reductions only, nothing stored
template <bool FP8>
__device__ __forceinline__ void index_k_row(uint4 ra, uint4 rb, int p, int64_t row, const float* __restrict__ sg,
                                            const float* __restrict__ sb, float eps,
                                            const float* __restrict__ inv_freq, void* __restrict__ cache,
                                            float* __restrict__ k_scale, int j) {
    float v[16];  // dims 8j..8j+7, then 64+8j..64+8j+7
    unpack_bf16x8(ra, v);
    unpack_bf16x8(rb, v + 8);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc += v[i];
    const float mean = group_sum8(acc) * (1.f / kID);
    float d2 = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) d2 = fmaf(v[i] - mean, v[i] - mean, d2);
    const float inv = 1.f / sqrtf(group_sum8(d2) * (1.f / kID) + eps);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float4* g4 = reinterpret_cast<const float4*>(sg + 64 * h + 8 * j);
        const float4* b4 = reinterpret_cast<const float4*>(sb + 64 * h + 8 * j);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float4 g = g4[q], b = b4[q];
            float* w = v + 8 * h + 4 * q;
            w[0] = fmaf((w[0] - mean) * inv, g.x, b.x);
            w[1] = fmaf((w[1] - mean) * inv, g.y, b.y);
            w[2] = fmaf((w[2] - mean) * inv, g.z, b.z);
            w[3] = fmaf((w[3] - mean) * inv, g.w, b.w);
        }
    }
    if (inv_freq) {
        const float4 f4 = __ldg(reinterpret_cast<const float4*>(inv_freq) + j);  // pairs 4j..4j+3
        const float fr[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float c, s;
            rope_cs(p, fr[u], c, s);
            const float x0 = v[2 * u], x1 = v[2 * u + 1];
            v[2 * u] = fmaf(x0, c, -x1 * s);
            v[2 * u + 1] = fmaf(x0, s, x1 * c);
        }
    }
    if (FP8) {
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (row < 0) return;  // after the group's shuffles
        const float scale = m > 0.f ? m / 448.f : 1.f;
        const float rs = 1.f / scale;
        uint2* dst = reinterpret_cast<uint2*>(static_cast<uint8_t*>(cache) + row * kID);
        dst[j] = make_uint2(pack_e4m3x4(v[0] * rs, v[1] * rs, v[2] * rs, v[3] * rs),
                            pack_e4m3x4(v[4] * rs, v[5] * rs, v[6] * rs, v[7] * rs));
        dst[8 + j] = make_uint2(pack_e4m3x4(v[8] * rs, v[9] * rs, v[10] * rs, v[11] * rs),
                                pack_e4m3x4(v[12] * rs, v[13] * rs, v[14] * rs, v[15] * rs));
        if (j == 0) k_scale[row] = scale;
    } else {
        if (row < 0) return;
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(cache) + row * kID);
        dst[j] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                            pack_bf16x2(v[6], v[7]));
        dst[8 + j] = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]), pack_bf16x2(v[12], v[13]),
                                pack_bf16x2(v[14], v[15]));
    }
}

template <bool FP8>
__global__ void __launch_bounds__(128) index_k_insert_kernel(const __nv_bfloat16* __restrict__ x,
                                                             const float* __restrict__ gamma,
                                                             const float* __restrict__ beta, float eps,
                                                             const int32_t* __restrict__ pos,
                                                             const float* __restrict__ inv_freq,
                                                             const int64_t* __restrict__ slot, int32_t n,
                                                             void* __restrict__ cache, float* __restrict__ k_scale,
                                                             int64_t num_rows, int32_t* d_status) {
    static_assert(kID == 32 * kWarpsPerCta, "one gamma and beta value per thread");
    __shared__ __align__(16) float sg[kID], sb[kID];
    pdl_enter();
    sg[threadIdx.x] = gamma[threadIdx.x];
    sb[threadIdx.x] = beta[threadIdx.x];
    __syncthreads();
    const int j = threadIdx.x & (kKeyLanes - 1);
    // key groups: kKeysPerWarp consecutive keys, one per warp at a time
    const int64_t groups = ((int64_t)n + kKeysPerWarp - 1) / kKeysPerWarp;
    const int64_t stride = (int64_t)gridDim.x * kWarpsPerCta;
    const int sub = (threadIdx.x & 31) / kKeyLanes;
    for (int64_t g0 = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5); g0 < groups; g0 += kUnroll * stride) {
        int64_t r[kUnroll];
        int p[kUnroll];
        uint4 ra[kUnroll], rb[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t t = (g0 + u * stride) * kKeysPerWarp + sub;
            r[u] = -1;
            p[u] = 0;
            ra[u] = rb[u] = make_uint4(0u, 0u, 0u, 0u);
            if (t < n) {
                r[u] = __ldg(slot + t);
                p[u] = __ldg(pos + t);
                const uint4* src = reinterpret_cast<const uint4*>(x + t * kID);
                ra[u] = __ldcs(src + j);
                rb[u] = __ldcs(src + 8 + j);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            // every lane takes part in the group reductions; only valid rows are stored
            const bool live = r[u] >= 0 && r[u] < num_rows && p[u] >= 0;
            if (r[u] >= num_rows || (r[u] >= 0 && p[u] < 0)) {
                if (j == 0) report(d_status, DSA_ERR_BAD_INPUT);
            }
            index_k_row<FP8>(ra[u], rb[u], p[u], live ? r[u] : -1, sg, sb, eps, inv_freq, cache, k_scale, j);
        }
    }
}

// ---------------------------------------------------------------------------
// latent row: the 512 latent dims copied (bf16) or e4m3 with one fp32 scale per
// 128 (fp8_ds_mla: [0,512) codes, [512,528) four scales, [528,656) the RoPE dims
// bf16), the 64 RoPE dims rotated.  Lane l: latent dims 16l..16l+15 (group l / 8)
// and RoPE pair l.
template <bool FP8>
__device__ __forceinline__ void latent_row(uint4 r0, uint4 r1, uint32_t pe, int p, int64_t row,
                                           const float* __restrict__ inv_freq, uint8_t* __restrict__ latent,
                                           int lane) {
    float x0 = bf16_lo(pe), x1 = bf16_hi(pe);
    if (inv_freq) {
        float c, s;
        rope_cs(p, __ldg(inv_freq + lane), c, s);
        const float y0 = fmaf(x0, c, -x1 * s), y1 = fmaf(x0, s, x1 * c);
        x0 = y0;
        x1 = y1;
    }
    if (FP8) {
        uint8_t* dst = latent + row * kDsRow;
        const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        float v[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = bf16_lo(w[i]);
            v[2 * i + 1] = bf16_hi(w[i]);
        }
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));  // within 8 lanes
        const float scale = m > 0.f ? m / 448.f : 1.f;
        const float rs = 1.f / scale;
        uint4 codes;
        codes.x = pack_e4m3x4(v[0] * rs, v[1] * rs, v[2] * rs, v[3] * rs);
        codes.y = pack_e4m3x4(v[4] * rs, v[5] * rs, v[6] * rs, v[7] * rs);
        codes.z = pack_e4m3x4(v[8] * rs, v[9] * rs, v[10] * rs, v[11] * rs);
        codes.w = pack_e4m3x4(v[12] * rs, v[13] * rs, v[14] * rs, v[15] * rs);
        reinterpret_cast<uint4*>(dst)[lane] = codes;
        if ((lane & 7) == 0) reinterpret_cast<float*>(dst + kMV)[lane >> 3] = scale;
        reinterpret_cast<uint32_t*>(dst + kMV + 16)[lane] = pack_bf16x2(x0, x1);
    } else {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(latent) + row * kMD;
        uint4* d4 = reinterpret_cast<uint4*>(dst + 16 * lane);
        d4[0] = r0;
        d4[1] = r1;
        reinterpret_cast<uint32_t*>(dst + kMV)[lane] = pack_bf16x2(x0, x1);
    }
}

template <bool FP8>
__global__ void __launch_bounds__(128) latent_insert_kernel(const __nv_bfloat16* __restrict__ c_kv,
                                                            const __nv_bfloat16* __restrict__ k_pe,
                                                            const int32_t* __restrict__ pos,
                                                            const float* __restrict__ inv_freq,
                                                            const int64_t* __restrict__ slot, int32_t n,
                                                            uint8_t* __restrict__ latent, int64_t num_rows,
                                                            int32_t* d_status) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int64_t stride = (int64_t)gridDim.x * kWarpsPerCta;
    for (int64_t t0 = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5); t0 < n; t0 += kUnroll * stride) {
        int64_t r[kUnroll];
        int p[kUnroll];
        uint4 r0[kUnroll], r1[kUnroll];
        uint32_t pe[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t t = t0 + u * stride;
            r[u] = -1;
            p[u] = 0;
            r0[u] = r1[u] = make_uint4(0u, 0u, 0u, 0u);
            pe[u] = 0u;
            if (t < n) {
                r[u] = __ldg(slot + t);
                p[u] = __ldg(pos + t);
                const uint4* src = reinterpret_cast<const uint4*>(c_kv + t * kMV + 16 * lane);
                r0[u] = __ldcs(src);
                r1[u] = __ldcs(src + 1);
                pe[u] = __ldcs(reinterpret_cast<const unsigned int*>(k_pe + t * (kMD - kMV)) + lane);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t row = insert_row(r[u], p[u], num_rows, d_status);
            if (row >= 0) latent_row<FP8>(r0[u], r1[u], pe[u], p[u], row, inv_freq, latent, lane);
        }
    }
}

// ---------------------------------------------------------------------------
// attention query: RoPE on dims 512..575, then every dim of head h times
// f_h = s_h ln(pos+1) + b_h.  One warp per (query, head); lane l: dims
// 16l..16l+15 and RoPE pair l.
__global__ void __launch_bounds__(128) mla_q_prep_kernel(const __nv_bfloat16* __restrict__ q,
                                                         const float* __restrict__ ss, const float* __restrict__ sb,
                                                         const float* __restrict__ inv_freq,
                                                         const int32_t* __restrict__ q_pos, int32_t num_q,
                                                         __nv_bfloat16* __restrict__ q_out, int32_t* d_status) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int64_t wi = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);  // (query, head)
    if (wi >= (int64_t)num_q * kMH) return;
    const int64_t t = wi / kMH;
    const int h = (int)(wi - t * kMH);
    const int p = __ldg(q_pos + t);
    if (p < 0) {
        if (lane == 0) report(d_status, DSA_ERR_BAD_INPUT);
        return;
    }
    const float f = fmaf(__ldg(ss + h), logf((float)p + 1.f), __ldg(sb + h));
    const __nv_bfloat16* qi = q + wi * kMD;
    __nv_bfloat16* qo = q_out + wi * kMD;
    const uint4* src = reinterpret_cast<const uint4*>(qi + 16 * lane);
    uint4 r[2] = {src[0], src[1]};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        uint32_t* w = reinterpret_cast<uint32_t*>(&r[k]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            w[i] = pack_bf16x2(bf16_lo(w[i]) * f, bf16_hi(w[i]) * f);
        }
    }
    uint4* d4 = reinterpret_cast<uint4*>(qo + 16 * lane);
    d4[0] = r[0];
    d4[1] = r[1];
    const uint32_t pe = reinterpret_cast<const uint32_t*>(qi + kMV)[lane];
    float x0 = bf16_lo(pe), x1 = bf16_hi(pe);
    if (inv_freq) {
        float c, s;
        rope_cs(p, __ldg(inv_freq + lane), c, s);
        const float y0 = fmaf(x0, c, -x1 * s), y1 = fmaf(x0, s, x1 * c);
        x0 = y0;
        x1 = y1;
    }
    reinterpret_cast<uint32_t*>(qo + kMV)[lane] = pack_bf16x2(x0 * f, x1 * f);
}

constexpr int kTokensPerCta = kWarpsPerCta;

// a grid of a few waves of CTAs (16 per SM) walking the items (keys in groups
// of kKeysPerWarp, latent rows, query heads), one per warp at a time
unsigned insert_grid(int64_t items) {
    static int sms = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
            sms = n;
        else
            sms = 148;
    });
    const int64_t need = (items + kTokensPerCta - 1) / kTokensPerCta;
    return (unsigned)std::min<int64_t>(need, (int64_t)sms * 16);
}

}  // namespace

cudaError_t launch_index_k_insert(const void* x, const float* gamma, const float* beta, float eps, const int32_t* pos,
                                  const float* inv_freq, const int64_t* slot, int32_t n, void* cache, float* k_scale,
                                  bool fp8, int64_t num_rows, int32_t* d_status, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const dim3 grid(insert_grid(((int64_t)n + kKeysPerWarp - 1) / kKeysPerWarp));
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    return fp8 ? launch_pdl(index_k_insert_kernel<true>, grid, dim3(128), 0, stream, 1, xb, gamma, beta, eps, pos,
                            inv_freq, slot, n, cache, k_scale, num_rows, d_status)
               : launch_pdl(index_k_insert_kernel<false>, grid, dim3(128), 0, stream, 1, xb, gamma, beta, eps, pos,
                            inv_freq, slot, n, cache, k_scale, num_rows, d_status);
}

cudaError_t launch_latent_insert(const void* c_kv, const void* k_pe, const int32_t* pos, const float* inv_freq,
                                 const int64_t* slot, int32_t n, void* latent, bool fp8, int64_t num_rows,
                                 int32_t* d_status, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const dim3 grid(insert_grid(n));
    const __nv_bfloat16* cb = static_cast<const __nv_bfloat16*>(c_kv);
    const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(k_pe);
    uint8_t* out = static_cast<uint8_t*>(latent);
    return fp8 ? launch_pdl(latent_insert_kernel<true>, grid, dim3(128), 0, stream, 1, cb, kb, pos, inv_freq, slot, n,
                            out, num_rows, d_status)
               : launch_pdl(latent_insert_kernel<false>, grid, dim3(128), 0, stream, 1, cb, kb, pos, inv_freq, slot, n,
                            out, num_rows, d_status);
}

cudaError_t launch_mla_q_prep(const void* q, const float* ssmax_s, const float* ssmax_b, const float* inv_freq,
                              const int32_t* q_pos, int32_t num_q, void* q_out, int32_t* d_status,
                              cudaStream_t stream) {
    if (num_q <= 0) return cudaSuccess;
    const dim3 grid((unsigned)(((int64_t)num_q * kMH + kTokensPerCta - 1) / kTokensPerCta));
    return launch_pdl(mla_q_prep_kernel, grid, dim3(128), 0, stream, 1, static_cast<const __nv_bfloat16*>(q), ssmax_s,
                      ssmax_b, inv_freq, q_pos, num_q, static_cast<__nv_bfloat16*>(q_out), d_status);
}

}  // namespace dsa
