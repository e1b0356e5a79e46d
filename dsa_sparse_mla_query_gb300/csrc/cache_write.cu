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

#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr double kTwoPiHi = 0x1.921fb58p+2;  // 2 pi = hi + mid + lo, the first two 26 bits each
constexpr double kTwoPiMid = -0x1.dde974p-25;
constexpr double kTwoPiLo = 0x1.1a62633145c07p-52;
constexpr double kInvTwoPiD = 0x1.45f306dc9c883p-3;

// cos and sin of pos * inv_freq: the angle exact in fp64, reduced by 2 pi
// (Cody & Waite, exact for |k| < 2^27), then fp32 sincos
__device__ __forceinline__ void rope_cs(int pos, float inv_freq, float& c, float& s) {
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

// the physical row of new token t, or -1 (skipped: a negative slot; reported: a
// slot past the cache or a negative position)
__device__ __forceinline__ int64_t insert_row(const int64_t* slot, const int32_t* pos, int64_t t, int64_t num_rows,
                                              int32_t* d_status) {
    const int64_t r = __ldg(slot + t);
    if (r < 0) return -1;
    if (r >= num_rows || __ldg(pos + t) < 0) {
        if ((threadIdx.x & 31) == 0) report(d_status, DSA_ERR_BAD_INPUT);
        return -1;
    }
    return r;
}

// ---------------------------------------------------------------------------
// indexer key: LayerNorm over the 128 dims (biased variance), RoPE on dims
// 0..63, then bf16 or e4m3 with one fp32 scale per row.  Lane l: dims 4l..4l+3.
template <bool FP8>
__global__ void __launch_bounds__(128) index_k_insert_kernel(const __nv_bfloat16* __restrict__ x,
                                                             const float* __restrict__ gamma,
                                                             const float* __restrict__ beta, float eps,
                                                             const int32_t* __restrict__ pos,
                                                             const float* __restrict__ inv_freq,
                                                             const int64_t* __restrict__ slot, int32_t n,
                                                             void* __restrict__ cache, float* __restrict__ k_scale,
                                                             int64_t num_rows, int32_t* d_status) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    for (int64_t t = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5); t < n; t += (int64_t)gridDim.x * 4) {
    const int64_t row = insert_row(slot, pos, t, num_rows, d_status);
    if (row < 0) continue;
    const uint2 raw = *reinterpret_cast<const uint2*>(x + t * kID + 4 * lane);
    const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(&raw);
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __bfloat162float(xb[i]);
    const float mean = warp_sum((v[0] + v[1]) + (v[2] + v[3])) * (1.f / kID);
    float d2 = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) d2 = fmaf(v[i] - mean, v[i] - mean, d2);
    const float inv = 1.f / sqrtf(warp_sum(d2) * (1.f / kID) + eps);
    const float4 g = *reinterpret_cast<const float4*>(gamma + 4 * lane);
    const float4 b = *reinterpret_cast<const float4*>(beta + 4 * lane);
    const float gv[4] = {g.x, g.y, g.z, g.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = fmaf((v[i] - mean) * inv, gv[i], bv[i]);
    if (inv_freq && lane < 16) {  // pairs 2 lane and 2 lane + 1
        const int p = __ldg(pos + t);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            float c, s;
            rope_cs(p, __ldg(inv_freq + 2 * lane + u), c, s);
            const float x0 = v[2 * u], x1 = v[2 * u + 1];
            v[2 * u] = fmaf(x0, c, -x1 * s);
            v[2 * u + 1] = fmaf(x0, s, x1 * c);
        }
    }
    if (FP8) {
        float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float scale = m > 0.f ? m / 448.f : 1.f;
        reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(cache) + row * kID)[lane] =
            pack_e4m3x4(v[0] / scale, v[1] / scale, v[2] / scale, v[3] / scale);
        if (lane == 0) k_scale[row] = scale;
    } else {
        reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(cache) + row * kID)[lane] =
            make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
    }
    }
}

// ---------------------------------------------------------------------------
// latent row: the 512 latent dims copied (bf16) or e4m3 with one fp32 scale per
// 128 (fp8_ds_mla: [0,512) codes, [512,528) four scales, [528,656) the RoPE dims
// bf16), the 64 RoPE dims rotated.  Lane l: latent dims 16l..16l+15 (group l / 8)
// and RoPE pair l.
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
    for (int64_t t = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5); t < n; t += (int64_t)gridDim.x * 4) {
    const int64_t row = insert_row(slot, pos, t, num_rows, d_status);
    if (row < 0) continue;
    const uint4* src = reinterpret_cast<const uint4*>(c_kv + t * kMV + 16 * lane);
    const uint4 r0 = src[0], r1 = src[1];
    // the RoPE pair of this lane
    const uint32_t pe = reinterpret_cast<const uint32_t*>(k_pe + t * (kMD - kMV))[lane];
    float x0 = __bfloat162float(__ushort_as_bfloat16((unsigned short)(pe & 0xFFFF)));
    float x1 = __bfloat162float(__ushort_as_bfloat16((unsigned short)(pe >> 16)));
    if (inv_freq) {
        float c, s;
        rope_cs(__ldg(pos + t), __ldg(inv_freq + lane), c, s);
        const float y0 = fmaf(x0, c, -x1 * s), y1 = fmaf(x0, s, x1 * c);
        x0 = y0;
        x1 = y1;
    }
    if (FP8) {
        uint8_t* dst = latent + row * kDsRow;
        float v[16];
        const __nv_bfloat16* b0 = reinterpret_cast<const __nv_bfloat16*>(&r0);
        const __nv_bfloat16* b1 = reinterpret_cast<const __nv_bfloat16*>(&r1);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[i] = __bfloat162float(b0[i]);
            v[8 + i] = __bfloat162float(b1[i]);
        }
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));  // within 8 lanes
        const float scale = m > 0.f ? m / 448.f : 1.f;
        uint4 codes;
        codes.x = pack_e4m3x4(v[0] / scale, v[1] / scale, v[2] / scale, v[3] / scale);
        codes.y = pack_e4m3x4(v[4] / scale, v[5] / scale, v[6] / scale, v[7] / scale);
        codes.z = pack_e4m3x4(v[8] / scale, v[9] / scale, v[10] / scale, v[11] / scale);
        codes.w = pack_e4m3x4(v[12] / scale, v[13] / scale, v[14] / scale, v[15] / scale);
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
            const float a = __bfloat162float(__ushort_as_bfloat16((unsigned short)(w[i] & 0xFFFF)));
            const float b = __bfloat162float(__ushort_as_bfloat16((unsigned short)(w[i] >> 16)));
            w[i] = pack_bf16x2(a * f, b * f);
        }
    }
    uint4* d4 = reinterpret_cast<uint4*>(qo + 16 * lane);
    d4[0] = r[0];
    d4[1] = r[1];
    const uint32_t pe = reinterpret_cast<const uint32_t*>(qi + kMV)[lane];
    float x0 = __bfloat162float(__ushort_as_bfloat16((unsigned short)(pe & 0xFFFF)));
    float x1 = __bfloat162float(__ushort_as_bfloat16((unsigned short)(pe >> 16)));
    if (inv_freq) {
        float c, s;
        rope_cs(p, __ldg(inv_freq + lane), c, s);
        const float y0 = fmaf(x0, c, -x1 * s), y1 = fmaf(x0, s, x1 * c);
        x0 = y0;
        x1 = y1;
    }
    reinterpret_cast<uint32_t*>(qo + kMV)[lane] = pack_bf16x2(x0 * f, x1 * f);
}

constexpr int kTokensPerCta = 4;  // a warp per token

// a grid of a few waves of CTAs (16 per SM) walking the tokens
unsigned insert_grid(int64_t items) {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                       cudaSuccess || sms <= 0)
            sms = 148;
    }
    const int64_t need = (items + kTokensPerCta - 1) / kTokensPerCta;
    return (unsigned)std::min<int64_t>(need, (int64_t)sms * 16);
}

}  // namespace

cudaError_t launch_index_k_insert(const void* x, const float* gamma, const float* beta, float eps, const int32_t* pos,
                                  const float* inv_freq, const int64_t* slot, int32_t n, void* cache, float* k_scale,
                                  bool fp8, int64_t num_rows, int32_t* d_status, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const dim3 grid(insert_grid(n));
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
