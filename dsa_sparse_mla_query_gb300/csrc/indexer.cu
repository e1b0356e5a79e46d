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
//   rotated dims (angle and rotation in fp64) are split into hi + lo 16-bit
//   parts, so the contraction runs over K = 192 columns [hi | lo | unrotated]
//   against key dims [0..63 | 0..63 | 64..127] and reproduces the fp64 query to
//   ~2^-17 relative.  That keeps the top-k boundary exact (see dsa_topk).
//   e4m3 keys decode exactly to f16, so the fp8 path runs the same contraction
//   in f16 and multiplies the per-row scale after the relu-weighted sum
//   (scale >= 0).
#include "dsa_internal.cuh"

namespace dsa {

// ---------------------------------------------------------------------------
// query preparation: q' [Q, 32, KP] (KP = 192 RoPE, 128 NoPE), w' [Q, 32]
template <typename T>
__device__ __forceinline__ T from_double(double x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_double<__nv_bfloat16>(double x) { return __double2bfloat16(x); }
template <>
__device__ __forceinline__ __half from_double<__half>(double x) { return __double2half(x); }
template <typename T>
__device__ __forceinline__ double to_double(T x);
template <>
__device__ __forceinline__ double to_double<__nv_bfloat16>(__nv_bfloat16 x) { return (double)__bfloat162float(x); }
template <>
__device__ __forceinline__ double to_double<__half>(__half x) { return (double)__half2float(x); }

template <typename T>
__global__ void __launch_bounds__(128) qprep_kernel(const __nv_bfloat16* __restrict__ q, const float* __restrict__ w,
                                                    const float* __restrict__ ss, const float* __restrict__ sb,
                                                    const float* __restrict__ inv_freq, dsa_seqs s, int num_q,
                                                    T* __restrict__ qp, float* __restrict__ wp,
                                                    int32_t* d_status) {
    const int t = blockIdx.x;
    const bool rope = inv_freq != nullptr;
    const int KP = rope ? 192 : 128;
    __shared__ double cs[32], sn[32];
    __shared__ double sgn[32];
    __shared__ int ok;
    const int b = seq_of(s.q_start, s.num_seqs, t);
    const int pos = __ldg(s.q_pos + t);
    if (threadIdx.x == 0) {
        const int ctx = __ldg(s.ctx_len + b);
        ok = (pos >= 0 && pos < ctx && ctx <= s.max_ctx);
        if (!ok) report(d_status, DSA_ERR_BAD_INPUT);
    }
    if (threadIdx.x < 32) {
        const int h = threadIdx.x;
        double f = (double)__ldg(ss + h) * log((double)pos + 1.0) + (double)__ldg(sb + h);
        sgn[h] = f < 0.0 ? -1.0 : 1.0;
        wp[(int64_t)t * kIH + h] = (float)((double)__ldg(w + (int64_t)t * kIH + h) * fabs(f) / 64.0);
        if (rope) {
            double th = (double)pos * (double)__ldg(inv_freq + h);
            sincos(th, &sn[h], &cs[h]);
        }
    }
    __syncthreads();
    const __nv_bfloat16* qt = q + (int64_t)t * kIH * kID;
    T* out = qp + (int64_t)t * kIH * KP;
    for (int e = threadIdx.x; e < kIH * 64; e += blockDim.x) {
        const int h = e >> 6, p = e & 63;  // pair p = dims (2p, 2p+1)
        double x0 = (double)__bfloat162float(qt[h * kID + 2 * p]);
        double x1 = (double)__bfloat162float(qt[h * kID + 2 * p + 1]);
        const double g = ok ? sgn[h] : 0.0;
        T* o = out + h * KP;
        if (rope && p < 32) {
            double y0 = g * (x0 * cs[p] - x1 * sn[p]);
            double y1 = g * (x0 * sn[p] + x1 * cs[p]);
            T h0 = from_double<T>(y0), h1 = from_double<T>(y1);
            o[2 * p] = h0;
            o[2 * p + 1] = h1;
            o[64 + 2 * p] = from_double<T>(y0 - to_double<T>(h0));
            o[64 + 2 * p + 1] = from_double<T>(y1 - to_double<T>(h1));
        } else {
            const int col = rope ? 64 + 2 * p : 2 * p;
            o[col] = from_double<T>(g * x0);
            o[col + 1] = from_double<T>(g * x1);
        }
    }
}

// ---------------------------------------------------------------------------
// scores: one CTA = 128 keys of one sequence x NQ queries of that sequence.
// 8 warps, warp w owns keys 16w..16w+15 (the MMA M rows); N = NQ*32 heads.
constexpr int kTileKeys = 128;
constexpr int kKeyStride = kID + 8;  // 16-bit elements per key row in smem (pad: no ldmatrix bank conflicts)

template <int NQ, int KP>
struct IdxSmem {
    static constexpr int kQStride = KP + 8;
    static constexpr size_t q_bytes = (size_t)NQ * kIH * kQStride * 2;
    static constexpr size_t k_bytes = (size_t)kTileKeys * kKeyStride * 2;
    static constexpr size_t raw_bytes = (size_t)kTileKeys * kID;  // e4m3 staging
    static constexpr size_t out_bytes = (size_t)NQ * kTileKeys * 4;
    static constexpr size_t total = q_bytes + k_bytes + raw_bytes + out_bytes + NQ * kIH * 4 + kTileKeys * 4 + 64;
};

template <int NQ, int KP, bool FP8>
__global__ void __launch_bounds__(256) index_scores_kernel(const uint16_t* __restrict__ qp,
                                                           const float* __restrict__ wp,
                                                           const void* __restrict__ k_idx,
                                                           const float* __restrict__ k_scale, dsa_seqs s,
                                                           float* __restrict__ scores, int64_t ld,
                                                           int32_t* d_status) {
    using L = IdxSmem<NQ, KP>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint16_t* sq = reinterpret_cast<uint16_t*>(smem);
    uint16_t* sk = reinterpret_cast<uint16_t*>(smem + L::q_bytes);
    uint8_t* sraw = smem + L::q_bytes + L::k_bytes;
    float* sout = reinterpret_cast<float*>(smem + L::q_bytes + L::k_bytes + L::raw_bytes);
    float* sw = sout + NQ * kTileKeys;
    float* sscale = sw + NQ * kIH;
    int* spos = reinterpret_cast<int*>(sscale + kTileKeys);

    const int b = blockIdx.y;
    const int ctx = __ldg(s.ctx_len + b);
    const int j0 = blockIdx.x * kTileKeys;
    if (ctx > s.max_ctx || ctx < 0) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0) report(d_status, DSA_ERR_BAD_INPUT);
        return;
    }
    if (j0 >= ctx) return;
    const int qs = __ldg(s.q_start + b), qe = __ldg(s.q_start + b + 1);
    if (qe - qs > s.max_q_per_seq || qe < qs) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0) report(d_status, DSA_ERR_BAD_INPUT);
        return;
    }
    const int q0 = qs + blockIdx.z * NQ;
    if (q0 >= qe) return;
    const int nq = min(NQ, qe - q0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    int maxpos = -1;
    if (tid < NQ) {
        int p = tid < nq ? __ldg(s.q_pos + q0 + tid) : -1;
        if (tid < nq && (p < 0 || p >= ctx)) {
            report(d_status, DSA_ERR_BAD_INPUT);
            p = -1;
        }
        spos[tid] = p;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < NQ; ++i) maxpos = max(maxpos, spos[i]);
    const int jn = min(kTileKeys, ctx - j0);

    if (j0 > maxpos) {  // fully masked tile: -inf only
        for (int e = tid; e < nq * jn; e += blockDim.x) {
            const int qi = e / jn, jj = e % jn;
            scores[(int64_t)(q0 + qi) * ld + j0 + jj] = -INFINITY;
        }
        return;
    }

    // ---- stage q' rows and w'
    {
        const int chunks_per_row = KP / 8;  // 16-byte chunks
        for (int e = tid; e < NQ * kIH * chunks_per_row; e += blockDim.x) {
            const int r = e / chunks_per_row, c = e % chunks_per_row;
            const int qi = r / kIH;
            const bool v = qi < nq;
            const uint16_t* src = qp + ((int64_t)(q0 + (v ? qi : 0)) * kIH + (r % kIH)) * KP + c * 8;
            cp_async16(sq + r * L::kQStride + c * 8, src, v);
        }
        for (int e = tid; e < NQ * kIH; e += blockDim.x) {
            const int qi = e / kIH;
            sw[e] = qi < nq ? __ldg(wp + (int64_t)(q0 + qi) * kIH + (e % kIH)) : 0.f;
        }
    }
    // ---- stage the key tile
    bool bad_row = false;
    if (!FP8) {
        const uint16_t* kb = reinterpret_cast<const uint16_t*>(k_idx);
        for (int e = tid; e < kTileKeys * 16; e += blockDim.x) {
            const int r = e >> 4, c = e & 15;
            int64_t row = r < jn ? phys_row(s, b, j0 + r) : -1;
            if (r < jn && row < 0) bad_row = true;
            cp_async16(sk + r * kKeyStride + c * 8, kb + (row < 0 ? 0 : row) * kID + c * 8, row >= 0);
        }
        cp_async_commit();
        if (tid < kTileKeys) sscale[tid] = 1.f;
        cp_async_wait<0>();
    } else {
        const uint8_t* kb = reinterpret_cast<const uint8_t*>(k_idx);
        for (int e = tid; e < kTileKeys * 8; e += blockDim.x) {
            const int r = e >> 3, c = e & 7;
            int64_t row = r < jn ? phys_row(s, b, j0 + r) : -1;
            if (r < jn && row < 0) bad_row = true;
            cp_async16(sraw + r * kID + c * 16, kb + (row < 0 ? 0 : row) * kID + c * 16, row >= 0);
        }
        cp_async_commit();
        if (tid < kTileKeys) {
            int64_t row = tid < jn ? phys_row(s, b, j0 + tid) : -1;
            float sc = row >= 0 ? __ldg(k_scale + row) : 0.f;
            if (sc < 0.f) {
                report(d_status, DSA_ERR_BAD_INPUT);
                sc = 0.f;
            }
            sscale[tid] = sc;
        }
        cp_async_wait<0>();
        __syncthreads();
        // e4m3 -> f16 (exact), 8 codes per step
        for (int e = tid; e < kTileKeys * 16; e += blockDim.x) {
            const int r = e >> 4, c = e & 15;
            uint2 raw = *reinterpret_cast<const uint2*>(sraw + r * kID + c * 8);
            uint4 o;
            o.x = e4m3x2_to_f16x2((uint16_t)(raw.x & 0xFFFF));
            o.y = e4m3x2_to_f16x2((uint16_t)(raw.x >> 16));
            o.z = e4m3x2_to_f16x2((uint16_t)(raw.y & 0xFFFF));
            o.w = e4m3x2_to_f16x2((uint16_t)(raw.y >> 16));
            *reinterpret_cast<uint4*>(sk + r * kKeyStride + c * 8) = o;
        }
    }
    if (bad_row) report(d_status, DSA_ERR_BAD_INPUT);
    __syncthreads();

    // ---- contraction on the tensor cores
    constexpr int NT = NQ * 4;  // n-tiles of 8 heads
    float acc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    const uint16_t* arow = sk + (warp * 16 + (lane & 15)) * kKeyStride + (lane >> 4) * 8;
    const int bl = lane & 7, bm = lane >> 3;
#pragma unroll
    for (int ks = 0; ks < KP / 16; ++ks) {
        int kd;  // key dim of this k-step
        if (KP == 192) kd = ks < 4 ? ks * 16 : (ks < 8 ? (ks - 4) * 16 : 64 + (ks - 8) * 16);
        else kd = ks * 16;
        uint32_t a[4];
        ldsm_x4(a[0], a[1], a[2], a[3], arow + kd);
#pragma unroll
        for (int nt = 0; nt < NT; nt += 2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(b0, b1, b2, b3, sq + ((nt + (bm >> 1)) * 8 + bl) * L::kQStride + ks * 16 + (bm & 1) * 8);
            if (FP8) {
                mma_f16(acc[nt], a, b0, b1);
                mma_f16(acc[nt + 1], a, b2, b3);
            } else {
                mma_bf16(acc[nt], a, b0, b1);
                mma_bf16(acc[nt + 1], a, b2, b3);
            }
        }
    }
    // ---- epilogue: relu, head weights, sum over 32 heads
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
        float p0 = 0.f, p1 = 0.f;  // keys g and g+8 of this warp
#pragma unroll
        for (int n4 = 0; n4 < 4; ++n4) {
            const int nt = qi * 4 + n4;
            const int h = n4 * 8 + 2 * c;
            const float w0 = sw[qi * kIH + h], w1 = sw[qi * kIH + h + 1];
            p0 += w0 * fmaxf(acc[nt][0], 0.f) + w1 * fmaxf(acc[nt][1], 0.f);
            p1 += w0 * fmaxf(acc[nt][2], 0.f) + w1 * fmaxf(acc[nt][3], 0.f);
        }
        p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
        p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
        p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
        p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
        if (c == 0) {
            const int r0 = warp * 16 + g, r1 = r0 + 8;
            const int pos = spos[qi];
            sout[qi * kTileKeys + r0] = (j0 + r0 <= pos) ? p0 * sscale[r0] : -INFINITY;
            sout[qi * kTileKeys + r1] = (j0 + r1 <= pos) ? p1 * sscale[r1] : -INFINITY;
        }
    }
    __syncthreads();
    for (int e = tid; e < nq * jn; e += blockDim.x) {
        const int qi = e / jn, jj = e % jn;
        scores[(int64_t)(q0 + qi) * ld + j0 + jj] = sout[qi * kTileKeys + jj];
    }
}

template <int NQ, int KP, bool FP8>
static cudaError_t launch_scores_t(const void* qp, const float* wp, const void* k_idx, const float* k_scale,
                                   const dsa_seqs& s, float* scores, int64_t ld, int32_t* d_status,
                                   cudaStream_t stream) {
    using L = IdxSmem<NQ, KP>;
    auto kern = index_scores_kernel<NQ, KP, FP8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::total);
    if (e != cudaSuccess) return e;
    dim3 grid((s.max_ctx + kTileKeys - 1) / kTileKeys, s.num_seqs, (s.max_q_per_seq + NQ - 1) / NQ);
    kern<<<grid, 256, L::total, stream>>>(reinterpret_cast<const uint16_t*>(qp), wp, k_idx, k_scale, s, scores, ld,
                                          d_status);
    return cudaGetLastError();
}

template <int NQ>
static cudaError_t launch_scores_nq(bool rope, bool fp8, const void* qp, const float* wp, const void* k_idx,
                                    const float* k_scale, const dsa_seqs& s, float* scores, int64_t ld,
                                    int32_t* d_status, cudaStream_t stream) {
    if (rope)
        return fp8 ? launch_scores_t<NQ, 192, true>(qp, wp, k_idx, k_scale, s, scores, ld, d_status, stream)
                   : launch_scores_t<NQ, 192, false>(qp, wp, k_idx, k_scale, s, scores, ld, d_status, stream);
    return fp8 ? launch_scores_t<NQ, 128, true>(qp, wp, k_idx, k_scale, s, scores, ld, d_status, stream)
               : launch_scores_t<NQ, 128, false>(qp, wp, k_idx, k_scale, s, scores, ld, d_status, stream);
}

cudaError_t launch_index_scores(const void* q_idx, const float* w, const float* ssmax_s, const float* ssmax_b,
                                const float* inv_freq, const void* k_idx, const float* k_scale, dsa_dtype k_dtype,
                                const dsa_seqs& s, int num_q, float* scores, int64_t ld, const Workspace& ws,
                                int32_t* d_status, cudaStream_t stream) {
    const bool fp8 = k_dtype == DSA_FP8_E4M3_ROWSCALE;
    const bool rope = inv_freq != nullptr;
    if (fp8)
        qprep_kernel<__half><<<num_q, 128, 0, stream>>>(
            reinterpret_cast<const __nv_bfloat16*>(q_idx), w, ssmax_s, ssmax_b, inv_freq, s, num_q,
            reinterpret_cast<__half*>(ws.qprep), ws.wprep, d_status);
    else
        qprep_kernel<__nv_bfloat16><<<num_q, 128, 0, stream>>>(
            reinterpret_cast<const __nv_bfloat16*>(q_idx), w, ssmax_s, ssmax_b, inv_freq, s, num_q,
            reinterpret_cast<__nv_bfloat16*>(ws.qprep), ws.wprep, d_status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int mq = s.max_q_per_seq;
    if (mq <= 1) return launch_scores_nq<1>(rope, fp8, ws.qprep, ws.wprep, k_idx, k_scale, s, scores, ld, d_status, stream);
    if (mq <= 2) return launch_scores_nq<2>(rope, fp8, ws.qprep, ws.wprep, k_idx, k_scale, s, scores, ld, d_status, stream);
    if (mq <= 4) return launch_scores_nq<4>(rope, fp8, ws.qprep, ws.wprep, k_idx, k_scale, s, scores, ld, d_status, stream);
    return launch_scores_nq<8>(rope, fp8, ws.qprep, ws.wprep, k_idx, k_scale, s, scores, ld, d_status, stream);
}

}  // namespace dsa
