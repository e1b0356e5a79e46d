// dsa_internal.cuh -- shared device helpers and launcher declarations of the
// sm_103a DSA decode library.  Not part of the public ABI (include/dsa.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa.h"

namespace dsa {

constexpr int kIH = DSA_INDEX_HEADS;   // 32
constexpr int kID = DSA_INDEX_DIM;     // 128
constexpr int kRopeDims = 64;          // rotated dims of an index head
constexpr int kMH = DSA_MLA_HEADS;     // 64
constexpr int kMD = DSA_MLA_DIM;       // 576
constexpr int kMV = DSA_MLA_VDIM;      // 512
constexpr int kDsRow = DSA_DS_MLA_ROW; // 656

// kernel tags in a timeout's device status (bits 8-15)
constexpr int kTagIndexer = 1, kTagMla = 2, kTagMlaFp8 = 3, kTagMlaNvfp4 = 4, kTagIndexerNvfp4 = 5;

// ---------------------------------------------------------------------------
// device-side error reporting: first error wins, never traps
__device__ __forceinline__ void report(int32_t* d_status, int32_t code) {
    if (d_status) atomicCAS(d_status, 0, code);
}

// sequence of query row t (q_start is a CSR offset array of B+1 entries)
__device__ __forceinline__ int seq_of(const int32_t* q_start, int B, int t) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(q_start + mid) <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// physical row of token j of sequence b; -1 when the page table or base
// points outside the cache
__device__ __forceinline__ int64_t phys_row(const dsa_seqs& s, int b, int64_t j) {
    int64_t row;
    if (s.page_table) {
        int64_t p = j / s.page_size;
        if (p >= s.max_pages) return -1;
        int64_t page = __ldg(s.page_table + (int64_t)b * s.max_pages + p);
        row = page * s.page_size + (j - p * s.page_size);
        if (page < 0) return -1;
    } else {
        row = __ldg(s.seq_base + b) + j;
    }
    return (row >= 0 && row < s.num_rows) ? row : -1;
}

// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch.  The kernels of a layer run back to back on
// one stream; each is launched with programmatic stream serialisation, lets
// its own dependents launch at once and waits (griddepcontrol.wait: until the
// preceding kernel has completed and its writes are visible) before its first
// access to global memory.  The next kernel's CTAs are thus placed and ready
// while the previous one drains, and no kernel reads anything early.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 2^x on the special-function unit (PTX ex2.approx.ftz.f32): relative error
// near 2^-22, subnormal results flushed to zero, 2^-inf = 0.  Ample for
// softmax probabilities, which are rounded to bf16 right after.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// two OCP e4m3 codes (low byte first) -> f16x2, exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
    return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

// Launch with programmatic stream serialisation (and a cluster of cluster_x
// CTAs along x when cluster_x > 1).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       int cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---------------------------------------------------------------------------
// launchers (host)
struct Workspace {
    // carved from the caller's workspace, 256-byte aligned pieces
    void* qprep;      // q' [Q, 32, KP] bf16 or f16, or [Q, 3, 32, 128] e4m3 parts (kQprepBytes per query)
    float* wprep;     // w' [Q, 32]
    float* mla_part;  // O partials [Q, splits, 64, 512]
    float* mla_ml;    // (m, l) partials [Q, splits, 64, 2]
    float* scores;    // [Q, ld] for dsa_decode_layer
    int64_t scores_ld;
};

constexpr int kQprepBytes = 4 * kIH * kID;  // per query: >= 32 x 192 16-bit values and 3 x 32 x 128 e4m3
// The attention's split count per query, and the scratch its partials take
// (none for one split or a two-split cluster pair), with the partials held to
// `cap` bytes (fewer splits otherwise)
constexpr size_t kNoCap = ~size_t(0);
int mla_splits(int num_q, int k, size_t cap = kNoCap);
size_t mla_part_bytes(int num_q, int k, size_t cap = kNoCap);  // fp32 partial outputs
size_t mla_ml_bytes(int num_q, int k, size_t cap = kNoCap);    // their (max, sum) pairs
int mla_launches(int num_q, int k, size_t cap = kNoCap);       // kernels one attention call enqueues
size_t workspace_bytes(const dsa_seqs& s, int num_q, int k, int64_t* scores_ld);
Workspace carve_workspace(void* base, const dsa_seqs& s, int num_q, int k);

cudaError_t launch_index_scores(const void* q_idx, const float* w, const float* ssmax_s, const float* ssmax_b,
                                const float* inv_freq, const void* k_idx, const float* k_scale, dsa_dtype k_dtype,
                                const dsa_seqs& s, int num_q, float* scores, int64_t ld, float* gmax, int64_t ldg,
                                const Workspace& ws, int32_t* d_status, cudaStream_t stream,
                                const void* k_block_scales = nullptr, float k_global = 1.f);
// NVFP4 index keys: codes [rows, 64], E4M3 block scales [rows, 8], tensor scale k_global
cudaError_t launch_index_scores_nvfp4(const void* q_idx, const float* w, const float* ssmax_s, const float* ssmax_b,
                                      const float* inv_freq, const void* k_codes, const void* k_block_scales,
                                      float k_global, const dsa_seqs& s, int num_q, float* scores, int64_t ld,
                                      float* gmax, int64_t ldg, const Workspace& ws, int32_t* d_status,
                                      cudaStream_t stream);
cudaError_t launch_topk(const float* scores, int64_t ld, const dsa_seqs& s, int num_q, int k, int32_t* idx,
                        int32_t* topk_len, const Workspace& ws, int32_t* d_status, cudaStream_t stream);
cudaError_t launch_sparse_mla(const void* q, const void* latent, dsa_dtype latent_dtype, const dsa_seqs& s,
                              int num_q, const int32_t* idx, const int32_t* topk_len, int k, float sm_scale,
                              void* out, float* lse, const Workspace& ws, int32_t* d_status, cudaStream_t stream,
                              size_t scratch_cap = kNoCap, const void* lat_scales = nullptr, float lat_global = 1.f);

}  // namespace dsa
