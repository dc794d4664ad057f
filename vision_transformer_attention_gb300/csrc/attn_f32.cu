// attn_f32.cu -- fp32 relative-position attention on CUDA cores.
//
// The exact-precision path (fp32 inputs, fp32 arithmetic, expf), used where a
// result within 1e-4 of the fp64 definition is required: tf32 tensor-core
// products round operands to 10 mantissa bits and would miss that bound.
//
// One thread owns one query row. Logits follow the unified form of
// "Rethinking and Improving Relative Position Encoding for Vision Transformer"
// (eq. 13, with the contextual key / query terms of eqs. 15-16 and the bias
// mode scalar of eq. 14 inside the 1/sqrt(d) scaling) and the Swin form of
// "Swin Transformer, section 3.2" (bias added after the scaling). The value term is eq. 17. The softmax takes
// two passes over the keys, one for the row maximum and normaliser and one
// for the weighted sum, so nothing needs rescaling. With Cross tables (iRPE
// eqs. 22-24) a pair's joint id a*span + b selects table rows a and span + b,
// and every term is the sum of the two rows' terms.
#include "vta_internal.h"
#include "sm103_ptx.cuh"

#include <cmath>

namespace vta {
namespace {

constexpr int kRows = 64;  // query rows per block (one per thread)
constexpr int kKeys = 64;  // keys staged in shared memory per step
constexpr int kMaxD = 64;

struct SmemF32 {
    float k[kKeys][kMaxD];
    float v[kKeys][kMaxD];
};

// The table rows of a pair: {id, -1}, or for Cross tables {a, span + b} of the
// joint id a*span + b. Ids outside the table (which the call's host check and
// the kernel's scan of the table report) are clamped into it.
struct Rows {
    int r0, r1;
};

__device__ __forceinline__ Rows bucket_of(const F32AttnArgs &a, int i, int j) {
    // class token (iRPE section 4.1): token 0, every pair with it in the last bucket
    if (a.cls) {
        if (i == 0 || j == 0) return Rows{a.num_buckets - 1, -1};
        --i;
        --j;
    }
    const int cols = 2 * a.W - 1;
    const int off = (i / a.W - j / a.W + a.H - 1) * cols + (i % a.W - j % a.W + a.W - 1);
    int id = a.lut ? __ldg(a.lut + off) : off;
    const int nid = (a.cross_span > 0 ? a.cross_span * a.cross_span : a.num_buckets) - a.cls;
    id = id < 0 ? 0 : (id >= nid ? nid - 1 : id);
    if (a.cross_span > 0) return Rows{id / a.cross_span, a.cross_span + id % a.cross_span};
    return Rows{id, -1};
}

// Offset of head `head`'s contextual tables: 0 when one table serves every head.
__device__ __forceinline__ size_t table_offset(const F32AttnArgs &a, int head) {
    return a.tab_heads > 1 ? static_cast<size_t>(head) * a.num_buckets * a.d : 0;
}

__device__ __forceinline__ float table_terms(const F32AttnArgs &a, const float (&qi)[kMaxD],
                                             const float *kj, int id, int head) {
    float s = 0.f;
    const size_t toff = table_offset(a, head);
    if (a.tab_k) {
        const float *r = a.tab_k + toff + static_cast<size_t>(id) * a.d;
#pragma unroll
        for (int c = 0; c < kMaxD; ++c)
            if (c < a.d) s = fmaf(qi[c], __ldg(r + c), s);
    }
    if (a.tab_q) {
        const float *r = a.tab_q + toff + static_cast<size_t>(id) * a.d;
        for (int c = 0; c < a.d; ++c) s = fmaf(kj[c], __ldg(r + c), s);
    }
    if (a.bias && a.bias_inside)
        s += __ldg(a.bias + static_cast<size_t>(id) * a.bias_heads + (a.bias_heads == 1 ? 0 : head));
    return s;
}

__device__ __forceinline__ float logit(const F32AttnArgs &a, const float (&qi)[kMaxD],
                                       const float *kj, Rows ids, int head) {
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxD; ++c)
        if (c < a.d) s = fmaf(qi[c], kj[c], s);
    // the contextual terms and the iRPE bias (eqs. 13-16), inside the scaling
    s += table_terms(a, qi, kj, ids.r0, head);
    if (ids.r1 >= 0) s += table_terms(a, qi, kj, ids.r1, head);
    const int id = ids.r0;
    if (a.bias) {
        const float b = a.bias_inside ? 0.f
                      : __ldg(a.bias + static_cast<size_t>(id) * a.bias_heads +
                              (a.bias_heads == 1 ? 0 : head));
        s *= a.scale;
        s += b;  // Swin: after the scaling
    } else {
        s *= a.scale;
    }
    return s;
}

__global__ void __launch_bounds__(kRows) attn_f32_kernel(F32AttnArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SmemF32 &sm = *reinterpret_cast<SmemF32 *>(smem_raw);
    const int slice = blockIdx.y;
    const int head = slice % a.heads;
    const int i = blockIdx.x * kRows + threadIdx.x;
    const bool row_ok = i < a.N;
    const size_t base = static_cast<size_t>(slice) * a.N * a.d;
    const float *q = a.q + base;
    const float *k = a.k + base;
    const float *v = a.v + base;

    // one block scans the offset table once: an id outside the table sets the
    // status bit (bucket_of clamps it, so no read leaves the tables)
    if (a.lut != nullptr && blockIdx.x == 0 && blockIdx.y == 0) {
        const int bound = (a.cross_span > 0 ? a.cross_span * a.cross_span : a.num_buckets) - a.cls;
        const int len = (2 * a.H - 1) * (2 * a.W - 1);
        for (int e = threadIdx.x; e < len; e += blockDim.x) {
            const int id = __ldg(a.lut + e);
            if (id < 0 || id >= bound) atomicOr(a.status, kStatusBadBucket);
        }
    }

    float qi[kMaxD];
#pragma unroll
    for (int c = 0; c < kMaxD; ++c)
        qi[c] = (row_ok && c < a.d) ? q[static_cast<size_t>(i) * a.d + c] : 0.f;

    // pass 1: row maximum and normaliser, online over key blocks
    float m = -INFINITY, l = 0.f;
    for (int j0 = 0; j0 < a.N; j0 += kKeys) {
        const int nk = min(kKeys, a.N - j0);
        __syncthreads();
        for (int e = threadIdx.x; e < nk * a.d; e += blockDim.x)
            sm.k[e / a.d][e % a.d] = k[static_cast<size_t>(j0) * a.d + e];
        __syncthreads();
        if (row_ok) {
            for (int jj = 0; jj < nk; ++jj) {
                const float x = logit(a, qi, sm.k[jj], bucket_of(a, i, j0 + jj), head);
                if (x > m) {
                    l = l * expf(m - x) + 1.f;
                    m = x;
                } else {
                    l += expf(x - m);
                }
            }
        }
    }
    const float inv_l = 1.f / l;

    // pass 2: weighted sum of the values plus the value-side table (eq. 17)
    float acc[kMaxD];
#pragma unroll
    for (int c = 0; c < kMaxD; ++c) acc[c] = 0.f;
    for (int j0 = 0; j0 < a.N; j0 += kKeys) {
        const int nk = min(kKeys, a.N - j0);
        __syncthreads();
        for (int e = threadIdx.x; e < nk * a.d; e += blockDim.x) {
            sm.k[e / a.d][e % a.d] = k[static_cast<size_t>(j0) * a.d + e];
            sm.v[e / a.d][e % a.d] = v[static_cast<size_t>(j0) * a.d + e];
        }
        __syncthreads();
        if (row_ok) {
            for (int jj = 0; jj < nk; ++jj) {
                const Rows ids = bucket_of(a, i, j0 + jj);
                const float p = expf(logit(a, qi, sm.k[jj], ids, head) - m) * inv_l;
#pragma unroll
                for (int c = 0; c < kMaxD; ++c)
                    if (c < a.d) acc[c] = fmaf(p, sm.v[jj][c], acc[c]);
                if (a.tab_v) {
                    const float *tv = a.tab_v + table_offset(a, head);
                    const float *r = tv + static_cast<size_t>(ids.r0) * a.d;
#pragma unroll
                    for (int c = 0; c < kMaxD; ++c)
                        if (c < a.d) acc[c] = fmaf(p, __ldg(r + c), acc[c]);
                    if (ids.r1 >= 0) {
                        r = tv + static_cast<size_t>(ids.r1) * a.d;
#pragma unroll
                        for (int c = 0; c < kMaxD; ++c)
                            if (c < a.d) acc[c] = fmaf(p, __ldg(r + c), acc[c]);
                    }
                }
            }
        }
    }
    if (row_ok) {
        float *o = a.out + base + static_cast<size_t>(i) * a.d;
#pragma unroll
        for (int c = 0; c < kMaxD; ++c)
            if (c < a.d) o[c] = acc[c];
    }
}

}  // namespace

cudaError_t launch_attn_f32(const F32AttnArgs &args, cudaStream_t stream) {
    F32AttnArgs a = args;
    a.status = device_status_word();
    if (a.status == nullptr) return cudaErrorMemoryAllocation;
    const size_t smem = sizeof(SmemF32);
    cudaError_t err = cudaFuncSetAttribute(attn_f32_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    dim3 grid((a.N + kRows - 1) / kRows, a.slices);
    attn_f32_kernel<<<grid, kRows, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace vta
