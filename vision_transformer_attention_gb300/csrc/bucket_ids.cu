// bucket_ids.cu -- iRPE eq. 18 (piecewise index) with the eq. 25 Product
// mapping or the Euclidean mapping (section 3.2), evaluated on the GPU in
// double precision.
//
// "Rethinking and Improving Relative Position Encoding for Vision Transformer",
// Method: an axis offset x keeps its own integer index while |x| <= alpha; past
// alpha the index grows with log(|x| / alpha) / log(gamma / alpha), scaled into
// [alpha, beta], is rounded, capped at beta and truncated toward zero after the
// sign is applied. The Product id pairs the row and column indices into one
// entry of a (2h+1) x (2h+1) table with h = int(beta) (Pitfalls: the table is
// sized from int(beta), not from beta).
//
// The Euclidean id is g of the offset's length, rounded first as the original
// code does (half to even; a length sqrt(k) is never exactly a half), shifted
// by int(beta): ids int(beta)..2 int(beta) of 2 int(beta) + 1.
//
// The Cross mapping (eqs. 22-24) gives each pair a row bucket g(dr) + h and a
// column bucket span + g(dc) + h of a 2 span-row table (span = 2h + 1). Its
// offset table holds the pair of axis indices as one joint index
// (g(dr) + h) span + (g(dc) + h), the Product id, from which the attention
// kernels form the sum of the two entries; the expanded id map holds the two
// buckets as two N x N planes.
//
// The clip index of table 3 replaces g by a clip of each axis offset to
// [-h, h] and pairs the two as a Product id.
//
// A pair's id depends only on its offset, so the attention kernels read ids
// from a table indexed by offset: lut[(dr + H - 1) * (2W - 1) + dc + W - 1].
#include "rpe_attn.h"
#include "vta_internal.h"

#include <algorithm>
#include <cmath>

namespace vta {
namespace {

__device__ int piecewise_index_real(double x, double alpha, double beta, double gamma) {
    const double ax = fabs(x);
    if (ax <= alpha) return static_cast<int>(rint(x));  // rint: round half to even
    const double share = log(ax / alpha) / log(gamma / alpha);
    const double spread = rint(alpha + share * (beta - alpha));
    const double capped = fmin(beta, spread);
    return static_cast<int>(x > 0.0 ? capped : -capped);  // the cast truncates toward zero
}

__device__ int piecewise_index(int offset, double alpha, double beta, double gamma) {
    return piecewise_index_real(static_cast<double>(offset), alpha, beta, gamma);
}

__global__ void build_lut_kernel(int H, int W, int mode, double alpha, double beta,
                                 double gamma, int32_t *lut) {
    const int cols = 2 * W - 1;
    const int total = (2 * H - 1) * cols;
    const int half = static_cast<int>(beta);
    const int span = 2 * half + 1;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
        const int dr = e / cols - (H - 1);
        const int dc = e % cols - (W - 1);
        if (mode == RPE_MAP_EUCLIDEAN) {
            const double dist = rint(sqrt(static_cast<double>(dr) * dr + static_cast<double>(dc) * dc));
            lut[e] = piecewise_index_real(dist, alpha, beta, gamma) + half;
        } else if (mode == RPE_MAP_CLIP_PRODUCT) {
            const int cr = dr < -half ? -half : (dr > half ? half : dr);
            const int cc = dc < -half ? -half : (dc > half ? half : dc);
            lut[e] = (cr + half) * span + (cc + half);
        } else {  // Product, and the joint index of Cross
            const int gr = piecewise_index(dr, alpha, beta, gamma);
            const int gc = piecewise_index(dc, alpha, beta, gamma);
            lut[e] = (gr + half) * span + (gc + half);
        }
    }
}

// span > 0 (Cross): the joint index a span + b becomes row bucket a in the
// first N x N plane and column bucket span + b in the second.
__global__ void expand_ids_kernel(int H, int W, int span, const int32_t *__restrict__ lut,
                                  int32_t *__restrict__ ids) {
    const int N = H * W;
    const int cols = 2 * W - 1;
    const long long total = static_cast<long long>(N) * N;
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int i = static_cast<int>(e / N), j = static_cast<int>(e % N);
        const int dr = i / W - j / W, dc = i % W - j % W;
        const int id = lut[(dr + H - 1) * cols + (dc + W - 1)];
        if (span > 0) {
            ids[e] = id / span;
            ids[total + e] = span + id % span;
        } else {
            ids[e] = id;
        }
    }
}

}  // namespace

cudaError_t launch_build_bucket_lut(int H, int W, int mode, double alpha, double beta,
                                    double gamma, int32_t *lut, int32_t *ids, cudaStream_t stream) {
    const int total = (2 * H - 1) * (2 * W - 1);
    build_lut_kernel<<<(total + 255) / 256, 256, 0, stream>>>(H, W, mode, alpha, beta, gamma, lut);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess || ids == nullptr) return err;
    const long long n2 = static_cast<long long>(H * W) * (H * W);
    const int blocks = static_cast<int>(std::min<long long>((n2 + 255) / 256, 8LL * sm_count()));
    const int span = mode == RPE_MAP_CROSS ? 2 * static_cast<int>(beta) + 1 : 0;
    expand_ids_kernel<<<blocks, 256, 0, stream>>>(H, W, span, lut, ids);
    return cudaGetLastError();
}

}  // namespace vta
