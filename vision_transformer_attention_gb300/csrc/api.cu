// api.cu -- the C ABI declared in include/rpe_attn.h: argument checks, the
// per-device status word, TMA tensor-map encoding and the kernel launches.
// Every check happens on the host before any launch; nothing here computes
// attention on the CPU.
#include "rpe_attn.h"
#include "vta_internal.h"
#include "sm103_ptx.cuh"

#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

namespace vta {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned *g_status[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

// Split-tail workspaces, one per (device, stream), each sized once for the
// largest tail any launch on that device can have.
struct SplitWs {
    float *ws;
    int *cnt;
};
std::map<std::pair<int, cudaStream_t>, SplitWs> g_split;

// Offset tables whose ids are known to lie in [0, bound): the tables
// rpe_build_bucket_ids wrote and the tables an attention call has checked,
// keyed by device address.
struct LutInfo {
    int H, W, bound;
    bool row_runs;  // each id forms one run along any grid row of keys
};
std::map<const void *, LutInfo> g_luts;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int status_of(cudaError_t err) { return err == cudaSuccess ? RPE_OK : RPE_ERR_CUDA; }

// bf16 iRPE launches: a request whose tables do not fit in shared memory comes
// back as cudaErrorNotSupported before anything is launched
int status_of_bf16(cudaError_t err) {
    return err == cudaErrorNotSupported ? RPE_ERR_UNSUPPORTED : status_of(err);
}

// Kernel of rpe_wait_probe: waits on a barrier that nothing arrives at.
__global__ void wait_probe_kernel(WaitCtl wc) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_wait(&bar, 0, wc, kStatusTimeoutProbe, nullptr);
    }
}

}  // namespace

unsigned *device_status_word() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_status[dev] == nullptr) {
        void *p = nullptr;
        if (cudaMalloc(&p, 256) != cudaSuccess) return nullptr;
        if (cudaMemset(p, 0, 256) != cudaSuccess) {
            cudaFree(p);
            return nullptr;
        }
        g_status[dev] = static_cast<unsigned *>(p);
    }
    return g_status[dev];
}

bool stream_split_workspace(cudaStream_t stream, size_t floats_per_item, float **ws,
                            int **counters) {
    const int dev = current_device();
    if (dev < 0) return false;
    std::lock_guard<std::mutex> lock(g_mutex);
    const auto key = std::make_pair(dev, stream);
    auto it = g_split.find(key);
    if (it == g_split.end()) {
        // no allocation while the stream is being captured: the launch then
        // runs every item whole
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
            return false;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms < 1 || 2 * ((sms + 1) / 2) > kSplitCounters)
            return false;
        // a tail has at most half a grid of items, a grid at most one CTA per SM
        const size_t items = static_cast<size_t>(sms + 1) / 2;
        void *w = nullptr, *c = nullptr;
        if (cudaMalloc(&w, items * floats_per_item * sizeof(float)) != cudaSuccess) return false;
        if (cudaMalloc(&c, kSplitCounters * sizeof(int)) != cudaSuccess ||
            cudaMemset(c, 0, kSplitCounters * sizeof(int)) != cudaSuccess) {
            cudaFree(w);
            if (c != nullptr) cudaFree(c);
            return false;
        }
        it = g_split.emplace(key, SplitWs{static_cast<float *>(w), static_cast<int *>(c)}).first;
    }
    *ws = it->second.ws;
    *counters = it->second.cnt;
    return true;
}

void lut_register(const int32_t *lut, int H, int W, int bound, bool row_runs) {
    std::lock_guard<std::mutex> lock(g_mutex);
    g_luts[lut] = LutInfo{H, W, bound, row_runs};
}

// True if, in the offset table h (ids in [0, 256)), the ids that one query
// column sees along any grid row of W keys form one run each: an id does not
// come back once another id has followed it.
bool lut_row_runs(const std::vector<int32_t> &h, int H, int W) {
    const int cols = 2 * W - 1;
    for (int r = 0; r < 2 * H - 1; ++r)
        for (int qx = 0; qx < W; ++qx) {
            bool ended[256] = {};
            int prev = -1;
            for (int kx = 0; kx < W; ++kx) {
                const int id = h[static_cast<size_t>(r) * cols + (qx - kx + W - 1)];
                if (id == prev) continue;
                if (id < 0 || id >= 256 || ended[id]) return false;
                if (prev >= 0) ended[prev] = true;
                prev = id;
            }
        }
    return true;
}

int lut_check(const int32_t *lut, int H, int W, int limit, cudaStream_t stream, bool *row_runs) {
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        auto it = g_luts.find(lut);
        if (it != g_luts.end() && it->second.H == H && it->second.W == W &&
            it->second.bound <= limit) {
            if (row_runs != nullptr) *row_runs = it->second.row_runs;
            return RPE_OK;
        }
    }
    // a table not yet known: read it back once (a synchronous copy, which a
    // stream capture does not allow)
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return RPE_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return RPE_ERR_UNSUPPORTED;
    const size_t n = static_cast<size_t>(2 * H - 1) * (2 * W - 1);
    std::vector<int32_t> host(n);
    if (cudaMemcpyAsync(host.data(), lut, n * sizeof(int32_t), cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return RPE_ERR_CUDA;
    int lo = INT_MAX, hi = INT_MIN;
    for (const int32_t id : host) {
        lo = id < lo ? id : lo;
        hi = id > hi ? id : hi;
    }
    if (lo < 0 || hi >= limit) return RPE_ERR_INVALID_ARG;
    const bool runs = lut_row_runs(host, H, W);
    lut_register(lut, H, W, hi + 1, runs);
    if (row_runs != nullptr) *row_runs = runs;
    return RPE_OK;
}

int sm_count() {
    const int dev = current_device();
    if (dev < 0) return 1;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_sms[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sms[dev] = n > 0 ? n : 1;
    }
    return g_sms[dev];
}

bool encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, int rank, const void *base,
                       const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                       CUtensorMapSwizzle swizzle) {
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (g_encode == nullptr) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return false;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    cuuint64_t gdim[5];
    cuuint64_t gstride[4];
    cuuint32_t bdim[5];
    cuuint32_t estride[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estride[i] = 1;
        if (i + 1 < rank) gstride[i] = strides_bytes[i];
    }
    const CUresult r = g_encode(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void *>(base),
                                gdim, gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

cudaError_t launch_wait_probe(unsigned long long limit_ns, cudaStream_t stream) {
    unsigned *status = device_status_word();
    if (status == nullptr) return cudaErrorMemoryAllocation;
    wait_probe_kernel<<<1, 32, 0, stream>>>(WaitCtl{status, limit_ns});
    return cudaGetLastError();
}

}  // namespace vta

using namespace vta;

extern "C" {

int rpe_build_bucket_ids(int H, int W, int mode, double alpha, double beta, double gamma,
                         int32_t *bucket_lut, int32_t *ids, int *num_buckets, void *stream) {
    if (H < 1 || W < 1 || mode < RPE_MAP_PRODUCT || mode > RPE_MAP_CLIP_PRODUCT ||
        bucket_lut == nullptr || num_buckets == nullptr)
        return RPE_ERR_INVALID_ARG;
    if (!std::isfinite(alpha) || !std::isfinite(beta) || !std::isfinite(gamma) || alpha <= 0.0 ||
        alpha > beta || beta > gamma || beta >= 127.0)
        return RPE_ERR_INVALID_ARG;
    // the offset table's (2H-1)(2W-1) entries, and the N x N expansion when asked for,
    // are indexed with 32-bit ints
    const long long n = static_cast<long long>(H) * W;
    if (H > 32768 || W > 32768 || (2LL * H - 1) * (2LL * W - 1) >= (1LL << 31) ||
        (ids != nullptr && n * n >= (1LL << 31)))
        return RPE_ERR_INVALID_ARG;
    const int half = static_cast<int>(beta);
    const int span = 2 * half + 1;
    const int nb = mode == RPE_MAP_EUCLIDEAN ? span : mode == RPE_MAP_CROSS ? 2 * span : span * span;
    if (nb > 256) return RPE_ERR_INVALID_ARG;
    if (!aligned16(bucket_lut) || (ids != nullptr && !aligned16(ids))) return RPE_ERR_INVALID_ARG;
    *num_buckets = nb;
    const int rc = status_of(launch_build_bucket_lut(H, W, mode, alpha, beta, gamma, bucket_lut,
                                                     ids, static_cast<cudaStream_t>(stream)));
    // every id the kernel writes lies below the bucket count (for Cross: below
    // span^2, the joint index)
    // Product, clip and Cross ids are monotone in the column offset for a fixed
    // row offset, so each id forms one run along a grid row of keys; Euclidean
    // ids (a distance) repeat on both sides of the query column
    if (rc == RPE_OK)
        lut_register(bucket_lut, H, W, mode == RPE_MAP_CROSS ? span * span : nb,
                     mode != RPE_MAP_EUCLIDEAN);
    return rc;
}

int rpe_attn_fwd(const void *q, const void *k, const void *v, const void *table_q,
                 const void *table_k, const void *table_v, const int32_t *bucket_lut,
                 int num_buckets, int B, int heads, int H, int W, int d, unsigned terms, int dtype,
                 void *out, void *stream) {
    if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || bucket_lut == nullptr)
        return RPE_ERR_INVALID_ARG;
    if (B < 1 || heads < 1 || H < 1 || W < 1 || d < 1 || num_buckets < 1) return RPE_ERR_INVALID_ARG;
    if ((terms & ~63u) != 0) return RPE_ERR_INVALID_ARG;
    const int cross_span = (terms & RPE_TABLES_CROSS) ? num_buckets / 2 : 0;
    const int tab_heads = (terms & RPE_TABLES_PER_HEAD) ? heads : 1;
    const int cls = (terms & RPE_CLS_TOKEN) ? 1 : 0;
    terms &= 7u;
    if (((terms & RPE_TERM_K) && table_k == nullptr) || ((terms & RPE_TERM_Q) && table_q == nullptr) ||
        ((terms & RPE_TERM_V) && table_v == nullptr))
        return RPE_ERR_INVALID_ARG;
    if (dtype != RPE_DTYPE_BF16 && dtype != RPE_DTYPE_F32) return RPE_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, out, bucket_lut,
                          (terms & RPE_TERM_Q) ? table_q : nullptr,
                          (terms & RPE_TERM_K) ? table_k : nullptr,
                          (terms & RPE_TERM_V) ? table_v : nullptr};
    for (const void *p : ptrs)
        if (p != nullptr && !aligned16(p)) return RPE_ERR_INVALID_ARG;
    const long long N = static_cast<long long>(H) * W + cls;  // token 0: the class token
    const long long slices = static_cast<long long>(B) * heads;
    if (N > 65536 || num_buckets > 256) return RPE_ERR_UNSUPPORTED;
    if (cross_span > 0 && (num_buckets % 2 != 0 || cross_span * cross_span > 64 || cls))
        return RPE_ERR_UNSUPPORTED;
    if (cls && num_buckets < 2) return RPE_ERR_INVALID_ARG;
    if (slices * N * d >= (1LL << 40)) return RPE_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == RPE_DTYPE_F32) {
        if (d > 64 || slices > 65535) return RPE_ERR_UNSUPPORTED;
    } else if (d != 64 || num_buckets > 128 || ((terms & RPE_TERM_Q) && num_buckets > 64)) {
        // bf16: up to 128 buckets for the key and value terms (two 64-bucket
        // halves), 64 for the query term
        return RPE_ERR_UNSUPPORTED;
    }
    bool row_runs = false;
    const int lut_rc = lut_check(bucket_lut, H, W,
                                 (cross_span > 0 ? cross_span * cross_span : num_buckets) - cls, st,
                                 &row_runs);
    if (lut_rc != RPE_OK) return lut_rc;
    if (dtype == RPE_DTYPE_F32) {
        F32AttnArgs a{};
        a.cross_span = cross_span;
        a.cls = cls;
        a.q = static_cast<const float *>(q);
        a.k = static_cast<const float *>(k);
        a.v = static_cast<const float *>(v);
        a.out = static_cast<float *>(out);
        a.slices = static_cast<int>(slices);
        a.heads = heads;
        a.N = static_cast<int>(N);
        a.d = d;
        a.H = H;
        a.W = W;
        a.lut = bucket_lut;
        a.num_buckets = num_buckets;
        a.tab_k = (terms & RPE_TERM_K) ? static_cast<const float *>(table_k) : nullptr;
        a.tab_q = (terms & RPE_TERM_Q) ? static_cast<const float *>(table_q) : nullptr;
        a.tab_v = (terms & RPE_TERM_V) ? static_cast<const float *>(table_v) : nullptr;
        a.tab_heads = tab_heads;
        a.bias = nullptr;
        a.bias_heads = 1;
        a.bias_inside = false;
        a.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
        return status_of(launch_attn_f32(a, st));
    }
    RpeBf16Args a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.tab_q = (terms & RPE_TERM_Q) ? table_q : nullptr;
    a.tab_k = (terms & RPE_TERM_K) ? table_k : nullptr;
    a.tab_v = (terms & RPE_TERM_V) ? table_v : nullptr;
    a.out = out;
    a.lut = bucket_lut;
    a.num_buckets = num_buckets;
    a.B = B;
    a.heads = heads;
    a.H = H;
    a.W = W;
    a.d = d;
    a.terms = terms;
    a.cross_span = cross_span;
    a.tab_heads = tab_heads;
    a.cls = cls;
    a.lut_row_runs = row_runs;
    return status_of_bf16(launch_rpe_bf16(a, st));
}

int rpe_attn_bias_fwd(const void *q, const void *k, const void *v, const float *bias_table,
                      int bias_heads, const int32_t *bucket_lut, int num_buckets,
                      unsigned flags, int B, int heads, int H, int W, int d, int dtype,
                      void *out, void *stream) {
    if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || bias_table == nullptr ||
        bucket_lut == nullptr)
        return RPE_ERR_INVALID_ARG;
    if (B < 1 || heads < 1 || H < 1 || W < 1 || d < 1 || num_buckets < 1) return RPE_ERR_INVALID_ARG;
    if (bias_heads != 1 && bias_heads != heads) return RPE_ERR_INVALID_ARG;
    if ((flags & ~static_cast<unsigned>(RPE_TABLES_CROSS | RPE_CLS_TOKEN)) != 0)
        return RPE_ERR_INVALID_ARG;
    const int cross_span = (flags & RPE_TABLES_CROSS) ? num_buckets / 2 : 0;
    const int cls = (flags & RPE_CLS_TOKEN) ? 1 : 0;
    if (dtype != RPE_DTYPE_BF16 && dtype != RPE_DTYPE_F32) return RPE_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, out, bucket_lut, bias_table};
    for (const void *p : ptrs)
        if (!aligned16(p)) return RPE_ERR_INVALID_ARG;
    const long long N = static_cast<long long>(H) * W + cls;  // token 0: the class token
    const long long slices = static_cast<long long>(B) * heads;
    if (N > 65536 || num_buckets > 256) return RPE_ERR_UNSUPPORTED;
    if (cross_span > 0 && (num_buckets % 2 != 0 || cross_span * cross_span > 64 || cls))
        return RPE_ERR_UNSUPPORTED;
    if (cls && num_buckets < 2) return RPE_ERR_INVALID_ARG;
    if (slices * N * d >= (1LL << 40)) return RPE_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == RPE_DTYPE_F32) {
        if (d > 64 || slices > 65535) return RPE_ERR_UNSUPPORTED;
    } else if (d != 64 || num_buckets > 128) {
        // bf16: the two-warpgroup kernel (W in {14, 56}, no class token) or the
        // general kernel
        return RPE_ERR_UNSUPPORTED;
    }
    const int lut_rc = lut_check(bucket_lut, H, W,
                                 (cross_span > 0 ? cross_span * cross_span : num_buckets) - cls, st,
                                 nullptr);
    if (lut_rc != RPE_OK) return lut_rc;
    if (dtype == RPE_DTYPE_F32) {
        F32AttnArgs a{};
        a.cross_span = cross_span;
        a.cls = cls;
        a.q = static_cast<const float *>(q);
        a.k = static_cast<const float *>(k);
        a.v = static_cast<const float *>(v);
        a.out = static_cast<float *>(out);
        a.slices = static_cast<int>(slices);
        a.heads = heads;
        a.N = static_cast<int>(N);
        a.d = d;
        a.H = H;
        a.W = W;
        a.lut = bucket_lut;
        a.num_buckets = num_buckets;
        a.bias = bias_table;
        a.bias_heads = bias_heads;
        a.bias_inside = true;
        a.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
        return status_of(launch_attn_f32(a, st));
    }
    RpeBf16Args a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.lut = bucket_lut;
    a.num_buckets = num_buckets;
    a.B = B;
    a.heads = heads;
    a.H = H;
    a.W = W;
    a.d = d;
    a.terms = 0;
    a.bias = bias_table;
    a.bias_heads = bias_heads;
    a.cross_span = cross_span;
    a.cls = cls;
    return status_of_bf16(launch_rpe_bf16(a, st));
}

int swin_window_attn_fwd(const void *q, const void *k, const void *v, const float *bias_table,
                         int num_windows, int heads, int M, int d, int dtype, void *out,
                         void *stream) {
    if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || bias_table == nullptr)
        return RPE_ERR_INVALID_ARG;
    if (num_windows < 1 || heads < 1 || M < 1 || d < 1) return RPE_ERR_INVALID_ARG;
    if (dtype != RPE_DTYPE_BF16 && dtype != RPE_DTYPE_F32) return RPE_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, out, bias_table};
    for (const void *p : ptrs)
        if (!aligned16(p)) return RPE_ERR_INVALID_ARG;
    const long long units = static_cast<long long>(num_windows) * heads;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == RPE_DTYPE_F32) {
        if (M < 2 || M > 8 || d > 64 || units > 65535) return RPE_ERR_UNSUPPORTED;
        F32AttnArgs a{};
        a.q = static_cast<const float *>(q);
        a.k = static_cast<const float *>(k);
        a.v = static_cast<const float *>(v);
        a.out = static_cast<float *>(out);
        a.slices = static_cast<int>(units);
        a.heads = heads;
        a.N = M * M;
        a.d = d;
        a.H = M;
        a.W = M;
        a.lut = nullptr;  // the bucket of a pair is its shifted, flattened offset
        a.num_buckets = (2 * M - 1) * (2 * M - 1);
        a.bias = bias_table;
        a.bias_heads = heads;
        a.bias_inside = false;
        a.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
        return status_of(launch_attn_f32(a, st));
    }
    if (M != 7 || (d != 32 && d != 64) || heads > swin_bf16_max_heads() || units >= (1LL << 30))
        return RPE_ERR_UNSUPPORTED;
    SwinBf16Args a{q, k, v, out, bias_table, num_windows, heads, M, d};
    return status_of(launch_swin_bf16(a, st));
}

int swin_window_attn_fwd_fmap(const void *q, const void *k, const void *v,
                              const float *bias_table, int batch, int img_h, int img_w,
                              int heads, int M, int d, void *out, void *stream) {
    if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || bias_table == nullptr)
        return RPE_ERR_INVALID_ARG;
    if (batch < 1 || img_h < 1 || img_w < 1 || heads < 1 || M < 1 || d < 1)
        return RPE_ERR_INVALID_ARG;
    if (img_h % M != 0 || img_w % M != 0) return RPE_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, out, bias_table};
    for (const void *p : ptrs)
        if (!aligned16(p)) return RPE_ERR_INVALID_ARG;
    const long long units =
        static_cast<long long>(batch) * (img_h / M) * (img_w / M) * static_cast<long long>(heads);
    if (M != 7 || (d != 32 && d != 64) || heads > swin_bf16_max_heads() || units >= (1LL << 30) ||
        img_h >= (1 << 24) || img_w >= (1 << 24))
        return RPE_ERR_UNSUPPORTED;
    SwinFmapArgs a{q, k, v, out, bias_table, batch, img_h, img_w, heads, M, d};
    return status_of(launch_swin_bf16_fmap(a, static_cast<cudaStream_t>(stream)));
}

int rpe_device_status(unsigned *status, int clear) {
    if (status == nullptr) return RPE_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return RPE_ERR_CUDA;
    unsigned *word = device_status_word();
    if (word == nullptr) return RPE_ERR_CUDA;
    unsigned host = 0;
    if (cudaMemcpy(&host, word, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess)
        return RPE_ERR_CUDA;
    if (clear && host != 0 && cudaMemset(word, 0, sizeof(host)) != cudaSuccess) return RPE_ERR_CUDA;
    *status = host;
    if (host & kStatusTimeoutMask) return RPE_ERR_TIMEOUT;
    return host ? RPE_ERR_INVALID_ARG : RPE_OK;
}

int rpe_wait_probe(uint64_t limit_ns, void *stream) {
    const unsigned long long lim = limit_ns ? limit_ns : 1000000ull;
    if (lim > kDefaultWaitNs) return RPE_ERR_INVALID_ARG;
    return status_of(launch_wait_probe(lim, static_cast<cudaStream_t>(stream)));
}

int rpe_release_stream(void *stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return RPE_OK;  // nothing allocated
    std::lock_guard<std::mutex> lock(g_mutex);
    auto it = g_split.find(std::make_pair(dev, static_cast<cudaStream_t>(stream)));
    if (it == g_split.end()) return RPE_OK;
    const bool ok = cudaFree(it->second.ws) == cudaSuccess && cudaFree(it->second.cnt) == cudaSuccess;
    g_split.erase(it);
    return ok ? RPE_OK : RPE_ERR_CUDA;
}

int rpe_shutdown(void) {
    std::lock_guard<std::mutex> lock(g_mutex);
    int rc = RPE_OK;
    int cur = -1;
    const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
    auto fail = [&]() { if (rc == RPE_OK) rc = RPE_ERR_CUDA; };
    for (auto &kv : g_split) {
        if (cudaSetDevice(kv.first.first) != cudaSuccess || cudaFree(kv.second.ws) != cudaSuccess ||
            cudaFree(kv.second.cnt) != cudaSuccess)
            fail();
    }
    g_split.clear();
    for (int d = 0; d < kMaxDevices; ++d) {
        if (g_status[d] == nullptr) continue;
        if (cudaSetDevice(d) != cudaSuccess || cudaFree(g_status[d]) != cudaSuccess) fail();
        g_status[d] = nullptr;
    }
    g_luts.clear();
    if (have_cur && cudaSetDevice(cur) != cudaSuccess) fail();
    return rc;
}

const char *rpe_status_string(int status) {
    switch (status) {
        case RPE_OK: return "ok";
        case RPE_ERR_INVALID_ARG: return "invalid argument";
        case RPE_ERR_UNSUPPORTED: return "unsupported shape, type or size";
        case RPE_ERR_CUDA: return "CUDA error";
        case RPE_ERR_TIMEOUT: return "an in-kernel wait timed out";
        default: return "unknown status";
    }
}

}  // extern "C"
