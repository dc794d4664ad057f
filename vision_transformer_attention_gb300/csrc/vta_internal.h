// vta_internal.h -- host-side declarations shared by the .cu files of the
// library (launchers, tensor maps and the device status word). Not part of
// the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <utility>
#include <cstdint>

namespace vta {

struct WaitCtl;

// Device status word of the current device (allocated on first use; NULL if
// that failed) and the default bound on in-kernel waits.
unsigned *device_status_word();

// Workspace of the split tail items of the two-warpgroup kernel for launches on
// `stream` of the current device: floats_per_item fp32 for each of up to
// ceil(SMs / 2) tail items and kSplitCounters arrival counters (zero between
// launches: the last arrival resets its counter). Allocated on the stream's
// first use, at that size, and kept: launches on one stream run in order, and
// launches on different streams use different workspaces, so no two launches
// in flight share one. False (nothing allocated) while the stream is being
// captured and has no workspace yet, or if an allocation failed; the launch
// then runs every item whole.
constexpr int kSplitCounters = 4096;
bool stream_split_workspace(cudaStream_t stream, size_t floats_per_item, float **ws,
                            int **counters);

// Offset tables of bucket ids. lut_register records that the table at `lut`
// for an H x W grid holds only ids in [0, bound). lut_check returns RPE_OK if
// the table is known to hold only ids below `limit`; otherwise it reads the
// table back once on `stream` (synchronously), checks it and records it:
// RPE_ERR_INVALID_ARG for an id outside [0, limit), RPE_ERR_UNSUPPORTED if
// the stream is being captured (no synchronous copy is possible there).
// row_runs records (and lut_check reports, when the pointer is not null)
// whether each id forms one run along any grid row of keys.
void lut_register(const int32_t *lut, int H, int W, int bound, bool row_runs);
int lut_check(const int32_t *lut, int H, int W, int limit, cudaStream_t stream, bool *row_runs);
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s

// Number of SMs of the current device (cached per device).
// Launches kernel with programmatic stream serialization: its prologue may
// overlap the tail of the previous kernel in the stream. Only for kernels that
// call griddep_wait() before reading any input.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

int sm_count();

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point.
// dims / strides are innermost-first; strides_bytes has rank-1 entries.
bool encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, int rank, const void *base,
                       const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                       CUtensorMapSwizzle swizzle);

// ---- launchers (each returns the cudaError_t of its launch) ----

cudaError_t launch_build_bucket_lut(int H, int W, int mode, double alpha, double beta, double gamma,
                                    int32_t *lut, int32_t *ids, cudaStream_t stream);

struct F32AttnArgs {
    const float *q, *k, *v;
    float *out;
    int slices, heads, N, d, H, W;
    const int32_t *lut;  // offset -> bucket; NULL: the bucket is the offset index
    int num_buckets;
    const float *tab_k, *tab_q, *tab_v;  // [num_buckets, d] or NULL
    const float *bias;                   // [num_buckets, bias_heads] or NULL
    int bias_heads;                      // columns of bias: 1 (shared by all heads) or heads
    bool bias_inside;                    // added before the scaling (iRPE bias mode) or after (Swin)
    float scale;
    int cross_span = 0;  // > 0: Cross tables (row buckets, then column buckets); ids are joint a*span+b
    int tab_heads = 1;   // contextual tables: 1 shared, or heads (table h for head h)
    int cls = 0;         // 1: token 0 is a class token, its pairs in bucket num_buckets - 1
    unsigned *status = nullptr;  // device status word (set by launch_attn_f32)
};
cudaError_t launch_attn_f32(const F32AttnArgs &a, cudaStream_t stream);

struct SwinBf16Args {
    const void *q, *k, *v;
    void *out;
    const float *bias_table;
    int num_windows, heads, M, d;
};
cudaError_t launch_swin_bf16(const SwinBf16Args &a, cudaStream_t stream);
// Most heads the bf16 Swin kernels take (their shared-memory bias table).
int swin_bf16_max_heads();
// Swin window attention on channels-last feature maps [batch][img_h][img_w][heads][d]:
// windows are read from and written back to the maps by the kernel's TMA boxes.
struct SwinFmapArgs {
    const void *q, *k, *v;
    void *out;
    const float *bias_table;
    int batch, img_h, img_w, heads, M, d;
};
cudaError_t launch_swin_bf16_fmap(const SwinFmapArgs &a, cudaStream_t stream);

struct RpeBf16Args {
    const void *q, *k, *v, *tab_q, *tab_k, *tab_v;
    void *out;
    const int32_t *lut;
    int num_buckets, B, heads, H, W, d;
    unsigned terms;
    const float *bias = nullptr;  // bias mode: fp32 [num_buckets, bias_heads], inside the scaling
    int bias_heads = 0;
    int cross_span = 0;  // > 0: Cross tables (row buckets, then column buckets); ids are joint a*span+b
    int tab_heads = 1;   // contextual tables: 1 shared, or heads (table h for head h)
    int cls = 0;         // 1: token 0 is a class token, its pairs in bucket num_buckets - 1
    // the offset table's ids form one run per grid row of keys: along each
    // row of W keys, seen from any query column, an id does not come back
    // once another id has followed it (Product, clip and Cross tables)
    bool lut_row_runs = false;
};
cudaError_t launch_rpe_bf16(const RpeBf16Args &a, cudaStream_t stream);

// The two-warpgroup kernel for the key term alone (or no term) on grids whose
// width it is specialised for. Returns false (and launches nothing) when it
// does not cover the request; *err then stays untouched.
bool launch_rpe_bf16_pingpong(const RpeBf16Args &a, cudaStream_t stream, cudaError_t *err);
// The same kernel with the query and / or value terms (W = 14, shared tables,
// at most 64 buckets, an even number of query tiles, and for the value term
// an offset table whose ids form one run per grid row of keys).
bool launch_rpe_bf16_pingpong_qv(const RpeBf16Args &a, cudaStream_t stream, cudaError_t *err);

cudaError_t launch_wait_probe(unsigned long long limit_ns, cudaStream_t stream);

}  // namespace vta
