/*
 * rpe_attn.h -- C ABI of the GB300 relative-position attention library
 * (libvta_gb300.so). Plain pointers and sizes only; no C++ or torch types.
 *
 * Sources, by page title and section:
 *   iRPE  = "Rethinking and Improving Relative Position Encoding for Vision
 *           Transformer": Method (eq. 13 unified logit, eq. 15 contextual key,
 *           eq. 16 contextual query, eq. 17 contextual value, eq. 18 piecewise
 *           index, eq. 25 Product mapping, eqs. 26-28 efficient computation).
 *   SWIN  = "Swin Transformer, section 3.2 and Table 4": SoftMax(QK^T/sqrt(d) + B)V.
 *   SWIN2D= "Swin 的二维 RPE" (Swin's 2D RPE), sections 3.1-3.2: the compact
 *           (2M-1) x (2M-1) table read at the offset shifted by M-1.
 *
 * Conventions shared by every call
 *   - Tokens of an H x W grid are numbered row-major: token i sits at
 *     (i / W, i % W). An offset is query minus key, (dr, dc) = (r_i - r_j,
 *     c_i - c_j).
 *   - Device pointers must be 16-byte aligned and point to contiguous
 *     row-major memory of the stated shape. The caller owns every buffer;
 *     the library never frees or keeps a caller pointer after the call.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream). Argument errors are detected on the
 *     host before any launch and return RPE_ERR_INVALID_ARG or
 *     RPE_ERR_UNSUPPORTED; a failed launch returns RPE_ERR_CUDA.
 *   - Every wait inside a kernel is bounded (2 s of GPU time). A wait that
 *     runs out sets a bit in a per-device status word and the kernel returns
 *     early, leaving its output undefined; rpe_device_status() reads the word.
 *     The word (256 bytes per device, made on the first call on that device)
 *     and the split-tail workspaces described at rpe_attn_fwd are the
 *     library's only device allocations.
 *   - There is no CPU fallback: without a usable sm_103 GPU the calls
 *     return RPE_ERR_CUDA.
 */
#ifndef VTA_GB300_RPE_ATTN_H
#define VTA_GB300_RPE_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum {
    RPE_OK = 0,
    RPE_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size or flag      */
    RPE_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels implement     */
    RPE_ERR_CUDA = 3,        /* a CUDA runtime / driver call failed              */
    RPE_ERR_TIMEOUT = 4      /* a bounded in-kernel wait ran out (device status) */
};

/* Offset-to-bucket mappings (iRPE section 3.2): Product and Cross (directed),
 * Euclidean (undirected), and the clip index of iRPE table 3 paired as a
 * Product. Quantization is not built. */
enum { RPE_MAP_PRODUCT = 0, RPE_MAP_EUCLIDEAN = 1, RPE_MAP_CROSS = 2, RPE_MAP_CLIP_PRODUCT = 3 };

/* Which contextual terms rpe_attn_fwd adds (iRPE eqs. 15-17). RPE_TABLES_CROSS
 * (also a flag of rpe_attn_bias_fwd) says the tables are laid out for the
 * Cross mapping: 2 * span rows, the row buckets 0..span-1 then the column
 * buckets span..2 span-1, with bucket_lut holding the joint index
 * a * span + b of row bucket a and column bucket span + b (as
 * rpe_build_bucket_ids writes it for RPE_MAP_CROSS); each pair's term is then
 * the sum of its row and column entries (eqs. 22-24). span = num_buckets / 2. */
enum { RPE_TERM_K = 1, RPE_TERM_Q = 2, RPE_TERM_V = 4, RPE_TABLES_CROSS = 8 };

/* Flag of rpe_attn_fwd: the contextual tables are [heads, num_buckets, d], one
 * per head (head h reads table h), instead of one [num_buckets, d] table
 * shared by every head (iRPE section 4.2, table 2). */
enum { RPE_TABLES_PER_HEAD = 16 };

/* Flag of rpe_attn_fwd and rpe_attn_bias_fwd: token 0 is a class token (iRPE
 * section 4.1). q, k, v and out then hold N = H * W + 1 tokens, token t >= 1
 * being grid token t - 1, and every pair involving token 0 takes the extra
 * bucket num_buckets - 1 (the offset table's ids lie below it). Not combined
 * with RPE_TABLES_CROSS. */
enum { RPE_CLS_TOKEN = 32 };

/* Element types of q, k, v, out and the iRPE tables. */
enum { RPE_DTYPE_BF16 = 0, RPE_DTYPE_F32 = 1 };

/*
 * rpe_build_bucket_ids -- iRPE eq. 18 with the eq. 25 (Product) or the
 * Euclidean mapping (section 3.2), evaluated on the GPU in double precision.
 *
 * For an H x W grid and index-function constants 0 < alpha <= beta <= gamma
 * (the code's ratio r gives alpha = r, beta = 2r, gamma = 8r), with
 * h = int(beta):
 *   RPE_MAP_PRODUCT:   the piecewise index g of every axis offset, the row and
 *                      column indices paired into one bucket
 *                        id = (g(dr) + h) * (2h + 1) + (g(dc) + h),
 *                      (2h + 1)^2 buckets;
 *   RPE_MAP_EUCLIDEAN: g of the offset's Euclidean length, rounded (half to
 *                      even) before the index as the original code does,
 *                        id = g(rint(sqrt(dr^2 + dc^2))) + h,
 *                      2h + 1 buckets (ids h..2h occur);
 *   RPE_MAP_CROSS:     a row bucket g(dr) + h and a column bucket
 *                      (2h + 1) + g(dc) + h, 2 (2h + 1) buckets; the offset
 *                      table holds the joint index (the Product id above),
 *                      which the attention calls split with RPE_TABLES_CROSS;
 *   RPE_MAP_CLIP_PRODUCT: each axis offset clipped to [-h, h] (iRPE table 3,
 *                      the clip index in place of g), paired as
 *                        id = (clip(dr) + h) * (2h + 1) + (clip(dc) + h),
 *                      (2h + 1)^2 buckets; alpha and gamma are checked but
 *                      not used.
 * Outputs (device, int32, written on `stream`):
 *   bucket_lut [(2H-1) * (2W-1)]  id of offset (dr, dc) at
 *                                 (dr + H - 1) * (2W - 1) + (dc + W - 1).
 *                                 rpe_attn_fwd consumes this form: every
 *                                 mapping on the pages is translation
 *                                 invariant, so the N x N map is this table
 *                                 read at each pair's offset.
 *   ids        [N * N] or NULL    the expanded map (query i, key j at i*N + j),
 *                                 N = H * W, read from the same table; for
 *                                 RPE_MAP_CROSS [2 * N * N]: the row buckets,
 *                                 then the column buckets.
 *   num_buckets (host int*)       set to the mapping's bucket count.
 * Errors (RPE_ERR_INVALID_ARG): H or W < 1 or > 32768, N*N >= 2^31 with ids
 * requested (without ids any grid the attention calls take is served), alpha <= 0,
 * alpha > beta or beta > gamma or a non-finite constant, an unknown mode, a
 * NULL bucket_lut or num_buckets, more than 256 buckets.
 */
int rpe_build_bucket_ids(int H, int W, int mode, double alpha, double beta,
                         double gamma, int32_t *bucket_lut, int32_t *ids,
                         int *num_buckets, void *stream);

/*
 * rpe_attn_fwd -- iRPE contextual attention on an H x W grid (eqs. 13, 15-17),
 * forward only, the contextual terms computed the efficient way (eqs. 26-28).
 *
 *   e_ij  = ( q_i.k_j + [K] q_i.R^K[id] + [Q] k_j.R^Q[id] ) / sqrt(d)
 *   out_i = sum_j softmax_j(e_ij) * ( v_j + [V] R^V[id] ),   id = id(i, j)
 *
 * q, k, v, out : device [B, heads, N, d], N = H * W, element type `dtype`.
 * table_q/k/v  : device [num_buckets, d], same element type, shared by all
 *                heads, or [heads, num_buckets, d] with RPE_TABLES_PER_HEAD;
 *                NULL for a term whose bit is not set in `terms` (a table
 *                whose bit is off is not read).
 * bucket_lut   : device int32 [(2H-1) * (2W-1)] from rpe_build_bucket_ids, or
 *                any table of ids indexed the same way. Every id must lie in
 *                [0, num_buckets) ([0, num_buckets - 1) with RPE_CLS_TOKEN,
 *                whose last bucket is the class token's; [0, span^2) for
 *                Cross tables). A table rpe_build_bucket_ids wrote is known
 *                to satisfy this; any other table is read back and checked on
 *                its first use with this grid (a synchronous copy of its
 *                (2H-1)(2W-1) ids on `stream`; RPE_ERR_UNSUPPORTED if `stream`
 *                is being captured, so make that first call outside a
 *                capture) and an id out of range returns RPE_ERR_INVALID_ARG
 *                before any launch. The check is remembered per device
 *                address: a table rewritten in place by other means after
 *                its check is caught by the kernel instead, which sets a
 *                status bit that rpe_device_status reports as
 *                RPE_ERR_INVALID_ARG (the id is clamped meanwhile, so no read
 *                leaves the tables). The check also records whether, seen
 *                from any query column, each id forms one run along a grid
 *                row of keys (true of Product, clip and Cross tables, false
 *                of Euclidean ones); the fast value-term path (bf16, W = 14)
 *                needs it. A table rewritten in place so that this no longer
 *                holds is reported the same way.
 * terms        : OR of RPE_TERM_K / RPE_TERM_Q / RPE_TERM_V (0 = plain attention),
 *                plus RPE_TABLES_CROSS for tables of the Cross mapping,
 *                RPE_TABLES_PER_HEAD for one table per head and RPE_CLS_TOKEN
 *                for a class token at token 0 (then N = H * W + 1).
 * Supported: RPE_DTYPE_BF16 with d == 64 (tcgen05 tensor cores, fp32
 * accumulation, probabilities rounded to bf16 before the value products);
 * RPE_DTYPE_F32 with d <= 64 and B * heads <= 65535 (fp32 on CUDA cores);
 * B * heads * N * d < 2^40 for both; 1 <= num_buckets <= 256
 * for fp32, <= 128 for bf16 (<= 64 with RPE_TERM_Q); with RPE_TABLES_CROSS
 * num_buckets even and (num_buckets / 2)^2 <= 64; N <= 65536. Anything else
 * returns RPE_ERR_UNSUPPORTED.
 * bf16 kernels keep the offset table ((2H-1)(2W-1) bytes, 2(2H-1)(2W-1) + 1
 * with a class token) and the per-bucket tables of one query tile in one
 * SM's shared memory. A request for which they do not fit returns
 * RPE_ERR_UNSUPPORTED before any launch. With 64 buckets the offset table may
 * take 147,968 bytes for plain attention, 107,008 with the key or the value
 * term, 105,984 with the query term, 65,024 to 66,048 with two terms and
 * 24,064 with all three (square grids up to 192, 164, 163, 127 and 78 on a
 * side); fewer buckets leave a little more room. The key and value terms
 * together take at most 110 buckets on a 14 x 14 grid, 100 on 56 x 56. fp32
 * reads the offset table from global memory and has no such limit.
 * Device memory: the library allocates, on first use per device and never
 * frees, a status word and, for bf16 calls on the two-warpgroup kernel whose
 * last round of (batch, head) work items fills at most half the GPU, one
 * workspace per stream (about 10 MB with 152 SMs, sized once for the largest
 * tail, never grown) through which two CTAs merge a split item. Calls on
 * different streams never share a workspace, so overlapping calls are safe; a
 * CUDA graph captured on a stream uses that stream's workspace, so two
 * replays of such graphs must not overlap one another or a call on that
 * stream. A stream's first split call allocates; under stream capture,
 * where no allocation is made, a stream without a workspace runs every item
 * whole (same result, a little slower).
 */
int rpe_attn_fwd(const void *q, const void *k, const void *v,
                 const void *table_q, const void *table_k, const void *table_v,
                 const int32_t *bucket_lut, int num_buckets,
                 int B, int heads, int H, int W, int d,
                 unsigned terms, int dtype, void *out, void *stream);

/*
 * rpe_attn_bias_fwd -- iRPE bias mode on an H x W grid (eqs. 13-14): a learned
 * scalar per bucket, added to the content logit before the scaling,
 *
 *   e_ij  = ( q_i.k_j + b[id(i, j)][h] ) / sqrt(d)
 *   out_i = sum_j softmax_j(e_ij) v_j
 *
 * q, k, v, out : device [B, heads, N, d], N = H * W, element type `dtype`.
 * bias_table   : device float32 [num_buckets, bias_heads] (bucket-major);
 *                bias_heads = heads (column h for head h) or 1 (one table
 *                shared by every head).
 * bucket_lut, num_buckets: as for rpe_attn_fwd (any mapping).
 * flags        : 0, or RPE_TABLES_CROSS for a Cross-mapping table (the bias
 *                of a pair is then b[a][h] + b[span + b'][h] for its joint
 *                index a * span + b'), or RPE_CLS_TOKEN (token 0 is a class
 *                token whose pairs take bias row num_buckets - 1).
 * Supported: RPE_DTYPE_F32 on any grid with d <= 64, num_buckets <= 256 and
 * B * heads <= 65535;
 * RPE_DTYPE_BF16 on any grid with d == 64 and num_buckets <= 128 (Cross as
 * for rpe_attn_fwd; W in {14, 56} without a class token runs on the
 * two-warpgroup kernel, everything else on the general one).
 * Errors as for rpe_attn_fwd.
 */
int rpe_attn_bias_fwd(const void *q, const void *k, const void *v, const float *bias_table,
                      int bias_heads, const int32_t *bucket_lut, int num_buckets,
                      unsigned flags, int B, int heads, int H, int W, int d, int dtype,
                      void *out, void *stream);

/*
 * swin_window_attn_fwd -- Swin window attention with the relative bias
 * (SWIN; SWIN2D 3.1-3.2), forward only:
 *
 *   out = SoftMax( Q K^T / sqrt(d) + B ) V,
 *   B[i, j] = table[ (dr + M - 1) * (2M - 1) + (dc + M - 1) ][ head ]
 *
 * q, k, v, out : device [num_windows, heads, M*M, d], element type `dtype`
 *                (windows already partitioned; token i of a window sits at
 *                (i / M, i % M)).
 * bias_table   : device float32 [(2M-1)^2, heads] (bucket-major).
 * Supported: RPE_DTYPE_BF16 with M == 7, d in {32, 64}, heads <= 32 and
 * num_windows * heads < 2^30 (tcgen05 tensor cores); RPE_DTYPE_F32 with
 * 2 <= M <= 8, d <= 64 and num_windows * heads <= 65535 (fp32 on CUDA cores).
 * Anything else returns RPE_ERR_UNSUPPORTED.
 */
int swin_window_attn_fwd(const void *q, const void *k, const void *v,
                         const float *bias_table, int num_windows, int heads,
                         int M, int d, int dtype, void *out, void *stream);

/*
 * swin_window_attn_fwd_noalloc -- swin_window_attn_fwd for callers that must
 * not allocate device memory. The pages have no counterpart: this is a
 * library-integration entry point, not part of the method.
 *
 * Same arguments, layouts, math and output as swin_window_attn_fwd on its
 * bf16 path (dtype is implicitly RPE_DTYPE_BF16; M == 7, d in {32, 64},
 * heads <= 32; anything else returns RPE_ERR_UNSUPPORTED). The difference is
 * where the kernel's scratch lives. swin_window_attn_fwd allocates a small
 * status buffer with cudaMalloc on its first call on a device; some callers
 * cannot allow that (pipelines that forbid allocation once running, processes
 * whose device memory is reserved up front by a pooling allocator, code that
 * runs only where allocation is not permitted). This variant instead uses a
 * fixed file-scope device array of 256 bytes (64 words) that every GPU which
 * loads the library holds until the process exits; a call needs one word of
 * it (its status word), whatever the problem size, and a request needing more
 * than the array holds would return RPE_ERR_UNSUPPORTED. The call itself
 * performs no cudaMalloc, cudaFree or other allocation.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress with that device current); make that first call
 *     before any stream capture.
 *   - Every call clears the status word (an async memset on `stream`) before
 *     its kernel runs; the array otherwise keeps the last call's contents.
 *   - All calls share the array, so calls that overlap on the GPU (different
 *     streams, no ordering between them) race on the status word.
 *   - A bounded-wait timeout inside this variant sets a bit in its own word,
 *     not in the word rpe_device_status reads: swin_noalloc_status reads it.
 */
int swin_window_attn_fwd_noalloc(const void *q, const void *k, const void *v,
                                 const float *bias_table, int num_windows, int heads,
                                 int M, int d, void *out, void *stream);

/*
 * swin_noalloc_status -- the status word of swin_window_attn_fwd_noalloc on
 * the current device (no counterpart on the pages; the same bits as
 * rpe_device_status). Synchronises the device, copies the word out of the
 * fixed array (cudaMemcpyFromSymbol, no allocation) into *status and, when
 * `clear` is non-zero, writes 0 back. Returns RPE_ERR_TIMEOUT if any bit was
 * set, RPE_ERR_CUDA if a CUDA call failed, else RPE_OK.
 */
int swin_noalloc_status(unsigned *status, int clear);

/*
 * swin_noalloc_status_word -- the device address of that status word on the
 * current device (a 4-byte unsigned inside the fixed array), for callers that
 * read or clear it with their own stream-ordered copies instead of the
 * synchronising swin_noalloc_status. No allocation; the address stays valid
 * until the process exits.
 */
int swin_noalloc_status_word(unsigned **word);

/*
 * swin_window_attn_fwd_fmap -- swin_window_attn_fwd with the window partition
 * (and its reverse) fused into the kernel (SWIN 3.2: self-attention inside
 * non-overlapping M x M windows that tile the feature map).
 *
 * q, k, v, out : device bf16 feature maps [batch, img_h, img_w, heads * d],
 *                channels-last (head h of pixel (y, x) at channels
 *                [h * d, (h + 1) * d)). Window (wy, wx) of an image covers rows
 *                [wy M, wy M + M) and columns [wx M, wx M + M); its token i is
 *                pixel (wy M + i / M, wx M + i % M). Every window and head is
 *                attended exactly as swin_window_attn_fwd does for the same
 *                window cut out of the map, and out receives the result at the
 *                same pixels and channels.
 * bias_table   : device float32 [(2M-1)^2, heads], as for swin_window_attn_fwd.
 * Requires img_h and img_w to be multiples of M (else RPE_ERR_INVALID_ARG),
 * M == 7, d in {32, 64}, heads <= 32 (else RPE_ERR_UNSUPPORTED); pointers
 * 16-byte aligned. The library owns nothing the caller passes; the call is
 * asynchronous on `stream`.
 */
int swin_window_attn_fwd_fmap(const void *q, const void *k, const void *v,
                              const float *bias_table, int batch, int img_h, int img_w,
                              int heads, int M, int d, void *out, void *stream);

/*
 * rpe_device_status -- synchronises the current device and returns, through
 * *status, the word the kernels set when a bounded wait ran out (bits 0-4)
 * or an offset table held an id out of range (bit 5); 0 = none. Clears the
 * word when `clear` is non-zero. Returns RPE_ERR_TIMEOUT if a wait ran out,
 * else RPE_ERR_INVALID_ARG if a table was bad, RPE_ERR_CUDA if synchronising
 * failed, else RPE_OK.
 */
int rpe_device_status(unsigned *status, int clear);

/*
 * rpe_wait_probe -- runs the bounded-wait routine every kernel uses on a
 * barrier that nothing ever arrives at, with a bound of `limit_ns`
 * nanoseconds (1 ms if 0), so that a test can see the wait run out and set
 * the status word without faulting or hanging the GPU.
 */
int rpe_wait_probe(uint64_t limit_ns, void *stream);

/* rpe_status_string -- a static description of a status code. */
const char *rpe_status_string(int status);

/*
 * rpe_release_stream -- frees the split-tail workspace the library keeps for
 * `stream` on the current device, if there is one (see rpe_attn_fwd, "Device
 * memory"); call it before destroying a stream that ran such calls. No work
 * on the stream that may use the workspace may be pending (cudaFree waits for
 * the device anyway) and no captured graph that uses it may be replayed
 * afterwards. The stream's next split call allocates again. Returns RPE_OK
 * (also when there was nothing to free) or RPE_ERR_CUDA.
 */
int rpe_release_stream(void *stream);

/*
 * rpe_shutdown -- frees every device allocation the library has made (the
 * status words and the split-tail workspaces, on every device) and forgets
 * the offset tables it has recorded as checked. Call it when no library work
 * is pending or being captured; no graph captured before it may be replayed
 * after it. The next call allocates again. The no-allocation Swin entry
 * point's fixed array is not an allocation and stays. Returns RPE_OK, or
 * RPE_ERR_CUDA for the first failure (the rest is still freed).
 */
int rpe_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* VTA_GB300_RPE_ATTN_H */
