// swin_attn_sm103.cu -- Swin window attention with the relative-position bias
// on sm_103a tensor cores (tcgen05 + TMEM + TMA), bf16 in, fp32 accumulate.
//
// What it computes ("Swin Transformer, section 3.2 and Table 4"):
//     out = SoftMax(Q K^T / sqrt(d) + B) V inside every M x M window, where
// B[i, j] is read from the compact (2M-1) x (2M-1) per-head table at the
// pair's offset shifted by M-1 and flattened row-major ("Swin 的二维 RPE",
// sections 3.1-3.2).
//
// Design. A (window, head) pair -- a "unit" -- has n = M*M <= 64 tokens, so
// two units share one 128-row tensor-core tile: unit 2t sits in rows 0..63
// of tile t and unit 2t+1 in rows 64..127. One 3D TMA box per operand
// ([2 units][64 rows][d], rows past n zero-filled) stages Q, K and V. A
// single M=128, N=128 MMA gives every query row its own unit's scores in
// one 64-column half of S (the other half, cross-unit, is ignored). One
// thread per row reads its half from TMEM, adds the bias from a shared-memory
// copy of the table (the per-key offset is a compile-time immediate because
// M is a template parameter), takes the softmax in base 2 and writes bf16
// probabilities back into tensor memory over the scores, as the A operand of
// P V: columns [32 s, 32 s + 32) hold slot s's keys in pairs, the other 32
// columns of the row are zero, so a single M=128, N=d, K=128 MMA gives P V,
// written to columns [64, 64 + d) (scores no longer needed). The epilogue
// scales by 1/rowsum, converts to bf16 and leaves through a TMA store that
// drops the padding rows. No n x n bias is ever formed in global memory.
//
// The kernel is persistent (grid = a multiple of the SM count), double-
// buffers Q/K/V so the next tile's loads overlap this tile's work, stages
// the output tile in the Q buffer it no longer needs, and uses 128
// tensor-memory columns and about 50 KB of shared memory per CTA at d = 32
// (four CTAs per SM, overlapping one another's latencies; two at d = 64).
#include "rpe_attn.h"
#include "vta_internal.h"
#include "sm103_ptx.cuh"

#include <cmath>
#include <mutex>

namespace vta {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Division by a divisor fixed for the whole launch, as one multiply-high, an
// add and a shift (Granlund and Montgomery, "Division by invariant integers
// using multiplication", 1994, section 4): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, n / d = (mulhi(m, n) + n) >> l for
// 0 <= n < 2^31 (the sum then stays below 2^32).
struct FastDiv {
    uint32_t d, m, l;
};

FastDiv make_fastdiv(int d) {
    FastDiv f{static_cast<uint32_t>(d < 1 ? 1 : d), 0u, 0u};
    while ((1ull << f.l) < f.d) ++f.l;
    f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << f.l) - f.d)) / f.d + 1);
    return f;
}

__device__ __forceinline__ int fast_div(const FastDiv &f, int n) {
    return static_cast<int>((__umulhi(f.m, static_cast<uint32_t>(n)) + static_cast<uint32_t>(n)) >> f.l);
}

template <int M, int D>
struct SwinTile {
    static constexpr int kN = M * M;            // tokens per window
    static constexpr int kRowBytes = D * 2;     // one bf16 row of q/k/v/out
    static constexpr uint32_t kSwz = (D == 32) ? kSwizzle64B : kSwizzle128B;
    static constexpr int kSbo = 8 * kRowBytes;  // stride between 8-row groups
    static constexpr int kOperBytes = 128 * kRowBytes;
    static constexpr int kStageBytes = 3 * kOperBytes;
    static constexpr int kNB = (2 * M - 1) * (2 * M - 1);
    static constexpr int kNBPad = (kNB + 3) & ~3;
    static constexpr int kMaxHeads = 32;
    static constexpr int kSmemFixed = 1024 + 2 * kStageBytes;
    static int smem_bytes(int heads) { return kSmemFixed + heads * kNBPad * 4; }
    static constexpr int kCtasPerSm = (D == 32) ? 4 : 2;
    static constexpr uint32_t kColO = 64;  // O after P V (scores dead by then)
    static_assert(kN <= 64, "a window must fit one 64-row slot");
};

// FM = false: q/k/v/out are [units][n][d] (windows already partitioned), one
// 3D box per operand and tile. FM = true: they are channels-last feature maps
// [batch][img_h][img_w][heads][d] and a unit is (image, window row, window
// column, head) in that order; one 5D box [1][M][M][1][d] per unit and operand
// reads the window straight from the map (and writes it back), so no
// partition or reverse copy exists.
template <int M, int D, bool FM>
__global__ void __launch_bounds__(128, SwinTile<M, D>::kCtasPerSm)
    swin_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_o, const float *__restrict__ bias_table,
                     FastDiv heads, int units, int tiles, FastDiv wins_y, FastDiv wins_x,
                     float scale_log2e, WaitCtl wc) {
    using T = SwinTile<M, D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *stage_base = smem;
    float *bias_s = reinterpret_cast<float *>(smem + 2 * T::kStageBytes);

    __shared__ __align__(8) uint64_t bar_load[2];
    __shared__ __align__(8) uint64_t bar_s;
    __shared__ __align__(8) uint64_t bar_o;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;

    griddep_launch_dependents();
    const int tid = threadIdx.x;
    const int warp = tid >> 5;

    if (tid == 0) {
        mbar_init(&bar_load[0], 1);
        mbar_init(&bar_load[1], 1);
        mbar_init(&bar_s, 1);
        mbar_init(&bar_o, 1);
        abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_o);
    }
    if (warp == 0) tmem_alloc(&tmem_base_s, 128);
    if constexpr (FM) {
        // a window's box fills rows 0..n-1 of its 64-row slot; rows n..63 of
        // both slots of every operand and stage must hold finite values (zero)
        // for the products. The boxes never write them, so the first loads
        // may land while these stores run.
        constexpr int kPadRows = 64 - T::kN;
        constexpr int kRowChunks = T::kRowBytes / 16;
        constexpr int kPadChunks = 2 * 3 * 2 * kPadRows * kRowChunks;  // stages x operands x slots
        for (int e = tid; e < kPadChunks; e += blockDim.x) {
            const int c = e % kRowChunks;
            const int row = (e / kRowChunks) % kPadRows;
            const int blk = e / (kRowChunks * kPadRows);  // (stage * 3 + operand) * 2 + slot
            st_shared_v4(smem_u32(stage_base) + (blk >> 1) * T::kOperBytes +
                             ((blk & 1) * 64 + T::kN + row) * T::kRowBytes + c * 16,
                         0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
    }
    const int nheads = static_cast<int>(heads.d);

    // Thread 0's bookkeeping of work in flight, for draining after an abort.
    uint32_t loads_pending = 0;  // bit s: stage s has a load not yet waited for
    uint32_t load_uses[2] = {0, 0};
    uint64_t *mma_bar_pending = nullptr;
    uint32_t mma_parity_pending = 0;

    // feature-map coordinates (head, first column, first row, image) of a unit
    auto unit_coords = [&](int u, int &h, int &x0, int &y0, int &b) {
        const int win = fast_div(heads, u);
        h = u - win * nheads;
        const int wrow = fast_div(wins_x, win);  // window row over all images
        x0 = (win - wrow * static_cast<int>(wins_x.d)) * M;
        b = fast_div(wins_y, wrow);
        y0 = (wrow - b * static_cast<int>(wins_y.d)) * M;
    };
    auto issue_load = [&](int tile, int stage) {
        uint8_t *sb = stage_base + stage * T::kStageBytes;
        if constexpr (FM) {
            // both slots are always loaded (an odd last tile repeats its unit
            // in slot 1, whose rows are discarded), so no slot's rows 0..n-1
            // are ever read before a load has written them
            mbar_arrive_expect_tx(&bar_load[stage], 3 * 2 * T::kN * T::kRowBytes);
            for (int s2 = 0; s2 < 2; ++s2) {
                int h, x0, y0, b;
                unit_coords(2 * tile + s2 < units ? 2 * tile + s2 : units - 1, h, x0, y0, b);
                uint8_t *dst = sb + s2 * 64 * T::kRowBytes;
                tma_load_5d(dst, &tm_q, &bar_load[stage], 0, h, x0, y0, b);
                tma_load_5d(dst + T::kOperBytes, &tm_k, &bar_load[stage], 0, h, x0, y0, b);
                tma_load_5d(dst + 2 * T::kOperBytes, &tm_v, &bar_load[stage], 0, h, x0, y0, b);
            }
        } else {
            mbar_arrive_expect_tx(&bar_load[stage], 3 * T::kOperBytes);
            tma_load_3d(sb, &tm_q, &bar_load[stage], 0, 0, 2 * tile);
            tma_load_3d(sb + T::kOperBytes, &tm_k, &bar_load[stage], 0, 0, 2 * tile);
            tma_load_3d(sb + 2 * T::kOperBytes, &tm_v, &bar_load[stage], 0, 0, 2 * tile);
        }
        loads_pending |= 1u << stage;
    };

    // nothing above reads an input: it may overlap the previous kernel
    griddep_wait();
    // the first tile's loads overlap the bias-table copy below (thread 0
    // initialised the barriers itself)
    if (tid == 0 && static_cast<int>(blockIdx.x) < tiles) issue_load(blockIdx.x, 0);

    // Bias table -> shared memory, head-major, pre-multiplied by log2(e).
    for (int e = tid; e < nheads * T::kNB; e += blockDim.x) {
        const int h = e / T::kNB, b = e % T::kNB;
        bias_s[h * T::kNBPad + b] = __ldg(bias_table + static_cast<size_t>(b) * nheads + h) * kLog2e;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    constexpr uint32_t kIdescS = idesc_bf16(128, 128, false, false);
    constexpr uint32_t kIdescO = idesc_bf16(128, D, false, true);
    const WaitCtl drain{wc.status, kDefaultWaitNs};


    // Per-thread constants: which unit slot and which row of it this thread owns.
    const int slot = tid >> 6;
    const int r = tid & 63;
    const int rr = (r < T::kN) ? r : 0;
    const int bias_base = (rr / M) * (2 * M - 1) + (rr % M) + (M - 1) * (2 * M - 1) + (M - 1);
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

    int it = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++it) {
        const int stage = it & 1;
        uint8_t *sb = stage_base + stage * T::kStageBytes;

        // ---- thread 0: S = Q K^T for this tile, then the next tile's loads
        if (tid == 0 && !abort_flag) {
            if (mbar_wait(&bar_load[stage], load_uses[stage] & 1, wc, kStatusTimeoutLoad,
                          &abort_flag)) {
                loads_pending &= ~(1u << stage);
                ++load_uses[stage];
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t a = smem_desc(smem_u32(sb) + kk * 32, 16, T::kSbo, T::kSwz);
                    const uint64_t b =
                        smem_desc(smem_u32(sb + T::kOperBytes) + kk * 32, 16, T::kSbo, T::kSwz);
                    mma_bf16_ss(tmem, a, b, kIdescS, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bar_s);
                mma_bar_pending = &bar_s;
                mma_parity_pending = it & 1;
                // the other stage's Q buffer staged the previous tile's output:
                // its TMA store must have read it before the next load lands there
                const int next = tile + gridDim.x;
                if (next < tiles) {
                    bulk_wait_read_all();
                    issue_load(next, stage ^ 1);
                }
            }
        }

        // ---- every thread: softmax of its own row over its own unit's keys
        const int unit = 2 * tile + slot;
        const bool row_ok = (r < T::kN) && (unit < units);
        float l = 1.f;
        if (mbar_wait(&bar_s, it & 1, wc, kStatusTimeoutMma, &abort_flag)) {
            if (tid == 0) mma_bar_pending = nullptr;
            tc_fence_after();
            uint32_t s0[32], s1[32];
            const uint32_t taddr = tmem + lane_off + slot * 64;
            tmem_ld32(taddr, s0);
            tmem_ld32(taddr + 32, s1);
            tmem_ld_wait();
            tmem_ready(s0);
            tmem_ready(s1);
            const int uu = unit < units ? unit : 0;
            const int h = uu - fast_div(heads, uu) * nheads;
            const float *bp = bias_s + h * T::kNBPad + bias_base;
            float x[T::kN];
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < T::kN; ++j) {
                constexpr int kSide = 2 * M - 1;
                const int kterm = (j / M) * kSide + (j % M);
                const float s = __uint_as_float(j < 32 ? s0[j & 31] : s1[j & 31]);
                x[j] = fmaf(s, scale_log2e, bp[-kterm]);
                mx = fmaxf(mx, x[j]);
            }
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < T::kN; ++j) {
                x[j] = ex2_approx(x[j] - mx);
                sum += x[j];
            }
            l = sum;
            // P over the scores: this slot's 32 columns, then 32 zero columns
            // for the other slot's keys (read above, not needed any more)
            uint32_t w[32], z[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const int j0 = 2 * c;
                const float a = (row_ok && j0 < T::kN) ? x[j0 < T::kN ? j0 : 0] : 0.f;
                const float b = (row_ok && j0 + 1 < T::kN) ? x[j0 + 1 < T::kN ? j0 + 1 : 0] : 0.f;
                w[c] = pack_bf16x2(a, b);
                z[c] = 0u;
            }
            tmem_st32(tmem + lane_off + slot * 32, w);
            tmem_st32(tmem + lane_off + (slot ^ 1) * 32, z);
            tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- thread 0: O = P V
        if (tid == 0 && !abort_flag) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t b = smem_desc(
                    smem_u32(sb + 2 * T::kOperBytes) + kk * 16 * T::kRowBytes, 16, T::kSbo, T::kSwz);
                mma_bf16_ts(tmem + T::kColO, tmem + kk * 8, b, kIdescO, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bar_o);
            mma_bar_pending = &bar_o;
            mma_parity_pending = it & 1;
        }

        // ---- every thread: normalise its row and stage it for the TMA store
        if (mbar_wait(&bar_o, it & 1, wc, kStatusTimeoutMma, &abort_flag)) {
            if (tid == 0) mma_bar_pending = nullptr;
            tc_fence_after();
            const float inv = row_ok ? 1.f / l : 0.f;
            // the output tile is staged in this stage's Q buffer (Q is dead
            // once S is formed)
            const uint32_t orow = smem_u32(sb) + tid * T::kRowBytes;
#pragma unroll
            for (int half = 0; half < D / 32; ++half) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + T::kColO + half * 32, o);
                tmem_ld_wait(o);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int chunk = half * 4 + c;
                    const int phys = (D == 32) ? (chunk ^ ((tid >> 1) & 3)) : (chunk ^ (tid & 7));
                    st_shared_v4(orow + (phys << 4),
                                 pack_bf16x2(__uint_as_float(o[8 * c + 0]) * inv,
                                             __uint_as_float(o[8 * c + 1]) * inv),
                                 pack_bf16x2(__uint_as_float(o[8 * c + 2]) * inv,
                                             __uint_as_float(o[8 * c + 3]) * inv),
                                 pack_bf16x2(__uint_as_float(o[8 * c + 4]) * inv,
                                             __uint_as_float(o[8 * c + 5]) * inv),
                                 pack_bf16x2(__uint_as_float(o[8 * c + 6]) * inv,
                                             __uint_as_float(o[8 * c + 7]) * inv));
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        const int aborted = __syncthreads_or(abort_flag);
        if (aborted) break;
        if (tid == 0) {
            if constexpr (FM) {
                const int nu = 2 * tile + 1 < units ? 2 : 1;
                for (int s2 = 0; s2 < nu; ++s2) {
                    int h, x0, y0, b;
                    unit_coords(2 * tile + s2, h, x0, y0, b);
                    tma_store_5d(&tm_o, sb + s2 * 64 * T::kRowBytes, 0, h, x0, y0, b);
                }
            } else {
                tma_store_3d(&tm_o, sb, 0, 0, 2 * tile);
            }
            bulk_commit_group();
        }
    }

    // ---- drain: nothing of this CTA may be in flight when it exits
    if (tid == 0) {
        for (int s = 0; s < 2; ++s)
            if (loads_pending & (1u << s))
                mbar_wait(&bar_load[s], load_uses[s] & 1, drain, kStatusTimeoutDrain, nullptr);
        if (mma_bar_pending != nullptr)
            mbar_wait(mma_bar_pending, mma_parity_pending, drain, kStatusTimeoutDrain, nullptr);
        bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

// The bf16 launch of pre-partitioned windows, shared by swin_window_attn_fwd
// (status = the library's allocated status word) and the no-allocation entry
// point (status = a word of its fixed array, cleared on `stream` first because
// that array keeps the previous call's contents).
template <int M, int D>
cudaError_t launch_swin_tmpl(const SwinBf16Args &a, unsigned *status, bool clear_status,
                             cudaStream_t stream) {
    using T = SwinTile<M, D>;
    if (a.heads > T::kMaxHeads) return cudaErrorInvalidValue;
    const int units = a.num_windows * a.heads;
    const int tiles = (units + 1) / 2;
    const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(T::kN),
                              static_cast<uint64_t>(units)};
    const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2,
                                 static_cast<uint64_t>(T::kN) * D * 2};
    const uint32_t box[3] = {static_cast<uint32_t>(D), 64, 2};
    const CUtensorMapSwizzle swz =
        (D == 32) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    CUtensorMap tq, tk, tv, to;
    if (!encode_tensor_map(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.q, dims, strides, box, swz) ||
        !encode_tensor_map(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.k, dims, strides, box, swz) ||
        !encode_tensor_map(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.v, dims, strides, box, swz) ||
        !encode_tensor_map(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.out, dims, strides, box, swz))
        return cudaErrorInvalidValue;
    const int smem = T::smem_bytes(a.heads);
    cudaError_t err = cudaFuncSetAttribute(swin_bf16_kernel<M, D, false>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           T::smem_bytes(T::kMaxHeads));
    if (err != cudaSuccess) return err;
    if (status == nullptr) return cudaErrorMemoryAllocation;
    if (clear_status) {
        err = cudaMemsetAsync(status, 0, sizeof(unsigned), stream);
        if (err != cudaSuccess) return err;
    }
    const int grid = std::min(tiles, sm_count() * T::kCtasPerSm);
    const float scale_log2e = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D))) * kLog2e;
    return launch_pdl(swin_bf16_kernel<M, D, false>, dim3(grid), dim3(128), smem, stream, tq, tk, tv, to,
                      a.bias_table, make_fastdiv(a.heads), units, tiles, make_fastdiv(1),
                      make_fastdiv(1), scale_log2e, WaitCtl{status, kDefaultWaitNs});
}

template <int M, int D>
cudaError_t launch_swin_fmap_tmpl(const SwinFmapArgs &a, cudaStream_t stream) {
    using T = SwinTile<M, D>;
    if (a.heads > T::kMaxHeads) return cudaErrorInvalidValue;
    const int wins_y = a.img_h / M, wins_x = a.img_w / M;
    const int units = a.batch * wins_y * wins_x * a.heads;
    const int tiles = (units + 1) / 2;
    const uint64_t row = static_cast<uint64_t>(a.heads) * D * 2;  // bytes per pixel
    const uint64_t dims[5] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.heads),
                              static_cast<uint64_t>(a.img_w), static_cast<uint64_t>(a.img_h),
                              static_cast<uint64_t>(a.batch)};
    const uint64_t strides[4] = {static_cast<uint64_t>(D) * 2, row, row * a.img_w,
                                 row * a.img_w * a.img_h};
    const uint32_t box[5] = {static_cast<uint32_t>(D), 1, M, M, 1};
    const CUtensorMapSwizzle swz =
        (D == 32) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tq, tk, tv, to;
    if (!encode_tensor_map(&tq, bf, 5, a.q, dims, strides, box, swz) ||
        !encode_tensor_map(&tk, bf, 5, a.k, dims, strides, box, swz) ||
        !encode_tensor_map(&tv, bf, 5, a.v, dims, strides, box, swz) ||
        !encode_tensor_map(&to, bf, 5, a.out, dims, strides, box, swz))
        return cudaErrorInvalidValue;
    const int smem = T::smem_bytes(a.heads);
    cudaError_t err = cudaFuncSetAttribute(swin_bf16_kernel<M, D, true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           T::smem_bytes(T::kMaxHeads));
    if (err != cudaSuccess) return err;
    unsigned *status = device_status_word();
    if (status == nullptr) return cudaErrorMemoryAllocation;
    const int grid = std::min(tiles, sm_count() * T::kCtasPerSm);
    const float scale_log2e = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D))) * kLog2e;
    return launch_pdl(swin_bf16_kernel<M, D, true>, dim3(grid), dim3(128), smem, stream, tq, tk,
                      tv, to, a.bias_table, make_fastdiv(a.heads), units, tiles,
                      make_fastdiv(wins_y), make_fastdiv(wins_x), scale_log2e,
                      WaitCtl{status, kDefaultWaitNs});
}

}  // namespace

cudaError_t launch_swin_bf16(const SwinBf16Args &a, cudaStream_t stream) {
    if (a.M == 7 && a.d == 32) return launch_swin_tmpl<7, 32>(a, device_status_word(), false, stream);
    if (a.M == 7 && a.d == 64) return launch_swin_tmpl<7, 64>(a, device_status_word(), false, stream);
    return cudaErrorInvalidValue;
}

int swin_bf16_max_heads() { return SwinTile<7, 32>::kMaxHeads < SwinTile<7, 64>::kMaxHeads
                                       ? SwinTile<7, 32>::kMaxHeads : SwinTile<7, 64>::kMaxHeads; }

cudaError_t launch_swin_bf16_fmap(const SwinFmapArgs &a, cudaStream_t stream) {
    if (a.M == 7 && a.d == 32) return launch_swin_fmap_tmpl<7, 32>(a, stream);
    if (a.M == 7 && a.d == 64) return launch_swin_fmap_tmpl<7, 64>(a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace vta

// ---------------------------------------------------------------------------
// swin_window_attn_fwd_noalloc: the same bf16 Swin kernel for callers that
// must not allocate device memory.
//
// The regular entry point keeps its kernels' status word (the only scratch
// the kernel writes besides its output) in a 256-byte buffer that the library
// allocates with cudaMalloc on the first call on each device. Some callers
// cannot allow that allocation: code that must not call cudaMalloc once it is
// running (real-time or certified pipelines, processes whose memory is fully
// reserved up front by a pooling allocator or a framework), and code that
// only ever runs inside a region where allocation is forbidden. This variant
// keeps that scratch in a fixed, file-scope device array instead, so a call
// allocates nothing.
// ---------------------------------------------------------------------------
namespace vta {
namespace {

// Scratch of the no-allocation variant: kNoAllocWords 32-bit words (256 bytes)
// of device memory that every GPU loading this library holds until the
// process exits. A call uses word 0 as its kernel's status word.
constexpr int kNoAllocWords = 64;
constexpr int kNoAllocWordsPerCall = 1;
static __device__ __align__(256) unsigned g_swin_noalloc_scratch[kNoAllocWords];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
unsigned *g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device. In host code the
// array's name is only a host-side stand-in, so its device address is looked
// up once per device (with that device current) and cached.
cudaError_t noalloc_scratch(unsigned **out) {
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        err = cudaGetSymbolAddress(&ptr, g_swin_noalloc_scratch);
        if (err != cudaSuccess) return err;
        g_noalloc_ptr[dev] = static_cast<unsigned *>(ptr);
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace vta

extern "C" int swin_window_attn_fwd_noalloc(const void *q, const void *k, const void *v,
                                            const float *bias_table, int num_windows,
                                            int heads, int M, int d, void *out,
                                            void *stream) {
    using namespace vta;
    if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || bias_table == nullptr)
        return RPE_ERR_INVALID_ARG;
    if (num_windows < 1 || heads < 1 || M < 1 || d < 1) return RPE_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, out, bias_table};
    for (const void *p : ptrs)
        if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0) return RPE_ERR_INVALID_ARG;
    const long long units = static_cast<long long>(num_windows) * heads;
    if (M != 7 || (d != 32 && d != 64) || heads > swin_bf16_max_heads() || units >= (1LL << 30))
        return RPE_ERR_UNSUPPORTED;
    // every call needs kNoAllocWordsPerCall words of the fixed array, whatever its shape
    if (kNoAllocWordsPerCall > kNoAllocWords) return RPE_ERR_UNSUPPORTED;
    unsigned *status = nullptr;
    if (noalloc_scratch(&status) != cudaSuccess) return RPE_ERR_CUDA;
    SwinBf16Args a{q, k, v, out, bias_table, num_windows, heads, M, d};
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t err = (d == 32) ? launch_swin_tmpl<7, 32>(a, status, true, st)
                                : launch_swin_tmpl<7, 64>(a, status, true, st);
    return err == cudaSuccess ? RPE_OK : RPE_ERR_CUDA;
}

extern "C" int swin_noalloc_status(unsigned *status, int clear) {
    using namespace vta;
    if (status == nullptr) return RPE_ERR_INVALID_ARG;
    unsigned *word = nullptr;
    if (noalloc_scratch(&word) != cudaSuccess) return RPE_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return RPE_ERR_CUDA;
    unsigned host = 0;
    if (cudaMemcpyFromSymbol(&host, g_swin_noalloc_scratch, sizeof(host), 0,
                             cudaMemcpyDeviceToHost) != cudaSuccess)
        return RPE_ERR_CUDA;
    if (clear && host != 0) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_swin_noalloc_scratch, &zero, sizeof(zero), 0,
                               cudaMemcpyHostToDevice) != cudaSuccess)
            return RPE_ERR_CUDA;
    }
    *status = host;
    return host ? RPE_ERR_TIMEOUT : RPE_OK;
}

extern "C" int swin_noalloc_status_word(unsigned **word) {
    using namespace vta;
    if (word == nullptr) return RPE_ERR_INVALID_ARG;
    unsigned *p = nullptr;
    if (noalloc_scratch(&p) != cudaSuccess) return RPE_ERR_CUDA;
    *word = p;
    return RPE_OK;
}
