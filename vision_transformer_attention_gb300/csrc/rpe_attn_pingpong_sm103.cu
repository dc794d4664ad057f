// rpe_attn_pingpong_sm103.cu -- iRPE contextual-key attention (or plain
// attention) on sm_103a with two softmax warpgroups per CTA.
//
// Same computation as rpe_attn_sm103.cu for the key term ("Rethinking and
// Improving Relative Position Encoding for Vision Transformer", eqs. 13, 15
// and the efficient form of eqs. 26-28): logits (q_i.k_j + q_i.R^K[id])/sqrt(d)
// with QR = Q R^K^T formed once per query tile on the tensor core and read per
// score by bucket id, softmax, P V. This kernel is the fast path for the
// key-term-only and no-term requests on grids of width W in {14, 56}:
//
//   * Two softmax warpgroups, each owning a 128-row query tile of the same
//     (batch, head) slice, share every K/V tile and take turns on the tensor
//     core: while one converts its scores, the other's QK^T or PV runs.
//   * P is written back into the score columns of tensor memory as bf16 and
//     the PV product reads its A operand from there (no shared-memory copy).
//   * Key tiles hold whole grid rows (126 keys for W = 14, 112 for W = 56), so
//     within a tile the offset-table position of key jj is a compile-time
//     constant: each score's bucket id is one shared-memory byte load at an
//     immediate offset from a per-tile base.
//   * Work items (slice, pair of query tiles) are ordered full pairs first so
//     that the static round-robin assignment stays balanced.
//
// Warps 0-3: softmax warpgroup 0; 4-7: warpgroup 1; warpgroup 2 (warps 8-11):
// warp 8 TMA producer, warp 9 MMA issuer, warps 10-11 idle. Tensor memory
// (512 columns): warpgroup w owns [256w, 256w + 256): scores / P at +0
// (128 columns), O at +128 (64), QR at +192 (64).
#include "vta_internal.h"
#include "sm103_ptx.cuh"

#include <algorithm>
#include <cmath>

namespace vta {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kD = 64;
constexpr int kTileBytes = 128 * 128;  // one 128-row x 64-column bf16 tile
constexpr int kThreads = 384;
// Register split (launch: 384 threads x 168 = 64,512): control warpgroup 96,
// softmax warpgroups 200 -> 128 x 96 + 256 x 200 = 63,488.
constexpr int kRegsControl = 96;
constexpr int kRegsSoftmax = 200;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * 168, "register split");
constexpr float kRescaleLog2 = 8.f;
constexpr int kMaxStages = 3;

template <int W>
struct Geo {
    static constexpr int R = 128 / W;               // grid rows per key tile
    static constexpr int KT = R * W;                // keys per tile
    static constexpr int NS = (KT + 15) / 16 * 16;  // N of QK^T, K of PV
    static constexpr int COLS = 2 * W - 1;          // offset-table row length
};

struct PPParams {
    int N, H, nb, nkt, qtiles, pairs_full, slices, items, nst;
    uint32_t off_q, off_kv, off_rk, off_qr, off_lut;
    int lut_len, lut_pad;
    const int32_t *lut;
    __nv_bfloat16 *out;
    float c;  // log2(e) / sqrt(d)
    WaitCtl wc;
};

struct PPBars {
    uint64_t tab_full, q_full, q_empty;
    uint64_t kv_full[kMaxStages], kv_empty[kMaxStages];
    uint64_t qr_full[2], qr_empty[2], s_full[2], p_full[2], o_full[2], o_empty[2];
};

struct Item {
    int slice, qt0;
    bool has_b;
};

// Full pairs of query tiles first (slice-major), then the odd last tiles.
__device__ __forceinline__ Item decode_item(const PPParams &P, int item) {
    Item r;
    const int nfull = P.slices * P.pairs_full;
    if (item < nfull) {
        r.slice = item / P.pairs_full;
        r.qt0 = 2 * (item % P.pairs_full);
        r.has_b = true;
    } else {
        r.slice = item - nfull;
        r.qt0 = P.qtiles - 1;
        r.has_b = false;
    }
    return r;
}

// AND-reduction over the 128 threads of softmax warpgroup wg (named barrier 1 + wg).
__device__ __forceinline__ bool wg_red_and(int wg, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(1 + wg)
        : "memory");
    return r != 0;
}

// One 32-key chunk of a tile for one query row: logits in log2 units
// (x = S c + QR'[id]; keys past the grid -- only in the last tile -- are set
// to -inf), an online update of the row's reference max m and sum l, and the
// chunk's probabilities written into tensor memory as 16 columns of bf16
// pairs over the already-read scores. The 32 bucket ids are loaded first and
// the 32 QR' values next, so the two dependent shared-memory loads of each
// score overlap those of the other 31.
//
// The reference max moves only when the chunk's max exceeds it by more than
// 2^8 (rare after the first chunk); then O (earlier tiles) and the P columns of
// this tile's earlier chunks are rescaled, warp-uniformly, in tensor memory.
template <int W, bool HK, int Q>
__device__ __forceinline__ void softmax_chunk(uint32_t tS, uint32_t tO, const uint8_t *lut_t,
                                              const float *qr_t, float c, int nvalid,
                                              bool o_live, float &m, float &l) {
    using G = Geo<W>;
    if constexpr (Q * 32 < G::KT) {
        uint32_t s[32];
        tmem_ld32(tS + Q * 32, s);
        tmem_ld_wait();
        float x[32];
        if constexpr (HK) {
            int id[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int jj = Q * 32 + j;
                const int C = (jj / W) * G::COLS + (jj % W);
                id[j] = (jj < G::KT) ? lut_t[-C] : 0;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = qr_t[id[j] * 128];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int jj = Q * 32 + j;
                x[j] = (jj < G::KT) ? fmaf(__uint_as_float(s[j]), c, x[j]) : -INFINITY;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int jj = Q * 32 + j;
                x[j] = (jj < G::KT) ? __uint_as_float(s[j]) * c : -INFINITY;
            }
        }
        if (Q * 32 + 32 > nvalid) {  // the chunk reaches past the grid's last row
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (Q * 32 + j >= nvalid) x[j] = -INFINITY;
        }
        float cmax = x[0];
#pragma unroll
        for (int j = 1; j < 32; ++j) cmax = fmaxf(cmax, x[j]);
        float alpha = 1.f;
        if (cmax > m + kRescaleLog2) {
            alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - cmax);
            m = cmax;
            l *= alpha;
        }
        if ((o_live || Q > 0) && __any_sync(~0u, alpha < 1.f)) {
            tmem_st_wait();
            if (o_live) {
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t o[16];
                    tmem_ld16(tO + q * 16, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st16(tO + q * 16, o);
                }
            }
#pragma unroll 1
            for (int q = 0; q < Q; ++q) {
                uint32_t pp[16];
                tmem_ld16(tS + q * 16, pp);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float lo = __uint_as_float(pp[e] << 16) * alpha;
                    const float hi = __uint_as_float(pp[e] & 0xFFFF0000u) * alpha;
                    pp[e] = pack_bf16x2(lo, hi);
                }
                tmem_st16(tS + q * 16, pp);
            }
        }
        float sum = 0.f;
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float p0 = ex2_approx(x[2 * e] - m);
            const float p1 = ex2_approx(x[2 * e + 1] - m);
            sum += p0 + p1;
            pk[e] = pack_bf16x2(p0, p1);
        }
        l += sum;
        tmem_st16(tS + Q * 16, pk);
    }
}

template <int W, bool HK>
__global__ void __launch_bounds__(kThreads, 1)
    rpe_pingpong_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_rk, const PPParams P) {
    using G = Geo<W>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ PPBars bars;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const WaitCtl &wc = P.wc;
    const WaitCtl drain{wc.status, kDefaultWaitNs};

    uint8_t *sQ = smem + P.off_q;    // two query tiles
    uint8_t *sKV = smem + P.off_kv;  // stage s: K at 2s tiles, V at 2s + 1
    uint8_t *sRK = smem + P.off_rk;
    float *sQR = reinterpret_cast<float *>(smem + P.off_qr);  // [2][nb][128]
    uint8_t *sLut = smem + P.off_lut + P.lut_pad;

    if (tid == 0) {
        mbar_init(&bars.tab_full, 1);
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.q_empty, 1);
        for (int i = 0; i < kMaxStages; ++i) {
            mbar_init(&bars.kv_full[i], 1);
            mbar_init(&bars.kv_empty[i], 1);
        }
        for (int w = 0; w < 2; ++w) {
            mbar_init(&bars.qr_full[w], 1);
            mbar_init(&bars.qr_empty[w], 128);
            mbar_init(&bars.s_full[w], 1);
            mbar_init(&bars.p_full[w], 128);
            mbar_init(&bars.o_full[w], 1);
            mbar_init(&bars.o_empty[w], 128);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&tmem_base_s, 512);
    if (HK) {
        // offset table as bytes, ids clamped into [0, nb). Keys past the last
        // grid row (masked later) index up to lut_pad bytes before the table;
        // those bytes hold bucket 0 so every read stays in bounds.
        for (int e = tid; e < P.lut_pad; e += kThreads) sLut[e - P.lut_pad] = 0;
        for (int e = tid; e < P.lut_len; e += kThreads) {
            const int id = __ldg(P.lut + e);
            sLut[e] = static_cast<uint8_t>(id < 0 ? 0 : (id >= P.nb ? P.nb - 1 : id));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (warp >= 8) {
        regs_dealloc<kRegsControl>();
        if (warp == 8) {
            // -------------------------------------------- TMA producer
            if (lane == 0) {
                prefetch_tmap(&tm_q);
                prefetch_tmap(&tm_k);
                prefetch_tmap(&tm_v);
                if (HK) {
                    mbar_arrive_expect_tx(&bars.tab_full, kTileBytes / 2);
                    tma_load_2d(sRK, &tm_rk, &bars.tab_full, 0, 0);
                }
                int g = 0, it = 0, last_q = -1;
                int last_use[kMaxStages] = {-1, -1, -1};
                bool ok = true;
                for (int item = blockIdx.x; ok && item < P.items; item += gridDim.x, ++it) {
                    const Item I = decode_item(P, item);
                    if (!(ok = mbar_wait(&bars.q_empty, (it & 1) ^ 1, wc, kStatusTimeoutSync,
                                         &abort_flag)))
                        break;
                    mbar_arrive_expect_tx(&bars.q_full, (I.has_b ? 2 : 1) * kTileBytes);
                    tma_load_3d(sQ, &tm_q, &bars.q_full, 0, I.qt0 * 128, I.slice);
                    if (I.has_b)
                        tma_load_3d(sQ + kTileBytes, &tm_q, &bars.q_full, 0, (I.qt0 + 1) * 128,
                                    I.slice);
                    last_q = it;
                    for (int kt = 0; kt < P.nkt; ++kt, ++g) {
                        const int st = g % P.nst, use = g / P.nst;
                        if (!(ok = mbar_wait(&bars.kv_empty[st], (use & 1) ^ 1, wc,
                                             kStatusTimeoutSync, &abort_flag)))
                            break;
                        uint8_t *kb = sKV + st * 2 * kTileBytes;
                        mbar_arrive_expect_tx(&bars.kv_full[st], 2 * kTileBytes);
                        tma_load_3d(kb, &tm_k, &bars.kv_full[st], 0, kt * G::KT, I.slice);
                        tma_load_3d(kb + kTileBytes, &tm_v, &bars.kv_full[st], 0, kt * G::KT,
                                    I.slice);
                        last_use[st] = use;
                    }
                }
                // drain: the most recent load on every barrier has landed
                if (HK) mbar_wait(&bars.tab_full, 0, drain, kStatusTimeoutDrain, nullptr);
                if (last_q >= 0)
                    mbar_wait(&bars.q_full, last_q & 1, drain, kStatusTimeoutDrain, nullptr);
                for (int st = 0; st < kMaxStages; ++st)
                    if (last_use[st] >= 0)
                        mbar_wait(&bars.kv_full[st], last_use[st] & 1, drain, kStatusTimeoutDrain,
                                  nullptr);
            }
            __syncwarp();
        } else if (warp == 9) {
            // -------------------------------------------- MMA issuer
            if (lane == 0) {
                constexpr uint32_t kIdS = idesc_bf16(128, G::NS, false, false);
                constexpr uint32_t kIdQR = idesc_bf16(128, 64, false, false);
                constexpr uint32_t kIdO = idesc_bf16(128, 64, false, true);
                uint64_t *last_bar = nullptr;
                uint32_t last_par = 0;
                auto commit = [&](uint64_t *bar, uint32_t parity) {
                    mma_commit(bar);
                    last_bar = bar;
                    last_par = parity;
                };
                auto issue_s = [&](int w, int st) {
                    const uint32_t aQ = smem_u32(sQ + w * kTileBytes);
                    const uint32_t aK = smem_u32(sKV + st * 2 * kTileBytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ss(tmem + w * 256, smem_desc(aQ + kk * 32, 16, 1024, kSwizzle128B),
                                    smem_desc(aK + kk * 32, 16, 1024, kSwizzle128B), kIdS, kk > 0);
                };
                bool ok = true;
                if (HK) ok = mbar_wait(&bars.tab_full, 0, wc, kStatusTimeoutLoad, &abort_flag);
                int g = 0, it = 0;
                int ci[2] = {0, 0}, cs[2] = {0, 0}, cp[2] = {0, 0};
                for (int item = blockIdx.x; ok && item < P.items; item += gridDim.x, ++it) {
                    const Item I = decode_item(P, item);
                    const int nw = I.has_b ? 2 : 1;
                    if (!(ok = mbar_wait(&bars.q_full, it & 1, wc, kStatusTimeoutLoad, &abort_flag)))
                        break;
                    tc_fence_after();
                    if (HK) {
                        for (int w = 0; w < nw && ok; ++w) {
                            if (!(ok = mbar_wait(&bars.qr_empty[w], (ci[w] & 1) ^ 1, wc,
                                                 kStatusTimeoutSync, &abort_flag)))
                                break;
                            tc_fence_after();
                            const uint32_t aQ = smem_u32(sQ + w * kTileBytes);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_bf16_ss(tmem + w * 256 + 192,
                                            smem_desc(aQ + kk * 32, 16, 1024, kSwizzle128B),
                                            smem_desc(smem_u32(sRK) + kk * 32, 16, 1024,
                                                      kSwizzle128B),
                                            kIdQR, kk > 0);
                            commit(&bars.qr_full[w], ci[w] & 1);
                        }
                        if (!ok) break;
                    }
                    {
                        const int st = g % P.nst;
                        if (!(ok = mbar_wait(&bars.kv_full[st], (g / P.nst) & 1, wc,
                                             kStatusTimeoutLoad, &abort_flag)))
                            break;
                        tc_fence_after();
                        for (int w = 0; w < nw; ++w) {
                            issue_s(w, st);
                            commit(&bars.s_full[w], cs[w] & 1);
                            ++cs[w];
                        }
                        if (P.nkt == 1) commit(&bars.q_empty, it & 1);
                    }
                    for (int kt = 0; ok && kt < P.nkt; ++kt, ++g) {
                        const int st = g % P.nst;
                        const bool last = kt == P.nkt - 1;
                        const int stn = (g + 1) % P.nst;
                        for (int w = 0; w < nw; ++w) {
                            if (!(ok = mbar_wait(&bars.p_full[w], cp[w] & 1, wc,
                                                 kStatusTimeoutSync, &abort_flag)))
                                break;
                            ++cp[w];
                            if (kt == 0 && !(ok = mbar_wait(&bars.o_empty[w], (ci[w] & 1) ^ 1, wc,
                                                            kStatusTimeoutSync, &abort_flag)))
                                break;
                            tc_fence_after();
                            const uint32_t aV = smem_u32(sKV + st * 2 * kTileBytes + kTileBytes);
#pragma unroll
                            for (int kk = 0; kk < G::NS / 16; ++kk)
                                mma_bf16_ts(tmem + w * 256 + 128, tmem + w * 256 + kk * 8,
                                            smem_desc(aV + kk * 2048, 16, 1024, kSwizzle128B), kIdO,
                                            (kt > 0 || kk > 0) ? 1u : 0u);
                            if (last) {
                                commit(&bars.o_full[w], ci[w] & 1);
                            } else {
                                // this warpgroup's next scores overwrite its P only after
                                // the P V above (tcgen05.mma from one thread run in order)
                                if (w == 0 &&
                                    !(ok = mbar_wait(&bars.kv_full[stn], ((g + 1) / P.nst) & 1, wc,
                                                     kStatusTimeoutLoad, &abort_flag)))
                                    break;
                                issue_s(w, stn);
                                commit(&bars.s_full[w], cs[w] & 1);
                                ++cs[w];
                                if (w == nw - 1 && kt + 1 == P.nkt - 1) commit(&bars.q_empty, it & 1);
                            }
                        }
                        if (!ok) break;
                        commit(&bars.kv_empty[st], (g / P.nst) & 1);
                    }
                    for (int w = 0; w < nw; ++w) ++ci[w];
                }
                // drain: tcgen05 work completes in order, so the last commit covers it all
                if (last_bar != nullptr)
                    mbar_wait(last_bar, last_par, drain, kStatusTimeoutDrain, nullptr);
            }
            __syncwarp();
        }
    } else {
        regs_alloc<kRegsSoftmax>();
        // ------------------------------------------------ softmax warpgroups
        const int wg = warp >> 2;
        const int lw = warp & 3;
        const int t = tid & 127;
        const uint32_t lane_off = static_cast<uint32_t>(lw * 32) << 16;
        const uint32_t tS = tmem + wg * 256, tO = tS + 128, tQR = tS + 192;
        float *qr_t = sQR + wg * P.nb * 128 + t;
        int it_w = 0, s_cnt = 0;
        for (int item = blockIdx.x; item < P.items; item += gridDim.x) {
            const Item I = decode_item(P, item);
            if (wg == 1 && !I.has_b) continue;
            const int qt = I.qt0 + wg;
            const int i = qt * 128 + t;
            const bool warp_active = qt * 128 + lw * 32 < P.N;
            const int ic = i < P.N ? i : P.N - 1;
            const int base_i = (ic / W) * G::COLS + (ic % W) + (P.H - 1) * G::COLS + (W - 1);
            if (HK) {
                bool ok = __all_sync(~0u, mbar_wait(&bars.qr_full[wg], it_w & 1, wc,
                                                    kStatusTimeoutMma, &abort_flag));
                if (!wg_red_and(wg, ok)) break;
                tc_fence_after();
                if (warp_active) {
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tQR + lane_off, r0);
                    tmem_ld32(tQR + lane_off + 32, r1);
                    tmem_ld_wait();
#pragma unroll
                    for (int b = 0; b < 64; ++b)
                        if (b < P.nb)
                            qr_t[b * 128] = __uint_as_float(b < 32 ? r0[b & 31] : r1[b & 31]) * P.c;
                }
                tc_fence_before();
                mbar_arrive(&bars.qr_empty[wg]);
            }
            float m = -INFINITY, l = 0.f;
            bool aborted = false;
            for (int kt = 0; kt < P.nkt; ++kt) {
                bool ok = __all_sync(~0u, mbar_wait(&bars.s_full[wg], s_cnt & 1, wc,
                                                    kStatusTimeoutMma, &abort_flag));
                ++s_cnt;
                if (!wg_red_and(wg, ok)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                if (warp_active) {
                    const int rj0 = kt * G::R;
                    const int nvalid = min(G::R, P.H - rj0) * W;
                    const uint8_t *lut_t = sLut + (base_i - rj0 * G::COLS);
                    const uint32_t tSl = tS + lane_off, tOl = tO + lane_off;
                    softmax_chunk<W, HK, 0>(tSl, tOl, lut_t, qr_t, P.c, nvalid, kt > 0, m, l);
                    softmax_chunk<W, HK, 1>(tSl, tOl, lut_t, qr_t, P.c, nvalid, kt > 0, m, l);
                    softmax_chunk<W, HK, 2>(tSl, tOl, lut_t, qr_t, P.c, nvalid, kt > 0, m, l);
                    softmax_chunk<W, HK, 3>(tSl, tOl, lut_t, qr_t, P.c, nvalid, kt > 0, m, l);
                    tmem_st_wait();
                }
                tc_fence_before();
                mbar_arrive(&bars.p_full[wg]);
            }
            if (!wg_red_and(wg, !aborted)) break;
            bool ok = __all_sync(~0u, mbar_wait(&bars.o_full[wg], it_w & 1, wc, kStatusTimeoutMma,
                                                &abort_flag));
            if (!wg_red_and(wg, ok)) break;
            tc_fence_after();
            uint32_t o0[32], o1[32];
            if (warp_active) {
                tmem_ld32(tO + lane_off, o0);
                tmem_ld32(tO + lane_off + 32, o1);
                tmem_ld_wait();
            }
            tc_fence_before();
            mbar_arrive(&bars.o_empty[wg]);
            if (i < P.N) {
                const float inv = 1.f / l;
                uint4 *dst = reinterpret_cast<uint4 *>(P.out + (static_cast<size_t>(I.slice) * P.N + i) * kD);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t *src = c < 4 ? o0 + 8 * c : o1 + 8 * (c - 4);
                    uint4 v;
                    v.x = pack_bf16x2(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv);
                    v.y = pack_bf16x2(__uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv);
                    v.z = pack_bf16x2(__uint_as_float(src[4]) * inv, __uint_as_float(src[5]) * inv);
                    v.w = pack_bf16x2(__uint_as_float(src[6]) * inv, __uint_as_float(src[7]) * inv);
                    dst[c] = v;
                }
            }
            ++it_w;
        }
    }
    tc_fence_before();
    asm volatile("barrier.sync 0;" ::: "memory");
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

template <int W, bool HK>
cudaError_t launch_pp(const RpeBf16Args &a, cudaStream_t stream) {
    using G = Geo<W>;
    PPParams p{};
    const int N = a.H * a.W;
    p.N = N;
    p.H = a.H;
    p.nb = a.num_buckets;
    p.nkt = (a.H + G::R - 1) / G::R;
    p.qtiles = (N + 127) / 128;
    p.pairs_full = p.qtiles / 2;
    p.slices = a.B * a.heads;
    p.items = p.slices * p.pairs_full + ((p.qtiles & 1) ? p.slices : 0);
    p.lut_len = (2 * a.H - 1) * (2 * a.W - 1);
    p.lut_pad = static_cast<int>(align_up(G::R * G::COLS, 16));
    p.lut = a.lut;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.c = static_cast<float>(kLog2e / std::sqrt(static_cast<double>(kD)));
    const uint32_t cap = 227 * 1024 - 1024;
    uint32_t total = 0;
    for (int nst = kMaxStages; nst >= 2; --nst) {
        uint32_t off = 0;
        p.off_q = off;
        off += 2 * kTileBytes;
        p.off_kv = off;
        off += nst * 2 * kTileBytes;
        p.off_rk = off;
        if (HK) off += kTileBytes / 2;
        p.off_qr = off;
        if (HK) off += align_up(2 * p.nb * 512, 1024);
        p.off_lut = off;
        if (HK) off += p.lut_pad + align_up(p.lut_len, 16);
        total = 1024 + off;
        p.nst = nst;
        if (total <= cap) break;
    }
    if (total > cap) return cudaErrorInvalidValue;
    unsigned *status = device_status_word();
    if (status == nullptr) return cudaErrorMemoryAllocation;
    p.wc = WaitCtl{status, kDefaultWaitNs};
    const uint64_t dims[3] = {kD, static_cast<uint64_t>(N), static_cast<uint64_t>(p.slices)};
    const uint64_t strides[2] = {kD * 2, static_cast<uint64_t>(N) * kD * 2};
    const uint32_t box[3] = {kD, 128, 1};
    const uint64_t tdims[2] = {kD, static_cast<uint64_t>(a.num_buckets)};
    const uint64_t tstrides[1] = {kD * 2};
    const uint32_t tbox[2] = {kD, 64};
    const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
    CUtensorMap tq, tk, tv, trk;
    if (!encode_tensor_map(&tq, bf, 3, a.q, dims, strides, box, sw) ||
        !encode_tensor_map(&tk, bf, 3, a.k, dims, strides, box, sw) ||
        !encode_tensor_map(&tv, bf, 3, a.v, dims, strides, box, sw) ||
        !encode_tensor_map(&trk, bf, 2, HK ? a.tab_k : a.q, tdims, tstrides, tbox, sw))
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(rpe_pingpong_kernel<W, HK>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(total));
    if (err != cudaSuccess) return err;
    const int grid = std::min(p.items, sm_count());
    rpe_pingpong_kernel<W, HK><<<grid, kThreads, total, stream>>>(tq, tk, tv, trk, p);
    return cudaGetLastError();
}

}  // namespace

bool launch_rpe_bf16_pingpong(const RpeBf16Args &a, cudaStream_t stream, cudaError_t *err) {
    if (a.d != kD || (a.terms & ~1u) != 0) return false;
    const bool hk = (a.terms & 1u) != 0;
    if (a.W == 14)
        *err = hk ? launch_pp<14, true>(a, stream) : launch_pp<14, false>(a, stream);
    else if (a.W == 56)
        *err = hk ? launch_pp<56, true>(a, stream) : launch_pp<56, false>(a, stream);
    else
        return false;
    return true;
}

}  // namespace vta
