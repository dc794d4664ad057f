// rpe_attn_sm103.cu -- iRPE contextual attention on sm_103a tensor cores
// (tcgen05 + TMEM + TMA), bf16 in, fp32 accumulate.
//
// What it computes ("Rethinking and Improving Relative Position Encoding for
// Vision Transformer", Method, eqs. 13 and 15-17), per (batch, head) slice:
//     e_ij  = ( q_i.k_j + [K] q_i.R^K[id] + [Q] k_j.R^Q[id] ) / sqrt(d)
//     out_i = sum_j softmax_j(e_ij) ( v_j + [V] R^V[id] ),   id = id(i, j)
// with the contextual terms taken the efficient way of eqs. 26-28: every
// query is dotted with every bucket vector once (QR = Q R^K^T, a small
// tensor-core product per query tile), every key likewise (KR = K R^Q^T per
// key tile), and a score picks its term by bucket id; the value term sums the
// probabilities per bucket (PB) and multiplies by R^V once per query tile.
// Bucket ids come from a shared-memory copy of the offset table built by
// rpe_build_bucket_ids; no n x n bias or id map is read from global memory.
//
// Cross tables (eqs. 22-24: a row bucket a and a column bucket span + b per
// pair, their terms added) are staged with the row buckets at rows 0.. and
// the column buckets at rows 32.. of the shared-memory table, so one product
// gives both halves' QR / KR columns; the copies into shared memory then hold
// the joint entry a*span + b as the fp32 sum of the two, and the per-score
// gather is the same as for one bucket per pair. For the value term the joint
// probability sums are reduced to per-row-bucket and per-column-bucket sums
// before the PB R^V product.
//
// Structure (one CTA per SM, persistent over (slice, 128-query tile) items):
//   warp 4  TMA producer: Q tile, then 128-key K/V tiles into a ring.
//   warp 5  MMA issuer:   QR = Q R^K^T, S = Q K^T (+ KR = K R^Q^T) into one of
//                         two TMEM score buffers, O += P V, O += PB R^V.
//   warps 0-3 softmax:    one thread per query row. Reads its score row from
//                         TMEM, adds the gathered terms, keeps a running max
//                         and sum (online softmax over key tiles; the O
//                         accumulator is rescaled only when the max grows by
//                         more than 2^8, otherwise the stale max is kept),
//                         writes bf16 probabilities as the K-major A operand
//                         of P V, then normalises O and stores it.
// Hand-offs use mbarriers; every wait is bounded (see sm103_ptx.cuh).
#include "vta_internal.h"
#include "sm103_ptx.cuh"

#include <algorithm>
#include <cmath>

namespace vta {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kD = 64;           // head dim (bytes per row: 128)
constexpr int kBM = 128;         // query rows per tile
constexpr int kBN = 128;         // keys per tile
constexpr int kTileBytes = 128 * 128;  // one 128-row bf16 tile of q / k / v
constexpr int kKRStride = 65;    // floats per key row of KR in shared memory (odd)
constexpr float kRescaleLog2 = 8.f;    // keep a stale max while the new one is within 2^8

// TMEM column map (512 columns allocated: the CTA owns the whole SM)
constexpr uint32_t kColS = 0;     // two 128-column score buffers
constexpr uint32_t kColO = 256;   // 64 columns, output accumulator
constexpr uint32_t kColQR = 320;  // 64 columns, Q R^K^T
constexpr uint32_t kColKR = 384;  // two 64-column buffers, K R^Q^T

constexpr int kThreads = 192;

struct RpeParams {
    int N, H, W, nb, nkt, qtiles, items, nst;
    int cross;     // Cross tables: span (nb = span^2 joint ids); 0 otherwise
    int tab_row2;  // table row staged at shared-memory row 32: span (Cross) or 32
    int tab_heads, heads;  // tab_heads 1: tables shared by every head; heads: one per head
    int nr;        // 64-row halves of each table: 1, or 2 for 65..128 buckets (K and V terms)
    int cls;       // 1: token 0 is a class token (bucket nb - 1 for all its pairs)
    // iRPE bias mode (with HK): a scalar per bucket and head, [num_buckets, bias_heads]
    // fp32, takes the place of the contextual key term: the table a row gathers
    // from holds the item's head's scaled bias instead of its QR' product, and no
    // R^K is loaded or multiplied
    const float *bias;
    int bias_heads;
    uint32_t off_q, off_kv, off_p, off_rk, off_rq, off_rv, off_qr, off_kr, off_pb, off_kterm,
        off_lut;
    int lut_len;
    const int32_t *lut;
    __nv_bfloat16 *out;
    float c;  // log2(e) / sqrt(d)
    WaitCtl wc;
};

struct Bars {
    uint64_t tab_full, tab_empty, q_full, q_empty, qr_full, qr_empty, o_full, o_empty, p_full, p_empty;
    uint64_t kv_full[2], kv_empty[2], s_full[2], s_empty[2];
};

__device__ __forceinline__ bool bar_red_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void softmax_bar() { named_bar_sync(1, 128); }

// EXT: the extended table forms (Cross tables, 65..128 buckets in two 64-row
// halves, one table per head); the other instantiations keep the code for one
// shared table of at most 64 buckets.
template <bool HK, bool HQ, bool HV, bool EXT>
__global__ void __launch_bounds__(kThreads, 1)
    rpe_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_rk,
                    const __grid_constant__ CUtensorMap tm_rq,
                    const __grid_constant__ CUtensorMap tm_rv, const RpeParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ Bars bars;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const WaitCtl &wc = P.wc;
    const WaitCtl drain{wc.status, kDefaultWaitNs};

    uint8_t *sQ = smem + P.off_q;
    uint8_t *sKV = smem + P.off_kv;  // stage s: K at s*2*kTileBytes, V after it
    uint8_t *sP = smem + P.off_p;
    float *sQR = reinterpret_cast<float *>(smem + P.off_qr);
    float *sKR = reinterpret_cast<float *>(smem + P.off_kr);
    float *sPB = reinterpret_cast<float *>(smem + P.off_pb);
    int *sKterm = reinterpret_cast<int *>(smem + P.off_kterm);
    uint8_t *sLut = smem + P.off_lut;

    if (tid == 0) {
        mbar_init(&bars.tab_full, 1);
        mbar_init(&bars.tab_empty, 1);
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.q_empty, 1);
        mbar_init(&bars.qr_full, 1);
        mbar_init(&bars.qr_empty, 128);
        mbar_init(&bars.o_full, 1);
        mbar_init(&bars.o_empty, 128);
        mbar_init(&bars.p_full, 128);
        mbar_init(&bars.p_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.kv_full[i], 1);
            mbar_init(&bars.kv_empty[i], 1);
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.s_empty[i], 128);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&tmem_base_s, 512);
    // bucket-id table: int32 in global -> uint8 in shared memory. The call
    // checked its ids on the host (once per table); an id outside [0, bound)
    // -- the class bucket excluded -- sets the status bit and is clamped so a
    // bad table can never index past shared memory.
    {
        const int bound = P.nb - (EXT && P.cls ? 1 : 0);
        for (int e = tid; e < P.lut_len; e += kThreads) {
            const int id = __ldg(P.lut + e);
            if (id < 0 || id >= bound) atomicOr(wc.status, kStatusBadBucket);
            sLut[e] = static_cast<uint8_t>(id < 0 ? 0 : (id >= bound ? bound - 1 : id));
        }
    }
    // Class token (iRPE section 4.1): entries lut_len..2 lut_len hold the extra
    // bucket nb - 1. The class key's offset term reaches there from every patch
    // query and the class query's base reaches there for every key, so a pair
    // with token 0 reads the extra bucket through the same gather.
    if (EXT && P.cls)
        for (int e = P.lut_len + tid; e <= 2 * P.lut_len; e += kThreads)
            sLut[e] = static_cast<uint8_t>(P.nb - 1);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (warp == 4) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            uint32_t tab_bytes = 0;
            const int nr = EXT ? P.nr : 1;
            const bool rk = HK && P.bias == nullptr;  // bias mode reads no R^K
            if (rk) tab_bytes += nr * (kTileBytes / 2);
            if (HQ) tab_bytes += nr * (kTileBytes / 2);
            if (HV) tab_bytes += nr * (kTileBytes / 2);
            // each table as 32-row boxes of table `head` ([tab_heads][rows][d]):
            // rows 0.. and rows tab_row2.. (then 64.. and 96.. for a second half)
            auto load_table = [&](uint8_t *dst, const CUtensorMap *m, int head) {
                tma_load_3d(dst, m, &bars.tab_full, 0, 0, head);
                tma_load_3d(dst + 4096, m, &bars.tab_full, 0, P.tab_row2, head);
                for (int r = 2; r < 2 * nr; ++r)
                    tma_load_3d(dst + r * 4096, m, &bars.tab_full, 0, 32 * r, head);
            };
            auto load_tables = [&](int head) {
                mbar_arrive_expect_tx(&bars.tab_full, tab_bytes);
                if (rk) load_table(smem + P.off_rk, &tm_rk, head);
                if (HQ) load_table(smem + P.off_rq, &tm_rq, head);
                if (HV) load_table(smem + P.off_rv, &tm_rv, head);
            };
            // Shared tables are loaded once. Per-head tables are loaded for every
            // item once the previous item's products are done with them, after
            // the item's first K/V tile so that load is not held up.
            const bool per_head = EXT && tab_bytes != 0 && P.tab_heads > 1;
            if (tab_bytes && !per_head) load_tables(0);
            int g = 0, w = 0;
            int last_kv_use[2] = {-1, -1};
            int last_q = -1, last_tab = -1;
            for (int item = blockIdx.x; item < P.items; item += gridDim.x, ++w) {
                const int slice = item / P.qtiles, qt = item % P.qtiles;
                if (!mbar_wait(&bars.q_empty, (w & 1) ^ 1, wc, kStatusTimeoutSync, &abort_flag)) break;
                mbar_arrive_expect_tx(&bars.q_full, kTileBytes);
                tma_load_3d(sQ, &tm_q, &bars.q_full, 0, qt * kBM, slice);
                last_q = w;
                bool ok = true;
                for (int kt = 0; kt < P.nkt; ++kt, ++g) {
                    const int st = g % P.nst, use = g / P.nst;
                    if (!mbar_wait(&bars.kv_empty[st], (use & 1) ^ 1, wc, kStatusTimeoutSync,
                                   &abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t *kb = sKV + st * 2 * kTileBytes;
                    mbar_arrive_expect_tx(&bars.kv_full[st], 2 * kTileBytes);
                    tma_load_3d(kb, &tm_k, &bars.kv_full[st], 0, kt * kBN, slice);
                    tma_load_3d(kb + kTileBytes, &tm_v, &bars.kv_full[st], 0, kt * kBN, slice);
                    last_kv_use[st] = use;
                    if (per_head && kt == 0) {
                        if (w > 0 && !mbar_wait(&bars.tab_empty, (w - 1) & 1, wc, kStatusTimeoutSync,
                                                &abort_flag)) {
                            ok = false;
                            break;
                        }
                        load_tables(slice % P.heads);
                        last_tab = w;
                    }
                }
                if (!ok) break;
            }
            // drain: the most recent load on every barrier has landed
            if (tab_bytes && !per_head) mbar_wait(&bars.tab_full, 0, drain, kStatusTimeoutDrain, nullptr);
            if (last_tab >= 0) mbar_wait(&bars.tab_full, last_tab & 1, drain, kStatusTimeoutDrain, nullptr);
            if (last_q >= 0) mbar_wait(&bars.q_full, last_q & 1, drain, kStatusTimeoutDrain, nullptr);
            for (int st = 0; st < 2; ++st)
                if (last_kv_use[st] >= 0)
                    mbar_wait(&bars.kv_full[st], last_kv_use[st] & 1, drain, kStatusTimeoutDrain,
                              nullptr);
        }
        __syncwarp();
    } else if (warp == 5) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
            constexpr uint32_t kIdT = idesc_bf16(128, 64, false, false);   // Q R^K^T, K R^Q^T
            constexpr uint32_t kIdO = idesc_bf16(128, 64, false, true);    // P V, PB R^V
            const uint32_t aQ = smem_u32(sQ);
            uint64_t *last_bar = nullptr;
            uint32_t last_par = 0;
            auto commit = [&](uint64_t *bar, uint32_t parity) {
                mma_commit(bar);
                last_bar = bar;
                last_par = parity;
            };
            bool ok = true;
            const bool rk = HK && P.bias == nullptr;  // bias mode: no Q R^K^T
            const bool per_head = EXT && (rk || HQ || HV) && P.tab_heads > 1;
            if ((rk || HQ || HV) && !per_head)
                ok = mbar_wait(&bars.tab_full, 0, wc, kStatusTimeoutLoad, &abort_flag);
            int g = 0, w = 0, pr = 0;
            uint32_t qrc = 0;  // QR rounds issued (one per 64-row half of R^K)
            for (int item = blockIdx.x; ok && item < P.items; item += gridDim.x, ++w) {
                if (!(ok = mbar_wait(&bars.q_full, w & 1, wc, kStatusTimeoutLoad, &abort_flag))) break;
                if (per_head && !(ok = mbar_wait(&bars.tab_full, w & 1, wc, kStatusTimeoutLoad, &abort_flag)))
                    break;
                tc_fence_after();
                // QR = Q R^K^T, one 64-bucket half per round through the same
                // 64 TMEM columns (the softmax warps copy each round out)
                for (int r = 0; rk && ok && r < (EXT ? P.nr : 1); ++r, ++qrc) {
                    if (!(ok = mbar_wait(&bars.qr_empty, (qrc & 1) ^ 1, wc, kStatusTimeoutSync,
                                         &abort_flag)))
                        break;
                    tc_fence_after();
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ss(tmem + kColQR, smem_desc(aQ + kk * 32, 16, 1024, kSwizzle128B),
                                    smem_desc(smem_u32(smem + P.off_rk) + r * (kTileBytes / 2) + kk * 32,
                                              16, 1024, kSwizzle128B),
                                    kIdT, kk > 0);
                    commit(&bars.qr_full, qrc & 1);
                }
                if (!ok) break;
                // S for key tile g (and KR with it); returns false on abort
                auto issue_s = [&](int gg, int kt) -> bool {
                    const int st = gg % P.nst, b = gg & 1;
                    if (!mbar_wait(&bars.kv_full[st], (gg / P.nst) & 1, wc, kStatusTimeoutLoad,
                                   &abort_flag))
                        return false;
                    if (!mbar_wait(&bars.s_empty[b], ((gg >> 1) & 1) ^ 1, wc, kStatusTimeoutSync,
                                   &abort_flag))
                        return false;
                    tc_fence_after();
                    const uint32_t aK = smem_u32(sKV + st * 2 * kTileBytes);
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ss(tmem + kColS + b * 128,
                                    smem_desc(aQ + kk * 32, 16, 1024, kSwizzle128B),
                                    smem_desc(aK + kk * 32, 16, 1024, kSwizzle128B), kIdS, kk > 0);
                    if (HQ)
                        for (int kk = 0; kk < 4; ++kk)
                            mma_bf16_ss(tmem + kColKR + b * 64,
                                        smem_desc(aK + kk * 32, 16, 1024, kSwizzle128B),
                                        smem_desc(smem_u32(smem + P.off_rq) + kk * 32, 16, 1024,
                                                  kSwizzle128B),
                                        kIdT, kk > 0);
                    commit(&bars.s_full[b], (gg >> 1) & 1);
                    if (kt == P.nkt - 1) commit(&bars.q_empty, w & 1);
                    return true;
                };
                if (!(ok = issue_s(g, 0))) break;
                // With two K/V stages the next tile's S is issued before this tile's
                // P V, so the tensor core works while the softmax warps do; with one
                // stage the next tile's load needs this P V to free the stage first.
                const bool early_s = P.nst > 1;
                for (int kt = 0; kt < P.nkt; ++kt, ++g) {
                    if (early_s && kt + 1 < P.nkt && !(ok = issue_s(g + 1, kt + 1))) break;
                    if (kt == 0 && !(ok = mbar_wait(&bars.o_empty, (w & 1) ^ 1, wc,
                                                    kStatusTimeoutSync, &abort_flag)))
                        break;
                    if (!(ok = mbar_wait(&bars.p_full, pr & 1, wc, kStatusTimeoutSync, &abort_flag)))
                        break;
                    ++pr;
                    tc_fence_after();
                    const int st = g % P.nst;
                    const uint32_t aV = smem_u32(sKV + st * 2 * kTileBytes + kTileBytes);
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16_ss(tmem + kColO,
                                    smem_desc(smem_u32(sP) + (kk >> 2) * kTileBytes + (kk & 3) * 32,
                                              16, 1024, kSwizzle128B),
                                    smem_desc(aV + kk * 2048, 16, 1024, kSwizzle128B), kIdO,
                                    (kt > 0 || kk > 0) ? 1u : 0u);
                    commit(&bars.p_empty, (pr - 1) & 1);
                    commit(&bars.kv_empty[st], (g / P.nst) & 1);
                    if (!early_s && kt + 1 < P.nkt && !(ok = issue_s(g + 1, kt + 1))) break;
                }
                if (!ok) break;
                if (HV) {
                    if (!(ok = mbar_wait(&bars.p_full, pr & 1, wc, kStatusTimeoutSync, &abort_flag)))
                        break;
                    ++pr;
                    tc_fence_after();
                    for (int kk = 0; kk < 4 * (EXT ? P.nr : 1); ++kk)
                        mma_bf16_ss(tmem + kColO,
                                    smem_desc(smem_u32(sP) + (kk >> 2) * kTileBytes + (kk & 3) * 32,
                                              16, 1024, kSwizzle128B),
                                    smem_desc(smem_u32(smem + P.off_rv) + kk * 2048, 16, 1024,
                                              kSwizzle128B),
                                    kIdO, 1u);
                    commit(&bars.p_empty, (pr - 1) & 1);
                }
                commit(&bars.o_full, w & 1);
                // every product of the item that reads the tables is done with them
                if (per_head) commit(&bars.tab_empty, w & 1);
            }
            // drain: tcgen05 work completes in order, so the last commit covers it all
            if (last_bar != nullptr) mbar_wait(last_bar, last_par, drain, kStatusTimeoutDrain, nullptr);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax warps 0-3
        const int t = tid;  // query row within the tile == TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const int cols = 2 * P.W - 1;
        float *qr_t = sQR + t;
        float *pb_t = sPB + t;
        const uint32_t prow = smem_u32(sP) + t * 128;
        int g = 0, w = 0, pw = 0;
        uint32_t qrc = 0;  // QR rounds copied
        for (int item = blockIdx.x; item < P.items; item += gridDim.x, ++w) {
            const int slice = item / P.qtiles, qt = item % P.qtiles;
            const int i = qt * kBM + t;
            const int ic = i < P.N ? i : P.N - 1;
            const int centre = (P.H - 1) * cols + (P.W - 1);  // offset (0, 0)
            const bool cls = EXT && P.cls;
            const int pi = cls ? ic - 1 : ic;                    // grid position of the query
            const int base_i = pi < 0 ? P.lut_len + centre : (pi / P.W) * cols + (pi % P.W) + centre;
            const uint8_t *lut_i = sLut + base_i;
            bool qr_ok = true;
            if (HK && P.bias != nullptr) {
                // bias mode (eq. 14): the item's head's bias for every bucket,
                // scaled like the logits (inside the 1/sqrt(d) scaling), in this
                // row of the table; a Cross table's joint id a*span + b takes row
                // bucket a plus column bucket span + b
                const int col = P.bias_heads == 1 ? 0 : slice % P.heads;
                for (int b = 0; b < P.nb; ++b) {
                    float v;
                    if (EXT && P.cross)
                        v = __ldg(P.bias + (b / P.cross) * P.bias_heads + col) +
                            __ldg(P.bias + (P.cross + b % P.cross) * P.bias_heads + col);
                    else
                        v = __ldg(P.bias + b * P.bias_heads + col);
                    qr_t[b * 128] = v * P.c;
                }
            }
            for (int r = 0; HK && P.bias == nullptr && r < (EXT ? P.nr : 1); ++r, ++qrc) {
                // one round per item unless EXT: the item counter is the phase
                const uint32_t qph = EXT ? qrc : static_cast<uint32_t>(w);
                bool ok = __all_sync(~0u, mbar_wait(&bars.qr_full, qph & 1, wc, kStatusTimeoutMma,
                                                    &abort_flag));
                if (!bar_red_and(ok)) {
                    qr_ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem + lane_off + kColQR, r0);
                tmem_ld32(tmem + lane_off + kColQR + 32, r1);
                tmem_ld_wait();
                tmem_ready(r0);
                tmem_ready(r1);
                if (EXT && P.cross) {
#pragma unroll
                    for (int a = 0; a < 8; ++a)
#pragma unroll
                        for (int b = 0; b < 8; ++b)
                            if (a < P.cross && b < P.cross)
                                qr_t[(a * P.cross + b) * 128] =
                                    (__uint_as_float(r0[a]) + __uint_as_float(r1[b])) * P.c;
                } else {
                    float *qr_r = qr_t + r * 64 * 128;
                    const int nb_r = P.nb - r * 64;
#pragma unroll
                    for (int b = 0; b < 64; ++b)
                        if (b < nb_r) qr_r[b * 128] = __uint_as_float(b < 32 ? r0[b & 31] : r1[b & 31]) * P.c;
                }
                tc_fence_before();
                mbar_arrive(&bars.qr_empty);
            }
            if (!qr_ok) break;
            if (HV)
                for (int b = 0; b < P.nb; ++b) pb_t[b * 128] = 0.f;
            float m = -INFINITY, l = 0.f;
            bool aborted = false;
            for (int kt = 0; kt < P.nkt; ++kt, ++g) {
                const int b = g & 1;
                bool ok = __all_sync(~0u, mbar_wait(&bars.s_full[b], (g >> 1) & 1, wc,
                                                    kStatusTimeoutMma, &abort_flag));
                if (!bar_red_and(ok)) {  // also: everyone is done with the previous tile
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const int kbase = kt * kBN;
                {
                    const int j = kbase + t < P.N ? kbase + t : P.N - 1;  // clamp padding keys
                    const int pj = cls ? j - 1 : j;                       // grid position of the key
                    sKterm[t] = pj < 0 ? centre - P.lut_len : (pj / P.W) * cols + (pj % P.W);
                }
                if (HQ) {
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tmem + lane_off + kColKR + b * 64, r0);
                    tmem_ld32(tmem + lane_off + kColKR + b * 64 + 32, r1);
                    tmem_ld_wait();
                    tmem_ready(r0);
                    tmem_ready(r1);
                    float *kr = sKR + t * kKRStride;
                    if (EXT && P.cross) {
#pragma unroll
                        for (int a = 0; a < 8; ++a)
#pragma unroll
                            for (int bb = 0; bb < 8; ++bb)
                                if (a < P.cross && bb < P.cross)
                                    kr[a * P.cross + bb] =
                                        (__uint_as_float(r0[a]) + __uint_as_float(r1[bb])) * P.c;
                    } else {
#pragma unroll
                        for (int bb = 0; bb < 64; ++bb)
                            if (bb < P.nb) kr[bb] = __uint_as_float(bb < 32 ? r0[bb & 31] : r1[bb & 31]) * P.c;
                    }
                }
                softmax_bar();
                uint32_t s[128];
                {
                    uint32_t *s0 = s, *s1 = s + 32, *s2 = s + 64, *s3 = s + 96;
                    tmem_ld32(tmem + lane_off + kColS + b * 128, *reinterpret_cast<uint32_t(*)[32]>(s0));
                    tmem_ld32(tmem + lane_off + kColS + b * 128 + 32, *reinterpret_cast<uint32_t(*)[32]>(s1));
                    tmem_ld32(tmem + lane_off + kColS + b * 128 + 64, *reinterpret_cast<uint32_t(*)[32]>(s2));
                    tmem_ld32(tmem + lane_off + kColS + b * 128 + 96, *reinterpret_cast<uint32_t(*)[32]>(s3));
                    tmem_ld_wait(s);
                }
                tc_fence_before();
                mbar_arrive(&bars.s_empty[b]);  // S[b] and KR[b] are read

                // pass 1: logits in log2 units, running max
                const int nvalid = min(kBN, P.N - kbase);
                const int4 *kt4 = reinterpret_cast<const int4 *>(sKterm);
                float mloc = -INFINITY;
#pragma unroll
                for (int q4 = 0; q4 < 32; ++q4) {
                    const int4 kv = kt4[q4];
                    const int kts[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int jj = q4 * 4 + e;
                        float x = __uint_as_float(s[jj]) * P.c;
                        if (HK || HQ || HV) {
                            const int id = lut_i[-kts[e]];
                            if (HK) x += qr_t[id * 128];
                            if (HQ) x += sKR[jj * kKRStride + id];
                        }
                        x = (jj < nvalid) ? x : -INFINITY;
                        s[jj] = __float_as_uint(x);
                        mloc = fmaxf(mloc, x);
                    }
                }
                // lazy rescale: move the reference max only when it grows by > 2^8
                float alpha = 1.f;
                if (mloc > m + kRescaleLog2) {
                    alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - mloc);
                    m = mloc;
                    l *= alpha;
                    if (HV)
                        for (int bb = 0; bb < P.nb; ++bb) pb_t[bb * 128] *= alpha;
                }
                // P buffer free (the previous P V is done) -> rescale O if needed
                ok = __all_sync(~0u, mbar_wait(&bars.p_empty, (pw & 1) ^ 1, wc, kStatusTimeoutMma,
                                               &abort_flag));
                ++pw;
                if (!ok) {
                    aborted = true;
                    continue;  // the next tile's reduction breaks out uniformly
                }
                tc_fence_after();
                if (kt > 0 && __any_sync(~0u, alpha < 1.f)) {
                    uint32_t o0[32], o1[32];
                    tmem_ld32(tmem + lane_off + kColO, o0);
                    tmem_ld32(tmem + lane_off + kColO + 32, o1);
                    tmem_ld_wait();
                    tmem_ready(o0);
                    tmem_ready(o1);
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        o0[c] = __float_as_uint(__uint_as_float(o0[c]) * alpha);
                        o1[c] = __float_as_uint(__uint_as_float(o1[c]) * alpha);
                    }
                    tmem_st32(tmem + lane_off + kColO, o0);
                    tmem_st32(tmem + lane_off + kColO + 32, o1);
                    tmem_st_wait();
                }
                // pass 2: probabilities -> P (bf16, K-major, 128B swizzle), row sum, PB
                float sum = 0.f;
#pragma unroll
                for (int ch = 0; ch < 16; ++ch) {
                    uint32_t wv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j0 = ch * 8 + 2 * e;
                        const float p0 = ex2_approx(__uint_as_float(s[j0]) - m);
                        const float p1 = ex2_approx(__uint_as_float(s[j0 + 1]) - m);
                        sum += p0 + p1;
                        if (HV) {
                            if (j0 < nvalid) pb_t[static_cast<int>(lut_i[-sKterm[j0]]) * 128] += p0;
                            if (j0 + 1 < nvalid)
                                pb_t[static_cast<int>(lut_i[-sKterm[j0 + 1]]) * 128] += p1;
                        }
                        wv[e] = pack_bf16x2(p0, p1);
                    }
                    const int blk = ch >> 3, c = ch & 7;
                    st_shared_v4(prow + blk * kTileBytes + ((c ^ (t & 7)) << 4), wv[0], wv[1],
                                 wv[2], wv[3]);
                }
                l += sum;
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bars.p_full);
            }
            if (!bar_red_and(!aborted)) break;  // uniform across the four softmax warps
            if (HV) {
                // PB (bf16, buckets >= nb zero) into P's first block for O += PB R^V
                bool ok = __all_sync(~0u, mbar_wait(&bars.p_empty, (pw & 1) ^ 1, wc,
                                                    kStatusTimeoutMma, &abort_flag));
                ++pw;
                if (!bar_red_and(ok)) break;
                // Cross: slot a < 8 takes row bucket a's sum over the joint ids,
                // slot 32 + b column bucket span + b's (the staged table rows)
                float rsum[8], csum[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) rsum[a] = csum[a] = 0.f;
                if (EXT && P.cross) {
#pragma unroll
                    for (int a = 0; a < 8; ++a)
#pragma unroll
                        for (int b = 0; b < 8; ++b)
                            if (a < P.cross && b < P.cross) {
                                const float pv = pb_t[(a * P.cross + b) * 128];
                                rsum[a] += pv;
                                csum[b] += pv;
                            }
                }
                // buckets 0..63 in P's first block, 64..127 (if any) in its second
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    if (c >= 8 * (EXT ? P.nr : 1)) continue;
                    uint32_t wv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int b0 = c * 8 + 2 * e;
                        float v0, v1;
                        if (EXT && P.cross) {
                            v0 = b0 < 8 ? rsum[b0] : (b0 >= 32 && b0 < 40 ? csum[b0 - 32] : 0.f);
                            v1 = b0 + 1 < 8 ? rsum[b0 + 1]
                                            : (b0 + 1 >= 32 && b0 + 1 < 40 ? csum[b0 - 31] : 0.f);
                        } else {
                            v0 = b0 < P.nb ? pb_t[b0 * 128] : 0.f;
                            v1 = b0 + 1 < P.nb ? pb_t[(b0 + 1) * 128] : 0.f;
                        }
                        wv[e] = pack_bf16x2(v0, v1);
                    }
                    st_shared_v4(prow + (c >> 3) * kTileBytes + (((c & 7) ^ (t & 7)) << 4), wv[0], wv[1],
                                 wv[2], wv[3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bars.p_full);
            }
            // epilogue: O / l -> bf16 -> global
            bool ok = __all_sync(~0u, mbar_wait(&bars.o_full, w & 1, wc, kStatusTimeoutMma,
                                                &abort_flag));
            if (!bar_red_and(ok)) break;
            tc_fence_after();
            uint32_t o0[32], o1[32];
            tmem_ld32(tmem + lane_off + kColO, o0);
            tmem_ld32(tmem + lane_off + kColO + 32, o1);
            tmem_ld_wait();
            tmem_ready(o0);
            tmem_ready(o1);
            tc_fence_before();
            mbar_arrive(&bars.o_empty);
            if (i < P.N) {
                const float inv = 1.f / l;
                uint4 *dst = reinterpret_cast<uint4 *>(P.out + (static_cast<size_t>(slice) * P.N + i) * kD);
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

template <bool HK, bool HQ, bool HV, bool EXT>
cudaError_t launch_tmpl(const RpeBf16Args &a, cudaStream_t stream) {
    const int N = a.H * a.W + a.cls;  // the class token, if any, is token 0
    const int slices = a.B * a.heads;
    RpeParams p{};
    p.N = N;
    p.H = a.H;
    p.W = a.W;
    p.cross = a.cross_span;
    p.nb = a.cross_span > 0 ? a.cross_span * a.cross_span : a.num_buckets;
    p.tab_row2 = a.cross_span > 0 ? a.cross_span : 32;
    p.tab_heads = a.tab_heads;
    p.heads = a.heads;
    p.nr = a.num_buckets > 64 ? 2 : 1;
    p.nkt = (N + kBN - 1) / kBN;
    p.qtiles = (N + kBM - 1) / kBM;
    p.items = slices * p.qtiles;
    p.lut_len = (2 * a.H - 1) * (2 * a.W - 1);
    p.cls = a.cls;
    p.bias = a.bias;
    p.bias_heads = a.bias_heads;
    p.lut = a.lut;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.c = static_cast<float>(kLog2e / std::sqrt(static_cast<double>(kD)));

    const uint32_t smem_cap = 227 * 1024 - 1024;  // leave room for the static barriers
    for (int nst = 2; nst >= 1; --nst) {
        uint32_t off = 0;
        p.off_q = off;
        off += kTileBytes;
        p.off_kv = off;
        off += nst * 2 * kTileBytes;
        p.off_p = off;
        off += 2 * kTileBytes;
        p.off_rk = off;
        if (HK && a.bias == nullptr) off += p.nr * (kTileBytes / 2);
        p.off_rq = off;
        if (HQ) off += p.nr * (kTileBytes / 2);
        p.off_rv = off;
        if (HV) off += p.nr * (kTileBytes / 2);
        p.off_qr = off;
        if (HK) off += align_up(p.nb * 512, 1024);
        p.off_kr = off;
        if (HQ) off += align_up(128 * kKRStride * 4, 1024);
        p.off_pb = off;
        if (HV) off += align_up(p.nb * 512, 1024);
        p.off_kterm = off;
        off += 512;
        p.off_lut = off;
        off += align_up(a.cls ? 2 * p.lut_len + 1 : p.lut_len, 16);
        const uint32_t total = 1024 + std::max<uint32_t>(off, 120 * 1024);
        if (total <= smem_cap) {
            p.nst = nst;
            unsigned *status = device_status_word();
            if (status == nullptr) return cudaErrorMemoryAllocation;
            p.wc = WaitCtl{status, kDefaultWaitNs};
            const uint64_t dims[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(N),
                                      static_cast<uint64_t>(slices)};
            const uint64_t strides[2] = {kD * 2, static_cast<uint64_t>(N) * kD * 2};
            const uint32_t box[3] = {kD, 128, 1};
            // tables [tab_heads][num_buckets][d]
            const uint64_t tdims[3] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(a.num_buckets),
                                       static_cast<uint64_t>(a.tab_heads)};
            const uint64_t tstrides[2] = {kD * 2, static_cast<uint64_t>(a.num_buckets) * kD * 2};
            const uint32_t tbox[3] = {kD, 32, 1};
            CUtensorMap tq, tk, tv, trk, trq, trv;
            const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
            const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
            if (!encode_tensor_map(&tq, bf, 3, a.q, dims, strides, box, sw) ||
                !encode_tensor_map(&tk, bf, 3, a.k, dims, strides, box, sw) ||
                !encode_tensor_map(&tv, bf, 3, a.v, dims, strides, box, sw))
                return cudaErrorInvalidValue;
            // tables not in use get a valid (never read) map over q
            const void *rk = HK && a.bias == nullptr ? a.tab_k : a.q, *rq = HQ ? a.tab_q : a.q,
                       *rv = HV ? a.tab_v : a.q;
            if (!encode_tensor_map(&trk, bf, 3, rk, tdims, tstrides, tbox, sw) ||
                !encode_tensor_map(&trq, bf, 3, rq, tdims, tstrides, tbox, sw) ||
                !encode_tensor_map(&trv, bf, 3, rv, tdims, tstrides, tbox, sw))
                return cudaErrorInvalidValue;
            cudaError_t err = cudaFuncSetAttribute(rpe_bf16_kernel<HK, HQ, HV, EXT>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(total));
            if (err != cudaSuccess) return err;
            const int grid = std::min(p.items, sm_count());
            rpe_bf16_kernel<HK, HQ, HV, EXT><<<grid, kThreads, total, stream>>>(tq, tk, tv, trk, trq, trv, p);
            return cudaGetLastError();
        }
    }
    // the offset and bucket tables do not fit in shared memory: nothing launched
    return cudaErrorNotSupported;
}

}  // namespace

namespace {

template <bool EXT>
cudaError_t launch_terms(const RpeBf16Args &a, cudaStream_t stream) {
    const bool k = a.terms & 1u, q = a.terms & 2u, v = a.terms & 4u;
    if (!k && !q && !v) return launch_tmpl<false, false, false, EXT>(a, stream);
    if (k && !q && !v) return launch_tmpl<true, false, false, EXT>(a, stream);
    if (!k && q && !v) return launch_tmpl<false, true, false, EXT>(a, stream);
    if (!k && !q && v) return launch_tmpl<false, false, true, EXT>(a, stream);
    if (k && q && !v) return launch_tmpl<true, true, false, EXT>(a, stream);
    if (k && !q && v) return launch_tmpl<true, false, true, EXT>(a, stream);
    if (!k && q && v) return launch_tmpl<false, true, true, EXT>(a, stream);
    return launch_tmpl<true, true, true, EXT>(a, stream);
}

}  // namespace

cudaError_t launch_rpe_bf16(const RpeBf16Args &a, cudaStream_t stream) {
    cudaError_t err = cudaSuccess;
    if (launch_rpe_bf16_pingpong(a, stream, &err)) return err;
    if (a.bias != nullptr) {
        // bias mode on any grid (and with a class token): the key-term path with
        // the bias row in place of QR'
        RpeBf16Args b = a;
        b.terms = 1u;
        b.tab_heads = 1;
        if (b.cross_span > 0 || b.num_buckets > 64 || b.cls) return launch_tmpl<true, false, false, true>(b, stream);
        return launch_tmpl<true, false, false, false>(b, stream);
    }
    if (a.cross_span > 0 || a.num_buckets > 64 || a.tab_heads > 1 || a.cls)
        return launch_terms<true>(a, stream);
    return launch_terms<false>(a, stream);
}

}  // namespace vta
