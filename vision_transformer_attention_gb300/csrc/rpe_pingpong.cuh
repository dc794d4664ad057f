// rpe_pingpong.cuh -- iRPE attention on sm_103a with two query tiles per CTA,
// each softmaxed by one warpgroup with one thread per query row, the tensor
// core fed through a ring of tensor-memory score slots per tile: the kernel
// template and its launcher, instantiated by rpe_attn_pingpong_sm103.cu (key
// term, bias mode, no term) and rpe_attn_pingpong_qv_sm103.cu (with the query
// and / or value terms).
//
// Same computation as rpe_attn_sm103.cu ("Rethinking and Improving Relative
// Position Encoding for Vision Transformer", eqs. 13-17 and the efficient form
// of eqs. 26-28): logits (q_i.k_j + q_i.R^K[id] + k_j.R^Q[id])/sqrt(d), softmax,
// P V plus the value term sum_j p_ij R^V[id], with QR = Q R^K^T formed once
// per query tile and KR = K R^Q^T once per key tile on the tensor core and read
// per score by bucket id. It is the fast path on grids of width W in {14, 56}:
//
//   * One CTA per SM, persistent over items. An item is a pair of 128-row
//     query tiles of one (batch, head) slice (or a slice's odd last tile);
//     both tiles share every K/V tile. Warps 0-3 softmax tile 0 and warps 4-7
//     tile 1, one thread per query row; warp 8 is the TMA producer, warps 9
//     and 10 the MMA issuers of the two tiles (one elected thread each); warp
//     11 only takes part in the register split (setmaxnreg: 216 registers for
//     the softmax warps, 64 for the others).
//   * Key tiles hold whole grid rows: five or six rows at W = 14 (70 keys in
//     NS = 80 score columns, or 84 in 96, whichever leaves fewer score
//     columns per query row), one row (56 keys, NS = 64) at W = 56. K and V
//     arrive as KT-row TMA boxes in NS-row buffers whose last NS - KT rows
//     stay zero. Keys past the grid (last tile) get -9984 added by one extra
//     K = 16 product with constant operands, so the softmax never tests them.
//   * Each tile's group owns O (64 tensor-memory columns) and a ring of two
//     score slots. A "unit" is QR' = Q R^K^T (once per item) or one key tile's
//     scores; unit u goes into slot u mod 2 once unit u - 2 is consumed (its
//     QR' copied to shared memory, or its P V issued). The issuer is a
//     straight sequence of bounded blocking waits.
//   * Per tile each thread reads its row's scores in one tensor-memory round
//     trip, forms the logits x = S c + QR'[id] (+ KR[j][id]) (c = log2 e /
//     sqrt d) in registers -- the bucket ids come from the offset table in
//     shared memory, read as aligned words per grid row of keys and taken out
//     with byte permutes, and QR' lives in shared memory as [bucket][row] --
//     then writes p = 2^(x - m) as bf16 pairs over the scores, where the P V
//     product reads its A operand. The reference max m moves only when a
//     tile's max exceeds it by more than 2^8 (O is then rescaled).
//   * Query term (five-row tiles at W = 14): group 0's issuer forms KR of each
//     key tile in the 64 tensor-memory columns after the two groups' 224;
//     warps 0-2 of both groups copy it (lane = key) to a shared fp16 table.
//   * Value term: each row's probabilities go into per-bucket sums PB in
//     shared memory, one grid row of keys at a time; at the item's end PB
//     (bf16, in the staging tile) times R^V accumulates into O on the tensor
//     core.
//   * An item's epilogue runs after the next item's QR' copy (so the copy
//     overlaps the wait for the last P V); it stages the bf16 output tile in
//     the group's own 16 KB area with a 128-byte swizzle and writes it with
//     one TMA store (rows past the grid fall outside the tensor map).
//   * When the last round of items fills at most half the grid, each of its
//     items runs as two parts (halves of the key tiles) on two CTAs that
//     merge through a per-stream workspace (see item_at and the epilogue).
//
// Tensor memory (512 columns): group w owns [C w, C w + C), C = 256 (224 with
// the query term): O at +0, slot s at +64 + s NS (s 96 with a class token at
// W = 56, where NS = 64 is short of the widened QR' product); KR (query
// term) at 448.
#pragma once
#include "vta_internal.h"
#include "sm103_ptx.cuh"

#include <algorithm>
#include <cmath>

namespace vta {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kD = 64;
constexpr int kTileBytes = 128 * 128;  // one 128-row x 64-column bf16 tile
// NG softmax groups (query tiles) per CTA: warps 0..4NG-1 are the groups'
// warpgroups, warpgroup NG the control warps. Register split per CTA: control
// warpgroup 64 registers, softmax warps the rest of the launch allocation.
// NG = 2 (a pair of query tiles sharing every K/V tile, one CTA per SM) is
// used; NG = 1 (one query tile per CTA, two CTAs per SM, independent
// pipelines but twice the K/V traffic from L2) measured slower at both grid
// widths.
constexpr int kGroupsPerCta = 2;

template <int NG>
struct Layout {
    static constexpr int kThreads = 128 * (NG + 1);
    static constexpr int kCtasPerSm = NG == 1 ? 2 : 1;
    static constexpr int kRegsLaunch = NG == 2 ? 168 : 128;
    static constexpr int kRegsControl = 64;
    static constexpr int kRegsSoftmax = NG == 2 ? 216 : 192;
    static_assert(128 * kRegsControl + 128 * NG * kRegsSoftmax <= kThreads * kRegsLaunch,
                  "register split");
};
constexpr float kRescaleLog2 = 8.f;
constexpr int kMaxStages = 8;
constexpr int kMaxSlots = 3;       // score slots per group (see Geo::SLOTS)
constexpr uint32_t kColSlot0 = 64;  // within the group's columns
// With the query term (five-row key tiles, NS = 80) each group owns 224
// columns and K R^Q^T of the current key tile takes the last 64.
constexpr uint32_t kKrCol = 448;
// Bytes per key row of the shared K R^Q^T table (fp16, up to 72 buckets): 36
// words, so the sixteen-byte stores of eight consecutive keys hit distinct
// banks, and one key's 64 buckets span distinct banks for the gathers.
constexpr int kKrStride = 144;

template <int W, int RR>
struct Geo {
    static constexpr int R = RR;                    // grid rows per key tile
    static constexpr int KT = R * W;                // keys per tile
    static constexpr int NS = (KT + 15) / 16 * 16;  // N of QK^T, K of PV
    static constexpr int HS = NS;  // keys per thread and tile (one thread owns a row)
    static constexpr int COLS = 2 * W - 1;          // offset-table row length
    // one K or V buffer: the tile's KT rows (loaded) and NS - KT rows that stay
    // zero (the products read NS rows)
    static constexpr int KV_BYTES = NS * 128;
    // score slots of NS columns after O's 64 in the group's 256 (a third slot
    // where it fits, W = 56, measured slower: the tensor core, not the
    // prefetch depth, limits there)
    static constexpr int SLOTS = 2;
    static_assert(SLOTS >= 2 && SLOTS <= kMaxSlots, "slots");
    static_assert(NS <= 96 && HS % 16 == 0 && 2 * HS >= NS, "tile geometry");
};

struct PPParams {
    int N, H, nb, nkt, qtiles, pairs_full, slices, items, nst, nq;
    int single;  // 1: an item is one query tile (one group per CTA)
    int cross;     // Cross tables: span (nb = span^2 joint ids); 0 otherwise
    int tab_heads; // 1: one R^K shared by every head; heads: one per head
    int tab_row2;  // table row staged at shared-memory row 32: span (Cross) or 32
    const float *bias;  // bias mode: [nb, bias_heads] fp32
    int bias_heads, heads;
    uint32_t off_q, off_kv, off_rk, off_qr, qr_stride, off_lut, off_mask, off_stage;
    // query term: R^Q and the key tile's K R^Q^T [key][bucket] (fp16, scaled);
    // value term: R^V and each group's bucket sums PB [bucket][128 rows] (fp32)
    uint32_t off_rq, off_rv, off_kr, off_pb, pb_stride;
    int lut_len, lut_pad;
    int nvalid_last;  // keys of the last key tile that lie on the grid
    // Class token (token 0; its pairs take bucket nb - 1): the grid keys are
    // tokens 1.., the offset table is followed by cls_len bytes of the class
    // bucket from which the class query reads (its base offset cls_base), and
    // the class key is folded into each row in the epilogue, its value row
    // read from v_cls + slice * N * 64.
    int cls_len, cls_base;
    const uint16_t *v_cls;
    // Tail split: items [0, whole) run whole, in full rounds over the grid; the
    // `tail` items after them run as two parts on two CTAs, part A over key
    // tiles [0, ka), part B over [ka, nkt), merged by the later part through
    // ws (per (tail item, group, part): O [64][128], m [128], l [128]) and
    // the arrival counters cnt (one per tail item and group).
    int whole, tail, ka;
    float *ws;
    int *cnt;
    const int32_t *lut;
    float c;  // log2(e) / sqrt(d)
    WaitCtl wc;
};

struct PPBars {
    uint64_t tab_full;
    uint64_t q_full[2], q_empty[2];
    uint64_t kv_full[kMaxStages], kv_empty[kMaxStages];
    uint64_t slot_full[2][kMaxSlots], slot_done[2][kMaxSlots];
    uint64_t o_full[2], o_empty[2], pv_done[2];
    uint64_t fin[2];   // drain of each issuer
    // query term: K R^Q^T of a key tile in tensor memory (full: product done;
    // empty: copied out) and in shared memory (full: copied; empty: every
    // softmax warp has read it)
    uint64_t kr_tfull, kr_tempty, kr_sfull, kr_sempty;
    uint64_t pb_full[2];  // value term: the group's PB operand is staged
};

struct Item {
    int slice, qt0;
    bool has_b;
    int kt0, kt1;  // key tiles of this entry
    int part;      // 0: the whole item; 1, 2: part A, B of tail item tidx
    int tidx;
};

// Items: full pairs of query tiles (slice-major), then the odd last tiles,
// dealt round-robin over the CTAs (an odd tile takes about as long as a pair:
// the two groups of a pair run side by side). item_at<SP>(P, k) is the k-th item
// of this CTA, -1 past its last; every role walks the same sequence.
template <bool SP>
__device__ __forceinline__ Item decode_item(const PPParams &P, int entry) {
    Item r;
    int item = entry;
    r.kt0 = 0;
    r.kt1 = P.nkt;
    r.part = 0;
    r.tidx = 0;
    if (SP && entry >= P.items) {  // a part of a split tail item
        const int j = (entry - P.items) % P.tail;
        r.part = 1 + (entry - P.items) / P.tail;
        r.tidx = j;
        item = P.whole + j;
        if (r.part == 1)
            r.kt1 = P.ka;
        else
            r.kt0 = P.ka;
    }
    if (P.single) {
        r.slice = item / P.qtiles;
        r.qt0 = item % P.qtiles;
        r.has_b = false;
        return r;
    }
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

// The k-th entry of this CTA: whole items in full rounds, then the tail parts.
// With T <= G / 2 tail items on G CTAs, CTA c < T runs part A of tail item c
// and CTA T + j part B of tail item j, so no CTA runs more than one part and
// the last round takes about half an item. Entries >= items encode parts:
// items + j (A) and items + T + j (B).
template <bool SP>
__device__ __forceinline__ int item_at(const PPParams &P, int k) {
    const int G = gridDim.x, c = blockIdx.x;
    if (!SP || P.tail == 0) {
        const int item = c + k * G;
        return item < P.items ? item : -1;
    }
    const int r0 = P.whole / G;
    if (k < r0) return c + k * G;
    if (k > r0 || c >= 2 * P.tail) return -1;
    return P.items + c;  // c < T: A part of tail item c; else B part of tail item c - T
}

// AND-reduction of v over the nthreads threads that use named barrier id.
__device__ __forceinline__ bool red_and(int id, int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Multiply this row's O (64 columns) by alpha once the group's previous P V
// has completed. Out of line: it runs only when a row's reference max moves.
__device__ __forceinline__ bool rescale_o(float alpha, uint32_t tO, uint64_t *pv_bar,
                                       uint32_t pv_parity, const WaitCtl &wc,
                                       volatile int *abort, bool sleep) {
    if (!__all_sync(~0u, mbar_wait(pv_bar, pv_parity, wc, kStatusTimeoutMma, abort, sleep))) return false;
    tc_fence_after();
#pragma unroll 1
    for (int r = 0; r < 4; ++r) {
        uint32_t o[16];
        tmem_ld16(tO + r * 16, o);
        tmem_ld_wait(o);
#pragma unroll
        for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st16(tO + r * 16, o);
    }
    tmem_st_wait();
    return true;
}

// The QR' and K R^Q^T tables next to the query or value term are fp16: two
// bytes per entry like bf16, but with unit roundoff 2^-11 instead of 2^-8
// (the logits they feed reach tens of units; fp16's range is 65504).
__device__ __forceinline__ float f16_to_f32(uint16_t bits) { return __half2float(__ushort_as_half(bits)); }
__device__ __forceinline__ uint16_t f32_to_f16(float x) { return __half_as_ushort(__float2half_rn(x)); }
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    return static_cast<uint32_t>(f32_to_f16(lo)) | (static_cast<uint32_t>(f32_to_f16(hi)) << 16);
}

// One half (H2 = 0: keys [0, HS) of the tile, 1: keys [HS, 2 HS)) of one row's tile.
// The logits add terms read by bucket id: QM = 1, an fp32 table at stride QS
// floats per bucket (QR' rows: 128; a bias-mode row: 1); QM = 2, an fp16 QR'
// table at stride QS; KQ, the key tile's K R^Q^T [key][bucket] (fp16).
template <int W, int R, bool GATHER_, int H2, int QS = 128, int QM = GATHER_ ? 1 : 0, bool KQ = false>
struct HalfTile {
    static constexpr bool GATHER = QM != 0 || KQ;
    using G = Geo<W, R>;
    static constexpr int J0 = G::HS * H2;                       // first key of the half
    static constexpr int NK = (G::KT - J0 < G::HS) ? G::KT - J0 : G::HS;  // keys of the half
    static constexpr int NQ = (NK + 15) / 16;                   // 16-key chunks holding them

    // Grid rows of the tile that the half's keys lie on, and the key columns
    // [c_lo, c_hi) of each. The offset-table bytes of one grid row of keys are
    // contiguous (column c at byte c_hi - 1 - c from the lowest), so each run is
    // read as aligned words, realigned with a funnel shift, and each id taken
    // out with a byte permute: about one shared-memory wavefront per four ids.
    static constexpr int ROW_LO = J0 / W;
    static constexpr int ROW_HI = (J0 + NK - 1) / W;
    static constexpr int NROWS = ROW_HI - ROW_LO + 1;
    static constexpr int c_lo(int r) { return (J0 > r * W ? J0 : r * W) - r * W; }
    static constexpr int c_hi(int r) { return (J0 + NK < (r + 1) * W ? J0 + NK : (r + 1) * W) - r * W; }
    static constexpr int run_words(int r) { return (c_hi(r) - c_lo(r) + 3) / 4; }
    static constexpr int NA = (W < NK ? W : NK) / 4 + 1;  // >= run_words of any row
    static constexpr int first_chunk(int r) { return ((J0 > r * W ? J0 : r * W) - J0) / 16; }

    // Pass 1: x = S c + QR'[id] over the half's keys, 16 keys at a time, kept
    // in registers (s, the scores' own registers) for pass 2; returns the
    // half's max. lutw: the offset table as words; e0: byte index in it of the
    // tile's key 0 for this row; qr_t: this row's QR' for bucket 0 (buckets
    // 128 floats apart).
    static __device__ __forceinline__ float logits(uint32_t tS, const uint32_t *lutw, int e0,
                                                   const void *qr, const uint16_t *kr, float c,
                                                   uint32_t (&s)[NQ][16]) {
        uint32_t ida[NROWS][NA];
        float mx = -INFINITY;
        const float2 c2 = make_float2(c, c);
        // all of the row's scores in one tensor-memory round trip; its latency
        // overlaps the first chunk's gathers
#pragma unroll
        for (int q = 0; q < NQ; ++q) tmem_ld16(tS + J0 + 16 * q, s[q]);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int jc = J0 + 16 * q;
            float qv[16];
            if constexpr (GATHER) {
                // the id words of each grid row, read at the first chunk that needs them
#pragma unroll
                for (int rr = 0; rr < NROWS; ++rr) {
                    const int r = ROW_LO + rr;
                    if (first_chunk(r) != q) continue;
                    const int lo = e0 - (r * G::COLS + c_hi(r) - 1);  // may be negative (padding)
                    const uint32_t sh = static_cast<uint32_t>(lo & 3) * 8u;
                    const uint32_t *wp = lutw + (lo >> 2);
                    uint32_t wv[NA + 1];
#pragma unroll
                    for (int m = 0; m <= NA; ++m)
                        if (m <= run_words(r)) wv[m] = wp[m];
#pragma unroll
                    for (int m = 0; m < NA; ++m)
                        if (m < run_words(r)) ida[rr][m] = __funnelshift_r(wv[m], wv[m + 1], sh);
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int jj = jc + j;
                    if (jj < J0 + NK) {
                        const int r = jj / W, k = c_hi(r) - 1 - jj % W;
                        const uint32_t id = __byte_perm(ida[r - ROW_LO][k / 4], 0u, 0x4440u | (k % 4));
                        float g = 0.f;
                        if constexpr (QM == 1) g = static_cast<const float *>(qr)[id * QS];
                        if constexpr (QM == 2) g = f16_to_f32(static_cast<const uint16_t *>(qr)[id * QS]);
                        if constexpr (KQ) g += f16_to_f32(kr[jj * (kKrStride / 2) + id]);
                        qv[j] = g;
                    } else {
                        qv[j] = 0.f;
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) qv[j] = 0.f;
            }
            if (q == 0) {
                tmem_ld_wait();
#pragma unroll
                for (int qq = 0; qq < NQ; ++qq) tmem_ready(s[qq]);
            }
            float x[16];
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const float2 r = ffma2(make_float2(__uint_as_float(s[q][j]), __uint_as_float(s[q][j + 1])),
                                       c2, make_float2(qv[j], qv[j + 1]));
                x[j] = (jc + j < G::KT) ? r.x : -INFINITY;
                x[j + 1] = (jc + j + 1 < G::KT) ? r.y : -INFINITY;
            }
            const float a = fmax3(x[0], x[1], x[2]), b = fmax3(x[3], x[4], x[5]);
            const float d = fmax3(x[6], x[7], x[8]), e = fmax3(x[9], x[10], x[11]);
            const float f = fmax3(x[12], x[13], x[14]);
            mx = fmax3(mx, fmax3(a, b, d), fmax3(e, f, x[15]));
#pragma unroll
            for (int j = 0; j < 16; ++j) s[q][j] = __float_as_uint(x[j]);
        }
        return mx;
    }

    // Pass 2: p = 2^(x - m) as bf16 pairs from pass 1's registers; chunk q's
    // 8 columns go to J0 + 8q, over scores already read. Keys past the tile
    // contribute 0. Returns sum p; KEEP: p (fp32) also replaces x in xs.
    template <bool KEEP = false>
    static __device__ __forceinline__ float probs(uint32_t tS, float m, uint32_t (&xs)[NQ][16]) {
        float sum = 0.f;
        const float2 nm = make_float2(-m, -m);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int jc = J0 + 16 * q;
            float2 p[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float2 d = fadd2(make_float2(__uint_as_float(xs[q][2 * e]), __uint_as_float(xs[q][2 * e + 1])), nm);
                p[e] = make_float2(jc + 2 * e < G::KT ? ex2_approx(d.x) : 0.f,
                                   jc + 2 * e + 1 < G::KT ? ex2_approx(d.y) : 0.f);
            }
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) pk[e] = pack_bf16x2(p[e].x, p[e].y);
            if constexpr (KEEP) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    xs[q][2 * e] = __float_as_uint(p[e].x);
                    xs[q][2 * e + 1] = __float_as_uint(p[e].y);
                }
            }
            tmem_st8(tS + J0 + 8 * q, pk);
#pragma unroll
            for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
                for (int j = 0; j < w; ++j) p[j] = fadd2(p[2 * j], p[2 * j + 1]);
            sum += p[0].x + p[0].y;
        }
        return sum;
    }

    // Value term: adds each key's probability (pass 2 with KEEP) to its
    // bucket's sum PB[id] (pb_t: this row's entry of bucket 0, buckets 128
    // floats apart), one grid row of keys at a time over the first `rows`
    // rows of the tile. A grid row's sums are all loaded first; runs of equal
    // ids along the row are summed in registers and each run's total is added
    // at its last key, so no update waits for another through shared memory.
    // This needs every id to form one run per grid row of keys (the caller
    // has the offset table checked for that).
    static __device__ __forceinline__ void bucket_sums(const uint32_t *lutw, int e0, float *pb_t,
                                                       int rows, const uint32_t (&ps)[NQ][16]) {
        static_assert(H2 == 0 && G::HS == G::NS, "one half per tile");
        constexpr int NW = (W + 3) / 4;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r >= rows) break;
            const int lo = e0 - (r * G::COLS + W - 1);
            const uint32_t sh = static_cast<uint32_t>(lo & 3) * 8u;
            const uint32_t *wp = lutw + (lo >> 2);
            uint32_t wv[NW + 1], ida[NW];
#pragma unroll
            for (int m = 0; m <= NW; ++m) wv[m] = wp[m];
#pragma unroll
            for (int m = 0; m < NW; ++m) ida[m] = __funnelshift_r(wv[m], wv[m + 1], sh);
            uint32_t id[W];
            float old[W];
#pragma unroll
            for (int kx = 0; kx < W; ++kx) {
                const int k = W - 1 - kx;  // byte k of the row's run is key column kx
                id[kx] = __byte_perm(ida[k / 4], 0u, 0x4440u | (k % 4));
                old[kx] = pb_t[id[kx] * 128];
            }
            float run = 0.f;
#pragma unroll
            for (int kx = 0; kx < W; ++kx) {
                const int jj = r * W + kx;
                const float p = __uint_as_float(ps[jj / 16][jj % 16]);
                run = (kx > 0 && id[kx] == id[kx - 1]) ? run + p : p;
                if (kx == W - 1 || id[kx + 1] != id[kx]) pb_t[id[kx] * 128] = old[kx] + run;
            }
        }
    }
};

// Tensor-memory column (relative to the slot) of the A operand of P V step kk
// (keys 16 kk .. 16 kk + 15): half kk*16 / HS, chunk within it.
template <int W, int R>
__device__ __forceinline__ constexpr uint32_t p_col(int kk) {
    using G = Geo<W, R>;
    return static_cast<uint32_t>((16 * kk / G::HS) * G::HS + ((16 * kk) % G::HS) / 2);
}

// BM: iRPE bias mode (a scalar per bucket and head, inside the scaling) in
// place of the contextual key term; HK and BM are not both set. TF, the
// table form: bit 0, the table (R^K or the bias table) is laid out for the
// Cross mapping; bit 1, R^K is one table per head; bit 2, the tail items may
// run split in two parts (see item_at); bit 3, token 0 is a class token (with
// the key term); bit 4, 65..128 buckets (the QR' product in two rounds);
// bit 5, the contextual query term; bit 6, the contextual value term (bits 5
// and 6: W = 14 with five-row key tiles, shared tables, every item a pair of
// query tiles).
template <int W, int R, bool HK, int NG, bool BM, int TF>
__global__ void __launch_bounds__(Layout<NG>::kThreads, Layout<NG>::kCtasPerSm)
    rpe_pingpong_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_rk,
                        const __grid_constant__ CUtensorMap tm_kc,
                        const __grid_constant__ CUtensorMap tm_rq,
                        const __grid_constant__ CUtensorMap tm_rv,
                        const __grid_constant__ CUtensorMap tm_o, const PPParams P) {
    constexpr bool X = (TF & 1) != 0;   // Cross table
    constexpr bool PH = (TF & 2) != 0;  // one R^K per head
    constexpr bool SP = (TF & 4) != 0;  // the tail items may run split
    constexpr bool CL = (TF & 8) != 0;  // token 0 is a class token
    // 65..128 buckets: QR' in two rounds of 64 buckets (shared R^K of 128 rows)
    constexpr int NQR = (TF & 16) != 0 ? 2 : 1;
    // R^K goes with each item (per-head tables, or the class key rows)
    constexpr bool RK_ITEM = PH || CL;
    // the R^K buffer: 64 table rows, then (CL) the slice's first 16 keys; or
    // 128 table rows
    constexpr uint32_t kRkBytes = CL ? 80 * 128 : NQR * (kTileBytes / 2);
    constexpr bool HQ = (TF & 32) != 0;  // query term: K R^Q^T per key tile
    constexpr bool HV = (TF & 64) != 0;  // value term: bucket sums, then PB R^V
    // shared tables loaded once per CTA: R^K (unless it travels with each
    // item), R^Q, R^V
    constexpr bool TABS = (HK && !RK_ITEM) || HQ || HV;
    constexpr uint32_t kTabBytes = ((HK && !RK_ITEM) ? kRkBytes : 0u) +
                                   (HQ ? kTileBytes / 2 : 0u) + (HV ? kTileBytes / 2 : 0u);
    // with the query or value term the QR' table is fp16 (shared memory holds
    // K R^Q^T and PB besides)
    constexpr int QM = HK ? ((HQ || HV) ? 2 : 1) : 0;
    // tensor-memory columns per group: O and two score slots; 224 with the
    // query term, which leaves the last 64 for K R^Q^T
    constexpr uint32_t kGroupCols = HQ ? 224 : 256;
    using G = Geo<W, R>;
    using L = Layout<NG>;
    constexpr int kThreads = L::kThreads;
    static_assert(!(HQ || HV) || (W == 14 && R == 5 && NG == 2 && !X && !PH && !SP && !CL && !BM &&
                                  NQR == 1),
                  "query / value terms: W = 14, five-row tiles, shared tables");
    // score slots: NS columns apart, or 96 with a class token where NS < 80,
    // so that the widened QR' product (80 columns) fits in either slot
    constexpr uint32_t kSlotCols = (CL && G::NS < 80) ? 96u : static_cast<uint32_t>(G::NS);
    static_assert(kColSlot0 + 2 * kSlotCols <= kGroupCols, "tensor-memory columns per group");
    static_assert(!HQ || 2 * kGroupCols + 64 <= 512, "tensor-memory columns");
    // Softmax warps wait with the suspending try (fewer issue slots taken
    // from the warp sharing their scheduler) at W = 14, where that measured
    // faster, and spin at W = 56, where it measured slower; the single-thread
    // producer and issuers always spin (their reaction time matters more).
    constexpr bool kSleep = W == 14;
    extern __shared__ uint8_t smem_raw[];
    // aligned by pointer arithmetic, so the compiler keeps the shared address space
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ PPBars bars;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;
    __shared__ volatile int split_arrivals[2];  // per group: arrivals before this part

    griddep_launch_dependents();
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const WaitCtl &wc = P.wc;
    const WaitCtl drain{wc.status, kDefaultWaitNs};

    uint8_t *sQ = smem + P.off_q;    // nq buffers of two query tiles
    uint8_t *sKV = smem + P.off_kv;  // stage s: K at 2s buffers, V at 2s + 1
    uint8_t *sRK = smem + P.off_rk;
    uint8_t *sLut = smem + P.off_lut + P.lut_pad;

    if (tid == 0) {
        mbar_init(&bars.tab_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.q_full[i], 1);
            mbar_init(&bars.q_empty[i], NG);  // one arrival per group issuer
            mbar_init(&bars.o_full[i], 1);
            mbar_init(&bars.o_empty[i], 128);
            mbar_init(&bars.pv_done[i], 1);
            mbar_init(&bars.fin[i], 1);
            for (int s = 0; s < kMaxSlots; ++s) {
                mbar_init(&bars.slot_full[i][s], 1);
                mbar_init(&bars.slot_done[i][s], 128);
            }
        }
        for (int i = 0; i < kMaxStages; ++i) {
            mbar_init(&bars.kv_full[i], 1);
            mbar_init(&bars.kv_empty[i], NG);  // one arrival per group issuer
        }
        // query term: warps 0-2 of each group (lanes = keys 0..95) copy K R^Q^T;
        // all softmax threads read it
        mbar_init(&bars.kr_tfull, 1);
        mbar_init(&bars.kr_tempty, 3 * NG * 32);
        mbar_init(&bars.kr_sfull, 3 * NG * 32);
        mbar_init(&bars.kr_sempty, 4 * NG * 32);
        for (int i = 0; i < 2; ++i) mbar_init(&bars.pb_full[i], 128);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&tmem_base_s, 256 * NG);
    // K/V buffers: rows KT..NS-1 are never loaded and must hold finite values
    // (the loads write rows 0..KT-1 only, so they may land while these run)
    {
        constexpr int kPadChunks = (G::NS - G::KT) * 128 / 16;
        if constexpr (kPadChunks > 0)
            for (int e = tid; e < P.nst * 2 * kPadChunks; e += kThreads)
                st_shared_v4(smem_u32(sKV) + (e / kPadChunks) * G::KV_BYTES + G::KT * 128 +
                                 (e % kPadChunks) * 16,
                             0u, 0u, 0u, 0u);
    }
    // value term: the bucket sums start at zero (each item's staging step
    // zeroes them again)
    if (HV)
        for (int e = tid; e < NG * static_cast<int>(P.pb_stride) / 16; e += kThreads)
            st_shared_v4(smem_u32(smem + P.off_pb) + e * 16, 0u, 0u, 0u, 0u);
    // Masking operands for the last key tile (128 rows x 16 bf16, K-major, 32-byte
    // swizzle): A has -9984 in column 0 of every row, B has 1 in column 0 of
    // every key row past the grid, so A B^T adds -9984 to exactly those scores.
    {
        uint8_t *mk = smem + P.off_mask;
        for (int e = tid; e < 2 * 4096 / 16; e += kThreads) st_shared_v4(smem_u32(mk) + e * 16, 0u, 0u, 0u, 0u);
        __syncthreads();
        if (tid < 128) {
            const int r = tid;
            const int off = r * 32 + ((r >> 2) & 1) * 16;  // where column 0 of row r lives
            *reinterpret_cast<uint16_t *>(mk + off) = 0xC61Cu;  // bf16 -9984
            if (r >= P.nvalid_last) *reinterpret_cast<uint16_t *>(mk + 4096 + off) = 0x3F80u;  // bf16 1
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    // everything above touches no input: it may overlap the previous kernel
    griddep_wait();
    // The offset table goes to shared memory on the softmax warps, after the
    // roles split, so the producer's first loads overlap the copy. Named
    // barrier 3 tells its readers it is complete: the softmax warps and, with
    // the value term, the control warp of CTA 0 that checks its row runs.
    constexpr bool kLut = HK || BM || HQ || HV;
    const int lut_bar_count = 4 * NG * 32 + ((HV && blockIdx.x == 0) ? 32 : 0);
    if (warp >= 4 * NG) {
        regs_dealloc<L::kRegsControl>();
        if (warp == 4 * NG) {
            // -------------------------------------------- TMA producer
            if (lane == 0) {
                prefetch_tmap(&tm_q);
                prefetch_tmap(&tm_k);
                prefetch_tmap(&tm_v);
                if (TABS) mbar_arrive_expect_tx(&bars.tab_full, kTabBytes);
                if (HK && !RK_ITEM) {
                    // 32-row boxes: table rows 0.. and rows tab_row2.. (for Cross
                    // tables the column buckets land at row 32), then 64.. and 96..
                    tma_load_3d(sRK, &tm_rk, &bars.tab_full, 0, 0, 0);
                    tma_load_3d(sRK + 4096, &tm_rk, &bars.tab_full, 0, P.tab_row2, 0);
                    if (NQR == 2) {
                        tma_load_3d(sRK + 8192, &tm_rk, &bars.tab_full, 0, 64, 0);
                        tma_load_3d(sRK + 12288, &tm_rk, &bars.tab_full, 0, 96, 0);
                    }
                }
                // R^Q and R^V: 64 rows each (rows past the bucket count read as zero)
                if (HQ) {
                    tma_load_3d(smem + P.off_rq, &tm_rq, &bars.tab_full, 0, 0, 0);
                    tma_load_3d(smem + P.off_rq + 4096, &tm_rq, &bars.tab_full, 0, 32, 0);
                }
                if (HV) {
                    tma_load_3d(smem + P.off_rv, &tm_rv, &bars.tab_full, 0, 0, 0);
                    tma_load_3d(smem + P.off_rv + 4096, &tm_rv, &bars.tab_full, 0, 32, 0);
                }
                int g = 0, it = 0;
                int last_q[2] = {-1, -1};
                int last_use[kMaxStages];
                for (int st = 0; st < kMaxStages; ++st) last_use[st] = -1;
                bool ok = true;
                for (int item = item_at<SP>(P, 0); ok && item >= 0; item = item_at<SP>(P, ++it)) {
                    const Item I = decode_item<SP>(P, item);
                    const int qb = it % P.nq, quse = it / P.nq;
                    if (!(ok = mbar_wait(&bars.q_empty[qb], (quse & 1) ^ 1, wc, kStatusTimeoutSync,
                                         &abort_flag, false)))
                        break;
                    uint8_t *qd = sQ + qb * NG * kTileBytes;
                    // per-head tables travel with the item's Q tiles: the Q buffer's
                    // release (after both groups' last products) frees its table too
                    constexpr bool tab_item = HK && RK_ITEM;
                    mbar_arrive_expect_tx(&bars.q_full[qb], (I.has_b ? 2 : 1) * kTileBytes +
                                                                (tab_item ? kRkBytes : 0));
                    if (tab_item) {
                        uint8_t *rd = sRK + qb * kRkBytes;
                        const int head = PH ? I.slice % P.heads : 0;
                        tma_load_3d(rd, &tm_rk, &bars.q_full[qb], 0, 0, head);
                        tma_load_3d(rd + 4096, &tm_rk, &bars.q_full[qb], 0, P.tab_row2, head);
                        // keys 0..15 of the slice (key 0: the class token) as rows 64..79
                        if (CL) tma_load_3d(rd + 8192, &tm_kc, &bars.q_full[qb], 0, 0, I.slice);
                    }
                    tma_load_3d(qd, &tm_q, &bars.q_full[qb], 0, I.qt0 * 128, I.slice);
                    if (I.has_b)
                        tma_load_3d(qd + kTileBytes, &tm_q, &bars.q_full[qb], 0, (I.qt0 + 1) * 128,
                                    I.slice);
                    last_q[qb] = quse;
                    for (int kt = I.kt0; kt < I.kt1; ++kt, ++g) {
                        const int st = g % P.nst, use = g / P.nst;
                        if (!(ok = mbar_wait(&bars.kv_empty[st], (use & 1) ^ 1, wc,
                                             kStatusTimeoutSync, &abort_flag, false)))
                            break;
                        uint8_t *kb = sKV + st * 2 * G::KV_BYTES;
                        mbar_arrive_expect_tx(&bars.kv_full[st], 2 * G::KT * 128);
                        // the grid keys are tokens 1.. when token 0 is a class token
                        const int k0 = (CL ? 1 : 0) + kt * G::KT;
                        tma_load_3d(kb, &tm_k, &bars.kv_full[st], 0, k0, I.slice);
                        tma_load_3d(kb + G::KV_BYTES, &tm_v, &bars.kv_full[st], 0, k0, I.slice);
                        last_use[st] = use;
                    }
                }
                // drain: the most recent load on every barrier has landed
                if (TABS) mbar_wait(&bars.tab_full, 0, drain, kStatusTimeoutDrain, nullptr);
                for (int b = 0; b < 2; ++b)
                    if (last_q[b] >= 0)
                        mbar_wait(&bars.q_full[b], last_q[b] & 1, drain, kStatusTimeoutDrain, nullptr);
                for (int st = 0; st < kMaxStages; ++st)
                    if (last_use[st] >= 0)
                        mbar_wait(&bars.kv_full[st], last_use[st] & 1, drain, kStatusTimeoutDrain,
                                  nullptr);
            }
            __syncwarp();
        } else if (warp > 4 * NG && warp <= 5 * NG) {
            // -------------------------------------------- MMA issuer of group w
            // The order is fixed: unit u is issued once unit u - SLOTS has been
            // consumed (and, for a tile's scores, its P V issued), so
            // the issuer is a straight sequence of bounded blocking waits. For
            // items the group sits out it still releases the item's Q buffer and
            // K/V stages, each after the matching load has landed.
            const int w = warp - (4 * NG + 1);
            if (lane == 0) {
                constexpr uint32_t kIdS = idesc_bf16(128, G::NS, false, false);
                // QR' = Q R^K^T: 64 bucket columns, and (CL) 16 more against the
                // slice's first keys, of which column 64 is q . k_class
                constexpr uint32_t kIdQR = idesc_bf16(128, CL ? 80 : 64, false, false);
                constexpr uint32_t kIdO = idesc_bf16(128, 64, false, true);
                constexpr uint32_t kIdKR = idesc_bf16(128, 64, false, false);
                const uint64_t hi128 = smem_desc(0, 16, 1024, kSwizzle128B);
                const uint32_t tG = tmem + w * kGroupCols;
                const uint32_t aQ = smem_u32(sQ + w * kTileBytes);
                const uint32_t aKV = smem_u32(sKV);
                // outstanding units, oldest first: bits 0-3 stage, 4 QR unit, 5 first
                // tile of the item, 6 last tile of the item
                uint32_t pend0 = 0, pend1 = 0, pend2 = 0;
                int np = 0;
                uint32_t u = 0;  // units issued
                int ci = 0;      // items whose last P V was issued
                bool ok = true;
                if (TABS) ok = mbar_wait(&bars.tab_full, 0, wc, kStatusTimeoutLoad, &abort_flag, false);
                // consume the oldest outstanding unit: wait until the group has
                // released it, then issue its P V
                auto consume = [&]() {
                    const uint32_t x = pend0;
                    const uint32_t cu = u - np;
                    pend0 = pend1;
                    pend1 = pend2;
                    --np;
                    ok = ok && mbar_wait(&bars.slot_done[w][cu % G::SLOTS], (cu / G::SLOTS) & 1, wc,
                                         kStatusTimeoutSync, &abort_flag, false);
                    if (!ok || (x & 0x10u)) return;
                    if (x & 0x20u)
                        ok = mbar_wait(&bars.o_empty[w], (ci & 1) ^ 1, wc, kStatusTimeoutSync, &abort_flag, false);
                    if (!ok) return;
                    tc_fence_after();
                    const int st = x & 0xF;
                    const uint64_t dV = hi128 | ((aKV + (st * 2 + 1) * G::KV_BYTES) >> 4);
                    const uint32_t aP = tG + kColSlot0 + (cu % G::SLOTS) * kSlotCols;
                    const uint32_t acc0 = (x & 0x20u) ? 0u : 1u;
#pragma unroll
                    for (int kk = 0; kk < G::NS / 16; ++kk)
                        mma_bf16_ts(tG, aP + p_col<W, R>(kk), dV + kk * (2048 >> 4), kIdO,
                                    kk > 0 ? 1u : acc0);
                    mma_commit(&bars.pv_done[w]);
                    mma_commit(&bars.kv_empty[st]);
                    if (x & 0x40u) {
                        if (HV) {
                            // the value term: O += PB R^V once the group has staged
                            // its bucket sums (A: PB, 128 rows x 64 buckets, K-major
                            // in the staging tile; B: R^V [bucket][d], like V)
                            ok = mbar_wait(&bars.pb_full[w], ci & 1, wc, kStatusTimeoutSync, &abort_flag, false);
                            if (!ok) return;
                            tc_fence_after();
                            const uint64_t dPB = hi128 | (smem_u32(smem + P.off_stage + w * kTileBytes) >> 4);
                            const uint64_t dRV = hi128 | (smem_u32(smem + P.off_rv) >> 4);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_bf16_ss(tG, dPB + kk * 2, dRV + kk * (2048 >> 4), kIdO, 1u);
                        }
                        mma_commit(&bars.o_full[w]);
                        ++ci;
                    }
                };
                int g = 0, it = 0;
                for (int item = item_at<SP>(P, 0); ok && item >= 0; item = item_at<SP>(P, ++it)) {
                    const Item I = decode_item<SP>(P, item);
                    const int qb = it % P.nq;
                    ok = mbar_wait(&bars.q_full[qb], (it / P.nq) & 1, wc, kStatusTimeoutLoad, &abort_flag, false);
                    if (w == 1 && !I.has_b) {
                        // the outstanding units' P V release K/V stages that the
                        // loads below may be waiting for: issue them first
                        while (ok && np > 0) consume();
                        for (int kt = I.kt0; ok && kt < I.kt1; ++kt, ++g) {
                            const int st = g % P.nst;
                            ok = mbar_wait(&bars.kv_full[st], (g / P.nst) & 1, wc, kStatusTimeoutLoad,
                                           &abort_flag, false);
                            if (ok) mbar_arrive(&bars.kv_empty[st]);
                        }
                        if (ok) mbar_arrive(&bars.q_empty[qb]);
                        continue;
                    }
                    const uint64_t dQ = hi128 | ((aQ + qb * NG * kTileBytes) >> 4);
                    for (int kt = HK ? I.kt0 - NQR : I.kt0; ok && kt < I.kt1; ++kt) {
                        if (np == G::SLOTS) consume();
                        if (!ok) break;
                        const uint32_t slot = u % G::SLOTS;
                        const uint32_t dS = tG + kColSlot0 + slot * kSlotCols;
                        uint32_t code;
                        if (kt < I.kt0) {  // a QR' unit (round kt - kt0 + NQR)
                            tc_fence_after();
                            const uint32_t rk_off = (RK_ITEM ? qb * kRkBytes : 0) +
                                                    (kt - I.kt0 + NQR) * (kTileBytes / 2);
                            const uint64_t dRK = hi128 | (smem_u32(sRK + rk_off) >> 4);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_bf16_ss(dS, dQ + kk * 2, dRK + kk * 2, kIdQR, kk > 0);
                            code = 0x10u;
                        } else {
                            const int st = g % P.nst;
                            ok = mbar_wait(&bars.kv_full[st], (g / P.nst) & 1, wc, kStatusTimeoutLoad,
                                           &abort_flag, false);
                            if (!ok) break;
                            tc_fence_after();
                            const uint64_t dK = hi128 | ((aKV + st * 2 * G::KV_BYTES) >> 4);
                            if (HQ && w == 0) {
                                // the query term: K R^Q^T of this key tile (rows =
                                // keys; lanes past the tile's keys are not read),
                                // once the previous tile's copy has left tensor memory
                                ok = mbar_wait(&bars.kr_tempty, (g & 1) ^ 1, wc, kStatusTimeoutSync,
                                               &abort_flag, false);
                                if (!ok) break;
                                tc_fence_after();
                                const uint64_t dRQ = hi128 | (smem_u32(smem + P.off_rq) >> 4);
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    mma_bf16_ss(tmem + kKrCol, dK + kk * 2, dRQ + kk * 2, kIdKR, kk > 0);
                                mma_commit(&bars.kr_tfull);
                            }
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_bf16_ss(dS, dQ + kk * 2, dK + kk * 2, kIdS, kk > 0);
                            const bool last = kt == P.nkt - 1;
                            if (last && P.nvalid_last < G::KT) {
                                const uint64_t dMA = smem_desc(smem_u32(smem + P.off_mask), 16, 256, kSwizzle32B);
                                mma_bf16_ss(dS, dMA, dMA + (4096 >> 4), kIdS, 1u);
                            }
                            code = static_cast<uint32_t>(st) | (kt == I.kt0 ? 0x20u : 0u) | (kt == I.kt1 - 1 ? 0x40u : 0u);
                            ++g;
                        }
                        mma_commit(&bars.slot_full[w][slot]);
                        if (kt == I.kt1 - 1) mma_commit(&bars.q_empty[qb]);
                        if (np == 0) pend0 = code; else if (np == 1) pend1 = code; else pend2 = code;
                        ++np;
                        ++u;
                    }
                }
                while (ok && np > 0) consume();
                // drain: a last commit completes after every product this thread issued
                mma_commit(&bars.fin[w]);
                mbar_wait(&bars.fin[w], 0, drain, kStatusTimeoutDrain, nullptr);
            }
            __syncwarp();
        } else if (HV && blockIdx.x == 0) {
            named_bar_sync(3, lut_bar_count);
            // The value term's bucket sums rely on each id forming one run
            // along a grid row of keys, seen from any query column; the call
            // checked that once per table. A table rewritten in place since then
            // is caught here, by the otherwise idle control warp of one CTA (the
            // table is the same for all): one offset-table row and query column
            // per lane at a time (ids < 64).
            for (int e = lane; e < (2 * P.H - 1) * W; e += 32) {
                const uint8_t *row = sLut + (e / W) * G::COLS + (e % W) + (W - 1);
                unsigned long long ended = 0ull;
                int prev = -1;
                bool bad = false;
                for (int kx = 0; kx < W; ++kx) {
                    const int id = row[-kx];
                    if (id == prev) continue;
                    bad = bad || ((ended >> id) & 1ull) != 0ull;
                    if (prev >= 0) ended |= 1ull << prev;
                    prev = id;
                }
                if (bad) atomicOr(wc.status, kStatusBadBucket);
            }
        }
    } else {
        regs_alloc<L::kRegsSoftmax>();
        if (kLut) {
            // offset table as bytes. The call checked its ids on the host (once
            // per table); an id outside [0, bound) -- the class bucket excluded --
            // sets the status bit and is clamped so no read leaves shared memory.
            // Keys past the last grid row index up to lut_pad bytes before the
            // table; those bytes hold bucket 0 so every read stays in bounds
            // (those scores are masked).
            constexpr int kCopiers = 4 * NG * 32;
            const int bound = P.nb - (CL ? 1 : 0);
            auto clamp_id = [&](int id) -> uint32_t {
                if (id < 0 || id >= bound) atomicOr(wc.status, kStatusBadBucket);
                return static_cast<uint32_t>(id < 0 ? 0 : (id >= bound ? bound - 1 : id));
            };
            for (int e = tid; e < P.lut_pad; e += kCopiers) sLut[e - P.lut_pad] = 0;
            // four ids per 16-byte load (the table and sLut are 16-byte aligned),
            // stored as one word of four bytes; then the last lut_len % 4 ids
            const int n4 = P.lut_len >> 2;
            for (int e = tid; e < n4; e += kCopiers) {
                const int4 v = __ldg(reinterpret_cast<const int4 *>(P.lut) + e);
                reinterpret_cast<uint32_t *>(sLut)[e] =
                    clamp_id(v.x) | (clamp_id(v.y) << 8) | (clamp_id(v.z) << 16) | (clamp_id(v.w) << 24);
            }
            for (int e = 4 * n4 + tid; e < P.lut_len; e += kCopiers)
                sLut[e] = static_cast<uint8_t>(clamp_id(__ldg(P.lut + e)));
            if (CL)
                for (int e = tid; e < P.cls_len; e += kCopiers)
                    sLut[P.lut_len + e] = static_cast<uint8_t>(P.nb - 1);
            named_bar_sync(3, lut_bar_count);
        }
        // ------------------------------------------------ softmax groups
        // One thread per query row. Decisions to go on or stop are uniform per
        // warp within an item and over the whole group twice per item (at its
        // start and before the epilogue); a warp that stops mid-item goes
        // straight to the second group vote, so every group barrier is reached
        // by all of the group's warps.
        const int wg = warp >> 2;        // query tile of the pair
        const int lq = warp & 3;         // tensor-memory lane quarter
        const int t = lq * 32 + lane;    // row within the query tile
        const int group_bar = 1 + wg;
        const bool leader = lq == 0 && lane == 0;
        const uint32_t lane_off = static_cast<uint32_t>(lq * 32) << 16;
        const uint32_t tG = tmem + wg * kGroupCols;
        const uint32_t tOl = tG + lane_off;
        // The group's QR' table [bucket][128 rows], fp32 (fp16 with the query or
        // value term); a thread reads and writes only its own row of it.
        uint8_t *qr_base = smem + P.off_qr + wg * P.qr_stride;
        float *qr_t = reinterpret_cast<float *>(qr_base) + t;
        uint16_t *qr_h = reinterpret_cast<uint16_t *>(qr_base) + t;
        // query term: the key tile's K R^Q^T [key][bucket] (fp16, scaled), shared
        // by both groups; value term: this row's bucket sums PB [bucket][128 rows]
        const uint16_t *kr_tab = reinterpret_cast<const uint16_t *>(smem + P.off_kr);
        float *pb_t = reinterpret_cast<float *>(smem + P.off_pb + wg * P.pb_stride) + t;
        // bias mode: the item's head's bias row, scaled, in the same region
        float *bias_row = reinterpret_cast<float *>(qr_base);
        const uint32_t *lutw = reinterpret_cast<const uint32_t *>(sLut);
        uint32_t u = 0;  // this group's unit counter
        int it_w = 0, gw = 0;
        // The group's output staging tile (128 rows x 128 bytes, 128-byte
        // swizzle) for the TMA store; a thread writes only its own row.
        uint8_t *stage = smem + P.off_stage + wg * kTileBytes;
        const uint32_t stage_row = smem_u32(stage) + t * 128;
        // The item whose epilogue is still due. It runs after the next item's QR'
        // copy (or after the last item), so that the copy overlaps the wait for
        // the item's last P V.
        bool ok = true, due = false;
        Item D{};
        float due_m = 0.f, due_l = 1.f, due_xc = -INFINITY;
        auto epilogue = [&]() -> bool {
            const bool okd = ok && __all_sync(~0u, mbar_wait(&bars.o_full[wg], it_w & 1, wc,
                                                            kStatusTimeoutMma, &abort_flag, kSleep));
            // the previous TMA store has read the staging tile (the vote's
            // barrier orders this before the group's staging writes)
            if (leader) bulk_wait_read_all();
            if (!red_and(group_bar, 128, okd)) return false;
            tc_fence_after();
            const int dqt = D.qt0 + wg;
            const bool dactive = dqt * 128 + lq * 32 < P.N;
            float inv = 1.f / due_l;
            // CL: fold the class key into the row: reference max mm, O and l
            // scaled by 2^(m - mm), the key's weight 2^(x_c - mm) times v_class
            float o_scale = 1.f, p_cls = 0.f;
            const uint4 *v_cls = nullptr;
            if (CL && dactive) {
                const float mm = fmaxf(due_m, due_xc);
                o_scale = ex2_approx(due_m - mm);
                p_cls = ex2_approx(due_xc - mm);
                inv = 1.f / (due_l * o_scale + p_cls);
                v_cls = reinterpret_cast<const uint4 *>(P.v_cls + static_cast<size_t>(D.slice) * P.N * 64);
            }
            // A part of a split tail item hands its unnormalised state (O, m, l)
            // to the workspace and counts its arrival; the later of the two
            // parts merges the other's state into its own and writes the
            // output, the earlier one is done. No part waits for the other.
            float a_self = 1.f, a_other = 0.f;
            const float *other = nullptr;
            if (SP && D.part != 0) {
                constexpr size_t kSlot = 66 * 128;  // O [64][128], m [128], l [128]
                const size_t pair = static_cast<size_t>(D.tidx * 2 + wg) * 2;
                float *mine = P.ws + (pair + (D.part - 1)) * kSlot;
                if (dactive) {
#pragma unroll
                    for (int c2 = 0; c2 < 4; ++c2) {
                        uint32_t o[16];
                        tmem_ld16(tOl + 16 * c2, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int e = 0; e < 16; ++e) mine[(16 * c2 + e) * 128 + t] = __uint_as_float(o[e]);
                    }
                    mine[64 * 128 + t] = due_m;
                    mine[65 * 128 + t] = due_l;
                }
                __threadfence();
                named_bar_sync(group_bar, 128);
                if (leader) split_arrivals[wg] = atomicAdd(P.cnt + D.tidx * 2 + wg, 1);
                named_bar_sync(group_bar, 128);
                if (split_arrivals[wg] == 0) {
                    tc_fence_before();
                    mbar_arrive(&bars.o_empty[wg]);
                    ++it_w;
                    return true;
                }
                __threadfence();
                if (leader) P.cnt[D.tidx * 2 + wg] = 0;  // both arrived: ready for the next launch
                other = P.ws + (pair + (2 - D.part)) * kSlot;
                if (dactive) {
                    // symmetric in the two parts (separately rounded products, one
                    // sum), so the result does not depend on which part came later
                    const float m2 = __ldcg(other + 64 * 128 + t), l2 = __ldcg(other + 65 * 128 + t);
                    const float mm = fmaxf(due_m, m2);
                    a_self = ex2_approx(due_m - mm);
                    a_other = ex2_approx(m2 - mm);
                    inv = 1.f / (__fmul_rn(due_l, a_self) + __fmul_rn(l2, a_other));
                }
            }
            // normalise the row's 64 output columns into the staging tile, 16 at a time
#pragma unroll
            for (int c2 = 0; c2 < 4; ++c2) {
                uint32_t o[16];
                if (dactive) {
                    tmem_ld16(tOl + 16 * c2, o);
                    tmem_ld_wait(o);
                    if (other != nullptr) {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            o[e] = __float_as_uint(__fmul_rn(__uint_as_float(o[e]), a_self) +
                                                   __fmul_rn(__ldcg(other + (16 * c2 + e) * 128 + t), a_other));
                    }
                    if (CL) {
                        // 16 bf16 of v_class (the same row for every thread: broadcast)
                        const uint4 va = __ldg(v_cls + 2 * c2), vb = __ldg(v_cls + 2 * c2 + 1);
                        const uint32_t vw[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const uint32_t w = vw[e >> 1];
                            const float ve = __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
                            o[e] = __float_as_uint(fmaf(__uint_as_float(o[e]), o_scale, p_cls * ve));
                        }
                    }
                }
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const uint32_t *src = o + 8 * c;
                    const int chunk = 2 * c2 + c;
                    st_shared_v4(stage_row + ((chunk ^ (t & 7)) << 4),
                                 pack_bf16x2(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv),
                                 pack_bf16x2(__uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv),
                                 pack_bf16x2(__uint_as_float(src[4]) * inv, __uint_as_float(src[5]) * inv),
                                 pack_bf16x2(__uint_as_float(src[6]) * inv, __uint_as_float(src[7]) * inv));
                }
            }
            tc_fence_before();
            mbar_arrive(&bars.o_empty[wg]);
            fence_proxy_async_smem();
            named_bar_sync(group_bar, 128);
            if (leader) {
                // rows past the grid fall outside the tensor map and are not written
                tma_store_3d(&tm_o, stage, 0, dqt * 128, D.slice);
                bulk_commit_group();
            }
            ++it_w;
            return true;
        };
        for (int item = item_at<SP>(P, 0), k_item = 0; item >= 0; item = item_at<SP>(P, ++k_item)) {
            const Item I = decode_item<SP>(P, item);
            if (wg == 1 && !I.has_b) continue;
            const int qt = I.qt0 + wg;
            const int i = qt * 128 + t;
            const bool warp_active = qt * 128 + lq * 32 < P.N;
            const int ic = i < P.N ? i : P.N - 1;
            // the row's grid position (CL: token t >= 1 is grid token t - 1); the
            // class query reads the class-bucket region after the offset table
            const int pi = CL ? ic - 1 : ic;
            const int base_i = pi < 0 ? P.cls_base
                                      : (pi / W) * G::COLS + (pi % W) + (P.H - 1) * G::COLS + (W - 1);
            uint32_t slot = u % G::SLOTS;
            if (HK)
                ok = __all_sync(~0u, mbar_wait(&bars.slot_full[wg][slot], (u / G::SLOTS) & 1, wc,
                                               kStatusTimeoutMma, &abort_flag, kSleep)) && ok;
            if (!red_and(group_bar, 128, ok)) {
                ok = false;
                break;
            }
            if (BM) {
                // the item's bias row, pre-scaled like the logits (eq. 13: inside
                // the 1/sqrt(d) scaling); visible to the group after the barrier
                const int col = P.bias_heads == 1 ? 0 : I.slice % P.heads;
                if (t < P.nb) {
                    // Cross: joint id a*span + b takes row bucket a plus column bucket span + b
                    const int r0 = X ? t / P.cross : t;
                    float b = __ldg(P.bias + r0 * P.bias_heads + col);
                    if (X) b += __ldg(P.bias + (P.cross + t % P.cross) * P.bias_heads + col);
                    bias_row[t] = b * P.c;
                }
                named_bar_sync(group_bar, 128);
            }
            float xc = -INFINITY;  // CL: the class key's logit for this row
            if (HK) {
                tc_fence_after();
                if (warp_active) {
                    uint32_t r0[32], r1[32], rk[16];
                    tmem_ld32(tG + kColSlot0 + slot * kSlotCols + lane_off, r0);
                    tmem_ld32(tG + kColSlot0 + slot * kSlotCols + lane_off + 32, r1);
                    if (CL) tmem_ld16(tG + kColSlot0 + slot * kSlotCols + lane_off + 64, rk);
                    tmem_ld_wait();
                    tmem_ready(r0);
                    tmem_ready(r1);
                    if (CL) tmem_ready(rk);
                    if constexpr (X) {
                        // joint id a*span + b: row bucket a (column a) plus column
                        // bucket span + b (staged at table row 32 + b)
#pragma unroll
                        for (int a = 0; a < 8; ++a)
#pragma unroll
                            for (int b = 0; b < 8; ++b)
                                if (a < P.cross && b < P.cross)
                                    qr_t[(a * P.cross + b) * 128] =
                                        (__uint_as_float(r0[a]) + __uint_as_float(r1[b])) * P.c;
                    } else {
#pragma unroll
                        for (int b = 0; b < 64; ++b)
                            if (b < P.nb) {
                                const float qv = __uint_as_float(b < 32 ? r0[b] : r1[b - 32]) * P.c;
                                if (QM == 2)
                                    qr_h[b * 128] = f32_to_f16(qv);
                                else
                                    qr_t[b * 128] = qv;
                            }
                        // the class key: q . k_class plus the class bucket's term,
                        // both inside the scaling (eq. 13)
                        if (CL) xc = __uint_as_float(rk[0]) * P.c + qr_t[(P.nb - 1) * 128];
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars.slot_done[wg][slot]);
                ++u;
                // the second QR' round: buckets 64.. into rows 64.. of the table
                if (NQR == 2) {
                    slot = u % G::SLOTS;
                    ok = __all_sync(~0u, mbar_wait(&bars.slot_full[wg][slot], (u / G::SLOTS) & 1, wc,
                                                   kStatusTimeoutMma, &abort_flag, kSleep)) && ok;
                    if (ok) {
                        tc_fence_after();
                        if (warp_active) {
                            uint32_t r0[32], r1[32];
                            tmem_ld32(tG + kColSlot0 + slot * kSlotCols + lane_off, r0);
                            tmem_ld32(tG + kColSlot0 + slot * kSlotCols + lane_off + 32, r1);
                            tmem_ld_wait();
                            tmem_ready(r0);
                            tmem_ready(r1);
#pragma unroll
                            for (int b = 0; b < 64; ++b)
                                if (64 + b < P.nb)
                                    qr_t[(64 + b) * 128] = __uint_as_float(b < 32 ? r0[b] : r1[b - 32]) * P.c;
                        }
                        tc_fence_before();
                        mbar_arrive(&bars.slot_done[wg][slot]);
                        ++u;
                    }
                }
            }
            if (due && !epilogue()) {
                ok = false;
                break;
            }
            float m = -INFINITY, l = 0.f;
            for (int kt = I.kt0; kt < I.kt1; ++kt, ++gw, ++u) {
                if (HQ) {
                    // warps 0-2 of each group copy this key tile's K R^Q^T from
                    // tensor memory (lane = key) to the shared table, scaled
                    // like the logits: group w the buckets 32 w .. 32 w + 31
                    if (lq < 3) {
                        ok = __all_sync(~0u, mbar_wait(&bars.kr_tfull, gw & 1, wc, kStatusTimeoutMma,
                                                       &abort_flag, kSleep)) && ok;
                        if (!ok) break;
                        tc_fence_after();
                        uint32_t kr[32];
                        tmem_ld32(tmem + kKrCol + 32 * wg + lane_off, kr);
                        tmem_ld_wait();
                        tmem_ready(kr);
                        tc_fence_before();
                        mbar_arrive(&bars.kr_tempty);
                        ok = __all_sync(~0u, mbar_wait(&bars.kr_sempty, (gw & 1) ^ 1, wc,
                                                       kStatusTimeoutSync, &abort_flag, kSleep)) && ok;
                        if (!ok) break;
                        if (t < G::KT) {
                            const uint32_t dst = smem_u32(kr_tab) + t * kKrStride + wg * 64;
#pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4) {
                                const uint32_t *v = kr + 8 * c4;
                                st_shared_v4(dst + 16 * c4,
                                             pack_f16x2(__uint_as_float(v[0]) * P.c, __uint_as_float(v[1]) * P.c),
                                             pack_f16x2(__uint_as_float(v[2]) * P.c, __uint_as_float(v[3]) * P.c),
                                             pack_f16x2(__uint_as_float(v[4]) * P.c, __uint_as_float(v[5]) * P.c),
                                             pack_f16x2(__uint_as_float(v[6]) * P.c, __uint_as_float(v[7]) * P.c));
                            }
                        }
                        mbar_arrive(&bars.kr_sfull);
                    }
                    ok = __all_sync(~0u, mbar_wait(&bars.kr_sfull, gw & 1, wc, kStatusTimeoutSync,
                                                   &abort_flag, kSleep)) && ok;
                    if (!ok) break;
                }
                slot = u % G::SLOTS;
                ok = __all_sync(~0u, mbar_wait(&bars.slot_full[wg][slot], (u / G::SLOTS) & 1, wc,
                                               kStatusTimeoutMma, &abort_flag, kSleep)) && ok;
                if (!ok) break;
                tc_fence_after();
                const uint32_t tSl = tG + kColSlot0 + slot * kSlotCols + lane_off;
                const int e0 = base_i - kt * G::R * G::COLS;
                using Tile = HalfTile<W, R, HK || BM, 0, BM ? 1 : 128, BM ? 1 : QM, HQ>;
                if (warp_active) {
                    uint32_t xs[Tile::NQ][16];  // the row's logits, pass 1 to pass 2
                    const float mt = Tile::logits(tSl, lutw, e0,
                                                  BM ? static_cast<const void *>(bias_row)
                                                     : QM == 2 ? static_cast<const void *>(qr_h)
                                                               : static_cast<const void *>(qr_t),
                                                  kr_tab, P.c, xs);
                    if (HQ) mbar_arrive(&bars.kr_sempty);
                    // lazy rescale: the reference max moves only when it grows by > 2^8
                    float alpha = 1.f;
                    if (mt > m + kRescaleLog2) {
                        alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - mt);
                        m = mt;
                        l *= alpha;
                    }
                    if (kt > I.kt0 && __any_sync(~0u, alpha < 1.f)) {
                        ok = rescale_o(alpha, tOl, &bars.pv_done[wg], (gw - 1) & 1, wc, &abort_flag, kSleep);
                        // the bucket sums carry the same reference max as O
                        if (HV && alpha < 1.f) {
#pragma unroll 1
                            for (int b = 0; b < P.nb; ++b) pb_t[b * 128] *= alpha;
                        }
                    }
                    l += Tile::template probs<HV>(tSl, m, xs);
                    if (HV) {
                        // grid rows of this tile that lie on the grid
                        const int rows = min(G::R, P.H - kt * G::R);
                        Tile::bucket_sums(lutw, e0, pb_t, rows, xs);
                    }
                    tmem_st_wait();
                } else if (HQ) {
                    mbar_arrive(&bars.kr_sempty);
                }
                tc_fence_before();
                mbar_arrive(&bars.slot_done[wg][slot]);
            }
            if (HV) {
                // the item's bucket sums become the A operand of PB R^V: bf16, 128
                // rows x 64 buckets (K-major, 128-byte swizzle) in the group's
                // staging tile, once the previous output store has read it; the
                // sums go back to zero for the next item
                if (leader) bulk_wait_read_all();
                if (red_and(group_bar, 128, ok)) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int b = 8 * c + e;
                            v[e] = 0.f;
                            if (b < P.nb) {
                                v[e] = pb_t[b * 128];
                                pb_t[b * 128] = 0.f;
                            }
                        }
                        st_shared_v4(stage_row + ((c ^ (t & 7)) << 4), pack_bf16x2(v[0], v[1]),
                                     pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                     pack_bf16x2(v[6], v[7]));
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(&bars.pb_full[wg]);
                } else {
                    ok = false;
                }
            }
            due = true;
            D = I;
            due_m = m;
            due_xc = xc;
            due_l = l;
        }
        if (due) epilogue();
        if (leader) bulk_wait_all();
    }
    tc_fence_before();
    asm volatile("barrier.sync 0;" ::: "memory");
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256 * NG);
    }
}

uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

template <int W, int R, bool HK, int NG, bool BM, int TF>
cudaError_t launch_pp(const RpeBf16Args &a, cudaStream_t stream) {
    using G = Geo<W, R>;
    using L = Layout<NG>;
    PPParams p{};
    constexpr bool CL = (TF & 8) != 0;
    constexpr int NQR = (TF & 16) != 0 ? 2 : 1;
    constexpr bool HQ = (TF & 32) != 0, HV = (TF & 64) != 0;
    constexpr uint32_t kRkBytes = CL ? 80 * 128 : NQR * (kTileBytes / 2);
    const int N = a.H * a.W + (CL ? 1 : 0);  // tokens (token 0: the class token)
    p.N = N;
    p.H = a.H;
    p.cross = a.cross_span;
    p.nb = a.cross_span > 0 ? a.cross_span * a.cross_span : a.num_buckets;
    p.tab_row2 = a.cross_span > 0 ? a.cross_span : 32;
    p.tab_heads = a.tab_heads;
    p.nkt = (a.H + G::R - 1) / G::R;
    p.qtiles = (N + 127) / 128;
    p.pairs_full = p.qtiles / 2;
    p.slices = a.B * a.heads;
    p.single = NG == 1;
    p.items = NG == 1 ? p.slices * p.qtiles
                      : p.slices * p.pairs_full + ((p.qtiles & 1) ? p.slices : 0);
    p.lut_len = (2 * a.H - 1) * (2 * a.W - 1);
    p.lut_pad = static_cast<int>(align_up(G::R * G::COLS + 4, 16));
    p.nvalid_last = a.H * a.W - (p.nkt - 1) * G::KT;  // grid keys of the last tile
    // class-bucket region: the class query's offset reads reach back nkt R COLS
    // bytes from cls_base and forward less than W + 16
    p.cls_base = CL ? p.lut_len + 32 + p.nkt * G::R * G::COLS : 0;
    p.cls_len = CL ? 32 + p.nkt * G::R * G::COLS + W + 48 : 0;
    p.v_cls = static_cast<const uint16_t *>(a.v);
    p.lut = a.lut;
    p.c = static_cast<float>(kLog2e / std::sqrt(static_cast<double>(kD)));
    p.bias = a.bias;
    p.bias_heads = a.bias_heads;
    p.heads = a.heads;
    // per CTA: the SM's 228 KB less 1 KB reserved per CTA, less the kernel's
    // static shared memory
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, rpe_pingpong_kernel<W, R, HK, NG, BM, TF>) != cudaSuccess)
        return cudaErrorInvalidValue;
    const uint32_t cap = (228 / L::kCtasPerSm - 1) * 1024 - static_cast<uint32_t>(fa.sharedSizeBytes);
    uint32_t total = 0;
    // as many K/V stages as fit (up to kMaxStages) next to a double-buffered Q;
    // a single Q buffer only when that leaves fewer than three stages
    for (int nq = 2; nq >= 1; --nq) {
        p.nq = nq;
        uint32_t off = 0;
        p.off_q = off;
        off += nq * NG * kTileBytes;
        p.off_rk = off;
        if (HK) off += ((a.tab_heads > 1 || CL) ? nq : 1) * kRkBytes;
        p.off_rq = off;
        if (HQ) off += kTileBytes / 2;
        p.off_rv = off;
        if (HV) off += kTileBytes / 2;
        p.off_qr = off;
        // each group's QR' table (or bias row); fp16 next to the query or value term
        p.qr_stride = (HQ || HV) ? align_up(HK ? p.nb * 256 : 0, 16)
                                 : align_up(std::max(HK ? p.nb * 512 : 0, BM ? 512 : 0), 1024);
        off += NG * p.qr_stride;
        // the key tile's K R^Q^T [key][bucket], fp16
        p.off_kr = off;
        if (HQ) off += G::NS * kKrStride;
        // each group's bucket sums [bucket][128 rows], fp32
        p.off_pb = off;
        p.pb_stride = HV ? p.nb * 512 : 0;
        off += NG * p.pb_stride;
        off = align_up(off, 1024);
        // each group's output staging tile (128 rows x 128 bytes, 128-byte swizzle)
        p.off_stage = off;
        off += NG * kTileBytes;
        p.off_mask = off;
        off += 2 * 4096;
        p.off_lut = off;
        if (HK || BM || HQ || HV) off += p.lut_pad + align_up(p.lut_len + p.cls_len, 16) + 16;
        off = align_up(off, 1024);
        p.off_kv = off;
        const int room = static_cast<int>((cap - std::min(cap, 1024 + off)) / (2 * G::KV_BYTES));
        p.nst = std::min(room, kMaxStages);
        total = 1024 + off + p.nst * 2 * G::KV_BYTES;
        if (p.nst >= 3 || (nq == 1 && p.nst >= G::SLOTS)) break;
    }
    // an issuer waiting for tile t's K/V holds up to SLOTS - 1 earlier tiles;
    // NotSupported (nothing launched) lets the caller take another kernel
    if (p.nst < G::SLOTS || total > cap) return cudaErrorNotSupported;
    unsigned *status = device_status_word();
    if (status == nullptr) return cudaErrorMemoryAllocation;
    p.wc = WaitCtl{status, kDefaultWaitNs};
    const uint64_t dims[3] = {kD, static_cast<uint64_t>(N), static_cast<uint64_t>(p.slices)};
    const uint64_t strides[2] = {kD * 2, static_cast<uint64_t>(N) * kD * 2};
    const uint32_t box[3] = {kD, 128, 1};
    const uint32_t box_kv[3] = {kD, static_cast<uint32_t>(G::KT), 1};  // one key tile
    // tables [tab_heads][num_buckets][d]
    const uint64_t tdims[3] = {kD, static_cast<uint64_t>(a.num_buckets),
                               static_cast<uint64_t>(a.tab_heads)};
    const uint64_t tstrides[2] = {kD * 2, static_cast<uint64_t>(a.num_buckets) * kD * 2};
    const uint32_t tbox[3] = {kD, 32, 1};
    const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
    CUtensorMap tq, tk, tv, trk, to, tkc, trq, trv;
    const uint32_t box_kc[3] = {kD, 16, 1};  // the slice's first 16 keys (class token first)
    if (!encode_tensor_map(&tq, bf, 3, a.q, dims, strides, box, sw) ||
        !encode_tensor_map(&to, bf, 3, a.out, dims, strides, box, sw) ||
        !encode_tensor_map(&tk, bf, 3, a.k, dims, strides, box_kv, sw) ||
        !encode_tensor_map(&tkc, bf, 3, a.k, dims, strides, box_kc, sw) ||
        !encode_tensor_map(&tv, bf, 3, a.v, dims, strides, box_kv, sw) ||
        !encode_tensor_map(&trk, bf, 3, HK ? a.tab_k : a.q, tdims, tstrides, tbox, sw) ||
        !encode_tensor_map(&trq, bf, 3, HQ ? a.tab_q : a.q, tdims, tstrides, tbox, sw) ||
        !encode_tensor_map(&trv, bf, 3, HV ? a.tab_v : a.q, tdims, tstrides, tbox, sw))
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(rpe_pingpong_kernel<W, R, HK, NG, BM, TF>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(total));
    if (err != cudaSuccess) return err;
    const int grid = std::min(p.items, sm_count() * L::kCtasPerSm);
    // Tail split: the items of the last, partial round run as two parts each
    // (see item_at) when that round fills at most half the grid, so each CTA
    // runs one part at most. (With more, some CTAs would run two parts, and
    // at a few key tiles per item two parts cost more than a whole item: the
    // DeiT-S shape, 80 tail items on 152 SMs, measured 22.5 -> 32.3 us.)
    p.whole = p.items;
    p.tail = 0;
    p.ka = p.nkt;
    if constexpr ((TF & 4) != 0) {
        const int T = p.items % grid;
        if (T > 0 && p.nkt >= 2 && 2 * T <= grid && 2 * T <= kSplitCounters) {
            float *ws = nullptr;
            int *cnt = nullptr;
            if (stream_split_workspace(stream, 4 * 66 * 128, &ws, &cnt)) {
                p.whole = p.items - T;
                p.tail = T;
                p.ws = ws;
                p.cnt = cnt;
                p.ka = (p.nkt + 1) / 2;  // part A: the first half of the key tiles
            }
        }
    }
    return launch_pdl(rpe_pingpong_kernel<W, R, HK, NG, BM, TF>, dim3(grid), dim3(L::kThreads), total, stream,
                      tq, tk, tv, trk, tkc, trq, trv, to, p);
}

}  // namespace

}  // namespace vta
