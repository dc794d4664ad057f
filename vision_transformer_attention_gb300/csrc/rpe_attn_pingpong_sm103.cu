// rpe_attn_pingpong_sm103.cu -- instantiations of the two-warpgroup kernel
// (rpe_pingpong.cuh) for the key term alone, bias mode and plain attention,
// and the dispatch of bf16 requests to it.
#include "rpe_pingpong.cuh"

namespace vta {


namespace {

template <int W, int R>
cudaError_t launch_width(const RpeBf16Args &a, cudaStream_t stream, bool hk, bool bm) {
    constexpr int NG = kGroupsPerCta;
    const int tf = (a.cross_span > 0 ? 1 : 0) | (a.tab_heads > 1 ? 2 : 0);
    // the split-tail variant (shared, non-Cross tables only) when the last round
    // of items fills at most half the grid (the rule launch_pp applies)
    bool sp = false;
    if (tf == 0) {
        const int N = a.H * a.W, qtiles = (N + 127) / 128, slices = a.B * a.heads;
        const int items = slices * (qtiles / 2) + ((qtiles & 1) ? slices : 0);
        const int grid = std::min(items, sm_count() * Layout<NG>::kCtasPerSm);
        const int T = items % grid, nkt = (a.H + R - 1) / R;
        sp = T > 0 && nkt >= 2 && 2 * T <= grid;
    }
    if (bm) return (tf & 1) ? launch_pp<W, R, false, NG, true, 1>(a, stream)
                 : sp       ? launch_pp<W, R, false, NG, true, 4>(a, stream)
                            : launch_pp<W, R, false, NG, true, 0>(a, stream);
    // a class token: never split (the class key is folded into a whole item's
    // row state in its epilogue)
    if (a.cls) return (tf & 2) ? launch_pp<W, R, true, NG, false, 10>(a, stream)
                               : launch_pp<W, R, true, NG, false, 8>(a, stream);
    if (hk && a.num_buckets > 64) return launch_pp<W, R, true, NG, false, 16>(a, stream);
    if (hk) {
        switch (tf) {
            case 0: return sp ? launch_pp<W, R, true, NG, false, 4>(a, stream)
                              : launch_pp<W, R, true, NG, false, 0>(a, stream);
            case 1: return launch_pp<W, R, true, NG, false, 1>(a, stream);
            case 2: return launch_pp<W, R, true, NG, false, 2>(a, stream);
            default: return launch_pp<W, R, true, NG, false, 3>(a, stream);
        }
    }
    return sp ? launch_pp<W, R, false, NG, false, 4>(a, stream)
              : launch_pp<W, R, false, NG, false, 0>(a, stream);
}

}  // namespace

bool launch_rpe_bf16_pingpong(const RpeBf16Args &a, cudaStream_t stream, cudaError_t *err) {
    if (a.d != kD || (a.terms & ~7u) != 0) return false;
    if ((a.terms & 6u) != 0) return launch_rpe_bf16_pingpong_qv(a, stream, err);
    const bool hk = (a.terms & 1u) != 0;
    const bool bm = a.bias != nullptr;
    if (hk && bm) return false;
    // a class token: key term, shared or per-head (not Cross) tables; the
    // score slots hold the 80 columns of the widened QR' product
    if (a.cls && (!hk || a.cross_span > 0)) return false;
    // the QR' product and copy cover 64 buckets, or 128 in two rounds with one
    // shared, non-Cross table and no class token; a bias row, one per thread, 128
    const bool hk128 = a.cross_span == 0 && a.tab_heads == 1 && !a.cls;
    if ((hk && a.num_buckets > (hk128 ? 128 : 64)) || (bm && a.num_buckets > 128)) return false;
    if (a.W == 14)
        // key tiles of 5 or 6 grid rows (70 or 84 keys in 80 or 96 score
        // columns), whichever leaves fewer score columns per query row
        *err = ((a.H + 4) / 5) * 80 < ((a.H + 5) / 6) * 96 ? launch_width<14, 5>(a, stream, hk, bm)
                                                          : launch_width<14, 6>(a, stream, hk, bm);
    else if (a.W == 56)
        *err = launch_width<56, 1>(a, stream, hk, bm);
    else
        return false;
    // shared memory too small for this request: nothing was launched
    return *err != cudaErrorNotSupported;
}

}  // namespace vta
