// rpe_attn_pingpong_qv_sm103.cu -- instantiations of the two-warpgroup kernel
// (rpe_pingpong.cuh) with the contextual query and / or value terms, in their
// own translation unit so that they compile beside the key-term variants.
#include "rpe_pingpong.cuh"

namespace vta {

namespace {

template <bool HK, int QV>
cudaError_t launch_qv(const RpeBf16Args &a, cudaStream_t stream) {
    return launch_pp<14, 5, HK, kGroupsPerCta, false, QV>(a, stream);
}

}  // namespace

bool launch_rpe_bf16_pingpong_qv(const RpeBf16Args &a, cudaStream_t stream, cudaError_t *err) {
    const bool hk = (a.terms & 1u) != 0, hq = (a.terms & 2u) != 0, hv = (a.terms & 4u) != 0;
    if (a.d != kD || (!hq && !hv) || a.bias != nullptr || a.W != 14 || a.cross_span > 0 ||
        a.tab_heads > 1 || a.cls || a.num_buckets > 64)
        return false;
    // the value term's bucket sums take each grid row of keys in one batch
    if (hv && !a.lut_row_runs) return false;
    // every item is a pair of query tiles (both groups copy K R^Q^T)
    const int qtiles = (a.H * a.W + 127) / 128;
    if (qtiles % 2 != 0) return false;
    const int qv = (hq ? 32 : 0) | (hv ? 64 : 0);
    cudaError_t e;
    if (hk)
        e = qv == 32 ? launch_qv<true, 32>(a, stream)
          : qv == 64 ? launch_qv<true, 64>(a, stream)
                     : launch_qv<true, 96>(a, stream);
    else
        e = qv == 32 ? launch_qv<false, 32>(a, stream)
          : qv == 64 ? launch_qv<false, 64>(a, stream)
                     : launch_qv<false, 96>(a, stream);
    // shared memory too small for this bucket count: nothing was launched
    if (e == cudaErrorNotSupported) return false;
    *err = e;
    return true;
}

}  // namespace vta
