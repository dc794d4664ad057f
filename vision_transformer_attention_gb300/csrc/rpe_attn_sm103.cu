// rpe_attn_sm103.cu -- iRPE contextual attention on sm_103a tensor cores.
#include "vta_internal.h"

namespace vta {

cudaError_t launch_rpe_bf16(const RpeBf16Args &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace vta
