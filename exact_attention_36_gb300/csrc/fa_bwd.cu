// fa_bwd.cu -- fused attention backward for sm_103a (placeholder launcher
// until the backward kernels land).
#include "fa_common.cuh"

namespace fa {
cudaError_t launch_bwd(const BwdArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace fa
