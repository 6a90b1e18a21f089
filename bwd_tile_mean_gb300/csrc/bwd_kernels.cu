// bwd_kernels.cu -- placeholder launchers (backward kernels pending).
#include "vsa_internal.h"

namespace vsa {
cudaError_t launch_dvec(const Prob &, const void *, const void *, float *, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_bwd_dkdv(const Prob &, const BwdArgs &, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_bwd_dq(const Prob &, const BwdArgs &, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_compress_bwd(const Prob &, const void *, const void *, const float *, const float *,
                                const float *, float *, float *, float *, float *, float *, float *,
                                cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace vsa
