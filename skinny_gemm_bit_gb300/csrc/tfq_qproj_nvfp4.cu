// Instantiation unit: NVFP4 projection kernels (teams and warp workers; single matrix and
// gate + up).
#include "tfq_qproj.cuh"

namespace tfq {

cudaError_t launch_qproj_nvfp4(bool dual, const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl)
{
    if (plan.mode == 2)  // no streaming schedule for NVFP4
        return cudaErrorInvalidValue;
    return dual ? launch_qproj_t<kNvfp4, true, false>(plan, p, stream, pdl)
                : launch_qproj_t<kNvfp4, false, false>(plan, p, stream, pdl);
}

}  // namespace tfq
