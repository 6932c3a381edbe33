// Instantiation unit: NVFP4 projection kernels (warp workers; single matrix and gate + up).
#include "tfq_qproj.cuh"

namespace tfq {

cudaError_t launch_qproj_nvfp4(bool dual, const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl)
{
    if (plan.mode != 1)  // the planner gives NVFP4 weights warp workers or nothing
        return cudaErrorInvalidValue;
    return dual ? launch_qproj_warp<kNvfp4, true, false>(plan, p, stream, pdl)
                : launch_qproj_warp<kNvfp4, false, false>(plan, p, stream, pdl);
}

}  // namespace tfq
