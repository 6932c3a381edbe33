// Instantiation unit: NVFP4 MoE expert projection kernels (teams and warp workers; gate + up
// and down), each expert's fp32 scale read from the packed buffer's scale table.
#include "tfq_qproj.cuh"

namespace tfq {

cudaError_t launch_qproj_nvfp4_moe(bool dual, const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl)
{
    if (plan.mode != 0 && plan.mode != 1)  // no streaming schedule for NVFP4
        return cudaErrorInvalidValue;
    return dual ? launch_qproj_t<kNvfp4, true, true>(plan, p, stream, pdl)
                : launch_qproj_t<kNvfp4, false, true>(plan, p, stream, pdl);
}

}  // namespace tfq
