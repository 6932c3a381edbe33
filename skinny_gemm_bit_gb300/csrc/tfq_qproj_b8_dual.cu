// Instantiation unit: 8-bit, gate+up (SwiGLU) projection kernels.
#include "tfq_qproj.cuh"

namespace tfq {

cudaError_t launch_qproj_b8_dual(bool moe, const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl)
{
    return moe ? launch_qproj_t<8, true, true>(plan, p, stream, pdl)
               : launch_qproj_t<8, true, false>(plan, p, stream, pdl);
}

}  // namespace tfq
