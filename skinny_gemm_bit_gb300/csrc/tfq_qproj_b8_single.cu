// Instantiation unit: 8-bit, single matrix projection kernels (teams, warp workers, streaming).
#include "tfq_stream.cuh"

namespace tfq {

cudaError_t launch_qproj_b8_single(bool moe, const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl)
{
    if (!moe && plan.mode == 2)
        return launch_qstream<8>(plan, p, stream, pdl);
    return moe ? launch_qproj_t<8, false, true>(plan, p, stream, pdl)
               : launch_qproj_t<8, false, false>(plan, p, stream, pdl);
}

}  // namespace tfq
