// FP32 instantiations of the fused reduce-scatter kernels (N = 1..16).
#include "lpcoll_dda.cuh"

namespace lpc {
cudaError_t launch_scatter_f32(const DdaParams &p, int nranks, size_t n, bool lp,
                               cudaStream_t stream)
{
    return launch_scatter<LPCOLL_F32>(p, nranks, n, lp, stream);
}
}  // namespace lpc
