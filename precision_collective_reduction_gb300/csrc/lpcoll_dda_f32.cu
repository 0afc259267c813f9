// FP32 instantiations of the fused DDA allreduce kernels (N = 1..16).
#include "lpcoll_dda.cuh"

namespace lpc {
cudaError_t launch_dda_f32(const DdaParams &p, int nranks, size_t n, int mode,
                           cudaStream_t stream)
{
    return launch_dda<LPCOLL_F32>(p, nranks, n, mode, stream);
}
}  // namespace lpc
