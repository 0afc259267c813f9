// lpcoll_codec.cu -- the staged building blocks: lp_quantize (one rank's
// message -> FP8 payload), lp_dequantize (payload -> message) and lp_reduce
// (N payloads -> one FP32-summed message). Same unit decomposition and the
// same device arithmetic as the fused kernels, so a staged pipeline
// (quantize x N, reduce) gives bit-identical results to dda_flat_sim.
#include "lpcoll_dda.cuh"
#include "lpcoll_device.cuh"

namespace lpc {

template <int DT, bool FULL>
__device__ __forceinline__ void quantize_unit(const void *in, uint8_t *codes,
                                              float *scales, size_t n, size_t unit,
                                              int lane)
{
    constexpr int V = Fmt<DT>::kVec;
    const size_t e0 = (unit * 32 + lane) * V;
    const int cnt = FULL ? V : lane_count<DT>(n, e0);
    const uint4 raw = (FULL || cnt > 0) ? load_vec<DT>(in, e0, cnt)
                                        : make_uint4(0u, 0u, 0u, 0u);
    float x[V];
    widen<DT>(raw, x);
    float s;
    Codes<DT> c = quantize_lane<DT>(x, s);
    if (FULL || cnt > 0) {
        store_codes(codes, e0, cnt, c);
        if ((lane % Fmt<DT>::kGroup) == 0)
            __stcs(scales + e0 / kBlock, s);
    }
}

template <int DT>
__global__ void __launch_bounds__(kThreads)
quantize_kernel(const void *in, uint8_t *codes, float *scales, size_t n,
                size_t full_units, size_t total_units)
{
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    for (size_t u = warp; u < full_units; u += nwarps)
        quantize_unit<DT, true>(in, codes, scales, n, u, lane);
    if (total_units > full_units && warp == full_units % nwarps)
        quantize_unit<DT, false>(in, codes, scales, n, full_units, lane);
}

template <int DT, bool FULL>
__device__ __forceinline__ void dequantize_unit(const uint8_t *codes,
                                                const float *scales, void *out,
                                                size_t n, size_t unit, int lane)
{
    constexpr int V = Fmt<DT>::kVec;
    const size_t e0 = (unit * 32 + lane) * V;
    const int cnt = FULL ? V : lane_count<DT>(n, e0);
    if (!FULL && cnt == 0)
        return;
    const Codes<DT> c = load_codes<DT>(codes, e0, cnt);
    const float s = scales[e0 / kBlock];
    float v[V];
    dequantize_lane<DT>(c, s, v);
    store_vec<DT>(out, e0, cnt, narrow<DT>(v));
}

template <int DT>
__global__ void __launch_bounds__(kThreads)
dequantize_kernel(const uint8_t *codes, const float *scales, void *out, size_t n,
                  size_t full_units, size_t total_units)
{
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    for (size_t u = warp; u < full_units; u += nwarps)
        dequantize_unit<DT, true>(codes, scales, out, n, u, lane);
    if (total_units > full_units && warp == full_units % nwarps)
        dequantize_unit<DT, false>(codes, scales, out, n, full_units, lane);
}

template <int N, int DT, bool FULL>
__device__ __forceinline__ void reduce_unit(const ReduceParams &p, void *out,
                                            size_t n, size_t unit, int lane)
{
    constexpr int V = Fmt<DT>::kVec;
    const size_t e0 = (unit * 32 + lane) * V;
    const int cnt = FULL ? V : lane_count<DT>(n, e0);
    if (!FULL && cnt == 0)
        return;
    Codes<DT> c[N];
    float s[N];
#pragma unroll
    for (int r = 0; r < N; ++r) {
        c[r] = load_codes<DT>(p.codes[r], e0, cnt);
        s[r] = p.scales[r][e0 / kBlock];
    }
    float acc[V];
#pragma unroll
    for (int r = 0; r < N; ++r) {
        float v[V];
        dequantize_lane<DT>(c[r], s[r], v);
#pragma unroll
        for (int j = 0; j < V; ++j)
            acc[j] = (r == 0) ? v[j] : __fadd_rn(acc[j], v[j]);
    }
    store_vec<DT>(out, e0, cnt, narrow<DT>(acc));
}

template <int N, int DT>
__global__ void __launch_bounds__(kThreads)
reduce_kernel(const __grid_constant__ ReduceParams p, void *out, size_t n,
              size_t full_units, size_t total_units)
{
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    for (size_t u = warp; u < full_units; u += nwarps)
        reduce_unit<N, DT, true>(p, out, n, u, lane);
    if (total_units > full_units && warp == full_units % nwarps)
        reduce_unit<N, DT, false>(p, out, n, full_units, lane);
}

template <int DT>
cudaError_t launch_quantize_t(const void *in, uint8_t *codes, float *scales,
                              size_t n, cudaStream_t stream)
{
    size_t full, total;
    unit_counts<DT>(n, full, total);
    const int grid = wave_ctas(reinterpret_cast<const void *>(&quantize_kernel<DT>), total);
    quantize_kernel<DT><<<grid, kThreads, 0, stream>>>(in, codes, scales, n, full, total);
    return cudaGetLastError();
}

template <int DT>
cudaError_t launch_dequantize_t(const uint8_t *codes, const float *scales, void *out,
                                size_t n, cudaStream_t stream)
{
    size_t full, total;
    unit_counts<DT>(n, full, total);
    const int grid =
        wave_ctas(reinterpret_cast<const void *>(&dequantize_kernel<DT>), total);
    dequantize_kernel<DT><<<grid, kThreads, 0, stream>>>(codes, scales, out, n, full,
                                                         total);
    return cudaGetLastError();
}

template <int N, int DT>
cudaError_t launch_reduce_n(const ReduceParams &p, void *out, size_t n,
                            cudaStream_t stream)
{
    size_t full, total;
    unit_counts<DT>(n, full, total);
    const int grid =
        wave_ctas(reinterpret_cast<const void *>(&reduce_kernel<N, DT>), total);
    reduce_kernel<N, DT><<<grid, kThreads, 0, stream>>>(p, out, n, full, total);
    return cudaGetLastError();
}

template <int DT>
cudaError_t launch_reduce_t(const ReduceParams &p, int nranks, void *out, size_t n,
                            cudaStream_t stream)
{
    switch (nranks) {
#define LPC_CASE(K) \
    case K: return launch_reduce_n<K, DT>(p, out, n, stream);
        LPC_CASE(1) LPC_CASE(2) LPC_CASE(3) LPC_CASE(4) LPC_CASE(5) LPC_CASE(6)
        LPC_CASE(7) LPC_CASE(8) LPC_CASE(9) LPC_CASE(10) LPC_CASE(11) LPC_CASE(12)
        LPC_CASE(13) LPC_CASE(14) LPC_CASE(15) LPC_CASE(16)
#undef LPC_CASE
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_quantize(const void *in, int dtype, size_t n, uint8_t *codes,
                            float *scales, cudaStream_t stream)
{
    return dtype == LPCOLL_F32
               ? launch_quantize_t<LPCOLL_F32>(in, codes, scales, n, stream)
               : launch_quantize_t<LPCOLL_BF16>(in, codes, scales, n, stream);
}

cudaError_t launch_dequantize(const uint8_t *codes, const float *scales, size_t n,
                              void *out, int dtype, cudaStream_t stream)
{
    return dtype == LPCOLL_F32
               ? launch_dequantize_t<LPCOLL_F32>(codes, scales, out, n, stream)
               : launch_dequantize_t<LPCOLL_BF16>(codes, scales, out, n, stream);
}

cudaError_t launch_reduce(const ReduceParams &p, int nranks, size_t n, void *out,
                          int dtype, cudaStream_t stream)
{
    return dtype == LPCOLL_F32
               ? launch_reduce_t<LPCOLL_F32>(p, nranks, out, n, stream)
               : launch_reduce_t<LPCOLL_BF16>(p, nranks, out, n, stream);
}

}  // namespace lpc
