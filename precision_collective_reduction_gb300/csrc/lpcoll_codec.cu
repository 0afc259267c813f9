// lpcoll_codec.cu -- the staged building blocks: lp_quantize (one rank's
// message -> FP8 payload), lp_dequantize (payload -> message) and lp_reduce
// (N payloads -> one FP32-summed message). Same unit decomposition and the
// same device arithmetic as the fused kernels, so a staged pipeline
// (quantize x N, reduce) gives bit-identical results to dda_flat_sim.
#include "lpcoll_dda.cuh"
#include "lpcoll_device.cuh"

namespace lpc {

// Units per loop iteration; all loads of an iteration are issued before any
// of its units is processed. Measured on GB300 (8 x 64 Mi FP32): quantize
// and dequantize gain 52% with 4 units over 1 (8 units: slower), the 8-rank
// reduce 15% with 2 (4 units: its 16+ loads per unit spill, -40%).
constexpr int kQuantizeUnits = 4;
constexpr int kDequantizeUnits = 4;
constexpr int kReduceUnits = 2;
// The quantize kernel reads much more than it writes and takes all the
// resident CTAs it can get (8 per SM: +10% over 4).
constexpr int kQuantizeCtasPerSm = 8;

// Warp-units [u0, u0 + K) of one message of n elements; e0 / cnt per lane.
template <int DT, int K>
__device__ __forceinline__ void unit_lanes(size_t n, size_t u0, int lane, size_t (&e0)[K],
                                           int (&cnt)[K])
{
#pragma unroll
    for (int k = 0; k < K; ++k) {
        e0[k] = ((u0 + k) * 32 + lane) * Fmt<DT>::kVec;
        cnt[k] = lane_count<DT>(n, e0[k]);
    }
}

template <int DT>
__global__ void __launch_bounds__(kThreads)
quantize_kernel(const void *in, uint8_t *codes, float *scales, size_t n, size_t items)
{
    constexpr int K = kQuantizeUnits;
    constexpr int V = Fmt<DT>::kVec;
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    for (size_t it = warp; it < items; it += nwarps) {
        size_t e0[K];
        int cnt[K];
        unit_lanes<DT, K>(n, it * K, lane, e0, cnt);
        uint4 raw[K];
#pragma unroll
        for (int k = 0; k < K; ++k)
            raw[k] = cnt[k] > 0 ? load_vec<DT>(in, e0[k], cnt[k]) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            float x[V];
            widen<DT>(raw[k], x);
            float s;
            const Codes<DT> c = quantize_lane<DT>(x, s);
            if (cnt[k] > 0) {
                store_codes(codes, e0[k], cnt[k], c);
                if ((lane % Fmt<DT>::kGroup) == 0)
                    __stcs(scales + e0[k] / kBlock, s);
            }
        }
    }
}

template <int DT>
__global__ void __launch_bounds__(kThreads)
dequantize_kernel(const uint8_t *codes, const float *scales, void *out, size_t n,
                  size_t items)
{
    constexpr int K = kDequantizeUnits;
    constexpr int V = Fmt<DT>::kVec;
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    for (size_t it = warp; it < items; it += nwarps) {
        size_t e0[K];
        int cnt[K];
        unit_lanes<DT, K>(n, it * K, lane, e0, cnt);
        Codes<DT> c[K];
        float s[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if (cnt[k] > 0) {
                c[k] = load_codes<DT>(codes, e0[k], cnt[k]);
                s[k] = scales[e0[k] / kBlock];
            }
        }
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if (cnt[k] > 0) {
                float v[V];
                dequantize_lane<DT>(c[k], s[k], v);
                store_vec<DT>(out, e0[k], cnt[k], narrow<DT>(v));
            }
        }
    }
}

template <int N, int DT>
__global__ void __launch_bounds__(kThreads)
reduce_kernel(const __grid_constant__ ReduceParams p, void *out, size_t n, size_t items)
{
    constexpr int K = kReduceUnits;
    constexpr int V = Fmt<DT>::kVec;
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    for (size_t it = warp; it < items; it += nwarps) {
        size_t e0[K];
        int cnt[K];
        unit_lanes<DT, K>(n, it * K, lane, e0, cnt);
        Codes<DT> c[K][N];
        float s[K][N];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if (cnt[k] > 0) {
#pragma unroll
                for (int r = 0; r < N; ++r) {
                    c[k][r] = load_codes<DT>(p.codes[r], e0[k], cnt[k]);
                    s[k][r] = p.scales[r][e0[k] / kBlock];
                }
            }
        }
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if (cnt[k] > 0) {
                float acc[V];
#pragma unroll
                for (int r = 0; r < N; ++r) {
                    float v[V];
                    dequantize_lane<DT>(c[k][r], s[k][r], v);
#pragma unroll
                    for (int j = 0; j < V; ++j)
                        acc[j] = (r == 0) ? v[j] : __fadd_rn(acc[j], v[j]);
                }
                store_vec<DT>(out, e0[k], cnt[k], narrow<DT>(acc));
            }
        }
    }
}

// Items of K warp-units covering a message of n elements.
template <int DT, int K>
inline size_t items_of(size_t n)
{
    size_t full, units;
    unit_counts<DT>(n, full, units);
    return (units + K - 1) / K;
}

template <int DT>
cudaError_t launch_quantize_t(const void *in, uint8_t *codes, float *scales,
                              size_t n, cudaStream_t stream)
{
    const size_t items = items_of<DT, kQuantizeUnits>(n);
    const int grid = wave_ctas(reinterpret_cast<const void *>(&quantize_kernel<DT>), items,
                               kQuantizeCtasPerSm);
    quantize_kernel<DT><<<grid, kThreads, 0, stream>>>(in, codes, scales, n, items);
    return cudaGetLastError();
}

template <int DT>
cudaError_t launch_dequantize_t(const uint8_t *codes, const float *scales, void *out,
                                size_t n, cudaStream_t stream)
{
    const size_t items = items_of<DT, kDequantizeUnits>(n);
    const int grid =
        wave_ctas(reinterpret_cast<const void *>(&dequantize_kernel<DT>), items);
    dequantize_kernel<DT><<<grid, kThreads, 0, stream>>>(codes, scales, out, n, items);
    return cudaGetLastError();
}

template <int N, int DT>
cudaError_t launch_reduce_n(const ReduceParams &p, void *out, size_t n,
                            cudaStream_t stream)
{
    const size_t items = items_of<DT, kReduceUnits>(n);
    const int grid =
        wave_ctas(reinterpret_cast<const void *>(&reduce_kernel<N, DT>), items);
    reduce_kernel<N, DT><<<grid, kThreads, 0, stream>>>(p, out, n, items);
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
