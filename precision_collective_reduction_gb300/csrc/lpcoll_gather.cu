// lpcoll_gather.cu -- the collectives without a reduction: AllGather and
// AlltoAll over N emulated ranks, exact or low precision.
//
// Each warp takes one unit (32 x kVec elements) of one sender's data: it
// loads it, and in low precision quantizes it on the sender's blocks (one
// absmax scale per 128 elements counted from the start of what the sender
// sends), stores the codes and scales to the sender's wire payload, and
// dequantizes them in registers; then it writes the (dequantized) values to
// the receiving outputs. Warps stride over (sender, destination, unit)
// items, so each sender's data streams through HBM in order.
//
// Offsets that are not 16-byte aligned (a contribution or chunk length that
// is not a multiple of 16 bytes) take the element-by-element path for the
// accesses that need it; the choice is made once per launch (ALIGNED).
#include "lpcoll_dda.cuh"
#include "lpcoll_device.cuh"

namespace lpc {

// lane count argument for load_vec / store_vec / store_codes: a negative
// count asks for element-wise access of a full lane at an unaligned offset
template <int DT>
__device__ __forceinline__ int access_count(int cnt, bool aligned)
{
    return (aligned || cnt != Fmt<DT>::kVec) ? cnt : -cnt;
}

// One unit of sender r's contribution (m elements) to the AllGather.
template <int DT, bool LP, bool ALIGNED, bool FULL>
__device__ __forceinline__ void gather_unit(const DdaParams &p, int nranks, size_t m,
                                            int r, size_t u, int lane)
{
    constexpr int V = Fmt<DT>::kVec;
    const size_t e0 = (u * 32 + lane) * V;
    const int cnt = FULL ? V : lane_count<DT>(m, e0);
    const uint4 raw = (FULL || cnt > 0) ? load_vec<DT>(p.in[r], e0, cnt)
                                        : make_uint4(0u, 0u, 0u, 0u);
    float x[V];
    widen<DT>(raw, x);
    if constexpr (LP) {
        float s;
        const Codes<DT> c = quantize_lane<DT>(x, s);
        if (FULL || cnt > 0) {
            store_codes(p.codes[r], e0, cnt, c);
            if ((lane % Fmt<DT>::kGroup) == 0)
                __stcs(p.scales[r] + e0 / kBlock, s);
        }
        dequantize_lane<DT>(c, s, x);
    }
    if (FULL || cnt > 0) {
        const uint4 o = narrow<DT>(x);
        const size_t at = static_cast<size_t>(r) * m + e0;
        const int k = access_count<DT>(cnt, ALIGNED);
        for (int d = 0; d < nranks; ++d)
            store_vec<DT>(p.out[d], at, k, o);
    }
}

template <int DT, bool LP, bool ALIGNED>
__global__ void __launch_bounds__(kThreads)
gather_kernel(const __grid_constant__ DdaParams p, int nranks, size_t m,
              size_t units, size_t full_units)
{
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    const size_t items = static_cast<size_t>(nranks) * units;
    for (size_t it = warp; it < items; it += nwarps) {
        const int r = static_cast<int>(it / units);
        const size_t u = it - static_cast<size_t>(r) * units;
        if (u < full_units)
            gather_unit<DT, LP, ALIGNED, true>(p, nranks, m, r, u, lane);
        else
            gather_unit<DT, LP, ALIGNED, false>(p, nranks, m, r, u, lane);
    }
}

// One unit of chunk j (c elements) of sender r in the AlltoAll.
template <int DT, bool LP, bool ALIGNED, bool FULL>
__device__ __forceinline__ void alltoall_unit(const DdaParams &p, size_t c, size_t nbc,
                                              int r, int j, size_t u, int lane)
{
    constexpr int V = Fmt<DT>::kVec;
    const size_t e0 = (u * 32 + lane) * V;
    const int cnt = FULL ? V : lane_count<DT>(c, e0);
    const int k = access_count<DT>(cnt, ALIGNED);
    const size_t src = static_cast<size_t>(j) * c + e0;
    const uint4 raw = (FULL || cnt > 0) ? load_vec<DT>(p.in[r], src, k)
                                        : make_uint4(0u, 0u, 0u, 0u);
    float x[V];
    widen<DT>(raw, x);
    if constexpr (LP) {
        float s;
        const Codes<DT> cd = quantize_lane<DT>(x, s);
        if (FULL || cnt > 0) {
            store_codes(p.codes[r], src, k, cd);
            if ((lane % Fmt<DT>::kGroup) == 0)
                __stcs(p.scales[r] + static_cast<size_t>(j) * nbc + e0 / kBlock, s);
        }
        dequantize_lane<DT>(cd, s, x);
    }
    if (FULL || cnt > 0)
        store_vec<DT>(p.out[j], static_cast<size_t>(r) * c + e0, k, narrow<DT>(x));
}

template <int DT, bool LP, bool ALIGNED>
__global__ void __launch_bounds__(kThreads)
alltoall_kernel(const __grid_constant__ DdaParams p, int nranks, size_t c, size_t nbc,
                size_t units, size_t full_units)
{
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    const size_t per_sender = static_cast<size_t>(nranks) * units;
    const size_t items = static_cast<size_t>(nranks) * per_sender;
    for (size_t it = warp; it < items; it += nwarps) {
        const int r = static_cast<int>(it / per_sender);
        const size_t rest = it - static_cast<size_t>(r) * per_sender;
        const int j = static_cast<int>(rest / units);
        const size_t u = rest - static_cast<size_t>(j) * units;
        if (u < full_units)
            alltoall_unit<DT, LP, ALIGNED, true>(p, c, nbc, r, j, u, lane);
        else
            alltoall_unit<DT, LP, ALIGNED, false>(p, c, nbc, r, j, u, lane);
    }
}

template <int DT, bool LP, bool ALIGNED>
cudaError_t launch_gather_t(const DdaParams &p, int nranks, size_t m, cudaStream_t st)
{
    size_t full, units;
    unit_counts<DT>(m, full, units);
    const void *k = reinterpret_cast<const void *>(&gather_kernel<DT, LP, ALIGNED>);
    const int grid = wave_ctas(k, units * static_cast<size_t>(nranks));
    gather_kernel<DT, LP, ALIGNED><<<grid, kThreads, 0, st>>>(p, nranks, m, units, full);
    return cudaGetLastError();
}

template <int DT, bool LP, bool ALIGNED>
cudaError_t launch_alltoall_t(const DdaParams &p, int nranks, size_t c, cudaStream_t st)
{
    size_t full, units;
    unit_counts<DT>(c, full, units);
    const size_t nbc = (c + kBlock - 1) / kBlock;
    const void *k = reinterpret_cast<const void *>(&alltoall_kernel<DT, LP, ALIGNED>);
    const int grid =
        wave_ctas(k, units * static_cast<size_t>(nranks) * static_cast<size_t>(nranks));
    alltoall_kernel<DT, LP, ALIGNED><<<grid, kThreads, 0, st>>>(p, nranks, c, nbc, units,
                                                                 full);
    return cudaGetLastError();
}

template <int DT>
cudaError_t dispatch_gather(const DdaParams &p, int nranks, size_t m, bool lp,
                            cudaStream_t st)
{
    const bool aligned = (m * (16 / Fmt<DT>::kVec)) % 16 == 0;
    if (lp)
        return aligned ? launch_gather_t<DT, true, true>(p, nranks, m, st)
                       : launch_gather_t<DT, true, false>(p, nranks, m, st);
    return aligned ? launch_gather_t<DT, false, true>(p, nranks, m, st)
                   : launch_gather_t<DT, false, false>(p, nranks, m, st);
}

template <int DT>
cudaError_t dispatch_alltoall(const DdaParams &p, int nranks, size_t c, bool lp,
                              cudaStream_t st)
{
    const bool aligned = (c * (16 / Fmt<DT>::kVec)) % 16 == 0;
    if (lp)
        return aligned ? launch_alltoall_t<DT, true, true>(p, nranks, c, st)
                       : launch_alltoall_t<DT, true, false>(p, nranks, c, st);
    return aligned ? launch_alltoall_t<DT, false, true>(p, nranks, c, st)
                   : launch_alltoall_t<DT, false, false>(p, nranks, c, st);
}

cudaError_t launch_all_gather(const DdaParams &p, int nranks, size_t m, int dtype,
                              bool lp, cudaStream_t st)
{
    return dtype == LPCOLL_F32 ? dispatch_gather<LPCOLL_F32>(p, nranks, m, lp, st)
                               : dispatch_gather<LPCOLL_BF16>(p, nranks, m, lp, st);
}

cudaError_t launch_all_to_all(const DdaParams &p, int nranks, size_t c, int dtype,
                              bool lp, cudaStream_t st)
{
    return dtype == LPCOLL_F32 ? dispatch_alltoall<LPCOLL_F32>(p, nranks, c, lp, st)
                               : dispatch_alltoall<LPCOLL_BF16>(p, nranks, c, lp, st);
}

}  // namespace lpc
