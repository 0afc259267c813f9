// lpcoll_gather.cu -- the collectives without a reduction: AllGather and
// AlltoAll over N emulated ranks, exact or low precision.
//
// Each warp takes an item of kItemUnits consecutive units (32 x kVec
// elements each) of one sender's data: it loads them all, and in low
// precision quantizes them on the sender's blocks (one absmax scale per 128
// elements counted from the start of what the sender sends), stores the
// codes and scales to the sender's wire payload, and dequantizes them in
// registers; then it writes the (dequantized) values to the receiving
// outputs. Warps stride over (sender, destination, item), so each sender's
// data streams through HBM in order.
//
// Offsets that are not 16-byte aligned (a contribution or chunk length that
// is not a multiple of 16 bytes) take the element-by-element path for the
// accesses that need it; the choice is made once per launch (ALIGNED).
#include "lpcoll_dda.cuh"
#include "lpcoll_device.cuh"

namespace lpc {

// Units per work item: a warp loads kItemUnits consecutive units of one
// sender before processing them, so each lane keeps kItemUnits 16-byte loads
// in flight (one sender per item would leave the loop latency-bound). With
// 4 CTAs per SM, items of 4 units measured fastest on GB300 (8 units: -13%,
// 16 units: -50%).
constexpr int kItemUnits = 4;

// Quantize-dequantize (LP) or pass through the kItemUnits vectors of one
// item, whose lane offsets are e0[k] with cnt[k] valid elements; x receives
// the values to deliver.
template <int DT, bool LP>
__device__ __forceinline__ void encode_item(const DdaParams &p, int r, size_t code_base,
                                            size_t scale_base,
                                            const size_t (&e0)[kItemUnits],
                                            const int (&cnt)[kItemUnits],
                                            const uint4 (&raw)[kItemUnits], bool aligned,
                                            int lane, float (&x)[kItemUnits][Fmt<DT>::kVec])
{
#pragma unroll
    for (int k = 0; k < kItemUnits; ++k) {
        widen<DT>(raw[k], x[k]);
        if constexpr (LP) {
            float s;
            const Codes<DT> c = quantize_lane<DT>(x[k], s);
            if (cnt[k] > 0) {
                store_codes(p.codes[r], code_base + e0[k], access_count<DT>(cnt[k], aligned),
                            c);
                if ((lane % Fmt<DT>::kGroup) == 0)
                    __stcs(p.scales[r] + scale_base + e0[k] / kBlock, s);
            }
            dequantize_lane<DT>(c, s, x[k]);
        }
    }
}

// One item of sender r's contribution (m elements) to the AllGather:
// units [g kItemUnits, (g+1) kItemUnits).
template <int DT, bool LP, bool ALIGNED>
__device__ __forceinline__ void gather_item(const DdaParams &p, int nranks, size_t m,
                                            int r, size_t g, int lane)
{
    constexpr int V = Fmt<DT>::kVec;
    size_t e0[kItemUnits];
    int cnt[kItemUnits];
    uint4 raw[kItemUnits];
#pragma unroll
    for (int k = 0; k < kItemUnits; ++k) {
        e0[k] = ((g * kItemUnits + k) * 32 + lane) * V;
        cnt[k] = lane_count<DT>(m, e0[k]);
        raw[k] = cnt[k] > 0 ? load_vec<DT>(p.in[r], e0[k], cnt[k]) : make_uint4(0u, 0u, 0u, 0u);
    }
    float x[kItemUnits][V];
    encode_item<DT, LP>(p, r, 0, 0, e0, cnt, raw, true, lane, x);
    // output by output: each receiver's slice of the item is written as one
    // contiguous run (2% faster than unit by unit across all receivers)
    const size_t at = static_cast<size_t>(r) * m;
    uint4 o[kItemUnits];
#pragma unroll
    for (int k = 0; k < kItemUnits; ++k)
        o[k] = narrow<DT>(x[k]);
    for (int d = 0; d < nranks; ++d) {
#pragma unroll
        for (int k = 0; k < kItemUnits; ++k)
            if (cnt[k] > 0)
                store_vec<DT>(p.out[d], at + e0[k], access_count<DT>(cnt[k], ALIGNED), o[k]);
    }
}

template <int DT, bool LP, bool ALIGNED>
__global__ void __launch_bounds__(kThreads)
gather_kernel(const __grid_constant__ DdaParams p, int nranks, size_t m, size_t groups)
{
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    const size_t items = static_cast<size_t>(nranks) * groups;
    for (size_t it = warp; it < items; it += nwarps) {
        const int r = static_cast<int>(it / groups);
        gather_item<DT, LP, ALIGNED>(p, nranks, m, r, it - static_cast<size_t>(r) * groups,
                                     lane);
    }
}

// One item of chunk j (c elements) of sender r in the AlltoAll.
template <int DT, bool LP, bool ALIGNED>
__device__ __forceinline__ void alltoall_item(const DdaParams &p, size_t c, size_t nbc,
                                              int r, int j, size_t g, int lane)
{
    constexpr int V = Fmt<DT>::kVec;
    const size_t src = static_cast<size_t>(j) * c;
    size_t e0[kItemUnits];
    int cnt[kItemUnits];
    uint4 raw[kItemUnits];
#pragma unroll
    for (int k = 0; k < kItemUnits; ++k) {
        e0[k] = ((g * kItemUnits + k) * 32 + lane) * V;
        cnt[k] = lane_count<DT>(c, e0[k]);
        raw[k] = cnt[k] > 0 ? load_vec<DT>(p.in[r], src + e0[k], access_count<DT>(cnt[k], ALIGNED))
                            : make_uint4(0u, 0u, 0u, 0u);
    }
    // with every load issued, each unit goes all the way to its output before
    // the next one is widened (fewer live registers than holding all units)
    const size_t at = static_cast<size_t>(r) * c;
#pragma unroll
    for (int k = 0; k < kItemUnits; ++k) {
        float x[V];
        widen<DT>(raw[k], x);
        if constexpr (LP) {
            float s;
            const Codes<DT> cd = quantize_lane<DT>(x, s);
            if (cnt[k] > 0) {
                store_codes(p.codes[r], src + e0[k], access_count<DT>(cnt[k], ALIGNED), cd);
                if ((lane % Fmt<DT>::kGroup) == 0)
                    __stcs(p.scales[r] + static_cast<size_t>(j) * nbc + e0[k] / kBlock, s);
            }
            dequantize_lane<DT>(cd, s, x);
        }
        if (cnt[k] > 0)
            store_vec<DT>(p.out[j], at + e0[k], access_count<DT>(cnt[k], ALIGNED),
                          narrow<DT>(x));
    }
}

// At most 64 registers so that 4 CTAs fit per SM (7-9% faster than the 3
// its unconstrained 74 registers allow).
template <int DT, bool LP, bool ALIGNED>
__global__ void __launch_bounds__(kThreads, kCtasPerSmBusy)
alltoall_kernel(const __grid_constant__ DdaParams p, int nranks, size_t c, size_t nbc,
                size_t groups)
{
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    const size_t per_sender = static_cast<size_t>(nranks) * groups;
    const size_t items = static_cast<size_t>(nranks) * per_sender;
    for (size_t it = warp; it < items; it += nwarps) {
        const int r = static_cast<int>(it / per_sender);
        const size_t rest = it - static_cast<size_t>(r) * per_sender;
        const int j = static_cast<int>(rest / groups);
        alltoall_item<DT, LP, ALIGNED>(p, c, nbc, r, j, rest - static_cast<size_t>(j) * groups,
                                       lane);
    }
}

// Items of kItemUnits units covering a length of `len` elements.
template <int DT>
inline size_t item_groups(size_t len)
{
    size_t full, units;
    unit_counts<DT>(len, full, units);
    return (units + kItemUnits - 1) / kItemUnits;
}

template <int DT, bool LP, bool ALIGNED>
cudaError_t launch_gather_t(const DdaParams &p, int nranks, size_t m, cudaStream_t st)
{
    const size_t groups = item_groups<DT>(m);
    const void *k = reinterpret_cast<const void *>(&gather_kernel<DT, LP, ALIGNED>);
    const int grid = wave_ctas(k, groups * static_cast<size_t>(nranks));
    gather_kernel<DT, LP, ALIGNED><<<grid, kThreads, 0, st>>>(p, nranks, m, groups);
    return cudaGetLastError();
}

template <int DT, bool LP, bool ALIGNED>
cudaError_t launch_alltoall_t(const DdaParams &p, int nranks, size_t c, cudaStream_t st)
{
    const size_t groups = item_groups<DT>(c);
    const size_t nbc = (c + kBlock - 1) / kBlock;
    const void *k = reinterpret_cast<const void *>(&alltoall_kernel<DT, LP, ALIGNED>);
    const int grid =
        wave_ctas(k, groups * static_cast<size_t>(nranks) * static_cast<size_t>(nranks));
    alltoall_kernel<DT, LP, ALIGNED><<<grid, kThreads, 0, st>>>(p, nranks, c, nbc, groups);
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
