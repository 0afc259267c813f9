// lpcoll_dda.cuh -- the fused DDA allreduce kernels (flat, tree, exact).
//
// One launch does the whole collective for all N emulated ranks. Each warp
// takes a unit of 32 x kVec consecutive elements and, for that element range,
// plays every rank at once:
//   1. loads the N ranks' 16-byte vectors (all N loads issued back to back);
//   2. per rank: block absmax (group shuffle), scale, E4M3 codes, which are
//      stored to the rank's wire payload ("each rank publishes its data");
//   3. dequantizes in registers and sums in FP32, rank 0 first ("every rank
//      reads every rank's data and reduces locally": the N local reductions
//      are identical, so one sum serves all ranks);
//   4. tree only: requantizes the reduced block into the shard payload
//      (reduce-scatter: the block's owner is the rank whose shard holds it)
//      and replaces the sum by its dequantized value (all-gather);
//   5. writes the result to all N outputs, or, for a reduce-scatter, only to
//      the output of the rank whose shard holds the element.
// Every element is read before any output of its unit is written, so an
// output may alias its input.
//
// The warps stride over units (grid-stride loop); the grid is at most 2 CTAs
// per SM for large allreduces and 4 otherwise (kCtasPerSm / kCtasPerSmBusy),
// all resident at once, so the units of every rank stream through HBM in
// order.
#pragma once

#include "lpcoll_device.cuh"

namespace lpc {

// Reduce-scatter output: element e belongs to shard e / L and lands at
// e - owner * L in the owner's output. A lane's kVec elements go out as one
// 16-byte store when they lie in one shard at an aligned offset (always so
// when L is a whole number of 128-element blocks), else one by one.
template <int DT>
__device__ __forceinline__ void scatter_store(const DdaParams &p, size_t e0, int cnt,
                                              uint4 v)
{
    constexpr int V = Fmt<DT>::kVec;
    constexpr int ES = 16 / V;
    const size_t L = p.shard_len;
    const size_t owner = e0 / L;
    const size_t off = e0 - owner * L;
    if (off + static_cast<size_t>(cnt) <= L && ((off * ES) & 15) == 0) {
        store_vec<DT>(p.out[owner], off, cnt, v);
        return;
    }
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    for (int j = 0; j < cnt; ++j) {
        const size_t e = e0 + j;
        const size_t o = e / L;
        if (DT == LPCOLL_F32) {
            static_cast<uint32_t *>(p.out[o])[e - o * L] = w[j];
        } else {
            static_cast<uint16_t *>(p.out[o])[e - o * L] =
                static_cast<uint16_t>(w[j >> 1] >> (16 * (j & 1)));
        }
    }
}

// Units a warp takes per loop iteration: enough that each lane keeps about
// eight 16-byte loads in flight (N loads per unit) whatever the rank count.
template <int N>
__host__ __device__ constexpr int units_per_iter()
{
    return N >= 8 ? 1 : (N >= 4 ? 2 : (N >= 2 ? 4 : 8));
}

// Loads of one unit: the N ranks' 16-byte vectors of this lane.
template <int N, int DT, bool FULL>
__device__ __forceinline__ void load_unit(const DdaParams &p, size_t e0, int cnt,
                                          uint4 (&raw)[N])
{
#pragma unroll
    for (int r = 0; r < N; ++r)
        raw[r] = (FULL || cnt > 0) ? load_vec<DT>(p.in[r], e0, cnt)
                                   : make_uint4(0u, 0u, 0u, 0u);
}

// Everything after the loads: quantize / dequantize / reduce / requantize,
// then the output stores.
template <int N, int DT, int MODE, bool FULL>
__device__ __forceinline__ void process_unit(const DdaParams &p, size_t e0, int cnt,
                                             int lane, const uint4 (&raw)[N])
{
    using F = Fmt<DT>;
    constexpr int V = F::kVec;
    constexpr bool kExactSum = (MODE == kExact || MODE == kScatterExact);
    constexpr bool kScatter = (MODE == kScatterExact || MODE == kScatterLp);
    const bool leader = (lane % F::kGroup) == 0;

    float acc[V];
#pragma unroll
    for (int r = 0; r < N; ++r) {
        float x[V];
        widen<DT>(raw[r], x);
        if constexpr (kExactSum) {
#pragma unroll
            for (int j = 0; j < V; ++j)
                acc[j] = (r == 0) ? x[j] : __fadd_rn(acc[j], x[j]);
        } else {
            float s;
            Codes<DT> c = quantize_lane<DT>(x, s);
            if (FULL || cnt > 0) {
                store_codes(p.codes[r], e0, cnt, c);
                if (leader)
                    __stcs(p.scales[r] + e0 / kBlock, s);
            }
            float v[V];
            dequantize_lane<DT>(c, s, v);
#pragma unroll
            for (int j = 0; j < V; ++j)
                acc[j] = (r == 0) ? v[j] : __fadd_rn(acc[j], v[j]);
        }
    }

    if constexpr (MODE == kTree) {
        float s;
        Codes<DT> c = quantize_lane<DT>(acc, s);
        if (FULL || cnt > 0) {
            store_codes(p.shard_codes, e0, cnt, c);
            if (leader)
                __stcs(p.shard_scales + e0 / kBlock, s);
        }
        dequantize_lane<DT>(c, s, acc);
    }

    if (FULL || cnt > 0) {
        const uint4 o = narrow<DT>(acc);
        if constexpr (kScatter) {
            scatter_store<DT>(p, e0, cnt, o);
        } else {
#pragma unroll
            for (int r = 0; r < N; ++r)
                store_vec<DT>(p.out[r], e0, cnt, o);
        }
    }
}

template <int N, int DT, int MODE, bool FULL>
__device__ __forceinline__ void dda_unit(const DdaParams &p, size_t n, size_t unit,
                                         int lane)
{
    constexpr int V = Fmt<DT>::kVec;
    const size_t e0 = (unit * 32 + lane) * V;
    const int cnt = FULL ? V : lane_count<DT>(n, e0);
    uint4 raw[N];
    load_unit<N, DT, FULL>(p, e0, cnt, raw);
    process_unit<N, DT, MODE, FULL>(p, e0, cnt, lane, raw);
}

// K consecutive full units, all K x N loads issued before any processing.
template <int N, int DT, int MODE, int K>
__device__ __forceinline__ void dda_units(const DdaParams &p, size_t unit0, int lane)
{
    constexpr int V = Fmt<DT>::kVec;
    uint4 raw[K][N];
#pragma unroll
    for (int k = 0; k < K; ++k)
        load_unit<N, DT, true>(p, ((unit0 + k) * 32 + lane) * V, V, raw[k]);
#pragma unroll
    for (int k = 0; k < K; ++k)
        process_unit<N, DT, MODE, true>(p, ((unit0 + k) * 32 + lane) * V, V, lane, raw[k]);
}

template <int N, int DT, int MODE>
__global__ void __launch_bounds__(kThreads)
dda_kernel(const __grid_constant__ DdaParams p, size_t n, size_t full_units,
           size_t total_units)
{
    wait_prior_grid();
    constexpr int K = units_per_iter<N>();
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    size_t u = warp;
    if constexpr (K > 1) {
        // groups of K consecutive units, then the full units left over
        const size_t groups = full_units / K;
        for (size_t g = warp; g < groups; g += nwarps)
            dda_units<N, DT, MODE, K>(p, g * K, lane);
        u = groups * K + warp;
    }
    for (; u < full_units; u += nwarps)
        dda_unit<N, DT, MODE, true>(p, n, u, lane);
    // the ragged last unit (at most one) goes to the warp that would take it
    if (total_units > full_units && warp == full_units % nwarps)
        dda_unit<N, DT, MODE, false>(p, n, full_units, lane);
}

// Units of a message of n elements: all full units, then the ragged one.
template <int DT>
inline void unit_counts(size_t n, size_t &full, size_t &total)
{
    const size_t per = 32 * static_cast<size_t>(Fmt<DT>::kVec);
    full = n / per;
    total = (n + per - 1) / per;
}

// CTAs for a launch covering `units` warp-units: enough for every unit, at
// most min(resident CTAs per SM, cap) x SMs.
int wave_ctas(const void *kernel, size_t units, int cap = kCtasPerSmBusy);

template <int N, int DT, int MODE>
cudaError_t launch_dda_n(const DdaParams &p, size_t n, cudaStream_t stream)
{
    size_t full, total;
    unit_counts<DT>(n, full, total);
    const void *k = reinterpret_cast<const void *>(&dda_kernel<N, DT, MODE>);
    const size_t K = units_per_iter<N>();
    const bool scatter = (MODE == kScatterExact || MODE == kScatterLp);
    const size_t in_bytes = n * static_cast<size_t>(N) * (16 / Fmt<DT>::kVec);
    const int cap = (scatter || in_bytes < kSmallLaunchBytes) ? kCtasPerSmBusy : kCtasPerSm;
    const int grid = wave_ctas(k, (total + K - 1) / K, cap);
    return launch_kernel(dda_kernel<N, DT, MODE>, grid, stream, p, n, full, total);
}

template <int DT, int MODE>
cudaError_t launch_dda_mode(const DdaParams &p, int nranks, size_t n,
                            cudaStream_t stream)
{
    switch (nranks) {
#define LPC_CASE(K) \
    case K: return launch_dda_n<K, DT, MODE>(p, n, stream);
        LPC_CASE(1) LPC_CASE(2) LPC_CASE(3) LPC_CASE(4) LPC_CASE(5) LPC_CASE(6)
        LPC_CASE(7) LPC_CASE(8) LPC_CASE(9) LPC_CASE(10) LPC_CASE(11) LPC_CASE(12)
        LPC_CASE(13) LPC_CASE(14) LPC_CASE(15) LPC_CASE(16)
#undef LPC_CASE
    default: return cudaErrorInvalidValue;
    }
}

template <int DT>
cudaError_t launch_dda(const DdaParams &p, int nranks, size_t n, int mode,
                       cudaStream_t stream)
{
    switch (mode) {
    case kExact: return launch_dda_mode<DT, kExact>(p, nranks, n, stream);
    case kFlat: return launch_dda_mode<DT, kFlat>(p, nranks, n, stream);
    case kTree: return launch_dda_mode<DT, kTree>(p, nranks, n, stream);
    default: return cudaErrorInvalidValue;
    }
}

template <int DT>
cudaError_t launch_scatter(const DdaParams &p, int nranks, size_t n, bool lp,
                           cudaStream_t stream)
{
    return lp ? launch_dda_mode<DT, kScatterLp>(p, nranks, n, stream)
              : launch_dda_mode<DT, kScatterExact>(p, nranks, n, stream);
}

// Remember e as this thread's lpcoll_last_cuda_error() (lpcoll_api.cu).
void record_cuda_error(cudaError_t e);

// Defined in lpcoll_dda_f32.cu / lpcoll_dda_bf16.cu (allreduce) and
// lpcoll_scatter_f32.cu / lpcoll_scatter_bf16.cu (reduce-scatter).
cudaError_t launch_dda_f32(const DdaParams &p, int nranks, size_t n, int mode,
                           cudaStream_t stream);
cudaError_t launch_dda_bf16(const DdaParams &p, int nranks, size_t n, int mode,
                            cudaStream_t stream);
cudaError_t launch_scatter_f32(const DdaParams &p, int nranks, size_t n, bool lp,
                               cudaStream_t stream);
cudaError_t launch_scatter_bf16(const DdaParams &p, int nranks, size_t n, bool lp,
                                cudaStream_t stream);

}  // namespace lpc
