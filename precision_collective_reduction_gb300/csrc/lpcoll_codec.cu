// lpcoll_codec.cu -- the staged building blocks: lp_quantize (one rank's
// message -> FP8 payload), lp_dequantize (payload -> message) and lp_reduce
// (N payloads -> one FP32-summed message). They run the same device
// arithmetic as the fused kernels (block absmax, the two IEEE divisions of
// the block scale, RNE satfinite encoding, exact decoding, one rounded
// multiply, the rank-ordered FP32 sum), so a staged pipeline (quantize x N,
// reduce) gives bit-identical results to dda_flat_sim.
//
// Lane layouts. lp_dequantize uses the fused kernels' warp-unit (one 16-byte
// vector per lane, a block spread over 32 or 16 lanes). lp_quantize and
// lp_reduce use a wide layout: a lane holds 16 consecutive elements (four
// FP32 or two BF16 vectors), 8 lanes hold one 128-element block and a warp
// item covers 512 elements. A lane then moves its codes with one 16-byte
// access per rank, finds the block maximum in 3 shuffle steps and computes
// the block scale once per 16 elements instead of once per 4 or 8. Measured
// on GB300 (64 Mi FP32 elements per rank, L2 flushed): quantize 59.4 ->
// 52 us, the 8-rank reduce 147.4 -> 129.0 us; the same layout for dequantize
// was no faster.
#include "lpcoll_dda.cuh"
#include "lpcoll_device.cuh"
#include "lpcoll_wide.cuh"

namespace lpc {

// Units per warp item of the dequantize kernel; all loads of an item are
// issued before any of its units is processed. With the one-warp-per-item
// grid, 2 units measured 1-3% faster per call than 4 or 8 on GB300 (64 Mi
// FP32 49.8 against 50.2 us in a CUDA graph) and 1 unit 13-28% slower.
constexpr int kDequantizeUnits = 2;
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

// FP8 format FMT on blocks of G lanes (16 G elements): the main path is
// <DT, E4M3, 8>, the format / block-size variants the other instances.
template <int DT, int FMT, int G>
__global__ void __launch_bounds__(kThreads)
quantize_kernel(const void *in, uint8_t *codes, float *scales, size_t n, size_t items)
{
    wait_prior_grid();
    constexpr int V = Fmt<DT>::kVec;
    constexpr int S = kWideElems / V;
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    for (size_t it = warp; it < items; it += nwarps) {
        const size_t e0 = it * kWideItem + static_cast<size_t>(lane) * kWideElems;
        uint4 raw[S];
#pragma unroll
        for (int j = 0; j < S; ++j) {
            const int cnt = lane_count<DT>(n, e0 + j * V);
            raw[j] = cnt > 0 ? load_vec<DT>(in, e0 + j * V, cnt) : make_uint4(0u, 0u, 0u, 0u);
        }
        float x[kWideElems];
        wide_widen<DT>(raw, x);
        float s;
        uint32_t w[4];
        wide_quantize_fmt<FMT, G>(x, w, s);
        if (e0 < n) {
            wide_store_codes(codes, n, e0, w);
            if (lane % G == 0)
                store_scale(scales + e0 / (kWideElems * G), s);
        }
    }
}

template <int DT>
__global__ void __launch_bounds__(kThreads)
dequantize_kernel(const uint8_t *codes, const float *scales, void *out, size_t n,
                  size_t items)
{
    wait_prior_grid();
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
                s[k] = load_scale(scales + e0[k] / kBlock);
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

// Resident CTAs per SM the reduce kernel's registers are budgeted for: 4
// (64 registers) up to 9 ranks, where it needs no spill; the BF16 8-rank
// reduce then runs 6-10% faster than at the 80 registers (3 CTAs per SM)
// the compiler picks on its own (GB300, 8 x 8 Mi and 8 x 64 Mi elements).
// More ranks: 3 (10-11 ranks) or 2, the budgets of the registers they use
// unbudgeted (80, and 111-128).
template <int N>
constexpr int reduce_min_ctas()
{
    return N <= 9 ? 4 : (N <= 11 ? 3 : 2);
}

template <int N, int DT>
__global__ void __launch_bounds__(kThreads, reduce_min_ctas<N>())
reduce_kernel(const __grid_constant__ ReduceParams p, void *out, size_t n, size_t items)
{
    wait_prior_grid();
    __shared__ uint4 stage_all[kWarpsPerCta][kWideElems * 32 / 4];
    uint4 *stage = stage_all[threadIdx.x >> 5];
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    for (size_t it = warp; it < items; it += nwarps) {
        const size_t item_e0 = it * kWideItem;
        const size_t e0 = item_e0 + static_cast<size_t>(lane) * kWideElems;
        float acc[kWideElems];
        if (e0 < n) {
            uint4 c[N];
            float s[N];
#pragma unroll
            for (int r = 0; r < N; ++r) {
                c[r] = wide_load_codes(p.codes[r], n, e0);
                s[r] = load_scale(p.scales[r] + e0 / kBlock);
            }
#pragma unroll
            for (int r = 0; r < N; ++r) {
                float v[kWideElems];
                wide_dequant(c[r], s[r], v);
#pragma unroll
                for (int j = 0; j < kWideElems; ++j)
                    acc[j] = (r == 0) ? v[j] : __fadd_rn(acc[j], v[j]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < kWideElems; ++j)
                acc[j] = 0.0f;
        }
        wide_store_results<DT>(out, n, item_e0, acc, stage, lane);
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

// Warp items of the wide layout covering a message of n elements.
inline size_t wide_items(size_t n) { return (n + kWideItem - 1) / kWideItem; }

template <int DT, int FMT, int G>
cudaError_t launch_quantize_t(const void *in, uint8_t *codes, float *scales, size_t n,
                              cudaStream_t stream)
{
    const size_t items = wide_items(n);
    return launch_kernel(quantize_kernel<DT, FMT, G>, item_ctas(items), stream, in, codes,
                         scales, n, items);
}

// Block size (32, 64, 128 or 256 elements) -> lanes per block.
template <int DT, int FMT>
cudaError_t launch_quantize_blocks(const void *in, size_t n, int block, uint8_t *codes,
                                   float *scales, cudaStream_t stream)
{
    switch (block) {
    case 32: return launch_quantize_t<DT, FMT, 2>(in, codes, scales, n, stream);
    case 64: return launch_quantize_t<DT, FMT, 4>(in, codes, scales, n, stream);
    case 128: return launch_quantize_t<DT, FMT, 8>(in, codes, scales, n, stream);
    case 256: return launch_quantize_t<DT, FMT, 16>(in, codes, scales, n, stream);
    default: return cudaErrorInvalidValue;
    }
}

template <int DT>
cudaError_t launch_dequantize_t(const uint8_t *codes, const float *scales, void *out,
                                size_t n, cudaStream_t stream)
{
    const size_t items = items_of<DT, kDequantizeUnits>(n);
    return launch_kernel(dequantize_kernel<DT>, item_ctas(items), stream, codes, scales, out,
                         n, items);
}

template <int N, int DT>
cudaError_t launch_reduce_n(const ReduceParams &p, void *out, size_t n,
                            cudaStream_t stream)
{
    const size_t items = wide_items(n);
    return launch_kernel(reduce_kernel<N, DT>, item_ctas(items), stream, p, out, n, items);
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
               ? launch_quantize_t<LPCOLL_F32, LPCOLL_E4M3, kWideGroup>(in, codes, scales, n,
                                                                        stream)
               : launch_quantize_t<LPCOLL_BF16, LPCOLL_E4M3, kWideGroup>(in, codes, scales, n,
                                                                         stream);
}

cudaError_t launch_quantize_fmt(const void *in, int dtype, size_t n, int block, int fmt,
                                uint8_t *codes, float *scales, cudaStream_t stream)
{
    if (dtype == LPCOLL_F32)
        return fmt == LPCOLL_E4M3
                   ? launch_quantize_blocks<LPCOLL_F32, LPCOLL_E4M3>(in, n, block, codes,
                                                                    scales, stream)
                   : launch_quantize_blocks<LPCOLL_F32, LPCOLL_E5M2>(in, n, block, codes,
                                                                    scales, stream);
    return fmt == LPCOLL_E4M3
               ? launch_quantize_blocks<LPCOLL_BF16, LPCOLL_E4M3>(in, n, block, codes, scales,
                                                                 stream)
               : launch_quantize_blocks<LPCOLL_BF16, LPCOLL_E5M2>(in, n, block, codes, scales,
                                                                 stream);
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
