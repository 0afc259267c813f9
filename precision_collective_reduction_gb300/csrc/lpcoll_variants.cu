// lpcoll_variants.cu -- format and block-size variants of the staged building
// blocks: lp_dequantize_fmt and lp_reduce_fmt (lp_quantize_fmt is the
// quantize kernel of lpcoll_codec.cu, instantiated per format and block).
//
// The pages fix neither the FP8 format nor the scaling granularity; these
// entry points make both a parameter for ablations: OCP E4M3 (largest finite
// 448) or E5M2 (largest finite 57344), one FP32 absmax scale per block of 32,
// 64, 128 or 256 elements. The arithmetic is the main path's: s = a / max,
// codes = fp8(x * (max / a)) rounded to nearest even and saturated, values
// fl(fp8 * s), FP32 sums in rank order. With E4M3 and 128-element blocks the
// results equal lp_quantize / lp_dequantize / lp_reduce.
//
// Dequantize works on warp-units (32 lanes x 16 bytes, 4 units per warp
// iteration, all loads first). The reduce works on the wide lane layout (16
// elements per lane, so no lane's elements straddle a block of 32 or more)
// and, the rank count being a run-time value, issues the loads of 4 ranks at
// a time before it adds them in rank order; results go out through the
// warp's shared-memory stage.
#include "lpcoll_dda.cuh"
#include "lpcoll_device.cuh"
#include "lpcoll_wide.cuh"

namespace lpc {

template <int FMT>
__device__ __forceinline__ float2 dec2_fmt(uint32_t c2)
{
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
        static_cast<__nv_fp8x2_storage_t>(c2 & 0xFFFFu), Fp8<FMT>::kKind);
    return __half22float2(__half2(h));
}

template <int DT, int FMT>
__device__ __forceinline__ void decode_lane(Codes<DT> c, float s,
                                            float (&v)[Fmt<DT>::kVec])
{
    constexpr int V = Fmt<DT>::kVec;
    uint32_t words[V / 4];
    if constexpr (DT == LPCOLL_F32) {
        words[0] = c.w;
    } else {
        words[0] = c.w.x;
        words[1] = c.w.y;
    }
#pragma unroll
    for (int k = 0; k < V / 4; ++k) {
        const float2 lo = dec2_fmt<FMT>(words[k]);
        const float2 hi = dec2_fmt<FMT>(words[k] >> 16);
        v[4 * k + 0] = __fmul_rn(lo.x, s);
        v[4 * k + 1] = __fmul_rn(lo.y, s);
        v[4 * k + 2] = __fmul_rn(hi.x, s);
        v[4 * k + 3] = __fmul_rn(hi.y, s);
    }
}

// Units per loop iteration of the dequantize variant; all their loads are
// issued before any unit is processed (as in lp_dequantize).
constexpr int kVariantUnits = 4;
// Ranks whose loads the reduce variant issues together.
constexpr int kRankChunk = 4;

template <int DT, int FMT>
__global__ void __launch_bounds__(kThreads)
dequantize_fmt_kernel(const uint8_t *codes, const float *scales, void *out, size_t n,
                      int block, size_t groups)
{
    wait_prior_grid();
    constexpr int V = Fmt<DT>::kVec;
    constexpr int K = kVariantUnits;
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    for (size_t g = warp; g < groups; g += nwarps) {
        size_t e0[K];
        int cnt[K];
        Codes<DT> c[K];
        float s[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            e0[k] = ((g * K + k) * 32 + lane) * V;
            cnt[k] = lane_count<DT>(n, e0[k]);
            if (cnt[k] > 0) {
                c[k] = load_codes<DT>(codes, e0[k], cnt[k]);
                s[k] = load_scale(scales + e0[k] / block);
            }
        }
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if (cnt[k] > 0) {
                float v[V];
                decode_lane<DT, FMT>(c[k], s[k], v);
                store_vec<DT>(out, e0[k], cnt[k], narrow<DT>(v));
            }
        }
    }
}

// Registers budgeted for 4 resident CTAs per SM (64, no spill), as the main
// reduce kernel up to 9 ranks; the compiler alone picks 80 (3 CTAs per SM).
template <int DT, int FMT>
__global__ void __launch_bounds__(kThreads, 4)
reduce_fmt_kernel(const __grid_constant__ ReduceParams p, int nranks, void *out, size_t n,
                  int block_shift, size_t items)
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
#pragma unroll
        for (int j = 0; j < kWideElems; ++j)
            acc[j] = 0.0f;
        if (e0 < n) {
            const size_t b = e0 >> block_shift;
            for (int r0 = 0; r0 < nranks; r0 += kRankChunk) {
                uint4 c[kRankChunk];
                float s[kRankChunk];
#pragma unroll
                for (int k = 0; k < kRankChunk; ++k) {
                    if (r0 + k < nranks) {
                        c[k] = wide_load_codes(p.codes[r0 + k], n, e0);
                        s[k] = load_scale(p.scales[r0 + k] + b);
                    }
                }
#pragma unroll
                for (int k = 0; k < kRankChunk; ++k) {
                    if (r0 + k < nranks) {
                        float v[kWideElems];
                        wide_dequant_fmt<FMT>(c[k], s[k], v);
#pragma unroll
                        for (int j = 0; j < kWideElems; ++j)
                            acc[j] = (r0 + k == 0) ? v[j] : __fadd_rn(acc[j], v[j]);
                    }
                }
            }
        }
        wide_store_results<DT>(out, n, item_e0, acc, stage, lane);
    }
}

template <int DT, int FMT>
cudaError_t dequantize_fmt_t(const uint8_t *codes, const float *scales, size_t n,
                             int block, void *out, cudaStream_t st)
{
    size_t full, units;
    unit_counts<DT>(n, full, units);
    const size_t groups = (units + kVariantUnits - 1) / kVariantUnits;
    return launch_kernel(dequantize_fmt_kernel<DT, FMT>, item_ctas(groups), st, codes, scales,
                         out, n, block, groups);
}

template <int DT, int FMT>
cudaError_t reduce_fmt_t(const ReduceParams &p, int nranks, size_t n, int block,
                         void *out, cudaStream_t st)
{
    const size_t items = (n + kWideItem - 1) / kWideItem;
    int shift = 0;
    while ((1 << shift) < block)
        ++shift;
    return launch_kernel(reduce_fmt_kernel<DT, FMT>, item_ctas(items), st, p, nranks, out, n,
                         shift, items);
}

#define LPC_BY_TYPE(FN, DTYPE, FMT, ...)                                              \
    ((DTYPE) == LPCOLL_F32                                                           \
         ? ((FMT) == LPCOLL_E4M3 ? FN<LPCOLL_F32, LPCOLL_E4M3>(__VA_ARGS__)          \
                                 : FN<LPCOLL_F32, LPCOLL_E5M2>(__VA_ARGS__))         \
         : ((FMT) == LPCOLL_E4M3 ? FN<LPCOLL_BF16, LPCOLL_E4M3>(__VA_ARGS__)         \
                                 : FN<LPCOLL_BF16, LPCOLL_E5M2>(__VA_ARGS__)))

cudaError_t launch_dequantize_fmt(const uint8_t *codes, const float *scales, size_t n,
                                  int block, int fmt, void *out, int dtype, cudaStream_t st)
{
    return LPC_BY_TYPE(dequantize_fmt_t, dtype, fmt, codes, scales, n, block, out, st);
}

cudaError_t launch_reduce_fmt(const ReduceParams &p, int nranks, size_t n, int block,
                              int fmt, void *out, int dtype, cudaStream_t st)
{
    return LPC_BY_TYPE(reduce_fmt_t, dtype, fmt, p, nranks, n, block, out, st);
}

#undef LPC_BY_TYPE

}  // namespace lpc
