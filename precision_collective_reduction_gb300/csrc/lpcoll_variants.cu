// lpcoll_variants.cu -- format and block-size variants of the staged building
// blocks: lp_quantize_fmt, lp_dequantize_fmt, lp_reduce_fmt.
//
// The pages fix neither the FP8 format nor the scaling granularity; these
// entry points make both a parameter for ablations: OCP E4M3 (largest finite
// 448) or E5M2 (largest finite 57344), one FP32 absmax scale per block of 32,
// 64, 128 or 256 elements. The arithmetic is the main path's: s = a / max,
// codes = fp8(x * (max / a)) rounded to nearest even and saturated, values
// fl(fp8 * s), FP32 sums in rank order. With E4M3 and 128-element blocks the
// results equal lp_quantize / lp_dequantize / lp_reduce.
//
// Work decomposition: a warp-unit is 32 lanes x 16 bytes (kVec elements per
// lane), so a block spans block / kVec lanes; FP32 blocks of 256 span two
// units, which one warp then processes together (U = 2). A warp takes 4
// consecutive units per iteration, all loads first.
#include "lpcoll_dda.cuh"
#include "lpcoll_device.cuh"

namespace lpc {

template <int FMT> struct Fp8;
template <> struct Fp8<LPCOLL_E4M3> {
    static constexpr float kMax = 448.0f;
    static constexpr __nv_fp8_interpretation_t kKind = __NV_E4M3;
};
template <> struct Fp8<LPCOLL_E5M2> {
    static constexpr float kMax = 57344.0f;
    static constexpr __nv_fp8_interpretation_t kKind = __NV_E5M2;
};

// Largest |x| over groups of G lanes (G a power of two <= 32, uniform).
__device__ __forceinline__ float group_max_rt(float v, int G)
{
    for (int m = G >> 1; m >= 1; m >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
    return v;
}

template <int FMT>
__device__ __forceinline__ void block_scale_fmt(float amax, float &s, float &inv)
{
    inv = __fdiv_rn(Fp8<FMT>::kMax, amax);
    if (isinf(inv)) {
        inv = 0.0f;
        s = 0.0f;
    } else {
        s = __fdiv_rn(amax, Fp8<FMT>::kMax);
    }
}

// kVec values -> packed codes (element 0 in the low byte).
template <int DT, int FMT>
__device__ __forceinline__ Codes<DT> encode_lane(const float (&x)[Fmt<DT>::kVec],
                                                 float inv)
{
    constexpr int V = Fmt<DT>::kVec;
    uint32_t c2[V / 2];
#pragma unroll
    for (int j = 0; j < V / 2; ++j)
        c2[j] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(
            make_float2(__fmul_rn(x[2 * j], inv), __fmul_rn(x[2 * j + 1], inv)),
            __NV_SATFINITE, Fp8<FMT>::kKind));
    Codes<DT> c;
    if constexpr (DT == LPCOLL_F32)
        c.w = c2[0] | (c2[1] << 16);
    else
        c.w = make_uint2(c2[0] | (c2[1] << 16), c2[2] | (c2[3] << 16));
    return c;
}

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

// Units per loop iteration of the quantize / dequantize variants; all their
// loads are issued before any unit is processed (as in lp_quantize).
constexpr int kVariantUnits = 4;

// Quantize kVariantUnits consecutive units per iteration. A block covers G
// lanes of one unit (U = 1) or the whole of two units (U = 2: FP32 blocks of
// 256 elements); U divides kVariantUnits, so no block straddles iterations.
template <int DT, int FMT, int U>
__global__ void __launch_bounds__(kThreads)
quantize_fmt_kernel(const void *in, uint8_t *codes, float *scales, size_t n, int block,
                    size_t groups)
{
    wait_prior_grid();
    constexpr int V = Fmt<DT>::kVec;
    constexpr int K = kVariantUnits;
    const int lane = threadIdx.x & 31;
    const int G = (U == 2) ? 32 : block / V;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    for (size_t g = warp; g < groups; g += nwarps) {
        size_t e0[K];
        int cnt[K];
        uint4 raw[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            e0[k] = ((g * K + k) * 32 + lane) * V;
            cnt[k] = lane_count<DT>(n, e0[k]);
            raw[k] = cnt[k] > 0 ? load_vec<DT>(in, e0[k], cnt[k]) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < K; i += U) {
            float x[U][V];
            float amax = 0.0f;
#pragma unroll
            for (int k = 0; k < U; ++k) {
                widen<DT>(raw[i + k], x[k]);
                float a = 0.0f;
#pragma unroll
                for (int j = 0; j < V; ++j)
                    a = fmaxf(a, fabsf(x[k][j]));
                amax = fmaxf(amax, group_max_rt(a, G));
            }
            float s, inv;
            block_scale_fmt<FMT>(amax, s, inv);
#pragma unroll
            for (int k = 0; k < U; ++k) {
                if (cnt[i + k] > 0) {
                    store_codes(codes, e0[i + k], cnt[i + k], encode_lane<DT, FMT>(x[k], inv));
                    if (k == 0 && (lane % G) == 0)
                        scales[e0[i] / block] = s;
                }
            }
        }
    }
}

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
                s[k] = scales[e0[k] / block];
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

template <int DT, int FMT>
__global__ void __launch_bounds__(kThreads)
reduce_fmt_kernel(const __grid_constant__ ReduceParams p, int nranks, void *out, size_t n,
                  int block, size_t units)
{
    wait_prior_grid();
    constexpr int V = Fmt<DT>::kVec;
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    for (size_t u = warp; u < units; u += nwarps) {
        const size_t e0 = (u * 32 + lane) * V;
        const int cnt = lane_count<DT>(n, e0);
        if (cnt <= 0)
            continue;
        float acc[V];
        for (int r = 0; r < nranks; ++r) {
            float v[V];
            decode_lane<DT, FMT>(load_codes<DT>(p.codes[r], e0, cnt),
                                 p.scales[r][e0 / block], v);
#pragma unroll
            for (int j = 0; j < V; ++j)
                acc[j] = (r == 0) ? v[j] : __fadd_rn(acc[j], v[j]);
        }
        store_vec<DT>(out, e0, cnt, narrow<DT>(acc));
    }
}

template <int DT, int FMT>
cudaError_t quantize_fmt_t(const void *in, size_t n, int block, uint8_t *codes,
                           float *scales, cudaStream_t st)
{
    size_t full, units;
    unit_counts<DT>(n, full, units);
    const size_t groups = (units + kVariantUnits - 1) / kVariantUnits;
    if (block > 32 * Fmt<DT>::kVec) {  // FP32, block 256: two units per block
        const void *k = reinterpret_cast<const void *>(&quantize_fmt_kernel<DT, FMT, 2>);
        return launch_kernel(quantize_fmt_kernel<DT, FMT, 2>, wave_ctas(k, groups), st, in,
                             codes, scales, n, block, groups);
    }
    const void *k = reinterpret_cast<const void *>(&quantize_fmt_kernel<DT, FMT, 1>);
    return launch_kernel(quantize_fmt_kernel<DT, FMT, 1>, wave_ctas(k, groups), st, in, codes,
                         scales, n, block, groups);
}

template <int DT, int FMT>
cudaError_t dequantize_fmt_t(const uint8_t *codes, const float *scales, size_t n,
                             int block, void *out, cudaStream_t st)
{
    size_t full, units;
    unit_counts<DT>(n, full, units);
    const size_t groups = (units + kVariantUnits - 1) / kVariantUnits;
    const void *k = reinterpret_cast<const void *>(&dequantize_fmt_kernel<DT, FMT>);
    return launch_kernel(dequantize_fmt_kernel<DT, FMT>, wave_ctas(k, groups), st, codes,
                         scales, out, n, block, groups);
}

template <int DT, int FMT>
cudaError_t reduce_fmt_t(const ReduceParams &p, int nranks, size_t n, int block,
                         void *out, cudaStream_t st)
{
    size_t full, units;
    unit_counts<DT>(n, full, units);
    const void *k = reinterpret_cast<const void *>(&reduce_fmt_kernel<DT, FMT>);
    return launch_kernel(reduce_fmt_kernel<DT, FMT>, wave_ctas(k, units), st, p, nranks, out, n,
                         block, units);
}

#define LPC_BY_TYPE(FN, DTYPE, FMT, ...)                                              \
    ((DTYPE) == LPCOLL_F32                                                           \
         ? ((FMT) == LPCOLL_E4M3 ? FN<LPCOLL_F32, LPCOLL_E4M3>(__VA_ARGS__)          \
                                 : FN<LPCOLL_F32, LPCOLL_E5M2>(__VA_ARGS__))         \
         : ((FMT) == LPCOLL_E4M3 ? FN<LPCOLL_BF16, LPCOLL_E4M3>(__VA_ARGS__)         \
                                 : FN<LPCOLL_BF16, LPCOLL_E5M2>(__VA_ARGS__)))

cudaError_t launch_quantize_fmt(const void *in, int dtype, size_t n, int block, int fmt,
                                uint8_t *codes, float *scales, cudaStream_t st)
{
    return LPC_BY_TYPE(quantize_fmt_t, dtype, fmt, in, n, block, codes, scales, st);
}

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
