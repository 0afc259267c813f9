// lpcoll_wide.cuh -- the wide lane layout of the staged quantize and reduce
// kernels and of the low-precision all-to-all: a lane holds 16 consecutive
// elements of one message (four FP32 or two BF16 16-byte vectors), 8 lanes
// hold one 128-element block, and a warp item covers 512 elements. Against
// the one-vector-per-lane warp-unit of the fused allreduce kernels, a lane
// moves its 16 codes with one 16-byte access, finds the block maximum in 3
// shuffle steps instead of 5 (FP32) or 4 (BF16), and computes the block
// scale once per 16 elements instead of once per 4 or 8. The arithmetic per
// element is the same, so both layouts give bit-identical results.
#pragma once

#include "lpcoll_device.cuh"

namespace lpc {

// Wide layout: elements per lane, lanes per block, elements per warp item.
constexpr int kWideElems = 16;
constexpr int kWideGroup = kBlock / kWideElems;
constexpr int kWideItem = 32 * kWideElems;

// 16 codes of a wide lane starting at element e0 < n (missing ones read 0).
__device__ __forceinline__ uint4 wide_load_codes(const uint8_t *codes, size_t n, size_t e0)
{
    if (!LPC_READ_OK(codes + e0, n - e0 < kWideElems ? n - e0 : kWideElems))
        return make_uint4(0u, 0u, 0u, 0u);
    if (n - e0 >= kWideElems)
        return __ldcs(reinterpret_cast<const uint4 *>(codes + e0));
    const size_t c = n - e0;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < kWideElems; ++j)
        if (static_cast<size_t>(j) < c)
            w[j / 4] |= static_cast<uint32_t>(codes[e0 + j]) << (8 * (j % 4));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Store the codes of a wide lane starting at element e0 < n (one 16-byte
// store where the address allows it, else byte by byte).
__device__ __forceinline__ void wide_store_codes(uint8_t *codes, size_t n, size_t e0,
                                                 const uint32_t (&w)[4])
{
    if (!LPC_WRITE_OK(codes + e0, n - e0 < kWideElems ? n - e0 : kWideElems))
        return;
    if (n - e0 >= kWideElems && (reinterpret_cast<uintptr_t>(codes + e0) & 15u) == 0) {
        __stcs(reinterpret_cast<uint4 *>(codes + e0), make_uint4(w[0], w[1], w[2], w[3]));
        return;
    }
    const size_t c = n - e0;
#pragma unroll
    for (int j = 0; j < kWideElems; ++j)
        if (static_cast<size_t>(j) < c)
            codes[e0 + j] = static_cast<uint8_t>(w[j / 4] >> (8 * (j % 4)));
}

// OCP FP8 formats: largest finite value and the conversion's interpretation.
template <int FMT> struct Fp8;
template <> struct Fp8<LPCOLL_E4M3> {
    static constexpr float kMax = 448.0f;
    static constexpr __nv_fp8_interpretation_t kKind = __NV_E4M3;
};
template <> struct Fp8<LPCOLL_E5M2> {
    static constexpr float kMax = 57344.0f;
    static constexpr __nv_fp8_interpretation_t kKind = __NV_E5M2;
};

// v = fl(fp8(code) * s) for the 16 codes of a wide lane (the FP8 -> FP16
// conversion is exact for both formats).
template <int FMT>
__device__ __forceinline__ void wide_dequant_fmt(uint4 c, float s, float (&v)[kWideElems])
{
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const __half2_raw lo_h = __nv_cvt_fp8x2_to_halfraw2(
            static_cast<__nv_fp8x2_storage_t>(w[q] & 0xFFFFu), Fp8<FMT>::kKind);
        const __half2_raw hi_h = __nv_cvt_fp8x2_to_halfraw2(
            static_cast<__nv_fp8x2_storage_t>(w[q] >> 16), Fp8<FMT>::kKind);
        const float2 lo = __half22float2(__half2(lo_h));
        const float2 hi = __half22float2(__half2(hi_h));
        v[4 * q + 0] = __fmul_rn(lo.x, s);
        v[4 * q + 1] = __fmul_rn(lo.y, s);
        v[4 * q + 2] = __fmul_rn(hi.x, s);
        v[4 * q + 3] = __fmul_rn(hi.y, s);
    }
}

// The main path's E4M3 decoding.
__device__ __forceinline__ void wide_dequant(uint4 c, float s, float (&v)[kWideElems])
{
    wide_dequant_fmt<LPCOLL_E4M3>(c, s, v);
}

// Store the 16 results of every lane of a warp item (first element item_e0)
// through the warp's shared-memory stage, so that each global store
// instruction writes 32 consecutive 16-byte vectors instead of 32 vectors
// 64 (FP32) or 32 (BF16) bytes apart. The slot of a vector is XOR-swizzled
// so that neither the writes nor the reads of the stage conflict on banks.
// All 32 lanes call it; results of lanes past the end are not stored.
// ALIGNED: out + item_e0 is 16-byte aligned (else element stores).
template <int DT, bool ALIGNED = true>
__device__ __forceinline__ void wide_store_results(void *out, size_t n, size_t item_e0,
                                                   const float (&v)[kWideElems],
                                                   uint4 *stage, int lane)
{
    constexpr int V = Fmt<DT>::kVec;
    constexpr int S = kWideElems / V;  // vectors per lane: 4 or 2
#pragma unroll
    for (int j = 0; j < S; ++j) {
        float t[V];
#pragma unroll
        for (int i = 0; i < V; ++i)
            t[i] = v[j * V + i];
        const int x = S == 4 ? ((lane >> 1) & 3) : ((lane >> 2) & 1);
        stage[lane * S + (j ^ x)] = narrow<DT>(t);
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < S; ++k) {
        const int m = k * 32 + lane;  // vector m of the item, held by lane m / S
        const int src = m / S;
        const int x = S == 4 ? ((src >> 1) & 3) : ((src >> 2) & 1);
        const uint4 val = stage[src * S + ((m % S) ^ x)];
        const size_t e = item_e0 + static_cast<size_t>(m) * V;
        const int cnt = lane_count<DT>(n, e);
        if (cnt > 0)
            store_vec<DT>(out, e, access_count<DT>(cnt, ALIGNED), val);
    }
    __syncwarp();
}

// Quantize the 16 values of a wide lane on its block of G lanes (16 G
// elements): a = block max |x|, s = fl(a / max), codes = fp8(fl(x * fl(max /
// a))) rounded to nearest even and saturated; a block whose max / a
// overflows gets s = 0 and signed-zero codes. Packed codes: element 4q + i
// in byte i of w[q].
template <int FMT, int G>
__device__ __forceinline__ void wide_quantize_fmt(const float (&x)[kWideElems], uint32_t (&w)[4],
                                                  float &s)
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kWideElems; ++i)
        amax = fmaxf(amax, fabsf(x[i]));
    amax = group_max<G>(amax);
    float inv = __fdiv_rn(Fp8<FMT>::kMax, amax);
    if (isinf(inv)) {
        inv = 0.0f;
        s = 0.0f;
    } else {
        s = __fdiv_rn(amax, Fp8<FMT>::kMax);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(
            make_float2(__fmul_rn(x[4 * q], inv), __fmul_rn(x[4 * q + 1], inv)), __NV_SATFINITE,
            Fp8<FMT>::kKind);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(
            make_float2(__fmul_rn(x[4 * q + 2], inv), __fmul_rn(x[4 * q + 3], inv)),
            __NV_SATFINITE, Fp8<FMT>::kKind);
        w[q] = lo | (hi << 16);
    }
}

// The main path: E4M3 on 128-element blocks.
__device__ __forceinline__ void wide_quantize(const float (&x)[kWideElems], uint32_t (&w)[4],
                                              float &s)
{
    wide_quantize_fmt<LPCOLL_E4M3, kWideGroup>(x, w, s);
}

// The values of the S = 16 / kVec vectors of a wide lane.
template <int DT>
__device__ __forceinline__ void wide_widen(const uint4 (&raw)[kWideElems / Fmt<DT>::kVec],
                                           float (&x)[kWideElems])
{
    constexpr int V = Fmt<DT>::kVec;
#pragma unroll
    for (int j = 0; j < kWideElems / V; ++j) {
        float t[V];
        widen<DT>(raw[j], t);
#pragma unroll
        for (int i = 0; i < V; ++i)
            x[j * V + i] = t[i];
    }
}

}  // namespace lpc
