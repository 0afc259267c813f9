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

// v = fl(e4m3(code) * s) for the 16 codes of a wide lane.
__device__ __forceinline__ void wide_dequant(uint4 c, float s, float (&v)[kWideElems])
{
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 lo = dec2(w[q]);
        const float2 hi = dec2(w[q] >> 16);
        v[4 * q + 0] = __fmul_rn(lo.x, s);
        v[4 * q + 1] = __fmul_rn(lo.y, s);
        v[4 * q + 2] = __fmul_rn(hi.x, s);
        v[4 * q + 3] = __fmul_rn(hi.y, s);
    }
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

// Quantize the 16 values of a wide lane on its block (8-lane group): the
// packed codes (element 4q + i in byte i of w[q]) and the block scale s.
__device__ __forceinline__ void wide_quantize(const float (&x)[kWideElems], uint32_t (&w)[4],
                                              float &s)
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kWideElems; ++i)
        amax = fmaxf(amax, fabsf(x[i]));
    amax = group_max<kWideGroup>(amax);
    float inv;
    block_scale(amax, s, inv);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        w[q] = enc2(__fmul_rn(x[4 * q], inv), __fmul_rn(x[4 * q + 1], inv)) |
               (enc2(__fmul_rn(x[4 * q + 2], inv), __fmul_rn(x[4 * q + 3], inv)) << 16);
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
