// lpcoll_device.cuh -- device building blocks shared by the kernels of
// liblpcoll: 16-byte vector access, BF16 widening / narrowing, block absmax,
// the per-block FP8 scale, and E4M3 packing with the hardware cvt.
//
// Work decomposition used by every kernel: a "unit" is one warp-width of
// 16-byte vectors of one rank's message, i.e. 32 x kVec elements: one
// 128-element block for FP32 (4 elements per lane), two blocks for BF16
// (8 elements per lane, one block per half-warp). A block's absmax is
// therefore a shuffle reduction inside a group of kGroup lanes (32 or 16).
//
// All floating-point steps are single IEEE binary32 operations rounded to
// nearest even, written with the __f*_rn intrinsics so that the compiler can
// neither contract them into FMAs nor swap a division for a reciprocal.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lpcoll.h"

namespace lpc {

constexpr int kBlock = LPCOLL_BLOCK;  // elements per scale block
constexpr float kE4M3Max = 448.0f;    // largest finite E4M3 value
constexpr int kThreads = 256;         // threads per CTA of every kernel
constexpr int kWarpsPerCta = kThreads / 32;

// Grid size: one CTA per kWarpsPerCta work items (a warp-unit, a group of
// units, a wide item or a tile per warp, depending on the kernel), so that
// every warp takes one item. For messages of more than a wave this grid is
// far larger than what the GPU holds at once; the hardware hands out CTAs
// in index order as earlier ones finish, which balances the work across the
// SMs of both dies and keeps the addresses in flight close together. The
// kernels still loop over items with the grid as stride, so any grid gives
// the same results. Measured on GB300 (L2 flushed) against grids of 2-4
// resident CTAs per SM that stride over the whole message: FP32 8 x 256 MiB
// LP flat 737 -> 690 us and tree 756 -> 700 us, BF16 8 x 64 MiB tree 220 ->
// 199 us, BF16 8 x 16 MiB flat 53.9 -> 49.8 us, the 16 MiB BF16
// reduce-scatter / all-gather / all-to-all 4-7% faster, the staged quantize
// and dequantize of 64 Mi FP32 8% faster; messages of one wave or less are
// unchanged.
inline int item_ctas(size_t items)
{
    constexpr size_t kMaxGrid = 0x7FFFFFFF;
    const size_t g = (items + kWarpsPerCta - 1) / kWarpsPerCta;
    return static_cast<int>(g < 1 ? 1 : (g > kMaxGrid ? kMaxGrid : g));
}

// ---------------------------------------------------------------------------
// Launch. Every kernel of the library is launched with programmatic stream
// serialization (programmatic dependent launch), so the GPU may schedule it
// while the previous kernel of its stream is still running; its first
// instruction (wait_prior_grid) then waits until that kernel has completed
// and its memory writes are visible, so the stream order of all memory
// accesses is kept. What it saves is the gap between back-to-back launches:
// on GB300 the 8-rank 512 KiB decode allreduce went from 2.08 to 1.63 us per
// call in a CUDA graph and from 4.08 to 3.09 us launched back to back, with
// chained in-place calls bit-identical. No kernel triggers its dependents
// early (measured no faster).
// ---------------------------------------------------------------------------

__device__ __forceinline__ void wait_prior_grid()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Bounds-checked build (compiled with -DLPCOLL_DEBUG_BOUNDS; see
// lpcoll_debug_bounds_errors in lpcoll.h). Before its launches an entry
// point lists the buffers the call may touch, with the sizes its contract
// gives them: debug_begin(), then debug_range() per buffer (read-only for
// inputs, writable for outputs, wires and workspaces). The list is copied
// ahead of every launch into this translation unit's copy of
// g_debug_ranges, and every global load, store and bulk copy of the kernels
// first checks the bytes it touches against it (LPC_READ_OK /
// LPC_WRITE_OK). A failed check skips the access (a skipped load reads
// zeros), sets a flag and keeps the first bad address in a small managed
// record; nothing traps, so the context stays usable. In the normal build
// the list calls are empty and the checks are the constant true, so the
// kernels compile to the same code as without them.
// ---------------------------------------------------------------------------

constexpr int kDebugMaxRanges = 4 * LPCOLL_MAX_RANKS + 2;

struct DebugRanges {
    const char *lo[kDebugMaxRanges];
    const char *hi[kDebugMaxRanges];
    unsigned char writable[kDebugMaxRanges];
    int count;
    unsigned int *flag;            // set to 1 by the first failed check
    unsigned long long *first_bad;  // address of the first failed access
};

#ifdef LPCOLL_DEBUG_BOUNDS
void debug_begin();
void debug_range(const void *p, size_t bytes, bool writable);
const DebugRanges &debug_pending();

static __device__ DebugRanges g_debug_ranges;

static __device__ __noinline__ bool debug_access_ok(const void *p, size_t bytes, bool write)
{
    const char *a = static_cast<const char *>(p);
    const DebugRanges &d = g_debug_ranges;
    for (int i = 0; i < d.count; ++i)
        if (a >= d.lo[i] && a + bytes <= d.hi[i] && (!write || d.writable[i]))
            return true;
    if (d.flag != nullptr) {
        atomicCAS(d.first_bad, 0ull, reinterpret_cast<unsigned long long>(a));
        atomicOr(d.flag, 1u);
    }
    return false;
}
#define LPC_READ_OK(p, bytes) ::lpc::debug_access_ok((p), (bytes), false)
#define LPC_WRITE_OK(p, bytes) ::lpc::debug_access_ok((p), (bytes), true)
#else
inline void debug_begin() {}
inline void debug_range(const void *, size_t, bool) {}
#define LPC_READ_OK(p, bytes) true
#define LPC_WRITE_OK(p, bytes) true
#endif

// The launch helpers have internal linkage: in the bounds-checked build each
// translation unit must copy the buffer list into its own g_debug_ranges, so
// no two units may share one instantiation of them.
template <typename... Params, typename... Args>
static cudaError_t launch_kernel_smem(void (*kernel)(Params...), int grid, size_t smem,
                                      cudaStream_t stream, Args... args)
{
#ifdef LPCOLL_DEBUG_BOUNDS
    const cudaError_t de = cudaMemcpyToSymbolAsync(g_debug_ranges, &debug_pending(),
                                                   sizeof(DebugRanges), 0,
                                                   cudaMemcpyHostToDevice, stream);
    if (de != cudaSuccess)
        return de;
#endif
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename... Params, typename... Args>
static cudaError_t launch_kernel(void (*kernel)(Params...), int grid, cudaStream_t stream,
                                 Args... args)
{
    return launch_kernel_smem(kernel, grid, 0, stream, args...);
}

// What a fused launch computes: the allreduce (exact, LP flat, LP tree) or a
// reduce-scatter (exact or LP), whose result goes to the shard's owner only.
enum Mode { kExact = 0, kFlat = 1, kTree = 2, kScatterExact = 3, kScatterLp = 4 };

// Element format traits: elements per 16-byte vector and lanes per block.
template <int DT> struct Fmt;
template <> struct Fmt<LPCOLL_F32> {
    static constexpr int kVec = 4;
    static constexpr int kGroup = 32;
};
template <> struct Fmt<LPCOLL_BF16> {
    static constexpr int kVec = 8;
    static constexpr int kGroup = 16;
};

// Per-rank pointers of a fused allreduce launch (passed by value).
struct DdaParams {
    const void *in[LPCOLL_MAX_RANKS];
    void *out[LPCOLL_MAX_RANKS];
    uint8_t *codes[LPCOLL_MAX_RANKS];
    float *scales[LPCOLL_MAX_RANKS];
    uint8_t *shard_codes;
    float *shard_scales;
    size_t shard_len;  // reduce-scatter: elements per shard (last one shorter)
};

// Per-rank payload pointers of lp_reduce.
struct ReduceParams {
    const uint8_t *codes[LPCOLL_MAX_RANKS];
    const float *scales[LPCOLL_MAX_RANKS];
};

// ---------------------------------------------------------------------------
// Memory access. Messages move with plain 16-byte loads and stores (default
// cache policy: on GB300 it sustained 3-6% more HBM bandwidth than the
// evict-first hints at two CTAs per SM); the small code and scale stores are
// marked evict-first.
//
// The count argument `cnt` of load_vec / store_vec / store_codes:
//   cnt == kVec   a full lane at a 16-byte aligned address: one vector access;
//   0 < cnt < kVec  the lane holding the end of the data (the ragged unit):
//                 cnt element accesses; missing elements read as +0, which
//                 leaves a block maximum unchanged;
//   cnt < 0       -cnt elements at an address that may not be aligned for a
//                 vector access (see access_count): element accesses.
// ---------------------------------------------------------------------------

template <int DT>
__device__ __forceinline__ uint4 load_vec(const void *base, size_t e0, int cnt)
{
    constexpr int V = Fmt<DT>::kVec;
    constexpr int ES = 16 / V;  // element size in bytes
    const char *p = static_cast<const char *>(base) + e0 * ES;
    if (!LPC_READ_OK(p, static_cast<size_t>(cnt < 0 ? -cnt : cnt) * ES))
        return make_uint4(0u, 0u, 0u, 0u);
    if (cnt == V)
        return *reinterpret_cast<const uint4 *>(p);
    if (cnt < 0)
        cnt = -cnt;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (DT == LPCOLL_F32) {
        const uint32_t *q = reinterpret_cast<const uint32_t *>(p);
        for (int j = 0; j < cnt; ++j)
            w[j] = q[j];
    } else {
        const uint16_t *q = reinterpret_cast<const uint16_t *>(p);
        for (int j = 0; j < cnt; ++j)
            w[j >> 1] |= static_cast<uint32_t>(q[j]) << (16 * (j & 1));
    }
    v.x = w[0];
    v.y = w[1];
    v.z = w[2];
    v.w = w[3];
    return v;
}

template <int DT>
__device__ __forceinline__ void store_vec(void *base, size_t e0, int cnt, uint4 v)
{
    constexpr int V = Fmt<DT>::kVec;
    constexpr int ES = 16 / V;
    char *p = static_cast<char *>(base) + e0 * ES;
    if (!LPC_WRITE_OK(p, static_cast<size_t>(cnt < 0 ? -cnt : cnt) * ES))
        return;
    if (cnt == V) {
        *reinterpret_cast<uint4 *>(p) = v;
        return;
    }
    if (cnt < 0)
        cnt = -cnt;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if (DT == LPCOLL_F32) {
        uint32_t *q = reinterpret_cast<uint32_t *>(p);
        for (int j = 0; j < cnt; ++j)
            q[j] = w[j];
    } else {
        uint16_t *q = reinterpret_cast<uint16_t *>(p);
        for (int j = 0; j < cnt; ++j)
            q[j] = static_cast<uint16_t>(w[j >> 1] >> (16 * (j & 1)));
    }
}

// Count argument for an access of cnt valid elements at an offset that is
// vector-aligned only if `aligned` (uniform per launch) holds.
template <int DT>
__device__ __forceinline__ int access_count(int cnt, bool aligned)
{
    return (aligned || cnt != Fmt<DT>::kVec) ? cnt : -cnt;
}

// kVec codes of one lane, packed little-endian (element e0 in the low byte).
template <int DT> struct Codes;
template <> struct Codes<LPCOLL_F32> {
    uint32_t w;
};
template <> struct Codes<LPCOLL_BF16> {
    uint2 w;
};

__device__ __forceinline__ void store_codes(uint8_t *base, size_t e0, int cnt,
                                            Codes<LPCOLL_F32> c)
{
    if (!LPC_WRITE_OK(base + e0, static_cast<size_t>(cnt < 0 ? -cnt : cnt)))
        return;
    if (cnt == 4) {
        __stcs(reinterpret_cast<unsigned int *>(base + e0), c.w);
        return;
    }
    if (cnt < 0)
        cnt = -cnt;
    for (int j = 0; j < cnt; ++j)
        base[e0 + j] = static_cast<uint8_t>(c.w >> (8 * j));
}

__device__ __forceinline__ void store_codes(uint8_t *base, size_t e0, int cnt,
                                            Codes<LPCOLL_BF16> c)
{
    if (!LPC_WRITE_OK(base + e0, static_cast<size_t>(cnt < 0 ? -cnt : cnt)))
        return;
    if (cnt == 8) {
        __stcs(reinterpret_cast<uint2 *>(base + e0), c.w);
        return;
    }
    if (cnt < 0)
        cnt = -cnt;
    for (int j = 0; j < cnt; ++j) {
        uint32_t word = j < 4 ? c.w.x : c.w.y;
        base[e0 + j] = static_cast<uint8_t>(word >> (8 * (j & 3)));
    }
}

__device__ __forceinline__ Codes<LPCOLL_F32> load_codes_f32(const uint8_t *base,
                                                           size_t e0, int cnt)
{
    Codes<LPCOLL_F32> c;
    c.w = 0u;
    if (!LPC_READ_OK(base + e0, static_cast<size_t>(cnt)))
        return c;
    if (cnt == 4) {
        c.w = __ldcs(reinterpret_cast<const unsigned int *>(base + e0));
        return c;
    }
    for (int j = 0; j < cnt; ++j)
        c.w |= static_cast<uint32_t>(base[e0 + j]) << (8 * j);
    return c;
}

__device__ __forceinline__ Codes<LPCOLL_BF16> load_codes_bf16(const uint8_t *base,
                                                             size_t e0, int cnt)
{
    Codes<LPCOLL_BF16> c;
    c.w = make_uint2(0u, 0u);
    if (!LPC_READ_OK(base + e0, static_cast<size_t>(cnt)))
        return c;
    if (cnt == 8) {
        c.w = __ldcs(reinterpret_cast<const uint2 *>(base + e0));
        return c;
    }
    for (int j = 0; j < cnt; ++j) {
        uint32_t b = static_cast<uint32_t>(base[e0 + j]) << (8 * (j & 3));
        if (j < 4)
            c.w.x |= b;
        else
            c.w.y |= b;
    }
    return c;
}

template <int DT>
__device__ __forceinline__ Codes<DT> load_codes(const uint8_t *base, size_t e0, int cnt);
template <>
__device__ __forceinline__ Codes<LPCOLL_F32> load_codes<LPCOLL_F32>(const uint8_t *base,
                                                                   size_t e0, int cnt)
{
    return load_codes_f32(base, e0, cnt);
}
template <>
__device__ __forceinline__ Codes<LPCOLL_BF16> load_codes<LPCOLL_BF16>(const uint8_t *base,
                                                                     size_t e0, int cnt)
{
    return load_codes_bf16(base, e0, cnt);
}

// One block scale to / from a wire payload (stores marked evict-first).
__device__ __forceinline__ void store_scale(float *p, float s)
{
    if (LPC_WRITE_OK(p, sizeof(float)))
        __stcs(p, s);
}

__device__ __forceinline__ float load_scale(const float *p)
{
    return LPC_READ_OK(p, sizeof(float)) ? *p : 0.0f;
}

// ---------------------------------------------------------------------------
// Element formats
// ---------------------------------------------------------------------------

// 16 bytes -> kVec floats (FP32: reinterpretation; BF16: exact shift).
template <int DT>
__device__ __forceinline__ void widen(uint4 v, float (&x)[Fmt<DT>::kVec])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (DT == LPCOLL_F32) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            x[j] = __uint_as_float(w[j]);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            x[2 * j] = __uint_as_float(w[j] << 16);
            x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
}

// kVec floats -> 16 bytes (BF16: round to nearest even).
template <int DT>
__device__ __forceinline__ uint4 narrow(const float (&x)[Fmt<DT>::kVec])
{
    uint32_t w[4];
    if constexpr (DT == LPCOLL_F32) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            w[j] = __float_as_uint(x[j]);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * j], x[2 * j + 1]);
            w[j] = *reinterpret_cast<uint32_t *>(&h);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------------------
// FP8 block quantization
// ---------------------------------------------------------------------------

// Largest |x| over the kGroup lanes holding one block (max is exact, so the
// shuffle order does not matter).
template <int G>
__device__ __forceinline__ float group_max(float v)
{
#pragma unroll
    for (int m = G / 2; m >= 1; m >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
    return v;
}

// Block scale s = a/448 and element multiplier inv = 448/a, each one IEEE
// division. If 448/a overflows, the block is degenerate: s = inv = 0, which
// turns every element into a signed zero code.
__device__ __forceinline__ void block_scale(float amax, float &s, float &inv)
{
    inv = __fdiv_rn(kE4M3Max, amax);
    if (isinf(inv)) {
        inv = 0.0f;
        s = 0.0f;
    } else {
        s = __fdiv_rn(amax, kE4M3Max);
    }
}

// Two floats -> two E4M3 codes (a in the low byte), RNE, saturating.
__device__ __forceinline__ uint32_t enc2(float a, float b)
{
    return static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// Two E4M3 codes (low byte first) -> two exact floats (via FP16, exact).
__device__ __forceinline__ float2 dec2(uint32_t c2)
{
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
        static_cast<__nv_fp8x2_storage_t>(c2 & 0xFFFFu), __NV_E4M3);
    return __half22float2(__half2(h));
}

// Quantize the kVec values of this lane (block scale from its group):
// returns the packed codes and writes s.
template <int DT>
__device__ __forceinline__ Codes<DT> quantize_lane(const float (&x)[Fmt<DT>::kVec],
                                                   float &s)
{
    constexpr int V = Fmt<DT>::kVec;
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < V; ++j)
        amax = fmaxf(amax, fabsf(x[j]));
    amax = group_max<Fmt<DT>::kGroup>(amax);
    float inv;
    block_scale(amax, s, inv);
    uint32_t c2[V / 2];
#pragma unroll
    for (int j = 0; j < V / 2; ++j)
        c2[j] = enc2(__fmul_rn(x[2 * j], inv), __fmul_rn(x[2 * j + 1], inv));
    Codes<DT> c;
    if constexpr (DT == LPCOLL_F32) {
        c.w = c2[0] | (c2[1] << 16);
    } else {
        c.w = make_uint2(c2[0] | (c2[1] << 16), c2[2] | (c2[3] << 16));
    }
    return c;
}

// Dequantize this lane's codes with scale s: v = fl(e4m3 * s).
template <int DT>
__device__ __forceinline__ void dequantize_lane(Codes<DT> c, float s,
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
        float2 lo = dec2(words[k]);
        float2 hi = dec2(words[k] >> 16);
        v[4 * k + 0] = __fmul_rn(lo.x, s);
        v[4 * k + 1] = __fmul_rn(lo.y, s);
        v[4 * k + 2] = __fmul_rn(hi.x, s);
        v[4 * k + 3] = __fmul_rn(hi.y, s);
    }
}

// Number of valid elements of a lane whose first element is e0.
template <int DT>
__device__ __forceinline__ int lane_count(size_t n, size_t e0)
{
    constexpr int V = Fmt<DT>::kVec;
    return e0 >= n ? 0 : (n - e0 >= (size_t)V ? V : static_cast<int>(n - e0));
}

}  // namespace lpc
