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
// The grid has one warp per unit (or per group of units, see
// units_per_iter): item_ctas in lpcoll_device.cuh. The warps still stride
// over units, so any grid is correct, and no CTA waits on another.
//
// Tile path (TILES; see tile_path_built for where it is used): a CTA
// instead takes a tile of kTileUnits consecutive units (one per warp; one
// tile per CTA with the item_ctas grid), builds the tile's outputs, codes
// and scales in a shared-memory area, and one thread writes each of them
// with a single bulk copy (cp.async.bulk.global.shared::cta). The loads and
// the arithmetic are the same as on the direct path; only where the results
// go differs (the sink), so both paths give bit-identical results.
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
            uint32_t *q = static_cast<uint32_t *>(p.out[o]) + (e - o * L);
            if (LPC_WRITE_OK(q, 4))
                *q = w[j];
        } else {
            uint16_t *q = static_cast<uint16_t *>(p.out[o]) + (e - o * L);
            if (LPC_WRITE_OK(q, 2))
                *q = static_cast<uint16_t>(w[j >> 1] >> (16 * (j & 1)));
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

// The kVec codes of this lane for the element multiplier inv of its block.
template <int DT>
__device__ __forceinline__ Codes<DT> encode_with(const float (&x)[Fmt<DT>::kVec], float inv)
{
    constexpr int V = Fmt<DT>::kVec;
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

// Where a unit's results go. GlobalSink stores them straight to the
// caller's buffers (cnt valid elements at e0; FULL: cnt == kVec). TileSink
// writes them into the CTA's shared-memory tile, at the lane's element
// offset `off` within the tile, for the bulk copies that follow.
template <int N, int DT, int MODE, bool FULL>
struct GlobalSink {
    static constexpr bool kTile = false;
    const DdaParams &p;
    size_t e0;
    int cnt;
    __device__ __forceinline__ bool live() const { return FULL || cnt > 0; }
    __device__ __forceinline__ void codes(int r, Codes<DT> c) const
    {
        store_codes(p.codes[r], e0, cnt, c);
    }
    __device__ __forceinline__ void scale(int r, float s) const
    {
        store_scale(p.scales[r] + e0 / kBlock, s);
    }
    __device__ __forceinline__ void shard_codes(Codes<DT> c) const
    {
        store_codes(p.shard_codes, e0, cnt, c);
    }
    __device__ __forceinline__ void shard_scale(float s) const
    {
        store_scale(p.shard_scales + e0 / kBlock, s);
    }
    __device__ __forceinline__ void out(uint4 o) const
    {
        if constexpr (MODE == kScatterExact || MODE == kScatterLp) {
            scatter_store<DT>(p, e0, cnt, o);
        } else {
#pragma unroll
            for (int r = 0; r < N; ++r)
                store_vec<DT>(p.out[r], e0, cnt, o);
        }
    }
};

// Byte layout of one shared-memory tile buffer (kTileUnits units of every
// rank): the result, then per rank the codes and the scales, then the tree's
// shard codes and scales. Every part starts 16-byte aligned, as the bulk
// copies need.
constexpr int kTileUnits = kWarpsPerCta;
template <int N, int DT>
struct TileLayout {
    static constexpr int kElems = kTileUnits * 32 * Fmt<DT>::kVec;  // 1024 / 2048
    static constexpr int kBlocks = kElems / kBlock;
    static constexpr int kRes = 0;
    static constexpr int kCodes = kRes + kElems * (16 / Fmt<DT>::kVec);
    static constexpr int kScales = kCodes + N * kElems;
    static constexpr int kShardCodes = kScales + N * kBlocks * 4;
    static constexpr int kShardScales = kShardCodes + kElems;
    static constexpr int kBytes = kShardScales + kBlocks * 4;
    static_assert(kCodes % 16 == 0 && kScales % 16 == 0 && kShardCodes % 16 == 0 &&
                      kShardScales % 16 == 0 && kBytes % 16 == 0 && (kBlocks * 4) % 16 == 0,
                  "tile parts must be 16-byte aligned for bulk copies");
};

template <int N, int DT>
struct TileSink {
    static constexpr bool kTile = true;
    using L = TileLayout<N, DT>;
    unsigned char *tile;
    int off;  // element offset of this lane's first element in the tile
    __device__ __forceinline__ bool live() const { return true; }
    __device__ __forceinline__ void codes(int r, Codes<DT> c) const
    {
        *reinterpret_cast<Codes<DT> *>(tile + L::kCodes + r * L::kElems + off) = c;
    }
    __device__ __forceinline__ void scale(int r, float s) const
    {
        reinterpret_cast<float *>(tile + L::kScales)[r * L::kBlocks + off / kBlock] = s;
    }
    __device__ __forceinline__ void shard_codes(Codes<DT> c) const
    {
        *reinterpret_cast<Codes<DT> *>(tile + L::kShardCodes + off) = c;
    }
    __device__ __forceinline__ void shard_scale(float s) const
    {
        reinterpret_cast<float *>(tile + L::kShardScales)[off / kBlock] = s;
    }
    __device__ __forceinline__ void out(uint4 o) const
    {
        *reinterpret_cast<uint4 *>(tile + L::kRes + off * (16 / Fmt<DT>::kVec)) = o;
    }
};

// Everything after the loads: quantize / dequantize / reduce / requantize,
// then the results to the sink.
template <int N, int DT, int MODE, class Sink>
__device__ __forceinline__ void process_unit(const Sink &sink, int lane, const uint4 (&raw)[N])
{
    using F = Fmt<DT>;
    constexpr int V = F::kVec;
    constexpr bool kExactSum = (MODE == kExact || MODE == kScatterExact);
    const bool leader = (lane % F::kGroup) == 0;

    // Batched block scales: all ranks' block maxima first, then lane k of
    // each block group computes rank k's scale (the same two divisions,
    // once per rank instead of once per rank on every lane) and the scales
    // are shuffled back. Used by the tile path's tree, which it made 1.4%
    // faster (760.0 -> 749.5 us, 8 x 256 MiB FP32); the flat tile kernel
    // was 1.6% slower with it and the direct 16-rank tree 2.3% slower.
    constexpr bool kBatch = !kExactSum && MODE == kTree && Sink::kTile && N <= F::kGroup;
    float bs[kBatch ? N : 1], binv[kBatch ? N : 1];
    if constexpr (kBatch) {
        float amax[N];
#pragma unroll
        for (int r = 0; r < N; ++r) {
            float x[V];
            widen<DT>(raw[r], x);
            float a = 0.0f;
#pragma unroll
            for (int j = 0; j < V; ++j)
                a = fmaxf(a, fabsf(x[j]));
            amax[r] = group_max<F::kGroup>(a);
        }
        const int sub = lane % F::kGroup;  // the rank whose scale this lane computes
        const int base = lane - sub;       // first lane of this lane's block group
        float mine = amax[0];
#pragma unroll
        for (int r = 1; r < N; ++r)
            mine = (sub == r) ? amax[r] : mine;
        float ms, minv;
        block_scale(mine, ms, minv);
#pragma unroll
        for (int r = 0; r < N; ++r) {
            bs[r] = __shfl_sync(0xFFFFFFFFu, ms, base + r);
            binv[r] = __shfl_sync(0xFFFFFFFFu, minv, base + r);
        }
    }

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
            Codes<DT> c;
            if constexpr (kBatch) {
                s = bs[r];
                c = encode_with<DT>(x, binv[r]);
            } else {
                c = quantize_lane<DT>(x, s);
            }
            if (sink.live()) {
                sink.codes(r, c);
                if (leader)
                    sink.scale(r, s);
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
        if (sink.live()) {
            sink.shard_codes(c);
            if (leader)
                sink.shard_scale(s);
        }
        dequantize_lane<DT>(c, s, acc);
    }

    if (sink.live())
        sink.out(narrow<DT>(acc));
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
    process_unit<N, DT, MODE>(GlobalSink<N, DT, MODE, FULL>{p, e0, cnt}, lane, raw);
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
        process_unit<N, DT, MODE>(
            GlobalSink<N, DT, MODE, true>{p, ((unit0 + k) * 32 + lane) * V, V}, lane, raw[k]);
}

// One thread's bulk copy of `bytes` from shared to global memory; its
// completion is tracked with commit / wait groups.
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, uint32_t bytes)
{
    if (!LPC_WRITE_OK(gdst, bytes))
        return;
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(static_cast<uint32_t>(__cvta_generic_to_shared(ssrc))), "r"(bytes)
                 : "memory");
}

// Tile path. Full tiles (kTileUnits consecutive full units) go through the
// CTA's shared-memory tile and bulk copies, two tile buffers alternating;
// the units after the last full tile (fewer than kTileUnits full ones and
// the ragged one) take the direct path.
template <int N, int DT, int MODE>
__device__ __forceinline__ void dda_tiles(const DdaParams &p, size_t n, size_t full_units,
                                          size_t total_units)
{
    using L = TileLayout<N, DT>;
    constexpr int V = Fmt<DT>::kVec;
    constexpr int ES = 16 / V;
    extern __shared__ __align__(128) unsigned char tile_smem[];
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const size_t tiles = full_units / kTileUnits;
    size_t i = 0;
    for (size_t t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
        unsigned char *tile = tile_smem + (i & 1) * L::kBytes;
        if (threadIdx.x == 0)  // the copies of two tiles ago have read this buffer
            asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncthreads();
        const size_t e0 = ((t * kTileUnits + w) * 32 + lane) * V;
        uint4 raw[N];
        load_unit<N, DT, true>(p, e0, V, raw);
        process_unit<N, DT, MODE>(TileSink<N, DT>{tile, (w * 32 + lane) * V}, lane, raw);
        // the tile's generic-proxy writes must be visible to the bulk copies
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (threadIdx.x == 0) {
            const size_t eb = t * L::kElems;  // first element of the tile
            for (int r = 0; r < N; ++r)
                bulk_store(static_cast<char *>(p.out[r]) + eb * ES, tile + L::kRes,
                           L::kElems * ES);
            if constexpr (MODE != kExact) {
                for (int r = 0; r < N; ++r) {
                    bulk_store(p.codes[r] + eb, tile + L::kCodes + r * L::kElems, L::kElems);
                    bulk_store(p.scales[r] + eb / kBlock, tile + L::kScales + r * L::kBlocks * 4,
                               L::kBlocks * 4);
                }
            }
            if constexpr (MODE == kTree) {
                bulk_store(p.shard_codes + eb, tile + L::kShardCodes, L::kElems);
                bulk_store(p.shard_scales + eb / kBlock, tile + L::kShardScales,
                           L::kBlocks * 4);
            }
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
    }
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    const size_t u0 = tiles * kTileUnits;
    for (size_t u = u0 + warp; u < full_units; u += nwarps)
        dda_unit<N, DT, MODE, true>(p, n, u, lane);
    if (total_units > full_units && warp == (full_units - u0) % nwarps)
        dda_unit<N, DT, MODE, false>(p, n, full_units, lane);
    // the copies must have read the tiles (and landed) before the CTA exits
    if (threadIdx.x == 0)
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

template <int N, int DT, int MODE, bool TILES>
__global__ void __launch_bounds__(kThreads)
dda_kernel(const __grid_constant__ DdaParams p, size_t n, size_t full_units,
           size_t total_units)
{
    wait_prior_grid();
    if constexpr (TILES) {
        dda_tiles<N, DT, MODE>(p, n, full_units, total_units);
        return;
    }
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

// The direct path of dda_kernel with registers budgeted for 3 resident CTAs
// per SM (at most 80; a few bytes of spill). Left to itself the compiler
// gives the FP32 kernels of 14-16 ranks 84-98 registers, which leaves 2 CTAs
// per SM; with the budget they ran 4-7% faster on GB300 (2 GiB of input:
// 16 ranks flat 735.9 -> 705.2 us, 15 ranks tree 793.3 -> 742.0 us, 14 ranks
// tree 785.0 -> 735.9 us). 13 ranks and below, and BF16 at 12 and 16 ranks,
// were equal or slower with it. The loop repeats dda_kernel's instead of
// sharing a device function with it: with the loop in a shared function the
// compiler gave the BF16 8-rank kernels 65-68 registers instead of 64, one
// resident CTA per SM fewer.
template <int N, int DT, int MODE>
__global__ void __launch_bounds__(kThreads, 3)
dda_kernel_r3(const __grid_constant__ DdaParams p, size_t n, size_t full_units,
              size_t total_units)
{
    wait_prior_grid();
    constexpr int K = units_per_iter<N>();
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    size_t u = warp;
    if constexpr (K > 1) {
        const size_t groups = full_units / K;
        for (size_t g = warp; g < groups; g += nwarps)
            dda_units<N, DT, MODE, K>(p, g * K, lane);
        u = groups * K + warp;
    }
    for (; u < full_units; u += nwarps)
        dda_unit<N, DT, MODE, true>(p, n, u, lane);
    if (total_units > full_units && warp == full_units % nwarps)
        dda_unit<N, DT, MODE, false>(p, n, full_units, lane);
}

template <int N, int DT, int MODE>
constexpr bool register_budget_3()
{
    return DT == LPCOLL_F32 && N >= 14 && (MODE == kFlat || MODE == kTree);
}

// Units of a message of n elements: all full units, then the ragged one.
template <int DT>
inline void unit_counts(size_t n, size_t &full, size_t &total)
{
    const size_t per = 32 * static_cast<size_t>(Fmt<DT>::kVec);
    full = n / per;
    total = (n + per - 1) / per;
}

// Tile path policy, from measurements on GB300 (CUDA events, L2 flushed,
// LP, tile path against the direct path, both with the item_ctas grid):
//   FP32, 8 ranks: up to 512 MiB of input equal or slower (128 MiB flat
//     45.7 -> 47.7 us), 1 GiB equal (flat) / 1% faster (tree), 2 GiB
//     694.9 -> 688.8 us (flat) and 707.2 -> 697.0 us (tree), 4 GiB 1.1-1.2%
//     faster;
//   BF16, 8 ranks, 64 MiB to 1 GiB: equal or slower.
// With grids of 2-3 resident CTAs per SM (measured before item_ctas) it was
// also slower with 4, 12 and 16 ranks (4-11%) and equal for the exact
// allreduce. So it is taken for FP32 LP allreduces of 8 ranks and 1 GiB of
// input or more; everything else stays direct.
constexpr size_t kTileMinBytes = size_t(1) << 30;
template <int N, int DT, int MODE>
constexpr bool tile_path_built()
{
    return (MODE == kFlat || MODE == kTree) && DT == LPCOLL_F32 && N == 8;
}

template <int N, int DT, int MODE>
cudaError_t launch_dda_n(const DdaParams &p, size_t n, cudaStream_t stream)
{
    size_t full, total;
    unit_counts<DT>(n, full, total);
    if constexpr (tile_path_built<N, DT, MODE>()) {
        const size_t bytes = n * static_cast<size_t>(N) * (16 / Fmt<DT>::kVec);
        const size_t tiles = full / kTileUnits;
        constexpr size_t smem = 2 * static_cast<size_t>(TileLayout<N, DT>::kBytes);
        static_assert(smem <= 48 * 1024, "tile buffers must fit the default dynamic smem");
        if (bytes >= kTileMinBytes && tiles > 0) {
            // one tile per CTA, plus the warps for the units after the last tile
            const size_t rest = total - tiles * kTileUnits;
            const int grid = item_ctas(tiles * kWarpsPerCta > rest ? tiles * kWarpsPerCta : rest);
            return launch_kernel_smem(dda_kernel<N, DT, MODE, true>, grid, smem, stream, p, n,
                                      full, total);
        }
    }
    const size_t K = units_per_iter<N>();
    const int grid = item_ctas((total + K - 1) / K);
    if constexpr (register_budget_3<N, DT, MODE>())
        return launch_kernel(dda_kernel_r3<N, DT, MODE>, grid, stream, p, n, full, total);
    return launch_kernel(dda_kernel<N, DT, MODE, false>, grid, stream, p, n, full, total);
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
