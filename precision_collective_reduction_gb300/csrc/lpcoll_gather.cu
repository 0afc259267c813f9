// lpcoll_gather.cu -- the collectives without a reduction: AllGather and
// AlltoAll over N emulated ranks, exact or low precision.
//
// The low-precision AllGather of 16-byte-aligned contributions runs on
// tiles staged in shared memory and written with bulk copies
// (gather_tile_kernel). The exact AllGather (and the LP one at unaligned
// lengths) and the exact AlltoAll: each warp takes an item of kItemUnits
// consecutive units (32 x kVec elements each) of one sender's data: it loads
// them all, and in low precision quantizes them on the sender's blocks (one
// absmax scale per 128 elements counted from the start of what the sender
// sends), stores the codes and scales to the sender's wire payload, and
// dequantizes them in registers; then it writes the (dequantized) values to
// the receiving outputs. Warps stride over (sender, destination, item), so
// each sender's data streams through HBM in order.
//
// The low-precision AlltoAll uses the wide lane layout (16 elements per lane,
// 8 lanes per block, 512 elements per warp item; lpcoll_wide.cuh), with the
// results written through the warp's shared-memory stage. On GB300 it took
// the 8-rank all-to-all from 61.4 to 57.2 us (BF16, chunks of 1 Mi), 227.3 to
// 214.7 us (BF16, 4 Mi) and 783.4 to 719.7 us (FP32, 8 Mi).
//
// Offsets that are not 16-byte aligned (a contribution or chunk length that
// is not a multiple of 16 bytes) take the element-by-element path for the
// accesses that need it; the choice is made once per launch (ALIGNED).
#include <algorithm>

#include "lpcoll_dda.cuh"
#include "lpcoll_device.cuh"
#include "lpcoll_wide.cuh"

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
                    store_scale(p.scales[r] + scale_base + e0[k] / kBlock, s);
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
    wait_prior_grid();
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

// Low-precision AllGather of contributions whose byte length is a multiple
// of 16 (every output offset then 16-byte aligned): a CTA takes a tile of
// kWarpsPerCta consecutive units of one sender (one per warp), quantizes and
// dequantizes it into one of two shared-memory tile buffers, and one thread
// writes the tile to all N receivers, and its codes and scales to the
// sender's wire, with bulk copies (cp.async.bulk.global.shared::cta); the
// units after a sender's last full tile are stored directly. Measured on
// GB300 against the item kernel above (8 ranks, CUDA events, L2 flushed):
// 1 Mi BF16 contributions 28.7 -> 28.7 us, 4 Mi BF16 108.5 -> 102.4 us,
// 8 Mi FP32 420.1 -> 386.7 us (6427 GB/s), both with grids of 3 resident
// CTAs per SM (2 or 4: 3-6% slower); one unit per warp (2 or 4 units: slower
// above 1 Mi). The grid has one CTA per tile (item_ctas).
template <int DT>
struct AgTile {
    static constexpr int kUnits = kWarpsPerCta;
    static constexpr int kElems = kUnits * 32 * Fmt<DT>::kVec;
    static constexpr int kBlocks = kElems / kBlock;
    static constexpr int kRes = 0;
    static constexpr int kCodes = kElems * (16 / Fmt<DT>::kVec);
    static constexpr int kScales = kCodes + kElems;
    static constexpr int kBytes = kScales + kBlocks * 4;
    static_assert(kCodes % 16 == 0 && kScales % 16 == 0 && kBytes % 16 == 0 &&
                      (kBlocks * 4) % 16 == 0,
                  "tile parts must be 16-byte aligned for bulk copies");
};

template <int DT>
__global__ void __launch_bounds__(kThreads)
gather_tile_kernel(const __grid_constant__ DdaParams p, int nranks, size_t m,
                   size_t tiles_per_sender, size_t units_per_sender)
{
    wait_prior_grid();
    using L = AgTile<DT>;
    constexpr int V = Fmt<DT>::kVec;
    constexpr int ES = 16 / V;
    extern __shared__ __align__(128) unsigned char ag_smem[];
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const size_t tiles = static_cast<size_t>(nranks) * tiles_per_sender;
    size_t i = 0;
    for (size_t t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
        const int r = static_cast<int>(t / tiles_per_sender);
        const size_t tt = t - static_cast<size_t>(r) * tiles_per_sender;
        unsigned char *tile = ag_smem + (i & 1) * L::kBytes;
        if (threadIdx.x == 0)  // the copies of two tiles ago have read this buffer
            asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncthreads();
        const size_t e0 = ((tt * L::kUnits + w) * 32 + lane) * V;
        const int off = (w * 32 + lane) * V;
        float x[V];
        widen<DT>(load_vec<DT>(p.in[r], e0, V), x);
        float s;
        const Codes<DT> c = quantize_lane<DT>(x, s);
        *reinterpret_cast<Codes<DT> *>(tile + L::kCodes + off) = c;
        if ((lane % Fmt<DT>::kGroup) == 0)
            reinterpret_cast<float *>(tile + L::kScales)[off / kBlock] = s;
        dequantize_lane<DT>(c, s, x);
        *reinterpret_cast<uint4 *>(tile + L::kRes + off * ES) = narrow<DT>(x);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (threadIdx.x == 0) {
            const size_t eb = tt * L::kElems;
            const size_t at = static_cast<size_t>(r) * m + eb;
            for (int d = 0; d < nranks; ++d)
                bulk_store(static_cast<char *>(p.out[d]) + at * ES, tile + L::kRes,
                           L::kElems * ES);
            bulk_store(p.codes[r] + eb, tile + L::kCodes, L::kElems);
            bulk_store(p.scales[r] + eb / kBlock, tile + L::kScales, L::kBlocks * 4);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
    }
    // the units after each sender's full tiles (the ragged one included),
    // one per warp, stored directly
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    const size_t u0 = tiles_per_sender * L::kUnits;
    const size_t tail = units_per_sender - u0;
    for (size_t it = warp; it < static_cast<size_t>(nranks) * tail; it += nwarps) {
        const int r = static_cast<int>(it / tail);
        const size_t u = u0 + (it - static_cast<size_t>(r) * tail);
        const size_t e0 = (u * 32 + lane) * V;
        const int cnt = lane_count<DT>(m, e0);
        float x[V];
        widen<DT>(cnt > 0 ? load_vec<DT>(p.in[r], e0, cnt) : make_uint4(0u, 0u, 0u, 0u), x);
        float s;
        const Codes<DT> c = quantize_lane<DT>(x, s);
        dequantize_lane<DT>(c, s, x);
        if (cnt > 0) {
            store_codes(p.codes[r], e0, cnt, c);
            if ((lane % Fmt<DT>::kGroup) == 0)
                store_scale(p.scales[r] + e0 / kBlock, s);
            const uint4 o = narrow<DT>(x);
            for (int d = 0; d < nranks; ++d)
                store_vec<DT>(p.out[d], static_cast<size_t>(r) * m + e0, cnt, o);
        }
    }
    if (threadIdx.x == 0)  // the copies must have completed before the CTA exits
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// One item of chunk j (c elements) of sender r in the exact AlltoAll.
template <int DT, bool ALIGNED>
__device__ __forceinline__ void alltoall_item(const DdaParams &p, size_t c, int r, int j,
                                              size_t g, int lane)
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
    const size_t at = static_cast<size_t>(r) * c;
#pragma unroll
    for (int k = 0; k < kItemUnits; ++k)
        if (cnt[k] > 0)
            store_vec<DT>(p.out[j], at + e0[k], access_count<DT>(cnt[k], ALIGNED), raw[k]);
}

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kThreads)
alltoall_kernel(const __grid_constant__ DdaParams p, int nranks, size_t c, size_t groups)
{
    wait_prior_grid();
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    const size_t per_sender = static_cast<size_t>(nranks) * groups;
    const size_t items = static_cast<size_t>(nranks) * per_sender;
    for (size_t it = warp; it < items; it += nwarps) {
        const int r = static_cast<int>(it / per_sender);
        const size_t rest = it - static_cast<size_t>(r) * per_sender;
        const int j = static_cast<int>(rest / groups);
        alltoall_item<DT, ALIGNED>(p, c, r, j, rest - static_cast<size_t>(j) * groups, lane);
    }
}

// Low-precision AlltoAll, per element format: wide items per warp step (all
// their loads issued first) and the resident CTAs per SM the registers are
// budgeted for (__launch_bounds__). The grid has one warp per step
// (item_ctas). Measured on GB300 with 8 ranks and that grid: FP32 2 items at
// 3 CTAs per SM (chunks of 8 Mi: 674.4 us against 688.8 us with 1 item, 705
// with 4), BF16 2 items at 4 CTAs per SM (1 item: -18%; 4 items at 3 CTAs:
// -2% at chunks of 1 Mi, +1% at 4 Mi).
template <int DT> struct A2aLp;
template <> struct A2aLp<LPCOLL_F32> {
    static constexpr int kItems = 2;
    static constexpr int kCtas = 3;
};
template <> struct A2aLp<LPCOLL_BF16> {
    static constexpr int kItems = 2;
    static constexpr int kCtas = 4;
};

// One step of the low-precision AlltoAll: wide items [g K, (g+1) K) of chunk j
// (c elements) of sender r. Each is quantized on the chunk's own blocks, its
// codes and scale go to sender r's wire (scales of chunk j start at j nbc),
// and the dequantized values go to out[j] at r c.
template <int DT, bool ALIGNED>
__device__ __forceinline__ void alltoall_lp_step(const DdaParams &p, size_t c, size_t nbc,
                                                 int r, int j, size_t g, int lane,
                                                 uint4 *stage)
{
    constexpr int V = Fmt<DT>::kVec;
    constexpr int S = kWideElems / V;
    constexpr int K = A2aLp<DT>::kItems;
    constexpr int ES = 16 / V;
    const size_t src = static_cast<size_t>(j) * c;
    size_t e0[K];
    uint4 raw[K][S];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        e0[k] = (g * K + k) * kWideItem + static_cast<size_t>(lane) * kWideElems;
#pragma unroll
        for (int q = 0; q < S; ++q) {
            const size_t e = e0[k] + q * V;
            const int cnt = lane_count<DT>(c, e);
            raw[k][q] = cnt > 0 ? load_vec<DT>(p.in[r], src + e, access_count<DT>(cnt, ALIGNED))
                                : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    char *out = static_cast<char *>(p.out[j]) + static_cast<size_t>(r) * c * ES;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        float x[kWideElems];
        wide_widen<DT>(raw[k], x);
        float s;
        uint32_t w[4];
        wide_quantize(x, w, s);
        if (e0[k] < c) {
            wide_store_codes(p.codes[r] + src, c, e0[k], w);
            if (lane % kWideGroup == 0)
                store_scale(p.scales[r] + static_cast<size_t>(j) * nbc + e0[k] / kBlock, s);
        }
        wide_dequant(make_uint4(w[0], w[1], w[2], w[3]), s, x);
        wide_store_results<DT, ALIGNED>(out, c, (g * K + k) * kWideItem, x, stage, lane);
    }
}

template <int DT, bool ALIGNED>
__global__ void __launch_bounds__(kThreads, A2aLp<DT>::kCtas)
alltoall_lp_kernel(const __grid_constant__ DdaParams p, int nranks, size_t c, size_t nbc,
                   size_t groups)
{
    wait_prior_grid();
    __shared__ uint4 stage_all[kWarpsPerCta][kWideElems * 32 / 4];
    uint4 *stage = stage_all[threadIdx.x >> 5];
    const int lane = threadIdx.x & 31;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const size_t nwarps = (static_cast<size_t>(gridDim.x) * kThreads) >> 5;
    const size_t per_sender = static_cast<size_t>(nranks) * groups;
    const size_t items = static_cast<size_t>(nranks) * per_sender;
    for (size_t it = warp; it < items; it += nwarps) {
        const int r = static_cast<int>(it / per_sender);
        const size_t rest = it - static_cast<size_t>(r) * per_sender;
        const int j = static_cast<int>(rest / groups);
        alltoall_lp_step<DT, ALIGNED>(p, c, nbc, r, j, rest - static_cast<size_t>(j) * groups,
                                      lane, stage);
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
    if constexpr (LP && ALIGNED) {
        using L = AgTile<DT>;
        size_t full, units;
        unit_counts<DT>(m, full, units);
        const size_t tps = full / L::kUnits;
        constexpr size_t smem = 2 * static_cast<size_t>(L::kBytes);
        static_assert(smem <= 48 * 1024, "tile buffers must fit the default dynamic smem");
        // one CTA per tile, or enough warps for the units after the tiles
        const size_t tail_units = static_cast<size_t>(nranks) * (units - tps * L::kUnits);
        const size_t need = std::max(static_cast<size_t>(nranks) * tps,
                                     (tail_units + kWarpsPerCta - 1) / kWarpsPerCta);
        return launch_kernel_smem(gather_tile_kernel<DT>, item_ctas(need * kWarpsPerCta), smem,
                                  st, p, nranks, m, tps, units);
    }
    const size_t groups = item_groups<DT>(m);
    return launch_kernel(gather_kernel<DT, LP, ALIGNED>,
                         item_ctas(groups * static_cast<size_t>(nranks)), st, p, nranks, m,
                         groups);
}

template <int DT, bool LP, bool ALIGNED>
cudaError_t launch_alltoall_t(const DdaParams &p, int nranks, size_t c, cudaStream_t st)
{
    const size_t pairs = static_cast<size_t>(nranks) * static_cast<size_t>(nranks);
    if constexpr (LP) {
        const size_t per = static_cast<size_t>(kWideItem) * A2aLp<DT>::kItems;
        const size_t groups = (c + per - 1) / per;
        const size_t nbc = (c + kBlock - 1) / kBlock;
        return launch_kernel(alltoall_lp_kernel<DT, ALIGNED>, item_ctas(groups * pairs), st, p,
                             nranks, c, nbc, groups);
    } else {
        const size_t groups = item_groups<DT>(c);
        return launch_kernel(alltoall_kernel<DT, ALIGNED>, item_ctas(groups * pairs), st, p,
                             nranks, c, groups);
    }
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
