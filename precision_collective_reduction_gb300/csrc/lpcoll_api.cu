// lpcoll_api.cu -- the extern "C" entry points of liblpcoll.so: argument
// checks (all done on the host before anything is enqueued) and dispatch to
// the kernels. The semantics of each call are documented in
// include/lpcoll.h.
#include <cuda_runtime.h>
#include <stdint.h>

#include <initializer_list>
#ifdef LPCOLL_DEBUG_BOUNDS
#include <atomic>
#include <mutex>
#endif

#include "lpcoll.h"
#include "lpcoll_dda.cuh"

namespace lpc {

cudaError_t launch_quantize(const void *in, int dtype, size_t n, uint8_t *codes,
                            float *scales, cudaStream_t stream);
cudaError_t launch_dequantize(const uint8_t *codes, const float *scales, size_t n,
                              void *out, int dtype, cudaStream_t stream);
cudaError_t launch_reduce(const ReduceParams &p, int nranks, size_t n, void *out,
                          int dtype, cudaStream_t stream);
cudaError_t launch_all_gather(const DdaParams &p, int nranks, size_t m, int dtype,
                              bool lp, cudaStream_t st);
cudaError_t launch_quantize_fmt(const void *in, int dtype, size_t n, int block, int fmt,
                                uint8_t *codes, float *scales, cudaStream_t st);
cudaError_t launch_dequantize_fmt(const uint8_t *codes, const float *scales, size_t n,
                                  int block, int fmt, void *out, int dtype,
                                  cudaStream_t st);
cudaError_t launch_reduce_fmt(const ReduceParams &p, int nranks, size_t n, int block,
                              int fmt, void *out, int dtype, cudaStream_t st);
cudaError_t launch_all_to_all(const DdaParams &p, int nranks, size_t c, int dtype,
                              bool lp, cudaStream_t st);

namespace {

thread_local int g_last_cuda_error = 0;

inline bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

inline bool bad_dtype(int dtype) { return dtype != LPCOLL_F32 && dtype != LPCOLL_BF16; }

// NULL / alignment check of one per-rank pointer array.
template <class P>
int check_rank_array(P const *arr, int nranks)
{
    if (arr == nullptr)
        return LPCOLL_ERR_ARG;
    for (int r = 0; r < nranks; ++r)
        if (arr[r] == nullptr)
            return LPCOLL_ERR_RANK;
    for (int r = 0; r < nranks; ++r)
        if (misaligned(arr[r]))
            return LPCOLL_ERR_ALIGN;
    return LPCOLL_OK;
}

int check_ptr(const void *p)
{
    if (p == nullptr)
        return LPCOLL_ERR_ARG;
    return misaligned(p) ? LPCOLL_ERR_ALIGN : LPCOLL_OK;
}

int finish(cudaError_t e)
{
    if (e == cudaSuccess)
        return LPCOLL_OK;
    g_last_cuda_error = static_cast<int>(e);
    return LPCOLL_ERR_CUDA;
}

// First non-OK status of a list of checks (NULL before alignment is kept by
// the order in which callers list them).
int first_error(std::initializer_list<int> sts)
{
    int align = LPCOLL_OK;
    for (int s : sts) {
        if (s == LPCOLL_ERR_ALIGN) {
            if (align == LPCOLL_OK)
                align = s;
        } else if (s != LPCOLL_OK) {
            return s;
        }
    }
    return align;
}

size_t elem_bytes(int dtype) { return dtype == LPCOLL_F32 ? 4 : 2; }

size_t blocks_of(size_t n, int block) { return (n + block - 1) / block; }

// Bounds-checked build: the buffers of an allreduce-shaped call (inputs read,
// outputs and wires written, and the tree's shard payload when given).
void debug_dda_ranges(const void *const *in, void *const *out, int nranks, size_t n,
                      int dtype, int block, uint8_t *const *wire_codes,
                      float *const *wire_scales, const uint8_t *shard_codes,
                      const float *shard_scales)
{
    debug_begin();
    for (int r = 0; r < nranks; ++r) {
        debug_range(in[r], n * elem_bytes(dtype), false);
        debug_range(out[r], n * elem_bytes(dtype), true);
        if (block) {
            debug_range(wire_codes[r], n, true);
            debug_range(wire_scales[r], blocks_of(n, block) * sizeof(float), true);
        }
    }
    if (block && shard_codes != nullptr) {
        debug_range(shard_codes, n, true);
        debug_range(shard_scales, blocks_of(n, block) * sizeof(float), true);
    }
}

int dda_common(const void *const *in, void *const *out, int nranks, size_t n,
               int dtype, int block, uint8_t *const *wire_codes,
               float *const *wire_scales, uint8_t *shard_codes, float *shard_scales,
               bool tree, void *stream)
{
    if (bad_dtype(dtype) || nranks < 1 || nranks > LPCOLL_MAX_RANKS)
        return LPCOLL_ERR_ARG;
    if (block != 0 && block != LPCOLL_BLOCK)
        return LPCOLL_ERR_UNSUPPORTED;
    if (n == 0)
        return LPCOLL_OK;
    const bool lp = block != 0;
    int st = first_error({
        check_rank_array(in, nranks),
        check_rank_array(out, nranks),
        lp ? check_rank_array(wire_codes, nranks) : LPCOLL_OK,
        lp ? check_rank_array(wire_scales, nranks) : LPCOLL_OK,
        (lp && tree) ? check_ptr(shard_codes) : LPCOLL_OK,
        (lp && tree) ? check_ptr(shard_scales) : LPCOLL_OK,
    });
    if (st != LPCOLL_OK)
        return st;

    DdaParams p = {};
    for (int r = 0; r < nranks; ++r) {
        p.in[r] = in[r];
        p.out[r] = out[r];
        if (lp) {
            p.codes[r] = wire_codes[r];
            p.scales[r] = wire_scales[r];
        }
    }
    p.shard_codes = (lp && tree) ? shard_codes : nullptr;
    p.shard_scales = (lp && tree) ? shard_scales : nullptr;
    debug_dda_ranges(in, out, nranks, n, dtype, block, wire_codes, wire_scales, p.shard_codes,
                     p.shard_scales);
    const int mode = !lp ? kExact : (tree ? kTree : kFlat);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish(dtype == LPCOLL_F32 ? launch_dda_f32(p, nranks, n, mode, s)
                                      : launch_dda_bf16(p, nranks, n, mode, s));
}

// Checks shared by the collectives other than the allreduce; fills the
// per-rank pointers of p. out[r] may be NULL where out_empty(r) is true.
template <class Empty>
int collective_args(const void *const *in, void *const *out, int nranks, int block,
                    uint8_t *const *wire_codes, float *const *wire_scales, Empty out_empty,
                    DdaParams &p)
{
    int out_st = LPCOLL_OK;
    if (out == nullptr) {
        out_st = LPCOLL_ERR_ARG;
    } else {
        for (int r = 0; r < nranks && out_st != LPCOLL_ERR_RANK; ++r) {
            if (out[r] == nullptr && !out_empty(r))
                out_st = LPCOLL_ERR_RANK;
            else if (out[r] != nullptr && misaligned(out[r]))
                out_st = LPCOLL_ERR_ALIGN;
        }
    }
    int st = first_error({
        check_rank_array(in, nranks),
        out_st,
        block ? check_rank_array(wire_codes, nranks) : LPCOLL_OK,
        block ? check_rank_array(wire_scales, nranks) : LPCOLL_OK,
    });
    if (st != LPCOLL_OK)
        return st;
    for (int r = 0; r < nranks; ++r) {
        p.in[r] = in[r];
        p.out[r] = out[r];
        if (block) {
            p.codes[r] = wire_codes[r];
            p.scales[r] = wire_scales[r];
        }
    }
    return LPCOLL_OK;
}

// dtype / format / block of the *_fmt variants.
int check_variant(int dtype, int fmt, int block)
{
    if (bad_dtype(dtype) || (fmt != LPCOLL_E4M3 && fmt != LPCOLL_E5M2))
        return LPCOLL_ERR_ARG;
    if (block != 32 && block != 64 && block != 128 && block != 256)
        return LPCOLL_ERR_UNSUPPORTED;
    return LPCOLL_OK;
}

int check_common(int dtype, int nranks, int block)
{
    if (bad_dtype(dtype) || nranks < 1 || nranks > LPCOLL_MAX_RANKS)
        return LPCOLL_ERR_ARG;
    if (block != 0 && block != LPCOLL_BLOCK)
        return LPCOLL_ERR_UNSUPPORTED;
    return LPCOLL_OK;
}

#ifdef LPCOLL_DEBUG_BOUNDS
// The bounds-check record that kernels write (managed memory, one per
// process) and the buffer list of the calling thread's current call.
struct DebugRecord {
    unsigned int flag;
    unsigned int pad;
    unsigned long long first_bad;
};
std::mutex g_record_mutex;
DebugRecord *g_record = nullptr;
thread_local DebugRanges g_pending = {};
// lpcoll_debug_bounds_shrink: bytes taken off every buffer of the next call
std::atomic<size_t> g_shrink_next{0};
thread_local size_t g_shrink = 0;

DebugRecord *debug_record()
{
    std::lock_guard<std::mutex> lock(g_record_mutex);
    if (g_record == nullptr) {
        void *p = nullptr;
        if (cudaMallocManaged(&p, sizeof(DebugRecord)) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_record = static_cast<DebugRecord *>(p);
        g_record->flag = 0;
        g_record->first_bad = 0;
    }
    return g_record;
}
#endif

}  // namespace

#ifdef LPCOLL_DEBUG_BOUNDS
void debug_begin()
{
    DebugRecord *rec = debug_record();
    g_shrink = g_shrink_next.exchange(0);
    g_pending.count = 0;
    g_pending.flag = rec != nullptr ? &rec->flag : nullptr;
    g_pending.first_bad = rec != nullptr ? &rec->first_bad : nullptr;
}

void debug_range(const void *p, size_t bytes, bool writable)
{
    if (p == nullptr || g_pending.count >= kDebugMaxRanges)
        return;
    const int i = g_pending.count++;
    g_pending.lo[i] = static_cast<const char *>(p);
    g_pending.hi[i] = static_cast<const char *>(p) + (bytes > g_shrink ? bytes - g_shrink : 0);
    g_pending.writable[i] = writable ? 1 : 0;
}

const DebugRanges &debug_pending() { return g_pending; }
#endif

void record_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int>(e); }

}  // namespace lpc

using namespace lpc;

extern "C" {

int lp_quantize(const void *in, lpcoll_dtype dtype, size_t n, int block,
                uint8_t *codes, float *scales, void *stream)
{
    if (bad_dtype(dtype))
        return LPCOLL_ERR_ARG;
    if (block != LPCOLL_BLOCK)
        return LPCOLL_ERR_UNSUPPORTED;
    if (n == 0)
        return LPCOLL_OK;
    int st = first_error({check_ptr(in), check_ptr(codes), check_ptr(scales)});
    if (st != LPCOLL_OK)
        return st;
    debug_begin();
    debug_range(in, n * elem_bytes(dtype), false);
    debug_range(codes, n, true);
    debug_range(scales, blocks_of(n, block) * sizeof(float), true);
    return finish(launch_quantize(in, dtype, n, codes, scales,
                                  static_cast<cudaStream_t>(stream)));
}

int lp_dequantize(const uint8_t *codes, const float *scales, size_t n, int block,
                  void *out, lpcoll_dtype dtype, void *stream)
{
    if (bad_dtype(dtype))
        return LPCOLL_ERR_ARG;
    if (block != LPCOLL_BLOCK)
        return LPCOLL_ERR_UNSUPPORTED;
    if (n == 0)
        return LPCOLL_OK;
    int st = first_error({check_ptr(codes), check_ptr(scales), check_ptr(out)});
    if (st != LPCOLL_OK)
        return st;
    debug_begin();
    debug_range(codes, n, false);
    debug_range(scales, blocks_of(n, block) * sizeof(float), false);
    debug_range(out, n * elem_bytes(dtype), true);
    return finish(launch_dequantize(codes, scales, n, out, dtype,
                                    static_cast<cudaStream_t>(stream)));
}

int lp_reduce(const uint8_t *const *codes, const float *const *scales, int nranks,
              size_t n, int block, void *out, lpcoll_dtype dtype, void *stream)
{
    if (bad_dtype(dtype) || nranks < 1 || nranks > LPCOLL_MAX_RANKS)
        return LPCOLL_ERR_ARG;
    if (block != LPCOLL_BLOCK)
        return LPCOLL_ERR_UNSUPPORTED;
    if (n == 0)
        return LPCOLL_OK;
    int st = first_error({check_rank_array(codes, nranks),
                          check_rank_array(scales, nranks), check_ptr(out)});
    if (st != LPCOLL_OK)
        return st;
    ReduceParams p = {};
    debug_begin();
    for (int r = 0; r < nranks; ++r) {
        p.codes[r] = codes[r];
        p.scales[r] = scales[r];
        debug_range(codes[r], n, false);
        debug_range(scales[r], blocks_of(n, block) * sizeof(float), false);
    }
    debug_range(out, n * elem_bytes(dtype), true);
    return finish(launch_reduce(p, nranks, n, out, dtype,
                                static_cast<cudaStream_t>(stream)));
}

int dda_flat_sim(const void *const *in, void *const *out, int nranks, size_t n,
                 lpcoll_dtype dtype, int block, uint8_t *const *wire_codes,
                 float *const *wire_scales, void *stream)
{
    return dda_common(in, out, nranks, n, dtype, block, wire_codes, wire_scales,
                      nullptr, nullptr, false, stream);
}

int dda_tree_sim(const void *const *in, void *const *out, int nranks, size_t n,
                 lpcoll_dtype dtype, int block, uint8_t *const *wire_codes,
                 float *const *wire_scales, uint8_t *shard_codes,
                 float *shard_scales, void *stream)
{
    return dda_common(in, out, nranks, n, dtype, block, wire_codes, wire_scales,
                      shard_codes, shard_scales, true, stream);
}

int reduce_scatter_sim(const void *const *in, void *const *out, int nranks, size_t n,
                       lpcoll_dtype dtype, int block, uint8_t *const *wire_codes,
                       float *const *wire_scales, void *stream)
{
    int st = check_common(dtype, nranks, block);
    if (st != LPCOLL_OK || n == 0)
        return st;
    size_t per = (n + static_cast<size_t>(nranks) - 1) / static_cast<size_t>(nranks);
    if (block)
        per = (per + LPCOLL_BLOCK - 1) / LPCOLL_BLOCK * LPCOLL_BLOCK;
    DdaParams p = {};
    st = collective_args(in, out, nranks, block, wire_codes, wire_scales,
                         [&](int r) { return static_cast<size_t>(r) * per >= n; }, p);
    if (st != LPCOLL_OK)
        return st;
    p.shard_len = per;
    debug_begin();
    for (int r = 0; r < nranks; ++r) {
        const size_t lo = static_cast<size_t>(r) * per;
        debug_range(in[r], n * elem_bytes(dtype), false);
        if (lo < n)
            debug_range(out[r], (n - lo < per ? n - lo : per) * elem_bytes(dtype), true);
        if (block) {
            debug_range(wire_codes[r], n, true);
            debug_range(wire_scales[r], blocks_of(n, block) * sizeof(float), true);
        }
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return finish(dtype == LPCOLL_F32 ? launch_scatter_f32(p, nranks, n, block != 0, s)
                                      : launch_scatter_bf16(p, nranks, n, block != 0, s));
}

int all_gather_sim(const void *const *in, void *const *out, int nranks, size_t m,
                   lpcoll_dtype dtype, int block, uint8_t *const *wire_codes,
                   float *const *wire_scales, void *stream)
{
    int st = check_common(dtype, nranks, block);
    if (st != LPCOLL_OK || m == 0)
        return st;
    DdaParams p = {};
    st = collective_args(in, out, nranks, block, wire_codes, wire_scales,
                         [](int) { return false; }, p);
    if (st != LPCOLL_OK)
        return st;
    debug_begin();
    for (int r = 0; r < nranks; ++r) {
        debug_range(in[r], m * elem_bytes(dtype), false);
        debug_range(out[r], static_cast<size_t>(nranks) * m * elem_bytes(dtype), true);
        if (block) {
            debug_range(wire_codes[r], m, true);
            debug_range(wire_scales[r], blocks_of(m, block) * sizeof(float), true);
        }
    }
    return finish(launch_all_gather(p, nranks, m, dtype, block != 0,
                                    static_cast<cudaStream_t>(stream)));
}

int all_to_all_sim(const void *const *in, void *const *out, int nranks, size_t c,
                   lpcoll_dtype dtype, int block, uint8_t *const *wire_codes,
                   float *const *wire_scales, void *stream)
{
    int st = check_common(dtype, nranks, block);
    if (st != LPCOLL_OK || c == 0)
        return st;
    DdaParams p = {};
    st = collective_args(in, out, nranks, block, wire_codes, wire_scales,
                         [](int) { return false; }, p);
    if (st != LPCOLL_OK)
        return st;
    debug_begin();
    for (int r = 0; r < nranks; ++r) {
        const size_t all = static_cast<size_t>(nranks) * c;
        debug_range(in[r], all * elem_bytes(dtype), false);
        debug_range(out[r], all * elem_bytes(dtype), true);
        if (block) {
            debug_range(wire_codes[r], all, true);
            debug_range(wire_scales[r],
                        static_cast<size_t>(nranks) * blocks_of(c, block) * sizeof(float), true);
        }
    }
    return finish(launch_all_to_all(p, nranks, c, dtype, block != 0,
                                    static_cast<cudaStream_t>(stream)));
}

int lp_quantize_fmt(const void *in, lpcoll_dtype dtype, size_t n, int block,
                    lpcoll_fp8 fmt, uint8_t *codes, float *scales, void *stream)
{
    int st = check_variant(dtype, fmt, block);
    if (st != LPCOLL_OK || n == 0)
        return st;
    st = first_error({check_ptr(in), check_ptr(codes), check_ptr(scales)});
    if (st != LPCOLL_OK)
        return st;
    debug_begin();
    debug_range(in, n * elem_bytes(dtype), false);
    debug_range(codes, n, true);
    debug_range(scales, blocks_of(n, block) * sizeof(float), true);
    return finish(launch_quantize_fmt(in, dtype, n, block, fmt, codes, scales,
                                      static_cast<cudaStream_t>(stream)));
}

int lp_dequantize_fmt(const uint8_t *codes, const float *scales, size_t n, int block,
                      lpcoll_fp8 fmt, void *out, lpcoll_dtype dtype, void *stream)
{
    int st = check_variant(dtype, fmt, block);
    if (st != LPCOLL_OK || n == 0)
        return st;
    st = first_error({check_ptr(codes), check_ptr(scales), check_ptr(out)});
    if (st != LPCOLL_OK)
        return st;
    debug_begin();
    debug_range(codes, n, false);
    debug_range(scales, blocks_of(n, block) * sizeof(float), false);
    debug_range(out, n * elem_bytes(dtype), true);
    return finish(launch_dequantize_fmt(codes, scales, n, block, fmt, out, dtype,
                                        static_cast<cudaStream_t>(stream)));
}

int lp_reduce_fmt(const uint8_t *const *codes, const float *const *scales, int nranks,
                  size_t n, int block, lpcoll_fp8 fmt, void *out, lpcoll_dtype dtype,
                  void *stream)
{
    int st = check_variant(dtype, fmt, block);
    if (st == LPCOLL_OK && (nranks < 1 || nranks > LPCOLL_MAX_RANKS))
        st = LPCOLL_ERR_ARG;
    if (st != LPCOLL_OK || n == 0)
        return st;
    st = first_error({check_rank_array(codes, nranks), check_rank_array(scales, nranks),
                      check_ptr(out)});
    if (st != LPCOLL_OK)
        return st;
    ReduceParams p = {};
    debug_begin();
    for (int r = 0; r < nranks; ++r) {
        p.codes[r] = codes[r];
        p.scales[r] = scales[r];
        debug_range(codes[r], n, false);
        debug_range(scales[r], blocks_of(n, block) * sizeof(float), false);
    }
    debug_range(out, n * elem_bytes(dtype), true);
    return finish(launch_reduce_fmt(p, nranks, n, block, fmt, out, dtype,
                                    static_cast<cudaStream_t>(stream)));
}

const char *lpcoll_status_string(int status)
{
    switch (status) {
    case LPCOLL_OK: return "LPCOLL_OK";
    case LPCOLL_ERR_ARG: return "LPCOLL_ERR_ARG: invalid argument or NULL pointer";
    case LPCOLL_ERR_ALIGN: return "LPCOLL_ERR_ALIGN: device pointer not 16-byte aligned";
    case LPCOLL_ERR_UNSUPPORTED: return "LPCOLL_ERR_UNSUPPORTED: unsupported block size";
    case LPCOLL_ERR_RANK: return "LPCOLL_ERR_RANK: NULL pointer in a per-rank array";
    case LPCOLL_ERR_CUDA: return "LPCOLL_ERR_CUDA: kernel launch failed";
    default: return "LPCOLL: unknown status";
    }
}

int lpcoll_last_cuda_error(void) { return g_last_cuda_error; }

int lpcoll_debug_bounds_errors(unsigned long long *first_bad)
{
    if (first_bad != nullptr)
        *first_bad = 0;
#ifdef LPCOLL_DEBUG_BOUNDS
    const cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return -2;
    }
    DebugRecord *rec = debug_record();
    if (rec == nullptr)
        return -2;
    const int bad = rec->flag != 0 ? 1 : 0;
    if (first_bad != nullptr)
        *first_bad = rec->first_bad;
    rec->flag = 0;
    rec->first_bad = 0;
    return bad;
#else
    return -1;
#endif
}

void lpcoll_debug_bounds_shrink(size_t bytes)
{
#ifdef LPCOLL_DEBUG_BOUNDS
    g_shrink_next.store(bytes);
#else
    (void)bytes;
#endif
}

int lpcoll_version(void) { return 100; }

}  // extern "C"
