// lpcoll_host.cu -- lpcoll_host_allreduce: the allreduce of N rank messages
// that live in host memory, pipelined through a caller-provided device
// workspace.
//
// Every stage of the emulated collective works on independent 128-element
// blocks, so a message can be processed in chunks whose boundaries are
// multiples of 128 elements with the same results as one launch over the
// whole message. The workspace holds `slots` chunk slots (inputs, outputs,
// wires); chunk k goes through slot k % slots on three streams:
//
//   copy-in stream:  N host->device copies of chunk k (one cudaMemcpyAsync
//                    per rank), after the slot's previous results have left;
//   compute stream:  the flat and / or tree allreduce kernels on the slot;
//   copy-out stream: N device->host copies of every requested result.
//
// Events order the three stages of a chunk, so copies in both directions and
// the kernels of neighbouring chunks overlap. The call returns once the last
// result has reached host memory.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <initializer_list>
#include <vector>

#include "lpcoll.h"
#include "lpcoll_dda.cuh"

namespace lpc {
namespace {

constexpr size_t kAlign = 256;  // every sub-buffer of a slot starts 256-aligned
constexpr int kMaxSlots = 8;

// Test hook (lpcoll_debug_fail_host_enqueue): the index of the enqueue step
// of the next lpcoll_host_allreduce call that reports an error instead of
// calling CUDA, or -1.
std::atomic<long> g_fail_step{-1};

// Error code that an injected failure reports.
constexpr cudaError_t kInjectedError = cudaErrorInvalidValue;

// The enqueue steps of one call (copies, event records and waits, launches),
// counted so that a test can make the k-th one fail on the host.
struct Steps {
    long next = 0;
    long fail_at;
    Steps() : fail_at(g_fail_step.exchange(-1)) {}
    template <class F>
    void run(cudaError_t &e, F &&f)
    {
        if (e != cudaSuccess)
            return;
        e = (next++ == fail_at) ? kInjectedError : f();
    }
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Byte layout of one slot for a chunk of `chunk` elements.
struct SlotLayout {
    size_t in, out, codes, scales, bytes;  // per-rank strides and slot size
    bool flat, tree;
};

SlotLayout slot_layout(int nranks, size_t chunk, int dtype, int block, bool flat,
                       bool tree)
{
    SlotLayout L = {};
    const size_t es = dtype == LPCOLL_F32 ? 4 : 2;
    L.flat = flat;
    L.tree = tree;
    L.in = round_up(chunk * es, kAlign);
    L.out = L.in;
    L.codes = block ? round_up(chunk, kAlign) : 0;
    L.scales = block ? round_up((chunk + LPCOLL_BLOCK - 1) / LPCOLL_BLOCK * 4, kAlign) : 0;
    const size_t per_rank =
        L.in + L.out * ((flat ? 1 : 0) + (tree ? 1 : 0)) + L.codes + L.scales;
    L.bytes = per_rank * static_cast<size_t>(nranks) +
              ((block && tree) ? L.codes + L.scales : 0);
    return L;
}

struct Slot {
    char *in[LPCOLL_MAX_RANKS];
    char *out_flat[LPCOLL_MAX_RANKS];
    char *out_tree[LPCOLL_MAX_RANKS];
    uint8_t *codes[LPCOLL_MAX_RANKS];
    float *scales[LPCOLL_MAX_RANKS];
    uint8_t *shard_codes;
    float *shard_scales;
    cudaEvent_t in_done, computed, out_done;
    bool used;
};

void carve(Slot &s, char *base, const SlotLayout &L, int nranks, int block)
{
    char *p = base;
    for (int r = 0; r < nranks; ++r) {
        s.in[r] = p;
        p += L.in;
        s.out_flat[r] = L.flat ? p : nullptr;
        p += L.flat ? L.out : 0;
        s.out_tree[r] = L.tree ? p : nullptr;
        p += L.tree ? L.out : 0;
        s.codes[r] = block ? reinterpret_cast<uint8_t *>(p) : nullptr;
        p += L.codes;
        s.scales[r] = block ? reinterpret_cast<float *>(p) : nullptr;
        p += L.scales;
    }
    s.shard_codes = (block && L.tree) ? reinterpret_cast<uint8_t *>(p) : nullptr;
    p += (block && L.tree) ? L.codes : 0;
    s.shard_scales = (block && L.tree) ? reinterpret_cast<float *>(p) : nullptr;
}

cudaError_t launch_chunk(const Slot &s, bool tree, int nranks, size_t m, int dtype,
                         int block, cudaStream_t st)
{
    DdaParams p = {};
    for (int r = 0; r < nranks; ++r) {
        p.in[r] = s.in[r];
        p.out[r] = tree ? s.out_tree[r] : s.out_flat[r];
        p.codes[r] = s.codes[r];
        p.scales[r] = s.scales[r];
    }
    p.shard_codes = tree ? s.shard_codes : nullptr;
    p.shard_scales = tree ? s.shard_scales : nullptr;
    const int mode = !block ? kExact : (tree ? kTree : kFlat);
    return dtype == LPCOLL_F32 ? launch_dda_f32(p, nranks, m, mode, st)
                               : launch_dda_bf16(p, nranks, m, mode, st);
}

}  // namespace
}  // namespace lpc

using namespace lpc;

extern "C" void lpcoll_debug_fail_host_enqueue(long step)
{
    g_fail_step.store(step < 0 ? -1 : step);
}

extern "C" size_t lpcoll_host_workspace_bytes(int nranks, size_t chunk, lpcoll_dtype dtype,
                                              int block, int flat, int tree, int slots)
{
    if (nranks < 1 || nranks > LPCOLL_MAX_RANKS || chunk == 0 || slots < 1 ||
        (dtype != LPCOLL_F32 && dtype != LPCOLL_BF16))
        return 0;
    const size_t c = round_up(chunk, LPCOLL_BLOCK);
    return slot_layout(nranks, c, dtype, block, flat != 0, tree != 0).bytes *
           static_cast<size_t>(slots);
}

extern "C" int lpcoll_host_allreduce(const void *const *host_in, void *const *host_out_flat,
                                     void *const *host_out_tree, int nranks, size_t n,
                                     lpcoll_dtype dtype, int block, size_t chunk, int slots,
                                     void *workspace, size_t workspace_bytes,
                                     void *copy_in_stream, void *compute_stream,
                                     void *copy_out_stream)
{
    if ((dtype != LPCOLL_F32 && dtype != LPCOLL_BF16) || nranks < 1 ||
        nranks > LPCOLL_MAX_RANKS || slots < 1 || slots > kMaxSlots)
        return LPCOLL_ERR_ARG;
    if (block != 0 && block != LPCOLL_BLOCK)
        return LPCOLL_ERR_UNSUPPORTED;
    if (chunk == 0 || chunk % LPCOLL_BLOCK != 0)
        return LPCOLL_ERR_ARG;
    if (n == 0)
        return LPCOLL_OK;
    const bool flat = host_out_flat != nullptr, tree = host_out_tree != nullptr;
    if (host_in == nullptr || (!flat && !tree) || workspace == nullptr)
        return LPCOLL_ERR_ARG;
    for (int r = 0; r < nranks; ++r)
        if (host_in[r] == nullptr || (flat && host_out_flat[r] == nullptr) ||
            (tree && host_out_tree[r] == nullptr))
            return LPCOLL_ERR_RANK;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
        return LPCOLL_ERR_ALIGN;
    const SlotLayout L = slot_layout(nranks, chunk, dtype, block, flat, tree);
    if (workspace_bytes < L.bytes * static_cast<size_t>(slots))
        return LPCOLL_ERR_ARG;

    const size_t es = dtype == LPCOLL_F32 ? 4 : 2;
    cudaStream_t s_in = static_cast<cudaStream_t>(copy_in_stream);
    cudaStream_t s_cmp = static_cast<cudaStream_t>(compute_stream);
    cudaStream_t s_out = static_cast<cudaStream_t>(copy_out_stream);
    const size_t nchunks = (n + chunk - 1) / chunk;
    const int S = static_cast<int>(nchunks < static_cast<size_t>(slots) ? nchunks : slots);

    std::vector<Slot> slot(S);
    cudaError_t e = cudaSuccess;
    debug_begin();  // the kernels touch nothing but the workspace
    debug_range(workspace, workspace_bytes, true);
    for (int i = 0; i < S; ++i) {
        Slot &s = slot[i];
        carve(s, static_cast<char *>(workspace) + L.bytes * i, L, nranks, block);
        s.used = false;
        s.in_done = s.computed = s.out_done = nullptr;
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&s.in_done, cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&s.computed, cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&s.out_done, cudaEventDisableTiming);
    }

    Steps step;
    for (size_t k = 0; k < nchunks && e == cudaSuccess; ++k) {
        Slot &s = slot[k % S];
        const size_t lo = k * chunk;
        const size_t m = (n - lo < chunk) ? n - lo : chunk;
        if (s.used)
            step.run(e, [&] { return cudaStreamWaitEvent(s_in, s.out_done, 0); });
        for (int r = 0; r < nranks; ++r)
            step.run(e, [&] {
                return cudaMemcpyAsync(s.in[r], static_cast<const char *>(host_in[r]) + lo * es,
                                       m * es, cudaMemcpyHostToDevice, s_in);
            });
        step.run(e, [&] { return cudaEventRecord(s.in_done, s_in); });
        step.run(e, [&] { return cudaStreamWaitEvent(s_cmp, s.in_done, 0); });
        if (flat)
            step.run(e, [&] { return launch_chunk(s, false, nranks, m, dtype, block, s_cmp); });
        if (tree)
            step.run(e, [&] { return launch_chunk(s, true, nranks, m, dtype, block, s_cmp); });
        step.run(e, [&] { return cudaEventRecord(s.computed, s_cmp); });
        step.run(e, [&] { return cudaStreamWaitEvent(s_out, s.computed, 0); });
        for (int r = 0; r < nranks; ++r) {
            if (flat)
                step.run(e, [&] {
                    return cudaMemcpyAsync(static_cast<char *>(host_out_flat[r]) + lo * es,
                                           s.out_flat[r], m * es, cudaMemcpyDeviceToHost, s_out);
                });
            if (tree)
                step.run(e, [&] {
                    return cudaMemcpyAsync(static_cast<char *>(host_out_tree[r]) + lo * es,
                                           s.out_tree[r], m * es, cudaMemcpyDeviceToHost, s_out);
                });
        }
        step.run(e, [&] { return cudaEventRecord(s.out_done, s_out); });
        s.used = true;
    }
    // On success the results are in host memory once the copy-out stream has
    // drained. After an error, part of the pipeline may still be queued on
    // the other two streams (copies reading the caller's host inputs, kernels
    // writing the workspace): wait for all three, so that nothing this call
    // queued still touches the caller's buffers when it returns.
    const cudaError_t sync = cudaStreamSynchronize(s_out);
    if (e == cudaSuccess)
        e = sync;
    if (e != cudaSuccess) {
        cudaStreamSynchronize(s_in);
        cudaStreamSynchronize(s_cmp);
    }
    for (Slot &s : slot)
        for (cudaEvent_t ev : {s.in_done, s.computed, s.out_done})
            if (ev != nullptr)
                cudaEventDestroy(ev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        record_cuda_error(e);
        return LPCOLL_ERR_CUDA;
    }
    return LPCOLL_OK;
}
