// lpcoll_noalloc.cu -- dda_flat_sim_noalloc: the low-precision flat
// allreduce for callers that cannot allocate device memory.
//
// dda_flat_sim needs caller-provided wire buffers (each rank's FP8 codes and
// block scales). For an allreduce caller those are scratch: nobody reads them
// afterwards. Some callers have no way to get them: code running as a plugin
// inside a host framework that owns every byte of device memory and forbids
// private allocations, or latency-critical loops that must never enter
// cudaMalloc (which can synchronize the whole device). This entry point keeps
// the wire in a fixed-size array that lives in the library's own device
// image instead, and allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU on which this
// library's kernels are loaded holds its own copy of it (about 66 MiB) until
// the process exits. Host code cannot use the array's name as a device
// address (on the host it names a host-side shadow), so the address is looked
// up once per device with cudaGetSymbolAddress, with that device current, on
// the first call made while it is current. The cached address belongs to
// the device's current context: after cudaDeviceReset (or any other
// teardown of that context) it is stale, so the library must not be used
// across a device reset.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "lpcoll.h"
#include "lpcoll_dda.cuh"

namespace {

constexpr size_t kCodeBytes = LPCOLL_NOALLOC_MAX_ELEMS;  // one byte per element
constexpr size_t kRankAlign = 256;                       // per-rank region alignment
constexpr size_t kScaleFloats =
    LPCOLL_NOALLOC_MAX_ELEMS / LPCOLL_BLOCK + LPCOLL_MAX_RANKS * (kRankAlign / 4);
constexpr size_t kScratchBytes = kCodeBytes + kScaleFloats * sizeof(float);

// codes of all ranks at [0, kCodeBytes), then the scales of all ranks
static __device__ __align__(256) unsigned char g_wire_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned char *g_scratch_ptr[kMaxDevices] = {};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Device address of the scratch array on the current device.
cudaError_t scratch_address(unsigned char **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_wire_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_ptr[dev] = static_cast<unsigned char *>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

}  // namespace

extern "C" int dda_flat_sim_noalloc(const void *const *in, void *const *out,
                                    int nranks, size_t n, lpcoll_dtype dtype,
                                    void *stream)
{
    if ((dtype != LPCOLL_F32 && dtype != LPCOLL_BF16) || nranks < 1 ||
        nranks > LPCOLL_MAX_RANKS)
        return LPCOLL_ERR_ARG;
    if (n == 0)
        return LPCOLL_OK;
    const size_t code_stride = round_up(n, kRankAlign);
    if (n > LPCOLL_NOALLOC_MAX_ELEMS ||
        code_stride * static_cast<size_t>(nranks) > LPCOLL_NOALLOC_MAX_ELEMS)
        return LPCOLL_ERR_ARG;  // message too large for the fixed scratch
    if (in == nullptr || out == nullptr)
        return LPCOLL_ERR_ARG;
    for (int r = 0; r < nranks; ++r)
        if (in[r] == nullptr || out[r] == nullptr)
            return LPCOLL_ERR_RANK;
    for (int r = 0; r < nranks; ++r)
        if (misaligned(in[r]) || misaligned(out[r]))
            return LPCOLL_ERR_ALIGN;

    unsigned char *base = nullptr;
    cudaError_t e = scratch_address(&base);
    if (e != cudaSuccess) {
        cudaGetLastError();
        lpc::record_cuda_error(e);
        return LPCOLL_ERR_CUDA;
    }
    const size_t scale_stride = round_up((n + LPCOLL_BLOCK - 1) / LPCOLL_BLOCK,
                                         kRankAlign / sizeof(float));
    float *scales = reinterpret_cast<float *>(base + kCodeBytes);

    lpc::DdaParams p = {};
    const size_t es = dtype == LPCOLL_F32 ? 4 : 2;
    lpc::debug_begin();
    lpc::debug_range(base, kScratchBytes, true);
    for (int r = 0; r < nranks; ++r) {
        p.in[r] = in[r];
        p.out[r] = out[r];
        p.codes[r] = base + static_cast<size_t>(r) * code_stride;
        p.scales[r] = scales + static_cast<size_t>(r) * scale_stride;
        lpc::debug_range(in[r], n * es, false);
        lpc::debug_range(out[r], n * es, true);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = dtype == LPCOLL_F32 ? lpc::launch_dda_f32(p, nranks, n, lpc::kFlat, s)
                            : lpc::launch_dda_bf16(p, nranks, n, lpc::kFlat, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        lpc::record_cuda_error(e);
        return LPCOLL_ERR_CUDA;
    }
    return LPCOLL_OK;
}
