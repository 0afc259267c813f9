/*
 * lpcoll.h -- C ABI of liblpcoll.so: the data-parallel hot path of a
 * low-precision (FP8) collective reduction and of the DDA flat / tree
 * allreduce, with N ranks emulated as N buffers in one GPU's memory.
 *
 * The method is the one described on code-journey.com, "RCCLX: AMD GPU
 * communication, Meta open source" (Portuguese and Korean editions):
 *   - section "Funcionalidade Principal 1: Acesso Direto a Dados (DDA)":
 *     DDA flat (every rank reads every other rank's data directly and reduces
 *     locally) and DDA tree (reduce-scatter, then all-gather, each phase by
 *     direct access);
 *   - section "Funcionalidade Principal 2: Coletivos de Baixa Precisao":
 *     FP8 quantization of FP32 / BF16 payloads for messages of 16 MB and more,
 *     with FP32 kept for the arithmetic (feature table, rows "Tipos de Dados"
 *     and "Precisao do Calculo").
 * The pages fix neither the FP8 format nor the scaling. This library uses:
 *   - OCP E4M3 codes ("e4m3fn", largest finite 448), rounded to nearest even
 *     and saturated to +-448;
 *   - one FP32 scale per block of LPCOLL_BLOCK = 128 consecutive elements:
 *     s = a / 448 with a = max |x| over the block, codes = e4m3(x * (448 / a));
 *     a block whose 448 / a overflows (a == 0 or a < ~1.3e-36) gets s = 0 and
 *     signed-zero codes;
 *   - dequantized values fl(e4m3 * s), summed in FP32 in the fixed order rank
 *     0, 1, ..., N-1 starting from rank 0's value, no fused multiply-add;
 *   - BF16 results rounded to nearest even.
 *
 * Conventions shared by every entry point:
 *   - Every data pointer is a DEVICE pointer into memory the caller owns; the
 *     library allocates nothing, frees nothing and never synchronizes.
 *     Every device pointer must be 16-byte aligned (LPCOLL_ERR_ALIGN).
 *   - Pointer arrays (in[], out[], wire_codes[], ...) are HOST arrays of
 *     nranks device pointers; they are read during the call only.
 *   - dtype is LPCOLL_F32 (float) or LPCOLL_BF16 (bfloat16 stored as
 *     uint16); inputs and outputs of one call share it.
 *   - n is the element count per rank; any n >= 0 is accepted. A payload of
 *     n elements is codes[n] (one byte each, element order) plus
 *     scales[ceil(n / 128)] (block b covers elements [128 b, 128 b + 128)).
 *   - stream is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Work is enqueued on it and the call returns at once. Kernels
 *     are launched with programmatic dependent launch: one may be scheduled
 *     while the previous kernel of the stream still runs, but it touches no
 *     memory before that kernel has completed, so stream order holds for
 *     every buffer, also inside CUDA graph capture.
 *   - Resources: kernels of 256 threads, one warp per work item (grids
 *     grow with the message and may exceed what the GPU holds at once; no
 *     CTA ever waits on another). FP32 low-precision allreduces of 8 ranks
 *     with 1 GiB of input or more, and low-precision all-gathers of
 *     16-byte-aligned contributions, stage results in up to 46 KB of
 *     dynamic shared memory per CTA and write them with bulk (TMA) copies;
 *     every copy has completed when the kernel does.
 *   - Return value: LPCOLL_OK, or an lpcoll_status error found before any
 *     launch (nothing is enqueued then), or LPCOLL_ERR_CUDA if the launch
 *     itself failed (lpcoll_last_cuda_error() gives the cudaError_t).
 *     Checks, in order: dtype / nranks (LPCOLL_ERR_ARG), block
 *     (LPCOLL_ERR_UNSUPPORTED), n == 0 (LPCOLL_OK, nothing launched, pointers
 *     not inspected), NULL pointer (LPCOLL_ERR_RANK inside a per-rank array,
 *     else LPCOLL_ERR_ARG), misalignment (LPCOLL_ERR_ALIGN).
 *   - An output may be the very same buffer as an input (in place, as the
 *     pages' allreduce example works); any other overlap between buffers of
 *     one call is undefined.
 */
#ifndef LPCOLL_H
#define LPCOLL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { LPCOLL_F32 = 0, LPCOLL_BF16 = 1 } lpcoll_dtype;

/* FP8 formats of the *_fmt variants (the main path is E4M3). */
typedef enum { LPCOLL_E4M3 = 0, LPCOLL_E5M2 = 1 } lpcoll_fp8;

typedef enum {
    LPCOLL_OK = 0,
    LPCOLL_ERR_ARG = 1,         /* bad dtype, nranks, or a NULL pointer */
    LPCOLL_ERR_ALIGN = 2,       /* a device pointer not 16-byte aligned */
    LPCOLL_ERR_UNSUPPORTED = 3, /* block size other than 128 (or 0 where allowed) */
    LPCOLL_ERR_RANK = 4,        /* NULL entry in a per-rank pointer array */
    LPCOLL_ERR_CUDA = 5         /* the kernel launch failed */
} lpcoll_status;

#define LPCOLL_MAX_RANKS 16
#define LPCOLL_BLOCK 128

/* Quantize one rank's message into its FP8 payload (the "wire").
 * Pages: "Funcionalidade Principal 2", FP8 compression of FP32/BF16 data.
 *   in      n elements of dtype (device)
 *   block   must be 128
 *   codes   out: n bytes, codes[i] = e4m3(in[i] * 448 / a_b)   (device)
 *   scales  out: ceil(n/128) floats, scales[b] = a_b / 448      (device)   */
int lp_quantize(const void *in, lpcoll_dtype dtype, size_t n, int block,
                uint8_t *codes, float *scales, void *stream);

/* Expand one FP8 payload back to dtype: out[i] = cast(e4m3(codes[i]) * s_b).
 * Pages: the receiving side of the low-precision collectives.
 *   codes, scales   payload as written by lp_quantize (device)
 *   out             n elements of dtype (device)                           */
int lp_dequantize(const uint8_t *codes, const float *scales, size_t n,
                  int block, void *out, lpcoll_dtype dtype, void *stream);

/* Reduce nranks FP8 payloads into one output: dequantize each, sum in FP32
 * in rank order 0..nranks-1, cast to dtype.
 * Pages: "Precisao do Calculo", FP32 kept for the arithmetic.
 *   codes[r], scales[r]   payload of rank r (host array of device pointers)
 *   nranks                1..16
 *   out                   n elements of dtype (device)                     */
int lp_reduce(const uint8_t *const *codes, const float *const *scales,
              int nranks, size_t n, int block, void *out, lpcoll_dtype dtype,
              void *stream);

/* DDA flat allreduce over nranks emulated ranks, one fused launch.
 * Pages: "Funcionalidade Principal 1", bullet "Algoritmo DDA Flat".
 *   in[r]           rank r's message, n elements of dtype (device)
 *   out[r]          rank r's result, n elements of dtype (device); all nranks
 *                   outputs receive the same values; out[r] == in[r] allowed
 *   block           0: exact precision, out = cast(sum_r in[r]);
 *                   128: low precision, each rank's message is quantized into
 *                   wire_codes[r] / wire_scales[r] (written: the payload a
 *                   rank would expose to its peers) and the outputs are the
 *                   FP32 sum of the dequantized payloads
 *   wire_codes[r]   n bytes (device); ignored (may be NULL) when block == 0
 *   wire_scales[r]  ceil(n/128) floats (device); ignored when block == 0   */
int dda_flat_sim(const void *const *in, void *const *out, int nranks,
                 size_t n, lpcoll_dtype dtype, int block,
                 uint8_t *const *wire_codes, float *const *wire_scales,
                 void *stream);

/* DDA tree allreduce: reduce-scatter then all-gather, one fused launch.
 * Pages: "Funcionalidade Principal 1", bullet "Algoritmo DDA Tree".
 * Rank r owns shard r, elements [r L, min((r+1) L, n)) with
 * L = ceil(ceil(n/nranks)/128)*128, so shards are whole blocks.
 *   in, out, nranks, n, dtype, wire_codes, wire_scales   as dda_flat_sim
 *   block = 128: phase 1 quantizes each rank's message into its wire;
 *     phase 2 (reduce-scatter) sums the nranks payloads of each shard in
 *     FP32 and quantizes the reduced shard again into shard_codes (n bytes)
 *     and shard_scales (ceil(n/128) floats), indexed like the message;
 *     phase 3 (all-gather) writes the dequantized shard payload to every
 *     out[r], so outputs carry one more quantization than dda_flat_sim's.
 *   block = 0: exact precision, same result as dda_flat_sim with block 0;
 *     wire and shard pointers are ignored (may be NULL).                   */
int dda_tree_sim(const void *const *in, void *const *out, int nranks,
                 size_t n, lpcoll_dtype dtype, int block,
                 uint8_t *const *wire_codes, float *const *wire_scales,
                 uint8_t *shard_codes, float *shard_scales, void *stream);

/* Format and block-size variants of lp_quantize / lp_dequantize / lp_reduce,
 * for ablations (the pages fix neither; the main path is E4M3 with blocks of
 * 128). fmt: LPCOLL_E4M3 (largest finite 448) or LPCOLL_E5M2 (largest
 * finite 57344, Inf/NaN codes never produced: values saturate). block: 32,
 * 64, 128 or 256 elements per FP32 scale (else LPCOLL_ERR_UNSUPPORTED); a
 * payload of n elements is codes[n] plus scales[ceil(n/block)], block b
 * covering elements [b block, (b+1) block). Scale s = a / max, codes =
 * fp8(x * (max / a)), rounded to nearest even and saturated; values are
 * fl(fp8 * s), reduced in FP32 in rank order. With LPCOLL_E4M3 and block 128
 * they return exactly what the plain entry points return.                 */
int lp_quantize_fmt(const void *in, lpcoll_dtype dtype, size_t n, int block,
                    lpcoll_fp8 fmt, uint8_t *codes, float *scales, void *stream);
int lp_dequantize_fmt(const uint8_t *codes, const float *scales, size_t n,
                      int block, lpcoll_fp8 fmt, void *out, lpcoll_dtype dtype,
                      void *stream);
int lp_reduce_fmt(const uint8_t *const *codes, const float *const *scales,
                  int nranks, size_t n, int block, lpcoll_fp8 fmt, void *out,
                  lpcoll_dtype dtype, void *stream);

/* ReduceScatter over nranks emulated ranks: rank r receives shard r of the
 * sum of all ranks' messages. Pages: "Funcionalidade Principal 2", feature
 * table row "Operacoes Suportadas" (ReduceScatter).
 * Shard r is elements [r L, min((r+1) L, n)); L = ceil(n/nranks), rounded
 * up to a multiple of 128 when block = 128.
 *   in[r]       rank r's message, n elements of dtype (device)
 *   out[r]      shard r of the result, min(L, n - r L) elements (device);
 *               may be NULL when that count is <= 0
 *   block = 128: each rank's message is quantized into wire_codes[r] (n
 *               bytes) / wire_scales[r] (ceil(n/128) floats), and shard r is
 *               the FP32 sum of the dequantized payloads (rank order, cast
 *               to dtype): bit-equal to that shard of dda_flat_sim's output.
 *   block = 0:  exact FP32 sum of the inputs; wires ignored (may be NULL). */
int reduce_scatter_sim(const void *const *in, void *const *out, int nranks,
                       size_t n, lpcoll_dtype dtype, int block,
                       uint8_t *const *wire_codes, float *const *wire_scales,
                       void *stream);

/* AllGather: every rank receives all ranks' contributions in rank order.
 * Pages: "Operacoes Suportadas" (AllGather).
 *   in[r]       rank r's contribution, m elements of dtype (device)
 *   out[r]      nranks * m elements (device): out[r][q m + i] = contribution
 *               q, element i, for every r
 *   block = 128: each contribution is quantized on its own 128-element
 *               blocks into wire_codes[r] (m bytes) / wire_scales[r]
 *               (ceil(m/128) floats); every output, the sender's own
 *               included, holds the dequantized values.
 *   block = 0:  exact copies; wires ignored (may be NULL).
 * Any m works; when m * element size is not a multiple of 16 bytes the
 * outputs are written element by element (slower).                        */
int all_gather_sim(const void *const *in, void *const *out, int nranks,
                   size_t m, lpcoll_dtype dtype, int block,
                   uint8_t *const *wire_codes, float *const *wire_scales,
                   void *stream);

/* AlltoAll: rank r's message is nranks chunks of c elements, chunk j
 * addressed to rank j. Pages: "Operacoes Suportadas" (AlltoAll).
 *   in[r]       nranks * c elements of dtype (device)
 *   out[j]      nranks * c elements (device): out[j][r c + i] = chunk j of
 *               rank r, element i
 *   block = 128: every chunk is quantized on its own 128-element blocks
 *               (counted from the chunk's start): chunk j of rank r has its
 *               codes at wire_codes[r] + j c (nranks * c bytes in all) and
 *               its scales at wire_scales[r] + j ceil(c/128) (nranks *
 *               ceil(c/128) floats); receivers get the dequantized values.
 *   block = 0:  exact copies; wires ignored (may be NULL).
 * Any c works; when c * element size is not a multiple of 16 bytes the data
 * moves element by element (slower).                                      */
int all_to_all_sim(const void *const *in, void *const *out, int nranks,
                   size_t c, lpcoll_dtype dtype, int block,
                   uint8_t *const *wire_codes, float *const *wire_scales,
                   void *stream);

/* Allreduce of nranks messages that live in HOST memory, through a device
 * workspace the caller provides: the flat and / or tree allreduce of
 * dda_flat_sim / dda_tree_sim (same results, bit for bit), run chunk by
 * chunk with host->device copies, kernels and device->host copies of
 * different chunks overlapped. Pages: the allreduce of "Funcionalidade
 * Principal 1" fed from and returned to host memory.
 *   host_in[r]        rank r's message, n elements of dtype (host)
 *   host_out_flat[r]  n elements (host) receiving the flat allreduce, or the
 *                     whole array NULL to skip it
 *   host_out_tree[r]  the same for the tree allreduce; at least one of the
 *                     two arrays must be given
 *   block             0 (exact) or 128 (low precision)
 *   chunk             elements per chunk, a positive multiple of 128
 *   slots             chunks in flight, 1..8 (2 or more to overlap)
 *   workspace         device memory of workspace_bytes >=
 *                     lpcoll_host_workspace_bytes(...), 256-byte aligned;
 *                     its contents are scratch
 *   copy_in_stream, compute_stream, copy_out_stream   cudaStream_t as void*
 *                     (three distinct streams overlap; NULL serializes)
 * Host buffers should be pinned (page-locked) for the copies to overlap.
 * The call returns when every result is in host memory (it synchronizes
 * copy_out_stream). Errors: LPCOLL_ERR_ARG (dtype, nranks, slots, chunk,
 * workspace NULL or too small, no output), LPCOLL_ERR_UNSUPPORTED (block),
 * LPCOLL_ERR_RANK (NULL per-rank pointer), LPCOLL_ERR_ALIGN (workspace),
 * LPCOLL_ERR_CUDA (a copy, launch or event failed). After LPCOLL_ERR_CUDA
 * the call has still waited for all three streams, so nothing it queued
 * reads host_in or writes the outputs or the workspace any more: the caller
 * may free or reuse them at once (the outputs' contents are undefined).   */
size_t lpcoll_host_workspace_bytes(int nranks, size_t chunk, lpcoll_dtype dtype,
                                   int block, int flat, int tree, int slots);
int lpcoll_host_allreduce(const void *const *host_in, void *const *host_out_flat,
                          void *const *host_out_tree, int nranks, size_t n,
                          lpcoll_dtype dtype, int block, size_t chunk, int slots,
                          void *workspace, size_t workspace_bytes,
                          void *copy_in_stream, void *compute_stream,
                          void *copy_out_stream);

/* Test hook for the error path of lpcoll_host_allreduce; not part of the
 * method. The next call of lpcoll_host_allreduce that passes its argument
 * checks treats its enqueue step number `step` (0 = the first copy, event
 * record or wait, or launch it would queue, in queue order) as failed
 * without calling CUDA for it: the steps before it are queued as usual, none
 * after it, and the call returns LPCOLL_ERR_CUDA with
 * lpcoll_last_cuda_error() == cudaErrorInvalidValue. The hook then disarms
 * itself; a negative step disarms it at once. It lets a test drive the
 * error return with no failing GPU call.                                   */
void lpcoll_debug_fail_host_enqueue(long step);

/* dda_flat_sim with block = 128 for callers that cannot allocate device
 * memory. The pages have no counterpart: this exists for users of the
 * library, not for the method. Some callers cannot provide the wire buffers
 * that dda_flat_sim needs as scratch, for instance a plugin running inside a
 * host framework that owns all device memory, or a latency-critical loop
 * that must never call cudaMalloc (which can synchronize the device). This
 * call keeps every rank's FP8 wire payload in a fixed array inside the
 * library's device image and allocates nothing; it gives the same outputs as
 * dda_flat_sim with block = 128.
 *   in, out, nranks, n, dtype, stream   as dda_flat_sim; the caller still
 *                                       owns and passes inputs and outputs
 *   limit    nranks * ceil(n / 256) * 256 <= LPCOLL_NOALLOC_MAX_ELEMS
 *            (64 Mi elements over all ranks, e.g. 8 ranks of 8 Mi elements,
 *            a 16 MiB BF16 message); larger calls return LPCOLL_ERR_ARG and
 *            launch nothing.
 *   memory   every GPU on which the library's kernels are loaded holds the
 *            array (about 66 MiB) until the process exits. The first call
 *            with a device current looks up the array's device address on
 *            that device (cudaGetSymbolAddress) and keeps it for the life
 *            of the process; make that first call before any stream capture,
 *            and do not use this call across a device reset
 *            (cudaDeviceReset), after which the kept address is stale.
 *   sharing  all calls share the one array and it keeps the last call's
 *            wire payload (nothing in it needs to start at zero). Calls that
 *            overlap on the GPU (different streams, or threads) race on it:
 *            their outputs stay correct, since no kernel reads the array
 *            back, but its contents are then undefined.                    */
#define LPCOLL_NOALLOC_MAX_ELEMS (64u * 1024u * 1024u)
int dda_flat_sim_noalloc(const void *const *in, void *const *out, int nranks,
                         size_t n, lpcoll_dtype dtype, void *stream);

/* Bounds checks, a test tool with no counterpart in the method. The
 * bounds-checked build of this library (liblpcoll_debug_bounds.so, compiled
 * with -DLPCOLL_DEBUG_BOUNDS) makes every entry point list the buffers its
 * call may touch, with the sizes this header gives them (inputs read-only;
 * outputs, wires and workspaces writable), and checks every global load,
 * store and bulk copy of its kernels against that list before the access.
 * An access outside the list is skipped (a skipped load reads zeros) and
 * recorded; nothing traps, so the CUDA context stays usable. That build
 * allocates one small managed record on first use, copies the buffer list
 * to the device ahead of every launch into one list per source file of the
 * library (so its calls are slower, must not be captured into a CUDA graph,
 * and must not overlap on the GPU: calls on several streams or threads at
 * once would check against each other's lists), and is for tests only.
 *
 * lpcoll_debug_bounds_errors waits for the device (cudaDeviceSynchronize)
 * and returns 1 if any access failed its check since the previous call
 * (*first_bad, when first_bad is not NULL, receives the first such
 * address), 0 if none, -2 if the device or the record failed; it then
 * clears the record. The normal build returns -1 and checks nothing.
 *
 * lpcoll_debug_bounds_shrink(bytes) makes the next call of the
 * bounds-checked build list every buffer `bytes` shorter than its real
 * size, so that the kernels' last legitimate accesses fail the check (and
 * are skipped): it shows the checks fire without any access leaving the
 * real buffers. The normal build ignores it.                              */
int lpcoll_debug_bounds_errors(unsigned long long *first_bad);
void lpcoll_debug_bounds_shrink(size_t bytes);

/* Static, NUL-terminated name of a status code (never NULL). */
const char *lpcoll_status_string(int status);

/* cudaError_t of the most recent LPCOLL_ERR_CUDA returned to this thread
 * (0 if none). */
int lpcoll_last_cuda_error(void);

/* Library ABI version: 100 * major + minor. */
int lpcoll_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LPCOLL_H */
