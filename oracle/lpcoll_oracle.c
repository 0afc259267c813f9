/*
 * lpcoll_oracle.c -- CPU oracle for the low-precision (FP8) collective
 * reduction and the DDA flat / tree allreduce, with N ranks held as N
 * separate host buffers.
 *
 * TEST INFRASTRUCTURE. This file is the correctness reference that the tests
 * and the benchmark's CPU-baseline leg compare the CUDA library against. It is
 * plain, slow, single-threaded C, written step by step from the method as the
 * pages describe it, and it shares no code, header or table with the CUDA
 * library. Nothing in the library may call it.
 *
 * Build with -O2 -ffp-contract=off and never -ffast-math: every floating-point
 * step below is one IEEE-754 binary32 operation rounded to nearest-even, and a
 * fused multiply-add would change the results.
 *
 * Sources (the pages this follows; all three describe Meta's RCCLX):
 *   [CJ] code-journey.com "RCCLX: AMD GPU communication, Meta open source"
 *        (Portuguese edition; the Korean edition is a near-verbatim twin).
 *        Sections used:
 *        "Funcionalidade Principal 1: Acesso Direto a Dados (DDA)",
 *           bullets "Algoritmo DDA Flat" and "Algoritmo DDA Tree";
 *        "Funcionalidade Principal 2: Coletivos de Baixa Precisao",
 *           the paragraph on FP8 compression of >= 16 MB messages and the
 *           feature table rows "Tipos de Dados" (FP32, BF16 via FP8),
 *           "Precisao do Calculo" (FP32 kept for the arithmetic) and
 *           "Operacoes Suportadas" (AllReduce, AllGather, AlltoAll,
 *           ReduceScatter);
 *        "Guia Pratico e Perspectivas", the torch.full / allreduce(SUM)
 *           example.
 *
 * Readings where the pages are silent (each one is a choice of this library,
 * listed with its reason in the design notes):
 *   - FP8 flavour: OCP E4M3 ("e4m3fn": no infinities, NaN = S.1111.111,
 *     largest finite 448), encoded round-to-nearest-even, saturating to +-448.
 *   - Scale: one binary32 scale per block of 128 consecutive elements,
 *     s = a/448 with a = max |x| over the block; elements are encoded as
 *     e4m3(x * (448/a)), the reciprocal computed once per block.
 *   - Degenerate block (448/a is +Inf: a == 0 or a below ~1.3e-36): s = 0
 *     and every code is a signed zero.
 *   - Sum: binary32, fixed order rank 0, 1, ..., N-1, starting from rank 0's
 *     value (not from 0.0).
 *   - Every rank's own contribution is quantized too, so all N outputs agree.
 *   - Tree: the reduced shard is quantized again before the all-gather and
 *     every rank, the owner included, receives the dequantized value.
 *   - BF16 output: binary32 rounded to nearest-even on bit 16.
 *
 * Parity status: every function here is pinned by the CPU tests (exhaustive
 * codec checks against the OCP definition and an independent library
 * encoder, round-trip and error-bound invariants, brute-force FP64 bounds,
 * the closed form of the pages' torch.full example). Agreement with RCCLX's
 * own FP8 scheme is unpinned: the pages give no format, block size or
 * rounding rule for it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_UNSUPPORTED 3

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* Value of an OCP E4M3 code: sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits. Exponent field 0 holds subnormals M * 2^-9; S.1111.111 is NaN; there
 * are no infinities. Every value is exact in binary32. */
float orc_e4m3_decode(uint8_t c)
{
    int sign = c >> 7;
    int e = (c >> 3) & 15;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
    return (float)(sign ? -v : v);
}

/* Nearest E4M3 code to y, ties to the even code; finite values beyond 448 in
 * magnitude give +-448 (satfinite); NaN gives 0x7F; the sign of zero is kept.
 * y is widened to double (exact) and scaled by a power of two (exact), so the
 * one rounding is the nearbyint() in the default round-to-nearest-even mode. */
uint8_t orc_e4m3_encode(float y)
{
    uint32_t bits;
    uint8_t sign;
    double a, m;
    int k, e;

    memcpy(&bits, &y, sizeof bits);
    sign = (bits >> 31) ? 0x80 : 0x00;
    if (isnan(y))
        return 0x7F;
    a = fabs((double)y);
    if (a > 448.0)
        return sign | 0x7E;
    if (a < 0x1p-6) {
        /* subnormal spacing 2^-9; m == 8 lands on the smallest normal, whose
         * code (exponent 1, mantissa 0) is also 8. */
        m = nearbyint(a * 0x1p9);
        return sign | (uint8_t)m;
    }
    frexp(a, &k);       /* a = f * 2^k with f in [0.5, 1) */
    e = k - 1;          /* unbiased exponent, -6 .. 8 */
    m = nearbyint(ldexp(a, 3 - e)); /* 8 .. 16: implicit bit + 3 fraction bits */
    if (m == 16.0) {
        e += 1;
        m = 8.0;
    }
    return sign | (uint8_t)(((e + 7) << 3) | ((int)m - 8));
}

/* Value of an OCP E5M2 code: sign bit, 5 exponent bits (bias 15), 2 mantissa
 * bits. Exponent field 0 holds subnormals M * 2^-16; exponent field 31 holds
 * +-Inf (M = 0) and NaN (M != 0). Every value is exact in binary32. */
float orc_e5m2_decode(uint8_t c)
{
    int sign = c >> 7;
    int e = (c >> 2) & 31;
    int m = c & 3;
    double v;
    if (e == 31)
        return m ? NAN : (sign ? -INFINITY : INFINITY);
    if (e == 0)
        v = ldexp((double)m, -16);
    else
        v = ldexp((double)(4 + m), e - 17); /* (1 + m/4) * 2^(e-15) */
    return (float)(sign ? -v : v);
}

/* Nearest E5M2 code to y, ties to the even code; magnitudes beyond the
 * largest finite value 57344 (Inf included) give +-57344 (satfinite); NaN
 * gives 0x7F; the sign of zero is kept. Same one-rounding construction as
 * the E4M3 encoder. */
uint8_t orc_e5m2_encode(float y)
{
    uint32_t bits;
    uint8_t sign;
    double a, m;
    int k, e;

    memcpy(&bits, &y, sizeof bits);
    sign = (bits >> 31) ? 0x80 : 0x00;
    if (isnan(y))
        return 0x7F;
    a = fabs((double)y);
    if (a > 57344.0)
        return sign | 0x7B;
    if (a < 0x1p-14) {
        /* subnormal spacing 2^-16; m == 4 is the smallest normal (code 4) */
        m = nearbyint(a * 0x1p16);
        return sign | (uint8_t)m;
    }
    frexp(a, &k);
    e = k - 1;                      /* -14 .. 15 */
    m = nearbyint(ldexp(a, 2 - e)); /* 4 .. 8 */
    if (m == 8.0) {
        e += 1;
        m = 4.0;
    }
    return sign | (uint8_t)(((e + 15) << 2) | ((int)m - 4));
}

float orc_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even (on bit 16). */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(f))
        return (uint16_t)((u >> 16) | 0x0040);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float load_elem(const void *buf, int dtype, size_t i)
{
    if (dtype == ORC_F32)
        return ((const float *)buf)[i];
    return orc_bf16_to_f32(((const uint16_t *)buf)[i]);
}

static void store_elem(void *buf, int dtype, size_t i, float v)
{
    if (dtype == ORC_F32)
        ((float *)buf)[i] = v;
    else
        ((uint16_t *)buf)[i] = orc_f32_to_bf16(v);
}

/* ------------------------------------------------------------------------ */
/* Block quantization (the FP8 payload of [CJ] "Funcionalidade Principal 2")  */
/* ------------------------------------------------------------------------ */

/* Scale of a block whose largest magnitude is amax. Writes s (kept in the
 * payload) and inv (the multiplier applied to each element). Both are single
 * IEEE divisions. */
#define ORC_E4M3 0
#define ORC_E5M2 1

/* Largest finite value of the FP8 format: the value the block maximum maps to. */
static float fp8_max(int fmt)
{
    return fmt == ORC_E5M2 ? 57344.0f : 448.0f;
}

static uint8_t fp8_encode(int fmt, float y)
{
    return fmt == ORC_E5M2 ? orc_e5m2_encode(y) : orc_e4m3_encode(y);
}

static float fp8_decode(int fmt, uint8_t c)
{
    return fmt == ORC_E5M2 ? orc_e5m2_decode(c) : orc_e4m3_decode(c);
}

/* Scale of a block whose largest magnitude is amax, for format fmt: s =
 * amax / max (kept in the payload) and inv = max / amax (the multiplier
 * applied to each element), each one IEEE division; a block whose inv
 * overflows gets s = inv = 0. */
void orc_block_scale_fmt(float amax, int fmt, float *s, float *inv)
{
    float q = fp8_max(fmt) / amax;
    if (isinf(q)) {
        *s = 0.0f;
        *inv = 0.0f;
        return;
    }
    *s = amax / fp8_max(fmt);
    *inv = q;
}

void orc_block_scale(float amax, float *s, float *inv)
{
    orc_block_scale_fmt(amax, ORC_E4M3, s, inv);
}

/* The other reading of the scale step, off by default: elements encoded as
 * fp8(x / s), one IEEE division per element, instead of fp8(x * inv). The
 * pages fix neither; this switch exists only to count how often the two
 * readings give different codes, and nothing in the default path uses it. */
static int g_divide_reading = 0;

void orc_set_divide_reading(int on)
{
    g_divide_reading = on != 0;
}

/* Quantize values v[0..len) (one block) into codes[0..len) and return s. */
static float quantize_block_fmt(const float *v, size_t len, uint8_t *codes, int fmt)
{
    float amax = 0.0f, s, inv;
    size_t i;
    for (i = 0; i < len; i++)
        amax = fmaxf(amax, fabsf(v[i]));
    orc_block_scale_fmt(amax, fmt, &s, &inv);
    for (i = 0; i < len; i++) {
        if (inv == 0.0f) {
            codes[i] = signbit(v[i]) ? 0x80 : 0x00;
        } else {
            float y = v[i] * inv;
            if (g_divide_reading)
                y = v[i] / s;
            codes[i] = fp8_encode(fmt, y);
        }
    }
    return s;
}

static float quantize_block(const float *v, size_t len, uint8_t *codes)
{
    return quantize_block_fmt(v, len, codes, ORC_E4M3);
}

static float dequant_elem_fmt(const uint8_t *codes, const float *scales,
                              int block, size_t i, int fmt)
{
    float d = fp8_decode(fmt, codes[i]);
    float s = scales[i / (size_t)block];
    return d * s;
}

static float dequant_elem(const uint8_t *codes, const float *scales,
                          int block, size_t i)
{
    return dequant_elem_fmt(codes, scales, block, i, ORC_E4M3);
}

static int check_block(int block)
{
    return block == 128 ? ORC_OK : ORC_ERR_UNSUPPORTED;
}

/* Block sizes of the format / block-size variants. */
static int check_block_variant(int block)
{
    return (block == 32 || block == 64 || block == 128 || block == 256)
               ? ORC_OK : ORC_ERR_UNSUPPORTED;
}

static int check_dtype(int dtype)
{
    return (dtype == ORC_F32 || dtype == ORC_BF16) ? ORC_OK : ORC_ERR_ARG;
}

/* One rank's payload: codes[n] and scales[ceil(n/block)]. */
int orc_quantize(const void *in, int dtype, size_t n, int block,
                 uint8_t *codes, float *scales)
{
    float buf[128];
    size_t b, nb, lo, len, i;
    if (check_dtype(dtype) || check_block(block))
        return check_dtype(dtype) ? ORC_ERR_ARG : ORC_ERR_UNSUPPORTED;
    nb = (n + (size_t)block - 1) / (size_t)block;
    for (b = 0; b < nb; b++) {
        lo = b * (size_t)block;
        len = (n - lo < (size_t)block) ? n - lo : (size_t)block;
        for (i = 0; i < len; i++)
            buf[i] = load_elem(in, dtype, lo + i);
        scales[b] = quantize_block(buf, len, codes + lo);
    }
    return ORC_OK;
}

int orc_dequantize(const uint8_t *codes, const float *scales, size_t n,
                   int block, void *out, int dtype)
{
    size_t i;
    if (check_dtype(dtype) || check_block(block))
        return check_dtype(dtype) ? ORC_ERR_ARG : ORC_ERR_UNSUPPORTED;
    for (i = 0; i < n; i++)
        store_elem(out, dtype, i, dequant_elem(codes, scales, block, i));
    return ORC_OK;
}

/* Dequantize N payloads and sum them in binary32, rank 0 first, then ranks
 * 1..N-1 in order ("Precisao do Calculo": FP32 kept for the arithmetic). */
int orc_reduce(const uint8_t *const *codes, const float *const *scales,
               int nranks, size_t n, int block, void *out, int dtype)
{
    size_t i;
    int r;
    if (nranks < 1 || check_dtype(dtype) || check_block(block))
        return (nranks < 1 || check_dtype(dtype)) ? ORC_ERR_ARG
                                                  : ORC_ERR_UNSUPPORTED;
    for (i = 0; i < n; i++) {
        float sum = dequant_elem(codes[0], scales[0], block, i);
        for (r = 1; r < nranks; r++)
            sum = sum + dequant_elem(codes[r], scales[r], block, i);
        store_elem(out, dtype, i, sum);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* DDA flat allreduce ([CJ] "Algoritmo DDA Flat"): every rank reads the data */
/* of all ranks directly and reduces it locally into its own output.         */
/* ------------------------------------------------------------------------ */

/* block == 0: exact precision, the widened inputs summed in fixed order.
 * block == 128: low precision; each rank first publishes its FP8 payload in
 * wire_codes[r] / wire_scales[r], then every rank reduces the N payloads. */
int orc_flat(const void *const *in, void *const *out, int nranks, size_t n,
             int dtype, int block, uint8_t *const *wire_codes,
             float *const *wire_scales)
{
    int r, dst, st;
    size_t i;
    if (nranks < 1 || check_dtype(dtype))
        return ORC_ERR_ARG;
    if (block == 0) {
        for (dst = 0; dst < nranks; dst++) {
            for (i = 0; i < n; i++) {
                float sum = load_elem(in[0], dtype, i);
                for (r = 1; r < nranks; r++)
                    sum = sum + load_elem(in[r], dtype, i);
                store_elem(out[dst], dtype, i, sum);
            }
        }
        return ORC_OK;
    }
    if (check_block(block))
        return ORC_ERR_UNSUPPORTED;
    /* each rank publishes its own payload */
    for (r = 0; r < nranks; r++) {
        st = orc_quantize(in[r], dtype, n, block, wire_codes[r], wire_scales[r]);
        if (st)
            return st;
    }
    /* each rank reads all payloads and reduces locally */
    for (dst = 0; dst < nranks; dst++) {
        st = orc_reduce((const uint8_t *const *)wire_codes,
                        (const float *const *)wire_scales, nranks, n, block,
                        out[dst], dtype);
        if (st)
            return st;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* DDA tree allreduce ([CJ] "Algoritmo DDA Tree"): reduce-scatter, then      */
/* all-gather, each phase by direct access to the other ranks' data.         */
/* ------------------------------------------------------------------------ */

/* Shard r is elements [r*len, min((r+1)*len, n)) with len = ceil(n/N)
 * rounded up to a whole number of blocks (whole elements when block == 0). */
size_t orc_shard_len(size_t n, int nranks, int block)
{
    size_t per = (n + (size_t)nranks - 1) / (size_t)nranks;
    if (block > 0)
        per = (per + (size_t)block - 1) / (size_t)block * (size_t)block;
    return per;
}

/* block == 128: phase 1, each rank publishes its FP8 payload (wire_codes[r],
 * wire_scales[r]); phase 2 (reduce-scatter), rank r sums shard r of all N
 * payloads and quantizes the result again into the shard payload
 * (shard_codes / shard_scales, indexed like the input: element i, block
 * i/128); phase 3 (all-gather), every rank dequantizes every shard payload
 * into its output. block == 0: the same two phases without quantization. */
int orc_tree(const void *const *in, void *const *out, int nranks, size_t n,
             int dtype, int block, uint8_t *const *wire_codes,
             float *const *wire_scales, uint8_t *shard_codes,
             float *shard_scales)
{
    size_t per, lo, hi, b0, i, len;
    int r, owner, dst, st;
    float *reduced;

    if (nranks < 1 || check_dtype(dtype))
        return ORC_ERR_ARG;
    if (block != 0 && check_block(block))
        return ORC_ERR_UNSUPPORTED;
    if (n == 0)
        return ORC_OK;
    reduced = (float *)malloc(n * sizeof(float));
    if (!reduced)
        return ORC_ERR_ARG;
    per = orc_shard_len(n, nranks, block);

    if (block == 0) {
        /* reduce-scatter: owner sums its shard of every rank's input */
        for (owner = 0; owner < nranks; owner++) {
            lo = (size_t)owner * per;
            hi = lo + per < n ? lo + per : n;
            for (i = lo; i < hi; i++) {
                float sum = load_elem(in[0], dtype, i);
                for (r = 1; r < nranks; r++)
                    sum = sum + load_elem(in[r], dtype, i);
                reduced[i] = sum;
            }
        }
        /* all-gather: every rank copies every owner's shard */
        for (dst = 0; dst < nranks; dst++)
            for (i = 0; i < n; i++)
                store_elem(out[dst], dtype, i, reduced[i]);
        free(reduced);
        return ORC_OK;
    }

    /* phase 1: publish */
    for (r = 0; r < nranks; r++) {
        st = orc_quantize(in[r], dtype, n, block, wire_codes[r], wire_scales[r]);
        if (st) {
            free(reduced);
            return st;
        }
    }
    /* phase 2: reduce-scatter with requantization of each reduced shard */
    for (owner = 0; owner < nranks; owner++) {
        lo = (size_t)owner * per;
        hi = lo + per < n ? lo + per : n;
        for (i = lo; i < hi; i++) {
            float sum = dequant_elem(wire_codes[0], wire_scales[0], block, i);
            for (r = 1; r < nranks; r++)
                sum = sum + dequant_elem(wire_codes[r], wire_scales[r], block, i);
            reduced[i] = sum;
        }
        for (b0 = lo; b0 < hi; b0 += (size_t)block) {
            len = hi - b0 < (size_t)block ? hi - b0 : (size_t)block;
            shard_scales[b0 / (size_t)block] =
                quantize_block(reduced + b0, len, shard_codes + b0);
        }
    }
    /* phase 3: all-gather of the shard payloads */
    for (dst = 0; dst < nranks; dst++)
        for (i = 0; i < n; i++)
            store_elem(out[dst], dtype, i,
                       dequant_elem(shard_codes, shard_scales, block, i));
    free(reduced);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* The other low-precision collectives of [CJ] "Funcionalidade Principal 2", */
/* feature table row "Operacoes Suportadas": ReduceScatter, AllGather,       */
/* AlltoAll. Each rank publishes the FP8 payload of what it sends; the       */
/* receivers dequantize it.                                                  */
/* ------------------------------------------------------------------------ */

static size_t elem_size(int dtype) { return dtype == ORC_F32 ? 4 : 2; }

static const void *elem_ptr(const void *buf, int dtype, size_t i)
{
    return (const char *)buf + i * elem_size(dtype);
}

/* ReduceScatter: rank r ends with shard r (as defined by orc_shard_len) of
 * the sum over ranks. block == 128: every rank first publishes its payload
 * (wire_codes[r], wire_scales[r]); owner r then sums shard r of the N
 * dequantized payloads in rank order. block == 0: the inputs are summed
 * exactly. out[r] receives the min(L, n - rL) elements of shard r. */
int orc_reduce_scatter(const void *const *in, void *const *out, int nranks,
                       size_t n, int dtype, int block, uint8_t *const *wire_codes,
                       float *const *wire_scales)
{
    size_t per, lo, hi, i;
    int r, owner, st;
    if (nranks < 1 || check_dtype(dtype))
        return ORC_ERR_ARG;
    if (block != 0 && check_block(block))
        return ORC_ERR_UNSUPPORTED;
    if (n == 0)
        return ORC_OK;
    per = orc_shard_len(n, nranks, block);
    if (block) {
        for (r = 0; r < nranks; r++) {
            st = orc_quantize(in[r], dtype, n, block, wire_codes[r], wire_scales[r]);
            if (st)
                return st;
        }
    }
    for (owner = 0; owner < nranks; owner++) {
        lo = (size_t)owner * per;
        hi = lo + per < n ? lo + per : n;
        for (i = lo; i < hi; i++) {
            float sum;
            if (block) {
                sum = dequant_elem(wire_codes[0], wire_scales[0], block, i);
                for (r = 1; r < nranks; r++)
                    sum = sum + dequant_elem(wire_codes[r], wire_scales[r], block, i);
            } else {
                sum = load_elem(in[0], dtype, i);
                for (r = 1; r < nranks; r++)
                    sum = sum + load_elem(in[r], dtype, i);
            }
            store_elem(out[owner], dtype, i - lo, sum);
        }
    }
    return ORC_OK;
}

/* AllGather: rank r contributes m elements; every rank receives all N
 * contributions in rank order, out[d][r*m + i] = contribution r, element i.
 * block == 128: each rank publishes its contribution's payload (blocks
 * counted from the start of the contribution) and the receivers dequantize
 * it, so rank r's own copy is the dequantized value too. block == 0: exact
 * copies. */
int orc_all_gather(const void *const *in, void *const *out, int nranks, size_t m,
                   int dtype, int block, uint8_t *const *wire_codes,
                   float *const *wire_scales)
{
    size_t i;
    int r, dst, st;
    if (nranks < 1 || check_dtype(dtype))
        return ORC_ERR_ARG;
    if (block != 0 && check_block(block))
        return ORC_ERR_UNSUPPORTED;
    if (m == 0)
        return ORC_OK;
    if (block) {
        for (r = 0; r < nranks; r++) {
            st = orc_quantize(in[r], dtype, m, block, wire_codes[r], wire_scales[r]);
            if (st)
                return st;
        }
    }
    for (dst = 0; dst < nranks; dst++)
        for (r = 0; r < nranks; r++)
            for (i = 0; i < m; i++) {
                float v = block ? dequant_elem(wire_codes[r], wire_scales[r], block, i)
                                : load_elem(in[r], dtype, i);
                store_elem(out[dst], dtype, (size_t)r * m + i, v);
            }
    return ORC_OK;
}

/* AlltoAll: rank r's input is N chunks of c elements, chunk j addressed to
 * rank j; rank j's output holds the chunks it received in sender order,
 * out[j][r*c + i] = chunk j of rank r, element i. block == 128: rank r
 * publishes one payload per destination chunk (blocks counted from the start
 * of each chunk; chunk j's codes at wire_codes[r] + j*c, its scales at
 * wire_scales[r] + j*ceil(c/128)) and the receivers dequantize them.
 * block == 0: exact copies. */
int orc_all_to_all(const void *const *in, void *const *out, int nranks, size_t c,
                   int dtype, int block, uint8_t *const *wire_codes,
                   float *const *wire_scales)
{
    size_t i, nbc;
    int r, j, st;
    if (nranks < 1 || check_dtype(dtype))
        return ORC_ERR_ARG;
    if (block != 0 && check_block(block))
        return ORC_ERR_UNSUPPORTED;
    if (c == 0)
        return ORC_OK;
    nbc = block ? (c + (size_t)block - 1) / (size_t)block : 0;
    if (block) {
        for (r = 0; r < nranks; r++)
            for (j = 0; j < nranks; j++) {
                st = orc_quantize(elem_ptr(in[r], dtype, (size_t)j * c), dtype, c, block,
                                  wire_codes[r] + (size_t)j * c,
                                  wire_scales[r] + (size_t)j * nbc);
                if (st)
                    return st;
            }
    }
    for (j = 0; j < nranks; j++)
        for (r = 0; r < nranks; r++)
            for (i = 0; i < c; i++) {
                float v = block ? dequant_elem(wire_codes[r] + (size_t)j * c,
                                               wire_scales[r] + (size_t)j * nbc, block, i)
                                : load_elem(in[r], dtype, (size_t)j * c + i);
                store_elem(out[j], dtype, (size_t)r * c + i, v);
            }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Format and block-size variants of the staged building blocks (an          */
/* ablation: the pages fix neither the FP8 format nor the block). fmt is     */
/* ORC_E4M3 or ORC_E5M2; block is 32, 64, 128 or 256. With fmt = ORC_E4M3     */
/* and block = 128 they equal orc_quantize / orc_dequantize / orc_reduce.    */
/* ------------------------------------------------------------------------ */

int orc_quantize_fmt(const void *in, int dtype, size_t n, int block, int fmt,
                     uint8_t *codes, float *scales)
{
    float buf[256];
    size_t b, nb, lo, len, i;
    if (check_dtype(dtype) || (fmt != ORC_E4M3 && fmt != ORC_E5M2))
        return ORC_ERR_ARG;
    if (check_block_variant(block))
        return ORC_ERR_UNSUPPORTED;
    nb = (n + (size_t)block - 1) / (size_t)block;
    for (b = 0; b < nb; b++) {
        lo = b * (size_t)block;
        len = (n - lo < (size_t)block) ? n - lo : (size_t)block;
        for (i = 0; i < len; i++)
            buf[i] = load_elem(in, dtype, lo + i);
        scales[b] = quantize_block_fmt(buf, len, codes + lo, fmt);
    }
    return ORC_OK;
}

int orc_dequantize_fmt(const uint8_t *codes, const float *scales, size_t n,
                       int block, int fmt, void *out, int dtype)
{
    size_t i;
    if (check_dtype(dtype) || (fmt != ORC_E4M3 && fmt != ORC_E5M2))
        return ORC_ERR_ARG;
    if (check_block_variant(block))
        return ORC_ERR_UNSUPPORTED;
    for (i = 0; i < n; i++)
        store_elem(out, dtype, i, dequant_elem_fmt(codes, scales, block, i, fmt));
    return ORC_OK;
}

int orc_reduce_fmt(const uint8_t *const *codes, const float *const *scales,
                   int nranks, size_t n, int block, int fmt, void *out, int dtype)
{
    size_t i;
    int r;
    if (nranks < 1 || check_dtype(dtype) || (fmt != ORC_E4M3 && fmt != ORC_E5M2))
        return ORC_ERR_ARG;
    if (check_block_variant(block))
        return ORC_ERR_UNSUPPORTED;
    for (i = 0; i < n; i++) {
        float sum = dequant_elem_fmt(codes[0], scales[0], block, i, fmt);
        for (r = 1; r < nranks; r++)
            sum = sum + dequant_elem_fmt(codes[r], scales[r], block, i, fmt);
        store_elem(out, dtype, i, sum);
    }
    return ORC_OK;
}
