/* A C caller of liblpcoll.so: no Python, only the CUDA runtime for memory.
 *
 * Runs the pages' usage example (code-journey.com "RCCLX: AMD GPU
 * communication, Meta open source", section "Guia Pratico e Perspectivas"):
 * rank r holds a 10 x 20 float tensor filled with r and the ranks allreduce
 * with SUM. Exact flat and tree must give N(N-1)/2 in every element of every
 * rank; the low-precision flat allreduce must give identical outputs on all
 * ranks, within 2^-4 relative of that value. Prints "ok" and exits 0 on
 * success; exits 1 with a message otherwise. */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "lpcoll.h"

#define NR 8
#define ROWS 10
#define COLS 20

static int fail(const char *what, int st)
{
    fprintf(stderr, "%s failed: %s\n", what, lpcoll_status_string(st));
    return 1;
}

int main(void)
{
    const size_t n = ROWS * COLS;
    const size_t nb = (n + LPCOLL_BLOCK - 1) / LPCOLL_BLOCK;
    float host[NR][ROWS * COLS];
    void *in[NR], *out[NR];
    uint8_t *codes[NR];
    float *scales[NR];
    const float want = NR * (NR - 1) / 2.0f;
    int r, st, lp;
    size_t i;

    for (r = 0; r < NR; ++r) {
        for (i = 0; i < n; ++i)
            host[r][i] = (float)r;
        if (cudaMalloc(&in[r], n * sizeof(float)) != cudaSuccess ||
            cudaMalloc(&out[r], n * sizeof(float)) != cudaSuccess ||
            cudaMalloc((void **)&codes[r], n) != cudaSuccess ||
            cudaMalloc((void **)&scales[r], nb * sizeof(float)) != cudaSuccess) {
            fprintf(stderr, "cudaMalloc failed\n");
            return 1;
        }
        cudaMemcpy(in[r], host[r], n * sizeof(float), cudaMemcpyHostToDevice);
    }

    for (lp = 0; lp < 3; ++lp) {
        if (lp == 0)
            st = dda_flat_sim((const void *const *)in, out, NR, n, LPCOLL_F32, 0, NULL,
                              NULL, NULL);
        else if (lp == 1)
            st = dda_tree_sim((const void *const *)in, out, NR, n, LPCOLL_F32, 0, NULL,
                              NULL, NULL, NULL, NULL);
        else
            st = dda_flat_sim((const void *const *)in, out, NR, n, LPCOLL_F32,
                              LPCOLL_BLOCK, codes, scales, NULL);
        if (st != LPCOLL_OK)
            return fail(lp == 1 ? "dda_tree_sim" : "dda_flat_sim", st);
        if (cudaDeviceSynchronize() != cudaSuccess) {
            fprintf(stderr, "kernel failed\n");
            return 1;
        }
        for (r = 0; r < NR; ++r) {
            float back[ROWS * COLS];
            cudaMemcpy(back, out[r], n * sizeof(float), cudaMemcpyDeviceToHost);
            for (i = 0; i < n; ++i) {
                const int exact_ok = back[i] == want;
                const int lp_ok = fabsf(back[i] - want) <= want / 16.0f;
                if ((lp < 2 && !exact_ok) || (lp == 2 && !lp_ok)) {
                    fprintf(stderr, "mode %d rank %d element %zu: %g, want %g\n", lp, r,
                            i, back[i], want);
                    return 1;
                }
            }
        }
    }
    /* an argument error is reported without a launch */
    st = dda_flat_sim((const void *const *)in, out, NR, n, LPCOLL_F32, 64, codes, scales,
                      NULL);
    if (st != LPCOLL_ERR_UNSUPPORTED)
        return fail("block-size check", st);
    for (r = 0; r < NR; ++r) {
        cudaFree(in[r]);
        cudaFree(out[r]);
        cudaFree(codes[r]);
        cudaFree(scales[r]);
    }
    printf("ok\n");
    return 0;
}
