/*
 * CPU baseline of the Q4_0 dequant-matmul: the fused fp32 loop of the C++
 * DeepSeek engine page, run on the host cores with OpenMP.
 *
 * BENCHMARK INFRASTRUCTURE.  bench.py times it next to the GPU path as the
 * CPU point of comparison.  It is neither the oracle (that is oracle/, plain
 * fp64) nor part of the CUDA product path.
 *
 * What the page describes, restated:
 *   §3.4   the dequantisation fused into the inner loop: each block's fp16
 *          scale is widened once, its nibbles are unpacked in place (low
 *          nibble = even column, high nibble = odd column), and a * (q - 8) * d
 *          is accumulated in fp32; the weights are never written out
 *          dequantised.  The scale widening goes through a table of all
 *          65536 fp16 codes, as the page does.
 *   §3.2   the loop order that streams B row by row (k outer) instead of
 *          column by column.
 *   §3.3   OpenMP with schedule(static); here over COLUMN BLOCKS, because the
 *          page's split over the rows of A gives one thread at M = 1.  Each
 *          thread owns a contiguous range of column blocks and keeps its
 *          accumulators private (no false sharing of C).
 *   §7.2   one thread per physical core (the caller passes the count).
 * The fp16 table is built from the binary16 definition (sign, 5-bit exponent
 * with bias 15, subnormals, Inf/NaN).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <omp.h>

static float g_fp16[65536];
static int g_fp16_ready = 0;

static void build_fp16_table(void)
{
    for (int h = 0; h < 65536; h++) {
        int s = (h >> 15) & 1, e = (h >> 10) & 31, f = h & 1023;
        float v;
        if (e == 0)
            v = ldexpf((float)f, -24);
        else if (e == 31)
            v = f ? NAN : INFINITY;
        else
            v = ldexpf((float)(1024 + f), e - 25);
        g_fp16[h] = s ? -v : v;
    }
    g_fp16_ready = 1;
}

/* C [M, N] = A [M, K] . W, A and C fp32 row-major, B in the block layout
 * (K rows of ceil(N/32) blocks of 18 bytes).  M <= 8. */
int q4cpu_matmul(const float *A, const uint8_t *B, float *C, int64_t M, int64_t N, int64_t K,
                 int threads)
{
    if (M < 1 || M > 8 || N < 1 || K < 1 || threads < 1)
        return -1;
    if (!g_fp16_ready)
        build_fp16_table();
    const int64_t nb = (N + 31) / 32;
#pragma omp parallel num_threads(threads)
    {
        const int t = omp_get_thread_num(), nt = omp_get_num_threads();
        /* schedule(static): a contiguous share of the column blocks */
        const int64_t b0 = nb * t / nt, b1 = nb * (t + 1) / nt;
        const int64_t w = b1 - b0;
        float *acc = (float *)calloc((size_t)(M * w * 32 > 0 ? M * w * 32 : 1), sizeof(float));
        for (int64_t k = 0; k < K; k++) {
            const uint8_t *row = B + (k * nb + b0) * 18;
            float a[8];
            for (int64_t m = 0; m < M; m++)
                a[m] = A[m * K + k];
            for (int64_t b = 0; b < w; b++) {
                const uint8_t *blk = row + b * 18;
                const float d = g_fp16[blk[0] | (blk[1] << 8)];
                /* the block's 32 codes, unpacked once: even columns from low
                 * nibbles, odd columns from high nibbles */
                float wq[32];
                for (int l = 0; l < 16; l++) {
                    const int q = blk[2 + l];
                    wq[2 * l] = (float)((q & 15) - 8);
                    wq[2 * l + 1] = (float)((q >> 4) - 8);
                }
                for (int64_t m = 0; m < M; m++) {
                    const float ad = a[m] * d;
                    float *c = acc + (m * w + b) * 32;
                    for (int l = 0; l < 32; l++)
                        c[l] += ad * wq[l];
                }
            }
        }
        for (int64_t m = 0; m < M; m++)
            for (int64_t b = 0; b < w; b++)
                for (int l = 0; l < 32; l++) {
                    const int64_t j = (b0 + b) * 32 + l;
                    if (j < N)
                        C[m * N + j] = acc[(m * w + b) * 32 + l];
                }
        free(acc);
    }
    return 0;
}
