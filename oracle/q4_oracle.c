/*
 * Q4_0 oracle: a plain, slow, obviously correct CPU reference of the
 * weight-only Q4_0 dequant-matmul, in fp64.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark load this library.  The CUDA product path never links,
 * imports or calls it, and it shares no code, header, table or constant with
 * the CUDA sources.
 *
 * Sources (pages of the reference material, cited by title and section):
 *   [Eng]  "用两千行 C++ 重写一个 DeepSeek 推理引擎" (C++ DeepSeek engine page)
 *          §2.2 block_q4_0 and dequantize; §2.3 row-major layout and column
 *          padding to a multiple of 32; §3.1 textbook triple loop; §3.2
 *          reordered i-k-j loop that zeroes C first; §3.4 fused dequant
 *          matmul; §7.1 little-endian files.
 *   [KT]   "KTransformers DeepSeek-V2 异构 MoE 推理…" page, «优化三» (160
 *          routed experts, 6 active per token, run as batched GEMVs) and
 *          «规则二» (gate -> top-k indices and weights -> experts).
 *
 * Everything is computed in fp64.  Each product a*w is exact in fp64 (a has
 * at most 24 significant bits, w = (q-8)*d at most 15), so the only error of
 * the oracle is the fp64 summation, at most about K*2^-53*sum|a*w|.
 *
 * Q8_0 (q4o_q8_*): [Eng §2.1-§2.2] names the format but prints no layout;
 * the reading used here is stated beside the functions.
 *
 * Pins: every function here is pinned by a CPU test against something other
 * than itself (library conversions over all 65536 codes, hand-built blocks,
 * exact rational sums, one-hot and zero cases, linearity, padding invariance,
 * closed forms of SiLU).  No function is parity-unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QO_BLOCK 32
#define QO_BLOCK_BYTES 18

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* IEEE 754 binary16 -> fp64, from the format's definition: 1 sign bit,
 * 5 exponent bits with bias 15, 10 fraction bits; exponent 0 is zero or
 * subnormal (f * 2^-24), exponent 31 is Inf (f == 0) or NaN.
 * [Eng §2.2: the block scale d is fp16, widened by fp16_to_fp32.] */
double q4o_fp16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 -> fp64: 1 sign bit, 8 exponent bits with bias 127, 7 fraction
 * bits; exponent 0 is zero or subnormal (f * 2^-133), 255 is Inf or NaN. */
double q4o_bf16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 255;
    int f = h & 127;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);   /* (1 + f/128) * 2^(e-127) */
    return sign ? -v : v;
}

/* fp64 -> bfloat16 bits, round to nearest with ties to even, from the
 * definition: keep 8 significant bits (normal range) or quantum 2^-133
 * (subnormal range); values that round to >= 2^128 become Inf. */
uint16_t q4o_f64_to_bf16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x))
        return (uint16_t)(sign | 0x7FC0);
    if (isinf(x))
        return (uint16_t)(sign | 0x7F80);
    if (a == 0.0)
        return sign;
    int e;
    double m = frexp(a, &e);              /* a = m * 2^e, m in [0.5, 1) */
    int expo = e - 1;                     /* a = 1.xxx * 2^expo */
    double quantum_exp = (expo < -126) ? -133 : (double)(expo - 7);
    double y = ldexp(a, -(int)quantum_exp);   /* a in units of the quantum */
    double fl = floor(y);
    double r = fl;
    double diff = y - fl;
    if (diff > 0.5 || (diff == 0.5 && fmod(fl, 2.0) != 0.0))
        r = fl + 1.0;
    double v = ldexp(r, (int)quantum_exp);
    if (v >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80);
    /* encode v (exact in bf16 now) */
    if (v < ldexp(1.0, -126)) {
        return (uint16_t)(sign | (uint16_t)ldexp(v, 133));   /* subnormal */
    }
    m = frexp(v, &e);
    expo = e - 1;
    int frac = (int)(ldexp(m, 8)) - 128;     /* m*256 in [128, 256) */
    return (uint16_t)(sign | (uint16_t)((expo + 127) << 7) | (uint16_t)frac);
}

/* Activation element i of a buffer of dtype 0 = fp32, 1 = bf16 bits. */
static double act_at(const void *A, int dtype, int64_t i)
{
    if (dtype == 0) {
        float f;
        memcpy(&f, (const char *)A + 4 * i, 4);
        return (double)f;
    }
    uint16_t h;
    memcpy(&h, (const char *)A + 2 * i, 2);
    return q4o_bf16_to_f64(h);
}

/* ------------------------------------------------------------------ */
/* Q4_0 block access                                                   */
/* ------------------------------------------------------------------ */

/* Scale of block (k, b): bytes 0-1 of the block, little-endian fp16
 * [Eng §2.2 struct block_q4_0; §7.1 the files are little-endian]. */
static double block_scale(const uint8_t *blk)
{
    uint16_t h = (uint16_t)(blk[0] | (blk[1] << 8));
    return q4o_fp16_to_f64(h);
}

/* Nibble l of a block: byte l/2 of qs; low nibble for even l, high nibble
 * for odd l [Eng §2.2 dequantize]. */
static int block_nibble(const uint8_t *blk, int l)
{
    uint8_t packed = blk[2 + l / 2];
    return (l % 2 == 0) ? (packed & 0x0F) : (packed >> 4);
}

/* Weight W[k, j] = (q - 8) * fp16_to_fp32(d) [Eng §2.2], where block
 * (k, j/32) sits at byte (k*nb + j/32)*18 of B: K rows, each of nb blocks
 * running along the output columns [Eng §2.3, §3.4 block = &B[k*(N/32)]]. */
static double weight_at(const uint8_t *B, int64_t nb, int64_t k, int64_t j)
{
    const uint8_t *blk = B + (k * nb + j / QO_BLOCK) * QO_BLOCK_BYTES;
    int q = block_nibble(blk, (int)(j % QO_BLOCK));
    return (double)(q - 8) * block_scale(blk);
}

/* ------------------------------------------------------------------ */
/* Dequantisation                                                      */
/* ------------------------------------------------------------------ */

/* W [K, N] fp32 = (q - 8) * d for every real column j < N [Eng §2.2].
 * (q-8)*d has at most 15 significant bits, so the fp32 value is exact. */
void q4o_dequant_f32(const uint8_t *B, int64_t K, int64_t N, float *W)
{
    int64_t nb = (N + QO_BLOCK - 1) / QO_BLOCK;
    for (int64_t k = 0; k < K; k++)
        for (int64_t j = 0; j < N; j++)
            W[k * N + j] = (float)weight_at(B, nb, k, j);
}

/* W [K, N] as bf16 bits: bf16_rn((q - 8) * d), the 16-bit tile value the
 * tensor-core path multiplies. */
void q4o_dequant_bf16(const uint8_t *B, int64_t K, int64_t N, uint16_t *W)
{
    int64_t nb = (N + QO_BLOCK - 1) / QO_BLOCK;
    for (int64_t k = 0; k < K; k++)
        for (int64_t j = 0; j < N; j++)
            W[k * N + j] = q4o_f64_to_bf16(weight_at(B, nb, k, j));
}

/* ------------------------------------------------------------------ */
/* Matmul                                                              */
/* ------------------------------------------------------------------ */

/* One output row: c[j] = sum_k a[k] * W[k, j], s[j] = sum_k |a[k] * W[k, j]|.
 * Loop order k -> block -> l, c zeroed first and overwritten: the fused
 * dequant loop of [Eng §3.4] with the zeroing of [Eng §3.2], in fp64. */
static void row_matmul(const double *a, const uint8_t *B, int64_t N, int64_t K,
                       double *c, double *s)
{
    int64_t nb = (N + QO_BLOCK - 1) / QO_BLOCK;
    for (int64_t j = 0; j < N; j++) {
        c[j] = 0.0;
        if (s)
            s[j] = 0.0;
    }
    for (int64_t k = 0; k < K; k++) {
        double av = a[k];
        const uint8_t *row = B + k * nb * QO_BLOCK_BYTES;
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *blk = row + b * QO_BLOCK_BYTES;
            double d = block_scale(blk);
            for (int l = 0; l < QO_BLOCK; l++) {
                int64_t j = b * QO_BLOCK + l;
                if (j >= N)
                    break;          /* padding column: never stored */
                int q = block_nibble(blk, l);
                double p = av * (double)(q - 8) * d;
                c[j] += p;
                if (s)
                    s[j] += fabs(p);
            }
        }
    }
}

/* c[j] = sum_k a[k] * |W[k, j]|: the first-order carry of per-row errors a[k]
 * through one matrix (used by the tolerance of the expert chain). */
static void row_matmul_abs(const double *a, const uint8_t *B, int64_t N, int64_t K,
                           double *c)
{
    int64_t nb = (N + QO_BLOCK - 1) / QO_BLOCK;
    for (int64_t j = 0; j < N; j++)
        c[j] = 0.0;
    for (int64_t k = 0; k < K; k++) {
        const uint8_t *row = B + k * nb * QO_BLOCK_BYTES;
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *blk = row + b * QO_BLOCK_BYTES;
            double d = fabs(block_scale(blk));
            for (int l = 0; l < QO_BLOCK; l++) {
                int64_t j = b * QO_BLOCK + l;
                if (j >= N)
                    break;
                c[j] += a[k] * fabs((double)(block_nibble(blk, l) - 8)) * d;
            }
        }
    }
}

/* c[j] = sum_k |a[k]| * |d_kj| * (q_kj + 8): the magnitudes of the two sums
 * the GPU's exact-dequant decode accumulates for output j, sum a*d*q and
 * 8 * sum a*d, whose difference is the product (used by the rounding bound
 * of the expert chain). */
static void row_matmul_absq(const double *a, const uint8_t *B, int64_t N, int64_t K,
                            double *c)
{
    int64_t nb = (N + QO_BLOCK - 1) / QO_BLOCK;
    for (int64_t j = 0; j < N; j++)
        c[j] = 0.0;
    for (int64_t k = 0; k < K; k++) {
        double av = fabs(a[k]);
        const uint8_t *row = B + k * nb * QO_BLOCK_BYTES;
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *blk = row + b * QO_BLOCK_BYTES;
            double d = fabs(block_scale(blk));
            for (int l = 0; l < QO_BLOCK; l++) {
                int64_t j = b * QO_BLOCK + l;
                if (j >= N)
                    break;
                c[j] += av * d * (double)(block_nibble(blk, l) + 8);
            }
        }
    }
}

/* C [M, N] = A [M, K] . W, with S [M, N] = sum_k |A[i,k] * W[k,j]| (may be
 * NULL).  A is fp32 (a_dtype 0) or bf16 bits (a_dtype 1), row-major.
 * [Eng §3.4 matmul_q4_0; C is overwritten as in §3.2.] */
void q4o_matmul(const void *A, int a_dtype, const uint8_t *B,
                int64_t M, int64_t N, int64_t K, double *C, double *S)
{
    double *a = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    for (int64_t i = 0; i < M; i++) {
        for (int64_t k = 0; k < K; k++)
            a[k] = act_at(A, a_dtype, i * K + k);
        row_matmul(a, B, N, K, C + i * N, S ? S + i * N : NULL);
    }
    free(a);
}

/* Same product by the textbook route: dequantise W first, then the i-j-k
 * triple loop of [Eng §3.1], in fp64.  A cross-check of q4o_matmul. */
void q4o_matmul_naive(const void *A, int a_dtype, const uint8_t *B,
                      int64_t M, int64_t N, int64_t K, double *C)
{
    int64_t nb = (N + QO_BLOCK - 1) / QO_BLOCK;
    double *W = (double *)malloc(sizeof(double) * (size_t)(K * N > 0 ? K * N : 1));
    for (int64_t k = 0; k < K; k++)
        for (int64_t j = 0; j < N; j++)
            W[k * N + j] = weight_at(B, nb, k, j);
    for (int64_t i = 0; i < M; i++)
        for (int64_t j = 0; j < N; j++) {
            double sum = 0.0;
            for (int64_t k = 0; k < K; k++)
                sum += act_at(A, a_dtype, i * K + k) * W[k * N + j];
            C[i * N + j] = sum;
        }
    free(W);
}

/* ------------------------------------------------------------------ */
/* Routed experts                                                      */
/* ------------------------------------------------------------------ */

static double sigmoid(double g) { return 1.0 / (1.0 + exp(-g)); }

/* out[t, :] = sum_{k=0..topk-1} w[t,k] * down_e( SiLU(gate_e(x_t)) * up_e(x_t) )
 * with e = idx[t,k], summed in slot order k.  SiLU(g) = g * sigmoid(g).
 * Weights per expert e: W_gate[e], W_up[e] are H x I (K = H, N = I) and
 * W_down[e] is I x H, each in the Q4_0 block layout above.  Slots whose index
 * lies outside [0, E) contribute nothing.  [KT «优化三»: routed experts as
 * batched GEMVs, 6 of 160 per token; «规则二»: gate -> top-k -> experts.]
 *
 * tol[t, j] (may be NULL) bounds the deviation of an fp32 evaluation of the
 * chain from out, to first order.  The pages state a tolerance for one
 * matmul only; carried through the chain it exceeds the output itself, so
 * the chain's bound is taken from the rounding of fp32 arithmetic instead:
 *   - one matmul output over K rows, evaluated as the sums sum a*d*q and
 *     8 * sum a*d in fp32 by a summation tree of depth at most
 *     D(K) = ceil(K/32) + 40, is off by at most gamma(D) * Sq with
 *     Sq = sum_k |a_k * d_kj| * (q_kj + 8) and gamma(n) = n*u / (1 - n*u),
 *     u = 2^-24 (the standard bound for floating-point sums);
 *   - SiLU(g) * u in fp32, with exp from a library routine of a few ulp, is
 *     off by at most (8 + 2|g|) * u relative;
 *   - the errors dg, du of gate and up reach h = SiLU(g) * u as
 *     |SiLU'(g) * u| * dg + |SiLU(g)| * du, and those of h reach the down
 *     output as sum_i |Wd[i, j]| * dh_i;
 *   - the weighted sum over topk slots adds gamma(topk) * sum_k |w_k * y_k|;
 *   - 1e-6 is added once, the absolute term of the pages' tolerance.
 * g, u, h (may be NULL) receive the per-slot stage values [T*topk, I]. */
/* The chain above with the slot weights in fp64 (w64) or fp32 (w32), and an
 * extra tolerance term wrel * |w_k| * |y_k[j]| for weights known only to a
 * relative error wrel (0 for exact weights). */
#define QO_U (1.0 / 16777216.0)
static double qo_gamma(double n) { return n * QO_U / (1.0 - n * QO_U); }
static double qo_depth(int64_t K) { return (double)((K + 31) / 32) + 40.0; }

static void moe_core(const void *x, int x_dtype,
                     const uint8_t *Wg, const uint8_t *Wu, const uint8_t *Wd,
                     const int32_t *idx, const float *w32, const double *w64, double wrel,
                     int64_t T, int64_t topk, int64_t E, int64_t H, int64_t I,
                     double *out, double *tol, double *g_out, double *u_out, double *h_out)
{
    int64_t nbI = (I + QO_BLOCK - 1) / QO_BLOCK;
    int64_t nbH = (H + QO_BLOCK - 1) / QO_BLOCK;
    size_t up_bytes = (size_t)(H * nbI * QO_BLOCK_BYTES);
    size_t down_bytes = (size_t)(I * nbH * QO_BLOCK_BYTES);
    double gam_gu = qo_gamma(qo_depth(H));
    double gam_d = qo_gamma(qo_depth(I));
    double gam_sum = qo_gamma((double)topk);

    double *xt = (double *)malloc(sizeof(double) * (size_t)H);
    double *g = (double *)malloc(sizeof(double) * (size_t)I);
    double *qg = (double *)malloc(sizeof(double) * (size_t)I);
    double *u = (double *)malloc(sizeof(double) * (size_t)I);
    double *qu = (double *)malloc(sizeof(double) * (size_t)I);
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    double *dh = (double *)malloc(sizeof(double) * (size_t)I);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    double *qy = (double *)malloc(sizeof(double) * (size_t)H);
    double *prop = (double *)malloc(sizeof(double) * (size_t)H);
    double *wy = (double *)malloc(sizeof(double) * (size_t)H);

    for (int64_t t = 0; t < T; t++) {
        for (int64_t i = 0; i < H; i++)
            xt[i] = act_at(x, x_dtype, t * H + i);
        for (int64_t j = 0; j < H; j++) {
            out[t * H + j] = 0.0;
            wy[j] = 0.0;
            if (tol)
                tol[t * H + j] = 1e-6;
        }
        for (int64_t k = 0; k < topk; k++) {
            int64_t slot = t * topk + k;
            int32_t e = idx[slot];
            double wk = w64 ? w64[slot] : (double)w32[slot];
            if (e < 0 || e >= E) {
                if (g_out) for (int64_t i = 0; i < I; i++) g_out[slot * I + i] = 0.0;
                if (u_out) for (int64_t i = 0; i < I; i++) u_out[slot * I + i] = 0.0;
                if (h_out) for (int64_t i = 0; i < I; i++) h_out[slot * I + i] = 0.0;
                continue;
            }
            const uint8_t *wg = Wg + (size_t)e * up_bytes;
            const uint8_t *wu = Wu + (size_t)e * up_bytes;
            const uint8_t *wd = Wd + (size_t)e * down_bytes;
            row_matmul(xt, wg, I, H, g, NULL);
            row_matmul(xt, wu, I, H, u, NULL);
            if (tol) {
                row_matmul_absq(xt, wg, I, H, qg);
                row_matmul_absq(xt, wu, I, H, qu);
            }
            for (int64_t i = 0; i < I; i++) {
                double sgm = sigmoid(g[i]);
                double silu = g[i] * sgm;
                double dsilu = sgm * (1.0 + g[i] * (1.0 - sgm));
                h[i] = silu * u[i];
                if (tol)
                    dh[i] = fabs(dsilu * u[i]) * gam_gu * qg[i]
                          + fabs(silu) * gam_gu * qu[i]
                          + (8.0 + 2.0 * fabs(g[i])) * QO_U * fabs(h[i]);
                if (g_out) g_out[slot * I + i] = g[i];
                if (u_out) u_out[slot * I + i] = u[i];
                if (h_out) h_out[slot * I + i] = h[i];
            }
            row_matmul(h, wd, H, I, y, NULL);
            for (int64_t j = 0; j < H; j++)
                out[t * H + j] += wk * y[j];
            if (tol) {
                /* prop[j] = sum_i dh[i] * |Wd[i, j]| */
                row_matmul_abs(dh, wd, H, I, prop);
                row_matmul_absq(h, wd, H, I, qy);
                for (int64_t j = 0; j < H; j++) {
                    tol[t * H + j] += fabs(wk) * (prop[j] + gam_d * qy[j] + wrel * fabs(y[j]));
                    wy[j] += fabs(wk * y[j]);
                }
            }
        }
        if (tol)
            for (int64_t j = 0; j < H; j++)
                tol[t * H + j] += gam_sum * wy[j];
    }
    free(xt); free(g); free(qg); free(u); free(qu); free(h); free(dh); free(y); free(qy);
    free(prop); free(wy);
}

void q4o_moe(const void *x, int x_dtype,
             const uint8_t *Wg, const uint8_t *Wu, const uint8_t *Wd,
             const int32_t *idx, const float *w,
             int64_t T, int64_t topk, int64_t E, int64_t H, int64_t I,
             double *out, double *tol, double *g_out, double *u_out, double *h_out)
{
    moe_core(x, x_dtype, Wg, Wu, Wd, idx, w, NULL, 0.0, T, topk, E, H, I,
             out, tol, g_out, u_out, h_out);
}

/* SiLU(g) = g * sigmoid(g) in fp64, exposed for its closed-form pins. */
double q4o_silu(double g) { return g * sigmoid(g); }

/* ------------------------------------------------------------------ */
/* Router of the routed experts                                        */
/* ------------------------------------------------------------------ */

/* For each token t [KTransformers page, «规则二»: the gate gives the top-k
 * indices and weights]: p = softmax(logits[t]) with the largest logit
 * subtracted before exp [engine page §5.1], the k largest p in descending
 * order (equal p: the lower expert index first), and their weights
 * renormalised to sum to one, w_k = p_k / sum_j p_j over the k chosen.  All
 * arithmetic in fp64. */
void q4o_moe_gate(const float *logits, int64_t T, int64_t E, int64_t topk,
                  int32_t *idx, double *w)
{
    double *p = (double *)malloc(sizeof(double) * (size_t)(E > 0 ? E : 1));
    unsigned char *taken = (unsigned char *)malloc((size_t)(E > 0 ? E : 1));
    for (int64_t t = 0; t < T; t++) {
        const float *l = logits + t * E;
        double mx = (double)l[0];
        for (int64_t e = 1; e < E; e++)
            if ((double)l[e] > mx)
                mx = (double)l[e];
        double sum = 0.0;
        for (int64_t e = 0; e < E; e++) {
            p[e] = exp((double)l[e] - mx);
            sum += p[e];
        }
        for (int64_t e = 0; e < E; e++) {
            p[e] /= sum;
            taken[e] = 0;
        }
        double wsum = 0.0;
        for (int64_t k = 0; k < topk; k++) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; e++)      /* ascending: ties keep the lower index */
                if (!taken[e] && (best < 0 || p[e] > p[best]))
                    best = e;
            taken[best] = 1;
            idx[t * topk + k] = (int32_t)best;
            w[t * topk + k] = p[best];
            wsum += p[best];
        }
        for (int64_t k = 0; k < topk; k++)
            w[t * topk + k] /= wsum;
    }
    free(p);
    free(taken);
}

/* One MoE block: the router above on the logits, the routed experts with its
 * fp64 weights, and, when Is > 0, a shared expert (S_gate, S_up: H x Is;
 * S_down: Is x H) that every token takes with weight 1, added after the
 * routed sum [KTransformers page, «规则二»: gate then experts; «优化三»: the
 * shared expert].  out and tol [T, H]; idx, w [T, topk] receive the routing.
 * tol carries the chain tolerance of both parts plus wrel * |w_k| * |y_k|
 * for router weights computed in fp32 (wrel = 2e-6). */
void q4o_moe_block(const void *x, int x_dtype, const float *logits,
                   const uint8_t *Wg, const uint8_t *Wu, const uint8_t *Wd,
                   int64_t T, int64_t topk, int64_t E, int64_t H, int64_t I,
                   const uint8_t *Sg, const uint8_t *Su, const uint8_t *Sd, int64_t Is,
                   double *out, double *tol, int32_t *idx, double *w)
{
    q4o_moe_gate(logits, T, E, topk, idx, w);
    moe_core(x, x_dtype, Wg, Wu, Wd, idx, NULL, w, 2e-6, T, topk, E, H, I,
             out, tol, NULL, NULL, NULL);
    if (Is <= 0)
        return;
    int32_t *sidx = (int32_t *)calloc((size_t)T, sizeof(int32_t));
    double *sw = (double *)malloc(sizeof(double) * (size_t)T);
    double *so = (double *)malloc(sizeof(double) * (size_t)(T * H));
    double *st = (double *)malloc(sizeof(double) * (size_t)(T * H));
    for (int64_t t = 0; t < T; t++)
        sw[t] = 1.0;
    moe_core(x, x_dtype, Sg, Su, Sd, sidx, NULL, sw, 0.0, T, 1, 1, H, Is,
             so, st, NULL, NULL, NULL);
    /* the shared rows are added to the routed sum in fp32: one more rounding */
    for (int64_t i = 0; i < T * H; i++) {
        if (tol)
            tol[i] += st[i] + QO_U * (fabs(out[i]) + fabs(so[i]));
        out[i] += so[i];
    }
    free(sidx); free(sw); free(so); free(st);
}

/* ------------------------------------------------------------------ */
/* Encoder (quantisation)                                              */
/* ------------------------------------------------------------------ */

/* x rounded to the nearest IEEE binary16 value, ties to even (5-bit
 * exponent with bias 15, 10-bit fraction, subnormals from 2^-24, values
 * that round above 65504 become infinity); returned as its 16 bits. */
uint16_t q4o_f64_to_fp16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x))
        return (uint16_t)(sign | 0x7E00);
    if (isinf(x))
        return (uint16_t)(sign | 0x7C00);
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);                   /* a = m * 2^e, m in [0.5, 1) */
    int expo = e - 1;                     /* a = 1.xxx * 2^expo */
    int quantum_exp = (expo < -14) ? -24 : expo - 10;
    double y = ldexp(a, -quantum_exp);    /* a in units of the quantum */
    double fl = floor(y);
    double r = fl;
    double diff = y - fl;
    if (diff > 0.5 || (diff == 0.5 && fmod(fl, 2.0) != 0.0))
        r = fl + 1.0;
    double v = ldexp(r, quantum_exp);
    if (v >= 65536.0)
        return (uint16_t)(sign | 0x7C00);
    if (v < ldexp(1.0, -14))
        return (uint16_t)(sign | (uint16_t)ldexp(v, 24));   /* subnormal */
    double m = frexp(v, &e);
    expo = e - 1;
    int frac = (int)ldexp(m, 11) - 1024;   /* m*2048 in [1024, 2048) */
    return (uint16_t)(sign | (uint16_t)((expo + 15) << 10) | (uint16_t)frac);
}

/* Q4_0 blocks of a K x N matrix W (row-major, fp32 or bf16 bits) in the
 * layout of [Eng §2.2-§2.3]: for each row k and block b (columns
 * 32b .. 32b+31), m = the element of largest magnitude (the first on ties),
 * d = m / -8 so that m maps to code 0, stored as fp16 (nearest even), and
 * code q_l = min(15, trunc(w_l * (1/d) + 8.5)) with every step an fp32
 * operation (no fused multiply-add; 1/d := 0 when d = 0); padding columns
 * (>= N) get code 8 (value 0).  The pages give no scale rule: this one makes
 * the largest magnitude exact and rounds the rest half up. */
void q4o_quantize(const void *W, int w_dtype, int64_t K, int64_t N, uint8_t *B)
{
    int64_t nb = (N + QO_BLOCK - 1) / QO_BLOCK;
    for (int64_t k = 0; k < K; k++) {
        for (int64_t b = 0; b < nb; b++) {
            float wv[QO_BLOCK];
            int n = (int)((N - b * QO_BLOCK) < QO_BLOCK ? (N - b * QO_BLOCK) : QO_BLOCK);
            for (int l = 0; l < n; l++)
                wv[l] = (float)act_at(W, w_dtype, k * N + b * QO_BLOCK + l);
            float amax = 0.0f, mx = 0.0f;
            for (int l = 0; l < n; l++) {
                float v = wv[l];
                if (amax < fabsf(v)) {
                    amax = fabsf(v);
                    mx = v;
                }
            }
            float d = mx / -8.0f;
            float id = (d != 0.0f) ? 1.0f / d : 0.0f;
            uint8_t *blk = B + (k * nb + b) * QO_BLOCK_BYTES;
            uint16_t h = q4o_f64_to_fp16((double)d);
            blk[0] = (uint8_t)(h & 0xFF);
            blk[1] = (uint8_t)(h >> 8);
            for (int l = 0; l < QO_BLOCK; l++) {
                int q = 8;
                if (l < n) {
                    float t = wv[l] * id;
                    t = t + 8.5f;
                    q = (int)t;
                    if (q > 15)
                        q = 15;
                    if (q < 0)
                        q = 0;
                }
                if (l % 2 == 0)
                    blk[2 + l / 2] = (uint8_t)q;
                else
                    blk[2 + l / 2] |= (uint8_t)(q << 4);
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* Q8_0 (a second format behind the same interface)                    */
/* ------------------------------------------------------------------ */
/* [Eng §2.1-§2.2] names Q8_0 beside Q4_0 (8-bit codes, about 60% of Q4_0's
 * decode speed on its CPU) but prints no layout for it.  Reading, by analogy
 * with the page's block_q4_0 and its §2.3 layout: a block is { fp16 d
 * (little-endian); int8 q[32] } = 34 bytes covering 32 consecutive output
 * columns of one row k; K rows of nb = ceil(N/32) blocks; element l of a block
 * is the two's-complement byte q[l]; W[k, 32b + l] = q * d.  Columns >= N are
 * padding and never read into an output. */
#define QO_Q8_BYTES 34

static double q8_weight_at(const uint8_t *B, int64_t nb, int64_t k, int64_t j)
{
    const uint8_t *blk = B + (k * nb + j / QO_BLOCK) * QO_Q8_BYTES;
    int q = (int)blk[2 + j % QO_BLOCK];
    if (q >= 128)
        q -= 256;                          /* two's complement */
    return (double)q * block_scale(blk);
}

/* W [K, N] fp32 = q * d: at most 8 x 11 significant bits, exact in fp32. */
void q4o_q8_dequant_f32(const uint8_t *B, int64_t K, int64_t N, float *W)
{
    int64_t nb = (N + QO_BLOCK - 1) / QO_BLOCK;
    for (int64_t k = 0; k < K; k++)
        for (int64_t j = 0; j < N; j++)
            W[k * N + j] = (float)q8_weight_at(B, nb, k, j);
}

/* C [M, N] = A . W for Q8_0 weights, S = sum_k |A[i,k] * W[k,j]| (may be
 * NULL), in fp64 with the k -> block -> l order of [Eng §3.4].  Each product
 * is exact in fp64 (24 + 19 bits). */
void q4o_q8_matmul(const void *A, int a_dtype, const uint8_t *B,
                   int64_t M, int64_t N, int64_t K, double *C, double *S)
{
    int64_t nb = (N + QO_BLOCK - 1) / QO_BLOCK;
    for (int64_t i = 0; i < M; i++) {
        double *c = C + i * N;
        double *s = S ? S + i * N : NULL;
        for (int64_t j = 0; j < N; j++) {
            c[j] = 0.0;
            if (s)
                s[j] = 0.0;
        }
        for (int64_t k = 0; k < K; k++) {
            double av = act_at(A, a_dtype, i * K + k);
            for (int64_t j = 0; j < N; j++) {
                double p = av * q8_weight_at(B, nb, k, j);
                c[j] += p;
                if (s)
                    s[j] += fabs(p);
            }
        }
    }
}
