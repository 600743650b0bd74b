/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the decode projection GEMM and
 * the MoE decode block.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline / reference legs of the benchmark load this file. The CUDA path
 * never links, includes or calls it, and it shares no code, header, table or
 * helper with the CUDA path.
 *
 * Every function states the definition it writes out. The method's sources
 * are four web pages about the Kimi K3 decode path on GB300; they describe
 * the operations in words only:
 *   - "vLLM 如何用智能体辅助优化 Kimi K3 解码性能", Part 1 §1 "针对工作负载调优形状":
 *     skinny projections y = x·Wᵀ at batch 1-2 by a small-matrix kernel and at
 *     larger batch by split-K. Both compute the same product.
 *   - same page, Part 1 §3 "改进 MoE 调度与重叠": router scores, routed experts,
 *     and a shared expert whose output is added.
 * The pages print no formula, shape, dtype or worked example. Shapes, dtypes,
 * the top-8 renormalised softmax gates and the SwiGLU expert come from the
 * workload definitions that accompany them (hidden 7168, 384 experts, top-8,
 * intermediate 2048, bf16 weights, fp32 accumulation, bf16 output).
 *
 * Arithmetic: every product and sum in double precision, in the plain order
 * k = 0..K-1. No blocking, fusion or reordering. bf16 operands are decoded
 * bit-exactly (a bf16 value is the top half of an IEEE binary32 word).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> double. The 16 bits are the high half of a binary32
 * word; the conversion to double is exact. */
static double bf16_to_f64(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double orc_bf16_to_f64(uint16_t b) { return bf16_to_f64(b); }

void orc_bf16_to_f64_array(const uint16_t* in, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_to_f64(in[i]);
}

/* double -> bf16 bit pattern, round to nearest, ties to even, written from the
 * definition of the format: 8 significant bits, binary32's exponent range,
 * subnormal quantum 2^-133, overflow to infinity. */
uint16_t orc_f64_to_bf16_bits(double v) {
    if (isnan(v)) return (uint16_t)0x7FC0;
    uint16_t sign = signbit(v) ? (uint16_t)0x8000 : (uint16_t)0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int e;
    double m = frexp(a, &e);             /* a = m * 2^e, m in [0.5, 1) */
    if (e < -125) {                      /* below the smallest normal 2^-126 */
        double q = nearbyint(ldexp(a, 133)); /* count of 2^-133 quanta */
        return (uint16_t)(sign | (uint16_t)q); /* q == 128 is the smallest normal */
    }
    double q = nearbyint(ldexp(m, 8));   /* significand with 8 bits: [128, 256] */
    if (q == 256.0) { q = 128.0; e += 1; }
    int field = e + 126;                 /* biased exponent: a = 1.f * 2^(e-1) */
    if (field >= 255) return (uint16_t)(sign | 0x7F80);
    return (uint16_t)(sign | (uint16_t)(field << 7) | (uint16_t)((int)q - 128));
}

void orc_f64_to_bf16_array(const double* in, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16_bits(in[i]);
}

/* Round a double to the nearest bf16 value (ties to even), returned as double. */
double orc_round_bf16(double v) { return bf16_to_f64(orc_f64_to_bf16_bits(v)); }

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Projection GEMM, "vLLM 如何用智能体辅助优化 Kimi K3 解码性能" Part 1 §1:
 *   y[m,n]      = sum_k x[m,k] * W[n,k]
 *   absref[m,n] = sum_k |x[m,k] * W[n,k]|   (the tolerance's reference scale)
 * x is [M,K] bf16 row-major, W is [N,K] bf16 row-major. absref may be NULL. */
void orc_linear(const uint16_t* x, const uint16_t* W, int64_t M, int64_t N,
                int64_t K, double* y, double* absref) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            const uint16_t* xr = x + m * K;
            const uint16_t* wr = W + n * K;
            double acc = 0.0, accabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = bf16_to_f64(xr[k]) * bf16_to_f64(wr[k]);
                acc += p;
                accabs += fabs(p);
            }
            y[m * N + n] = acc;
            if (absref) absref[m * N + n] = accabs;
        }
    }
}

/* Same product with double activations a[M,K] (used for the second GEMM of
 * an expert, whose input is the fp64 SwiGLU hidden vector). */
void orc_linear_f64act(const double* a, const uint16_t* W, int64_t M, int64_t N,
                       int64_t K, double* y, double* absref) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            const double* ar = a + m * K;
            const uint16_t* wr = W + n * K;
            double acc = 0.0, accabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = ar[k] * bf16_to_f64(wr[k]);
                acc += p;
                accabs += fabs(p);
            }
            y[m * N + n] = acc;
            if (absref) absref[m * N + n] = accabs;
        }
    }
}

/* Split-K form of the same product (same page, Part 1 §1: "split-K spreads
 * the GEMM over more workers"). K is cut into S contiguous chunks
 * [s*K/S, (s+1)*K/S); chunk s gives a partial sum; y is the sum of the
 * partials in the order s = 0..S-1. */
void orc_linear_splitk(const uint16_t* x, const uint16_t* W, int64_t M, int64_t N,
                       int64_t K, int64_t S, double* y) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double total = 0.0;
            for (int64_t s = 0; s < S; ++s) {
                int64_t k0 = s * K / S, k1 = (s + 1) * K / S;
                double part = 0.0;
                for (int64_t k = k0; k < k1; ++k)
                    part += bf16_to_f64(x[m * K + k]) * bf16_to_f64(W[n * K + k]);
                total += part;
            }
            y[m * N + n] = total;
        }
    }
}

/* Top-k selection and gates for one token, by a full sort.
 * Order: value descending, ties broken by the smaller expert index.
 * Gates: softmax over all E logits followed by renormalisation over the k
 * selected equals exp(l_j - l_max) / sum_{j' selected} exp(l_j' - l_max);
 * that closed form is what is computed. */
typedef struct { double v; int64_t i; } orc_pair;

static int orc_pair_cmp(const void* pa, const void* pb) {
    const orc_pair* a = (const orc_pair*)pa;
    const orc_pair* b = (const orc_pair*)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->i < b->i) ? -1 : (a->i > b->i) ? 1 : 0;
}

int orc_topk(const double* logits, int64_t M, int64_t E, int64_t k,
             int32_t* idx, double* gates) {
    if (k < 1 || k > E) return -1;
    orc_pair* buf = (orc_pair*)malloc(sizeof(orc_pair) * (size_t)E);
    if (!buf) return -2;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t e = 0; e < E; ++e) { buf[e].v = logits[m * E + e]; buf[e].i = e; }
        qsort(buf, (size_t)E, sizeof(orc_pair), orc_pair_cmp);
        double lmax = buf[0].v, denom = 0.0;
        for (int64_t j = 0; j < k; ++j) denom += exp(buf[j].v - lmax);
        for (int64_t j = 0; j < k; ++j) {
            idx[m * k + j] = (int32_t)buf[j].i;
            if (gates) gates[m * k + j] = exp(buf[j].v - lmax) / denom;
        }
    }
    free(buf);
    return 0;
}

/* SwiGLU hidden vector of one expert for c token rows.
 * W13 is [2I, H] bf16: rows 0..I-1 are the gate projection W1, rows I..2I-1
 * the up projection W3.
 *   a = x·W1ᵀ, b = x·W3ᵀ, h = silu(a) * b, silu(z) = z / (1 + e^-z).
 * round_h != 0 rounds h to bf16 (a diagnostic; the fp64 reference leaves it
 * unrounded). */
void orc_swiglu_hidden(const uint16_t* xrows, const uint16_t* W13, int64_t c,
                       int64_t H, int64_t I, int round_h, double* h) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t t = 0; t < c; ++t) {
        for (int64_t i = 0; i < I; ++i) {
            const uint16_t* xr = xrows + t * H;
            const uint16_t* w1 = W13 + i * H;
            const uint16_t* w3 = W13 + (I + i) * H;
            double a = 0.0, b = 0.0;
            for (int64_t k = 0; k < H; ++k) {
                double xv = bf16_to_f64(xr[k]);
                a += xv * bf16_to_f64(w1[k]);
                b += xv * bf16_to_f64(w3[k]);
            }
            double v = a / (1.0 + exp(-a)) * b;
            h[t * I + i] = round_h ? orc_round_bf16(v) : v;
        }
    }
}

/* silu(z) = z / (1 + e^-z), exposed so the tests can pin it. */
double orc_silu(double z) { return z / (1.0 + exp(-z)); }
