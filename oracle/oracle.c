/*
 * oracle.c - plain, slow CPU reference of the batched q8_0 decode step.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code, header, table
 * or helper with the CUDA library: every function here is written from the
 * definition of the operation, in double precision, with no blocking, fusion
 * or reordering.  Where the method takes an integer decision from a floating
 * value (activation quantization) the decision is taken in fp32, the
 * precision the method stores activations in.
 *
 * Build: gcc -O2 -ffp-contract=off (no fast-math), so every float/double
 * operation is a single IEEE-754 operation; -fopenmp spreads the loops over
 * independent outputs (rows, heads, blocks) across host threads.  Every
 * output is still computed by one thread with the serial code below, in the
 * same order, so the results do not depend on the thread count
 * (orc_set_threads; 1 by default).
 *
 * Sources ("pages"):
 *   [P1] "feat(qwen4exp): exact 4-slot concurrent serving", section "How it
 *        stays exact" (batch-invariant MMVQ: a 4-row batch uses the same
 *        arithmetic as one row).
 *   [P4] "#1209 Speed up concurrent generation, fix QFUSE ...", section "What
 *        changed and why", item 2 (the activation quantizer's division and
 *        rounding convention).
 *   [P5] "antirez/ds4 pull 604", section 2 and "Commit walkthrough" (q8_0
 *        narrow-batch matmul: each 32-weight block read once and dotted
 *        against every token; multi-sequence decode attention, one query per
 *        sequence against its own KV; pos-vector RoPE; per-sequence KV append).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK 32 /* q8_0 block length [P5, Commit walkthrough: "each 32-weight block"] */

#ifdef _OPENMP
#include <omp.h>
#endif

static int orc_threads = 1;

/* Threads the loops below use (>= 1); returns the previous value. */
int orc_set_threads(int n)
{
    int old = orc_threads;
    orc_threads = n < 1 ? 1 : n;
    return old;
}

/* Whether the library was built with OpenMP (otherwise everything runs on one thread). */
int orc_parallel(void)
{
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}

/* IEEE-754 binary16 -> double, from the format definition:
 * normal (e in 1..30): (1024 + m) * 2^(e - 25); subnormal: m * 2^-24. */
double orc_half_to_double(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return s ? -v : v;
}

/* float -> binary16, round to nearest even (the KV cache stores f16). */
uint16_t orc_float_to_half(float f)
{
    _Float16 h = (_Float16)f;
    uint16_t u;
    memcpy(&u, &h, 2);
    return u;
}

uint16_t orc_double_to_half(double f)
{
    _Float16 h = (_Float16)f;
    uint16_t u;
    memcpy(&u, &h, 2);
    return u;
}

/*
 * Activation quantization to q8_0 blocks [P4 item 2; P5 Commit walkthrough].
 * Per block of 32 fp32 values: amax = max|x| (NaN entries skipped),
 * d = amax / 127 (fp32 division, round to nearest), q = round(x / d) with the
 * quotient an fp32 division and round() half away from zero, clamped to
 * [-127, 127]; a block with d == 0 quantizes to all zeros, and a NaN
 * quotient quantizes to 0.  x is [T][ldx] (first K used), q is [T][K],
 * d is [T][K/32].
 */
void orc_quantize_act(const float* x, int T, int K, int64_t ldx, int8_t* q, float* d)
{
    int nb = K / QK;
#pragma omp parallel for collapse(2) schedule(static) num_threads(orc_threads)
    for (int t = 0; t < T; ++t) {
        for (int b = 0; b < nb; ++b) {
            const float* xb = x + (int64_t)t * ldx + (int64_t)b * QK;
            float amax = 0.0f;
            for (int i = 0; i < QK; ++i) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            float dd = amax / 127.0f;
            d[(int64_t)t * nb + b] = dd;
            for (int i = 0; i < QK; ++i) {
                int v = 0;
                if (dd != 0.0f) {
                    float r = xb[i] / dd;
                    if (r == r) {
                        float rr = roundf(r);
                        if (rr > 127.0f) rr = 127.0f;
                        if (rr < -127.0f) rr = -127.0f;
                        v = (int)rr;
                    }
                }
                q[(int64_t)t * K + (int64_t)b * QK + i] = (int8_t)v;
            }
        }
    }
}

/*
 * The half-scale form of the quantizer [P4 item 2: a fused producer must match
 * the consuming quantizer's finite-half guards and division/rounding
 * convention].  Reading: the block scale amax / 127 (fp32 division) is stored
 * as the nearest binary16; a scale that overflows binary16 is stored as the
 * largest finite half (65504); the codes are round-half-away(x / s) against
 * the stored scale s (fp32 division), clamped to [-127, 127], 0 when s == 0
 * or the quotient is NaN.  d receives binary16 bits [T][K/32].
 */
void orc_quantize_act_f16(const float* x, int T, int K, int64_t ldx, int8_t* q, uint16_t* d)
{
    int nb = K / QK;
#pragma omp parallel for collapse(2) schedule(static) num_threads(orc_threads)
    for (int t = 0; t < T; ++t) {
        for (int b = 0; b < nb; ++b) {
            const float* xb = x + (int64_t)t * ldx + (int64_t)b * QK;
            float amax = 0.0f;
            for (int i = 0; i < QK; ++i) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            _Float16 h = (_Float16)(amax / 127.0f);
            if (isinf((float)h)) h = (_Float16)65504.0f;
            uint16_t bits;
            memcpy(&bits, &h, 2);
            d[(int64_t)t * nb + b] = bits;
            float s = (float)h;
            for (int i = 0; i < QK; ++i) {
                int v = 0;
                if (s != 0.0f) {
                    float r = xb[i] / s;
                    if (r == r) {
                        float rr = roundf(r);
                        if (rr > 127.0f) rr = 127.0f;
                        if (rr < -127.0f) rr = -127.0f;
                        v = (int)rr;
                    }
                }
                q[(int64_t)t * K + (int64_t)b * QK + i] = (int8_t)v;
            }
        }
    }
}

/* Per-block integer dots: out[t][n][b] = sum_i wq[n][32b+i] * aq[t][32b+i]. */
void orc_block_dots(const int8_t* wq, int N, int K, const int8_t* aq, int T, int32_t* out)
{
    int nb = K / QK;
#pragma omp parallel for collapse(2) schedule(static) num_threads(orc_threads)
    for (int t = 0; t < T; ++t)
        for (int n = 0; n < N; ++n)
            for (int b = 0; b < nb; ++b) {
                int32_t s = 0;
                for (int i = 0; i < QK; ++i)
                    s += (int32_t)wq[(int64_t)n * K + (int64_t)b * QK + i] *
                         (int32_t)aq[(int64_t)t * K + (int64_t)b * QK + i];
                out[((int64_t)t * N + n) * nb + b] = s;
            }
}

/*
 * q8_0 x q8_0 matvec [P5 Commit walkthrough "narrow-batch q8_0 matmul"; P1]:
 *   y[t][n] = sum_b (wd[n][b] * ad[t][b]) * sum_i wq[n][32b+i] * aq[t][32b+i]
 * wq int8 [N][K] row-major, wd binary16 [N][K/32], aq int8 [T][K],
 * ad fp32 [T][K/32]; y double [T][N].  Accumulated in double, blocks in
 * ascending order.
 */
void orc_matvec(const int8_t* wq, const uint16_t* wd, int N, int K,
                const int8_t* aq, const float* ad, int T, double* y)
{
    int nb = K / QK;
#pragma omp parallel for collapse(2) schedule(static) num_threads(orc_threads)
    for (int t = 0; t < T; ++t)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int b = 0; b < nb; ++b) {
                int64_t s = 0;
                const int8_t* w = wq + (int64_t)n * K + (int64_t)b * QK;
                const int8_t* a = aq + (int64_t)t * K + (int64_t)b * QK;
                for (int i = 0; i < QK; ++i) s += (int64_t)w[i] * (int64_t)a[i];
                double scale = orc_half_to_double(wd[(int64_t)n * nb + b]) * (double)ad[(int64_t)t * nb + b];
                acc += scale * (double)s;
            }
            y[(int64_t)t * N + n] = acc;
        }
}

/* RMSNorm: y = x / sqrt(mean(x^2) + eps) * gamma, per row of length H. */
void orc_rmsnorm(const double* x, int T, int H, const float* gamma, double eps, double* y)
{
#pragma omp parallel for schedule(static) num_threads(orc_threads)
    for (int t = 0; t < T; ++t) {
        const double* xr = x + (int64_t)t * H;
        double ss = 0.0;
        for (int i = 0; i < H; ++i) ss += xr[i] * xr[i];
        double r = 1.0 / sqrt(ss / (double)H + eps);
        for (int i = 0; i < H; ++i) y[(int64_t)t * H + i] = xr[i] * r * (double)gamma[i];
    }
}

/*
 * Pos-vector RoPE [P5 Commit walkthrough: each token at its own position;
 * the per-element math is that of a single-token launch at that position].
 * Half-split pairing: dims (i, i + D/2) for i < D/2 rotate by the angle
 * pos[t] * theta^(-2i/D).  x is [T][n_heads][D], rotated in place.
 */
void orc_rope(double* x, int T, int n_heads, int D, const int32_t* pos, double theta)
{
    int half = D / 2;
#pragma omp parallel for collapse(2) schedule(static) num_threads(orc_threads)
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < n_heads; ++h) {
            double* xr = x + ((int64_t)t * n_heads + h) * D;
            for (int i = 0; i < half; ++i) {
                double ang = (double)pos[t] * pow(theta, -2.0 * (double)i / (double)D);
                double c = cos(ang), s = sin(ang);
                double x0 = xr[i], x1 = xr[i + half];
                xr[i] = x0 * c - x1 * s;
                xr[i + half] = x0 * s + x1 * c;
            }
        }
}

/*
 * One query row of multi-sequence decode attention [P5 Commit walkthrough:
 * one query token per sequence attending to its own cache].  GQA: query head
 * h reads KV head h / (Hq / Hkv).  Keys 0..L-1 of the row's own cache;
 * k, v are binary16 with element (g, j, d) at g*head_stride + j*tok_stride + d.
 * Naive softmax in double: out[h] = sum_j softmax_j(scale * q[h].k_j) v_j.
 */
void orc_attention_row(const double* q, const uint16_t* k, const uint16_t* v, int L,
                       int Hq, int Hkv, int D, int64_t head_stride, int64_t tok_stride,
                       double scale, double* out)
{
    int group = Hq / Hkv;
#pragma omp parallel for schedule(static) num_threads(orc_threads)
    for (int h = 0; h < Hq; ++h) {
        double* s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        int g = h / group;
        const double* qh = q + (int64_t)h * D;
        double m = -INFINITY;
        for (int j = 0; j < L; ++j) {
            const uint16_t* kj = k + g * head_stride + j * tok_stride;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qh[d] * orc_half_to_double(kj[d]);
            s[j] = scale * dot;
            if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (int j = 0; j < L; ++j) {
            s[j] = exp(s[j] - m);
            l += s[j];
        }
        for (int d = 0; d < D; ++d) {
            double o = 0.0;
            for (int j = 0; j < L; ++j)
                o += s[j] * orc_half_to_double(v[g * head_stride + j * tok_stride + d]);
            out[(int64_t)h * D + d] = L > 0 ? o / l : 0.0;
        }
        free(s);
    }
}

/* SwiGLU: h[t][i] = silu(gu[t][i]) * gu[t][F + i], silu(z) = z / (1 + e^-z);
 * the gate half comes first in the concatenated gate||up output. */
void orc_swiglu(const double* gu, int T, int F, double* h)
{
#pragma omp parallel for collapse(2) schedule(static) num_threads(orc_threads)
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < F; ++i) {
            double g = gu[(int64_t)t * 2 * F + i];
            double u = gu[(int64_t)t * 2 * F + F + i];
            h[(int64_t)t * F + i] = g / (1.0 + exp(-g)) * u;
        }
}

/* Index of the largest entry of each row; ties go to the lowest index,
 * NaN entries are never chosen (an all-NaN row gives 0). */
void orc_argmax(const float* x, int T, int V, int32_t* out)
{
    for (int t = 0; t < T; ++t) {
        const float* r = x + (int64_t)t * V;
        int best = 0;
        float bv = -INFINITY;
        int found = 0;
        for (int i = 0; i < V; ++i) {
            if (r[i] != r[i]) continue;
            if (!found || r[i] > bv) {
                bv = r[i];
                best = i;
                found = 1;
            }
        }
        out[t] = best;
    }
}
