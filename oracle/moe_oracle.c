/*
 * moe_oracle.c -- plain fp64 CPU oracle of the MoE layer forward with router
 * replay.  TEST INFRASTRUCTURE ONLY: the CUDA product path never includes,
 * links, loads or calls this file.  See moe_oracle.h for the definition it
 * computes and the passages it follows.
 *
 * Style rule of this file: every function is the plain definition written
 * out, loops in the order the definition reads, fp64 throughout.  OpenMP
 * parallelism is only ever across independent outputs (tokens, rows); the
 * summation order of every individual output is the one written here.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- exact decoders ------------------------------------------------------ */

double oracle_bf16_to_f64(uint16_t h) {
    /* bf16 is the top half of an IEEE binary32 pattern. */
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_e4m3_to_f64(uint8_t b) {
    /* OCP 8-bit E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits,
     * no infinities, S.1111.111 is NaN. [TR] §6.1 Kernels: MXFP8 values. */
    int sign = (b >> 7) & 1;
    int ex = (b >> 3) & 0xF;
    int man = b & 7;
    double v;
    if (ex == 15 && man == 7) return NAN;
    if (ex == 0)
        v = ldexp((double)man, -9);          /* subnormal: man/8 * 2^(1-7) */
    else
        v = ldexp(8.0 + man, ex - 7 - 3);    /* (1 + man/8) * 2^(ex-7) */
    return sign ? -v : v;
}

double oracle_e8m0_to_f64(uint8_t s) {
    /* E8M0 block scale: 2^(s-127); 0xFF is NaN. [TR] §6.1: MXFP8 scale. */
    if (s == 0xFF) return NAN;
    return ldexp(1.0, (int)s - 127);
}

/* ---- NVFP4 ([TR] §6.1 Kernels: FP4 E2M1 values, an E4M3 scale per 16 values,
 * an FP32 scale per token; IEEE division in the quantiser) ------------------ */

double oracle_e2m1_to_f64(uint8_t code) {
    /* sign bit 3; exponent bits 2..1 with bias 1; mantissa bit 0. */
    int sign = (code >> 3) & 1;
    int ex = (code >> 1) & 3;
    int man = code & 1;
    double v = ex == 0 ? 0.5 * man : ldexp(1.0 + 0.5 * man, ex - 1);
    return sign ? -v : v;
}

uint8_t oracle_e2m1_round(float vf) {
    /* the nearest of the eight magnitudes; on a tie the even code; beyond the
     * largest magnitude, the largest (saturation) */
    const double a = fabs((double)vf);
    int best = a >= 6.0 ? 7 : 0;
    for (int m = 1; m < 8 && best != 7; ++m) {
        const double dm = fabs(a - oracle_e2m1_to_f64((uint8_t)m));
        const double db = fabs(a - oracle_e2m1_to_f64((uint8_t)best));
        if (dm < db || (dm == db && m % 2 == 0)) best = m;
    }
    return (uint8_t)((vf < 0.0f && best != 0) ? (best | 8) : best);
}

uint8_t oracle_e4m3_round(float vf) {
    /* E4M3 (fn): normals (1 + m/8) * 2^(e-7), e = 1..15 (448 the largest),
     * subnormals m/8 * 2^-6.  Round to nearest, ties to even, saturate. */
    const double v = (double)vf;
    if (!(v > 0.0)) return 0;
    if (v >= 448.0) return 0x7E;
    int e;
    frexp(v, &e);
    int ex = e - 1; /* 2^ex <= v < 2^(ex+1) */
    if (ex < -6) return (uint8_t)nearbyint(ldexp(v, 9)); /* multiples of 2^-9; 8 -> 2^-6 */
    double m = nearbyint(ldexp(v, 3 - ex));                /* 8 .. 16 */
    if (m == 16.0) {
        m = 8.0;
        ex += 1;
    }
    const int code = ((ex + 7) << 3) | ((int)m - 8);
    return (uint8_t)(code > 0x7E ? 0x7E : code);
}

void oracle_nvfp4_quantize_rows(const float *x, int64_t R, int64_t K, uint8_t *codes,
                                uint8_t *bscale, float *rscale) {
    /* fp32 arithmetic throughout (built with -ffp-contract=off), divisions
     * correctly rounded as the IEEE standard defines them. */
    for (int64_t r = 0; r < R; ++r) {
        const float *row = x + r * K;
        float amax = 0.0f;
        for (int64_t i = 0; i < K; ++i) amax = fmaxf(amax, fabsf(row[i]));
        const float s = amax / 2688.0f; /* 6 * 448 */
        rscale[r] = s;
        for (int64_t b = 0; b < K / 16; ++b) {
            float bmax = 0.0f;
            for (int64_t i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(row[16 * b + i]));
            uint8_t S = 0;
            if (s > 0.0f) {
                const float sixth = bmax / 6.0f;
                S = oracle_e4m3_round(sixth / s);
            }
            bscale[r * (K / 16) + b] = S;
            const float denom = (float)oracle_e4m3_to_f64(S) * s;
            for (int64_t i = 0; i < 16; ++i) {
                const int64_t c = 16 * b + i;
                codes[r * K + c] = denom > 0.0f ? oracle_e2m1_round(row[c] / denom) : 0;
            }
        }
    }
}

double oracle_round_bf16(double v) {
    /* 8 significant bits, ties to even; bf16 shares fp32's exponent range
     * (subnormal spacing 2^-133); beyond the largest finite value -> inf. */
    if (v == 0.0 || !isfinite(v)) return v;
    int e;
    frexp(v, &e);
    int ex = e - 1;
    if (ex < -126) ex = -126;
    const double r = ldexp(nearbyint(ldexp(v, 7 - ex)), ex - 7);
    if (fabs(r) > 0x1.FEp127) return copysign(INFINITY, v);
    return r;
}

/* Quantise rows and return the values the GEMM uses: e2m1 * e4m3 * row scale. */
static void nvfp4_quantised_values(const float *x, int64_t R, int64_t K, double *out) {
    uint8_t *codes = (uint8_t *)malloc((size_t)(R * K));
    uint8_t *bs = (uint8_t *)malloc((size_t)(R * K / 16));
    float *rs = (float *)malloc((size_t)R * sizeof(float));
    oracle_nvfp4_quantize_rows(x, R, K, codes, bs, rs);
    for (int64_t r = 0; r < R; ++r)
        for (int64_t i = 0; i < K; ++i)
            out[r * K + i] = oracle_e2m1_to_f64(codes[r * K + i]) *
                             oracle_e4m3_to_f64(bs[r * (K / 16) + i / 16]) * (double)rs[r];
    free(rs);
    free(bs);
    free(codes);
}

void oracle_mx_qdq_rows(const double *in, int64_t R, int64_t K, double *out) {
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t b = 0; b < K / 32; ++b) {
            const double *v = in + r * K + 32 * b;
            double *o = out + r * K + 32 * b;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) amax = fmax(amax, fabs(v[i]));
            int X = -127;
            if (amax > 0.0) {
                int e;
                frexp(amax, &e); /* amax = m * 2^e, m in [0.5, 1): floor(log2) = e - 1 */
                X = e - 1 - 8;
                if (X < -127) X = -127;
                if (X > 127) X = 127;
            }
            for (int i = 0; i < 32; ++i) {
                const double s = ldexp(fabs(v[i]), -X); /* exact: a power of two */
                const double q = oracle_e4m3_to_f64(oracle_e4m3_round((float)s));
                o[i] = ldexp(v[i] < 0.0 ? -q : q, X);
            }
        }
    }
}

double oracle_matrix_elem(const oracle_matrix *m, int64_t K, int64_t r, int64_t c) {
    if (m->fmt == ORACLE_W_BF16)
        return oracle_bf16_to_f64(((const uint16_t *)m->values)[r * K + c]);
    if (m->fmt == ORACLE_W_NVFP4) {
        const uint8_t byte = ((const uint8_t *)m->values)[r * (K / 2) + c / 2];
        const uint8_t code = (c & 1) ? (byte >> 4) : (byte & 15);
        return oracle_e2m1_to_f64(code) * oracle_e4m3_to_f64(m->scales[r * (K / 16) + c / 16]) *
               (double)m->tscale;
    }
    /* MXFP8: one E8M0 scale per 32 consecutive elements along K. */
    double q = oracle_e4m3_to_f64(((const uint8_t *)m->values)[r * K + c]);
    double sc = oracle_e8m0_to_f64(m->scales[r * (K / 32) + c / 32]);
    return q * sc;
}

/* ---- routing --------------------------------------------------------------- */

void oracle_router_logits(const uint16_t *x, const uint16_t *wr, const float *bias,
                          int64_t T, int64_t d, int64_t E, double *logits) {
    /* [TD] "每层有一个门控": the gate is a linear map of the hidden state. */
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; ++t) {
        for (int64_t e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int64_t j = 0; j < d; ++j)
                acc += oracle_bf16_to_f64(x[t * d + j]) * oracle_bf16_to_f64(wr[e * d + j]);
            if (bias) acc += (double)bias[e];
            logits[t * E + e] = acc;
        }
    }
}

/* a ranks before b: larger logit first, equal logits -> lower expert id. */
static int ranks_before(double la, int64_t a, double lb, int64_t b) {
    if (la > lb) return 1;
    if (la < lb) return 0;
    return a < b;
}

void oracle_select_topk(const double *logits, int64_t T, int64_t E, int64_t k,
                        int32_t *ids) {
    /* [TD]: the gate picks 8 of 384 experts per token.  Selection: k rounds,
     * each taking the best expert not yet chosen. */
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; ++t) {
        const double *l = logits + t * E;
        unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
        for (int64_t s = 0; s < k; ++s) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
            }
            taken[best] = 1;
            ids[t * k + s] = (int32_t)best;
        }
        free(taken);
    }
}

int64_t oracle_check_ids(const int32_t *ids, int64_t T, int64_t E, int64_t k,
                         uint8_t *valid) {
    int64_t bad = 0;
    for (int64_t t = 0; t < T; ++t) {
        int ok = 1;
        for (int64_t s = 0; s < k; ++s) {
            int32_t e = ids[t * k + s];
            if (e < 0 || e >= E) ok = 0;
            for (int64_t s2 = 0; s2 < s; ++s2)
                if (ids[t * k + s2] == e) ok = 0;
        }
        valid[t] = (uint8_t)ok;
        bad += !ok;
    }
    return bad;
}

void oracle_gate_weights(const double *logits, const int32_t *ids, int64_t T,
                         int64_t E, int64_t k, double *gates) {
    /* [TR] §6.2: under replay the router still computes the gate scores, over
     * the replayed experts.  Softmax over all E followed by renormalisation
     * over the chosen set equals the softmax of the chosen logits, since the
     * common denominator cancels. */
    for (int64_t t = 0; t < T; ++t) {
        const double *l = logits + t * E;
        double m = -INFINITY;
        for (int64_t s = 0; s < k; ++s) {
            double v = l[ids[t * k + s]];
            if (v > m) m = v;
        }
        double den = 0.0;
        for (int64_t s = 0; s < k; ++s) den += exp(l[ids[t * k + s]] - m);
        for (int64_t s = 0; s < k; ++s)
            gates[t * k + s] = exp(l[ids[t * k + s]] - m) / den;
    }
}

void oracle_filter_replay(const double *logits, const int32_t *ids_in, int64_t T,
                          int64_t E, int64_t k, double tau, int32_t *ids_out,
                          int32_t *n_replaced) {
    int32_t *own = (int32_t *)malloc((size_t)k * sizeof(int32_t));
    unsigned char *kept = (unsigned char *)malloc((size_t)k);
    for (int64_t t = 0; t < T; ++t) {
        const double *l = logits + t * E;
        const int32_t *in = ids_in + t * k;
        int32_t *out = ids_out + t * k;
        oracle_select_topk(l, 1, E, k, own);
        /* threshold from the router's own k-th choice */
        const double thr = tau > 0.0 ? l[own[k - 1]] + log(tau) : -INFINITY;
        for (int64_t s = 0; s < k; ++s) {
            kept[s] = l[in[s]] >= thr;
            out[s] = in[s];
        }
        int32_t replaced = 0;
        int64_t next = 0; /* next own candidate to try */
        for (int64_t s = 0; s < k; ++s) {
            if (kept[s]) continue;
            for (;;) {
                int32_t c = own[next++];
                int taken = 0;
                for (int64_t s2 = 0; s2 < k; ++s2)
                    if ((kept[s2] || s2 < s) && out[s2] == c) taken = 1;
                if (!taken) {
                    out[s] = c;
                    break;
                }
            }
            ++replaced;
        }
        if (n_replaced) n_replaced[t] = replaced;
    }
    free(kept);
    free(own);
}

/* ---- dispatch: stable counting sort -------------------------------------- */

void oracle_counting_sort(const int32_t *ids, int64_t n_pairs, int64_t E,
                          int32_t *cnt, int32_t *off, int32_t *perm, int32_t *inv) {
    /* [TR] §6.1: tokens are dispatched to their experts and combined back.
     * On one device, dispatch is a grouping of the (token, slot) pairs by
     * expert that keeps the pair order inside each group. */
    int32_t *next = (int32_t *)malloc((size_t)(E > 0 ? E : 1) * sizeof(int32_t));
    for (int64_t e = 0; e < E; ++e) cnt[e] = 0;
    for (int64_t i = 0; i < n_pairs; ++i) cnt[ids[i]] += 1;
    off[0] = 0;
    for (int64_t e = 0; e < E; ++e) off[e + 1] = off[e] + cnt[e];
    for (int64_t e = 0; e < E; ++e) next[e] = off[e];
    for (int64_t i = 0; i < n_pairs; ++i) {
        int32_t dst = next[ids[i]]++;
        perm[dst] = (int32_t)i;
        inv[i] = dst;
    }
    free(next);
}

/* ---- expert FFN ------------------------------------------------------------ */

static double silu(double a) { return a / (1.0 + exp(-a)); }

void oracle_expert_ffn(const uint16_t *x, int64_t n, int64_t d, int64_t F,
                       const oracle_matrix *wg, const oracle_matrix *wu,
                       const oracle_matrix *wd, double *y) {
    /* SwiGLU expert: h_f = silu(x . Wg[f]) * (x . Wu[f]);  y = sum_f h_f Wd[:, f].
     * [TR] §6.1 and Fig. 10: the grouped expert GEMMs. */
    double *xd = (double *)malloc((size_t)(n * d) * sizeof(double));
    double *h = (double *)malloc((size_t)(n * F) * sizeof(double));
    const int nv = wg->fmt == ORACLE_W_NVFP4;
    const int mxa = wg->fmt == ORACLE_W_MXFP8_ACT;
    if (mxa) {
        /* MXFP8 expert compute: the token rows enter the GEMM quantised along d */
        for (int64_t i = 0; i < n * d; ++i) xd[i] = oracle_bf16_to_f64(x[i]);
        oracle_mx_qdq_rows(xd, n, d, xd);
    } else if (nv) {
        /* NVFP4 forward: the token rows enter the GEMM quantised */
        float *xf = (float *)malloc((size_t)(n * d) * sizeof(float));
        for (int64_t i = 0; i < n * d; ++i) xf[i] = (float)oracle_bf16_to_f64(x[i]);
        nvfp4_quantised_values(xf, n, d, xd);
        free(xf);
    } else {
        for (int64_t i = 0; i < n * d; ++i) xd[i] = oracle_bf16_to_f64(x[i]);
    }

    int64_t f;
#pragma omp parallel for schedule(static)
    for (f = 0; f < F; ++f) {
        for (int64_t r = 0; r < n; ++r) {
            double a = 0.0, b = 0.0;
            for (int64_t j = 0; j < d; ++j) {
                a += xd[r * d + j] * oracle_matrix_elem(wg, d, f, j);
                b += xd[r * d + j] * oracle_matrix_elem(wu, d, f, j);
            }
            h[r * F + f] = silu(a) * b;
        }
    }
    if (mxa) {
        /* h is stored in bf16 and quantised along F, row by row */
        for (int64_t i = 0; i < n * F; ++i) h[i] = oracle_round_bf16(h[i]);
        oracle_mx_qdq_rows(h, n, F, h);
    }
    if (nv) {
        /* h is stored in bf16 and quantised again, row by row */
        float *hf = (float *)malloc((size_t)(n * F) * sizeof(float));
        for (int64_t i = 0; i < n * F; ++i) hf[i] = (float)oracle_round_bf16(h[i]);
        nvfp4_quantised_values(hf, n, F, h);
        free(hf);
    }
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < d; ++i) {
        for (int64_t r = 0; r < n; ++r) {
            double acc = 0.0;
            for (int64_t ff = 0; ff < F; ++ff)
                acc += h[r * F + ff] * oracle_matrix_elem(wd, F, i, ff);
            y[r * d + i] = acc;
        }
    }
    free(h);
    free(xd);
}

/* ---- combine ----------------------------------------------------------------- */

void oracle_combine(const double *y_slots, const double *gates,
                    const double *y_shared, const uint8_t *valid, int64_t T,
                    int64_t k, int64_t d, double *out) {
    /* [TR] §6.1: combine; [TD]/[CH]: expert outputs are added in one fixed
     * order -- slot 0 first, then 1, ..., then the always-on shared expert. */
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t i = 0; i < d; ++i) {
            double acc = 0.0;
            if (!valid || valid[t]) {
                for (int64_t s = 0; s < k; ++s)
                    acc += gates[t * k + s] * y_slots[(t * k + s) * d + i];
                if (y_shared) acc += y_shared[t * d + i];
            }
            out[t * d + i] = acc;
        }
    }
}

int oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

int oracle_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
