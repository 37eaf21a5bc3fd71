/*
 * moe_oracle.c -- CPU oracle for the MoE FFN layer with SelectedSoftmax
 * routing.  TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and
 * the benchmark's CPU-baseline leg; never by the CUDA product path.  It shares
 * no code, header or table with the CUDA library.
 *
 * Plain C, fp64 throughout.  It reads the same storage bytes as the GPU path
 * (fp32, bf16 bit patterns, 34-byte Q8_0 blocks, 36-byte affine 4-bit blocks,
 * 144-byte Q4_K or 210-byte Q6_K super-blocks) and widens them exactly.
 * Steps follow the pages in order:
 *
 *   1. router projection: logit[t,e] = sum_i x[t,i] * W_r[e,i]
 *      ("New Community Model: ZONOS3-Mini (Zyphra) - #1271", §Summary:
 *       MoE routing runs through MoeModule).
 *   2-4. SelectedSoftmax ("... - #1271", §Framework change): rank experts by
 *      raw logit plus a per-expert selection bias, keep the top k, and weigh
 *      the kept experts by the softmax of their logits (the unbiased ones).
 *      Equal ranking scores are broken in favour of the lower expert index.
 *   5. SwiGLU expert FFN ("zonos2.cpp internals", §Recommended: expert stacks
 *      ffn_{gate,up,down}_exps; "... - #1271", §Summary: SwiGLU FFN):
 *      h = SiLU(W_g[e] x) * (W_u[e] x), y = W_d[e] h, SiLU(z) = z / (1+e^-z).
 *   6. combine: out[t] = sum_j w[t,j] * y_j   (residual streams are F32,
 *      "zonos2.cpp internals", §Notes; the oracle keeps fp64).
 *
 * Token grouping (histogram, exclusive scan, stable permutation) is implied by
 * grouped expert compute (ggml mul_mat_id, "zonos2.cpp internals",
 * §Performance); the oracle writes it out by brute force.
 */
#include "moe_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---------------------------------------------------------- exact widening */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16 -> double, written from the format's definition. */
static double f16_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24);                 /* subnormal / zero */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + mant), expo - 25);  /* (1.m) * 2^(e-15) */
    return sign ? -v : v;
}

/* OCP 8-bit floating point, E4M3 -> double, written from the format's
 * definition: sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent
 * field 0 is subnormal (0.m * 2^-6), exponent 15 with mantissa 7 is NaN, and
 * there are no infinities (largest finite 1.75 * 2^8 = 448). */
static double e4m3_to_double(uint8_t b)
{
    const int sign = b >> 7, expo = (b >> 3) & 15, mant = b & 7;
    double v;
    if (expo == 15 && mant == 7)
        v = NAN;
    else if (expo == 0)
        v = ldexp((double)mant, -9);                  /* (m / 8) * 2^-6 */
    else
        v = ldexp((double)(8 + mant), expo - 10);     /* (1 + m / 8) * 2^(e-7) */
    return sign ? -v : v;
}

/* Decode row `row` of a [rows, cols] matrix stored as `dt` into out[cols]. */
static void decode_row(const void *base, int dt, size_t row, int cols, double *out)
{
    if (dt == ORACLE_F32) {
        const float *p = (const float *)base + row * (size_t)cols;
        for (int c = 0; c < cols; ++c) out[c] = (double)p[c];
    } else if (dt == ORACLE_BF16) {
        const uint16_t *p = (const uint16_t *)base + row * (size_t)cols;
        for (int c = 0; c < cols; ++c) out[c] = bf16_bits_to_double(p[c]);
    } else if (dt == ORACLE_Q8_0) { /* per row cols/32 blocks of {fp16 scale, int8 q[32]} */
        const uint8_t *p = (const uint8_t *)base + row * (size_t)(cols / 32) * 34;
        for (int b = 0; b < cols / 32; ++b) {
            const uint8_t *blk = p + (size_t)b * 34;
            double scale = f16_bits_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
            for (int i = 0; i < 32; ++i)
                out[b * 32 + i] = scale * (double)(int8_t)blk[2 + i];
        }
    } else if (dt == ORACLE_Q4_K) {
        /* Q4_K ("zonos2.cpp internals", §Recommended: F16 spine + K-quant
         * experts, 4.50 bits per weight; the pages give no byte layout, this
         * is the GGUF one): per row cols/256 super-blocks of 144 bytes
         * {fp16 d, fp16 dmin, 12 bytes of six-bit sub-block scales sc[8] and
         * mins m[8], 128 bytes of 4-bit codes}.  Sub-block j holds values
         * 32j .. 32j+31: value = d * sc[j] * q - dmin * m[j].  Six-bit fields:
         * for j < 4, sc[j] = low 6 bits of byte j and m[j] = low 6 bits of
         * byte j+4; for j >= 4, sc[j] = (low nibble of byte j+4) + 16 * (top 2
         * bits of byte j-4) and m[j] = (high nibble of byte j+4) + 16 * (top 2
         * bits of byte j).  Codes: the 32-byte run c (c = 0..3) holds sub-block
         * 2c in its low nibbles and sub-block 2c+1 in its high nibbles, value i
         * of each in byte i of the run. */
        const uint8_t *p = (const uint8_t *)base + row * (size_t)(cols / 256) * 144;
        for (int b = 0; b < cols / 256; ++b) {
            const uint8_t *blk = p + (size_t)b * 144;
            const double d = f16_bits_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
            const double dmin = f16_bits_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
            const uint8_t *s = blk + 4, *qs = blk + 16;
            for (int j = 0; j < 8; ++j) {
                int sc, m;
                if (j < 4) {
                    sc = s[j] & 63;
                    m = s[j + 4] & 63;
                } else {
                    sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
                    m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
                }
                const uint8_t *run = qs + 32 * (j / 2);
                for (int i = 0; i < 32; ++i) {
                    const int q = (j % 2) ? (run[i] >> 4) : (run[i] & 15);
                    out[b * 256 + 32 * j + i] = d * (double)sc * (double)q - dmin * (double)m;
                }
            }
        }
    } else if (dt == ORACLE_Q6_K) {
        /* Q6_K ("zonos2.cpp internals", §Recommended: F16 spine + K-quant
         * experts, 6.56 bits per weight, "the sweet spot"; the pages give no
         * byte layout, this is the GGUF one): per row cols/256 super-blocks of
         * 210 bytes {ql[128]: low 4 bits of the codes, qh[64]: their top 2
         * bits, int8 scales[16], fp16 d}.  Value v (0..255) lies in half
         * h = v / 128 at u = v % 128, with g = u / 32 and l = u % 32: its low
         * bits are the low (g < 2) or high (g >= 2) nibble of
         * ql[64h + l + 32 (g % 2)], its top bits bits 2g, 2g+1 of qh[32h + l];
         * the 6-bit code q decodes as d * scales[v / 16] * (q - 32). */
        const uint8_t *p = (const uint8_t *)base + row * (size_t)(cols / 256) * 210;
        for (int b = 0; b < cols / 256; ++b) {
            const uint8_t *blk = p + (size_t)b * 210;
            const uint8_t *ql = blk, *qh = blk + 128;
            const int8_t *sc = (const int8_t *)(blk + 192);
            const double d = f16_bits_to_double((uint16_t)(blk[208] | (blk[209] << 8)));
            for (int v = 0; v < 256; ++v) {
                const int h = v / 128, u = v % 128, g = u / 32, l = u % 32;
                const uint8_t lo_byte = ql[64 * h + l + 32 * (g % 2)];
                const int lo = g < 2 ? (lo_byte & 15) : (lo_byte >> 4);
                const int hi = (qh[32 * h + l] >> (2 * g)) & 3;
                const int q = lo | (hi << 4);
                out[b * 256 + v] = d * (double)sc[v / 16] * (double)(q - 32);
            }
        }
    } else if (dt == ORACLE_FP8) {
        /* fp8 experts ("zonos2" sglang-omni cookbook, §Benchmark Results: the
         * served configurations run "fp8"; the pages fix neither the 8-bit
         * variant nor the scaling, so this is a reading): E4M3 codes with one
         * fp32 scale per row (output channel), stored per row as {fp32 scale,
         * codes[cols]}; value = scale * E4M3(code). */
        const uint8_t *p = (const uint8_t *)base + row * (size_t)(cols + 4);
        float scale;
        memcpy(&scale, p, sizeof scale);
        for (int c = 0; c < cols; ++c) out[c] = (double)scale * e4m3_to_double(p[4 + c]);
    } else { /* ORACLE_Q4_A64 ("Zyphra-ZONOS2-4bit", §How this was quantized:
              * experts at 4 bits, groups of 64, affine; the byte layout is this
              * library's): per row cols/64 blocks of {fp16 scale, fp16 bias,
              * 32 bytes: value 2j in the low nibble of byte j, 2j+1 in the high},
              * value = scale * q + bias */
        const uint8_t *p = (const uint8_t *)base + row * (size_t)(cols / 64) * 36;
        for (int b = 0; b < cols / 64; ++b) {
            const uint8_t *blk = p + (size_t)b * 36;
            double scale = f16_bits_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
            double bias = f16_bits_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
            for (int j = 0; j < 32; ++j) {
                out[b * 64 + 2 * j] = scale * (double)(blk[4 + j] & 15) + bias;
                out[b * 64 + 2 * j + 1] = scale * (double)(blk[4 + j] >> 4) + bias;
            }
        }
    }
}

static int valid_act(int dt) { return dt == ORACLE_F32 || dt == ORACLE_BF16; }
static int valid_w(int dt)
{
    return dt == ORACLE_F32 || dt == ORACLE_BF16 || dt == ORACLE_Q8_0 || dt == ORACLE_Q4_A64 ||
           dt == ORACLE_Q4_K || dt == ORACLE_Q6_K || dt == ORACLE_FP8;
}

/* ------------------------------------------------------------ thread helper */
typedef void (*range_fn)(void *ctx, int begin, int end);
struct range_job { range_fn fn; void *ctx; int begin, end; };

static void *range_trampoline(void *p)
{
    struct range_job *j = (struct range_job *)p;
    j->fn(j->ctx, j->begin, j->end);
    return NULL;
}

int oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* Run fn over [0, n) split into contiguous ranges, one per thread. */
static void parallel_for(int n, int nthreads, range_fn fn, void *ctx)
{
    if (nthreads <= 0) nthreads = oracle_default_threads();
    if (nthreads > n) nthreads = n;
    if (nthreads <= 1) {
        if (n > 0) fn(ctx, 0, n);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    struct range_job *jobs = (struct range_job *)malloc(sizeof(struct range_job) * (size_t)nthreads);
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].fn = fn;
        jobs[i].ctx = ctx;
        jobs[i].begin = (int)((long long)n * i / nthreads);
        jobs[i].end = (int)((long long)n * (i + 1) / nthreads);
        if (pthread_create(&th[i], NULL, range_trampoline, &jobs[i]) == 0)
            started = i + 1;
        else
            break;
    }
    /* any range whose thread could not start runs here */
    for (int i = started; i < nthreads; ++i) fn(ctx, jobs[i].begin, jobs[i].end);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(jobs);
    free(th);
}

/* ------------------------------------------------- step 1: router logits */
struct logits_ctx {
    const void *x; int x_dt; int d; const void *w_r; int E; double *logits;
};

static void logits_range(void *p, int t0, int t1)
{
    struct logits_ctx *c = (struct logits_ctx *)p;
    double *xr = (double *)malloc(sizeof(double) * (size_t)c->d);
    double *wr = (double *)malloc(sizeof(double) * (size_t)c->d);
    for (int t = t0; t < t1; ++t) {
        decode_row(c->x, c->x_dt, (size_t)t, c->d, xr);
        for (int e = 0; e < c->E; ++e) {
            decode_row(c->w_r, c->x_dt, (size_t)e, c->d, wr);
            double acc = 0.0;
            for (int i = 0; i < c->d; ++i) acc += xr[i] * wr[i];
            c->logits[(size_t)t * c->E + e] = acc;
        }
    }
    free(wr);
    free(xr);
}

int oracle_router_logits(const void *x, int x_dt, int T, int d, const void *w_router,
                         int E, double *logits, int nthreads)
{
    if (T < 0 || d <= 0 || E <= 0 || !valid_act(x_dt)) return -1;
    if (T == 0) return 0;
    if (!x || !w_router || !logits) return -1;
    struct logits_ctx c = { x, x_dt, d, w_router, E, logits };
    parallel_for(T, nthreads, logits_range, &c);
    return 0;
}

/* -------------------------------------------- steps 2-4: SelectedSoftmax */
int oracle_selected_softmax(const double *logits, const float *bias, int T, int E, int k,
                            int32_t *topk_idx, double *topk_w, double *margin)
{
    if (T < 0 || E <= 0 || k < 1 || k > E) return -1;
    double *score = (double *)malloc(sizeof(double) * (size_t)E);
    char *taken = (char *)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const double *l = logits + (size_t)t * E;
        /* 2. ranking score = raw logit + selection bias */
        for (int e = 0; e < E; ++e) score[e] = l[e] + (bias ? (double)bias[e] : 0.0);
        memset(taken, 0, (size_t)E);
        /* 3. top-k by repeated arg-max: higher score first, lower index on ties */
        double kth = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || score[e] > score[best]) best = e;
            }
            taken[best] = 1;
            topk_idx[(size_t)t * k + j] = best;
            kth = score[best];
        }
        if (margin) {
            if (k == E) {
                margin[t] = INFINITY;
            } else {
                double next = -INFINITY;
                for (int e = 0; e < E; ++e)
                    if (!taken[e] && score[e] > next) next = score[e];
                margin[t] = kth - next;
            }
        }
        /* 4. weights: softmax over the selected experts' unbiased logits */
        double m = -INFINITY;
        for (int j = 0; j < k; ++j) {
            double v = l[topk_idx[(size_t)t * k + j]];
            if (v > m) m = v;
        }
        double den = 0.0;
        for (int j = 0; j < k; ++j) den += exp(l[topk_idx[(size_t)t * k + j]] - m);
        for (int j = 0; j < k; ++j)
            topk_w[(size_t)t * k + j] = exp(l[topk_idx[(size_t)t * k + j]] - m) / den;
    }
    free(taken);
    free(score);
    return 0;
}

/* ------------------------------ other scoring modes: activation before rank
 * "New Community Model: ZONOS3-Mini (Zyphra) - #1271", §Framework change: the
 * framework's older modes apply a softmax or a sigmoid to the router logits
 * before ranking, and so weigh the experts differently from SelectedSoftmax.
 * The pages give no formulas; the reading taken here:
 *   p = softmax over all E logits (mode 1) or p = sigmoid(logit) (mode 2);
 *   ranking score = p + selection bias; top k, higher first, lower index on ties;
 *   weights = p of the selected experts, not renormalised (renormalised
 *   softmax-before-rank weights would equal SelectedSoftmax's).
 * Mode 0 is SelectedSoftmax. */
int oracle_route_scored(const double *logits, const float *bias, int T, int E, int k, int mode,
                        int32_t *topk_idx, double *topk_w, double *margin)
{
    if (mode == 0) return oracle_selected_softmax(logits, bias, T, E, k, topk_idx, topk_w, margin);
    if (T < 0 || E <= 0 || k < 1 || k > E || (mode != 1 && mode != 2)) return -1;
    double *prob = (double *)malloc(sizeof(double) * (size_t)E);
    double *score = (double *)malloc(sizeof(double) * (size_t)E);
    char *taken = (char *)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const double *l = logits + (size_t)t * E;
        if (mode == 1) {
            double m = -INFINITY;
            for (int e = 0; e < E; ++e) if (l[e] > m) m = l[e];
            double den = 0.0;
            for (int e = 0; e < E; ++e) den += exp(l[e] - m);
            for (int e = 0; e < E; ++e) prob[e] = exp(l[e] - m) / den;
        } else {
            for (int e = 0; e < E; ++e) prob[e] = 1.0 / (1.0 + exp(-l[e]));
        }
        for (int e = 0; e < E; ++e) score[e] = prob[e] + (bias ? (double)bias[e] : 0.0);
        memset(taken, 0, (size_t)E);
        double kth = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || score[e] > score[best]) best = e;
            }
            taken[best] = 1;
            topk_idx[(size_t)t * k + j] = best;
            topk_w[(size_t)t * k + j] = prob[best];
            kth = score[best];
        }
        if (margin) {
            if (k == E) {
                margin[t] = INFINITY;
            } else {
                double next = -INFINITY;
                for (int e = 0; e < E; ++e)
                    if (!taken[e] && score[e] > next) next = score[e];
                margin[t] = kth - next;
            }
        }
    }
    free(taken);
    free(score);
    free(prob);
    return 0;
}

int oracle_softmax_of_set(const double *logits, int T, int E, int k, const int32_t *topk_idx,
                          double *topk_w)
{
    for (int t = 0; t < T; ++t) {
        const double *l = logits + (size_t)t * E;
        double m = -INFINITY;
        for (int j = 0; j < k; ++j) {
            int e = topk_idx[(size_t)t * k + j];
            if (e < 0 || e >= E) return -1;
            if (l[e] > m) m = l[e];
        }
        double den = 0.0;
        for (int j = 0; j < k; ++j) den += exp(l[topk_idx[(size_t)t * k + j]] - m);
        for (int j = 0; j < k; ++j)
            topk_w[(size_t)t * k + j] = exp(l[topk_idx[(size_t)t * k + j]] - m) / den;
    }
    return 0;
}

/* ------------------------------------------------------ token grouping */
int oracle_permute(const int32_t *topk_idx, int T, int k, int E, int32_t *counts,
                   int32_t *offsets, int32_t *perm_tok, int32_t *inv)
{
    if (T < 0 || k < 1 || E <= 0) return -1;
    size_t n = (size_t)T * (size_t)k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (size_t i = 0; i < n; ++i) {
        int e = topk_idx[i];
        if (e < 0 || e >= E) return -1;
        counts[e] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    /* stable: within an expert, slots in increasing flat order (t, then j) */
    for (int e = 0; e < E; ++e) {
        int32_t pos = offsets[e];
        for (size_t i = 0; i < n; ++i) {
            if (topk_idx[i] != e) continue;
            perm_tok[pos] = (int32_t)(i / (size_t)k);
            inv[i] = pos;
            ++pos;
        }
    }
    return 0;
}

/* ---------------------------------------- steps 5-6: experts + combine */
struct combine_ctx {
    const void *x; int x_dt; int d;
    const int32_t *idx; const double *w; int k;
    const void *w_gate, *w_up, *w_down; int w_dt; int E; int F;
    double *out;
};

static void combine_range(void *p, int t0, int t1)
{
    struct combine_ctx *c = (struct combine_ctx *)p;
    int d = c->d, F = c->F;
    double *xr = (double *)malloc(sizeof(double) * (size_t)d);
    double *row = (double *)malloc(sizeof(double) * (size_t)(d > F ? d : F));
    double *h = (double *)malloc(sizeof(double) * (size_t)F);
    for (int t = t0; t < t1; ++t) {
        double *o = c->out + (size_t)t * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        decode_row(c->x, c->x_dt, (size_t)t, d, xr);
        for (int j = 0; j < c->k; ++j) {
            int e = c->idx[(size_t)t * c->k + j];
            double wt = c->w[(size_t)t * c->k + j];
            /* gate and up projections, SiLU(gate) * up */
            for (int f = 0; f < F; ++f) {
                decode_row(c->w_gate, c->w_dt, (size_t)e * F + f, d, row);
                double g = 0.0;
                for (int i = 0; i < d; ++i) g += row[i] * xr[i];
                decode_row(c->w_up, c->w_dt, (size_t)e * F + f, d, row);
                double u = 0.0;
                for (int i = 0; i < d; ++i) u += row[i] * xr[i];
                h[f] = g / (1.0 + exp(-g)) * u;
            }
            /* down projection, weighted by the routing weight */
            for (int i = 0; i < d; ++i) {
                decode_row(c->w_down, c->w_dt, (size_t)e * d + i, F, row);
                double y = 0.0;
                for (int f = 0; f < F; ++f) y += row[f] * h[f];
                o[i] += wt * y;
            }
        }
    }
    free(h);
    free(row);
    free(xr);
}

int oracle_expert_combine(const void *x, int x_dt, int T, int d, const int32_t *topk_idx,
                          const double *topk_w, int k, const void *w_gate, const void *w_up,
                          const void *w_down, int w_dt, int E, int F, double *out, int nthreads)
{
    if (T < 0 || d <= 0 || F <= 0 || E <= 0 || k < 1 || !valid_act(x_dt) || !valid_w(w_dt))
        return -1;
    if (w_dt == ORACLE_Q8_0 && (d % 32 || F % 32)) return -1;
    if (w_dt == ORACLE_Q4_A64 && (d % 64 || F % 64)) return -1;
    if ((w_dt == ORACLE_Q4_K || w_dt == ORACLE_Q6_K) && (d % 256 || F % 256)) return -1;
    for (size_t i = 0; i < (size_t)T * k; ++i)
        if (topk_idx[i] < 0 || topk_idx[i] >= E) return -1;
    if (T == 0) return 0;
    struct combine_ctx c = { x, x_dt, d, topk_idx, topk_w, k, w_gate, w_up, w_down,
                             w_dt, E, F, out };
    parallel_for(T, nthreads, combine_range, &c);
    return 0;
}

int oracle_moe_forward(const void *x, int x_dt, int T, int d, const void *w_router,
                       const float *bias, int E, int k, const void *w_gate, const void *w_up,
                       const void *w_down, int w_dt, int F, double *out, int32_t *topk_idx,
                       double *topk_w, double *margin, int nthreads)
{
    return oracle_moe_forward_scored(x, x_dt, T, d, w_router, bias, E, k, 0, w_gate, w_up,
                                     w_down, w_dt, F, out, topk_idx, topk_w, margin, nthreads);
}

int oracle_moe_forward_scored(const void *x, int x_dt, int T, int d, const void *w_router,
                              const float *bias, int E, int k, int mode, const void *w_gate,
                              const void *w_up, const void *w_down, int w_dt, int F, double *out,
                              int32_t *topk_idx, double *topk_w, double *margin, int nthreads)
{
    if (T < 0 || k < 1 || k > E) return -1;
    if (T == 0) return 0;
    double *logits = (double *)malloc(sizeof(double) * (size_t)T * E);
    int rc = oracle_router_logits(x, x_dt, T, d, w_router, E, logits, nthreads);
    if (rc == 0) rc = oracle_route_scored(logits, bias, T, E, k, mode, topk_idx, topk_w, margin);
    if (rc == 0)
        rc = oracle_expert_combine(x, x_dt, T, d, topk_idx, topk_w, k, w_gate, w_up, w_down,
                                   w_dt, E, F, out, nthreads);
    free(logits);
    return rc;
}
