/*
 * oracle.c — plain, slow CPU oracle for one top-k Mixture-of-Experts layer.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * bench's CPU-baseline leg load this library. The CUDA library never links,
 * includes or calls it, and it shares no code with the CUDA library.
 *
 * What the layer computes. The pages establish that every decoder layer of
 * Muse Spark is a Mixture-of-Experts layer whose tokens each pick 8 of 256
 * experts ("How SGLang-TorchTPU accelerated an 816B-parameter MoE on TPU v7",
 * section "Introduction"), that per-expert outputs are combined after the
 * experts run ("TensorSharp Muse Spark benchmark", section "Performance"),
 * and that summing per-expert partials in bf16 hurt quality (same page,
 * section "Answer quality"), so every sum here is taken in double. The pages
 * leave the gate, renormalisation, FFN type and tie rule open; this oracle
 * takes the plainest reading, stated with each function:
 *
 *   logit[t,e] = fp32( sum_c x[t,c] * Wr[e,c] ) (+ bias[e])
 *   p[t,:]     = softmax(logit[t,:]) over all E experts (double)
 *   ids[t,:]   = the k experts of largest p, ties to the lower expert id,
 *                listed by descending p
 *   w[t,j]     = p[t,ids[t,j]] / sum_j' p[t,ids[t,j']]
 *   h          = silu(Wg[e] x) * (Wu[e] x),  silu(g) = g / (1 + exp(-g))
 *   Y[t,j]     = Wd[e] h                      (e = ids[t,j])
 *   y[t]       = sum_j w[t,j] Y[t,j]          (j ascending)
 *
 * NVFP4 expert weights (the same page, section "Results and interpretation",
 * names NVFP4 expert weights) are 16-element blocks of E2M1 codes with one
 * E4M3 scale per block and one fp32 scale per tensor; the oracle owns its own
 * quantiser and codec tables (OCP Microscaling Formats v1.0 for E2M1, OCP FP8
 * for E4M3). Decisions that produce integer codes are taken in fp32, the
 * precision the CUDA quantiser uses.
 *
 * Parity pins for every function here live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int d, E, k, I;
    int fmt;                          /* 0: bf16 experts, 1: nvfp4 experts */
    const uint16_t *w_router;         /* [E, d] bf16 bits */
    const float *router_bias;         /* [E] fp32 or NULL */
    const uint16_t *w_gate, *w_up;    /* [E, I, d] bf16 bits */
    const uint16_t *w_down;           /* [E, d, I] bf16 bits */
    const uint8_t *q_gate, *q_up;     /* [E, I, d/2] packed E2M1, low nibble = even k */
    const uint8_t *q_down;            /* [E, d, I/2] */
    const uint8_t *s_gate, *s_up;     /* [E, I, d/16] E4M3 block scales */
    const uint8_t *s_down;            /* [E, d, I/16] */
    const float *g_gate, *g_up, *g_down; /* [E] per-tensor fp32 scales */
    int expert_norm;                  /* 1: RMS-normalise each expert output before the sum */
} orc_layer;

/* RMS normalisation of an expert output before the weighted sum, eps 1e-6,
 * no learned scale. Reading of "Muse Spark normalises each expert's output,
 * then combines" ("TensorSharp Muse Spark benchmark", section "Performance"). */
#define ORC_EXPERT_NORM_EPS 1e-6

/* ------------------------------------------------------------------------- */
/* number formats                                                             */
/* ------------------------------------------------------------------------- */

double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* round-to-nearest-even fp32 -> bf16 */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* nearest integer of a non-negative double, exact halves to the even integer */
static double rne_nonneg(double q)
{
    double f = floor(q);
    double frac = q - f;
    if (frac > 0.5)
        return f + 1.0;
    if (frac < 0.5)
        return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * Exponent field 0 is subnormal: 0.5 * m. */
float orc_e2m1_decode(uint8_t c)
{
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    float mag = (e == 0) ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, e - 1);
    return s ? -mag : mag;
}

/* E4M3 (OCP FP8, no infinities): sign bit 7, exponent bits 6..3 (bias 7),
 * mantissa bits 2..0; exponent field 0 is subnormal m/8 * 2^-6; S.1111.111 is NaN. */
float orc_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    float mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexpf((float)m / 8.0f, -6);
    else
        mag = ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return s ? -mag : mag;
}

/* Nearest E2M1 code to v, exact ties to the even code, magnitudes above 6
 * saturate to 6. The sign bit copies the sign of v (so -0.1 gives code 8).
 * Written as a search over the 8 magnitudes: the definition, not a trick. */
uint8_t orc_e2m1_encode(float v)
{
    int neg = signbit(v) ? 1 : 0;
    float a = fabsf(v);
    int best = 0;
    float bestd = INFINITY;
    for (int c = 0; c < 8; ++c) {
        float dd = fabsf(a - orc_e2m1_decode((uint8_t)c));
        if (dd < bestd || (dd == bestd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bestd = dd;
        }
    }
    return (uint8_t)((neg << 3) | best);
}

/* Nearest E4M3 code to a non-negative v, ties to even mantissa, values at or
 * above 448 (the largest finite E4M3) saturate to 448. */
uint8_t orc_e4m3_encode(float v)
{
    if (!(v > 0.0f))
        return 0;
    if (v >= 448.0f)
        return 0x7E;
    int ex;
    double fr = frexp((double)v, &ex);   /* v = fr * 2^ex, fr in [0.5, 1) */
    int E = ex - 1;                      /* v = (2 fr) * 2^E */
    if (E < -6) {                        /* subnormal range: multiples of 2^-9 */
        double r = rne_nonneg(ldexp((double)v, 9));
        return (uint8_t)r;               /* r == 8 is code 0x08 = 2^-6 */
    }
    double r = rne_nonneg((2.0 * fr - 1.0) * 8.0);
    if (r == 8.0) {
        r = 0.0;
        E += 1;
    }
    int code = ((E + 7) << 3) | (int)r;
    if (code > 0x7E)
        code = 0x7E;
    return (uint8_t)code;
}

/* NVFP4 quantiser for one tensor W[rows, K] (bf16), blocks of 16 along K:
 *   s_t   = amax|W| / (6 * 448)            (1 if W is all zero)
 *   s_b   = E4M3( (amax_block / 6) / s_t )
 *   code  = E2M1( w / (E4M3dec(s_b) * s_t) ), 0 where that scale is 0
 * All in fp32, as the CUDA quantiser computes it. */
void orc_quantize_nvfp4(const uint16_t *W, int rows, int K, uint8_t *q, uint8_t *s, float *g)
{
    float amax = 0.0f;
    for (long long i = 0; i < (long long)rows * K; ++i) {
        float a = fabsf((float)orc_bf16_to_double(W[i]));
        if (a > amax)
            amax = a;
    }
    float st = (amax > 0.0f) ? amax / 2688.0f : 1.0f;
    *g = st;
    int nb = K / 16;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        for (int b = 0; b < nb; ++b) {
            const uint16_t *blk = W + (long long)r * K + b * 16;
            float bmax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float a = fabsf((float)orc_bf16_to_double(blk[i]));
                if (a > bmax)
                    bmax = a;
            }
            float sbf = (bmax / 6.0f) / st;
            uint8_t sc = orc_e4m3_encode(sbf);
            s[(long long)r * nb + b] = sc;
            float scale = orc_e4m3_decode(sc) * st;
            uint8_t codes[16];
            for (int i = 0; i < 16; ++i) {
                float w = (float)orc_bf16_to_double(blk[i]);
                codes[i] = (scale == 0.0f) ? 0 : orc_e2m1_encode(w / scale);
            }
            uint8_t *qo = q + (long long)r * (K / 2) + b * 8;
            for (int i = 0; i < 8; ++i)
                qo[i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
        }
    }
}

/* w = (E2M1(code) * E4M3(scale)) * s_t in fp32 (the first product is exact) */
void orc_dequant_nvfp4_row(const uint8_t *q, const uint8_t *s, float g, int K, float *out)
{
    for (int c = 0; c < K; ++c) {
        uint8_t byte = q[c / 2];
        uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
        float v = orc_e2m1_decode(code) * orc_e4m3_decode(s[c / 16]);
        out[c] = v * g;
    }
}

/* ------------------------------------------------------------------------- */
/* routing                                                                    */
/* ------------------------------------------------------------------------- */

/* Router: logits in double, rounded once to fp32, bias added in fp32. */
void orc_router_logits(const uint16_t *x, const uint16_t *wr, const float *bias,
                       int T, int d, int E, float *logits)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += orc_bf16_to_double(x[(long long)t * d + c]) *
                       orc_bf16_to_double(wr[(long long)e * d + c]);
            float l = (float)acc;
            if (bias)
                l = l + bias[e];
            logits[(long long)t * E + e] = l;
        }
    }
}

typedef struct {
    double p;
    int e;
} pe_pair;

static int cmp_p_desc_e_asc(const void *a, const void *b)
{
    const pe_pair *x = (const pe_pair *)a, *y = (const pe_pair *)b;
    if (x->p > y->p)
        return -1;
    if (x->p < y->p)
        return 1;
    return (x->e < y->e) ? -1 : (x->e > y->e);
}

/* softmax over all E in double */
static void softmax_row(const float *l, int E, double *p)
{
    double m = -INFINITY;
    for (int e = 0; e < E; ++e)
        if ((double)l[e] > m)
            m = (double)l[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) {
        p[e] = exp((double)l[e] - m);
        z += p[e];
    }
    for (int e = 0; e < E; ++e)
        p[e] /= z;
}

/* Top-k by a full sort of all E experts on (p descending, id ascending), then
 * renormalise the k kept probabilities to sum to 1. gap[t] is the fp32 logit
 * of the k-th kept expert minus that of the best expert left out (+inf when
 * k == E). */
void orc_select_topk(const float *logits, int T, int E, int k,
                     int32_t *ids, double *w, double *gap)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (long long)t * E;
        double *p = (double *)malloc(sizeof(double) * E);
        pe_pair *pr = (pe_pair *)malloc(sizeof(pe_pair) * E);
        softmax_row(l, E, p);
        for (int e = 0; e < E; ++e) {
            pr[e].p = p[e];
            pr[e].e = e;
        }
        qsort(pr, (size_t)E, sizeof(pe_pair), cmp_p_desc_e_asc);
        double s = 0.0;
        for (int j = 0; j < k; ++j)
            s += pr[j].p;
        for (int j = 0; j < k; ++j) {
            ids[(long long)t * k + j] = pr[j].e;
            w[(long long)t * k + j] = pr[j].p / s;
        }
        if (gap)
            gap[t] = (k < E) ? (double)l[pr[k - 1].e] - (double)l[pr[k].e] : INFINITY;
        free(p);
        free(pr);
    }
}

/* Renormalised weights for a given (forced) expert set: p(ids_j) / sum p(ids). */
void orc_weights_for_ids(const float *logits, int T, int E, int k, const int32_t *ids, double *w)
{
    double *p = (double *)malloc(sizeof(double) * E);
    for (int t = 0; t < T; ++t) {
        softmax_row(logits + (long long)t * E, E, p);
        double s = 0.0;
        for (int j = 0; j < k; ++j)
            s += p[ids[(long long)t * k + j]];
        for (int j = 0; j < k; ++j)
            w[(long long)t * k + j] = p[ids[(long long)t * k + j]] / s;
    }
    free(p);
}

/* Token permutation: counts per expert, exclusive prefix sum, then a stable
 * counting sort that walks tokens in ascending order, so the rows of every
 * expert hold its tokens in ascending token order. pos[t,j] is the row of
 * (token t, slot j) in the permuted order. */
void orc_permute(const int32_t *ids, int T, int k, int E,
                 int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *pos)
{
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (long long i = 0; i < (long long)T * k; ++i)
        counts[ids[i]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int e = ids[(long long)t * k + j];
            int r = offsets[e] + fill[e];
            fill[e] += 1;
            perm[r] = t;
            pos[(long long)t * k + j] = r;
        }
    }
    free(fill);
}

/* ------------------------------------------------------------------------- */
/* expert FFN and combine                                                     */
/* ------------------------------------------------------------------------- */

/* One row of an expert matrix as doubles. which: 0 gate, 1 up, 2 down. */
static void weight_row(const orc_layer *L, int which, int e, int row, double *out, float *tmp)
{
    int K = (which == 2) ? L->I : L->d;
    int rows = (which == 2) ? L->d : L->I;
    long long idx = (long long)e * rows + row;
    if (L->fmt == 0) {
        const uint16_t *base = which == 0 ? L->w_gate : which == 1 ? L->w_up : L->w_down;
        const uint16_t *src = base + idx * K;
        for (int c = 0; c < K; ++c)
            out[c] = orc_bf16_to_double(src[c]);
    } else {
        const uint8_t *qb = which == 0 ? L->q_gate : which == 1 ? L->q_up : L->q_down;
        const uint8_t *sb = which == 0 ? L->s_gate : which == 1 ? L->s_up : L->s_down;
        const float *gb = which == 0 ? L->g_gate : which == 1 ? L->g_up : L->g_down;
        orc_dequant_nvfp4_row(qb + idx * (K / 2), sb + idx * (K / 16), gb[e], K, tmp);
        for (int c = 0; c < K; ++c)
            out[c] = (double)tmp[c];
    }
}

/* SwiGLU expert e on one token: h[i] = silu(Wg[e,i,:].x) * (Wu[e,i,:].x),
 * Y[c] = Wd[e,c,:].h, all in double. */
void orc_expert_ffn(const orc_layer *L, int e, const uint16_t *x_row, double *h, double *Y)
{
    int d = L->d, I = L->I;
    int K = d > I ? d : I;
    double *xr = (double *)malloc(sizeof(double) * d);
    double *row = (double *)malloc(sizeof(double) * K);
    float *tmp = (float *)malloc(sizeof(float) * K);
    for (int c = 0; c < d; ++c)
        xr[c] = orc_bf16_to_double(x_row[c]);
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        weight_row(L, 0, e, i, row, tmp);
        for (int c = 0; c < d; ++c)
            g += row[c] * xr[c];
        weight_row(L, 1, e, i, row, tmp);
        for (int c = 0; c < d; ++c)
            u += row[c] * xr[c];
        h[i] = g / (1.0 + exp(-g)) * u;
    }
    for (int c = 0; c < d; ++c) {
        double acc = 0.0;
        weight_row(L, 2, e, c, row, tmp);
        for (int i = 0; i < I; ++i)
            acc += row[i] * h[i];
        Y[c] = acc;
    }
    free(xr);
    free(row);
    free(tmp);
}

/* Full layer for a list of tokens (all T when tokens == NULL).
 * forced_ids: NULL, or [T, k] expert ids to use instead of the oracle's own
 * selection (weights then follow orc_weights_for_ids). Outputs are per listed
 * token: ids_out, w_out [n, k], gap_out [n], Y_out [n, k, d] (may be NULL),
 * y_out [n, d]. */
void orc_forward(const orc_layer *L, const uint16_t *x, int T,
                 const int32_t *tokens, int n, const int32_t *forced_ids,
                 int32_t *ids_out, double *w_out, double *gap_out,
                 double *Y_out, double *y_out)
{
    int d = L->d, E = L->E, k = L->k;
    if (!tokens)
        n = T;
    float *lg = (float *)malloc(sizeof(float) * (size_t)n * E);
    uint16_t *xs = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)n * d);
    for (int a = 0; a < n; ++a) {
        int t = tokens ? tokens[a] : a;
        memcpy(xs + (long long)a * d, x + (long long)t * d, sizeof(uint16_t) * d);
    }
    orc_router_logits(xs, L->w_router, L->router_bias, n, d, E, lg);
    orc_select_topk(lg, n, E, k, ids_out, w_out, gap_out);
    if (forced_ids) {
        for (int a = 0; a < n; ++a) {
            int t = tokens ? tokens[a] : a;
            for (int j = 0; j < k; ++j)
                ids_out[(long long)a * k + j] = forced_ids[(long long)t * k + j];
        }
        orc_weights_for_ids(lg, n, E, k, ids_out, w_out);
    }
    double *Yall = Y_out ? Y_out : (double *)malloc(sizeof(double) * (size_t)n * k * d);
#pragma omp parallel for schedule(dynamic, 1)
    for (long long item = 0; item < (long long)n * k; ++item) {
        int a = (int)(item / k);
        double *h = (double *)malloc(sizeof(double) * L->I);
        orc_expert_ffn(L, ids_out[item], xs + (long long)a * d, h, Yall + item * d);
        free(h);
    }
    /* per-slot factor: 1, or 1 / sqrt(mean(Y^2) + eps) when normalising */
    double *fac = (double *)malloc(sizeof(double) * (size_t)n * k);
    for (long long item = 0; item < (long long)n * k; ++item) {
        fac[item] = 1.0;
        if (L->expert_norm) {
            double ss = 0.0;
            for (int c = 0; c < d; ++c)
                ss += Yall[item * d + c] * Yall[item * d + c];
            fac[item] = 1.0 / sqrt(ss / d + ORC_EXPERT_NORM_EPS);
        }
    }
    for (int a = 0; a < n; ++a) {
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j)
                acc += w_out[(long long)a * k + j] * (Yall[((long long)a * k + j) * d + c] * fac[(long long)a * k + j]);
            y_out[(long long)a * d + c] = acc;
        }
    }
    free(fac);
    if (!Y_out)
        free(Yall);
    free(lg);
    free(xs);
}

/* ------------------------------------------------------------------------- */
/* pre-norm and residual between stacked layers                              */
/* ------------------------------------------------------------------------- */

/* u = x / sqrt(mean(x^2) + eps), no learned scale, double -> fp32 -> bf16.
 * The page on the TPU megakernel ("Key optimisations") places a norm after
 * the 62 layers; the stacked workload puts one before every layer. */
void orc_rmsnorm(const uint16_t *x, int T, int d, double eps, uint16_t *u)
{
    for (int t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int c = 0; c < d; ++c) {
            double v = orc_bf16_to_double(x[(long long)t * d + c]);
            ss += v * v;
        }
        double r = 1.0 / sqrt(ss / d + eps);
        for (int c = 0; c < d; ++c)
            u[(long long)t * d + c] =
                orc_f32_to_bf16((float)(orc_bf16_to_double(x[(long long)t * d + c]) * r));
    }
}

/* x_next = bf16( fp32( x + y ) ) */
void orc_residual_add(const uint16_t *x, const double *y, long long n, uint16_t *out)
{
    for (long long i = 0; i < n; ++i)
        out[i] = orc_f32_to_bf16((float)(orc_bf16_to_double(x[i]) + y[i]));
}

/* ------------------------------------------------------------------------- */

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
