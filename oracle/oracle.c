/*
 * oracle.c -- plain, slow, single-threaded CPU oracle for the routed-expert
 * MoE layer and the Engram gather-decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load this library.  It shares no code,
 * header, table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * Sources (page title, then section):
 *   [I]  strix-llama.cpp issue "Feature Request: support DeepSeek V4.1 Flash
 *        with bounded SSD expert caching"
 *   [S]  Strata-DSV4.1 README
 *   [V]  vllm.cpp PR "DeepSeek-V4-Flash-Vision tower" (device MoE router notes)
 *
 * Readings taken where the pages are silent (each listed in the design notes):
 *   R1  router logit order "LANE32": 32 partial sums, partial j accumulates
 *       fmaf over c = j, j+32, ... in ascending c from +0.0f, then a butterfly
 *       p_j <- p_j + p_(j xor o) for o = 16, 8, 4, 2, 1; z = p_0.
 *   R2  s = 1 / (1 + e) in float, e = exp(-z) by Cody-Waite range reduction
 *       (n = rint(x * log2 e), r = x - n*ln2 in two float parts) and the
 *       degree-7 Taylor polynomial of exp(r) in Horner form with fmaf; x is
 *       clamped below at -30 (there 1 + e == 1) and x > 88 gives s = 0.  Every
 *       step is one IEEE float operation, so any conforming machine gets the
 *       same bits.
 *   R3  key = s + b (float); order by key descending, id ascending; a NaN key
 *       ranks below every number.
 *   R4  S = (((s_0 + s_1) + s_2) + ...) in slot order; w_j = s_j / S.
 *   R5  stable counting sort of pair ids p = t*k + j by expert id.
 *   R6  FFN in FP64 on exactly dequantised weights, no SwiGLU clamp.
 *   R10 Engram head sum: acc = v_0, then acc = acc + v_h (float), h ascending.
 *   R12 router variant score s = sqrt(softplus(z)) in float (see or_sqrt_softplus).
 *   Q2_K code packing: code i = (qs[i/4] >> 2*(i%4)) & 3; sub-block j holds
 *       weights 16j..16j+15 (the field order is given, the bit packing is not).
 *   Q8_0 field order: fp16 d first, then int8 q[32].
 *   Layer-stack norm: weight-free RMS norm with a LANE32 sum of squares,
 *       eps = 1e-6, r = 1/sqrtf(mean + eps), u = bf16(x * r).
 *
 * Built with -ffp-contract=off so that no multiply-add is fused except where
 * fmaf() is written out.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "oracle.h"

/* ------------------------------------------------------------------------- */
/* scalar formats                                                             */
/* ------------------------------------------------------------------------- */

/* IEEE binary16 -> float (exact). */
float or_f16_to_f32(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    float v;
    if (e == 0)
        v = ldexpf((float)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexpf((float)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return s ? -v : v;
}

float or_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* float -> bf16, round to nearest even; NaN -> canonical 0x7FC0. */
uint16_t or_bf16_rne(float f)
{
    uint32_t u;
    if (isnan(f))
        return 0x7FC0;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* double -> bf16 with a single rounding: round to float with round-to-odd
 * (24 bits >= 8 + 2), then float -> bf16 to nearest even. */
uint16_t or_bf16_rne_f64(double x)
{
    float f;
    uint32_t u;
    if (isnan(x))
        return 0x7FC0;
    f = (float)x;
    if ((double)f != x && !isinf(x)) {
        if (fabs((double)f) > fabs(x))
            f = nextafterf(f, 0.0f);
        memcpy(&u, &f, 4);
        u |= 1u;
        memcpy(&f, &u, 4);
    }
    return or_bf16_rne(f);
}

/* OCP FP8 E4M3: bias 7, no infinity, S.1111.111 is NaN. */
float or_e4m3_to_f32(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    float v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexpf((float)m, -9);                  /* m/8 * 2^-6 */
    else
        v = ldexpf((float)(8 + m), e - 10);        /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* E8M0 scale: 2^(e-127); 0xFF is NaN. */
float or_e8m0_to_f32(uint8_t e)
{
    if (e == 255)
        return NAN;
    return ldexpf(1.0f, (int)e - 127);
}

/* ------------------------------------------------------------------------- */
/* block formats                                                              */
/* ------------------------------------------------------------------------- */

/* Q2_K: 84 bytes per 256 weights -- scales[16], qs[64], fp16 d, fp16 dmin.
 * w_i = (d * sc_j) * q_i - dmin * m_j, j = i / 16, sc_j = scales[j] & 15,
 * m_j = scales[j] >> 4.  Every product is exact in float, so the one rounding
 * is the subtraction. */
void or_dequant_q2k(const uint8_t *blk, int64_t nblk, float *out)
{
    for (int64_t b = 0; b < nblk; ++b) {
        const uint8_t *p = blk + b * 84;
        float d = or_f16_to_f32((uint16_t)(p[80] | (p[81] << 8)));
        float dmin = or_f16_to_f32((uint16_t)(p[82] | (p[83] << 8)));
        for (int i = 0; i < 256; ++i) {
            int j = i / 16;
            int sc = p[j] & 15, m = p[j] >> 4;
            int q = (p[16 + i / 4] >> (2 * (i % 4))) & 3;
            float a = (d * (float)sc) * (float)q;
            float c = dmin * (float)m;
            out[b * 256 + i] = a - c;
        }
    }
}

/* Q8_0: 34 bytes per 32 weights -- fp16 d, int8 q[32]; w_i = d * q_i. */
void or_dequant_q8_0(const uint8_t *blk, int64_t nblk, float *out)
{
    for (int64_t b = 0; b < nblk; ++b) {
        const uint8_t *p = blk + b * 34;
        float d = or_f16_to_f32((uint16_t)(p[0] | (p[1] << 8)));
        for (int i = 0; i < 32; ++i)
            out[b * 32 + i] = d * (float)(int8_t)p[2 + i];
    }
}

/* ------------------------------------------------------------------------- */
/* Engram gather-decode ([I] "Feature Description": 264-byte rows of 256 E4M3   */
/* values and 8 E8M0 scales; "DeepSeek V4.1 Engram graph integration": rows per */
/* token gathered from the layer's table)                                      */
/* ------------------------------------------------------------------------- */

/* out[t][tau*256 + c] = bf16(sum_h e4m3(row[c]) * e8m0(row[256 + c/32])),
 * rows = table_tau[ids[t][tau][h]].  An id outside [0, n_rows) decodes as +0
 * and sets bit 2 of *err. */
void or_engram_gather(const uint8_t *const *tables, const int64_t *n_rows, int n_tables,
                      const int64_t *ids, int T, int H, uint16_t *out, int32_t *err)
{
    for (int t = 0; t < T; ++t)
        for (int tau = 0; tau < n_tables; ++tau)
            for (int c = 0; c < 256; ++c) {
                float acc = 0.0f;
                for (int h = 0; h < H; ++h) {
                    int64_t r = ids[((int64_t)t * n_tables + tau) * H + h];
                    float v;
                    if (r < 0 || r >= n_rows[tau]) {
                        v = 0.0f;
                        if (err)
                            *err |= 2;
                    } else {
                        const uint8_t *row = tables[tau] + r * 264;
                        v = or_e4m3_to_f32(row[c]) * or_e8m0_to_f32(row[256 + c / 32]);
                    }
                    acc = (h == 0) ? v : acc + v;
                }
                out[((int64_t)t * n_tables + tau) * 256 + c] = or_bf16_rne(acc);
            }
}

/* ------------------------------------------------------------------------- */
/* router ([S] "Results": selection-only route bias, mixing weights exact;     */
/* [V] router notes: weights gathered from the unbiased scores)                */
/* ------------------------------------------------------------------------- */

/* R1: LANE32 logit of one (token, expert). */
static float lane32_dot(const uint16_t *x, const float *wr, int d, int E, int e)
{
    float p[32], q[32];
    for (int j = 0; j < 32; ++j) {
        p[j] = 0.0f;
        for (int c = j; c < d; c += 32)
            p[j] = fmaf(or_bf16_to_f32(x[c]), wr[(int64_t)c * E + e], p[j]);
    }
    for (int o = 16; o >= 1; o >>= 1) {
        for (int j = 0; j < 32; ++j)
            q[j] = p[j] + p[j ^ o];
        memcpy(p, q, sizeof p);
    }
    return p[0];
}

/* R2: the router's sigmoid (see the header comment). */
float or_sigmoid(float z)
{
    const float LOG2E = 1.44269504088896341f;
    const float LN2_HI = 0.693359375f;              /* 355/512: n * LN2_HI is exact */
    const float LN2_LO = -2.12194440054690583e-4f;  /* ln 2 - LN2_HI */
    float x = -z;
    if (isnan(x))
        return x;
    if (x > 88.0f)
        return 0.0f;
    if (x < -30.0f)
        x = -30.0f;
    float n = rintf(x * LOG2E);
    float r = fmaf(-n, LN2_HI, x);
    r = fmaf(-n, LN2_LO, r);
    /* exp(r) = sum r^k / k!, k = 0..7 */
    float p = 1.0f / 5040.0f;
    p = fmaf(p, r, 1.0f / 720.0f);
    p = fmaf(p, r, 1.0f / 120.0f);
    p = fmaf(p, r, 1.0f / 24.0f);
    p = fmaf(p, r, 1.0f / 6.0f);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    float e = ldexpf(p, (int)n);
    return 1.0f / (1.0f + e);
}

/* R3: does (ka, ia) rank before (kb, ib)? */
static int ranks_before(float ka, int ia, float kb, int ib)
{
    int na = isnan(ka), nb = isnan(kb);
    if (na != nb)
        return !na;
    if (!na && ka != kb)
        return ka > kb;
    return ia < ib;
}

void or_route(const uint16_t *x, const float *wr, const float *bias, int T, int d, int E, int k,
              int32_t *ids, float *w, float *z_out, float *s_out)
{
    float *s = (float *)malloc(sizeof(float) * (size_t)E);
    float *key = (float *)malloc(sizeof(float) * (size_t)E);
    int *used = (int *)malloc(sizeof(int) * (size_t)E);
    for (int t = 0; t < T; ++t) {
        const uint16_t *xt = x + (int64_t)t * d;
        for (int e = 0; e < E; ++e) {
            float z = lane32_dot(xt, wr, d, E, e);
            s[e] = or_sigmoid(z);                                        /* R2 */
            key[e] = s[e] + (bias ? bias[e] : 0.0f);                 /* R3 */
            used[e] = 0;
            if (z_out)
                z_out[(int64_t)t * E + e] = z;
            if (s_out)
                s_out[(int64_t)t * E + e] = s[e];
        }
        /* top-k by repeated selection of the best unused expert */
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!used[e] && (best < 0 || ranks_before(key[e], e, key[best], best)))
                    best = e;
            used[best] = 1;
            ids[t * k + j] = best;
        }
        /* R4: weights from the unbiased scores, sum in slot order */
        float S = 0.0f;
        for (int j = 0; j < k; ++j)
            S = (j == 0) ? s[ids[t * k]] : S + s[ids[t * k + j]];
        for (int j = 0; j < k; ++j)
            w[t * k + j] = s[ids[t * k + j]] / S;
    }
    free(s);
    free(key);
    free(used);
}

/* ------------------------------------------------------------------------- */
/* router variants ([V] device router notes, the per-row rule of               */
/* "SqrtSoftplusRouteTopk")                                                    */
/* ------------------------------------------------------------------------- */

/* R12: exp(x) for -87 <= x <= 0 in float, every step one IEEE operation: Cody-Waite reduction
 * n = rint(x log2 e), r = x - n ln2 (two float parts), the degree-7 Taylor polynomial of exp(r)
 * in Horner form with fmaf, scaled by 2^n (n >= -126, so the scaling is exact). */
static float or_exp_neg(float x)
{
    const float LOG2E = 1.44269504088896341f;
    const float LN2_HI = 0.693359375f;
    const float LN2_LO = -2.12194440054690583e-4f;
    float n = rintf(x * LOG2E);
    float r = fmaf(-n, LN2_HI, x);
    r = fmaf(-n, LN2_LO, r);
    float p = 1.0f / 5040.0f;
    p = fmaf(p, r, 1.0f / 720.0f);
    p = fmaf(p, r, 1.0f / 120.0f);
    p = fmaf(p, r, 1.0f / 24.0f);
    p = fmaf(p, r, 1.0f / 6.0f);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    return ldexpf(p, (int)n);
}

/* R12: s = sqrt(softplus(z)) in float.  softplus(z) = max(z, 0) + log1p(exp(-|z|)); e =
 * exp(-|z|) as above (|z| > 87: e = 0); log1p(e) = 2 atanh(u) with u = e / (2 + e) <= 1/3, as
 * 2u (1 + v/3 + v^2/5 + ... + v^7/15), v = u^2, Horner with fmaf; then sqrtf.  Every step is one
 * IEEE float operation. */
float or_sqrt_softplus(float z)
{
    if (isnan(z))
        return z;
    const float a = fabsf(z);
    const float e = (a > 87.0f) ? 0.0f : or_exp_neg(-a);
    const float u = e / (2.0f + e);
    const float v = u * u;
    float q = 1.0f / 15.0f;
    q = fmaf(q, v, 1.0f / 13.0f);
    q = fmaf(q, v, 1.0f / 11.0f);
    q = fmaf(q, v, 1.0f / 9.0f);
    q = fmaf(q, v, 1.0f / 7.0f);
    q = fmaf(q, v, 1.0f / 5.0f);
    q = fmaf(q, v, 1.0f / 3.0f);
    q = fmaf(q, v, 1.0f);
    const float l = 2.0f * (u * q);
    const float sp = (z > 0.0f ? z : 0.0f) + l;
    return sqrtf(sp);
}

/* Router with the per-row rule of the device router notes ([V]):
 *   score_fn 0: s = or_sigmoid(z) (R2); 1: s = or_sqrt_softplus(z) (R12).
 *   Row t is media when vbias and media are both given and media[t] != 0; a media row's key is
 *   s + vbias, a text row's s + bias (bias NULL: 0).  Selection as R3.
 *   tid2eid [vocab][k] (or NULL) with tok [T]: on such a hash layer a TEXT row's ids are
 *   tid2eid[tok[t]][0..k) in table order (no key, no bias); media rows select as above.
 *   Weights (R4) from the unbiased s of the row's ids, S in slot order.
 *   Hash rows: tok[t] outside [0, vocab) sets err bit 2 and gives ids -1, weights 0; a table id
 *   outside [0, E) sets err bit 1, is written as it is, and counts s = 0. */
void or_route_ex(const uint16_t *x, const float *wr, const float *bias, int T, int d, int E, int k,
                 int score_fn, const float *vbias, const uint8_t *media, const int32_t *tid2eid,
                 const int32_t *tok, int vocab, int32_t *ids, float *w, int32_t *err)
{
    float *s = (float *)malloc(sizeof(float) * (size_t)E);
    float *key = (float *)malloc(sizeof(float) * (size_t)E);
    int *used = (int *)malloc(sizeof(int) * (size_t)E);
    float sel[64];
    for (int t = 0; t < T; ++t) {
        const uint16_t *xt = x + (int64_t)t * d;
        const int is_media = vbias && media && media[t] != 0;
        const float *rb = is_media ? vbias : bias;
        for (int e = 0; e < E; ++e) {
            float z = lane32_dot(xt, wr, d, E, e);
            s[e] = score_fn == 1 ? or_sqrt_softplus(z) : or_sigmoid(z);
            key[e] = s[e] + (rb ? rb[e] : 0.0f);
            used[e] = 0;
        }
        int32_t *it = ids + (int64_t)t * k;
        float *wt = w + (int64_t)t * k;
        if (tid2eid && !is_media) {
            if (tok[t] < 0 || tok[t] >= vocab) {
                *err |= 2;
                for (int j = 0; j < k; ++j) {
                    it[j] = -1;
                    wt[j] = 0.0f;
                }
                continue;
            }
            for (int j = 0; j < k; ++j) {
                const int32_t id = tid2eid[(int64_t)tok[t] * k + j];
                it[j] = id;
                if (id < 0 || id >= E) {
                    *err |= 1;
                    sel[j] = 0.0f;
                } else {
                    sel[j] = s[id];
                }
            }
        } else {
            for (int j = 0; j < k; ++j) {
                int best = -1;
                for (int e = 0; e < E; ++e)
                    if (!used[e] && (best < 0 || ranks_before(key[e], e, key[best], best)))
                        best = e;
                used[best] = 1;
                it[j] = best;
                sel[j] = s[best];
            }
        }
        float S = 0.0f;
        for (int j = 0; j < k; ++j)
            S = (j == 0) ? sel[0] : S + sel[j];
        for (int j = 0; j < k; ++j)
            wt[j] = sel[j] / S;
    }
    free(s);
    free(key);
    free(used);
}

/* ------------------------------------------------------------------------- */
/* permutation ([S] DSpark verify: the union of the pass's experts served once */
/* per layer; [I] expert store: request-union planning)                        */
/* ------------------------------------------------------------------------- */

/* R5.  Pairs whose id lies outside [0, E) are kept after every group, in pair
 * order (offsets[E] counts valid pairs only), and set bit 1 of *err. */
void or_permute(const int32_t *ids, int T, int k, int E, int32_t *offsets, int32_t *perm,
                int32_t *inv, int32_t *active, int32_t *n_active, int32_t *err)
{
    int P = T * k;
    int32_t *fill = (int32_t *)calloc((size_t)E + 1, sizeof(int32_t));
    for (int e = 0; e <= E; ++e)
        offsets[e] = 0;
    for (int p = 0; p < P; ++p) {
        int e = ids[p];
        if (e >= 0 && e < E)
            offsets[e + 1]++;
        else if (err)
            *err |= 1;
    }
    for (int e = 0; e < E; ++e)
        offsets[e + 1] += offsets[e];
    int bad = offsets[E];
    for (int p = 0; p < P; ++p) {
        int e = ids[p];
        int pos = (e >= 0 && e < E) ? offsets[e] + fill[e]++ : bad++;
        perm[pos] = p;
        inv[p] = pos;
    }
    int na = 0;
    for (int e = 0; e < E; ++e)
        if (offsets[e + 1] > offsets[e])
            active[na++] = e;
    for (int a = na; a < E; ++a)
        active[a] = -1;
    *n_active = na;
    free(fill);
}

/* ------------------------------------------------------------------------- */
/* expert FFN ([S] "Verifying it": expert tier against a dequantised F32       */
/* reference; V4-Flash "How fast is it?": SwiGLU)                              */
/* ------------------------------------------------------------------------- */

static double *dequant_matrix_f64(int fmt, const uint8_t *bytes, int rows, int cols)
{
    int64_t n = (int64_t)rows * cols;
    float *f = (float *)malloc(sizeof(float) * (size_t)n);
    double *m = (double *)malloc(sizeof(double) * (size_t)n);
    if (fmt == OR_FMT_Q2_K)
        or_dequant_q2k(bytes, n / 256, f);
    else
        or_dequant_q8_0(bytes, n / 32, f);
    for (int64_t i = 0; i < n; ++i)
        m[i] = (double)f[i];
    free(f);
    return m;
}

/* y[i][:] = down * (silu(gate * x_i) .* (up * x_i)) in FP64 for n rows x_i.
 * gate, up: [F][d]; down: [d][F]; quant blocks run along the inner axis. */
void or_expert_ffn(int fmt, const uint8_t *gate, const uint8_t *up, const uint8_t *down, int d, int F,
                   const uint16_t *xs, int n, double *y)
{
    double *G = dequant_matrix_f64(fmt, gate, F, d);
    double *U = dequant_matrix_f64(fmt, up, F, d);
    double *D = dequant_matrix_f64(fmt, down, d, F);
    double *xv = (double *)malloc(sizeof(double) * (size_t)d);
    double *h = (double *)malloc(sizeof(double) * (size_t)F);
    for (int i = 0; i < n; ++i) {
        for (int c = 0; c < d; ++c)
            xv[c] = (double)or_bf16_to_f32(xs[(int64_t)i * d + c]);
        for (int r = 0; r < F; ++r) {
            double g = 0.0, u = 0.0;
            const double *gr = G + (int64_t)r * d, *ur = U + (int64_t)r * d;
            for (int c = 0; c < d; ++c) {
                g += gr[c] * xv[c];
                u += ur[c] * xv[c];
            }
            h[r] = g / (1.0 + exp(-g)) * u;
        }
        for (int o = 0; o < d; ++o) {
            double acc = 0.0;
            const double *dr = D + (int64_t)o * F;
            for (int r = 0; r < F; ++r)
                acc += dr[r] * h[r];
            y[(int64_t)i * d + o] = acc;
        }
    }
    free(G);
    free(U);
    free(D);
    free(xv);
    free(h);
}

/* ------------------------------------------------------------------------- */
/* one MoE layer: route, run each selected expert once over its tokens, add    */
/* the always-on shared expert, mix with the renormalised weights ([S] "How it */
/* works", step 4: shared expert plus routed sum)                              */
/* ------------------------------------------------------------------------- */

/* gate_e/up_e/down_e: host arrays of E pointers to each routed expert's bytes
 * (an unselected expert may be NULL).  sh_*: shared expert (Q8_0) or NULL when
 * F_shared == 0.  out: BF16 [T][d]; out_f64 (optional): the value before the
 * final rounding.  ids/w (optional outputs, [T][k]).  Returns 0, or -1 when a
 * selected expert's pointer is NULL. */
int or_moe_layer(const uint16_t *x, int T, int d, int E, int k, int F, const float *wr,
                 const float *bias, const uint8_t *const *gate_e, const uint8_t *const *up_e,
                 const uint8_t *const *down_e, const uint8_t *sh_gate, const uint8_t *sh_up,
                 const uint8_t *sh_down, int F_shared, uint16_t *out, double *out_f64,
                 int32_t *ids_out, float *w_out)
{
    int P = T * k, rc = 0;
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)P);
    float *w = (float *)malloc(sizeof(float) * (size_t)P);
    double *acc = (double *)calloc((size_t)T * d, sizeof(double));
    uint16_t *xs = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)T * d);
    double *y = (double *)malloc(sizeof(double) * (size_t)T * d);
    int *rows = (int *)malloc(sizeof(int) * (size_t)P);

    or_route(x, wr, bias, T, d, E, k, ids, w, NULL, NULL);
    if (F_shared > 0 && sh_gate) {
        or_expert_ffn(OR_FMT_Q8_0, sh_gate, sh_up, sh_down, d, F_shared, x, T, y);
        for (int64_t i = 0; i < (int64_t)T * d; ++i)
            acc[i] = y[i];
    }
    for (int e = 0; e < E; ++e) {
        int n = 0;
        for (int p = 0; p < P; ++p)
            if (ids[p] == e)
                rows[n++] = p;
        if (n == 0)
            continue;
        if (!gate_e[e] || !up_e[e] || !down_e[e]) {
            rc = -1;
            goto done;
        }
        for (int i = 0; i < n; ++i)
            memcpy(xs + (int64_t)i * d, x + (int64_t)(rows[i] / k) * d, sizeof(uint16_t) * (size_t)d);
        or_expert_ffn(OR_FMT_Q2_K, gate_e[e], up_e[e], down_e[e], d, F, xs, n, y);
        for (int i = 0; i < n; ++i) {
            int t = rows[i] / k;
            double wt = (double)w[rows[i]];
            for (int c = 0; c < d; ++c)
                acc[(int64_t)t * d + c] += wt * y[(int64_t)i * d + c];
        }
    }
    for (int64_t i = 0; i < (int64_t)T * d; ++i) {
        out[i] = or_bf16_rne_f64(acc[i]);
        if (out_f64)
            out_f64[i] = acc[i];
    }
    if (ids_out)
        memcpy(ids_out, ids, sizeof(int32_t) * (size_t)P);
    if (w_out)
        memcpy(w_out, w, sizeof(float) * (size_t)P);
done:
    free(ids);
    free(w);
    free(acc);
    free(xs);
    free(y);
    free(rows);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* layer-stack step (speculative verify batch through a stack of MoE layers,  */
/* [S] "Latest (2026-10-14)": one batched verify pass of 1 + 4 rows)           */
/* ------------------------------------------------------------------------- */

/* x_new = bf16(x + moe * scale), product then sum, each rounded to float. */
void or_residual(const uint16_t *x, const uint16_t *moe, int T, int d, float scale, uint16_t *x_new)
{
    for (int64_t i = 0; i < (int64_t)T * d; ++i) {
        float m = or_bf16_to_f32(moe[i]) * scale;
        x_new[i] = or_bf16_rne(or_bf16_to_f32(x[i]) + m);
    }
}

/* Weight-free RMS norm: LANE32 sum of squares (as R1 with w = x), mean by a
 * float division by d, r = 1 / sqrtf(mean + eps), u = bf16(x * r). */
void or_rmsnorm(const uint16_t *x, int T, int d, float eps, uint16_t *u)
{
    for (int t = 0; t < T; ++t) {
        const uint16_t *xt = x + (int64_t)t * d;
        float p[32], q[32];
        for (int j = 0; j < 32; ++j) {
            p[j] = 0.0f;
            for (int c = j; c < d; c += 32) {
                float v = or_bf16_to_f32(xt[c]);
                p[j] = fmaf(v, v, p[j]);
            }
        }
        for (int o = 16; o >= 1; o >>= 1) {
            for (int j = 0; j < 32; ++j)
                q[j] = p[j] + p[j ^ o];
            memcpy(p, q, sizeof p);
        }
        float mean = p[0] / (float)d;
        float r = 1.0f / sqrtf(mean + eps);
        for (int c = 0; c < d; ++c)
            u[(int64_t)t * d + c] = or_bf16_rne(or_bf16_to_f32(xt[c]) * r);
    }
}

/* ------------------------------------------------------------------------- */
/* Engram gate and residual injection ([I] "Placement"), in FP64               */
/* ------------------------------------------------------------------------- */

/* kv[t][n] = sum_c rows[t][c] * w[n][c] (FP64; rows and w BF16, w stored [N][K], rows of w are
 * the outputs).  The product of the gathered rows and engram_kv.weight. */
void or_engram_kv(const uint16_t *rows, const uint16_t *w, int T, int K, int N, double *kv)
{
    for (int t = 0; t < T; ++t) {
        const uint16_t *r = rows + (int64_t)t * K;
        for (int n = 0; n < N; ++n) {
            const uint16_t *wn = w + (int64_t)n * K;
            double acc = 0.0;
            for (int c = 0; c < K; ++c)
                acc += (double)or_bf16_to_f32(r[c]) * (double)or_bf16_to_f32(wn[c]);
            kv[(int64_t)t * N + n] = acc;
        }
    }
}

/* For every token t (mask NULL or mask[t] == 0) and branch h < 4, with key_h = kv[t][h W ..],
 * value = kv[t][4 W ..] (four keys, then the shared value, each width W):
 *   dot = sum_i r[h,i] qn[h,i] kn[h,i] key[h,i]
 *   dot *= 1/sqrt(mean(r[h,:]^2) + eps) * 1/sqrt(mean(key[h,:]^2) + eps) * 1/sqrt(W)
 *   gate = sigmoid(copysign(sqrt(max(|dot|, 1e-6)), dot))
 *   r[h,i] = bf16(r[h,i] + gate * bf16(value[i]))
 * in FP64 with one rounding to BF16 at each bf16(); masked tokens keep r unchanged.  resid is
 * [T][4][W] BF16, updated in place; gate_out [T][4] (or NULL) receives the gates (0 for masked
 * tokens). */
void or_engram_gate(const double *kv, uint16_t *resid, const float *qn, const float *kn, const uint8_t *mask,
                    int T, int W, double eps, double *gate_out)
{
    for (int t = 0; t < T; ++t) {
        const double *kvt = kv + (int64_t)t * 5 * W;
        for (int h = 0; h < 4; ++h) {
            uint16_t *r = resid + ((int64_t)t * 4 + h) * W;
            if (mask && mask[t]) {
                if (gate_out)
                    gate_out[t * 4 + h] = 0.0;
                continue;
            }
            const double *key = kvt + (int64_t)h * W;
            double dot = 0.0, rr = 0.0, kk = 0.0;
            for (int i = 0; i < W; ++i) {
                const double ri = (double)or_bf16_to_f32(r[i]);
                dot += ri * (double)qn[h * W + i] * (double)kn[h * W + i] * key[i];
                rr += ri * ri;
                kk += key[i] * key[i];
            }
            dot *= 1.0 / sqrt(rr / W + eps);
            dot *= 1.0 / sqrt(kk / W + eps);
            dot *= 1.0 / sqrt((double)W);
            const double m = sqrt(fabs(dot) > 1e-6 ? fabs(dot) : 1e-6);
            const double g = 1.0 / (1.0 + exp(-copysign(m, dot)));
            if (gate_out)
                gate_out[t * 4 + h] = g;
            const double *val = kvt + (int64_t)4 * W;
            for (int i = 0; i < W; ++i) {
                const double vb = (double)or_bf16_to_f32(or_bf16_rne_f64(val[i]));
                r[i] = or_bf16_rne_f64((double)or_bf16_to_f32(r[i]) + g * vb);
            }
        }
    }
}
