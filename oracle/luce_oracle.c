/*
 * luce_oracle.c -- plain, single-threaded CPU oracle of the routed-MoE FFN
 * decode step (Q8_0 experts x q8_1 activations) and of the greedy argmax.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path
 * (the CUDA library and its Python binding) never calls it, and the two
 * share no code, header, table or helper.
 *
 * Pages cited (by title):
 *   [PR826] Lucebox PR #826 "feat(ds41): two-box expert-parallel serving".
 *           Sections used: the commit "fused DS4.1 decode kernels" (router
 *           select+weights over the same logits, expert grouping, q8_1
 *           activation memo, column-range Q8_0 products, argmax pair/pick);
 *           the commit "fused routed combine and q8_1 inputs for the hybrid
 *           owners" (masked combine, clamped routed SwiGLU); the commit
 *           "RDNA4 Q8_0 gate/up pair" (gate and up products fused with the
 *           SwiGLU); the code review "moe_combine_masked_kernel indexes
 *           valid with an unchecked (possibly -1) route id" (masked ids).
 *   The Q8_0 / q8_1 block layouts are the ggml ones the pages name
 *   (block_q8_0 in the review of the whole-row-lane slice): 32 int8 values
 *   with an fp16 scale d (Q8_0, 34 B) and additionally an fp16 s = d*sum(q)
 *   (q8_1, 36 B).
 *
 * Precision.  Every accumulation whose precision the pages leave open (dot
 * products, SwiGLU, router softmax) is carried out in double.  Steps where a
 * floating-point value decides an integer (the q8_1 quantization) are done
 * in fp32, the precision of the quantized format's own definition.  The
 * route-weighted combine is done in fp32 with every product and every sum
 * rounded separately, because [PR826, commit "fused routed combine ..."]
 * states exactly that rounding.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared (no fast-math):
 * every float operation below is one IEEE operation, in program order.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define LO_QK 32
#define LO_Q8_0_BYTES 34
#define LO_Q8_1_BYTES 36
#define LO_QK_K 256       /* values of a Q4_K super-block */
#define LO_Q4_K_BYTES 144 /* d, dmin (fp16), 12 bytes of scales, 128 bytes of codes */

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary16 conversion, written from the format definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; subnormals
 * have exponent field 0 and value fraction * 2^-24.  Encoding rounds to
 * nearest, ties to even (the IEEE default rounding attribute).          */

uint16_t lo_fp16_encode(float f)
{
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t exp = (x >> 23) & 0xffu;
    uint32_t man = x & 0x7fffffu;

    if (exp == 0xffu) /* inf or nan */
        return (uint16_t)(sign | 0x7c00u | (man ? 0x200u : 0u));
    if (exp == 0u) /* fp32 zero or subnormal: below 2^-126, rounds to zero */
        return (uint16_t)sign;

    int e = (int)exp - 127; /* value = 1.man * 2^e */
    if (e > 15)
        return (uint16_t)(sign | 0x7c00u);
    if (e >= -14) {
        /* normal binary16: keep the top 10 of 23 fraction bits */
        uint32_t keep = man >> 13;
        uint32_t rest = man & 0x1fffu;
        uint32_t r = ((uint32_t)(e + 15) << 10) + keep;
        if (rest > 0x1000u || (rest == 0x1000u && (keep & 1u)))
            r += 1u; /* a carry out of the fraction bumps the exponent */
        if (r >= 0x7c00u)
            return (uint16_t)(sign | 0x7c00u);
        return (uint16_t)(sign | r);
    }
    /* subnormal binary16: count units of 2^-24.
     * value = mf * 2^(e-23) with mf = 1.man as a 24-bit integer, so the
     * number of 2^-24 units is mf * 2^(e+1) = mf >> shift, shift = -(e+1). */
    uint32_t mf = man | 0x800000u;
    int shift = -(e + 1); /* >= 14 here */
    if (shift > 24)
        return (uint16_t)sign; /* below half a unit: rounds to zero */
    uint32_t q = mf >> shift;
    uint32_t rem = mf & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u)))
        q += 1u; /* may reach 0x400, the smallest normal: still correct */
    return (uint16_t)(sign | q);
}

float lo_fp16_decode(uint16_t h)
{
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t exp = (h >> 10) & 0x1fu;
    uint32_t man = h & 0x3ffu;
    uint32_t bits;
    if (exp == 0u) {
        /* zero or subnormal: man * 2^-24, exact in fp32 */
        float v = ldexpf((float)man, -24);
        return sign ? -v : v;
    }
    if (exp == 0x1fu)
        bits = sign | 0x7f800000u | (man << 13);
    else
        bits = sign | ((exp - 15u + 127u) << 23) | (man << 13);
    float f;
    memcpy(&f, &bits, 4);
    return f;
}

static uint16_t rd_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr_u16(uint8_t *p, uint16_t v)
{
    p[0] = (uint8_t)(v & 0xffu);
    p[1] = (uint8_t)(v >> 8);
}

/* ------------------------------------------------------------------------ */
/* q8_1 quantization of one 32-value block ([PR826, commit "fused DS4.1
 * decode kernels"]: the FFN input is quantized once to q8_1 rows shared by
 * every expert).  Definition of the block: d = max|x| / 127, q = round(x/d)
 * (half away from zero), stored fp16 d and fp16 s = d * sum(q).
 * Reading: the division and rounding use the fp32 d, before it is rounded
 * to fp16; an all-zero block stores d = s = 0 and q = 0.                 */
void lo_quantize_q8_1_block(const float *x, uint8_t *out)
{
    float amax = 0.0f;
    for (int i = 0; i < LO_QK; i++) {
        float a = fabsf(x[i]);
        if (a > amax)
            amax = a;
    }
    float d = amax / 127.0f;
    int sum = 0;
    for (int i = 0; i < LO_QK; i++) {
        int q = 0;
        if (amax != 0.0f)
            q = (int)roundf(x[i] / d);
        out[4 + i] = (uint8_t)(int8_t)q;
        sum += q;
    }
    float s = d * (float)sum;
    wr_u16(out + 0, lo_fp16_encode(d));
    wr_u16(out + 2, lo_fp16_encode(s));
}

/* x: [n_rows][K] fp32, K % 32 == 0  ->  out: [n_rows][K/32] q8_1 blocks */
void lo_quantize_q8_1(const float *x, int64_t n_rows, int64_t K, uint8_t *out)
{
    int64_t nb = K / LO_QK;
    for (int64_t r = 0; r < n_rows; r++)
        for (int64_t b = 0; b < nb; b++)
            lo_quantize_q8_1_block(x + r * K + b * LO_QK, out + (r * nb + b) * LO_Q8_1_BYTES);
}

/* ------------------------------------------------------------------------ */
/* One row dot product of a Q8_0 weight row with a q8_1 activation row over
 * K values: sum over blocks b of d_w[b] * d_x[b] * isum[b], where
 * isum[b] = sum_i qw[b][i] * qx[b][i] is an exact integer.  Accumulated in
 * double in block order.  *terms receives sum_b |d_w d_x isum_b|, the scale
 * of the rounding error any fp32 evaluation of the same sum can make.     */
double lo_dot_q8_0_q8_1(const uint8_t *w_row, const uint8_t *x_row, int64_t K, double *terms)
{
    int64_t nb = K / LO_QK;
    double acc = 0.0, tabs = 0.0;
    for (int64_t b = 0; b < nb; b++) {
        const uint8_t *wb = w_row + b * LO_Q8_0_BYTES;
        const uint8_t *xb = x_row + b * LO_Q8_1_BYTES;
        int32_t isum = 0;
        for (int i = 0; i < LO_QK; i++)
            isum += (int32_t)(int8_t)wb[2 + i] * (int32_t)(int8_t)xb[4 + i];
        double dw = (double)lo_fp16_decode(rd_u16(wb));
        double dx = (double)lo_fp16_decode(rd_u16(xb));
        double t = dw * dx * (double)isum;
        acc += t;
        tabs += fabs(t);
    }
    if (terms)
        *terms = tabs;
    return acc;
}

/* The exact integer block sums of one row dot (for bit-exact checks of the
 * integer part of the products).                                          */
void lo_block_isums(const uint8_t *w_row, const uint8_t *x_row, int64_t K, int32_t *isum)
{
    int64_t nb = K / LO_QK;
    for (int64_t b = 0; b < nb; b++) {
        const uint8_t *wb = w_row + b * LO_Q8_0_BYTES;
        const uint8_t *xb = x_row + b * LO_Q8_1_BYTES;
        int32_t s = 0;
        for (int i = 0; i < LO_QK; i++)
            s += (int32_t)(int8_t)wb[2 + i] * (int32_t)(int8_t)xb[4 + i];
        isum[b] = s;
    }
}

/* y[r] = W[r] . x for r < rows, W: [rows][K/32] Q8_0 blocks. */
void lo_matvec_q8_0(const uint8_t *W, int64_t rows, int64_t K, const uint8_t *xq, double *y, double *terms)
{
    int64_t rb = (K / LO_QK) * LO_Q8_0_BYTES;
    for (int64_t r = 0; r < rows; r++)
        y[r] = lo_dot_q8_0_q8_1(W + r * rb, xq, K, terms ? &terms[r] : 0);
}

/* ------------------------------------------------------------------------ */
/* SwiGLU of [PR826, commits "RDNA4 Q8_0 gate/up pair" and "fused routed
 * combine ..."]: h = silu(g) * u, silu(g) = g / (1 + exp(-g)).  The clamped
 * routed form is silu(min(g, L)) * clamp(u, -L, L).  Reading: clamp <= 0
 * means unclamped; the limit L = 10 of the clamped workloads is an input. */
double lo_silu(double g) { return g / (1.0 + exp(-g)); }

double lo_swiglu(double g, double u, double clamp)
{
    if (clamp > 0.0) {
        if (g > clamp)
            g = clamp;
        if (u > clamp)
            u = clamp;
        if (u < -clamp)
            u = -clamp;
    }
    return lo_silu(g) * u;
}

/* Tolerance scale of h from the tolerances of g and u, to first order:
 * |dh| <= |silu(g)| |du| + |u| |silu'(g)| |dg|, with |silu'| <= 1.1.       */
static double swiglu_terms(double g, double u, double tg, double tu, double clamp)
{
    if (clamp > 0.0) {
        if (g > clamp)
            g = clamp;
        if (u > clamp)
            u = clamp;
        if (u < -clamp)
            u = -clamp;
    }
    return fabs(lo_silu(g)) * tu + fabs(u) * 1.1 * tg;
}

/* ------------------------------------------------------------------------ */
/* Router select + weights ([PR826, commit "fused DS4.1 decode kernels"]:
 * the selection and the weights are read from the same logits, in one
 * launch).
 * Per token: score_e = logit_e + bias_e in fp32; the k largest scores are
 * selected, best first, ties to the lower expert index; the weights are the
 * softmax of the selected *unbiased* logits.  Readings: bias affects
 * selection only; softmax over the k selected logits, no extra scaling; a
 * NaN score is taken as -infinity (below every number), so the order is
 * total and a token always selects k distinct experts.                    */
void lo_route_topk(const float *logits, const float *bias, int T, int E, int k, int32_t *ids, double *weights)
{
    for (int t = 0; t < T; t++) {
        const float *l = logits + (int64_t)t * E;
        int32_t *id = ids + (int64_t)t * k;
        for (int j = 0; j < k; j++) {
            int best = -1;
            float bs = 0.0f;
            for (int e = 0; e < E; e++) {
                int taken = 0;
                for (int i = 0; i < j; i++)
                    if (id[i] == e)
                        taken = 1;
                if (taken)
                    continue;
                float s = bias ? l[e] + bias[e] : l[e];
                if (s != s)
                    s = -INFINITY; /* a NaN score ranks below every number */
                if (best < 0 || s > bs) { /* strict: ties keep the lower index */
                    best = e;
                    bs = s;
                }
            }
            id[j] = best;
        }
        double m = (double)l[id[0]];
        for (int j = 1; j < k; j++)
            if ((double)l[id[j]] > m)
                m = (double)l[id[j]];
        double den = 0.0;
        for (int j = 0; j < k; j++)
            den += exp((double)l[id[j]] - m);
        for (int j = 0; j < k; j++)
            weights[(int64_t)t * k + j] = exp((double)l[id[j]] - m) / den;
    }
}

/* ------------------------------------------------------------------------ */
/* Expert grouping ([PR826, commit "fused DS4.1 decode kernels"]: a single
 * grouping per MoE layer, used by gate, up and down).  The T*k routes
 * r = t*k + j are sorted by expert id, stable in r.  Masked routes (id < 0,
 * [PR826, review of moe_combine_masked_kernel]) are left out.  counts[e],
 * offsets[e] = sum of counts below e (offsets[E] = number of kept routes),
 * routes[offsets[e] ...] = the route indices of expert e in increasing r;
 * the unused tail of routes[] is filled with -1.                          */
void lo_moe_group(const int32_t *ids, int T, int k, int E, int32_t *counts, int32_t *offsets, int32_t *routes)
{
    int64_t R = (int64_t)T * k;
    for (int e = 0; e < E; e++)
        counts[e] = 0;
    for (int64_t r = 0; r < R; r++)
        if (ids[r] >= 0 && ids[r] < E)
            counts[ids[r]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; e++)
        offsets[e + 1] = offsets[e] + counts[e];
    int64_t pos = 0;
    for (int e = 0; e < E; e++)
        for (int64_t r = 0; r < R; r++)
            if (ids[r] == e)
                routes[pos++] = (int32_t)r;
    for (; pos < R; pos++)
        routes[pos] = -1;
}

/* ------------------------------------------------------------------------ */
/* Gate/up pair with SwiGLU ([PR826, commit "RDNA4 Q8_0 gate/up pair"]: the
 * gate and up products on the same activations, the GLU of the two in the
 * same launch).  For every kept route r = t*k + j with expert e = ids[r]:
 *   g_i = Wg[e][i] . xq[t],  u_i = Wu[e][i] . xq[t],  h[r][i] = swiglu(g_i, u_i)
 * and, when the shared expert is given, for every token t the same with
 * Ws_g, Ws_u into row T*k + t (the shared expert always runs, weight 1).
 * Rows of masked routes are left untouched.  h_terms receives the error
 * scale of each h (see swiglu_terms).                                     */
void lo_glu_pair(const uint8_t *wg, const uint8_t *wu, const uint8_t *wsg, const uint8_t *wsu, const uint8_t *xq,
                 const int32_t *ids, int T, int k, int E, int H, int I, double clamp, double *h, double *h_terms)
{
    int64_t rowb = (int64_t)(H / LO_QK) * LO_Q8_0_BYTES;
    int64_t xrow = (int64_t)(H / LO_QK) * LO_Q8_1_BYTES;
    int64_t nrows = (int64_t)T * k + (wsg ? T : 0);
    for (int64_t r = 0; r < nrows; r++) {
        const uint8_t *G, *U;
        int t;
        if (r < (int64_t)T * k) {
            int e = ids[r];
            if (e < 0 || e >= E)
                continue;
            t = (int)(r / k);
            G = wg + (int64_t)e * I * rowb;
            U = wu + (int64_t)e * I * rowb;
        } else {
            t = (int)(r - (int64_t)T * k);
            G = wsg;
            U = wsu;
        }
        for (int i = 0; i < I; i++) {
            double tg, tu;
            double g = lo_dot_q8_0_q8_1(G + i * rowb, xq + t * xrow, H, &tg);
            double u = lo_dot_q8_0_q8_1(U + i * rowb, xq + t * xrow, H, &tu);
            h[r * I + i] = lo_swiglu(g, u, clamp);
            if (h_terms)
                h_terms[r * I + i] = swiglu_terms(g, u, tg, tu, clamp);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Down product and masked, route-weighted combine ([PR826, commit "fused
 * routed combine ..."]: masking, weighting and summing the routes is one
 * launch whose combine rounds each product and each sum on its own).  For
 * every token t and output row n:
 *   y[r][n]  = Wd[ids[r]][n] . hq[r]      (r = t*k + j, ids[r] >= 0)
 *   yS[t][n] = Ws_d[n] . hq[T*k + t]      (when the shared expert is given)
 *   out[t][n] = 0; for j = 0..k-1 with ids >= 0: out = fl(out + fl(w * y));
 *   then out = fl(out + yS)
 * with w and y rounded to fp32 and every product and sum rounded to fp32.
 * Reading: the shared expert is added last, with weight 1.  out_terms gets
 * sum_j |w_j| * terms(y_j) + terms(yS).                                   */
void lo_down_combine(const uint8_t *wd, const uint8_t *wsd, const uint8_t *hq, const int32_t *ids,
                     const float *weights, int T, int k, int E, int H, int I, float *out, double *out_terms)
{
    int64_t rowb = (int64_t)(I / LO_QK) * LO_Q8_0_BYTES;
    int64_t hrow = (int64_t)(I / LO_QK) * LO_Q8_1_BYTES;
    for (int t = 0; t < T; t++) {
        for (int n = 0; n < H; n++) {
            float acc = 0.0f;
            double tt = 0.0;
            for (int j = 0; j < k; j++) {
                int64_t r = (int64_t)t * k + j;
                int e = ids[r];
                if (e < 0 || e >= E)
                    continue;
                double ty;
                double y = lo_dot_q8_0_q8_1(wd + ((int64_t)e * H + n) * rowb, hq + r * hrow, I, &ty);
                float w = weights[r];
                float p = w * (float)y;
                acc = acc + p;
                tt += fabs((double)w) * ty;
            }
            if (wsd) {
                double ty;
                double y = lo_dot_q8_0_q8_1(wsd + (int64_t)n * rowb, hq + ((int64_t)T * k + t) * hrow, I, &ty);
                acc = acc + (float)y;
                tt += ty;
            }
            out[(int64_t)t * H + n] = acc;
            if (out_terms)
                out_terms[(int64_t)t * H + n] = tt;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Greedy argmax ([PR826, commit "fused DS4.1 decode kernels"]: the greedy
 * token is found exactly by an argmax done as pairs and a pick).  Per row: the first
 * index of the maximum value (ties to the lower index; -0 equals +0).     */
void lo_argmax(const float *logits, int R, int64_t V, int32_t *idx, float *val)
{
    for (int r = 0; r < R; r++) {
        const float *x = logits + (int64_t)r * V;
        int64_t best = 0;
        for (int64_t v = 1; v < V; v++)
            if (x[v] > x[best])
                best = v;
        idx[r] = (int32_t)best;
        if (val)
            val[r] = x[best];
    }
}

/* ------------------------------------------------------------------------ */
/* Q4_K weights ([PR826], commit "fused DS4.1 decode kernels": wide Q4_K
 * products are among the layer's matrix products).  The pages name the
 * format without defining it; this is the ggml K-quant layout the name
 * refers to: a super-block of 256 values in 8 sub-blocks of 32, 144 bytes:
 * fp16 d, fp16 dmin, 12 bytes that pack 8 six-bit scales sc_j and 8 six-bit
 * mins m_j, then 128 bytes of 4-bit codes.  Sub-block j takes the low
 * (j even) or high (j odd) nibbles of bytes 32 (j / 2) .. 32 (j / 2) + 31;
 * value i of sub-block j is d sc_j q_i - dmin m_j.  Scales and mins: for
 * j < 4, sc_j = s[j] & 63 and m_j = s[j + 4] & 63; for j >= 4 the low four
 * bits come from s[j + 4] (sc: low nibble, m: high nibble) and the high two
 * bits from the top bits of s[j - 4] (sc) and s[j] (m).                   */
void lo_q4_k_scale_min(const uint8_t *s, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* One Q4_K row times one q8_1 row over K values (K a multiple of 256; q8_1
 * block b = 8 sb + j pairs with sub-block j of super-block sb).  Per
 * sub-block: d sc_j d8 isum_j - dmin m_j s8, with isum_j = sum_i q_i qx_i an
 * exact integer, d8 the block's fp16 scale and s8 its fp16 s = d8 sum(qx)
 * as stored (the form that reads the mins against the stored sum).  Reading:
 * the stored s (rounded to fp16) is part of the definition, so the result
 * differs from the dequantized product by at most dmin m_j |s8 - d8 sum qx|.
 * Accumulated in double; *terms receives sum_j (|d sc d8 isum| + |dmin m s8|). */
double lo_dot_q4_k_q8_1(const uint8_t *w_row, const uint8_t *x_row, int64_t K, double *terms)
{
    int64_t nsb = K / LO_QK_K;
    double acc = 0.0, tabs = 0.0;
    for (int64_t sb = 0; sb < nsb; sb++) {
        const uint8_t *w = w_row + sb * LO_Q4_K_BYTES;
        const double d = (double)lo_fp16_decode(rd_u16(w));
        const double dmin = (double)lo_fp16_decode(rd_u16(w + 2));
        const uint8_t *qs = w + 16;
        for (int j = 0; j < 8; j++) {
            const uint8_t *xb = x_row + (sb * 8 + j) * LO_Q8_1_BYTES;
            int sc, m;
            lo_q4_k_scale_min(w + 4, j, &sc, &m);
            int32_t isum = 0;
            for (int i = 0; i < LO_QK; i++) {
                const int q = (j & 1) ? (qs[32 * (j / 2) + i] >> 4) : (qs[32 * (j / 2) + i] & 15);
                isum += q * (int32_t)(int8_t)xb[4 + i];
            }
            const double d8 = (double)lo_fp16_decode(rd_u16(xb));
            const double s8 = (double)lo_fp16_decode(rd_u16(xb + 2));
            const double t1 = d * (double)sc * d8 * (double)isum;
            const double t2 = dmin * (double)m * s8;
            acc += t1 - t2;
            tabs += fabs(t1) + fabs(t2);
        }
    }
    if (terms)
        *terms = tabs;
    return acc;
}

/* Gate/up pair with SwiGLU as lo_glu_pair, with Q4_K gate and up rows. */
void lo_glu_q4k(const uint8_t *wg, const uint8_t *wu, const uint8_t *wsg, const uint8_t *wsu, const uint8_t *xq,
                const int32_t *ids, int T, int k, int E, int H, int I, double clamp, double *h, double *h_terms)
{
    int64_t rowb = (int64_t)(H / LO_QK_K) * LO_Q4_K_BYTES;
    int64_t xrow = (int64_t)(H / LO_QK) * LO_Q8_1_BYTES;
    int64_t nrows = (int64_t)T * k + (wsg ? T : 0);
    for (int64_t r = 0; r < nrows; r++) {
        const uint8_t *G, *U;
        int t;
        if (r < (int64_t)T * k) {
            int e = ids[r];
            if (e < 0 || e >= E)
                continue;
            t = (int)(r / k);
            G = wg + (int64_t)e * I * rowb;
            U = wu + (int64_t)e * I * rowb;
        } else {
            t = (int)(r - (int64_t)T * k);
            G = wsg;
            U = wsu;
        }
        for (int i = 0; i < I; i++) {
            double tg, tu;
            double g = lo_dot_q4_k_q8_1(G + i * rowb, xq + t * xrow, H, &tg);
            double u = lo_dot_q4_k_q8_1(U + i * rowb, xq + t * xrow, H, &tu);
            h[r * I + i] = lo_swiglu(g, u, clamp);
            if (h_terms)
                h_terms[r * I + i] = swiglu_terms(g, u, tg, tu, clamp);
        }
    }
}

/* Down product and masked, route-weighted combine as lo_down_combine, with
 * Q4_K down rows (same rounding of the combine). */
void lo_down_combine_q4k(const uint8_t *wd, const uint8_t *wsd, const uint8_t *hq, const int32_t *ids,
                         const float *weights, int T, int k, int E, int H, int I, float *out, double *out_terms)
{
    int64_t rowb = (int64_t)(I / LO_QK_K) * LO_Q4_K_BYTES;
    int64_t hrow = (int64_t)(I / LO_QK) * LO_Q8_1_BYTES;
    for (int t = 0; t < T; t++) {
        for (int n = 0; n < H; n++) {
            float acc = 0.0f;
            double tt = 0.0;
            for (int j = 0; j < k; j++) {
                int64_t r = (int64_t)t * k + j;
                int e = ids[r];
                if (e < 0 || e >= E)
                    continue;
                double ty;
                double y = lo_dot_q4_k_q8_1(wd + ((int64_t)e * H + n) * rowb, hq + r * hrow, I, &ty);
                float w = weights[r];
                float p = w * (float)y;
                acc = acc + p;
                tt += fabs((double)w) * ty;
            }
            if (wsd) {
                double ty;
                double y = lo_dot_q4_k_q8_1(wsd + (int64_t)n * rowb, hq + ((int64_t)T * k + t) * hrow, I, &ty);
                acc = acc + (float)y;
                tt += ty;
            }
            out[(int64_t)t * H + n] = acc;
            if (out_terms)
                out_terms[(int64_t)t * H + n] = tt;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Argmax of a vocabulary split across ranks ([PR826], commit "fused DS4.1
 * decode kernels": the argmax pair/pick of a vocabulary split across ranks,
 * exact; the cluster runtime commit: the greedy verify head with its
 * vocabulary split across the ranks).  Shard s reports the pair
 * (vals[s][r], idxs[s][r]): its first maximum and that column's index in
 * the whole vocabulary.  The pick keeps the largest value and, among equal
 * values, the lower index, which is the first maximum of the whole row.    */
void lo_argmax_pick(const float *vals, const int32_t *idxs, int S, int R, int32_t *idx, float *val)
{
    for (int r = 0; r < R; r++) {
        float bv = vals[r];
        int32_t bi = idxs[r];
        for (int s = 1; s < S; s++) {
            const float v = vals[(int64_t)s * R + r];
            const int32_t i = idxs[(int64_t)s * R + r];
            if (v > bv || (v == bv && i < bi)) {
                bv = v;
                bi = i;
            }
        }
        idx[r] = bi;
        if (val)
            val[r] = bv;
    }
}

/* ------------------------------------------------------------------------ */
/* The step before the router ([PR826], commit "fused DS4.1 decode kernels":
 * RMS norm among the fused launches; the HC pre-mix commit: an RMS norm
 * whose sum of squares and products run in F32).  Readings: the standard
 * RMS norm, xn_i = x_i * gamma_i / sqrt(mean_i x_i^2 + eps) with eps a
 * parameter, and the router logits are the product of the normed row with
 * the router matrix W_r [E][H] held in F32.  Computed in double: xn [T][H],
 * logits [T][E] and, per logit, the error scale sum_i |W_r[e][i] xn_i|.   */
void lo_rmsnorm_router(const float *x, const float *gamma, double eps, const float *w_router, int T, int E, int H,
                       double *xn, double *logits, double *terms)
{
    for (int t = 0; t < T; t++) {
        const float *xt = x + (int64_t)t * H;
        double ss = 0.0;
        for (int i = 0; i < H; i++)
            ss += (double)xt[i] * (double)xt[i];
        const double r = 1.0 / sqrt(ss / (double)H + eps);
        double *xnt = xn + (int64_t)t * H;
        for (int i = 0; i < H; i++)
            xnt[i] = (double)xt[i] * r * (double)gamma[i];
        for (int e = 0; e < E; e++) {
            const float *w = w_router + (int64_t)e * H;
            double acc = 0.0, mag = 0.0;
            for (int i = 0; i < H; i++) {
                acc += (double)w[i] * xnt[i];
                mag += fabs((double)w[i] * xnt[i]);
            }
            logits[(int64_t)t * E + e] = acc;
            terms[(int64_t)t * E + e] = mag;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Array forms of the fp16 conversions, for the Python wrapper.            */
void lo_fp16_encode_n(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = lo_fp16_encode(x[i]);
}

void lo_fp16_decode_n(const uint16_t *h, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = lo_fp16_decode(h[i]);
}
