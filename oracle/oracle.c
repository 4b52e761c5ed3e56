/*
 * oracle.c -- plain, slow CPU oracle of OSCAR-style INT2 KV caching.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg load it.  It shares no code, header, table or constant
 * generator with the CUDA path.
 *
 * Source: the axbrief.com page "Together AI's OSCAR breaks the 2-bit KV cache
 * accuracy barrier", sections "attention-statistics rotation + Triton kernels"
 * (key rotation R_K = U_Q * H_Had * P_br with U_Q the eigenvectors of
 * C_Q = (1/N) sum q_n^T q_n; clipping c_K = 0.96, c_V = 0.92; per-token
 * asymmetric INT2 in groups of G_K = 64 channels; a read path that unpacks,
 * dequantises and inverse-rotates inside attention) and "OSCAR release"
 * (BF16 sink and recent-window tokens kept beside the INT2 history).
 *
 * Precision: the write path is the exact fp32 contract both sides must meet bit
 * for bit (the rotation is a serial fp32 fused multiply-add chain in ascending
 * input-channel order; IEEE division; round-half-even); everything else
 * (covariance, eigen-decomposition, dequantisation, attention) is fp64.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no fast-math, no contraction).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D 128
#define GROUP 64

/* ---------------------------------------------------------------- number formats */

/* bf16 -> fp32: bf16 is the top half of an fp32 bit pattern. */
static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* IEEE-754 binary16 -> fp32 (exact), from the format definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
float or_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
    return (float)(sign ? -v : v);
}

/* fp32 -> IEEE-754 binary16, round to nearest, ties to even. */
uint16_t or_f32_to_f16(float x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs((double)x);
    if (isnan(x))
        return 0x7e00;
    if (isinf(x))
        return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: the unit is 2^-24; a result of 1024 units is the
         * smallest normal, whose bit pattern is also 1024. */
        double r = nearbyint(a * ldexp(1.0, 24));
        return sign | (uint16_t)r;
    }
    int e;
    frexp(a, &e);                 /* a = m * 2^e, m in [0.5, 1) */
    e -= 1;                       /* a = (1.f) * 2^e */
    double unit = ldexp(1.0, e - 10);
    double r = nearbyint(a / unit);   /* 1024 .. 2048, exact quotient */
    if (r >= 2048.0) {
        r = 1024.0;
        e += 1;
    }
    if (e > 15)
        return sign | 0x7c00;     /* overflow to infinity */
    return sign | (uint16_t)(((e + 15) << 10) | ((int)r - 1024));
}

/* ---------------------------------------------------------------- rotation R_K */

/* Normalised Sylvester-Hadamard matrix, closed form H[i][j] = (-1)^popcount(i&j) / sqrt(128). */
void or_hadamard128(double *h)
{
    double s = 1.0 / sqrt((double)D);
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j)
            h[i * D + j] = (__builtin_popcount((unsigned)(i & j)) & 1) ? -s : s;
}

/* Reverse the 7 bits of i (0 <= i < 128). */
int or_bitrev7(int i)
{
    int r = 0;
    for (int b = 0; b < 7; ++b)
        if (i & (1 << b))
            r |= 1 << (6 - b);
    return r;
}

/* C = (1/N) sum_n q_n^T q_n over row vectors q_n (fp64 accumulation). */
void or_query_covariance(const float *q, long n, double *c)
{
    memset(c, 0, sizeof(double) * D * D);
    for (long t = 0; t < n; ++t) {
        const float *r = q + t * D;
        for (int i = 0; i < D; ++i) {
            double qi = r[i];
            for (int j = 0; j < D; ++j)
                c[i * D + j] += qi * (double)r[j];
        }
    }
    for (int i = 0; i < D * D; ++i)
        c[i] /= (double)n;
}

/*
 * Symmetric eigen-decomposition by the cyclic Jacobi method (Golub & Van Loan,
 * "Matrix Computations", section 8.5: the 2x2 symmetric Schur step and the
 * cyclic-by-row sweep).  a (n x n, row-major) is overwritten; evals gets the
 * eigenvalues in descending order and v (row-major, columns = eigenvectors)
 * the matching orthonormal eigenvectors, each column signed so that its
 * entry of largest magnitude is positive.  Returns the number of sweeps.
 */
int or_jacobi_eigh(double *a, int n, double *evals, double *v)
{
    double *w = (double *)malloc(sizeof(double) * n * n);
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j)
            v[i * n + j] = (i == j) ? 1.0 : 0.0;
    double fro = 0.0;
    for (int i = 0; i < n * n; ++i)
        fro += a[i] * a[i];
    fro = sqrt(fro);
    int sweep;
    for (sweep = 0; sweep < 100; ++sweep) {
        double off = 0.0;
        for (int p = 0; p < n; ++p)
            for (int q = 0; q < n; ++q)
                if (p != q)
                    off += a[p * n + q] * a[p * n + q];
        if (sqrt(off) <= 1e-15 * fro)
            break;
        for (int p = 0; p < n - 1; ++p) {
            for (int q = p + 1; q < n; ++q) {
                double apq = a[p * n + q];
                if (apq == 0.0)
                    continue;
                /* 2x2 symmetric Schur: choose (c, s) zeroing a_pq */
                double tau = (a[q * n + q] - a[p * n + p]) / (2.0 * apq);
                double t = (tau >= 0 ? 1.0 : -1.0) / (fabs(tau) + sqrt(1.0 + tau * tau));
                double c = 1.0 / sqrt(1.0 + t * t);
                double s = t * c;
                /* A <- J^T A J with J = rotation in the (p, q) plane */
                for (int k = 0; k < n; ++k) {          /* columns p, q */
                    double akp = a[k * n + p], akq = a[k * n + q];
                    a[k * n + p] = c * akp - s * akq;
                    a[k * n + q] = s * akp + c * akq;
                }
                for (int k = 0; k < n; ++k) {          /* rows p, q */
                    double apk = a[p * n + k], aqk = a[q * n + k];
                    a[p * n + k] = c * apk - s * aqk;
                    a[q * n + k] = s * apk + c * aqk;
                }
                for (int k = 0; k < n; ++k) {          /* V <- V J */
                    double vkp = v[k * n + p], vkq = v[k * n + q];
                    v[k * n + p] = c * vkp - s * vkq;
                    v[k * n + q] = s * vkp + c * vkq;
                }
            }
        }
    }
    /* sort descending (selection sort on an index list) */
    int *idx = (int *)malloc(sizeof(int) * n);
    for (int i = 0; i < n; ++i)
        idx[i] = i;
    for (int i = 0; i < n; ++i) {
        int best = i;
        for (int j = i + 1; j < n; ++j)
            if (a[idx[j] * n + idx[j]] > a[idx[best] * n + idx[best]])
                best = j;
        int tmp = idx[i];
        idx[i] = idx[best];
        idx[best] = tmp;
    }
    for (int j = 0; j < n; ++j) {
        int src = idx[j];
        evals[j] = a[src * n + src];
        int imax = 0;
        for (int i = 1; i < n; ++i)
            if (fabs(v[i * n + src]) > fabs(v[imax * n + src]))
                imax = i;
        double sg = v[imax * n + src] < 0 ? -1.0 : 1.0;
        for (int i = 0; i < n; ++i)
            w[i * n + j] = sg * v[i * n + src];
    }
    memcpy(v, w, sizeof(double) * n * n);
    free(idx);
    free(w);
    return sweep;
}

/*
 * R_K = U_Q * H_Had * P_br from query samples q (n x 128, fp32).
 * P_br[i][j] = 1 iff j = bitrev7(i), so (M P_br)[r][c] = M[r][bitrev7(c)].
 * rk64 (fp64) and rk (fp32, rounded to nearest) are both written when non-NULL;
 * evals (descending) likewise.
 */
void or_build_rk(const float *q, long n, double *rk64, float *rk, double *evals)
{
    double *c = (double *)malloc(sizeof(double) * D * D);
    double *u = (double *)malloc(sizeof(double) * D * D);
    double *h = (double *)malloc(sizeof(double) * D * D);
    double *uh = (double *)malloc(sizeof(double) * D * D);
    double ev[D];
    or_query_covariance(q, n, c);
    or_jacobi_eigh(c, D, ev, u);
    or_hadamard128(h);
    for (int r = 0; r < D; ++r)
        for (int i = 0; i < D; ++i) {
            double acc = 0.0;
            for (int k = 0; k < D; ++k)
                acc += u[r * D + k] * h[k * D + i];
            uh[r * D + i] = acc;
        }
    for (int r = 0; r < D; ++r)
        for (int col = 0; col < D; ++col) {
            double x = uh[r * D + or_bitrev7(col)];
            if (rk64)
                rk64[r * D + col] = x;
            if (rk)
                rk[r * D + col] = (float)x;
        }
    if (evals)
        memcpy(evals, ev, sizeof(ev));
    free(c);
    free(u);
    free(h);
    free(uh);
}

/* ---------------------------------------------------------------- write path */

/* k~_c = sum_j x_j R[j][c] as the serial chain acc <- fma(x_j, R[j][c], acc), j = 0..127, acc0 = +0. */
void or_rotate_f32(const float *x, const float *r, float *y)
{
    for (int c = 0; c < D; ++c) {
        float acc = 0.0f;
        for (int j = 0; j < D; ++j)
            acc = fmaf(x[j], r[j * D + c], acc);
        y[c] = acc;
    }
}

/*
 * Per-token asymmetric INT2 of one 128-channel vector y (fp32), groups of `group` channels
 * (64, the default G_K of the OSCAR page, or 128; any divisor of 128 works):
 *   mn, mx = group min / max;  lo = c*mn, hi = c*mx  (the clip);
 *   s = fp16(( hi - lo) / 3),  m = fp16(lo);
 *   code = min(max(rint((min(max(y, lo), hi) - m) / s), 0), 3), computed with
 *   the fp16-rounded s and m that are stored; s == 0 gives code 0.
 * Packing: channel 4i + j goes to bits 2j..2j+1 of byte i.
 * sm = [s_0, m_0, s_1, m_1, ...] (fp16 bit patterns, one pair per group: 2 * 128 / group).
 */
void or_quant_vec_g(const float *y, float clip, int group, uint8_t *codes, uint16_t *sm)
{
    uint8_t code[D];
    for (int g = 0; g < D / group; ++g) {
        const float *yg = y + g * group;
        float mn = yg[0], mx = yg[0];
        for (int c = 1; c < group; ++c) {
            mn = fminf(mn, yg[c]);
            mx = fmaxf(mx, yg[c]);
        }
        float lo = clip * mn;
        float hi = clip * mx;
        float s_exact = (hi - lo) / 3.0f;
        uint16_t s16 = or_f32_to_f16(s_exact);
        uint16_t m16 = or_f32_to_f16(lo);
        float s = or_f16_to_f32(s16);
        float m = or_f16_to_f32(m16);
        for (int c = 0; c < group; ++c) {
            float xc = fminf(fmaxf(yg[c], lo), hi);
            int q = 0;
            if (s != 0.0f) {
                float t = (xc - m) / s;
                float r = rintf(t);
                q = r < 0.0f ? 0 : (r > 3.0f ? 3 : (int)r);
            }
            code[g * group + c] = (uint8_t)q;
        }
        sm[2 * g] = s16;
        sm[2 * g + 1] = m16;
    }
    for (int i = 0; i < D / 4; ++i)
        codes[i] = (uint8_t)(code[4 * i] | (code[4 * i + 1] << 2) | (code[4 * i + 2] << 4) |
                             (code[4 * i + 3] << 6));
}

void or_quant_vec(const float *y, float clip, uint8_t *codes, uint16_t *sm)
{
    or_quant_vec_g(y, clip, GROUP, codes, sm);
}

/* n tokens of bf16 input (n x 128 bit patterns) -> codes (n x 32) + sm (n x 2 * 128 / group).
 * r == NULL: no rotation (values).  Also returns the fp32 rotated vectors if y_out != NULL. */
void or_quant_tokens_g(const uint16_t *x16, long n, const float *r, float clip, int group, uint8_t *codes,
                       uint16_t *sm, float *y_out)
{
    float x[D], y[D];
    for (long t = 0; t < n; ++t) {
        for (int j = 0; j < D; ++j)
            x[j] = bf16_to_f32(x16[t * D + j]);
        if (r)
            or_rotate_f32(x, r, y);
        else
            memcpy(y, x, sizeof(y));
        if (y_out)
            memcpy(y_out + t * D, y, sizeof(y));
        or_quant_vec_g(y, clip, group, codes + t * (D / 4), sm + t * (2 * D / group));
    }
}

void or_quant_tokens(const uint16_t *x16, long n, const float *r, float clip, uint8_t *codes,
                     uint16_t *sm, float *y_out)
{
    or_quant_tokens_g(x16, n, r, clip, GROUP, codes, sm, y_out);
}

/* x^ = m + code * s in fp64 (exact), n tokens, groups of `group` channels. */
void or_dequant_tokens_g(const uint8_t *codes, const uint16_t *sm, long n, int group, double *out)
{
    const int per = 2 * D / group;
    for (long t = 0; t < n; ++t)
        for (int c = 0; c < D; ++c) {
            int g = c / group;
            int code = (codes[t * (D / 4) + c / 4] >> (2 * (c % 4))) & 3;
            double s = or_f16_to_f32(sm[t * per + 2 * g]);
            double m = or_f16_to_f32(sm[t * per + 2 * g + 1]);
            out[t * D + c] = m + code * s;
        }
}

void or_dequant_tokens(const uint8_t *codes, const uint16_t *sm, long n, double *out)
{
    or_dequant_tokens_g(codes, sm, n, GROUP, out);
}

/* ---------------------------------------------------------------- read path */

/*
 * Decode attention of G query heads sharing one KV head, fp64:
 *   INT2 tokens:  logit = (q R_K) . k^ / sqrt(128)   (k^ dequantised, rotated domain)
 *   BF16 tokens:  logit = q . k / sqrt(128)          (sink + window, unrotated)
 *   out = sum_t softmax(logit)_t v_t with v^ dequantised for INT2 tokens.
 * The key rotation is applied to q, which equals inverse-rotating every key
 * because R_K is orthogonal.  r == NULL means R_K = I.
 * out: G x 128; lse: G (natural log of sum exp(logit)), may be NULL.
 */
void or_attention_g(int g_heads, const float *q, const float *r, long n_int2, int group_k, int group_v,
                    const uint8_t *k_codes, const uint16_t *k_sm, const uint8_t *v_codes,
                    const uint16_t *v_sm, long n_bf16, const uint16_t *k16, const uint16_t *v16,
                    double *out, double *lse)
{
    long n = n_int2 + n_bf16;
    double *logit = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
    double *kh = (double *)malloc(sizeof(double) * D * (n_int2 > 0 ? n_int2 : 1));
    double *vh = (double *)malloc(sizeof(double) * D * (n_int2 > 0 ? n_int2 : 1));
    or_dequant_tokens_g(k_codes, k_sm, n_int2, group_k, kh);
    or_dequant_tokens_g(v_codes, v_sm, n_int2, group_v, vh);
    double scale = 1.0 / sqrt((double)D);
    for (int hh = 0; hh < g_heads; ++hh) {
        const float *qh = q + hh * D;
        double qr[D];
        for (int c = 0; c < D; ++c) {
            double acc = 0.0;
            for (int j = 0; j < D; ++j)
                acc += (double)qh[j] * (r ? (double)r[j * D + c] : (j == c ? 1.0 : 0.0));
            qr[c] = acc;
        }
        double mx = -INFINITY;
        for (long t = 0; t < n_int2; ++t) {
            double acc = 0.0;
            for (int c = 0; c < D; ++c)
                acc += qr[c] * kh[t * D + c];
            logit[t] = acc * scale;
            if (logit[t] > mx)
                mx = logit[t];
        }
        for (long t = 0; t < n_bf16; ++t) {
            double acc = 0.0;
            for (int c = 0; c < D; ++c)
                acc += (double)qh[c] * (double)bf16_to_f32(k16[t * D + c]);
            logit[n_int2 + t] = acc * scale;
            if (logit[n_int2 + t] > mx)
                mx = logit[n_int2 + t];
        }
        double l = 0.0;
        double o[D];
        for (int c = 0; c < D; ++c)
            o[c] = 0.0;
        for (long t = 0; t < n; ++t) {
            double p = exp(logit[t] - mx);
            l += p;
            if (t < n_int2)
                for (int c = 0; c < D; ++c)
                    o[c] += p * vh[t * D + c];
            else
                for (int c = 0; c < D; ++c)
                    o[c] += p * (double)bf16_to_f32(v16[(t - n_int2) * D + c]);
        }
        for (int c = 0; c < D; ++c)
            out[hh * D + c] = n > 0 ? o[c] / l : 0.0;
        if (lse)
            lse[hh] = n > 0 ? mx + log(l) : -INFINITY;
    }
    free(logit);
    free(kh);
    free(vh);
}

void or_attention(int g_heads, const float *q, const float *r, long n_int2,
                  const uint8_t *k_codes, const uint16_t *k_sm, const uint8_t *v_codes,
                  const uint16_t *v_sm, long n_bf16, const uint16_t *k16, const uint16_t *v16,
                  double *out, double *lse)
{
    or_attention_g(g_heads, q, r, n_int2, GROUP, GROUP, k_codes, k_sm, v_codes, v_sm, n_bf16, k16, v16, out, lse);
}
