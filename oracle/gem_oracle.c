/*
 * gem_oracle.c — TEST INFRASTRUCTURE ONLY (see gem_oracle.h).
 *
 * Scalar fp64 reference of the decoder-layer step.  Every loop runs in the order the
 * definition states (sequential k in every dot product); OpenMP only splits
 * independent outputs (rows, heads), so results do not depend on the thread count.
 */
#include "gem_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- binary16 <-> double: IEEE-754 binary16 definition ------------------------- */

double gem_oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* zero / subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);   /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

uint16_t gem_oracle_double_to_half_via_f32(double v)
{
    float f = (float)v;                 /* binary32, round to nearest even */
    double a = fabs((double)f);
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    if (isnan(f))
        return (uint16_t)(sign | 0x7e00);
    if (isinf(f))
        return (uint16_t)(sign | 0x7c00);
    if (a < ldexp(1.0, -14)) {          /* subnormal range: multiples of 2^-24 */
        double q = nearbyint(a * ldexp(1.0, 24));  /* ties to even */
        return (uint16_t)(sign | (uint16_t)q);     /* q == 1024 is the smallest normal */
    }
    int ex;
    frexp(a, &ex);                      /* a = m * 2^ex, m in [0.5, 1) */
    int e = ex - 1;                     /* a in [2^e, 2^(e+1)) */
    double q = nearbyint(ldexp(a, 10 - e));  /* in [1024, 2048], ties to even */
    if (q == 2048.0) {
        q = 1024.0;
        e += 1;
    }
    if (e > 15)
        return (uint16_t)(sign | 0x7c00);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(q - 1024.0));
}

uint16_t gem_oracle_other_half_via_f32(double v)
{
    float f = (float)v;
    uint16_t h = gem_oracle_double_to_half_via_f32(v);
    double hv = gem_oracle_half_to_double(h);
    if (isnan(f) || hv == (double)f)
        return h;
    /* binary16 codes on a monotone integer line: +x -> x, -x -> -(x & 0x7fff) */
    int i = (h & 0x8000) ? -(int)(h & 0x7fff) : (int)h;
    i += hv > (double)f ? -1 : 1;
    return (uint16_t)(i < 0 ? (0x8000 | -i) : i);
}

/* ---- Q4_0 --------------------------------------------------------------------------
 * [GEM] "Verified model facts": Q4_0 matrices are rows of 32-weight blocks.  A block
 * is an 18-byte record: binary16 scale d (little endian), then 16 bytes of 4-bit
 * codes q; weight = (q - 8) * d.  Reading (GGML order, the pages do not spell it out):
 * byte j holds element j in its low nibble and element j + 16 in its high nibble.
 */
static inline const uint8_t *q4_block(const uint8_t *W, int64_t K, int64_t n, int64_t b)
{
    return W + (n * (K / 32) + b) * 18;
}

static inline double q4_scale(const uint8_t *blk)
{
    return gem_oracle_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
}

void gem_oracle_q4_0_dequant(const uint8_t *W, int64_t N, int64_t K, double *out)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < K / 32; ++b) {
            const uint8_t *blk = q4_block(W, K, n, b);
            double d = q4_scale(blk);
            double *w = out + n * K + 32 * b;
            for (int j = 0; j < 16; ++j) {
                w[j] = (double)((blk[2 + j] & 0x0f) - 8) * d;
                w[j + 16] = (double)((blk[2 + j] >> 4) - 8) * d;
            }
        }
}

/* Dot product of Q4_0 row n with x, k = 0 .. K-1 in order. */
static double q4_row_dot(const uint8_t *W, int64_t K, int64_t n, const double *x)
{
    double acc = 0.0;
    for (int64_t b = 0; b < K / 32; ++b) {
        const uint8_t *blk = q4_block(W, K, n, b);
        double d = q4_scale(blk);
        const double *xb = x + 32 * b;
        for (int j = 0; j < 16; ++j)
            acc += (double)((blk[2 + j] & 0x0f) - 8) * d * xb[j];
        for (int j = 0; j < 16; ++j)
            acc += (double)((blk[2 + j] >> 4) - 8) * d * xb[j + 16];
    }
    return acc;
}

int gem_oracle_q4_0_gemv_f64(const uint8_t *W, int64_t N, int64_t K, const double *x,
                             int64_t ldx, int B, double *y, int64_t ldy)
{
    if (K % 32 || N < 0 || B < 0)
        return 1;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int64_t n = 0; n < N; ++n)
            y[b * ldy + n] = q4_row_dot(W, K, n, x + b * ldx);
    return 0;
}

int gem_oracle_q4_0_gemv_f32(const uint8_t *W, int64_t N, int64_t K, const float *x,
                             int64_t ldx, int B, const float *residual, int64_t ldr,
                             double *y, int64_t ldy)
{
    if (K % 32 || N < 0 || B < 0)
        return 1;
    double *xd = malloc(sizeof(double) * (size_t)(K > 0 ? K : 1) * (size_t)(B > 0 ? B : 1));
    if (!xd)
        return 2;
    for (int b = 0; b < B; ++b)
        for (int64_t k = 0; k < K; ++k)
            xd[b * K + k] = (double)x[b * ldx + k];
    int rc = gem_oracle_q4_0_gemv_f64(W, N, K, xd, K, B, y, ldy);
    if (residual)
        for (int b = 0; b < B; ++b)
            for (int64_t n = 0; n < N; ++n)
                y[b * ldy + n] += (double)residual[b * ldr + n];
    free(xd);
    return rc;
}

/* ---- Q8_0 --------------------------------------------------------------------------
 * [GEM] "Verified model facts": the published layout keeps the token embedding (tied with
 * the output projection) as Q8_0.  A block is a 34-byte record: binary16 scale d (little
 * endian), then 32 signed 8-bit codes q (two's complement); weight j = q[j] * d.  Reading
 * (the pages name the type only): the GGML Q8_0 record, element j in byte 2 + j.
 */
static inline const uint8_t *q8_block(const uint8_t *W, int64_t K, int64_t n, int64_t b)
{
    return W + (n * (K / 32) + b) * 34;
}

void gem_oracle_q8_0_dequant(const uint8_t *W, int64_t N, int64_t K, double *out)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < K / 32; ++b) {
            const uint8_t *blk = q8_block(W, K, n, b);
            double d = gem_oracle_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
            for (int j = 0; j < 32; ++j)
                out[n * K + 32 * b + j] = (double)(int8_t)blk[2 + j] * d;
        }
}

/* y[b][n] = sum_k deq(W)[n][k] * x[b][k], k in order, fp64. */
int gem_oracle_q8_0_gemv_f64(const uint8_t *W, int64_t N, int64_t K, const double *x,
                             int64_t ldx, int B, double *y, int64_t ldy)
{
    if (K % 32 || N < 0 || B < 0)
        return 1;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int64_t n = 0; n < N; ++n) {
            const double *xb = x + b * ldx;
            double acc = 0.0;
            for (int64_t blk = 0; blk < K / 32; ++blk) {
                const uint8_t *p = q8_block(W, K, n, blk);
                double d = gem_oracle_half_to_double((uint16_t)(p[0] | (p[1] << 8)));
                for (int j = 0; j < 32; ++j)
                    acc += (double)(int8_t)p[2 + j] * d * xb[32 * blk + j];
            }
            y[b * ldy + n] = acc;
        }
    return 0;
}

/* ---- RMSNorm -----------------------------------------------------------------------
 * [GEM] "weighted RMSNorm over one or many heads"; [GELO] 05 apply_qk_norm.
 * Readings: eps is a caller parameter (1e-6 in the workloads); gamma multiplies as
 * stored (no 1 + gamma offset).
 */
void gem_oracle_rmsnorm(const double *x, int64_t n, const float *gamma, double eps,
                        double *out)
{
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i)
        ss += x[i] * x[i];
    double r = sqrt(ss / (double)n + eps);
    for (int64_t i = 0; i < n; ++i)
        out[i] = x[i] / r * (gamma ? (double)gamma[i] : 1.0);
}

/* ---- RoPE (NeoX pairing) -------------------------------------------------------------
 * [GEM] "NeoX/proportional RoPE"; [GELO] 02 p-RoPE: only the first rope_dim dims
 * rotate, the rest pass through.  Pair i couples dims i and i + rope_dim/2 and turns
 * by pos * theta^(-2i/rope_dim).  Reading: frequencies run over rope_dim.
 */
void gem_oracle_rope_neox(double *v, int d, int rope_dim, double pos, double theta)
{
    (void)d;
    int half = rope_dim / 2;
    for (int i = 0; i < half; ++i) {
        double w = pow(theta, -2.0 * (double)i / (double)rope_dim);
        double a = pos * w;
        double c = cos(a), s = sin(a);
        double u = v[i], t = v[i + half];
        v[i] = u * c - t * s;
        v[i + half] = u * s + t * c;
    }
}

/* ---- GQA decode attention -------------------------------------------------------------
 * [GELO] 02 (GQA, sliding window of the last W tokens), 05 (decode attends
 * n_kv = n_cache + 1 positions).  Readings: query head h uses KV head h / (n_q/n_kv);
 * the window includes the new token; softmax in fp64 with max subtraction.
 */
int gem_oracle_gqa_attention(const double *q, const uint16_t *k_cache,
                             const uint16_t *v_cache, int n_q, int n_kv, int d,
                             int64_t cap, int64_t pos, int window, double scale,
                             double *out, double *probs)
{
    if (n_kv <= 0 || n_q % n_kv || pos < 0)
        return 1;
    int64_t j0 = window ? (pos - window + 1 > 0 ? pos - window + 1 : 0) : 0;
    int64_t T = pos - j0 + 1;
    if ((window && window > cap) || (!window && pos >= cap))
        return 2;
    int G = n_q / n_kv;
    int rc = 0;
#pragma omp parallel for schedule(static)
    for (int h = 0; h < n_q; ++h) {
        int g = h / G;
        const double *qh = q + (int64_t)h * d;
        double *s = malloc(sizeof(double) * (size_t)T);
        if (!s) {
            rc = 3;
            continue;
        }
        double m = -INFINITY;
        for (int64_t t = 0; t < T; ++t) {
            int64_t j = j0 + t;
            int64_t slot = window ? j % window : j;
            const uint16_t *kr = k_cache + ((int64_t)g * cap + slot) * d;
            double acc = 0.0;
            for (int i = 0; i < d; ++i)
                acc += qh[i] * gem_oracle_half_to_double(kr[i]);
            s[t] = scale * acc;
            if (s[t] > m)
                m = s[t];
        }
        double den = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            s[t] = exp(s[t] - m);
            den += s[t];
        }
        double *oh = out + (int64_t)h * d;
        for (int i = 0; i < d; ++i)
            oh[i] = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            int64_t j = j0 + t;
            int64_t slot = window ? j % window : j;
            const uint16_t *vr = v_cache + ((int64_t)g * cap + slot) * d;
            double p = s[t] / den;
            if (probs)
                probs[(int64_t)h * T + t] = p;
            for (int i = 0; i < d; ++i)
                oh[i] += p * gem_oracle_half_to_double(vr[i]);
        }
        free(s);
    }
    return rc;
}

/* ---- Compact full-attention cache ---------------------------------------------------------
 * [GEM] "Verified model facts": on a full-attention layer (V = unweighted RMSNorm of the K
 * projection, K = key_norm-weighted RMSNorm of it, then RoPE) the cache can hold the V row
 * alone; the historical K row is rebuilt inside the attention as V * key_norm.  Reading (the
 * pages leave the rotation implicit): the rebuilt row is rotated at the row's own position,
 *   K_j = RoPE_j(V16_j * gamma_k),
 * evaluated in fp64 from the binary16 V row, since the standard cache stores the rotated K.
 * Full attention only: slot j holds position j.  q: [n_q][d] (already normalised and rotated
 * at pos); out: [n_q][d].
 */
int gem_oracle_gqa_attention_compact(const double *q, const uint16_t *v_cache, const float *gamma_k,
                                     int n_q, int n_kv, int d, int64_t cap, int64_t pos,
                                     int rope_dim, double theta, double scale, double *out)
{
    if (n_kv <= 0 || n_q % n_kv || pos < 0 || pos >= cap || rope_dim < 0 || rope_dim > d ||
        (rope_dim & 1))
        return 1;
    const int64_t T = pos + 1;
    const int G = n_q / n_kv;
    int rc = 0;
#pragma omp parallel for schedule(static)
    for (int g = 0; g < n_kv; ++g) {
        double *s = malloc(sizeof(double) * (size_t)T * (size_t)G);
        double *k = malloc(sizeof(double) * (size_t)d);
        if (!s || !k) {
            free(s);
            free(k);
            rc = 3;
            continue;
        }
        const uint16_t *vg = v_cache + (int64_t)g * cap * d;
        for (int64_t j = 0; j < T; ++j) {   /* rebuild K_j, then every head's score */
            for (int i = 0; i < d; ++i)
                k[i] = gem_oracle_half_to_double(vg[j * d + i]) * (gamma_k ? (double)gamma_k[i] : 1.0);
            gem_oracle_rope_neox(k, d, rope_dim, (double)j, theta);
            for (int hh = 0; hh < G; ++hh) {
                const double *qh = q + (int64_t)(g * G + hh) * d;
                double acc = 0.0;
                for (int i = 0; i < d; ++i)
                    acc += qh[i] * k[i];
                s[hh * T + j] = scale * acc;
            }
        }
        for (int hh = 0; hh < G; ++hh) {
            double *sh = s + hh * T;
            double m = -INFINITY;
            for (int64_t j = 0; j < T; ++j)
                if (sh[j] > m)
                    m = sh[j];
            double den = 0.0;
            for (int64_t j = 0; j < T; ++j) {
                sh[j] = exp(sh[j] - m);
                den += sh[j];
            }
            double *oh = out + (int64_t)(g * G + hh) * d;
            for (int i = 0; i < d; ++i)
                oh[i] = 0.0;
            for (int64_t j = 0; j < T; ++j) {
                const double w = sh[j] / den;
                for (int i = 0; i < d; ++i)
                    oh[i] += w * gem_oracle_half_to_double(vg[j * d + i]);
            }
        }
        free(s);
        free(k);
    }
    return rc;
}

/* ---- FFN activations --------------------------------------------------------------------
 * [GELO] 04/05: Qwen3 SwiGLU, silu(g) = g / (1 + e^-g).  [GELO] 04 (Gemma):
 * gelu_pytorch_tanh, 0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))).
 */
double gem_oracle_silu(double g) { return g / (1.0 + exp(-g)); }

double gem_oracle_gelu_tanh(double g)
{
    const double c = sqrt(2.0 / M_PI);
    return 0.5 * g * (1.0 + tanh(c * (g + 0.044715 * g * g * g)));
}

/* ---- One decoder layer step ----------------------------------------------------------------
 * Topology ([GELO] 06 figure notes, [GEM] stage groups): pre-norm, merged QKV
 * projection, per-head QK-norm, RoPE, KV append, GQA attention, O projection +
 * residual, pre-FFN norm, gate/up, gated activation, down projection + residual.
 * Gemma flags: V from the K projection by unweighted RMSNorm ([GEM] "Verified model
 * facts"); post-attention / post-FFN norms before each residual add (reading).
 */
int gem_oracle_decode_layer_ex(const gem_oracle_layer *L, int B, const double *x_in,
                               uint16_t *k_cache, uint16_t *v_cache, int64_t cap,
                               const int32_t *pos, double *x_out, double *qkv_out,
                               double *attn_out, double *h_out, double *kvnew_out,
                               const int8_t *flip)
{
    const int64_t H = L->H, d = L->d, nq = L->n_q, nkv = L->n_kv, F = L->F;
    const int64_t qdim = nq * d, kdim = nkv * d;
    const int64_t nqkv = qdim + kdim + (L->v_from_k ? 0 : kdim);
    int rc = 0;
    double *xn = malloc(sizeof(double) * H);
    double *qkv = malloc(sizeof(double) * nqkv);
    double *vrow = malloc(sizeof(double) * kdim);
    double *tmp = malloc(sizeof(double) * (d > H ? d : H));
    double *att = malloc(sizeof(double) * qdim);
    double *o = malloc(sizeof(double) * H);
    double *h = malloc(sizeof(double) * H);
    double *g = malloc(sizeof(double) * F);
    double *u = malloc(sizeof(double) * F);
    double *a = malloc(sizeof(double) * F);
    double *dn = malloc(sizeof(double) * H);
    if (!xn || !qkv || !vrow || !tmp || !att || !o || !h || !g || !u || !a || !dn) {
        rc = 3;
        goto done;
    }
    for (int b = 0; b < B; ++b) {
        const double *x = x_in + (int64_t)b * H;
        int64_t p = pos[b];
        uint16_t *kc = k_cache ? k_cache + (int64_t)b * nkv * cap * d : NULL;
        uint16_t *vc = v_cache + (int64_t)b * nkv * cap * d;
        /* a1 pre-attention RMSNorm, a2 QKV projection */
        gem_oracle_rmsnorm(x, H, L->g_attn, L->eps, xn);
        gem_oracle_q4_0_gemv_f64(L->w_qkv, nqkv, H, xn, H, 1, qkv, nqkv);
        double *q = qkv, *k = qkv + qdim;
        /* a3 value rows: V projection, or unweighted RMSNorm of the raw K projection */
        for (int64_t j = 0; j < nkv; ++j) {
            if (L->v_from_k)
                gem_oracle_rmsnorm(k + j * d, d, NULL, L->eps, vrow + j * d);
            else
                memcpy(vrow + j * d, qkv + qdim + kdim + j * d, sizeof(double) * d);
        }
        /* a3 per-head QK-norm, a4 RoPE */
        for (int64_t hh = 0; hh < nq; ++hh) {
            if (L->qk_norm) {
                gem_oracle_rmsnorm(q + hh * d, d, L->g_q, L->eps, tmp);
                memcpy(q + hh * d, tmp, sizeof(double) * d);
            }
            gem_oracle_rope_neox(q + hh * d, (int)d, L->rope_dim, (double)p, L->theta);
        }
        for (int64_t j = 0; j < nkv; ++j) {
            if (L->qk_norm) {
                gem_oracle_rmsnorm(k + j * d, d, L->g_k, L->eps, tmp);
                memcpy(k + j * d, tmp, sizeof(double) * d);
            }
            gem_oracle_rope_neox(k + j * d, (int)d, L->rope_dim, (double)p, L->theta);
        }
        if (qkv_out) {
            memcpy(qkv_out + (int64_t)b * nqkv, qkv, sizeof(double) * (qdim + kdim));
            if (!L->v_from_k)
                memcpy(qkv_out + (int64_t)b * nqkv + qdim + kdim, vrow, sizeof(double) * kdim);
        }
        /* a5 KV append at the new token's slot, rounded to binary16 via binary32 (a compact
         * cache keeps the V row only) */
        int64_t slot = L->window ? p % L->window : p;
        if (slot >= cap || p < 0 || (L->compact_kv && (L->window || !L->v_from_k))) {
            rc = 2;
            goto done;
        }
        for (int64_t j = 0; j < nkv; ++j)
            for (int64_t i = 0; i < d; ++i) {
                const int64_t fk = (((int64_t)b * 2 + 0) * nkv + j) * d + i;
                const int64_t fv = (((int64_t)b * 2 + 1) * nkv + j) * d + i;
                if (!L->compact_kv)
                    kc[(j * cap + slot) * d + i] = (flip && flip[fk])
                        ? gem_oracle_other_half_via_f32(k[j * d + i])
                        : gem_oracle_double_to_half_via_f32(k[j * d + i]);
                vc[(j * cap + slot) * d + i] = (flip && flip[fv])
                    ? gem_oracle_other_half_via_f32(vrow[j * d + i])
                    : gem_oracle_double_to_half_via_f32(vrow[j * d + i]);
                if (kvnew_out) {
                    kvnew_out[fk] = k[j * d + i];
                    kvnew_out[fv] = vrow[j * d + i];
                }
            }
        /* a6 attention */
        if (L->compact_kv)
            rc = gem_oracle_gqa_attention_compact(q, vc, L->g_k, (int)nq, (int)nkv, (int)d, cap, p,
                                                  L->rope_dim, L->theta, L->scale, att);
        else
            rc = gem_oracle_gqa_attention(q, kc, vc, (int)nq, (int)nkv, (int)d, cap, p,
                                          L->window, L->scale, att, NULL);
        if (rc)
            goto done;
        if (attn_out)
            memcpy(attn_out + (int64_t)b * qdim, att, sizeof(double) * qdim);
        /* a7 O projection + residual */
        gem_oracle_q4_0_gemv_f64(L->w_o, H, qdim, att, qdim, 1, o, H);
        if (L->post_norms) {
            gem_oracle_rmsnorm(o, H, L->g_post_attn, L->eps, tmp);
            for (int64_t i = 0; i < H; ++i)
                h[i] = x[i] + tmp[i];
        } else {
            for (int64_t i = 0; i < H; ++i)
                h[i] = x[i] + o[i];
        }
        if (h_out)
            memcpy(h_out + (int64_t)b * H, h, sizeof(double) * H);
        /* a8 pre-FFN RMSNorm, a9 gate/up, a10 gated activation */
        gem_oracle_rmsnorm(h, H, L->g_ffn, L->eps, xn);
        gem_oracle_q4_0_gemv_f64(L->w_gate, F, H, xn, H, 1, g, F);
        gem_oracle_q4_0_gemv_f64(L->w_up, F, H, xn, H, 1, u, F);
        for (int64_t i = 0; i < F; ++i)
            a[i] = (L->act ? gem_oracle_gelu_tanh(g[i]) : gem_oracle_silu(g[i])) * u[i];
        /* a11 down projection + residual */
        gem_oracle_q4_0_gemv_f64(L->w_down, H, F, a, F, 1, dn, H);
        double *xo = x_out + (int64_t)b * H;
        if (L->post_norms) {
            gem_oracle_rmsnorm(dn, H, L->g_post_ffn, L->eps, tmp);
            for (int64_t i = 0; i < H; ++i)
                xo[i] = h[i] + tmp[i];
        } else {
            for (int64_t i = 0; i < H; ++i)
                xo[i] = h[i] + dn[i];
        }
    }
done:
    free(xn); free(qkv); free(vrow); free(tmp); free(att); free(o); free(h);
    free(g); free(u); free(a); free(dn);
    return rc;
}

int gem_oracle_decode_layer_f64(const gem_oracle_layer *L, int B, const double *x_in,
                                uint16_t *k_cache, uint16_t *v_cache, int64_t cap,
                                const int32_t *pos, double *x_out, double *qkv_out,
                                double *attn_out, double *h_out)
{
    return gem_oracle_decode_layer_ex(L, B, x_in, k_cache, v_cache, cap, pos, x_out, qkv_out,
                                      attn_out, h_out, NULL, NULL);
}

int gem_oracle_decode_layer(const gem_oracle_layer *L, int B, const float *x_in,
                            uint16_t *k_cache, uint16_t *v_cache, int64_t cap,
                            const int32_t *pos, double *x_out, double *qkv_out,
                            double *attn_out, double *h_out)
{
    double *xd = malloc(sizeof(double) * (size_t)(B * L->H));
    if (!xd)
        return 3;
    for (int64_t i = 0; i < B * L->H; ++i)
        xd[i] = (double)x_in[i];
    int rc = gem_oracle_decode_layer_f64(L, B, xd, k_cache, v_cache, cap, pos, x_out,
                                         qkv_out, attn_out, h_out);
    free(xd);
    return rc;
}

/* [GEM] sampler note: equal logits are broken by token id (lowest wins).  Reading for
 * entries that are not numbers (the pages do not say): a NaN is never chosen; all NaN
 * (or n == 0) gives 0. */
int64_t gem_oracle_argmax(const double *v, int64_t n)
{
    int64_t best = -1;
    for (int64_t i = 0; i < n; ++i)
        if (!isnan(v[i]) && (best < 0 || v[i] > v[best]))
            best = i;
    return best < 0 ? 0 : best;
}

/* The k largest entries, largest first: the order ranks numbers by value (descending, -inf
 * included), equal values by index (ascending, as the argmax above), and places entries that are
 * not numbers after every number, by index.  [GEM] sampler note (top-k with ties broken by token
 * id); the NaN rank is this library's reading.  Plain selection: k scans over the n entries.
 * idx, val: [k]; 1 <= k <= n. */
static int oracle_before(const double *v, int64_t a, int64_t b)
{
    const int na = isnan(v[a]), nb = isnan(v[b]);
    if (na != nb)
        return nb;   /* a number comes before a NaN */
    if (!na && v[a] != v[b])
        return v[a] > v[b];
    return a < b;
}

int gem_oracle_topk(const double *v, int64_t n, int k, int64_t *idx, double *val)
{
    if (k < 1 || k > n)
        return 1;
    unsigned char *taken = calloc((size_t)n, 1);
    if (!taken)
        return 3;
    for (int r = 0; r < k; ++r) {
        int64_t best = -1;
        for (int64_t i = 0; i < n; ++i)
            if (!taken[i] && (best < 0 || oracle_before(v, i, best)))
                best = i;
        taken[best] = 1;
        idx[r] = best;
        val[r] = v[best];
    }
    free(taken);
    return 0;
}

int gem_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void gem_oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
