/*
 * Plain, slow, fp64 CPU oracle for the Q4_0 decode-step matrix-vector product
 * and the decoder-layer glue around it.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is used by the tests, by the
 * package's smoke check and by the CPU-baseline leg of the benchmark.  The
 * GPU library never includes, links or calls it, and it shares no code,
 * header, table or constant with the GPU library.
 *
 * What it computes, and where each step comes from:
 *   - Q4_0 block: 32 weights stored as an IEEE binary16 scale d followed by
 *     16 bytes of 4-bit codes; weight = (q - 8) * d.  The pages name the GGUF
 *     file format (PipeLLM, "Layer 1"/compatibility paragraph) and 4-bit
 *     weights (PIPO summary, Method, "Computation optimization") but print no
 *     layout; the layout is GGUF's Q4_0 as stated in the task definition:
 *     byte j of the codes holds element j in its low nibble and element j+16
 *     in its high nibble.
 *   - The product y[b][n] = sum_k W[n][k] * x[b][k] is written out as its
 *     plain definition (dequantise each weight, multiply, add in index order,
 *     fp64).  PIPO's "matrix-vector multiply directly on 4-bit quantized
 *     weights, avoiding dequantization" reaches the same value up to rounding
 *     order, so the definition is the oracle.
 *   - Decoder-layer glue (RMSNorm, context-1 attention, residual adds,
 *     SiLU-gated FFN) follows the plainest Llama-shaped reading of "a
 *     transformer layer's q/k/v/o/gate/up/down projections in sequence"
 *     (PIPO summary, Method, "Offloading architecture": the layer is the unit
 *     of the schedule).  Activations are rounded to binary16 at the points
 *     where the GPU stores binary16.  The residual sum is normalised after
 *     each add (post-norm); with the workloads' weights (codes uniform on
 *     0..15, so E[q - 8] = -1/2) a pre-norm residual stream overflows
 *     binary16 within two 8B-shaped layers.
 *
 * All floating-point work here is double precision.  The binary16 decoder
 * and the round-to-nearest-even encoder are written out below from the IEEE
 * 754 definition; nothing else from a library is used but libm's sqrt/exp.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#define ORA_QK 32          /* weights per Q4_0 block */
#define ORA_BLOCK_BYTES 18 /* 2-byte scale + 16 bytes of codes */

/* ------------------------------------------------------------------ */
/* IEEE 754 binary16                                                   */
/* ------------------------------------------------------------------ */

/* binary16 bit pattern -> double (exact: every binary16 value is a double). */
double ora_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);              /* zero and subnormals: m * 2^-24 */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25);  /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* double -> binary16, round to nearest, ties to even; overflow -> inf. */
uint16_t ora_double_to_half(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v))
        return (uint16_t)(sign | 0x7E00u);
    double a = fabs(v);
    if (a >= 65520.0)                           /* half-way above 65504 rounds to inf */
        return (uint16_t)(sign | 0x7C00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: value = m * 2^-24, m in [0, 1024]; m == 1024 is
         * the smallest normal and its encoding is 0x0400 as well */
        double m = rint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)m);
    }
    int E;
    (void)frexp(a, &E);                         /* a = f * 2^E, f in [0.5, 1) */
    int e = E - 1;                              /* a in [2^e, 2^(e+1)) */
    double m = rint(ldexp(a, 10 - e));          /* in [1024, 2048] */
    if (m == 2048.0) {
        m = 1024.0;
        e += 1;
    }
    if (e > 15)
        return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)(((e + 15) << 10) | ((int)m - 1024)));
}

void ora_half_to_double_n(const uint16_t *h, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = ora_half_to_double(h[i]);
}

void ora_double_to_half_n(const double *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = ora_double_to_half(v[i]);
}

/* ------------------------------------------------------------------ */
/* Q4_0 weights                                                        */
/* ------------------------------------------------------------------ */

/* The weight at (row n, column k) of a row-major Q4_0 matrix with k_dim
 * columns: block i = k / 32 of row n, element j = k % 32 of that block. */
static double ora_weight(const uint8_t *w, int64_t k_dim, int64_t n, int64_t k)
{
    int64_t blocks_per_row = k_dim / ORA_QK;
    const uint8_t *blk = w + (n * blocks_per_row + k / ORA_QK) * ORA_BLOCK_BYTES;
    int j = (int)(k % ORA_QK);
    uint16_t d_bits = (uint16_t)(blk[0] | (blk[1] << 8));   /* little-endian scale */
    const uint8_t *qs = blk + 2;
    int q = (j < 16) ? (qs[j] & 0x0F) : (qs[j - 16] >> 4);
    return (double)(q - 8) * ora_half_to_double(d_bits);
}

/* Dense dequantisation: out[n * k_dim + k] = W[n][k]. */
void ora_dequant(const uint8_t *w, int64_t n_rows, int64_t k_dim, double *out)
{
    for (int64_t n = 0; n < n_rows; n++)
        for (int64_t k = 0; k < k_dim; k++)
            out[n * k_dim + k] = ora_weight(w, k_dim, n, k);
}

/* y[b][n] = sum_k W[n][k] * x[b][k] for rows n in [row0, row1), and
 * s[b][n] = sum_k |W[n][k] * x[b][k]| (the scale of the error bound).
 * x is binary16 [batch][k_dim]; y and s are [batch][n_rows].  Products are
 * exact in double; the sum runs over k in index order. */
void ora_gemv(const uint8_t *w, const uint16_t *x, int64_t n_rows, int64_t k_dim,
              int batch, int64_t row0, int64_t row1, double *y, double *s)
{
    for (int b = 0; b < batch; b++) {
        const uint16_t *xb = x + (int64_t)b * k_dim;
        for (int64_t n = row0; n < row1; n++) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < k_dim; k++) {
                double p = ora_weight(w, k_dim, n, k) * ora_half_to_double(xb[k]);
                acc += p;
                mag += fabs(p);
            }
            y[(int64_t)b * n_rows + n] = acc;
            if (s)
                s[(int64_t)b * n_rows + n] = mag;
        }
    }
}

/* The same product on an explicit list of rows (for spot checks of large
 * matrices): y[b][i], s[b][i] for row rows[i]. */
void ora_gemv_rows(const uint8_t *w, const uint16_t *x, int64_t n_rows, int64_t k_dim,
                   int batch, const int64_t *rows, int64_t n_sel, double *y, double *s)
{
    (void)n_rows;
    for (int b = 0; b < batch; b++) {
        const uint16_t *xb = x + (int64_t)b * k_dim;
        for (int64_t i = 0; i < n_sel; i++) {
            int64_t n = rows[i];
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < k_dim; k++) {
                double p = ora_weight(w, k_dim, n, k) * ora_half_to_double(xb[k]);
                acc += p;
                mag += fabs(p);
            }
            y[(int64_t)b * n_sel + i] = acc;
            if (s)
                s[(int64_t)b * n_sel + i] = mag;
        }
    }
}

/* ------------------------------------------------------------------ */
/* Decoder-layer glue                                                  */
/* ------------------------------------------------------------------ */

/* RMSNorm with unit weight: x = f16(h / sqrt(mean(h^2) + eps)), per batch row. */
void ora_rmsnorm(const uint16_t *h, int batch, int64_t dim, double eps, uint16_t *x_out)
{
    for (int b = 0; b < batch; b++) {
        const uint16_t *hb = h + (int64_t)b * dim;
        double ss = 0.0;
        for (int64_t i = 0; i < dim; i++) {
            double v = ora_half_to_double(hb[i]);
            ss += v * v;
        }
        double r = 1.0 / sqrt(ss / (double)dim + eps);
        for (int64_t i = 0; i < dim; i++)
            x_out[(int64_t)b * dim + i] = ora_double_to_half(ora_half_to_double(hb[i]) * r);
    }
}

/* Attention over a context of one token: the softmax over a single key is 1
 * and rotary position 0 is the identity, so query head qh reads the value
 * head it is grouped with: attn[b][qh*hd + i] = f16(v[b][(qh / group)*hd + i]),
 * group = (q_dim / hd) / (kv_dim / hd). */
void ora_attn_ctx1(const double *v, int batch, int64_t q_dim, int64_t kv_dim, int64_t head_dim,
                   uint16_t *attn)
{
    int64_t n_q = q_dim / head_dim, n_kv = kv_dim / head_dim;
    int64_t group = n_q / n_kv;
    for (int b = 0; b < batch; b++)
        for (int64_t qh = 0; qh < n_q; qh++)
            for (int64_t i = 0; i < head_dim; i++)
                attn[(int64_t)b * q_dim + qh * head_dim + i] =
                    ora_double_to_half(v[(int64_t)b * kv_dim + (qh / group) * head_dim + i]);
}

/* Decode attention of one token over a KV cache (the decode loop over a
 * growing context that PipeLLM captures per context-length bucket, "Layer 1:
 * CUDA Graph Compilation"; the per-layer KV cache PIPO loads and saves with
 * the layer, Method, "Offloading architecture").  The cache holds binary16
 * keys and values, row t = position t, each row n_kv heads of head_dim
 * values (keys already carry their position encoding, as a cache stores
 * them).  For query head h and its value head g = h / (n_q / n_kv):
 *   s_t = (sum_i q[h][i] * k[t][g][i]) / sqrt(head_dim),  t < ctx
 *   p_t = exp(s_t - max_t s_t) / sum_t exp(s_t - max_t s_t)
 *   o[h][i] = sum_t p_t * v[t][g][i]
 * in double, q given in double.  sabs[h][i] = sum_t p_t |v[t][g][i]| (for the
 * accepted error bound). */
void ora_attn_decode(const double *q, const uint16_t *kc, const uint16_t *vc, int64_t ctx, int64_t n_q,
                     int64_t n_kv, int64_t head_dim, double *o, double *sabs, double *work)
{
    int64_t group = n_q / n_kv, kv_dim = n_kv * head_dim;
    double scale = 1.0 / sqrt((double)head_dim);
    for (int64_t h = 0; h < n_q; h++) {
        int64_t g = h / group;
        double mx = -INFINITY;
        for (int64_t t = 0; t < ctx; t++) {
            double sc = 0.0;
            for (int64_t i = 0; i < head_dim; i++)
                sc += q[h * head_dim + i] * ora_half_to_double(kc[t * kv_dim + g * head_dim + i]);
            work[t] = sc * scale;
            if (work[t] > mx) mx = work[t];
        }
        double den = 0.0;
        for (int64_t t = 0; t < ctx; t++) {
            work[t] = exp(work[t] - mx);
            den += work[t];
        }
        for (int64_t i = 0; i < head_dim; i++) {
            double acc = 0.0, aabs = 0.0;
            for (int64_t t = 0; t < ctx; t++) {
                double v = ora_half_to_double(vc[t * kv_dim + g * head_dim + i]);
                acc += work[t] / den * v;
                aabs += work[t] / den * fabs(v);
            }
            o[h * head_dim + i] = acc;
            sabs[h * head_dim + i] = aabs;
        }
    }
}

/* RMSNorm of a double vector (a residual sum): x = f16(t / sqrt(mean(t^2) + eps)). */
void ora_rmsnorm_d(const double *t, int batch, int64_t dim, double eps, uint16_t *x_out)
{
    for (int b = 0; b < batch; b++) {
        const double *tb = t + (int64_t)b * dim;
        double ss = 0.0;
        for (int64_t i = 0; i < dim; i++)
            ss += tb[i] * tb[i];
        double r = 1.0 / sqrt(ss / (double)dim + eps);
        for (int64_t i = 0; i < dim; i++)
            x_out[(int64_t)b * dim + i] = ora_double_to_half(tb[i] * r);
    }
}

/* Residual sum: t = z + o (z binary16, o and t double). */
void ora_add(const uint16_t *z, const double *o, int64_t n, double *t)
{
    for (int64_t i = 0; i < n; i++)
        t[i] = ora_half_to_double(z[i]) + o[i];
}

/* SiLU-gated product: act = f16(g / (1 + exp(-g)) * u). */
void ora_silu_mul(const double *g, const double *u, int64_t n, uint16_t *act)
{
    for (int64_t i = 0; i < n; i++)
        act[i] = ora_double_to_half(g[i] / (1.0 + exp(-g[i])) * u[i]);
}

/* One decoder layer, batch rows independent, with the residual sum
 * normalised after each add.  z is the layer's normalised binary16 input
 * [batch][hidden]; weight order q, k, v, o, gate, up, down (row-major Q4_0
 * each).  Writes t2 (double [batch][hidden], the last residual sum) and
 * z_out = f16(norm(t2)), the next layer's input.  work must hold
 * batch*(q_dim + 2*kv_dim + 3*hidden + 2*ffn) doubles and
 * batch*(hidden + q_dim + ffn) binary16 values in work16. */
void ora_layer(const uint8_t *const *wts, const uint16_t *z, int batch, int64_t hidden,
               int64_t q_dim, int64_t kv_dim, int64_t ffn, int64_t head_dim, double eps,
               double *work, uint16_t *work16, double *t2, uint16_t *z_out)
{
    double *q = work;
    double *k = q + (int64_t)batch * q_dim;
    double *v = k + (int64_t)batch * kv_dim;
    double *o = v + (int64_t)batch * kv_dim;
    double *t1 = o + (int64_t)batch * hidden;
    double *dn = t1 + (int64_t)batch * hidden;
    double *g = dn + (int64_t)batch * hidden;
    double *u = g + (int64_t)batch * ffn;
    uint16_t *attn = work16;
    uint16_t *z1 = attn + (int64_t)batch * q_dim;
    uint16_t *act = z1 + (int64_t)batch * hidden;

    ora_gemv(wts[0], z, q_dim, hidden, batch, 0, q_dim, q, 0);
    ora_gemv(wts[1], z, kv_dim, hidden, batch, 0, kv_dim, k, 0);
    ora_gemv(wts[2], z, kv_dim, hidden, batch, 0, kv_dim, v, 0);
    ora_attn_ctx1(v, batch, q_dim, kv_dim, head_dim, attn);
    ora_gemv(wts[3], attn, hidden, q_dim, batch, 0, hidden, o, 0);
    ora_add(z, o, (int64_t)batch * hidden, t1);
    ora_rmsnorm_d(t1, batch, hidden, eps, z1);
    ora_gemv(wts[4], z1, ffn, hidden, batch, 0, ffn, g, 0);
    ora_gemv(wts[5], z1, ffn, hidden, batch, 0, ffn, u, 0);
    ora_silu_mul(g, u, (int64_t)batch * ffn, act);
    ora_gemv(wts[6], act, hidden, ffn, batch, 0, hidden, dn, 0);
    ora_add(z1, dn, (int64_t)batch * hidden, t2);
    ora_rmsnorm_d(t2, batch, hidden, eps, z_out);
}

/* One decoder layer of one token at position pos with a per-layer KV cache
 * (batch 1): the layer of ora_layer with the context-1 attention replaced by
 * decode attention over the cache.  The cache rows 0..pos-1 hold the earlier
 * tokens' binary16 keys and values; this token's k and v are rounded to
 * binary16 and stored in row pos (the cache the layer carries, PIPO summary,
 * Method, "Offloading architecture"), then every query head attends over
 * rows 0..pos (ora_attn_decode) and the attention output is rounded to
 * binary16 before the o projection.  With pos = 0 the softmax over one key is
 * 1 and the layer is ora_layer.  kc, vc: [capacity][kv_dim] binary16,
 * updated in row pos.  work must hold q_dim + 2*kv_dim + 3*hidden + 2*ffn +
 * 2*q_dim + (pos + 1) doubles, work16 hidden + q_dim + ffn binary16 values. */
void ora_layer_kv(const uint8_t *const *wts, const uint16_t *z, int64_t hidden, int64_t q_dim, int64_t kv_dim,
                  int64_t ffn, int64_t head_dim, double eps, uint16_t *kc, uint16_t *vc, int64_t pos,
                  double *work, uint16_t *work16, double *t2, uint16_t *z_out)
{
    double *q = work;
    double *k = q + q_dim;
    double *v = k + kv_dim;
    double *o = v + kv_dim;
    double *t1 = o + hidden;
    double *dn = t1 + hidden;
    double *g = dn + hidden;
    double *u = g + ffn;
    double *att = u + ffn;
    double *sabs = att + q_dim;
    double *aw = sabs + q_dim;
    uint16_t *attn = work16;
    uint16_t *z1 = attn + q_dim;
    uint16_t *act = z1 + hidden;
    int64_t n_q = q_dim / head_dim, n_kv = kv_dim / head_dim;

    ora_gemv(wts[0], z, q_dim, hidden, 1, 0, q_dim, q, 0);
    ora_gemv(wts[1], z, kv_dim, hidden, 1, 0, kv_dim, k, 0);
    ora_gemv(wts[2], z, kv_dim, hidden, 1, 0, kv_dim, v, 0);
    ora_double_to_half_n(k, kv_dim, kc + pos * kv_dim);
    ora_double_to_half_n(v, kv_dim, vc + pos * kv_dim);
    ora_attn_decode(q, kc, vc, pos + 1, n_q, n_kv, head_dim, att, sabs, aw);
    ora_double_to_half_n(att, q_dim, attn);
    ora_gemv(wts[3], attn, hidden, q_dim, 1, 0, hidden, o, 0);
    ora_add(z, o, hidden, t1);
    ora_rmsnorm_d(t1, 1, hidden, eps, z1);
    ora_gemv(wts[4], z1, ffn, hidden, 1, 0, ffn, g, 0);
    ora_gemv(wts[5], z1, ffn, hidden, 1, 0, ffn, u, 0);
    ora_silu_mul(g, u, ffn, act);
    ora_gemv(wts[6], act, hidden, ffn, 1, 0, hidden, dn, 0);
    ora_add(z1, dn, hidden, t2);
    ora_rmsnorm_d(t2, 1, hidden, eps, z_out);
}
