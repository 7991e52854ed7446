/*
 * mla_oracle.c -- plain, slow, fp64 CPU oracle for MLA latent-KV decode.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
 * execute this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg use it. It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Every result is computed in double precision straight from the bf16 input
 * bits (widening bf16 -> double is exact), with no intermediate rounding. The
 * only rounding is the final bf16 store of a cache row in mla_oracle_append_kv,
 * because the latent cache is bf16 storage by definition.
 *
 * Sources (web pages; cited by address and section):
 *  [V2]   sheratonhq.com/news/191949, "DeepSeek-V2 teardown: how MLA and MoE cut
 *         the KV cache by 93.3%", section 2.1 (MHA -> MLA): only the latent c_t is
 *         cached; the cache shrinks from 2*n_h*d_h*l to d_c*l elements; W_UK can be
 *         absorbed into W_Q and W_UV into W_O; queries are also low-rank
 *         compressed; a separate decoupled-RoPE branch carries position.
 *  [MW]   zskr.cn/news/1409628, "LLM inference: from the memory wall to the
 *         compute wall", section 2.1 (joint low-rank projection hidden 7168 ->
 *         latent 512; scores = (Q W_DK^T) CKV^T; decoupled RoPE) and section 2.2
 *         (layer reordering: associativity of the matrix products).
 *  [V3]   fsdata.site/2026/11/deepseek-v3-mla-optimization, sections 1-2 (the
 *         latent is projected back per head on the fly; per-token cache element
 *         table for MHA).
 *
 * Readings where the pages are silent (each one is a parameter or a stated
 * convention, never hidden):
 *  - the cache row of a token is [c_kv (d_c) | k_rope (d_rope)], k_rope already
 *    rotated to the token's position;
 *  - RoPE rotates consecutive pairs (2i, 2i+1) counter-clockwise by
 *    pos * theta^(-2i/d_rope); pos is the 0-based token index in its sequence;
 *  - the softmax scale is a parameter (1/sqrt(d_nope + d_rope) in the workloads);
 *  - lse is the natural log of the sum of exp(scaled logits); an empty sequence
 *    gives out = 0 and lse = -inf;
 *  - no normalisation layers (the pages name none).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_RANGE 4

/* ---------------------------------------------------------------- bf16 */

static double bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 value, ties to even, straight from fp64
 * (no detour through fp32, which would round twice). bf16 keeps 8 significant
 * bits; normal exponents reach down to 2^-126 and subnormals step by 2^-133. */
uint16_t mla_oracle_f64_to_bf16(double x)
{
    if (isnan(x))
        return 0x7FC0;
    double a = fabs(x);
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isinf(a))
        return sign | 0x7F80;
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);               /* a = m * 2^e, m in [0.5, 1) */
    double quantum = (e - 1 < -126) ? ldexp(1.0, -133) : ldexp(1.0, e - 8);
    double r = nearbyint(a / quantum) * quantum;   /* default mode: ties to even */
    if (r >= ldexp(1.0, 128))
        return sign | 0x7F80;
    float f = (float)r;                            /* exact: r has <= 8 bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------- RoPE */

/* Rotate x[0..d_rope) in place: pair (2i, 2i+1) by angle pos * theta^(-2i/d_rope). */
static void rope_rotate(double *x, int d_rope, int pos, double theta)
{
    for (int i = 0; i < d_rope / 2; ++i) {
        double freq = pow(theta, -2.0 * (double)i / (double)d_rope);
        double ang = (double)pos * freq;
        double c = cos(ang), s = sin(ang);
        double x0 = x[2 * i], x1 = x[2 * i + 1];
        x[2 * i] = x0 * c - x1 * s;
        x[2 * i + 1] = x0 * s + x1 * c;
    }
}

void mla_oracle_rope(double *x, int n_rows, int d_rope, const int32_t *pos, double theta)
{
    for (int r = 0; r < n_rows; ++r)
        rope_rotate(x + (size_t)r * d_rope, d_rope, pos[r], theta);
}

/* ------------------------------------------------- cache-size closed forms */

/* [V2] 2.1: standard attention caches K and V for every head and layer. */
long long mla_oracle_kv_elements_mha(int layers, int heads, int head_dim)
{
    return (long long)layers * 2 * heads * head_dim;
}

/* [V2] 2.1 + decoupled RoPE: MLA caches one latent (d_c) and one shared rotated
 * key (d_rope) per token and layer. */
long long mla_oracle_kv_elements_mla(int layers, int d_c, int d_rope)
{
    return (long long)layers * (d_c + d_rope);
}

/* ------------------------------------------------------------ paged cache */

/* Address of token j of sequence b in the paged cache, or NULL when the block
 * table entry is outside the pool. */
static const uint16_t *cache_row(const uint16_t *cache, int num_blocks, int block_size,
                                 int row_len, const int32_t *block_table, int max_blocks,
                                 int b, int j)
{
    int blk = block_table[(size_t)b * max_blocks + j / block_size];
    if (blk < 0 || blk >= num_blocks)
        return NULL;
    return cache + ((size_t)blk * block_size + (size_t)(j % block_size)) * row_len;
}

/* ------------------------------------------------------------------ append */

/*
 * [V2] 2.1, [MW] 2.1: the new token's hidden state h is projected down to the
 * latent c_kv = h W_DKV (d_model -> d_c), and the decoupled key k_rope = RoPE(h W_KR)
 * (d_model -> d_rope). Only [c_kv | k_rope] is cached, at slot pos[b] of sequence b.
 *
 * h [B][d_model] bf16; w_dkr [(d_c+d_rope)][d_model] bf16 (row n is output n);
 * pos [B]; block_table [B][max_blocks]; kv_cache [num_blocks][block_size][d_c+d_rope].
 */
int mla_oracle_append_kv(const uint16_t *h, int B, int d_model, const uint16_t *w_dkr,
                         int d_c, int d_rope, const int32_t *pos, const int32_t *block_table,
                         int max_blocks, uint16_t *kv_cache, int num_blocks, int block_size,
                         double rope_theta)
{
    int D = d_c + d_rope;
    if (B < 0 || d_model <= 0 || d_c <= 0 || d_rope < 0 || (d_rope & 1) || block_size <= 0)
        return ORC_ERR_ARG;
    double *x = (double *)malloc(sizeof(double) * (size_t)D);
    if (!x)
        return ORC_ERR_ARG;
    int status = ORC_OK;
    for (int b = 0; b < B; ++b) {
        int p = pos[b];
        if (p < 0 || p / block_size >= max_blocks) {
            status = ORC_ERR_RANGE;
            continue;
        }
        int blk = block_table[(size_t)b * max_blocks + p / block_size];
        if (blk < 0 || blk >= num_blocks) {
            status = ORC_ERR_RANGE;
            continue;
        }
        for (int n = 0; n < D; ++n) {
            double acc = 0.0;
            for (int k = 0; k < d_model; ++k)
                acc += bf16_to_f64(h[(size_t)b * d_model + k]) *
                       bf16_to_f64(w_dkr[(size_t)n * d_model + k]);
            x[n] = acc;
        }
        rope_rotate(x + d_c, d_rope, p, rope_theta);
        uint16_t *dst = kv_cache + ((size_t)blk * block_size + (size_t)(p % block_size)) * D;
        for (int n = 0; n < D; ++n)
            dst[n] = mla_oracle_f64_to_bf16(x[n]);
    }
    free(x);
    return status;
}

/* ------------------------------------------------------------- fp8 cache */

/*
 * FP8 latent cache ("LLM inference: from the memory wall to the compute wall" §5 names a
 * mixed-precision FP8/FP16 KV cache as the next step; "DeepSeek V3 MLA optimisation" turns
 * on FP8 quantisation of the KV cache). The pages fix no format; the reading taken here:
 *  - each value is stored as an e4m3 code: 1 sign bit, 4 exponent bits with bias 7, 3
 *    mantissa bits; exponent field 0 holds the subnormals m/8 * 2^-6; there are no
 *    infinities and the all-ones code of either sign is NaN, so the largest finite
 *    magnitude is 1.75 * 2^8 = 448;
 *  - rounding is to the nearest value, ties to the even mantissa, and magnitudes beyond
 *    448 saturate to 448;
 *  - every cached row (one token: [c_kv | k_rope]) carries one power-of-two scale 2^e,
 *    e the smallest integer with max|x| * 2^-e <= 448 (e = 0 for an all-zero row), and the
 *    codes hold x * 2^-e. The dequantised value is code * 2^e, exactly.
 */

/* Value of an e4m3 code, straight from the format definition (NaN codes give NaN). */
double mla_oracle_e4m3_to_f64(uint8_t code)
{
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7)
        return NAN;
    double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* The e4m3 code nearest to x (ties to the even mantissa; saturating at 448; the sign of
 * x is kept, also for a result of zero). NaN gives the positive NaN code. */
uint8_t mla_oracle_f64_to_e4m3(double x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    if (a >= 448.0)
        return sign | 0x7E;
    /* spacing of the representable values around a: 2^-9 below 2^-6, else 2^(E-3) for
     * a in [2^E, 2^(E+1)) */
    double quantum;
    if (a < ldexp(1.0, -6)) {
        quantum = ldexp(1.0, -9);
    } else {
        int E;
        frexp(a, &E); /* a = f * 2^E with f in [0.5, 1) */
        quantum = ldexp(1.0, (E - 1) - 3);
    }
    double n = nearbyint(a / quantum); /* exact division; default mode: ties to even */
    double v = n * quantum;            /* may step up to the next binade: still exact */
    if (v > 448.0)
        v = 448.0;
    if (v < ldexp(1.0, -6))
        return sign | (uint8_t)(v / ldexp(1.0, -9)); /* subnormal or zero: m = v / 2^-9 */
    int E;
    double f = frexp(v, &E); /* v = f * 2^E, f in [0.5, 1); as 1.mmm * 2^(E-1) */
    int mant = (int)((2.0 * f - 1.0) * 8.0);
    return sign | (uint8_t)(((E - 1 + 7) << 3) | mant);
}

/* One row of D values -> e4m3 codes and the exponent e of its power-of-two scale. */
void mla_oracle_quantize_row_fp8(const double *x, int D, uint8_t *codes, int8_t *e_out)
{
    double mx = 0.0;
    for (int n = 0; n < D; ++n)
        if (fabs(x[n]) > mx)
            mx = fabs(x[n]);
    int e = 0;
    if (mx > 0.0) {
        e = (int)ceil(log2(mx / 448.0));
        while (ldexp(mx, -e) > 448.0) /* make e the smallest with mx * 2^-e <= 448 */
            ++e;
        while (ldexp(mx, -(e - 1)) <= 448.0)
            --e;
        if (e < -126) /* the stored scale 2^-e stays a normal float: rows below 2^-117 */
            e = -126;
    }
    for (int n = 0; n < D; ++n)
        codes[n] = mla_oracle_f64_to_e4m3(ldexp(x[n], -e));
    *e_out = (int8_t)e;
}

/* rows x D values -> codes [rows][D] and exps [rows]. */
void mla_oracle_quantize_rows_fp8(const double *x, long rows, int D, uint8_t *codes,
                                  int8_t *exps)
{
    for (long r = 0; r < rows; ++r)
        mla_oracle_quantize_row_fp8(x + r * D, D, codes + r * D, exps + r);
}

/* codes [rows][D], exps [rows] -> the dequantised values code * 2^e. */
void mla_oracle_dequantize_rows_fp8(const uint8_t *codes, const int8_t *exps, long rows, int D,
                                    double *out)
{
    for (long r = 0; r < rows; ++r)
        for (int n = 0; n < D; ++n)
            out[r * D + n] = ldexp(mla_oracle_e4m3_to_f64(codes[r * D + n]), exps[r]);
}

/* mla_oracle_append_kv into an FP8 cache: the projected, rotated row (fp64) is quantised
 * as above and written as codes into kv_codes [num_blocks][block_size][D] and its exponent
 * into kv_exps [num_blocks][block_size]. */
int mla_oracle_append_kv_fp8(const uint16_t *h, int B, int d_model, const uint16_t *w_dkr,
                             int d_c, int d_rope, const int32_t *pos, const int32_t *block_table,
                             int max_blocks, uint8_t *kv_codes, int8_t *kv_exps, int num_blocks,
                             int block_size, double rope_theta)
{
    int D = d_c + d_rope;
    if (B < 0 || d_model <= 0 || d_c <= 0 || d_rope < 0 || (d_rope & 1) || block_size <= 0)
        return ORC_ERR_ARG;
    double *x = (double *)malloc(sizeof(double) * (size_t)D);
    if (!x)
        return ORC_ERR_ARG;
    int status = ORC_OK;
    for (int b = 0; b < B; ++b) {
        int p = pos[b];
        if (p < 0 || p / block_size >= max_blocks) {
            status = ORC_ERR_RANGE;
            continue;
        }
        int blk = block_table[(size_t)b * max_blocks + p / block_size];
        if (blk < 0 || blk >= num_blocks) {
            status = ORC_ERR_RANGE;
            continue;
        }
        for (int n = 0; n < D; ++n) {
            double acc = 0.0;
            for (int k = 0; k < d_model; ++k)
                acc += bf16_to_f64(h[(size_t)b * d_model + k]) *
                       bf16_to_f64(w_dkr[(size_t)n * d_model + k]);
            x[n] = acc;
        }
        rope_rotate(x + d_c, d_rope, p, rope_theta);
        size_t slot = (size_t)blk * block_size + (size_t)(p % block_size);
        mla_oracle_quantize_row_fp8(x, D, kv_codes + slot * D, kv_exps + slot);
    }
    free(x);
    return status;
}

/* ---------------------------------------------------- attention, absorbed */

/*
 * [V2] 2.1 (W_UK absorbed into the query side), [MW] 2.1-2.2 (scores =
 * (Q W_DK^T) CKV^T after reordering): every head of sequence b scores the shared
 * cached rows directly in latent space,
 *     s_j = scale * (q_lat . c_kv_j + q_rope . k_rope_j),   j < L_b,
 * p = softmax(s), and the latent output is o_lat = sum_j p_j c_kv_j (W_UV is
 * applied afterwards, on the output side). lse = ln sum_j exp(s_j).
 *
 * q_lat [B][H][d_c], q_rope [B][H][d_rope] (double); cache bf16 bits as above;
 * out [B][H][d_c]; lse [B][H]. probs, when not NULL, receives p for (b=0, h=0)
 * (length >= L_0). Returns ORC_ERR_RANGE (and skips that token) when a block
 * table entry needed by a valid token is outside the pool.
 */
int mla_oracle_decode_absorbed(const double *q_lat, const double *q_rope,
                               const uint16_t *kv_cache, int num_blocks, int block_size,
                               const int32_t *block_table, int max_blocks,
                               const int32_t *seqlens, int B, int H, int d_c, int d_rope,
                               double scale, double *out, double *lse, double *probs)
{
    int D = d_c + d_rope;
    int bad = 0;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] < 0 || (seqlens[b] + block_size - 1) / block_size > max_blocks)
            return ORC_ERR_ARG;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int bh = 0; bh < B * H; ++bh) {
        int b = bh / H;
        int L = seqlens[b];
        const double *ql = q_lat + (size_t)bh * d_c;
        const double *qr = q_rope + (size_t)bh * d_rope;
        double *o = out + (size_t)bh * d_c;
        for (int c = 0; c < d_c; ++c)
            o[c] = 0.0;
        double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        unsigned char *ok = (unsigned char *)malloc((size_t)(L > 0 ? L : 1));
        double m = -INFINITY;
        for (int j = 0; j < L; ++j) {
            const uint16_t *row = cache_row(kv_cache, num_blocks, block_size, D, block_table,
                                            max_blocks, b, j);
            ok[j] = row != NULL;
            if (!row) {
                bad = 1;
                s[j] = -INFINITY;
                continue;
            }
            double dot = 0.0;
            for (int c = 0; c < d_c; ++c)
                dot += ql[c] * bf16_to_f64(row[c]);
            for (int r = 0; r < d_rope; ++r)
                dot += qr[r] * bf16_to_f64(row[d_c + r]);
            s[j] = scale * dot;
            if (s[j] > m)
                m = s[j];
        }
        double den = 0.0;
        for (int j = 0; j < L; ++j)
            if (ok[j])
                den += exp(s[j] - m);
        for (int j = 0; j < L; ++j) {
            if (!ok[j])
                continue;
            double p = exp(s[j] - m) / den;
            if (bh == 0 && probs)
                probs[j] = p;
            const uint16_t *row = cache_row(kv_cache, num_blocks, block_size, D, block_table,
                                            max_blocks, b, j);
            for (int c = 0; c < d_c; ++c)
                o[c] += p * bf16_to_f64(row[c]);
        }
        lse[bh] = (den > 0.0) ? m + log(den) : -INFINITY;
        free(s);
        free(ok);
    }
    return bad ? ORC_ERR_RANGE : ORC_OK;
}

/* ---------------------------------------------------- attention, expanded */

/*
 * The definition the absorbed form must equal ([V2] 2.1, [V3] section 1: the
 * latent is projected back per head when attention needs it). For head i and
 * cached token j:
 *     k_i,j = [ W_UK_i c_kv_j  (d_h) | k_rope_j (d_rope) ],   v_i,j = W_UV_i c_kv_j,
 *     s_j = scale * (q_nope_i . (W_UK_i c_kv_j) + q_rope_i . k_rope_j),
 *     o_i = sum_j softmax(s)_j v_i,j,   lse_i = ln sum_j exp(s_j).
 * This is ordinary multi-head attention with a decoupled RoPE key shared by
 * all heads; K and V are materialised explicitly, one token at a time.
 *
 * q_nope [B][H][d_h], q_rope [B][H][d_rope], w_uk [H][d_h][d_c], w_uv [H][d_v][d_c]
 * (double); out_v [B][H][d_v]; lse [B][H].
 */
int mla_oracle_decode_expanded(const double *q_nope, const double *q_rope,
                               const uint16_t *kv_cache, int num_blocks, int block_size,
                               const int32_t *block_table, int max_blocks,
                               const int32_t *seqlens, int B, int H, int d_c, int d_rope,
                               int d_h, int d_v, const double *w_uk, const double *w_uv,
                               double scale, double *out_v, double *lse)
{
    int D = d_c + d_rope;
    int bad = 0;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] < 0 || (seqlens[b] + block_size - 1) / block_size > max_blocks)
            return ORC_ERR_ARG;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int bh = 0; bh < B * H; ++bh) {
        int b = bh / H, i = bh % H;
        int L = seqlens[b];
        const double *qn = q_nope + (size_t)bh * d_h;
        const double *qr = q_rope + (size_t)bh * d_rope;
        const double *Wk = w_uk + (size_t)i * d_h * d_c;
        const double *Wv = w_uv + (size_t)i * d_v * d_c;
        double *o = out_v + (size_t)bh * d_v;
        int n = L > 0 ? L : 1;
        double *s = (double *)malloc(sizeof(double) * (size_t)n);
        double *V = (double *)malloc(sizeof(double) * (size_t)n * d_v);
        double *c = (double *)malloc(sizeof(double) * (size_t)d_c);
        double *k = (double *)malloc(sizeof(double) * (size_t)d_h);
        unsigned char *ok = (unsigned char *)malloc((size_t)n);
        double m = -INFINITY;
        for (int j = 0; j < L; ++j) {
            const uint16_t *row = cache_row(kv_cache, num_blocks, block_size, D, block_table,
                                            max_blocks, b, j);
            ok[j] = row != NULL;
            if (!row) {
                bad = 1;
                s[j] = -INFINITY;
                continue;
            }
            for (int cc = 0; cc < d_c; ++cc)
                c[cc] = bf16_to_f64(row[cc]);
            /* explicit per-head key: k = W_UK_i c */
            for (int d = 0; d < d_h; ++d) {
                double acc = 0.0;
                for (int cc = 0; cc < d_c; ++cc)
                    acc += Wk[(size_t)d * d_c + cc] * c[cc];
                k[d] = acc;
            }
            /* explicit per-head value: v = W_UV_i c */
            for (int d = 0; d < d_v; ++d) {
                double acc = 0.0;
                for (int cc = 0; cc < d_c; ++cc)
                    acc += Wv[(size_t)d * d_c + cc] * c[cc];
                V[(size_t)j * d_v + d] = acc;
            }
            double dot = 0.0;
            for (int d = 0; d < d_h; ++d)
                dot += qn[d] * k[d];
            for (int r = 0; r < d_rope; ++r)
                dot += qr[r] * bf16_to_f64(row[d_c + r]);
            s[j] = scale * dot;
            if (s[j] > m)
                m = s[j];
        }
        double den = 0.0;
        for (int j = 0; j < L; ++j)
            if (ok[j])
                den += exp(s[j] - m);
        for (int d = 0; d < d_v; ++d)
            o[d] = 0.0;
        for (int j = 0; j < L; ++j) {
            if (!ok[j])
                continue;
            double p = exp(s[j] - m) / den;
            for (int d = 0; d < d_v; ++d)
                o[d] += p * V[(size_t)j * d_v + d];
        }
        lse[bh] = (den > 0.0) ? m + log(den) : -INFINITY;
        free(s);
        free(V);
        free(c);
        free(k);
        free(ok);
    }
    return bad ? ORC_ERR_RANGE : ORC_OK;
}

/* ------------------------------------------------------- split-KV combine */

/*
 * Merge of attention results over disjoint token ranges of one (b, h). Each
 * part s carries its own normalised output o_s and lse_s. The merged result is
 * the softmax over the union of the ranges:
 *     lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) o_s.
 * Parts with lse_s = -inf (empty ranges) weigh zero; if every part is empty,
 * out = 0 and lse = -inf. (Not on the pages: split-KV decoding is this
 * implementation's choice; this is the exact identity it relies on.)
 *
 * o_part [B][S][H][d], lse_part [B][S][H]; out [B][H][d]; lse [B][H].
 */
void mla_oracle_combine(const double *o_part, const double *lse_part, int B, int S, int H,
                        int d, double *out, double *lse)
{
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            double m = -INFINITY;
            for (int s = 0; s < S; ++s) {
                double l = lse_part[((size_t)b * S + s) * H + h];
                if (l > m)
                    m = l;
            }
            double *o = out + ((size_t)b * H + h) * d;
            for (int c = 0; c < d; ++c)
                o[c] = 0.0;
            if (m == -INFINITY) {
                lse[(size_t)b * H + h] = -INFINITY;
                continue;
            }
            double den = 0.0;
            for (int s = 0; s < S; ++s) {
                double l = lse_part[((size_t)b * S + s) * H + h];
                if (l != -INFINITY)
                    den += exp(l - m);
            }
            double tot = m + log(den);
            for (int s = 0; s < S; ++s) {
                double l = lse_part[((size_t)b * S + s) * H + h];
                if (l == -INFINITY)
                    continue;
                double wgt = exp(l - tot);
                const double *op = o_part + (((size_t)b * S + s) * H + h) * d;
                for (int c = 0; c < d; ++c)
                    o[c] += wgt * op[c];
            }
            lse[(size_t)b * H + h] = tot;
        }
}

/* ------------------------------------------------------ absorbed projections */

/*
 * Query side ([V2] 2.1: queries are low-rank compressed too, a decoupled RoPE
 * branch carries position, and W_UK is absorbed into the query projection;
 * [MW] 2.2: compute Q W_DK^T first, by associativity):
 *     c_q      = h W_DQ                         (d_model -> q_lora)
 *     q_nope_i = c_q W_UQ_i                     (q_lora -> d_h, per head)
 *     q_rope_i = RoPE(c_q W_QR_i, pos)          (q_lora -> d_rope, per head)
 *     q_lat_i  = W_UK_i^T q_nope_i              (d_h -> d_c)
 *
 * h [B][d_model]; w_dq [q_lora][d_model]; w_uq [H*d_h][q_lora]; w_qr [H*d_rope][q_lora];
 * w_uk [H][d_h][d_c] (bf16 bits). Outputs (double): q_lat [B][H][d_c],
 * q_rope [B][H][d_rope], and q_nope [B][H][d_h] when not NULL.
 */
int mla_oracle_absorb_q(const uint16_t *h, int B, int d_model, const uint16_t *w_dq, int q_lora,
                        const uint16_t *w_uq, const uint16_t *w_qr, const uint16_t *w_uk, int H,
                        int d_h, int d_rope, int d_c, const int32_t *pos, double rope_theta,
                        double *q_lat, double *q_rope, double *q_nope)
{
    if (B < 0 || H <= 0 || (d_rope & 1))
        return ORC_ERR_ARG;
    double *cq = (double *)malloc(sizeof(double) * (size_t)q_lora);
    double *qn = (double *)malloc(sizeof(double) * (size_t)d_h);
    for (int b = 0; b < B; ++b) {
        for (int r = 0; r < q_lora; ++r) {
            double acc = 0.0;
            for (int k = 0; k < d_model; ++k)
                acc += bf16_to_f64(h[(size_t)b * d_model + k]) *
                       bf16_to_f64(w_dq[(size_t)r * d_model + k]);
            cq[r] = acc;
        }
        for (int i = 0; i < H; ++i) {
            for (int d = 0; d < d_h; ++d) {
                double acc = 0.0;
                const uint16_t *w = w_uq + ((size_t)i * d_h + d) * q_lora;
                for (int r = 0; r < q_lora; ++r)
                    acc += cq[r] * bf16_to_f64(w[r]);
                qn[d] = acc;
                if (q_nope)
                    q_nope[((size_t)b * H + i) * d_h + d] = acc;
            }
            double *qr = q_rope + ((size_t)b * H + i) * d_rope;
            for (int d = 0; d < d_rope; ++d) {
                double acc = 0.0;
                const uint16_t *w = w_qr + ((size_t)i * d_rope + d) * q_lora;
                for (int r = 0; r < q_lora; ++r)
                    acc += cq[r] * bf16_to_f64(w[r]);
                qr[d] = acc;
            }
            rope_rotate(qr, d_rope, pos[b], rope_theta);
            double *ql = q_lat + ((size_t)b * H + i) * d_c;
            const uint16_t *wk = w_uk + (size_t)i * d_h * d_c;
            for (int c = 0; c < d_c; ++c) {
                double acc = 0.0;
                for (int d = 0; d < d_h; ++d)
                    acc += qn[d] * bf16_to_f64(wk[(size_t)d * d_c + c]);
                ql[c] = acc;
            }
        }
    }
    free(cq);
    free(qn);
    return ORC_OK;
}

/*
 * Output side ([V2] 2.1: W_UV is absorbed into the output projection):
 *     o_v_i = W_UV_i o_lat_i   (d_c -> d_v, per head),   y = W_O [o_v_1 | ... | o_v_H].
 * o_lat [B][H][d_c] (double); w_uv [H][d_v][d_c]; w_o [d_model][H*d_v] (bf16 bits);
 * y [B][d_model] (double).
 */
int mla_oracle_out_absorb(const double *o_lat, int B, int H, int d_c, int d_v,
                          const uint16_t *w_uv, const uint16_t *w_o, int d_model, double *y)
{
    double *ov = (double *)malloc(sizeof(double) * (size_t)H * d_v);
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < H; ++i)
            for (int d = 0; d < d_v; ++d) {
                double acc = 0.0;
                const uint16_t *w = w_uv + ((size_t)i * d_v + d) * d_c;
                const double *o = o_lat + ((size_t)b * H + i) * d_c;
                for (int c = 0; c < d_c; ++c)
                    acc += bf16_to_f64(w[c]) * o[c];
                ov[(size_t)i * d_v + d] = acc;
            }
        for (int n = 0; n < d_model; ++n) {
            double acc = 0.0;
            const uint16_t *w = w_o + (size_t)n * H * d_v;
            for (int k = 0; k < H * d_v; ++k)
                acc += bf16_to_f64(w[k]) * ov[k];
            y[(size_t)b * d_model + n] = acc;
        }
    }
    free(ov);
    return ORC_OK;
}
