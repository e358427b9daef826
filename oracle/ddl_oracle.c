/*
 * ddl_oracle.c -- plain, slow, fp64 CPU reference of one batch-B decode step
 * of a GQA transformer decoder layer with 4-bit (or bf16) weights.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this file.  It shares no
 * code, header, table or constant with the CUDA library and includes none of
 * its files.
 *
 * Sources (cited as page title + section):
 *  - "把基础打牢" primer, §1.1 block pseudo-code: rmsnorm -> q,k,v projections
 *    -> split heads -> rope -> causal softmax attention -> merge heads ->
 *    y = x + attn Wo -> z = y + ffn(rmsnorm(y)).
 *  - same primer, §1.2 decode_step: per layer load the KV history, run the
 *    block on one new token, append its k,v to the cache.
 *  - Unsloth/Qwen-27B article (zhichai.top), §二.1 fused SwiGLU formula:
 *    silu(x Wg) elementwise-times (x Wu); §二.2 GQA: several query heads share
 *    one K/V head; §二.3 4-bit weights expanded with their scale on arrival.
 *  - roofline reply (zhichai.net), §五: RoPE rotates q and k by dimension pairs.
 *
 * Readings where the pages are silent (the plainest reading the rest supports):
 *  - RMSNorm: x * w / sqrt(mean(x^2) + eps), eps inside the root.
 *  - RoPE: half-split pairs (i, i + hd/2), theta_i = base^(-2i/hd), angle
 *    pos * theta_i, applied to q and k after the projection.
 *  - GQA mapping: query head h uses K/V head floor(h / (H_q / H_kv)).
 *  - INT4: symmetric, group 64 along K, s = bf16_rne(absmax / 7),
 *    q = clamp(round_half_even(w / s), -7, 7); all-zero group -> s = 0, q = 0;
 *    two codes per byte, even k in the low nibble, 4-bit two's complement.
 *  - The new k (after RoPE) and v are stored as bf16 (round to nearest even)
 *    and attention reads the stored values; nothing else is rounded.
 *  - No projection biases.
 *
 * Everything is fp64; bf16 values are widened exactly.  Loops run in the
 * plain order of the definitions; OpenMP only splits independent outputs.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 */

/* Exact widening of a bf16 bit pattern (the top half of an fp32). */
double orc_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round an fp64 value to the nearest bf16 (ties to even), one rounding.
 * bf16 = 1 sign, 8 exponent (bias 127, same range as fp32), 7 fraction bits;
 * subnormals have quantum 2^-133. */
uint16_t orc_bf16_from_f64(double x) {
    if (isnan(x)) return (uint16_t)(signbit(x) ? 0xFFC0u : 0x7FC0u);
    uint16_t sign = signbit(x) ? 0x8000u : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    int e2;
    frexp(a, &e2);                 /* a = m * 2^e2, m in [0.5, 1) */
    int qexp = e2 - 8;             /* 8 significant bits: quantum 2^(e2-8) */
    if (qexp < -133) qexp = -133;  /* subnormal quantum */
    double n = ldexp(a, -qexp);    /* exact: power-of-two scaling */
    double r = rint(n);            /* default mode: round half to even */
    double v = ldexp(r, qexp);
    if (v >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
    float f = (float)v;            /* exact: v has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

void orc_bf16_from_f64_array(const double* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_from_f64(x[i]);
}

/* ------------------------------------------------------------- INT4 codes */

#define ORC_GROUP 64

/* Code of weight k in row n of a packed [N][K/2] matrix. */
static int code_at(const uint8_t* q, int64_t K, int64_t n, int64_t k) {
    uint8_t byte = q[n * (K / 2) + k / 2];
    int nib = (k & 1) ? (byte >> 4) : (byte & 0xF);
    return nib >= 8 ? nib - 16 : nib; /* 4-bit two's complement */
}

/* Dequantized weight q * s (exact in fp64). */
static double w_int4(const uint8_t* q, const uint16_t* s, int64_t K,
                     int64_t n, int64_t k) {
    return (double)code_at(q, K, n, k) * orc_bf16_to_f64(s[n * (K / ORC_GROUP) + k / ORC_GROUP]);
}

/* Symmetric INT4 quantization, group 64 along K (4-bit weights expanded
 * with their per-group scale, Unsloth article §二.3). */
void orc_quantize_int4(const uint16_t* w, int64_t N, int64_t K,
                       uint8_t* q_out, uint16_t* s_out) {
    int64_t G = K / ORC_GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < G; ++g) {
            double absmax = 0.0;
            for (int64_t j = 0; j < ORC_GROUP; ++j) {
                double v = fabs(orc_bf16_to_f64(w[n * K + g * ORC_GROUP + j]));
                if (v > absmax) absmax = v;
            }
            uint16_t sb = orc_bf16_from_f64(absmax / 7.0);
            double s = orc_bf16_to_f64(sb);
            s_out[n * G + g] = sb;
            for (int64_t j = 0; j < ORC_GROUP; ++j) {
                int64_t k = g * ORC_GROUP + j;
                int c = 0;
                if (s != 0.0) {
                    double r = rint(orc_bf16_to_f64(w[n * K + k]) / s);
                    if (r > 7.0) r = 7.0;
                    if (r < -7.0) r = -7.0;
                    c = (int)r;
                }
                uint8_t nib = (uint8_t)(c & 0xF);
                uint8_t* byte = &q_out[n * (K / 2) + k / 2];
                if ((k & 1) == 0) *byte = nib;              /* even k: low nibble */
                else *byte = (uint8_t)(*byte | (nib << 4)); /* odd k: high nibble */
            }
        }
    }
}

/* Unpack codes to int8 [N][K] (for tests of the packed format). */
void orc_unpack_int4(const uint8_t* q, int64_t N, int64_t K, int8_t* codes) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) codes[n * K + k] = (int8_t)code_at(q, K, n, k);
}

/* ------------------------------------------------------------ primitives */

/* y[n] = sum_k W[n][k] x[k], W = q*s dequantized. */
void orc_gemv_int4(const uint8_t* q, const uint16_t* s, int64_t N, int64_t K,
                   const double* x, double* y) {
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += w_int4(q, s, K, n, k) * x[k];
        y[n] = acc;
    }
}

/* y[n] = sum_k W[n][k] x[k], W bf16 [N][K]. */
void orc_gemv_bf16(const uint16_t* w, int64_t N, int64_t K, const double* x, double* y) {
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += orc_bf16_to_f64(w[n * K + k]) * x[k];
        y[n] = acc;
    }
}

/* RMSNorm (primer §1.1 step 1): out = x * w / sqrt(mean(x^2) + eps). */
void orc_rmsnorm(const double* x, const uint16_t* w, int64_t D, double eps, double* out) {
    double ss = 0.0;
    for (int64_t i = 0; i < D; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss / (double)D + eps);
    for (int64_t i = 0; i < D; ++i) out[i] = x[i] * r * orc_bf16_to_f64(w[i]);
}

/* RoPE on one head vector in place: pair (i, i + hd/2) rotated by
 * pos * base^(-2i/hd) (roofline reply §五; primer §1.1 apply_rope). */
void orc_rope(double* v, int64_t hd, int64_t pos, double base) {
    int64_t half = hd / 2;
    for (int64_t i = 0; i < half; ++i) {
        double theta = pow(base, -2.0 * (double)i / (double)hd);
        double phi = (double)pos * theta;
        double c = cos(phi), sn = sin(phi);
        double a = v[i], b = v[i + half];
        v[i] = a * c - b * sn;
        v[i + half] = a * sn + b * c;
    }
}

/* Causal softmax attention of one new query token over keys 0..n_keys-1 of
 * one sequence (primer §1.1 step 6; GQA sharing, Unsloth article §二.2).
 * q: [H_q][hd]; kc, vc: [H_kv][s_max][hd] bf16; out: [H_q][hd].
 * probs (optional): [H_q][n_keys] softmax weights. */
void orc_attention(const double* q, const uint16_t* kc, const uint16_t* vc,
                   int64_t H_q, int64_t H_kv, int64_t hd, int64_t s_max,
                   int64_t n_keys, double* out, double* probs) {
    int64_t G = H_q / H_kv;
    double scale = 1.0 / sqrt((double)hd);
#pragma omp parallel for schedule(static)
    for (int64_t h = 0; h < H_q; ++h) {
        int64_t g = h / G;
        double* sc = (double*)malloc((size_t)n_keys * sizeof(double));
        double m = -INFINITY;
        for (int64_t t = 0; t < n_keys; ++t) {
            const uint16_t* kr = kc + (g * s_max + t) * hd;
            double acc = 0.0;
            for (int64_t d = 0; d < hd; ++d) acc += q[h * hd + d] * orc_bf16_to_f64(kr[d]);
            sc[t] = acc * scale;
            if (sc[t] > m) m = sc[t];
        }
        double l = 0.0;
        for (int64_t t = 0; t < n_keys; ++t) {
            sc[t] = exp(sc[t] - m);
            l += sc[t];
        }
        for (int64_t d = 0; d < hd; ++d) out[h * hd + d] = 0.0;
        for (int64_t t = 0; t < n_keys; ++t) {
            double p = sc[t] / l;
            if (probs) probs[h * n_keys + t] = p;
            const uint16_t* vr = vc + (g * s_max + t) * hd;
            for (int64_t d = 0; d < hd; ++d) out[h * hd + d] += p * orc_bf16_to_f64(vr[d]);
        }
        free(sc);
    }
}

/* ------------------------------------------------------------------ layer */

typedef struct {
    int64_t D, H_q, H_kv, head_dim, d_ff;
    double rope_base, eps;
} orc_shape;

/* A weight matrix [N][K]: INT4 (q [N][K/2], s [N][K/64]) when q != NULL,
 * otherwise bf16 w [N][K]. */
typedef struct {
    const uint8_t* q;
    const uint16_t* s;
    const uint16_t* w;
} orc_mat;

typedef struct {
    const uint16_t* norm1;
    orc_mat wq, wk, wv, wo;
    const uint16_t* norm2;
    orc_mat wg, wu, wd;
} orc_layer;

/* Optional per-stage outputs for one layer, each [B][...] fp64 (may be NULL). */
typedef struct {
    double* h;    /* [B][D]    rmsnorm(x, norm1) */
    double* q;    /* [B][Nq]   after RoPE */
    double* k;    /* [B][Nkv]  after RoPE, before bf16 storage */
    double* v;    /* [B][Nkv] */
    double* attn; /* [B][Nq]   merged heads */
    double* y;    /* [B][D] */
    double* a;    /* [B][d_ff] silu(g) * u */
} orc_stages;

static void gemv(const orc_mat* m, int64_t N, int64_t K, const double* x, double* y) {
    if (m->q) orc_gemv_int4(m->q, m->s, N, K, x, y);
    else orc_gemv_bf16(m->w, N, K, x, y);
}

/* One decode step of one layer for B sequences at the same position pos
 * (primer §1.2 decode_step body).  kc/vc: [B][H_kv][s_max][hd] bf16, slots
 * 0..pos-1 hold history; slot pos is written here.  x, z: [B][D]. */
int orc_layer_decode(const orc_shape* sh, const orc_layer* L, uint16_t* kc, uint16_t* vc,
                     int64_t s_max, int64_t B, int64_t pos, const double* x, double* z,
                     const orc_stages* st) {
    int64_t D = sh->D, hd = sh->head_dim, Hq = sh->H_q, Hkv = sh->H_kv, F = sh->d_ff;
    int64_t Nq = Hq * hd, Nkv = Hkv * hd;
    if (pos < 0 || pos >= s_max || Hq % Hkv != 0 || hd % 2 != 0) return -1;
    double* h = malloc(sizeof(double) * D);
    double* h2 = malloc(sizeof(double) * D);
    double* q = malloc(sizeof(double) * Nq);
    double* k = malloc(sizeof(double) * Nkv);
    double* v = malloc(sizeof(double) * Nkv);
    double* o = malloc(sizeof(double) * Nq);
    double* y = malloc(sizeof(double) * D);
    double* t = malloc(sizeof(double) * (D > F ? D : F));
    double* gg = malloc(sizeof(double) * F);
    double* uu = malloc(sizeof(double) * F);
    for (int64_t b = 0; b < B; ++b) {
        const double* xb = x + b * D;
        uint16_t* kcb = kc + b * Hkv * s_max * hd;
        uint16_t* vcb = vc + b * Hkv * s_max * hd;
        /* h = rmsnorm(x); q,k,v = h W */
        orc_rmsnorm(xb, L->norm1, D, sh->eps, h);
        gemv(&L->wq, Nq, D, h, q);
        gemv(&L->wk, Nkv, D, h, k);
        gemv(&L->wv, Nkv, D, h, v);
        /* split heads, rope on q and k */
        for (int64_t hh = 0; hh < Hq; ++hh) orc_rope(q + hh * hd, hd, pos, sh->rope_base);
        for (int64_t g = 0; g < Hkv; ++g) orc_rope(k + g * hd, hd, pos, sh->rope_base);
        /* append the new k, v to the cache (bf16) */
        for (int64_t g = 0; g < Hkv; ++g)
            for (int64_t d = 0; d < hd; ++d) {
                kcb[(g * s_max + pos) * hd + d] = orc_bf16_from_f64(k[g * hd + d]);
                vcb[(g * s_max + pos) * hd + d] = orc_bf16_from_f64(v[g * hd + d]);
            }
        /* attention over slots 0..pos, merge heads */
        orc_attention(q, kcb, vcb, Hq, Hkv, hd, s_max, pos + 1, o, NULL);
        /* y = x + attn Wo */
        gemv(&L->wo, D, Nq, o, t);
        for (int64_t i = 0; i < D; ++i) y[i] = xb[i] + t[i];
        /* z = y + ffn(rmsnorm(y)), ffn = (silu(h2 Wg) * (h2 Wu)) Wd */
        if (st && st->h) memcpy(st->h + b * D, h, sizeof(double) * D);
        orc_rmsnorm(y, L->norm2, D, sh->eps, h2);
        gemv(&L->wg, F, D, h2, gg);
        gemv(&L->wu, F, D, h2, uu);
        for (int64_t i = 0; i < F; ++i) gg[i] = gg[i] / (1.0 + exp(-gg[i])) * uu[i];
        gemv(&L->wd, D, F, gg, t);
        for (int64_t i = 0; i < D; ++i) z[b * D + i] = y[i] + t[i];
        if (st) {
            if (st->q) memcpy(st->q + b * Nq, q, sizeof(double) * Nq);
            if (st->k) memcpy(st->k + b * Nkv, k, sizeof(double) * Nkv);
            if (st->v) memcpy(st->v + b * Nkv, v, sizeof(double) * Nkv);
            if (st->attn) memcpy(st->attn + b * Nq, o, sizeof(double) * Nq);
            if (st->y) memcpy(st->y + b * D, y, sizeof(double) * D);
            if (st->a) memcpy(st->a + b * F, gg, sizeof(double) * F);
        }
    }
    free(h); free(h2); free(q); free(k); free(v); free(o); free(y); free(t); free(gg); free(uu);
    return 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
