/*
 * oracle.c - plain, slow CPU reference of the batch-1 quantized decode step.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load, call or link this code.  The engine
 * never does, and this file shares no code, header, table or helper with it.
 *
 * What it computes (one decoder step of a dense Qwen2/Qwen3-style
 * grouped-query-attention decoder whose linear layers hold weight-only
 * quantized codes):
 *   x  = embedding row of the token
 *   per layer:
 *     n   = RMSNorm(x)                              [naive Qwen engine, "RMSNorm"]
 *     q,k,v = W_{q,k,v} n (+ bias)                  [How To Construct..., §3-§4]
 *     (Qwen3 only) per-head RMSNorm of q and k
 *     RoPE on q and k at the token's position       [naive Qwen engine, "Rope"]
 *     k,v rounded to bfloat16 and stored at `pos`
 *     o_h = softmax(q_h . K_g / sqrt(d)) V_g  over positions 0..pos, g = h / (Hq/Hkv)
 *                                               [Bare-Metal LLM Inference on H100,
 *                                                "Architectural Blueprint" (GQA 7:1)]
 *     x  += W_o o
 *     n2  = RMSNorm(x)
 *     x  += W_down (silu(W_gate n2) * (W_up n2))   [naive Qwen engine, "SwiGLU"]
 *   logits = W_lm RMSNorm(x);  token = argmax (lowest index on ties)
 *                                               [FlashQwen, "Stage 5 - GPU argmax"]
 *
 * Weight formats:
 *   INT4, group 128, symmetric, zero point 0, one bfloat16 scale per group
 *   per output row: W[n][k] = code[n][k] * scale[n][k/128]
 *   ["How To Construct...", §3; "Bare-Metal...", "Architectural Blueprint"].
 *   Codes are two's-complement nibbles in [-8, 7] packed eight to a uint32 in
 *   the ValueShuffle order: logical lane i of an octet sits at bit shift
 *   {0,16,4,20,8,24,12,28}[i] ["How To Construct...", §7, the lane-map switch].
 *   Words are row-major, K-contiguous: word (n, k/8) holds codes k..k+7.
 *
 *   INT8, symmetric, one fp32 scale per output row, codes in natural byte
 *   order, row-major [N][K] ["FlashQwen", "Stage 8 - INT8 weight quantization"].
 *
 * Precision.  Compiled twice from this one file: with OR_REAL=float the
 * arithmetic is the FP32 decoder the acceptance criterion names; with
 * OR_REAL=double the same steps run in fp64, which bounds the fp32 variant's
 * own rounding.  Every sum is a plain left-to-right loop over its index, so
 * results do not depend on the number of OpenMP threads.  RoPE angles are
 * always formed in double.  The KV cache stores bfloat16 (round to nearest
 * even) in both variants, as the configuration prescribes.
 *
 * Readings taken where the pages are silent:
 *   - RoPE pairs element i with element i + d/2 of a head ("rotate half"),
 *     theta_i = base^(-2i/d), angle = pos * theta_i.
 *   - softmax scale is 1/sqrt(d); the new token attends to itself.
 *   - SwiGLU's gate (the matrix inside Swish) is gate_proj; silu(a) = a/(1+e^-a).
 *   - argmax ties resolve to the lowest index.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef OR_REAL
#define OR_REAL float
#define OR_PREFIX(name) or_f32_##name
#define OR_EXP expf
#define OR_SQRT sqrtf
#else
#define OR_PREFIX(name) or_f64_##name
#define OR_EXP exp
#define OR_SQRT sqrt
#endif

typedef OR_REAL real_t;

/* ------------------------------------------------------------------ */
/* bfloat16 storage                                                     */
/* ------------------------------------------------------------------ */

static inline float bf16_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* float -> bfloat16, round to nearest, ties to even (finite inputs). */
static inline uint16_t float_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ */
/* Integer work: pack / unpack (shared by both variants; defined once)  */
/* ------------------------------------------------------------------ */
#ifndef OR_DOUBLE_BUILD

/* ValueShuffle: logical lane i of an octet -> bit position of its nibble. */
static const int kLaneShift[8] = {0, 16, 4, 20, 8, 24, 12, 28};

/* codes[N][K] (int8 in [-8,7]) -> words[N][K/8].  K % 8 == 0. */
void or_pack_int4(const int8_t *codes, int64_t N, int64_t K, uint32_t *words) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t w = 0; w < K / 8; ++w) {
            uint32_t word = 0;
            for (int i = 0; i < 8; ++i) {
                uint32_t nib = (uint32_t)(uint8_t)codes[n * K + w * 8 + i] & 0xFu;
                word |= nib << kLaneShift[i];
            }
            words[n * (K / 8) + w] = word;
        }
}

/* words[N][K/8] -> codes[N][K]: mask four bits, sign-extend bit 3. */
void or_unpack_int4(const uint32_t *words, int64_t N, int64_t K, int8_t *codes) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t w = 0; w < K / 8; ++w) {
            uint32_t word = words[n * (K / 8) + w];
            for (int i = 0; i < 8; ++i) {
                int v = (int)((word >> kLaneShift[i]) & 0xFu);
                if (v & 0x8) v -= 16;
                codes[n * K + w * 8 + i] = (int8_t)v;
            }
        }
}

uint16_t or_bf16_round(float f) { return float_to_bf16(f); }

int64_t or_argmax(const float *v, int64_t n) {
    int64_t best = 0;
    for (int64_t i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}

/* Host threads of the parallel loops (timing only: results do not depend on it). */
int or_threads(void) { return omp_get_max_threads(); }
void or_set_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }

#endif /* !OR_DOUBLE_BUILD */

/* One INT4 code at (n, k) of a packed matrix with K columns. */
static inline int int4_code(const uint32_t *words, int64_t K, int64_t n, int64_t k) {
    static const int shift[8] = {0, 16, 4, 20, 8, 24, 12, 28};
    uint32_t word = words[n * (K / 8) + k / 8];
    int v = (int)((word >> shift[k % 8]) & 0xFu);
    return (v & 0x8) ? v - 16 : v;
}

/* ------------------------------------------------------------------ */
/* Elementwise pieces                                                   */
/* ------------------------------------------------------------------ */

/* RMSNorm: y_i = gamma_i * x_i / sqrt(mean(x^2) + eps)   [naive Qwen engine, "RMSNorm"] */
void OR_PREFIX(rmsnorm)(const real_t *x, const uint16_t *gamma, int64_t n, float eps, real_t *y) {
    real_t ss = 0;
    for (int64_t i = 0; i < n; ++i) ss += x[i] * x[i];
    real_t inv = (real_t)1 / OR_SQRT(ss / (real_t)n + (real_t)eps);
    for (int64_t i = 0; i < n; ++i) y[i] = (real_t)bf16_to_float(gamma[i]) * (x[i] * inv);
}

/* RoPE on n_heads heads of width d at position pos, in place.
 * [naive Qwen engine, "Rope": a 2-D rotation by a position-proportional angle] */
void OR_PREFIX(rope)(real_t *v, int64_t n_heads, int64_t d, int64_t pos, double base) {
    int64_t half = d / 2;
    for (int64_t h = 0; h < n_heads; ++h) {
        real_t *x = v + h * d;
        for (int64_t i = 0; i < half; ++i) {
            double theta = pow(base, -2.0 * (double)i / (double)d);
            double ang = (double)pos * theta;
            real_t c = (real_t)cos(ang), s = (real_t)sin(ang);
            real_t a = x[i], b = x[i + half];
            x[i] = a * c - b * s;
            x[i + half] = b * c + a * s;
        }
    }
}

/* softmax over n scores (max-subtracted). */
void OR_PREFIX(softmax)(const real_t *s, int64_t n, real_t *p) {
    real_t m = s[0];
    for (int64_t i = 1; i < n; ++i)
        if (s[i] > m) m = s[i];
    real_t z = 0;
    for (int64_t i = 0; i < n; ++i) {
        p[i] = OR_EXP(s[i] - m);
        z += p[i];
    }
    for (int64_t i = 0; i < n; ++i) p[i] /= z;
}

static inline real_t silu(real_t a) { return a / ((real_t)1 + OR_EXP(-a)); }

void OR_PREFIX(silu_mul)(const real_t *gate, const real_t *up, int64_t n, real_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = silu(gate[i]) * up[i];
}

/* ------------------------------------------------------------------ */
/* Matrix-vector products.  absacc (optional) receives sum_k |W_nk x_k|  */
/* so that tests can bound rounding error per output.                   */
/* ------------------------------------------------------------------ */

void OR_PREFIX(gemv_int4)(const uint32_t *words, const uint16_t *scales, const uint16_t *bias,
                          int64_t N, int64_t K, const real_t *x, real_t *y, real_t *absacc) {
    int64_t G = K / 128;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        real_t acc = 0, aacc = 0;
        for (int64_t k = 0; k < K; ++k) {
            real_t w = (real_t)int4_code(words, K, n, k) * (real_t)bf16_to_float(scales[n * G + k / 128]);
            acc += w * x[k];
            aacc += fabs((double)(w * x[k]));
        }
        if (bias) acc += (real_t)bf16_to_float(bias[n]);
        y[n] = acc;
        if (absacc) absacc[n] = aacc;
    }
}

void OR_PREFIX(gemv_int8)(const int8_t *codes, const float *scales, int64_t N, int64_t K,
                          const real_t *x, real_t *y, real_t *absacc) {
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        real_t acc = 0, aacc = 0;
        for (int64_t k = 0; k < K; ++k) {
            real_t w = (real_t)codes[n * K + k] * (real_t)scales[n];
            acc += w * x[k];
            aacc += fabs((double)(w * x[k]));
        }
        y[n] = acc;
        if (absacc) absacc[n] = aacc;
    }
}

void OR_PREFIX(gemv_bf16)(const uint16_t *w, int64_t N, int64_t K, const real_t *x, real_t *y,
                          real_t *absacc) {
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        real_t acc = 0, aacc = 0;
        for (int64_t k = 0; k < K; ++k) {
            real_t t = (real_t)bf16_to_float(w[n * K + k]) * x[k];
            acc += t;
            aacc += fabs((double)t);
        }
        y[n] = acc;
        if (absacc) absacc[n] = aacc;
    }
}

/* ------------------------------------------------------------------ */
/* Grouped-query attention of one new token over positions 0..T-1.      */
/* k_cache/v_cache: bfloat16 [T][Hkv][d] for one layer.                 */
/* ------------------------------------------------------------------ */
void OR_PREFIX(attention)(const real_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                          int64_t T, int64_t Hq, int64_t Hkv, int64_t d, real_t *out) {
    int64_t group = Hq / Hkv;
    real_t scale = (real_t)1 / OR_SQRT((real_t)d);
#pragma omp parallel for schedule(static)
    for (int64_t h = 0; h < Hq; ++h) {
        int64_t g = h / group;
        real_t *s = (real_t *)malloc(sizeof(real_t) * (size_t)T);
        real_t *p = (real_t *)malloc(sizeof(real_t) * (size_t)T);
        for (int64_t t = 0; t < T; ++t) {
            const uint16_t *kr = k_cache + (t * Hkv + g) * d;
            real_t dot = 0;
            for (int64_t i = 0; i < d; ++i) dot += q[h * d + i] * (real_t)bf16_to_float(kr[i]);
            s[t] = dot * scale;
        }
        OR_PREFIX(softmax)(s, T, p);
        for (int64_t i = 0; i < d; ++i) {
            real_t acc = 0;
            for (int64_t t = 0; t < T; ++t)
                acc += p[t] * (real_t)bf16_to_float(v_cache[(t * Hkv + g) * d + i]);
            out[h * d + i] = acc;
        }
        free(s);
        free(p);
    }
}

/* ------------------------------------------------------------------ */
/* The whole decoder step.                                              */
/* ------------------------------------------------------------------ */

/* Mirrors the field order of the Python-side ctypes structures. */
typedef struct {
    int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, mlp, vocab;
    float rms_eps, rope_base;
    int32_t qkv_bias, qk_norm, tied_lm_head;
    int32_t weight_format; /* 1 = INT4 group-128 bf16 scales, 2 = INT8 per-row fp32 scales */
} or_config;

typedef struct {
    const void *wq, *sq, *bq;
    const void *wk, *sk, *bk;
    const void *wv, *sv, *bv;
    const void *wo, *so;
    const void *wg, *sg;
    const void *wu, *su;
    const void *wd, *sd;
    const uint16_t *attn_norm, *mlp_norm, *q_norm, *k_norm;
} or_layer;

typedef struct {
    const uint16_t *embed;      /* bf16 [V][h] */
    const uint16_t *final_norm; /* bf16 [h] */
    const void *lm_head;        /* bf16 [V][h], or int8 [V][h] with lm_scale */
    const float *lm_scale;      /* fp32 [V] for the INT8 format, else NULL */
    const or_layer *layers;     /* [n_layers] */
} or_weights;

static void linear(const or_config *c, const void *w, const void *s, const void *b, int64_t N,
                   int64_t K, const real_t *x, real_t *y) {
    if (c->weight_format == 1)
        OR_PREFIX(gemv_int4)((const uint32_t *)w, (const uint16_t *)s, (const uint16_t *)b, N, K, x, y,
                             NULL);
    else {
        OR_PREFIX(gemv_int8)((const int8_t *)w, (const float *)s, N, K, x, y, NULL);
        if (b)
            for (int64_t n = 0; n < N; ++n) y[n] += (real_t)bf16_to_float(((const uint16_t *)b)[n]);
    }
}

/*
 * One decode step: consume `token` at position `pos`, append its K/V to the
 * caches (bf16 [L][t_max][Hkv][d]) and write the logits [V] (as float).
 * hidden_out (optional) receives the final residual x [h] before the last norm.
 * Returns 0, or -1 on bad arguments.
 */
int OR_PREFIX(step)(const or_config *c, const or_weights *W, uint16_t *k_cache, uint16_t *v_cache,
                    int64_t t_max, int32_t token, int64_t pos, float *logits, float *hidden_out) {
    const int64_t h = c->hidden, Hq = c->n_q_heads, Hkv = c->n_kv_heads, d = c->head_dim;
    const int64_t F = c->mlp, V = c->vocab;
    if (pos < 0 || pos >= t_max || token < 0 || token >= V || Hq % Hkv != 0 || Hq * d != h)
        return -1;

    real_t *x = calloc((size_t)h, sizeof(real_t));
    real_t *n = calloc((size_t)(F > h ? F : h), sizeof(real_t));
    real_t *q = calloc((size_t)(Hq * d), sizeof(real_t));
    real_t *k = calloc((size_t)(Hkv * d), sizeof(real_t));
    real_t *v = calloc((size_t)(Hkv * d), sizeof(real_t));
    real_t *o = calloc((size_t)h, sizeof(real_t));
    real_t *ga = calloc((size_t)F, sizeof(real_t));
    real_t *up = calloc((size_t)F, sizeof(real_t));
    real_t *u = calloc((size_t)F, sizeof(real_t));
    real_t *tmp = calloc((size_t)(V > F ? V : F), sizeof(real_t));

    for (int64_t i = 0; i < h; ++i) x[i] = (real_t)bf16_to_float(W->embed[(int64_t)token * h + i]);

    for (int64_t l = 0; l < c->n_layers; ++l) {
        const or_layer *L = &W->layers[l];
        uint16_t *kc = k_cache + l * t_max * Hkv * d;
        uint16_t *vc = v_cache + l * t_max * Hkv * d;

        OR_PREFIX(rmsnorm)(x, L->attn_norm, h, c->rms_eps, n);
        linear(c, L->wq, L->sq, c->qkv_bias ? L->bq : NULL, Hq * d, h, n, q);
        linear(c, L->wk, L->sk, c->qkv_bias ? L->bk : NULL, Hkv * d, h, n, k);
        linear(c, L->wv, L->sv, c->qkv_bias ? L->bv : NULL, Hkv * d, h, n, v);
        if (c->qk_norm) {
            for (int64_t hh = 0; hh < Hq; ++hh) {
                OR_PREFIX(rmsnorm)(q + hh * d, L->q_norm, d, c->rms_eps, tmp);
                memcpy(q + hh * d, tmp, sizeof(real_t) * (size_t)d);
            }
            for (int64_t hh = 0; hh < Hkv; ++hh) {
                OR_PREFIX(rmsnorm)(k + hh * d, L->k_norm, d, c->rms_eps, tmp);
                memcpy(k + hh * d, tmp, sizeof(real_t) * (size_t)d);
            }
        }
        OR_PREFIX(rope)(q, Hq, d, pos, (double)c->rope_base);
        OR_PREFIX(rope)(k, Hkv, d, pos, (double)c->rope_base);
        for (int64_t i = 0; i < Hkv * d; ++i) {
            kc[pos * Hkv * d + i] = float_to_bf16((float)k[i]);
            vc[pos * Hkv * d + i] = float_to_bf16((float)v[i]);
        }
        OR_PREFIX(attention)(q, kc, vc, pos + 1, Hq, Hkv, d, o);

        linear(c, L->wo, L->so, NULL, h, Hq * d, o, tmp);
        for (int64_t i = 0; i < h; ++i) x[i] += tmp[i];

        OR_PREFIX(rmsnorm)(x, L->mlp_norm, h, c->rms_eps, n);
        linear(c, L->wg, L->sg, NULL, F, h, n, ga);
        linear(c, L->wu, L->su, NULL, F, h, n, up);
        OR_PREFIX(silu_mul)(ga, up, F, u);
        linear(c, L->wd, L->sd, NULL, h, F, u, tmp);
        for (int64_t i = 0; i < h; ++i) x[i] += tmp[i];
    }

    if (hidden_out)
        for (int64_t i = 0; i < h; ++i) hidden_out[i] = (float)x[i];

    OR_PREFIX(rmsnorm)(x, W->final_norm, h, c->rms_eps, n);
    if (W->lm_scale)
        OR_PREFIX(gemv_int8)((const int8_t *)W->lm_head, W->lm_scale, V, h, n, tmp, NULL);
    else
        OR_PREFIX(gemv_bf16)((const uint16_t *)W->lm_head, V, h, n, tmp, NULL);
    for (int64_t i = 0; i < V; ++i) logits[i] = (float)tmp[i];

    free(x); free(n); free(q); free(k); free(v); free(o);
    free(ga); free(up); free(u); free(tmp);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Prompt prefill: the step above applied to n tokens at positions      */
/* pos0 .. pos0 + n - 1, with each linear layer evaluated for all rows  */
/* at once.  Every output element is the same sum as in the GEMV (k     */
/* ascending, the same dequantized weight, the same rounding), so the   */
/* result equals n calls of the step bit for bit; only the loops are    */
/* interchanged so that each weight row is unpacked once per block of   */
/* rows instead of once per token.                                      */
/* ------------------------------------------------------------------ */

/* W[n][k] for one output row n, as the GEMVs form it. */
static void dequant_row(const or_config *c, const void *w, const void *s, int64_t n, int64_t K, real_t *out) {
    if (c->weight_format == 1) {
        const uint32_t *words = (const uint32_t *)w;
        const uint16_t *scales = (const uint16_t *)s;
        for (int64_t k = 0; k < K; ++k)
            out[k] = (real_t)int4_code(words, K, n, k) * (real_t)bf16_to_float(scales[n * (K / 128) + k / 128]);
    } else {
        const int8_t *codes = (const int8_t *)w;
        for (int64_t k = 0; k < K; ++k) out[k] = (real_t)codes[n * K + k] * (real_t)((const float *)s)[n];
    }
}

/* Y[m][n] = sum_k W[n][k] X[m][k] (+ b[n]) for the M rows of X [M][K]. */
static void linear_rows(const or_config *c, const void *w, const void *s, const void *b, int64_t N,
                        int64_t K, const real_t *X, int64_t M, real_t *Y) {
    enum { NB = 16 };  /* output rows per block */
    real_t *XT = malloc(sizeof(real_t) * (size_t)(K * M));   /* X transposed: [K][M] */
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) XT[k * M + m] = X[m * K + k];
#pragma omp parallel
    {
        real_t *wb = malloc(sizeof(real_t) * (size_t)(NB * K));
        real_t *acc = malloc(sizeof(real_t) * (size_t)(NB * M));
#pragma omp for schedule(dynamic, 1)
        for (int64_t n0 = 0; n0 < N; n0 += NB) {
            const int64_t nb = N - n0 < NB ? N - n0 : NB;
            for (int64_t j = 0; j < nb; ++j) dequant_row(c, w, s, n0 + j, K, wb + j * K);
            for (int64_t i = 0; i < nb * M; ++i) acc[i] = 0;
            for (int64_t k = 0; k < K; ++k) {
                const real_t *xk = XT + k * M;
                for (int64_t j = 0; j < nb; ++j) {
                    const real_t wk = wb[j * K + k];
                    real_t *a = acc + j * M;
                    for (int64_t m = 0; m < M; ++m) a[m] += wk * xk[m];
                }
            }
            for (int64_t j = 0; j < nb; ++j)
                for (int64_t m = 0; m < M; ++m) {
                    real_t v = acc[j * M + m];
                    if (b) v += (real_t)bf16_to_float(((const uint16_t *)b)[n0 + j]);
                    Y[m * N + n0 + j] = v;
                }
        }
        free(wb);
        free(acc);
    }
    free(XT);
}

/*
 * Prefill: consume tokens[0..n-1] at positions pos0.., append their K/V, and
 * write the logits of the last token (the distribution of the first generated
 * token).  Returns 0, or -1 on bad arguments.
 */
int OR_PREFIX(prefill)(const or_config *c, const or_weights *W, uint16_t *k_cache, uint16_t *v_cache,
                       int64_t t_max, const int32_t *tokens, int64_t n_tok, int64_t pos0, float *logits) {
    const int64_t h = c->hidden, Hq = c->n_q_heads, Hkv = c->n_kv_heads, d = c->head_dim;
    const int64_t F = c->mlp, V = c->vocab, M = n_tok;
    if (M < 1 || pos0 < 0 || pos0 + M > t_max || Hq % Hkv != 0 || Hq * d != h) return -1;
    for (int64_t m = 0; m < M; ++m)
        if (tokens[m] < 0 || tokens[m] >= V) return -1;

    real_t *x = calloc((size_t)(M * h), sizeof(real_t));
    real_t *nrm = calloc((size_t)(M * h), sizeof(real_t));
    real_t *q = calloc((size_t)(M * Hq * d), sizeof(real_t));
    real_t *k = calloc((size_t)(M * Hkv * d), sizeof(real_t));
    real_t *v = calloc((size_t)(M * Hkv * d), sizeof(real_t));
    real_t *o = calloc((size_t)(M * h), sizeof(real_t));
    real_t *t = calloc((size_t)(M * h), sizeof(real_t));
    real_t *ga = calloc((size_t)(M * F), sizeof(real_t));
    real_t *up = calloc((size_t)(M * F), sizeof(real_t));
    real_t *u = calloc((size_t)(M * F), sizeof(real_t));
    real_t *tmp = calloc((size_t)(V > d ? V : d), sizeof(real_t));

    for (int64_t m = 0; m < M; ++m)
        for (int64_t i = 0; i < h; ++i) x[m * h + i] = (real_t)bf16_to_float(W->embed[(int64_t)tokens[m] * h + i]);

    for (int64_t l = 0; l < c->n_layers; ++l) {
        const or_layer *L = &W->layers[l];
        uint16_t *kc = k_cache + l * t_max * Hkv * d;
        uint16_t *vc = v_cache + l * t_max * Hkv * d;

        for (int64_t m = 0; m < M; ++m) OR_PREFIX(rmsnorm)(x + m * h, L->attn_norm, h, c->rms_eps, nrm + m * h);
        linear_rows(c, L->wq, L->sq, c->qkv_bias ? L->bq : NULL, Hq * d, h, nrm, M, q);
        linear_rows(c, L->wk, L->sk, c->qkv_bias ? L->bk : NULL, Hkv * d, h, nrm, M, k);
        linear_rows(c, L->wv, L->sv, c->qkv_bias ? L->bv : NULL, Hkv * d, h, nrm, M, v);
        for (int64_t m = 0; m < M; ++m) {
            real_t *qm = q + m * Hq * d, *km = k + m * Hkv * d, *vm = v + m * Hkv * d;
            const int64_t pos = pos0 + m;
            if (c->qk_norm) {
                for (int64_t hh = 0; hh < Hq; ++hh) {
                    OR_PREFIX(rmsnorm)(qm + hh * d, L->q_norm, d, c->rms_eps, tmp);
                    memcpy(qm + hh * d, tmp, sizeof(real_t) * (size_t)d);
                }
                for (int64_t hh = 0; hh < Hkv; ++hh) {
                    OR_PREFIX(rmsnorm)(km + hh * d, L->k_norm, d, c->rms_eps, tmp);
                    memcpy(km + hh * d, tmp, sizeof(real_t) * (size_t)d);
                }
            }
            OR_PREFIX(rope)(qm, Hq, d, pos, (double)c->rope_base);
            OR_PREFIX(rope)(km, Hkv, d, pos, (double)c->rope_base);
            for (int64_t i = 0; i < Hkv * d; ++i) {
                kc[pos * Hkv * d + i] = float_to_bf16((float)km[i]);
                vc[pos * Hkv * d + i] = float_to_bf16((float)vm[i]);
            }
        }
        /* row m attends to positions 0 .. pos0 + m (causal; its own K/V included) */
        for (int64_t m = 0; m < M; ++m)
            OR_PREFIX(attention)(q + m * Hq * d, kc, vc, pos0 + m + 1, Hq, Hkv, d, o + m * h);

        linear_rows(c, L->wo, L->so, NULL, h, Hq * d, o, M, t);
        for (int64_t i = 0; i < M * h; ++i) x[i] += t[i];

        for (int64_t m = 0; m < M; ++m) OR_PREFIX(rmsnorm)(x + m * h, L->mlp_norm, h, c->rms_eps, nrm + m * h);
        linear_rows(c, L->wg, L->sg, NULL, F, h, nrm, M, ga);
        linear_rows(c, L->wu, L->su, NULL, F, h, nrm, M, up);
        OR_PREFIX(silu_mul)(ga, up, M * F, u);
        linear_rows(c, L->wd, L->sd, NULL, h, F, u, M, t);
        for (int64_t i = 0; i < M * h; ++i) x[i] += t[i];
    }

    /* the last row only: its logits are the first generated token's */
    OR_PREFIX(rmsnorm)(x + (M - 1) * h, W->final_norm, h, c->rms_eps, nrm);
    if (W->lm_scale)
        OR_PREFIX(gemv_int8)((const int8_t *)W->lm_head, W->lm_scale, V, h, nrm, tmp, NULL);
    else
        OR_PREFIX(gemv_bf16)((const uint16_t *)W->lm_head, V, h, nrm, tmp, NULL);
    for (int64_t i = 0; i < V; ++i) logits[i] = (float)tmp[i];

    free(x); free(nrm); free(q); free(k); free(v); free(o); free(t);
    free(ga); free(up); free(u); free(tmp);
    return 0;
}
