/*
 * fg_oracle.c -- plain, slow, obviously-correct CPU oracle for the 4-bit
 * group-quantised, block-scheduled OPT decoder hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math (-fopenmp optional).  The
 * contraction switch matters: every float operation below is a separately
 * rounded IEEE binary32 operation unless fmaf() is written out.  OpenMP (when
 * present) only splits independent output rows or (sequence, head) pairs over
 * threads; no reduction is ever split, so results do not depend on the thread
 * count.
 *
 * Sources (web pages on FlexGen's 4-bit group-wise compression):
 *  - "FlexGen 完全拆解" (pinghaoyang.com.cn), section "权重压缩与 KV Cache 压缩":
 *    group-wise asymmetric min/max quantisation q = round((x-min)/(max-min)
 *    *(2^b-1)), dequantisation x^ = min + q/(2^b-1)*(max-min), b = 4, g = 64,
 *    tensors are dequantised to FP16 before use.
 *  - same page, section "从 Transformer 推理的数据流重新定义卸载": prefill
 *    K = XW_K, V = XW_V, Q = XW_Q; decode appends the new K/V row and attends
 *    one query position over all s+t cached rows.
 *  - bjbfmj.com/news/40234, section 6.3: two 4-bit codes packed per uint8 plus
 *    a per-group scale tensor.
 * The fixed arithmetic of the quantiser (fp32 min/max, scale=(M-m)/15 by IEEE
 * division, code=clamp(rint((x-m)/scale),0,15), all codes 0 when scale==0,
 * fp32 min and scale stored) is the reading this project adopts where the
 * pages leave the precision open; see the readings list in the design notes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_GROUP 64

/* ------------------------------------------------------------------------ */
/* IEEE binary16 <-> binary32, written from the format definition            */
/* (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits).             */
/* ------------------------------------------------------------------------ */

float or_h2f(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);              /* zero / subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);  /* (1 + f/1024) * 2^(e-15)    */
    return (float)(sign ? -v : v);              /* exact: fits in binary32      */
}

/* Round-to-nearest-even conversion of a binary32 value to binary16. */
uint16_t or_f2h(float x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs((double)x);
    if (isnan(x))
        return 0x7E00;
    if (a >= 65520.0)                            /* halfway to 2^16 rounds up to inf */
        return sign | 0x7C00;
    if (a < ldexp(1.0, -14)) {                   /* subnormal range: step 2^-24 */
        double q = nearbyint(a * ldexp(1.0, 24));   /* exact scaling, RNE */
        return sign | (uint16_t)q;               /* q == 1024 is the smallest normal */
    }
    int e2;
    frexp(a, &e2);                               /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;                              /* a in [2^E, 2^(E+1)) */
    double sig = nearbyint(ldexp(a, 10 - E));    /* in [1024, 2048], RNE */
    if (sig == 2048.0) {
        sig = 1024.0;
        E += 1;
    }
    if (E + 15 >= 31)
        return sign | 0x7C00;
    return sign | (uint16_t)(((E + 15) << 10) | ((int)sig - 1024));
}

void or_h2f_array(const uint16_t* h, float* f, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) f[i] = or_h2f(h[i]);
}

void or_f2h_array(const float* f, uint16_t* h, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) h[i] = or_f2h(f[i]);
}

int or_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void or_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* Group-wise 4-bit quantisation of one group of 64 values.                  */
/* Group = 64 consecutive elements along the contiguous (last) axis.          */
/* meta receives (min, scale); codes receives 32 bytes, element 2j in the     */
/* low nibble of byte j and element 2j+1 in the high nibble.                  */
/* ------------------------------------------------------------------------ */

/* a < b in the IEEE total order restricted to finite values: numeric order,
 * with -0 below +0 (so the sign of a zero minimum or maximum is defined by
 * the values, not by where they sit in the group). */
static int total_less(float a, float b)
{
    if (a < b) return 1;
    if (a > b) return 0;
    return signbit(a) && !signbit(b);
}

static void quantize_group(const uint16_t* x, uint8_t* codes, float* meta)
{
    float v[OR_GROUP];
    uint8_t q[OR_GROUP];
    for (int i = 0; i < OR_GROUP; ++i) v[i] = or_h2f(x[i]);

    float mn = v[0], mx = v[0];
    for (int i = 1; i < OR_GROUP; ++i) {
        if (total_less(v[i], mn)) mn = v[i];
        if (total_less(mx, v[i])) mx = v[i];
    }
    float range = mx - mn;          /* fp32 subtract */
    float scale = range / 15.0f;    /* fp32 IEEE divide, 15 = 2^4 - 1 levels */

    for (int i = 0; i < OR_GROUP; ++i) {
        if (scale == 0.0f) {
            q[i] = 0;
        } else {
            float t = (v[i] - mn) / scale;   /* fp32 subtract, fp32 divide */
            float r = rintf(t);              /* round half to even */
            if (r < 0.0f) r = 0.0f;
            if (r > 15.0f) r = 15.0f;
            q[i] = (uint8_t)r;
        }
    }
    for (int j = 0; j < OR_GROUP / 2; ++j)
        codes[j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
    meta[0] = mn;
    meta[1] = scale;
}

/* x: [rows][cols] fp16, cols % 64 == 0.
 * codes: [rows][cols/2] bytes; meta: [rows][cols/64][2] fp32. */
void or_quantize_g4(const uint16_t* x, int64_t rows, int64_t cols,
                    uint8_t* codes, float* meta)
{
    int64_t ng = cols / OR_GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t g = 0; g < ng; ++g)
            quantize_group(x + r * cols + g * OR_GROUP,
                           codes + r * (cols / 2) + g * (OR_GROUP / 2),
                           meta + (r * ng + g) * 2);
}

/* Dequantised value of code q in a group with (min, scale): the single-rounding
 * fused multiply-add q*scale + min in fp32, then rounded to fp16 (tensors are
 * dequantised to FP16 before use). */
static uint16_t dequant_one(int q, float mn, float scale)
{
    return or_f2h(fmaf((float)q, scale, mn));
}

void or_dequant_g4(const uint8_t* codes, const float* meta, int64_t rows,
                   int64_t cols, uint16_t* out)
{
    int64_t ng = cols / OR_GROUP;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            uint8_t byte = codes[r * (cols / 2) + c / 2];
            int q = (c & 1) ? (byte >> 4) : (byte & 0xF);
            const float* m = meta + (r * ng + c / OR_GROUP) * 2;
            out[r * cols + c] = dequant_one(q, m[0], m[1]);
        }
}

/* ------------------------------------------------------------------------ */
/* Linear layer: Y[m][n] = fp16( act(sum_k X[m][k]*W[n][k] + bias[n])        */
/*                               + residual[m][n] )                           */
/* X fp16 [M][K], W fp16 [N][K] (torch Linear layout), fp32 accumulation in   */
/* ascending k; order: +bias, then ReLU (act==1), then +residual, one final  */
/* rounding to fp16.  bias / residual may be NULL.                           */
/* ------------------------------------------------------------------------ */

void or_linear_f16(const uint16_t* X, int64_t M, int64_t K, const uint16_t* W,
                   int64_t N, const uint16_t* bias, const uint16_t* residual,
                   int act, uint16_t* Y)
{
    float* wf = (float*)malloc(sizeof(float) * (size_t)(N * K));
    or_h2f_array(W, wf, N * K);
#pragma omp parallel
    {
        float* xf = (float*)malloc(sizeof(float) * (size_t)K);
#pragma omp for schedule(static)
        for (int64_t m = 0; m < M; ++m) {
            or_h2f_array(X + m * K, xf, K);
            for (int64_t n = 0; n < N; ++n) {
                const float* w = wf + n * K;
                float acc = 0.0f;
                for (int64_t k = 0; k < K; ++k) acc += xf[k] * w[k];
                if (bias) acc += or_h2f(bias[n]);
                if (act == 1 && acc < 0.0f) acc = 0.0f;
                if (residual) acc += or_h2f(residual[m * N + n]);
                Y[m * N + n] = or_f2h(acc);
            }
        }
        free(xf);
    }
    free(wf);
}

/* Same contraction with an fp32 result and no epilogue (LM head logits). */
void or_linear_f16_f32out(const uint16_t* X, int64_t M, int64_t K,
                          const uint16_t* W, int64_t N, float* Y)
{
    float* wf = (float*)malloc(sizeof(float) * (size_t)(N * K));
    or_h2f_array(W, wf, N * K);
#pragma omp parallel
    {
        float* xf = (float*)malloc(sizeof(float) * (size_t)K);
#pragma omp for schedule(static)
        for (int64_t m = 0; m < M; ++m) {
            or_h2f_array(X + m * K, xf, K);
            for (int64_t n = 0; n < N; ++n) {
                const float* w = wf + n * K;
                float acc = 0.0f;
                for (int64_t k = 0; k < K; ++k) acc += xf[k] * w[k];
                Y[m * N + n] = acc;
            }
        }
        free(xf);
    }
    free(wf);
}

/* Linear layer whose weight is stored 4-bit: dequantise to fp16, then the
 * plain linear above. */
void or_linear_g4(const uint16_t* X, int64_t M, int64_t K, const uint8_t* codes,
                  const float* meta, int64_t N, const uint16_t* bias,
                  const uint16_t* residual, int act, uint16_t* Y)
{
    uint16_t* w = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(N * K));
    or_dequant_g4(codes, meta, N, K, w);
    or_linear_f16(X, M, K, w, N, bias, residual, act, Y);
    free(w);
}

/* ------------------------------------------------------------------------ */
/* LayerNorm over the last axis: mean and biased variance in fp32 (ascending */
/* sums), y = (x - mean) / sqrt(var + eps) * gamma + beta, rounded to fp16.  */
/* ------------------------------------------------------------------------ */

void or_layernorm(const uint16_t* x, int64_t rows, int64_t cols,
                  const uint16_t* gamma, const uint16_t* beta, float eps,
                  uint16_t* y)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * cols;
        float sum = 0.0f;
        for (int64_t c = 0; c < cols; ++c) sum += or_h2f(xr[c]);
        float mean = sum / (float)cols;
        float sq = 0.0f;
        for (int64_t c = 0; c < cols; ++c) {
            float dv = or_h2f(xr[c]) - mean;
            sq += dv * dv;
        }
        float var = sq / (float)cols;
        float denom = sqrtf(var + eps);
        for (int64_t c = 0; c < cols; ++c) {
            float v = (or_h2f(xr[c]) - mean) / denom;
            v = v * or_h2f(gamma[c]) + or_h2f(beta[c]);
            y[r * cols + c] = or_f2h(v);
        }
    }
}

/* Token embedding plus learned position embedding:
 * y[t] = fp16(E_tok[ids[t]] + E_pos[pos[t]]), one fp32 add per element. */
void or_embed(const int32_t* ids, const int32_t* pos, int64_t ntok,
              const uint16_t* e_tok, const uint16_t* e_pos, int64_t h1,
              uint16_t* y)
{
    for (int64_t t = 0; t < ntok; ++t)
        for (int64_t c = 0; c < h1; ++c)
            y[t * h1 + c] = or_f2h(or_h2f(e_tok[(int64_t)ids[t] * h1 + c]) +
                                   or_h2f(e_pos[(int64_t)pos[t] * h1 + c]));
}

/* ------------------------------------------------------------------------ */
/* 4-bit KV cache.  Per layer, K and V each hold                              */
/*   codes [B][H][cap][d/2] bytes and meta [B][H][cap][d/64][2] fp32,         */
/* one cache row per (sequence, head, position), grouped in 64s along the    */
/* head dimension.                                                            */
/* ------------------------------------------------------------------------ */

typedef struct {
    uint8_t* k_codes;
    uint8_t* v_codes;
    float* k_meta;
    float* v_meta;
    int32_t B, H, d, cap;
} or_kv4;

static int64_t kv_row(const or_kv4* c, int64_t b, int64_t h, int64_t t)
{
    return (b * c->H + h) * c->cap + t;
}

/* Quantise the K and V parts of one token's QKV row into cache slot t of
 * sequence b, for every head.  qkv_row: [3*h1] fp16 = q | k | v. */
static void store_kv_row(or_kv4* c, const uint16_t* qkv_row, int64_t b, int64_t t)
{
    int64_t d = c->d, h1 = (int64_t)c->H * d, ng = d / OR_GROUP;
    for (int64_t h = 0; h < c->H; ++h) {
        int64_t row = kv_row(c, b, h, t);
        for (int64_t g = 0; g < ng; ++g) {
            quantize_group(qkv_row + h1 + h * d + g * OR_GROUP,
                           c->k_codes + row * (d / 2) + g * (OR_GROUP / 2),
                           c->k_meta + (row * ng + g) * 2);
            quantize_group(qkv_row + 2 * h1 + h * d + g * OR_GROUP,
                           c->v_codes + row * (d / 2) + g * (OR_GROUP / 2),
                           c->v_meta + (row * ng + g) * 2);
        }
    }
}

/* Dequantise cache row (b,h,t) of K or V into d fp32 values (each first
 * rounded to fp16, as every dequantised tensor is). */
static void load_cache_row(const or_kv4* c, int is_v, int64_t b, int64_t h,
                           int64_t t, float* out)
{
    int64_t d = c->d, ng = d / OR_GROUP;
    int64_t row = kv_row(c, b, h, t);
    const uint8_t* codes = (is_v ? c->v_codes : c->k_codes) + row * (d / 2);
    const float* meta = (is_v ? c->v_meta : c->k_meta) + row * ng * 2;
    for (int64_t i = 0; i < d; ++i) {
        int q = (i & 1) ? (codes[i / 2] >> 4) : (codes[i / 2] & 0xF);
        const float* m = meta + (i / OR_GROUP) * 2;
        out[i] = or_h2f(dequant_one(q, m[0], m[1]));
    }
}

/* Prefill K/V store: token t of sequence b is row (b*s + t) of qkv
 * ([B*s][3*h1] fp16); it goes to cache slot t. */
void or_kv_store_prefill(const uint16_t* qkv, int32_t B, int32_t s,
                         uint8_t* k_codes, uint8_t* v_codes, float* k_meta,
                         float* v_meta, int32_t H, int32_t d, int32_t cap)
{
    or_kv4 c = {k_codes, v_codes, k_meta, v_meta, B, H, d, cap};
    int64_t ld = 3 * (int64_t)H * d;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < B; ++b)
        for (int64_t t = 0; t < s; ++t)
            store_kv_row(&c, qkv + (b * s + t) * ld, b, t);
}

/* Softmax-weighted sum over n rows with scores sc[0..n): two passes in fp32
 * (max, then sum of exp(score - max)), out[i] = (sum_j p_j v_j[i]) / sum_j p_j.
 * vrows: n x d fp32 values.  The result is rounded to fp16. */
static void softmax_weighted(const float* sc, const float* vrows, int64_t n,
                             int64_t d, float* p, uint16_t* out)
{
    float mx = sc[0];
    for (int64_t j = 1; j < n; ++j)
        if (sc[j] > mx) mx = sc[j];
    float l = 0.0f;
    for (int64_t j = 0; j < n; ++j) {
        p[j] = expf(sc[j] - mx);
        l += p[j];
    }
    for (int64_t i = 0; i < d; ++i) {
        float acc = 0.0f;
        for (int64_t j = 0; j < n; ++j) acc += p[j] * vrows[j * d + i];
        out[i] = or_f2h(acc / l);
    }
}

/* Causal prefill attention over fp16 Q/K/V taken straight from the QKV
 * projection (not yet stored, so not quantised).
 * qkv: [B*s][3*h1]; out: [B*s][h1]; score = (q . k) * (1/sqrt(d)).
 * pad: NULL, or [B] left-padding counts: sequence b's prompt fills slots
 * pad[b]..s-1, a query at slot i >= pad[b] attends keys pad[b]..i, and a
 * query in a padding slot outputs zeros. */
void or_prefill_attn(const uint16_t* qkv, int32_t B, int32_t s, int32_t H,
                     int32_t d, const int32_t* pad, uint16_t* out)
{
    int64_t h1 = (int64_t)H * d, ld = 3 * h1;
    float scale = 1.0f / sqrtf((float)d);
#pragma omp parallel
    {
        float* q = (float*)malloc(sizeof(float) * (size_t)d);
        float* kr = (float*)malloc(sizeof(float) * (size_t)d);
        float* sc = (float*)malloc(sizeof(float) * (size_t)s);
        float* p = (float*)malloc(sizeof(float) * (size_t)s);
        float* vr = (float*)malloc(sizeof(float) * (size_t)s * (size_t)d);
#pragma omp for collapse(2) schedule(static)
        for (int64_t b = 0; b < B; ++b)
            for (int64_t h = 0; h < H; ++h)
                for (int64_t i = 0; i < s; ++i) {
                    const int64_t p0 = pad ? pad[b] : 0;
                    uint16_t* o = out + (b * s + i) * h1 + h * d;
                    if (i < p0) {   /* padding slot */
                        for (int64_t c = 0; c < d; ++c) o[c] = 0;
                        continue;
                    }
                    or_h2f_array(qkv + (b * s + i) * ld + h * d, q, d);
                    for (int64_t j = p0; j <= i; ++j) {
                        or_h2f_array(qkv + (b * s + j) * ld + h1 + h * d, kr, d);
                        float dot = 0.0f;
                        for (int64_t c = 0; c < d; ++c) dot += q[c] * kr[c];
                        sc[j - p0] = dot * scale;
                        or_h2f_array(qkv + (b * s + j) * ld + 2 * h1 + h * d,
                                     vr + (j - p0) * d, d);
                    }
                    softmax_weighted(sc, vr, i + 1 - p0, d, p, o);
                }
        free(q);
        free(kr);
        free(sc);
        free(p);
        free(vr);
    }
}

/* Decode attention over the 4-bit cache.  qkv: [B][qkv_ld] fp16 rows, one
 * new token per sequence.  If do_append, the new k and v are first quantised
 * into slot pos; then the query attends over slots pad[b]..pos (pad NULL:
 * 0..pos), every row (the new one included) read through dequantisation.
 * out: [B][h1] fp16. */
void or_decode_attn_g4(const uint16_t* qkv, int64_t qkv_ld, uint8_t* k_codes,
                       uint8_t* v_codes, float* k_meta, float* v_meta,
                       int32_t B, int32_t H, int32_t d, int32_t cap,
                       int32_t pos, int32_t do_append, const int32_t* pad,
                       uint16_t* out)
{
    or_kv4 c = {k_codes, v_codes, k_meta, v_meta, B, H, d, cap};
    int64_t h1 = (int64_t)H * d, L = (int64_t)pos + 1;
    float scale = 1.0f / sqrtf((float)d);
    if (do_append)
        for (int64_t b = 0; b < B; ++b)
            store_kv_row(&c, qkv + b * qkv_ld, b, pos);
#pragma omp parallel
    {
        float* q = (float*)malloc(sizeof(float) * (size_t)d);
        float* kr = (float*)malloc(sizeof(float) * (size_t)d);
        float* sc = (float*)malloc(sizeof(float) * (size_t)L);
        float* p = (float*)malloc(sizeof(float) * (size_t)L);
        float* vr = (float*)malloc(sizeof(float) * (size_t)L * (size_t)d);
#pragma omp for collapse(2) schedule(static)
        for (int64_t b = 0; b < B; ++b)
            for (int64_t h = 0; h < H; ++h) {
                const int64_t p0 = pad ? pad[b] : 0;
                or_h2f_array(qkv + b * qkv_ld + h * d, q, d);
                for (int64_t j = p0; j < L; ++j) {
                    load_cache_row(&c, 0, b, h, j, kr);
                    float dot = 0.0f;
                    for (int64_t i = 0; i < d; ++i) dot += q[i] * kr[i];
                    sc[j - p0] = dot * scale;
                    load_cache_row(&c, 1, b, h, j, vr + (j - p0) * d);
                }
                softmax_weighted(sc, vr, L - p0, d, p, out + b * h1 + h * d);
            }
        free(q);
        free(kr);
        free(sc);
        free(p);
        free(vr);
    }
}

/* Uncompressed (fp16) KV cache: k, v [B][H][cap][d] fp16, the rows stored as
 * the QKV projection produced them.  This is the setting the pages compare
 * the 4-bit cache against ("FlexGen 完全拆解", results for input length 512:
 * FlexGen with and without 4-bit compression). */

/* Prefill store into the fp16 cache: token t of sequence b (row b*s + t of
 * qkv, [B*s][3*h1]) goes to slot t. */
void or_kv_store_prefill_f16(const uint16_t* qkv, int32_t B, int32_t s, uint16_t* k,
                             uint16_t* v, int32_t H, int32_t d, int32_t cap)
{
    int64_t h1 = (int64_t)H * d, ld = 3 * h1;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t t = 0; t < s; ++t)
            for (int64_t h = 0; h < H; ++h) {
                int64_t row = ((b * H + h) * cap + t) * d;
                memcpy(k + row, qkv + (b * s + t) * ld + h1 + h * d, sizeof(uint16_t) * (size_t)d);
                memcpy(v + row, qkv + (b * s + t) * ld + 2 * h1 + h * d, sizeof(uint16_t) * (size_t)d);
            }
}

/* Decode attention over the fp16 cache: optionally store the new k, v rows
 * (qkv row b) into slot pos, then for each (b, h) attend slots pad[b]..pos:
 * the same fp32 arithmetic as or_decode_attn_g4 with the cached rows read
 * as stored instead of dequantised. */
void or_decode_attn_f16(const uint16_t* qkv, int64_t qkv_ld, uint16_t* k, uint16_t* v,
                        int32_t B, int32_t H, int32_t d, int32_t cap, int32_t pos,
                        int32_t do_append, const int32_t* pad, uint16_t* out)
{
    int64_t h1 = (int64_t)H * d, L = (int64_t)pos + 1;
    float scale = 1.0f / sqrtf((float)d);
    if (do_append)
        for (int64_t b = 0; b < B; ++b)
            for (int64_t h = 0; h < H; ++h) {
                int64_t row = ((b * H + h) * cap + pos) * d;
                memcpy(k + row, qkv + b * qkv_ld + h1 + h * d, sizeof(uint16_t) * (size_t)d);
                memcpy(v + row, qkv + b * qkv_ld + 2 * h1 + h * d, sizeof(uint16_t) * (size_t)d);
            }
#pragma omp parallel
    {
        float* q = (float*)malloc(sizeof(float) * (size_t)d);
        float* kr = (float*)malloc(sizeof(float) * (size_t)d);
        float* sc = (float*)malloc(sizeof(float) * (size_t)L);
        float* p = (float*)malloc(sizeof(float) * (size_t)L);
        float* vr = (float*)malloc(sizeof(float) * (size_t)L * (size_t)d);
#pragma omp for collapse(2) schedule(static)
        for (int64_t b = 0; b < B; ++b)
            for (int64_t h = 0; h < H; ++h) {
                const int64_t p0 = pad ? pad[b] : 0;
                const int64_t base = (b * H + h) * cap;
                or_h2f_array(qkv + b * qkv_ld + h * d, q, d);
                for (int64_t j = p0; j < L; ++j) {
                    or_h2f_array(k + (base + j) * d, kr, d);
                    float dot = 0.0f;
                    for (int64_t i = 0; i < d; ++i) dot += q[i] * kr[i];
                    sc[j - p0] = dot * scale;
                    or_h2f_array(v + (base + j) * d, vr + (j - p0) * d, d);
                }
                softmax_weighted(sc, vr, L - p0, d, p, out + b * h1 + h * d);
            }
        free(q);
        free(kr);
        free(sc);
        free(p);
        free(vr);
    }
}

/* Number of rows kept by top-K sparse attention over n attended rows: the
 * keep_pct percent with the highest scores, rounded up (at least one row). */
int32_t or_topk_count(int64_t n, int32_t keep_pct)
{
    return (int32_t)((n * keep_pct + 99) / 100);
}

/* Order for the top-K choice: higher score first; equal scores (+0 and -0
 * compare equal) by ascending slot. */
static const float* g_rank_sc;
static int rank_cmp(const void* a, const void* b)
{
    int64_t i = *(const int64_t*)a, j = *(const int64_t*)b;
    float si = g_rank_sc[i], sj = g_rank_sc[j];
    if (si > sj) return -1;
    if (si < sj) return 1;
    return i < j ? -1 : (i > j ? 1 : 0);
}
static int slot_cmp(const void* a, const void* b)
{
    int64_t i = *(const int64_t*)a, j = *(const int64_t*)b;
    return i < j ? -1 : (i > j ? 1 : 0);
}

/* Top-K sparse decode attention over the 4-bit cache ("FlexGen 完全拆解",
 * section on the paper's further approximations: the attention scores are
 * computed from every cached key, and only the V rows of the highest-scoring
 * keep_pct percent are loaded).  Readings: the softmax is the full one over
 * all n attended rows (maximum and normaliser over every score); the rows not
 * kept contribute nothing to the weighted sum (no renormalisation); the count
 * kept is or_topk_count(n, keep_pct); equal scores are kept lowest slot
 * first; the new token's row is a candidate like any other.  Scores are
 * computed exactly as or_decode_attn_g4 computes them.
 * sel_in: NULL, or the kept slots to use instead of the oracle's own choice,
 * [B][H][kmax] (kmax = or_topk_count(pos+1, keep_pct)), each (b,h) list
 * ascending and -1 after its own count -- so the weighted sum can be checked
 * on another implementation's choice.  sel_out: NULL or [B][H][kmax], the
 * kept slots in that layout.  keep_pct in 1..100; 100 keeps every row and
 * equals or_decode_attn_g4. */
void or_decode_attn_topk_g4(const uint16_t* qkv, int64_t qkv_ld, uint8_t* k_codes,
                            uint8_t* v_codes, float* k_meta, float* v_meta,
                            int32_t B, int32_t H, int32_t d, int32_t cap,
                            int32_t pos, int32_t do_append, const int32_t* pad,
                            int32_t keep_pct, const int32_t* sel_in,
                            int32_t* sel_out, uint16_t* out)
{
    or_kv4 c = {k_codes, v_codes, k_meta, v_meta, B, H, d, cap};
    int64_t h1 = (int64_t)H * d, L = (int64_t)pos + 1;
    int64_t kmax = or_topk_count(L, keep_pct);
    float scale = 1.0f / sqrtf((float)d);
    if (do_append)
        for (int64_t b = 0; b < B; ++b)
            store_kv_row(&c, qkv + b * qkv_ld, b, pos);
    float* q = (float*)malloc(sizeof(float) * (size_t)d);
    float* kr = (float*)malloc(sizeof(float) * (size_t)d);
    float* vr = (float*)malloc(sizeof(float) * (size_t)d);
    float* sc = (float*)malloc(sizeof(float) * (size_t)L);
    float* p = (float*)malloc(sizeof(float) * (size_t)L);
    float* acc = (float*)malloc(sizeof(float) * (size_t)d);
    int64_t* idx = (int64_t*)malloc(sizeof(int64_t) * (size_t)L);
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h) {
            const int64_t p0 = pad ? pad[b] : 0, n = L - p0;
            const int64_t ksel = or_topk_count(n, keep_pct);
            or_h2f_array(qkv + b * qkv_ld + h * d, q, d);
            for (int64_t j = 0; j < n; ++j) {
                load_cache_row(&c, 0, b, h, p0 + j, kr);
                float dot = 0.0f;
                for (int64_t i = 0; i < d; ++i) dot += q[i] * kr[i];
                sc[j] = dot * scale;
            }
            /* the full softmax over all n rows */
            float mx = sc[0];
            for (int64_t j = 1; j < n; ++j)
                if (sc[j] > mx) mx = sc[j];
            float l = 0.0f;
            for (int64_t j = 0; j < n; ++j) {
                p[j] = expf(sc[j] - mx);
                l += p[j];
            }
            /* the kept rows, as offsets from slot p0, ascending */
            const int32_t* given = sel_in ? sel_in + (b * H + h) * kmax : NULL;
            if (given) {
                for (int64_t r = 0; r < ksel; ++r) idx[r] = given[r] - p0;
            } else {
                for (int64_t j = 0; j < n; ++j) idx[j] = j;
                g_rank_sc = sc;
                qsort(idx, (size_t)n, sizeof(int64_t), rank_cmp);
                qsort(idx, (size_t)ksel, sizeof(int64_t), slot_cmp);
            }
            for (int64_t i = 0; i < d; ++i) acc[i] = 0.0f;
            for (int64_t r = 0; r < ksel; ++r) {
                load_cache_row(&c, 1, b, h, p0 + idx[r], vr);
                for (int64_t i = 0; i < d; ++i) acc[i] += p[idx[r]] * vr[i];
            }
            for (int64_t i = 0; i < d; ++i) out[b * h1 + h * d + i] = or_f2h(acc[i] / l);
            if (sel_out) {
                int32_t* so = sel_out + (b * H + h) * kmax;
                for (int64_t r = 0; r < kmax; ++r) so[r] = r < ksel ? (int32_t)(p0 + idx[r]) : -1;
            }
        }
    free(q);
    free(kr);
    free(vr);
    free(sc);
    free(p);
    free(acc);
    free(idx);
}

/* Greedy choice: for each of B rows of V fp32 logits, the index of the
 * largest value (the lowest such index when several are equal). */
void or_argmax(const float* logits, int64_t B, int64_t V, int32_t* out)
{
    for (int64_t b = 0; b < B; ++b) {
        const float* r = logits + b * V;
        int64_t best = 0;
        for (int64_t v = 1; v < V; ++v)
            if (r[v] > r[best]) best = v;
        out[b] = (int32_t)best;
    }
}
