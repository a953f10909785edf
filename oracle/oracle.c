/*
 * oracle.c - plain, slow CPU reference for one batch-size-1 decode step of a
 * Llama-style decoder.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark may load this code.  It shares nothing with
 * the CUDA path: no headers, helpers, tables or kernels.
 *
 * What it computes is the unfused, sequential definition of the step: the
 * "simple, synchronous, unfused reference" that the fused path is compared
 * against layer by layer and token by token (stapisi.com/news/3904786,
 * section 6.3 "software engineering practice").  Fusion and in-kernel
 * pipelining change only the schedule of this computation, not its result
 * (cloud.baidu.com/article/9434380, section 4.2).
 *
 * Precision: weights and the K/V cache are bf16 (widened exactly); every
 * activation and every accumulation is double.  The only rounding steps are
 * the ones the method itself has: K and V are stored to the cache as bf16,
 * and the greedy argmax is taken over logits rounded to float, the precision
 * the GPU path decides it in.
 *
 * Operator list of one layer (cloud.baidu.com/article/9434380, section 5,
 * step 2, segments A/B/C): normalisation + Q/K/V projection + rotary position
 * encoding; attention scores + causal mask + softmax + output projection;
 * normalisation + FFN first layer + activation + FFN second layer + residual.
 * The normalisation is RMSNorm (developer.baidu.com/article/detail.html?id=
 * 8006242, section 4.1.2) and the activation is SwiGLU (Llama).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Weight-only INT8 form of the model's matrices (stapisi.com/news/3904786,
 * section 6: quantization fused into the kernels), see oracle_quantize_q8.
 * Index 0..6 = wq, wk, wv, wo, w_gate, w_up, w_down; per layer an int8
 * matrix [out][in] and its scales: one per output row, except w_down, one per
 * input column. */
typedef struct {
    const int8_t* const* q[7];
    const float* const* s[7];
    const int8_t* lm_q;   /* [vocab][hidden] */
    const float* lm_s;    /* [vocab] */
} oracle_q8;

typedef struct {
    int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab, max_seq;
    double rms_eps, rope_theta;
    const uint16_t* embed;      /* [vocab][hidden] */
    const uint16_t* lm_head;    /* [vocab][hidden]; equal to embed when tied */
    const uint16_t* final_norm; /* [hidden] */
    const uint16_t* const* attn_norm; /* per layer [hidden] */
    const uint16_t* const* wq;        /* per layer [n_q_heads*head_dim][hidden] */
    const uint16_t* const* wk;        /* per layer [n_kv_heads*head_dim][hidden] */
    const uint16_t* const* wv;        /* per layer [n_kv_heads*head_dim][hidden] */
    const uint16_t* const* wo;        /* per layer [hidden][n_q_heads*head_dim] */
    const uint16_t* const* ffn_norm;  /* per layer [hidden] */
    const uint16_t* const* w_gate;    /* per layer [ffn][hidden] */
    const uint16_t* const* w_up;      /* per layer [ffn][hidden] */
    const uint16_t* const* w_down;    /* per layer [hidden][ffn] */
    const oracle_q8* q8;              /* NULL: the bf16 matrices above; else these int8 ones */
} oracle_model;

/* bf16 bit pattern -> double (exact). */
static inline double bf2d(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

double oracle_bf16_to_double(uint16_t b) { return bf2d(b); }

/* double -> bf16 bit pattern: first to float (the GPU path's activation
 * precision), then to bf16, both rounding to nearest even. */
uint16_t oracle_round_bf16(double v) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* RMSNorm (developer.baidu.com/article/detail.html?id=8006242, section 4.1.2
 * names RMSNorm; Llama form): y_i = x_i / sqrt(mean_j(x_j^2) + eps) * g_i.
 * No mean subtraction and no bias. */
void oracle_rmsnorm(const double* x, const uint16_t* g, int n, double eps, double* y) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; ++i) y[i] = x[i] * inv * bf2d(g[i]);
}

/* y = W x for a bf16 matrix W [rows][cols] (row-major, [out, in]). */
void oracle_gemv(const uint16_t* W, int64_t rows, int64_t cols, const double* x, double* y) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* w = W + r * cols;
        double acc = 0.0;
        for (int64_t c = 0; c < cols; ++c) acc += bf2d(w[c]) * x[c];
        y[r] = acc;
    }
}

/* Weight-only INT8 quantization (stapisi.com/news/3904786, section 6 names
 * quantization among the work fused into kernels; the page gives no scheme,
 * the one taken is symmetric absmax per channel): for each group g of
 * weights (a row, or for col_scaled a column) of a bf16 matrix [rows][cols],
 * the scale is s_g = max|w| / 127 and each code is q = round(w / s_g), ties to
 * even, so w ~ q * s_g with |w - q s_g| <= s_g / 2 and |q| <= 127.  Both the
 * scale and the quotient are float operations rounded to nearest (the
 * precision the codes are decided in); a group of zeros gets s = 0, q = 0. */
void oracle_quantize_q8(const uint16_t* W, int64_t rows, int64_t cols, int col_scaled, int8_t* q, float* scale) {
    const int64_t ng = col_scaled ? cols : rows, len = col_scaled ? rows : cols;
    for (int64_t gi = 0; gi < ng; ++gi) {
        float amax = 0.0f;
        for (int64_t k = 0; k < len; ++k) {
            const int64_t idx = col_scaled ? k * cols + gi : gi * cols + k;
            const float w = (float)bf2d(W[idx]);
            if (fabsf(w) > amax) amax = fabsf(w);
        }
        const float sg = amax / 127.0f;
        scale[gi] = sg;
        for (int64_t k = 0; k < len; ++k) {
            const int64_t idx = col_scaled ? k * cols + gi : gi * cols + k;
            float c = 0.0f;
            if (sg > 0.0f) c = rintf((float)bf2d(W[idx]) / sg);
            if (c > 127.0f) c = 127.0f;
            if (c < -127.0f) c = -127.0f;
            q[idx] = (int8_t)c;
        }
    }
}

/* Weight-only INT4 quantization (stapisi.com/news/3904786, section 6, as for
 * INT8 above; the page names no scheme): the same symmetric absmax per group,
 * with 7 levels a side instead of 127, s_g = max|w| / 7 and q = round(w / s_g),
 * ties to even, clamped to [-7, 7]; both float operations rounded to nearest,
 * a group of zeros gets s = 0, q = 0.  The codes are returned one per int8_t
 * (the packing into nibbles is the GPU stream's business, not the method's);
 * oracle_gemv_q8 and the decode step read them like INT8 codes. */
void oracle_quantize_q4(const uint16_t* W, int64_t rows, int64_t cols, int col_scaled, int8_t* q, float* scale) {
    const int64_t ng = col_scaled ? cols : rows, len = col_scaled ? rows : cols;
    for (int64_t gi = 0; gi < ng; ++gi) {
        float amax = 0.0f;
        for (int64_t k = 0; k < len; ++k) {
            const float w = (float)bf2d(W[col_scaled ? k * cols + gi : gi * cols + k]);
            amax = fabsf(w) > amax ? fabsf(w) : amax;
        }
        const float s4 = amax / 7.0f;
        scale[gi] = s4;
        for (int64_t k = 0; k < len; ++k) {
            const int64_t at = col_scaled ? k * cols + gi : gi * cols + k;
            float code = s4 > 0.0f ? rintf((float)bf2d(W[at]) / s4) : 0.0f;
            code = code > 7.0f ? 7.0f : (code < -7.0f ? -7.0f : code);
            q[at] = (int8_t)code;
        }
    }
}

/* y = W' x for the dequantized matrix W'[r][c] = q[r][c] * s (s = scale[r],
 * or scale[c] when col_scaled), in double. */
void oracle_gemv_q8(const int8_t* q, const float* scale, int col_scaled, int64_t rows, int64_t cols, const double* x,
                    double* y) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const int8_t* w = q + r * cols;
        double acc = 0.0;
        for (int64_t c = 0; c < cols; ++c)
            acc += (double)w[c] * (double)(col_scaled ? scale[c] : scale[r]) * x[c];
        y[r] = acc;
    }
}

/* Matrix kind k (0..6 as in oracle_q8) of layer l: the bf16 matrix or its int8 form. */
static void mat_gemv(const oracle_model* m, int k, int l, const uint16_t* bf, int64_t rows, int64_t cols,
                     const double* x, double* y) {
    if (m->q8) oracle_gemv_q8(m->q8->q[k][l], m->q8->s[k][l], k == 6, rows, cols, x, y);
    else oracle_gemv(bf, rows, cols, x, y);
}

/* Rotary position encoding of one head vector v[hd] at position pos
 * (cloud.baidu.com/article/9434380, section 3 lists it among the decode
 * operators; the pages give no formula).  Llama "rotate-half" form: dims i and
 * i + hd/2 form a pair rotated by the angle pos * theta^(-2i/hd):
 *   v'_i        = v_i cos(a) - v_{i+hd/2} sin(a)
 *   v'_{i+hd/2} = v_{i+hd/2} cos(a) + v_i sin(a)                          */
void oracle_rope(double* v, int hd, int pos, double theta) {
    int half = hd / 2;
    for (int i = 0; i < half; ++i) {
        double inv_freq = pow(theta, -(2.0 * (double)i) / (double)hd);
        double a = (double)pos * inv_freq;
        double c = cos(a), s = sin(a);
        double x0 = v[i], x1 = v[i + half];
        v[i] = x0 * c - x1 * s;
        v[i + half] = x1 * c + x0 * s;
    }
}

/* Softmax with the maximum subtracted first, the overflow guard the pages ask
 * for (cloud.baidu.com/article/9434380, section 8, problem 4). */
void oracle_softmax(const double* s, int n, double* p) {
    double m = -INFINITY;
    for (int i = 0; i < n; ++i) if (s[i] > m) m = s[i];
    double sum = 0.0;
    for (int i = 0; i < n; ++i) { p[i] = exp(s[i] - m); sum += p[i]; }
    for (int i = 0; i < n; ++i) p[i] /= sum;
}

/* One query head over ctx cached positions (segment B of
 * cloud.baidu.com/article/9434380, section 5, step 2: scores + mask + softmax
 * + weighted sum).  K and V are bf16 [ctx][hd]; the causal mask is implicit:
 * only positions 0..ctx-1 (the current token included) are passed in.
 * out[d] = sum_p softmax_p(q . K_p / sqrt(hd)) V_p[d]. */
void oracle_attention_head(const double* q, const uint16_t* K, const uint16_t* V, int ctx, int hd, double* out) {
    double* s = (double*)malloc(sizeof(double) * (size_t)ctx);
    double* p = (double*)malloc(sizeof(double) * (size_t)ctx);
    double scale = 1.0 / sqrt((double)hd);
    for (int t = 0; t < ctx; ++t) {
        double acc = 0.0;
        for (int d = 0; d < hd; ++d) acc += q[d] * bf2d(K[(int64_t)t * hd + d]);
        s[t] = acc * scale;
    }
    oracle_softmax(s, ctx, p);
    for (int d = 0; d < hd; ++d) out[d] = 0.0;
    for (int t = 0; t < ctx; ++t)
        for (int d = 0; d < hd; ++d) out[d] += p[t] * bf2d(V[(int64_t)t * hd + d]);
    free(s);
    free(p);
}

/* SiLU activation x / (1 + e^-x); SwiGLU u_j = silu(gate_j) * up_j. */
double oracle_silu(double x) { return x / (1.0 + exp(-x)); }

/* Greedy token: index of the largest logit after rounding to float, the
 * lowest index on ties.  *nonfinite is set when any logit is NaN or infinite. */
int oracle_argmax_f32(const double* logits, int n, int* nonfinite) {
    int best = -1;
    float bv = 0.0f;
    *nonfinite = 0;
    for (int i = 0; i < n; ++i) {
        float v = (float)logits[i];
        if (!isfinite(v)) { *nonfinite = 1; continue; }
        if (best < 0 || v > bv) { best = i; bv = v; }
    }
    return best;
}

/* Sampling (cloud.baidu.com/article/9434380, section 5: step 1 names the
 * temperature among the sampling parameters, step 5 the sampling logic and the
 * stop condition on the fused path).  The pages name no sampling rule; the one
 * taken is exact sampling from softmax(logits / T) by the Gumbel-max rule:
 * the token is argmax_v (logit_v / T + G_v) with G_v independent standard
 * Gumbel noise, G = -ln(-ln U), U uniform on (0, 1).
 *
 * U comes from SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014): the generator's state starts
 * at the seed and advances by the constant 0x9E3779B97F4A7C15 before each
 * output; an output is the state passed through the mix
 *   z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31.
 * Output number i (0-based) therefore mixes seed + (i + 1) * 0x9E3779B97F4A7C15.
 * For token v at position pos, i = pos * 2^32 + v.  U = ((z >> 41) + 0.5) * 2^-23
 * (23 bits plus the half: 24 significant bits, exact in float; never 0 or 1).  Everything after U is fp32 (the precision the
 * GPU decides the token in): G = -logf(-logf(U)), key = fmaf(logit, 1/T, G),
 * with the logit rounded to float first. */
uint64_t oracle_splitmix64_output(uint64_t seed, uint64_t i) {
    uint64_t z = seed + (i + 1u) * 0x9E3779B97F4A7C15ull;   /* the state after i + 1 advances */
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    z ^= z >> 31;
    return z;
}

float oracle_uniform_f32(uint64_t seed, int pos, int v) {
    const uint64_t i = ((uint64_t)(uint32_t)pos << 32) | (uint32_t)v;
    const uint64_t z = oracle_splitmix64_output(seed, i);
    return ((float)(uint32_t)(z >> 41) + 0.5f) * (1.0f / 8388608.0f);
}

float oracle_gumbel_f32(uint64_t seed, int pos, int v) {
    const float u = oracle_uniform_f32(seed, pos, v);
    return -logf(-logf(u));
}

/* Sampled token: inv_temp <= 0 is the greedy argmax; otherwise the largest
 * key over the finite logits, the lowest index on ties.  *nonfinite as in
 * oracle_argmax_f32. */
int oracle_sample_f32(const double* logits, int n, float inv_temp, uint64_t seed, int pos, int* nonfinite) {
    if (!(inv_temp > 0.0f)) return oracle_argmax_f32(logits, n, nonfinite);
    int best = -1;
    float bk = 0.0f;
    *nonfinite = 0;
    for (int i = 0; i < n; ++i) {
        const float v = (float)logits[i];
        if (!isfinite(v)) { *nonfinite = 1; continue; }
        const float key = fmaf(v, inv_temp, oracle_gumbel_f32(seed, pos, i));
        if (best < 0 || key > bk) { best = i; bk = key; }
    }
    return best;
}

/* Nucleus (top-p) sampling (cloud.baidu.com/article/9434380, section 5,
 * step 1 names top-p beside the temperature as a fixed sampling parameter;
 * the page gives no rule, the one taken is the usual nucleus restriction made
 * independent of how ties are ordered): with x_v = float(logit_v) * (1/T) in
 * float and probabilities q_v = exp(x_v - max x) / sum_u exp(x_u - max x) in
 * double, token v is kept iff the probability of the tokens strictly more
 * probable than it is below p:  sum_{u : x_u > x_v} q_u < p.  The token is
 * then the Gumbel-max choice (as oracle_sample_f32) over the kept tokens only,
 * which samples from softmax(x) restricted to the kept set and renormalised.
 * top_p >= 1 keeps every token; inv_temp <= 0 is greedy.  Plain O(n log n):
 * sort by x descending and accumulate the mass of each group of equal x. */
static const float* g_sort_x;
static int cmp_x_desc(const void* a, const void* b) {
    const float xa = g_sort_x[*(const int*)a], xb = g_sort_x[*(const int*)b];
    return (xa < xb) - (xa > xb);
}

int oracle_sample_topp_f32(const double* logits, int n, float inv_temp, double top_p, uint64_t seed, int pos,
                           int* nonfinite) {
    if (!(inv_temp > 0.0f) || !(top_p < 1.0)) return oracle_sample_f32(logits, n, inv_temp, seed, pos, nonfinite);
    float* x = (float*)malloc(sizeof(float) * (size_t)n);
    int* idx = (int*)malloc(sizeof(int) * (size_t)n);
    unsigned char* keep = (unsigned char*)calloc((size_t)n, 1);
    int m = 0;
    *nonfinite = 0;
    for (int v = 0; v < n; ++v) {
        const float y = (float)logits[v];
        if (!isfinite(y)) { *nonfinite = 1; continue; }
        x[v] = y * inv_temp;
        idx[m++] = v;
    }
    int best = -1;
    if (m > 0) {
        g_sort_x = x;
        qsort(idx, (size_t)m, sizeof(int), cmp_x_desc);
        const double xmax = (double)x[idx[0]];
        double z = 0.0;
        for (int k = 0; k < m; ++k) z += exp((double)x[idx[k]] - xmax);
        double above = 0.0;                      /* mass of the tokens strictly more probable */
        for (int k = 0; k < m;) {
            int e = k;
            double grp = 0.0;
            while (e < m && x[idx[e]] == x[idx[k]]) { grp += exp((double)x[idx[e]] - xmax); ++e; }
            const int kept = above < top_p * z;
            for (int q = k; q < e; ++q) keep[idx[q]] = (unsigned char)kept;
            above += grp;
            k = e;
        }
        float bk = 0.0f;
        for (int v = 0; v < n; ++v) {
            if (!keep[v]) continue;
            const float key = fmaf((float)logits[v], inv_temp, oracle_gumbel_f32(seed, pos, v));
            if (best < 0 || key > bk) { best = v; bk = key; }
        }
    }
    free(x); free(idx); free(keep);
    return best;
}

/* One decode step: feed `token` at position `pos`, append its K/V to the
 * cache, return logits [vocab] and the final-norm hidden state [hidden].
 * kcache / vcache: bf16 [n_layers][n_kv_heads][max_seq][head_dim]; positions
 * 0..pos-1 must already hold the earlier steps' K (rotated) and V.
 * Returns 0, or -1 for bad arguments. */
int oracle_decode_step(const oracle_model* m, uint16_t* kcache, uint16_t* vcache, int token, int pos,
                       double* logits, double* hidden) {
    const int H = m->hidden, hd = m->head_dim, qh = m->n_q_heads, kvh = m->n_kv_heads, F = m->ffn;
    if (token < 0 || token >= m->vocab || pos < 0 || pos >= m->max_seq || qh % kvh != 0) return -1;
    const int group = qh / kvh;
    double* x = (double*)malloc(sizeof(double) * H);
    double* xn = (double*)malloc(sizeof(double) * H);
    double* q = (double*)malloc(sizeof(double) * (size_t)qh * hd);
    double* k = (double*)malloc(sizeof(double) * (size_t)kvh * hd);
    double* v = (double*)malloc(sizeof(double) * (size_t)kvh * hd);
    double* att = (double*)malloc(sizeof(double) * (size_t)qh * hd);
    double* o = (double*)malloc(sizeof(double) * H);
    double* gate = (double*)malloc(sizeof(double) * F);
    double* up = (double*)malloc(sizeof(double) * F);
    double* u = (double*)malloc(sizeof(double) * F);

    /* embedding row */
    for (int i = 0; i < H; ++i) x[i] = bf2d(m->embed[(int64_t)token * H + i]);

    for (int l = 0; l < m->n_layers; ++l) {
        /* segment A: RMSNorm, Q/K/V projections, RoPE on q and k, K/V append */
        oracle_rmsnorm(x, m->attn_norm[l], H, m->rms_eps, xn);
        mat_gemv(m, 0, l, m->wq[l], (int64_t)qh * hd, H, xn, q);
        mat_gemv(m, 1, l, m->wk[l], (int64_t)kvh * hd, H, xn, k);
        mat_gemv(m, 2, l, m->wv[l], (int64_t)kvh * hd, H, xn, v);
        for (int h = 0; h < qh; ++h) oracle_rope(q + (int64_t)h * hd, hd, pos, m->rope_theta);
        for (int g = 0; g < kvh; ++g) oracle_rope(k + (int64_t)g * hd, hd, pos, m->rope_theta);
        for (int g = 0; g < kvh; ++g) {
            int64_t base = (((int64_t)l * kvh + g) * m->max_seq + pos) * hd;
            for (int d = 0; d < hd; ++d) {
                kcache[base + d] = oracle_round_bf16(k[(int64_t)g * hd + d]);
                vcache[base + d] = oracle_round_bf16(v[(int64_t)g * hd + d]);
            }
        }
        /* segment B: attention over positions 0..pos; q head h reads kv head
         * h / (qh/kvh) (grouped-query attention), then output projection and
         * the residual add. */
#pragma omp parallel for schedule(static)
        for (int h = 0; h < qh; ++h) {
            int g = h / group;
            int64_t base = ((int64_t)l * kvh + g) * m->max_seq * hd;
            oracle_attention_head(q + (int64_t)h * hd, kcache + base, vcache + base, pos + 1, hd, att + (int64_t)h * hd);
        }
        mat_gemv(m, 3, l, m->wo[l], H, (int64_t)qh * hd, att, o);
        for (int i = 0; i < H; ++i) x[i] += o[i];
        /* segment C: RMSNorm, gate/up projections, SwiGLU, down projection,
         * residual add */
        oracle_rmsnorm(x, m->ffn_norm[l], H, m->rms_eps, xn);
        mat_gemv(m, 4, l, m->w_gate[l], F, H, xn, gate);
        mat_gemv(m, 5, l, m->w_up[l], F, H, xn, up);
        for (int j = 0; j < F; ++j) u[j] = oracle_silu(gate[j]) * up[j];
        mat_gemv(m, 6, l, m->w_down[l], H, F, u, o);
        for (int i = 0; i < H; ++i) x[i] += o[i];
    }
    /* final norm, LM head */
    oracle_rmsnorm(x, m->final_norm, H, m->rms_eps, hidden);
    if (m->q8) oracle_gemv_q8(m->q8->lm_q, m->q8->lm_s, 0, m->vocab, H, hidden, logits);
    else oracle_gemv(m->lm_head, m->vocab, H, hidden, logits);

    free(x); free(xn); free(q); free(k); free(v); free(att); free(o); free(gate); free(up); free(u);
    return 0;
}
