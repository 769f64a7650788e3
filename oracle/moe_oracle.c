/*
 * moe_oracle.c -- plain, slow CPU oracle for the DeepSeek-V3-style MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls this file;
 * only the tests, the smoke check and the benchmark's CPU-baseline leg use it.  It shares
 * no code, header, table or constant generator with the CUDA library.
 *
 * Sources (cited by page title and section):
 *  [P1] "从 1024 块 GPU 到 558 万美元：拆解 DeepSeek-V3 的算法-系统协同设计" (wsisp.com)
 *       §2.2 MoEGate listing (sigmoid gate, selection-only bias, group-limited top-k,
 *       weights from un-biased scores, normalisation, routed_scaling_factor);
 *       §2.3 dispatch skeleton (per-expert counts, argsort of the flat expert ids);
 *       §5.1 blockwise FP8 GEMM sketch (FP8 operands, per-block scales applied during
 *       accumulation, FP32 accumulation, output quantised as needed).
 *  [P2] "深入理解 DeepSeek-V3" -- Chinese précis of "Insights into DeepSeek-V3: Scaling
 *       Challenges and Reflections on Hardware for AI Architectures" (arXiv 2505.09343)
 *       §3.1 (8 routed + 1 shared expert per token; FP8 dispatch, BF16 combine);
 *       §3.2 (activations quantised in 1x128 tiles, weights in 128x128 blocks, each with
 *       a scale; FP32 accumulation requested).
 *  [OFP8] OCP "8-bit Floating Point Specification (OFP8)" rev 1.0, E4M3 encoding table.
 *
 * Readings of the pages where they are silent (each also listed in the design notes):
 *  - experts outside the kept groups are masked with -inf (the listing writes 0.0; the two
 *    agree whenever every selection score is positive);
 *  - ties in every top-k go to the lower index; slots are in descending selection score;
 *  - a block scale is amax/448 in FP32 (amax == 0 gives scale 1 and all-zero codes), and
 *    values are encoded as e4m3(v * (448/amax)) with round-to-nearest-even and saturation;
 *  - power-of-two mode (the *_pow2 entry points): [P2 §3.2] recommends tensor cores that
 *    take the scaling factors natively, as Blackwell's microscaling does, and microscaling
 *    scales are powers of two (an 8-bit exponent, 2^-127 .. 2^127).  The scale of a tile or
 *    block is then the smallest power of two s with 448 * s >= amax, clamped to that range,
 *    so no value saturates; codes = e4m3(v * 2^-e), an exact scaling (amax == 0 as above);
 *  - the expert FFN is SwiGLU: down(silu(gate(x)) * up(x)), no biases, gate rows 0..I-1
 *    and up rows I..2I-1 of the stacked first weight;
 *  - h goes from FP32 straight to FP8 1x128 tiles; expert outputs are BF16 and unweighted;
 *    the combine weights them in FP32 in slot order, adds the shared expert, rounds once;
 *  - the load-driven bias update is b_i += 1e-3 * sign(mean_load - load_i).
 *
 * Arithmetic: dot products accumulate in double and are rounded to float once, so the
 * oracle is the exact result up to that final rounding.  Products of two E4M3 values are
 * exact in double and a 128-term block sum of them is exact in double too.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------------------ */
/* number formats                                                                        */
/* ------------------------------------------------------------------------------------ */

/* BF16 -> FP32 is exact: the BF16 bits are the upper half of the FP32 bits. */
float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* FP32 -> BF16, round to nearest, ties to even (the IEEE default rounding). */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u); /* NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* [OFP8] E4M3: sign bit, 4 exponent bits (bias 7), 3 mantissa bits.  Exponent field 0
 * holds the subnormals m * 2^-9; S.1111.111 is NaN; there is no infinity, so the
 * largest finite magnitude is S.1111.110 = 1.75 * 2^8 = 448. */
double orc_e4m3_to_double(uint8_t code)
{
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* Magnitudes of the non-negative finite codes 0..126 (increasing in the code), filled once
 * from orc_e4m3_to_double. */
static double g_mag[127];
static int g_mag_ready = 0;

static void mag_init(void)
{
    if (g_mag_ready) return;
#pragma omp critical(orc_mag_init)
    {
        if (!g_mag_ready) {
            for (int c = 0; c < 127; ++c) g_mag[c] = orc_e4m3_to_double((uint8_t)c);
            g_mag_ready = 1;
        }
    }
}

static inline double e4m3_mag(int c) { return g_mag[c]; }

/* FP32 -> E4M3 by the definition of round-to-nearest-even with saturation to the largest
 * finite value: pick the representable magnitude nearest to |v|; on an exact tie pick the
 * code whose last bit is 0.  Magnitudes at or above 448 (including infinity) give 448.
 * NaN gives S.1111.111. */
uint8_t orc_f32_to_e4m3(float v)
{
    mag_init();
    if (isnan(v)) return 0x7f;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return sign | 0x7e;
    int lo = 0; /* largest code whose magnitude is <= a (binary search, fixed 7 steps) */
    for (int step = 64; step > 0; step >>= 1) {
        int m = lo + step;
        lo = (m <= 126 && e4m3_mag(m) <= a) ? m : lo;
    }
    double dlo = a - e4m3_mag(lo), dhi = e4m3_mag(lo + 1) - a; /* both exact in double */
    int c;
    if (dlo < dhi) c = lo;
    else if (dhi < dlo) c = lo + 1;
    else c = (lo & 1) ? lo + 1 : lo;
    return sign | (uint8_t)c;
}

/* Element i of an input array that is FP32 (is_bf16 == 0) or BF16 (is_bf16 != 0). */
static inline float load_elem(const void* p, int is_bf16, int64_t i)
{
    return is_bf16 ? orc_bf16_to_f32(((const uint16_t*)p)[i]) : ((const float*)p)[i];
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------------------ */
/* [P2 §3.2] fine-grained quantisation                                                   */
/* ------------------------------------------------------------------------------------ */

/* Exponent e of the power-of-two scale of a tile with amax > 0: the smallest integer with
 * 448 * 2^e >= amax (448 * 2^e is exact in double), clamped to [-127, 127], the range of an
 * 8-bit power-of-two scale. */
static int pow2_exponent(float amax)
{
    const double a = (double)amax;
    int e = (int)ceil(log2(a / 448.0));  /* first guess; corrected exactly below */
    while (e > -127 && ldexp(448.0, e - 1) >= a) --e;
    while (e < 127 && ldexp(448.0, e) < a) ++e;
    if (e < -127) e = -127;
    return e;
}

/* Encode one tile of n values (v[i*stride]) given its amax; writes codes and returns the
 * FP32 scale.  scale = amax/448; codes = e4m3(v * (448/amax)); amax == 0 -> scale 1.
 * pow2 != 0: scale = 2^e (pow2_exponent), codes = e4m3(v * 2^-e). */
static float quant_tile(float amax, int pow2, const void* src, int64_t base, int is_bf16, int64_t n,
                        int64_t stride, uint8_t* dst, int64_t dbase, int64_t dstride)
{
    if (amax == 0.0f) {
        for (int64_t i = 0; i < n; ++i) dst[dbase + i * dstride] = 0;
        return 1.0f;
    }
    if (pow2) {
        /* v * 2^-e is exact wherever the product is a normal float; below that the code is 0
         * whichever way the product rounds (E4M3's smallest step is 2^-9). */
        const int e = pow2_exponent(amax);
        for (int64_t i = 0; i < n; ++i) {
            float v = load_elem(src, is_bf16, base + i * stride);
            dst[dbase + i * dstride] = orc_f32_to_e4m3((float)ldexp((double)v, -e));
        }
        return (float)ldexp(1.0, e);
    }
    float mul = 448.0f / amax;
    for (int64_t i = 0; i < n; ++i) {
        float v = load_elem(src, is_bf16, base + i * stride);
        dst[dbase + i * dstride] = orc_f32_to_e4m3(v * mul);
    }
    return amax / 448.0f;
}

/* Activations: one scale per row per 128 consecutive columns.
 * x [rows, cols] (cols % 128 == 0) -> q [rows, cols] E4M3 codes, s [rows, cols/128]. */
static void quant_1x128(int64_t rows, int64_t cols, const void* x, int x_is_bf16, int pow2,
                        uint8_t* q, float* s)
{
    int64_t nb = cols / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            int64_t base = r * cols + b * 128;
            float amax = 0.0f;
            for (int64_t i = 0; i < 128; ++i) {
                float a = fabsf(load_elem(x, x_is_bf16, base + i));
                if (a > amax) amax = a;
            }
            s[r * nb + b] = quant_tile(amax, pow2, x, base, x_is_bf16, 128, 1, q, base, 1);
        }
    }
}

void orc_quant_1x128(int64_t rows, int64_t cols, const void* x, int x_is_bf16, uint8_t* q, float* s)
{
    quant_1x128(rows, cols, x, x_is_bf16, 0, q, s);
}

void orc_quant_1x128_pow2(int64_t rows, int64_t cols, const void* x, int x_is_bf16, uint8_t* q, float* s)
{
    quant_1x128(rows, cols, x, x_is_bf16, 1, q, s);
}

/* Weights: one scale per 128x128 block of each matrix.
 * w [n_mats, rows, cols] (rows, cols % 128 == 0) -> q same shape, s [n_mats, rows/128, cols/128]. */
static void quant_128x128(int64_t n_mats, int64_t rows, int64_t cols, const void* w, int w_is_bf16,
                          int pow2, uint8_t* q, float* s)
{
    int64_t rb = rows / 128, cb = cols / 128;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < n_mats; ++m) {
        for (int64_t i = 0; i < rb; ++i) {
            for (int64_t j = 0; j < cb; ++j) {
                int64_t base = m * rows * cols + i * 128 * cols + j * 128;
                float amax = 0.0f;
                for (int64_t r = 0; r < 128; ++r)
                    for (int64_t c = 0; c < 128; ++c) {
                        float a = fabsf(load_elem(w, w_is_bf16, base + r * cols + c));
                        if (a > amax) amax = a;
                    }
                float scale = 1.0f;
                for (int64_t r = 0; r < 128; ++r)
                    scale = quant_tile(amax, pow2, w, base + r * cols, w_is_bf16, 128, 1, q,
                                       base + r * cols, 1);
                s[(m * rb + i) * cb + j] = scale;
            }
        }
    }
}

void orc_quant_128x128(int64_t n_mats, int64_t rows, int64_t cols, const void* w, int w_is_bf16,
                       uint8_t* q, float* s)
{
    quant_128x128(n_mats, rows, cols, w, w_is_bf16, 0, q, s);
}

void orc_quant_128x128_pow2(int64_t n_mats, int64_t rows, int64_t cols, const void* w, int w_is_bf16,
                            uint8_t* q, float* s)
{
    quant_128x128(n_mats, rows, cols, w, w_is_bf16, 1, q, s);
}

/* ------------------------------------------------------------------------------------ */
/* [P1 §2.2] MoEGate                                                                     */
/* ------------------------------------------------------------------------------------ */

/* For every token: logits = x . Wg^T (accumulated in double, rounded to float), scores =
 * sigmoid(logits), selection scores c = scores + bias; group score = sum of the two largest
 * c in the group; keep the topk_group groups with the largest group scores; among experts
 * in kept groups take the top_k largest c; weights = scores at those experts, divided by
 * (their sum + 1e-20) when top_k > 1, then multiplied by routed_scaling_factor.
 *
 * x [T,H], Wg [E,H] (FP32 or BF16); bias [E].  Outputs: topk_idx/topk_w [T,K] in
 * descending-c slot order; scores_out [T,E] (may be NULL); margin [T] (may be NULL) =
 * min over the group cut (TG-th vs best dropped group score) and the expert cut (K-th vs
 * best unselected candidate c); +inf where a cut does not exist. */
void orc_gate(int64_t T, int H, int E, int G, int TG, int K, float rsf,
              const void* x, int x_is_bf16, const void* Wg, int w_is_bf16, const float* bias,
              int32_t* topk_idx, float* topk_w, float* scores_out, float* margin)
{
    int gsz = E / G;
    /* the gate weight widened to double once (exact) */
    double* wd = (double*)malloc(sizeof(double) * (size_t)E * H);
    for (int64_t i = 0; i < (int64_t)E * H; ++i) wd[i] = (double)load_elem(Wg, w_is_bf16, i);
#pragma omp parallel
    {
        float* s = (float*)malloc(sizeof(float) * E);
        float* c = (float*)malloc(sizeof(float) * E);
        float* gs = (float*)malloc(sizeof(float) * G);
        char* gkeep = (char*)malloc(G);
        char* taken = (char*)malloc(E);
        double* xd = (double*)malloc(sizeof(double) * H);
#pragma omp for schedule(dynamic, 16)
        for (int64_t t = 0; t < T; ++t) {
            for (int h = 0; h < H; ++h) xd[h] = (double)load_elem(x, x_is_bf16, t * H + h);
            /* logits and sigmoid scores */
            for (int e = 0; e < E; ++e) {
                const double* wr = wd + (int64_t)e * H;
                double acc = 0.0;
                for (int h = 0; h < H; ++h) acc += xd[h] * wr[h];
                float logit = (float)acc;
                s[e] = (float)(1.0 / (1.0 + exp(-(double)logit)));
                c[e] = s[e] + bias[e];
            }
            if (scores_out)
                for (int e = 0; e < E; ++e) scores_out[t * E + e] = s[e];
            /* group scores: sum of the two largest selection scores of each group */
            for (int g = 0; g < G; ++g) {
                float b1 = -INFINITY, b2 = -INFINITY;
                for (int j = 0; j < gsz; ++j) {
                    float v = c[g * gsz + j];
                    if (v > b1) { b2 = b1; b1 = v; }
                    else if (v > b2) b2 = v;
                }
                gs[g] = b1 + b2;
                gkeep[g] = 0;
            }
            /* keep topk_group groups: repeated arg-max, ties to the lower group index */
            float last_kept_gs = INFINITY;
            for (int r = 0; r < TG; ++r) {
                int best = -1;
                for (int g = 0; g < G; ++g)
                    if (!gkeep[g] && (best < 0 || gs[g] > gs[best])) best = g;
                gkeep[best] = 1;
                last_kept_gs = gs[best];
            }
            float best_dropped_gs = -INFINITY;
            for (int g = 0; g < G; ++g)
                if (!gkeep[g] && gs[g] > best_dropped_gs) best_dropped_gs = gs[g];
            /* top_k experts among kept groups (masked experts count as -inf) */
            for (int e = 0; e < E; ++e) taken[e] = 0;
            float last_c = INFINITY;
            for (int k = 0; k < K; ++k) {
                int best = -1;
                for (int e = 0; e < E; ++e) {
                    if (taken[e] || !gkeep[e / gsz]) continue;
                    if (best < 0 || c[e] > c[best]) best = e;
                }
                taken[best] = 1;
                topk_idx[t * K + k] = best;
                last_c = c[best];
            }
            float best_unsel_c = -INFINITY;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && gkeep[e / gsz] && c[e] > best_unsel_c) best_unsel_c = c[e];
            if (margin) {
                float mg = (TG < G) ? last_kept_gs - best_dropped_gs : INFINITY;
                float me = last_c - best_unsel_c;
                margin[t] = mg < me ? mg : me;
            }
            /* weights from the un-biased scores */
            float w[1024];
            for (int k = 0; k < K; ++k) w[k] = s[topk_idx[t * K + k]];
            if (K > 1) {
                float den = 0.0f;
                for (int k = 0; k < K; ++k) den = den + w[k];
                den = den + 1e-20f;
                for (int k = 0; k < K; ++k) w[k] = w[k] / den;
            }
            for (int k = 0; k < K; ++k) topk_w[t * K + k] = w[k] * rsf;
        }
        free(s); free(c); free(gs); free(gkeep); free(taken); free(xd);
    }
    free(wd);
}

/* ------------------------------------------------------------------------------------ */
/* [P1 §2.3] counts and permutation by expert                                            */
/* ------------------------------------------------------------------------------------ */

/* counts[e] = number of (token, slot) pairs routed to e.  Rows are ordered expert-major and,
 * within an expert, by ascending token index (the stable argsort of the flat expert ids).
 * With has_shared, slot group E holds every token once, in order, in rows [T*K, T*K + T).
 * offs [E+1+has_shared]: offs[e] = rows of the experts before e, offs[E] = T*K; perm_tok[row]
 * is the token of a row; row_of[t*K+k] is the row of (t, k).
 * An id outside [0, E) never comes out of the gate; the library contract (not the pages)
 * drops such a slot: it counts for no expert, row_of = -1, and the V valid slots fill rows
 * [0, V) while rows [V, T*K) get perm_tok = -1 (the last expert's range reaches T*K). */
void orc_permute(int64_t T, int E, int K, int has_shared, const int32_t* topk_idx,
                 int32_t* counts, int32_t* offs, int32_t* perm_tok, int32_t* row_of)
{
    int64_t* fill = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t i = 0; i < T * K; ++i)
        if (topk_idx[i] >= 0 && topk_idx[i] < E) counts[topk_idx[i]] += 1;
    offs[0] = 0;
    for (int e = 1; e < E; ++e) offs[e] = offs[e - 1] + counts[e - 1];
    int64_t n_valid = (int64_t)offs[E - 1] + counts[E - 1];
    offs[E] = (int32_t)(T * K);
    if (has_shared) offs[E + 1] = offs[E] + (int32_t)T;
    for (int64_t r = n_valid; r < T * K; ++r) perm_tok[r] = -1;
    for (int64_t t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int e = topk_idx[t * K + k];
            if (e < 0 || e >= E) {
                row_of[t * K + k] = -1;
                continue;
            }
            int64_t pos = offs[e] + fill[e]++;
            perm_tok[pos] = (int32_t)t;
            row_of[t * K + k] = (int32_t)pos;
        }
    if (has_shared)
        for (int64_t t = 0; t < T; ++t) perm_tok[offs[E] + t] = (int32_t)t;
    free(fill);
}

/* load-driven bias update: b_i += 1e-3 * sign(mean_load - load_i), mean_load = T*K/E.
 * The sign is taken in integers: sign(T*K - E*load_i). */
void orc_bias_update(int E, int64_t T, int K, const int32_t* counts, float* bias)
{
    for (int e = 0; e < E; ++e) {
        int64_t d = T * (int64_t)K - (int64_t)E * (int64_t)counts[e];
        int sgn = (d > 0) - (d < 0);
        bias[e] = bias[e] + 1e-3f * (float)sgn;
    }
}

/* ------------------------------------------------------------------------------------ */
/* [P1 §5.1][P2 §3.2] routed / shared SwiGLU expert with blockwise FP8 operands          */
/* ------------------------------------------------------------------------------------ */

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* One dot product of a 1x128-scaled activation row with a 128x128-scaled weight row:
 * sum_kb (sa[kb]*sb[kb]) * sum_{k in kb} dq(a_k)*dq(w_k), in double. */
static double block_dot(int K, const double* a_dq, const float* a_s, const uint8_t* w,
                        const float* w_s, const double* lut)
{
    double acc = 0.0;
    for (int kb = 0; kb < K / 128; ++kb) {
        double p = 0.0;
        for (int k = kb * 128; k < kb * 128 + 128; ++k) p += a_dq[k] * lut[w[k]];
        acc += ((double)a_s[kb] * (double)w_s[kb]) * p;
    }
    return acc;
}

/* rows x [n_rows] each through expert row_expert[r]:
 *   g_j = <x, W13[e, j]>, u_j = <x, W13[e, I + j]>      (1x128 x 128x128 blockwise, FP32 result)
 *   h_j = silu(g_j) * u_j                                (in double, rounded to FP32)
 *   hq, hs = 1x128 quantisation of h
 *   y_n = <hq, W2[e, n]>                                 (blockwise, rounded to BF16)
 * aq [n_rows, H] codes, as [n_rows, H/128]; W13 [nE, 2I, H], W13s [nE, 2I/128, H/128];
 * W2 [nE, H, I], W2s [nE, H/128, I/128].  gu_out [n_rows, 2I] (g then u, FP32),
 * h_out [n_rows, I] (FP32), hq_out/hs_out: each may be NULL; y_out [n_rows, H] BF16 bits. */
static void ffn_fp8(int64_t n_rows, int H, int I, const uint8_t* aq, const float* as,
                    const int32_t* row_expert, const uint8_t* W13, const float* W13s,
                    const uint8_t* W2, const float* W2s, int pow2, float* gu_out, float* h_out,
                    uint8_t* hq_out, float* hs_out, uint16_t* y_out)
{
    double lut[256];
    for (int c = 0; c < 256; ++c) lut[c] = orc_e4m3_to_double((uint8_t)c);
    int hb = H / 128, ib = I / 128;
#pragma omp parallel
    {
        double* a_dq = (double*)malloc(sizeof(double) * H);
        double* h_dq = (double*)malloc(sizeof(double) * I);
        float* h = (float*)malloc(sizeof(float) * I);
        uint8_t* hq = (uint8_t*)malloc(I);
        float* hs = (float*)malloc(sizeof(float) * ib);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r) {
            int64_t e = row_expert[r];
            const uint8_t* w13 = W13 + e * (int64_t)(2 * I) * H;
            const float* w13s = W13s + e * (int64_t)(2 * I / 128) * hb;
            const uint8_t* w2 = W2 + e * (int64_t)H * I;
            const float* w2s = W2s + e * (int64_t)hb * ib;
            for (int k = 0; k < H; ++k) a_dq[k] = lut[aq[r * H + k]];
            const float* sa = as + r * hb;
            for (int j = 0; j < I; ++j) {
                float g = (float)block_dot(H, a_dq, sa, w13 + (int64_t)j * H,
                                           w13s + (int64_t)(j / 128) * hb, lut);
                float u = (float)block_dot(H, a_dq, sa, w13 + (int64_t)(I + j) * H,
                                           w13s + (int64_t)((I + j) / 128) * hb, lut);
                h[j] = (float)(silu((double)g) * (double)u);
                if (gu_out) {
                    gu_out[r * 2 * I + j] = g;
                    gu_out[r * 2 * I + I + j] = u;
                }
            }
            quant_1x128(1, I, h, 0, pow2, hq, hs);
            for (int k = 0; k < I; ++k) h_dq[k] = lut[hq[k]];
            for (int n = 0; n < H; ++n) {
                float y = (float)block_dot(I, h_dq, hs, w2 + (int64_t)n * I,
                                           w2s + (int64_t)(n / 128) * ib, lut);
                y_out[r * H + n] = orc_f32_to_bf16(y);
            }
            if (h_out) memcpy(h_out + r * I, h, sizeof(float) * I);
            if (hq_out) memcpy(hq_out + r * I, hq, I);
            if (hs_out) memcpy(hs_out + r * ib, hs, sizeof(float) * ib);
        }
        free(a_dq); free(h_dq); free(h); free(hq); free(hs);
    }
}

void orc_ffn_fp8(int64_t n_rows, int H, int I, const uint8_t* aq, const float* as,
                 const int32_t* row_expert, const uint8_t* W13, const float* W13s,
                 const uint8_t* W2, const float* W2s, float* gu_out, float* h_out,
                 uint8_t* hq_out, float* hs_out, uint16_t* y_out)
{
    ffn_fp8(n_rows, H, I, aq, as, row_expert, W13, W13s, W2, W2s, 0, gu_out, h_out, hq_out, hs_out, y_out);
}

/* The same with h re-quantised in power-of-two mode (the operands come quantised by the
 * *_pow2 entry points; the blockwise sum itself is the same for either kind of scale). */
void orc_ffn_fp8_pow2(int64_t n_rows, int H, int I, const uint8_t* aq, const float* as,
                      const int32_t* row_expert, const uint8_t* W13, const float* W13s,
                      const uint8_t* W2, const float* W2s, float* gu_out, float* h_out,
                      uint8_t* hq_out, float* hs_out, uint16_t* y_out)
{
    ffn_fp8(n_rows, H, I, aq, as, row_expert, W13, W13s, W2, W2s, 1, gu_out, h_out, hq_out, hs_out, y_out);
}

/* The same expert FFN with every operand in FP32 and no quantisation (the all-FP32 layer):
 * g, u, y are double-accumulated dot products rounded to FP32; h = silu(g)*u rounded to FP32.
 * x [n_rows, H]; W13 [nE, 2I, H]; W2 [nE, H, I]; h_out [n_rows, I] may be NULL;
 * y_out [n_rows, H] FP32. */
void orc_ffn_f32(int64_t n_rows, int H, int I, const float* x, const int32_t* row_expert,
                 const float* W13, const float* W2, float* h_out, float* y_out)
{
#pragma omp parallel
    {
        float* h = (float*)malloc(sizeof(float) * I);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r) {
            int64_t e = row_expert[r];
            const float* w13 = W13 + e * (int64_t)(2 * I) * H;
            const float* w2 = W2 + e * (int64_t)H * I;
            const float* xr = x + r * H;
            for (int j = 0; j < I; ++j) {
                double g = 0.0, u = 0.0;
                for (int k = 0; k < H; ++k) {
                    g += (double)xr[k] * (double)w13[(int64_t)j * H + k];
                    u += (double)xr[k] * (double)w13[(int64_t)(I + j) * H + k];
                }
                h[j] = (float)(silu((double)(float)g) * (double)(float)u);
            }
            for (int n = 0; n < H; ++n) {
                double y = 0.0;
                for (int k = 0; k < I; ++k) y += (double)h[k] * (double)w2[(int64_t)n * I + k];
                y_out[r * H + n] = (float)y;
            }
            if (h_out) memcpy(h_out + r * I, h, sizeof(float) * I);
        }
        free(h);
    }
}

/* ------------------------------------------------------------------------------------ */
/* [P1 §2.3] combine; [P2 §3.1] BF16 combine payload                                     */
/* ------------------------------------------------------------------------------------ */

/* y[t] = sum_k w[t,k] * yk[t,k] (FP32, slot order) + ysh[t] (if given), one FP32 result per
 * element: each step is a separate FP32 multiply and FP32 add.  yk [n_tok, K, H] and ysh
 * [n_tok, H] are FP32 or BF16 (y_is_bf16); acc_out [n_tok, H] FP32. */
void orc_combine(int64_t n_tok, int K, int H, const void* yk, const void* ysh, int y_is_bf16,
                 const float* w, float* acc_out)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n_tok; ++t) {
        for (int n = 0; n < H; ++n) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                float prod = w[t * K + k] * load_elem(yk, y_is_bf16, (t * K + k) * H + n);
                acc = acc + prod;
            }
            if (ysh) acc = acc + load_elem(ysh, y_is_bf16, t * H + n);
            acc_out[t * H + n] = acc;
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* [P2 §3.2] LogFMT-nBit: a logarithmic code for 1x128 tiles of the combine payload      */
/* ------------------------------------------------------------------------------------ */

/* The précis' description (Insights into DeepSeek-V3 §3.2, LogFMT communication compression):
 * per 1x128 tile take the logarithm of the magnitudes and their min and max; the min is coded
 * S.00..01 and the max S.11..11, Step = (max - min) / (2^(n-1) - 2), zero is S.00..00, every
 * other value is rounded to an integer multiple K of Step, and K decodes to
 * exp(min + Step * (K - 1)); the rounding must happen in linear space (unbiased), and min is
 * held above max - ln(2^32).  Readings where the text is silent:
 *  - natural logarithm (the decoder is written with exp);
 *  - min and max run over the tile's non-zero values; a tile of zeros has min = Step = 0 and
 *    all codes zero; a tile whose non-zero magnitudes are all equal has Step = 0 and codes 1;
 *  - the tile's metadata travel as two FP32 numbers (min, Step), and the grid the decoder
 *    rebuilds from them, d(K) = exp(min + Step * (K - 1)), is the grid the encoder rounds to;
 *  - "rounding in linear space": a magnitude a is coded with the K whose d(K) is nearest to a
 *    (with d(0) = 0), ties to the larger K; K never exceeds 2^(n-1) - 1;
 *  - the sign is the top bit of the n-bit code (S), also for zero.
 * Decisions are taken in double on the FP32 metadata.  margin_out (may be NULL) receives, per
 * value, its distance to the decision midpoint as a fraction of the gap between the two
 * neighbouring grid values (+inf where no choice was made). */
static double logfmt_grid(double lmin, double step, int K)
{
    return K == 0 ? 0.0 : exp(lmin + step * (double)(K - 1));
}

void orc_logfmt_encode(int64_t rows, int64_t cols, const void* x, int x_is_bf16, int n_bits,
                       uint16_t* codes, float* lmin_out, float* step_out, float* margin_out)
{
    const int kmax = (1 << (n_bits - 1)) - 1;
    const int64_t tiles = cols / 128;
#pragma omp parallel for schedule(static)
    for (int64_t tt = 0; tt < rows * tiles; ++tt) {
        const int64_t base = (tt / tiles) * cols + (tt % tiles) * 128;
        double amax = 0.0, amin = INFINITY;
        for (int j = 0; j < 128; ++j) {
            double a = fabs((double)load_elem(x, x_is_bf16, base + j));
            if (a > 0.0) {
                if (a > amax) amax = a;
                if (a < amin) amin = a;
            }
        }
        float lmin_f = 0.0f, step_f = 0.0f;
        if (amax > 0.0) {
            double lmax = log(amax), lmn = log(amin);
            if (lmn < lmax - 32.0 * log(2.0)) lmn = lmax - 32.0 * log(2.0);
            lmin_f = (float)lmn;
            step_f = (float)((lmax - lmn) / (double)(kmax - 1));
        }
        lmin_out[tt] = lmin_f;
        step_out[tt] = step_f;
        for (int j = 0; j < 128; ++j) {
            float v = load_elem(x, x_is_bf16, base + j);
            uint16_t sgn = signbit(v) ? (uint16_t)(1u << (n_bits - 1)) : 0;
            double a = fabs((double)v);
            int K = 0;
            double mg = INFINITY;
            if (a > 0.0) {
                if (step_f == 0.0f) {
                    K = 1;
                } else {
                    double r = (log(a) - (double)lmin_f) / (double)step_f + 1.0;
                    int k0 = r < 0.0 ? 0 : (r > (double)kmax ? kmax : (int)floor(r));
                    if (k0 >= kmax) {
                        K = kmax;
                    } else {
                        double lo = logfmt_grid(lmin_f, step_f, k0), hi = logfmt_grid(lmin_f, step_f, k0 + 1);
                        double mid = 0.5 * (lo + hi);
                        K = a >= mid ? k0 + 1 : k0;
                        mg = fabs(a - mid) / (hi - lo);
                    }
                }
            }
            codes[base + j] = sgn | (uint16_t)K;
            if (margin_out) margin_out[base + j] = (float)mg;
        }
    }
}

/* Decode: K = code & (2^(n-1) - 1); value = +-exp(min + Step * (K - 1)) for K >= 1, +-0 for
 * K = 0, in double, rounded to FP32. */
void orc_logfmt_decode(int64_t rows, int64_t cols, const uint16_t* codes, int n_bits,
                       const float* lmin, const float* step, float* out)
{
    const int kmask = (1 << (n_bits - 1)) - 1;
    const int64_t tiles = cols / 128;
#pragma omp parallel for schedule(static)
    for (int64_t tt = 0; tt < rows * tiles; ++tt) {
        const int64_t base = (tt / tiles) * cols + (tt % tiles) * 128;
        for (int j = 0; j < 128; ++j) {
            uint16_t c = codes[base + j];
            double m = logfmt_grid(lmin[tt], step[tt], c & kmask);
            out[base + j] = (float)((c >> (n_bits - 1)) & 1 ? -m : m);
        }
    }
}
