/*
 * CPU oracle for the MoE layer hot path: router -> dispatch -> SwiGLU experts -> combine.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, single-threaded definition that the
 * CUDA library is checked against. Only the tests, the smoke check and the bench's CPU-baseline
 * leg load it. It shares no code, header, table or constant generator with the CUDA library.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no -ffast-math: every float
 * operation below is one IEEE-754 operation rounded to nearest even, in the order written).
 *
 * Sources (web pages, cited by title and section):
 *  [SMoE]  "7.13 Serving Mixture-of-Experts: Expert Parallelism & All-to-All Inference"
 *          (llm-stack-book), sections "Expert Parallelism Mechanics: Dispatch, Compute,
 *          Combine" (router, per-rank dispatch, grouped expert FFN, weighted combine; the
 *          single-process reference layer), "DeepEP: A Production All-to-All Kernel" (FP8 E4M3
 *          dispatch with a BF16 combine; fixed-size padded receive buffers), "Hot-Expert Skew
 *          at Decode and Load Balancing" (shared experts).
 *  [LK]    "Mixture-of-experts serving" (learn-kernels), paragraph 1 (DeepSeek-V3 layer: one
 *          shared expert plus 256 routed, 8 active, sigmoid affinity with a per-expert bias)
 *          and paragraph 3 (group-limited routing).
 *  [OS]    "One-Sided Expert-Parallel All-to-All for Mixture-of-Experts Inference over NVLink"
 *          (abstract): each source pushes into rank-major buffers on the target without a
 *          metadata exchange, and the grouped GEMMs read those buffers in place.
 *
 * Readings where the pages are silent (each restated where it is used):
 *  R-a  The gate GEMM is fp32. Its summation order is fixed so two implementations can agree
 *       bit for bit: d is cut into 16 equal chunks, each chunk is a sequential fused
 *       multiply-add chain from index 0 of the chunk, and the 16 partials are added by a
 *       balanced pairwise tree.
 *  R-b  The sigmoid is the logistic 1/(1+e^-z) with e^-z from Cody-Waite range reduction and a
 *       degree-7 Taylor polynomial (one fixed sequence of float operations).
 *  R-c  The group score is the sum of the two largest selection keys of the group; groups are
 *       contiguous blocks of E/n_group experts.
 *  R-d  Ties in any top-k (groups or experts) go to the lower index.
 *  R-e  The gate weights are the selected raw sigmoid scores divided by their sum (summed in
 *       selection order) and multiplied by the routing scale.
 *  R-f  Token t belongs to source rank t / (T/R); expert e lives on rank e / (E/R).
 *  R-g  Rank-major receive layout: destination rank r, then source rank s, a segment of
 *       cap = (T/R) * min(k, E/R) rows; inside a segment rows are grouped by local expert in
 *       ascending order, and by token index inside an expert. One row per (token, expert).
 *  R-h  Expert FFN is SwiGLU: h = silu(x Wg^T) * (x Wu^T), rounded to the GEMM input format,
 *       then o = h Wd^T rounded to bf16. The shared expert is the same on every token.
 *  R-i  FP8: per-row 1x128 blocks, scale = amax/448 (1 when amax is 0), code = e4m3 with
 *       round-to-nearest-even and saturation of value/scale; weights e4m3 with one fp32 scale
 *       per 128x128 block.
 *  R-l  FP8 with power-of-two scales (the second FP8 recipe): the same blocks as R-i, but each
 *       block's fp32 scale is the smallest power of two 2^e with amax <= 448 * 2^e, e kept in
 *       [-126, 127] (scale 1 when amax is 0), so value / scale is exact; weight block scales
 *       are powers of two as well. The pages fix e4m3 payloads with fp32 block scales, not the
 *       scale values; powers of two are the values the block-scaled tensor-core MMA applies.
 *  R-j  Combine: y = bf16(sum_i w_i * o_i + sh) with the sum taken in fp64 here.
 *  R-k  Redundant experts ([SMoE] "Hot-Expert Skew", redundant experts; exercise 5,
 *       imbalance_factor_replicated): a deployment has S expert slots on each of the R ranks
 *       (R*S >= E). The R*S - E spare slots hold extra copies, given one at a time to the expert
 *       with the largest estimated load per copy (ties: lower expert). Every copy carries an
 *       equal share of its expert's load, and copies are placed largest first onto the least
 *       loaded rank that still has a free slot (ties: lower expert, lower copy, lower rank);
 *       a rank's slots are ordered by (expert, copy). Each source rank splits its own tokens of
 *       an expert evenly over the copies: its j-th token of expert e (counted in token order)
 *       goes to copy (j + s) mod copies(e), copies numbered in slot order. The receive layout
 *       is R-g with slots in place of experts and cap = (T/R) * min(k, S).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------------
 * Number formats
 * ------------------------------------------------------------------------------------------ */
static float f32_of_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_of_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

float oracle_bf16_to_f32(uint16_t h) { return f32_of_bits((uint32_t)h << 16); }

/* Round fp32 to the nearest bf16, ties to even. */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u = bits_of_f32(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u); /* quiet NaN */
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* e4m3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field
 * 0 holds subnormals m/8 * 2^-6; S.1111.111 is NaN; there is no infinity; largest finite 448. */
float oracle_e4m3_to_f32(uint8_t q) {
    int s = q >> 7, e = (q >> 3) & 15, m = q & 7;
    float v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexpf((float)m, -9);            /* m/8 * 2^-6 */
    else v = ldexpf((float)(8 + m), e - 7 - 3);      /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* fp32 -> e4m3 code, round to nearest even, values beyond +-448 saturate to +-448. */
uint8_t oracle_f32_to_e4m3(float x) {
    if (isnan(x)) return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    float a = fabsf(x);
    if (a > 448.0f) return sign | 0x7e;              /* 1.110b * 2^8 = 448 */
    /* Spacing of the e4m3 grid around a: 2^(E-3) in binade [2^E, 2^(E+1)), E >= -6;
     * 2^-9 below the smallest normal 2^-6. */
    int E;
    if (a < ldexpf(1.0f, -6)) E = -6;
    else { int e2; frexpf(a, &e2); E = e2 - 1; }
    float q = rintf(ldexpf(a, 3 - E));              /* a / spacing, exact; then RNE */
    float v = ldexpf(q, E - 3);                     /* rounded magnitude */
    if (v == 0.0f) return sign;
    if (v < ldexpf(1.0f, -6)) return sign | (uint8_t)q;           /* subnormal: m = q */
    int e2; frexpf(v, &e2);
    int Ev = e2 - 1;                                 /* v may have moved up one binade */
    int mant = (int)(ldexpf(v, -Ev) * 8.0f) - 8;
    return sign | (uint8_t)((Ev + 7) << 3) | (uint8_t)mant;
}

/* ------------------------------------------------------------------------------------------
 * Router  [LK paragraph 1: sigmoid affinity + per-expert bias; paragraph 3: group-limited
 * routing; SMoE "Expert Parallelism Mechanics", router step: top-k then renormalise]
 * ------------------------------------------------------------------------------------------ */

/* e^z for the sigmoid (reading R-b). Cody-Waite: n = rint(z*log2 e), r = z - n*ln2 in two
 * pieces (hi has 9 significant bits so n*hi is exact for |n| < 2^15), e^r by the Taylor
 * series to degree 7 in Horner form (|r| <= ln2/2 so the remainder is below 2^-27), result
 * scaled by 2^n built from exponent bits. z is clamped to [-87, 87] so 2^n stays normal. */
float oracle_exp(float z) {
    const float LOG2E = 1.44269504088896341f;
    const float LN2_HI = 0.693359375f;
    const float LN2_LO = -2.12194440e-4f;
    if (z > 87.0f) z = 87.0f;
    if (z < -87.0f) z = -87.0f;
    float n = rintf(z * LOG2E);
    float r = fmaf(-n, LN2_HI, z);
    r = fmaf(-n, LN2_LO, r);
    float p = 1.98412698e-4f;              /* 1/7! */
    p = fmaf(p, r, 1.38888889e-3f);        /* 1/6! */
    p = fmaf(p, r, 8.33333333e-3f);        /* 1/5! */
    p = fmaf(p, r, 4.16666667e-2f);        /* 1/4! */
    p = fmaf(p, r, 1.66666667e-1f);        /* 1/3! */
    p = fmaf(p, r, 0.5f);                  /* 1/2! */
    p = fmaf(p, r, 1.0f);                  /* 1/1! */
    p = fmaf(p, r, 1.0f);                  /* 1/0! */
    float two_n = f32_of_bits((uint32_t)((int)n + 127) << 23);
    return p * two_n;
}

float oracle_sigmoid(float z) { return 1.0f / (1.0f + oracle_exp(-z)); }

/* z = x . w in fp32 with the canonical order of reading R-a. Requires d % 16 == 0. */
float oracle_logit(const uint16_t* x, const float* w, int d) {
    float part[16];
    int L = d / 16;
    for (int c = 0; c < 16; ++c) {
        float acc = 0.0f;
        for (int i = c * L; i < (c + 1) * L; ++i) acc = fmaf(oracle_bf16_to_f32(x[i]), w[i], acc);
        part[c] = acc;
    }
    for (int width = 16; width > 1; width /= 2)
        for (int j = 0; j < width / 2; ++j) part[j] = part[2 * j] + part[2 * j + 1];
    return part[0];
}

/* a ranks before b: larger key first, then lower index (reading R-d). */
static int ranks_before(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

/* Group-limited top-k on one token's scores s [E] and bias [E] (readings R-c, R-d, R-e).
 * Writes idx [k] in selection order and w [k]. */
static void select_token(int E, int k, int n_group, int topk_group, float route_scale,
                         const float* s, const float* bias, float* v, float* gscore, char* gkeep,
                         char* taken, int32_t* idx, float* w) {
    int gs = E / n_group;
    for (int e = 0; e < E; ++e) v[e] = s[e] + bias[e];     /* bias steers selection only */
    /* group score: sum of the two largest keys in the group */
    for (int g = 0; g < n_group; ++g) {
        int b1 = -1, b2 = -1;
        for (int e = g * gs; e < (g + 1) * gs; ++e) {
            if (b1 < 0 || ranks_before(v[e], e, v[b1], b1)) { b2 = b1; b1 = e; }
            else if (b2 < 0 || ranks_before(v[e], e, v[b2], b2)) b2 = e;
        }
        gscore[g] = (b2 >= 0) ? v[b1] + v[b2] : v[b1];
        gkeep[g] = 0;
    }
    for (int r = 0; r < topk_group; ++r) {
        int best = -1;
        for (int g = 0; g < n_group; ++g)
            if (!gkeep[g] && (best < 0 || ranks_before(gscore[g], g, gscore[best], best)))
                best = g;
        gkeep[best] = 1;
    }
    /* top-k experts among the kept groups */
    memset(taken, 0, E);
    float sum = 0.0f;
    for (int i = 0; i < k; ++i) {
        int best = -1;
        for (int e = 0; e < E; ++e)
            if (gkeep[e / gs] && !taken[e] && (best < 0 || ranks_before(v[e], e, v[best], best)))
                best = e;
        taken[best] = 1;
        idx[i] = best;
        sum += s[best];                     /* raw sigmoid, summed in selection order */
    }
    for (int i = 0; i < k; ++i) w[i] = (s[idx[i]] / sum) * route_scale;
}

static int route_shape_ok(int d, int E, int k, int n_group, int topk_group) {
    return !(d % 16 || n_group < 1 || E % n_group || topk_group < 1 || topk_group > n_group ||
             k < 1 || k > topk_group * (E / n_group));
}

/* Selection alone, from given sigmoid scores [T][E]. Returns 0, or -1 on a bad shape. */
int oracle_select(int T, int E, int k, int n_group, int topk_group, float route_scale,
                  const float* scores, const float* bias, int32_t* topk_idx, float* topk_w) {
    if (!route_shape_ok(16, E, k, n_group, topk_group)) return -1;
    float* v = (float*)malloc(sizeof(float) * E);
    float* gscore = (float*)malloc(sizeof(float) * n_group);
    char* gkeep = (char*)malloc(n_group);
    char* taken = (char*)malloc(E);
    for (int t = 0; t < T; ++t)
        select_token(E, k, n_group, topk_group, route_scale, scores + (size_t)t * E, bias, v,
                     gscore, gkeep, taken, topk_idx + (size_t)t * k, topk_w + (size_t)t * k);
    free(v); free(gscore); free(gkeep); free(taken);
    return 0;
}

/* Route T tokens. x bf16 [T][d]; w_gate fp32 [E][d]; bias fp32 [E].
 * Outputs topk_idx [T][k] (selection order), topk_w [T][k]; optionally logits [T][E] and
 * scores [T][E] (the sigmoid affinities). Returns 0, or -1 on a bad shape. */
int oracle_route(int T, int d, int E, int k, int n_group, int topk_group, float route_scale,
                 const uint16_t* x, const float* w_gate, const float* bias,
                 int32_t* topk_idx, float* topk_w, float* logits_out, float* scores_out) {
    if (!route_shape_ok(d, E, k, n_group, topk_group)) return -1;
    float* s = (float*)malloc(sizeof(float) * E);
    float* v = (float*)malloc(sizeof(float) * E);
    float* gscore = (float*)malloc(sizeof(float) * n_group);
    char* gkeep = (char*)malloc(n_group);
    char* taken = (char*)malloc(E);
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            float z = oracle_logit(x + (size_t)t * d, w_gate + (size_t)e * d, d);
            s[e] = oracle_sigmoid(z);
            if (logits_out) logits_out[(size_t)t * E + e] = z;
            if (scores_out) scores_out[(size_t)t * E + e] = s[e];
        }
        select_token(E, k, n_group, topk_group, route_scale, s, bias, v, gscore, gkeep, taken,
                     topk_idx + (size_t)t * k, topk_w + (size_t)t * k);
    }
    free(s); free(v); free(gscore); free(gkeep); free(taken);
    return 0;
}

/* ------------------------------------------------------------------------------------------
 * Dispatch  [SMoE "Expert Parallelism Mechanics", dispatch step: rows for the same
 * destination made contiguous, one row per (token, expert); OS abstract: push into rank-major
 * buffers on the target with no metadata exchange; SMoE "DeepEP": fixed-size padded buffers]
 * ------------------------------------------------------------------------------------------ */

/* counts [R][E]: rows source s sends to expert e. offsets [R][E]: first row of expert e inside
 * segment (rank(e), s), i.e. the exclusive sum of counts[s][e'] over experts e' < e on the same
 * rank. row_of [T][k]: receive row of (t, i). src_tok [R*R*cap] (nullable): token of each
 * receive row, -1 for rows left empty. Returns 0, or -1 on a bad shape. */
int oracle_dispatch_index(int T, int E, int k, int R, const int32_t* topk_idx,
                          int32_t* counts, int32_t* offsets, int32_t* row_of, int32_t* src_tok) {
    if (T % R || E % R) return -1;
    int Ts = T / R, Er = E / R;
    int cap = Ts * (k < Er ? k : Er);
    memset(counts, 0, sizeof(int32_t) * R * E);
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < k; ++i) counts[(t / Ts) * E + topk_idx[(size_t)t * k + i]] += 1;
    for (int s = 0; s < R; ++s)
        for (int e = 0; e < E; ++e) {
            int acc = 0;
            for (int e2 = (e / Er) * Er; e2 < e; ++e2) acc += counts[s * E + e2];
            offsets[s * E + e] = acc;
        }
    if (src_tok)
        for (long r = 0; r < (long)R * R * cap; ++r) src_tok[r] = -1;
    int32_t* run = (int32_t*)calloc((size_t)R * E, sizeof(int32_t));
    for (int t = 0; t < T; ++t) {               /* tokens in ascending order: stable */
        int s = t / Ts;
        for (int i = 0; i < k; ++i) {
            int e = topk_idx[(size_t)t * k + i];
            int r = e / Er;
            int row = (r * R + s) * cap + offsets[s * E + e] + run[s * E + e]++;
            row_of[(size_t)t * k + i] = row;
            if (src_tok) src_tok[row] = t;
        }
    }
    free(run);
    return 0;
}

/* Reading R-l: the smallest power of two 2^e, -126 <= e <= 127, with amax <= 448 * 2^e (1 when
 * amax is 0). Found by stepping e, every comparison exact in double. */
float oracle_pow2_scale(float amax) {
    if (!(amax > 0.0f)) return 1.0f;
    int e = 0;
    while (e < 127 && ldexp(448.0, e) < (double)amax) ++e;
    while (e > -126 && ldexp(448.0, e - 1) >= (double)amax) --e;
    return (float)ldexp(1.0, e);
}

/* 1x128 block quantisation of one row of n floats (n % 128 == 0): amax per block, scale =
 * amax / 448 (reading R-i; 1 if amax == 0) or its power of two (reading R-l, pow2 != 0),
 * code = e4m3(value / scale). */
void oracle_quant_row_e4m3_ex(const float* v, int n, uint8_t* q, float* scales, int pow2) {
    for (int b = 0; b < n / 128; ++b) {
        float amax = 0.0f;
        for (int c = b * 128; c < (b + 1) * 128; ++c) if (fabsf(v[c]) > amax) amax = fabsf(v[c]);
        float scale = pow2 ? oracle_pow2_scale(amax) : (amax > 0.0f ? amax / 448.0f : 1.0f);
        scales[b] = scale;
        for (int c = b * 128; c < (b + 1) * 128; ++c) q[c] = oracle_f32_to_e4m3(v[c] / scale);
    }
}

void oracle_quant_row_e4m3(const float* v, int n, uint8_t* q, float* scales) {
    oracle_quant_row_e4m3_ex(v, n, q, scales, 0);
}

/* Copy payload rows. bf16 mode: recv[row] = x[t]. fp8 mode (recv_scales != NULL): recv holds
 * e4m3 codes of x[t] and recv_scales[row][d/128] its block scales; a token is quantised once
 * and its codes written to each of its k rows. Unfilled rows are left untouched. */
void oracle_dispatch_payload_ex(int T, int d, int k, const uint16_t* x, const int32_t* row_of,
                                void* recv, float* recv_scales, int pow2) {
    float* xf = (float*)malloc(sizeof(float) * d);
    uint8_t* q = (uint8_t*)malloc(d);
    float* sc = (float*)malloc(sizeof(float) * (d / 128 + 1));
    for (int t = 0; t < T; ++t) {
        if (recv_scales) {
            for (int c = 0; c < d; ++c) xf[c] = oracle_bf16_to_f32(x[(size_t)t * d + c]);
            oracle_quant_row_e4m3_ex(xf, d, q, sc, pow2);
        }
        for (int i = 0; i < k; ++i) {
            long row = row_of[(size_t)t * k + i];
            if (recv_scales) {
                memcpy((uint8_t*)recv + row * d, q, d);
                memcpy(recv_scales + row * (d / 128), sc, sizeof(float) * (d / 128));
            } else {
                memcpy((uint16_t*)recv + row * d, x + (size_t)t * d, sizeof(uint16_t) * d);
            }
        }
    }
    free(xf); free(q); free(sc);
}

void oracle_dispatch_payload(int T, int d, int k, const uint16_t* x, const int32_t* row_of,
                             void* recv, float* recv_scales) {
    oracle_dispatch_payload_ex(T, d, k, x, row_of, recv, recv_scales, 0);
}

/* ------------------------------------------------------------------------------------------
 * Expert FFN  [SMoE "Expert Parallelism Mechanics": per-expert up-projection, activation,
 * down-projection on the rows that expert received; LK paragraph 1 and SMoE "Hot-Expert Skew":
 * the shared expert runs on every token. SwiGLU form per reading R-h.]
 * ------------------------------------------------------------------------------------------ */
static double silu(double g) { return g / (1.0 + exp(-g)); }

/* One input row through one bf16 SwiGLU expert. w13 [2F][d] (rows 0..F-1 gate, F..2F-1 up),
 * w2 [d][F]. out: bf16 [d]. h_out (nullable): the bf16-rounded intermediate, as floats [F].
 * out_exact (nullable): the down projection's fp64 sums before their rounding to bf16 [d]. */
void oracle_swiglu_row_bf16(int d, int F, const uint16_t* x, const uint16_t* w13,
                            const uint16_t* w2, uint16_t* out, float* h_out, double* out_exact) {
    double* xv = (double*)malloc(sizeof(double) * d);
    double* h = (double*)malloc(sizeof(double) * F);
    for (int c = 0; c < d; ++c) xv[c] = oracle_bf16_to_f32(x[c]);
    for (int f = 0; f < F; ++f) {
        double g = 0.0, u = 0.0;
        const uint16_t* wg = w13 + (size_t)f * d;
        const uint16_t* wu = w13 + (size_t)(F + f) * d;
        for (int c = 0; c < d; ++c) {
            g += xv[c] * oracle_bf16_to_f32(wg[c]);
            u += xv[c] * oracle_bf16_to_f32(wu[c]);
        }
        h[f] = oracle_bf16_to_f32(oracle_f32_to_bf16((float)(silu(g) * u)));
        if (h_out) h_out[f] = (float)h[f];
    }
    for (int c = 0; c < d; ++c) {
        double o = 0.0;
        const uint16_t* wd = w2 + (size_t)c * F;
        for (int f = 0; f < F; ++f) o += h[f] * oracle_bf16_to_f32(wd[f]);
        out[c] = oracle_f32_to_bf16((float)o);
        if (out_exact) out_exact[c] = o;
    }
    free(xv); free(h);
}

/* One row through one e4m3 SwiGLU expert. xq [d] codes with xs [d/128] scales; w13q [2F][d]
 * with w13s [2F/128][d/128]; w2q [d][F] with w2s [d/128][F/128]. h is re-quantised 1x128 before
 * the down projection (reading R-i, or R-l when pow2 != 0). out: bf16 [d]. h_out (nullable): dequantised h [F].
 * out_exact (nullable): the down projection's fp64 sums before their rounding to bf16 [d]. */
void oracle_swiglu_row_fp8_ex(int d, int F, const uint8_t* xq, const float* xs,
                              const uint8_t* w13q, const float* w13s, const uint8_t* w2q,
                              const float* w2s, uint16_t* out, float* h_out, double* out_exact,
                              int pow2) {
    int db = d / 128, fb = F / 128;
    double* xv = (double*)malloc(sizeof(double) * d);
    float* hf = (float*)calloc((size_t)F, sizeof(float));
    uint8_t* hq = (uint8_t*)malloc(F);
    float* hs = (float*)malloc(sizeof(float) * fb);
    for (int c = 0; c < d; ++c) xv[c] = (double)oracle_e4m3_to_f32(xq[c]) * xs[c / 128];
    for (int f = 0; f < F; ++f) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < d; ++c) {
            double wg = (double)oracle_e4m3_to_f32(w13q[(size_t)f * d + c]) * w13s[(f / 128) * db + c / 128];
            double wu = (double)oracle_e4m3_to_f32(w13q[(size_t)(F + f) * d + c]) *
                        w13s[((F + f) / 128) * db + c / 128];
            g += xv[c] * wg;
            u += xv[c] * wu;
        }
        hf[f] = (float)(silu(g) * u);
    }
    oracle_quant_row_e4m3_ex(hf, F, hq, hs, pow2);
    for (int f = 0; f < F; ++f) {
        hf[f] = oracle_e4m3_to_f32(hq[f]) * hs[f / 128];
        if (h_out) h_out[f] = hf[f];
    }
    for (int c = 0; c < d; ++c) {
        double o = 0.0;
        for (int f = 0; f < F; ++f)
            o += (double)hf[f] * ((double)oracle_e4m3_to_f32(w2q[(size_t)c * F + f]) * w2s[(c / 128) * fb + f / 128]);
        out[c] = oracle_f32_to_bf16((float)o);
        if (out_exact) out_exact[c] = o;
    }
    free(xv); free(hf); free(hq); free(hs);
}

void oracle_swiglu_row_fp8(int d, int F, const uint8_t* xq, const float* xs,
                           const uint8_t* w13q, const float* w13s, const uint8_t* w2q,
                           const float* w2s, uint16_t* out, float* h_out, double* out_exact) {
    oracle_swiglu_row_fp8_ex(d, F, xq, xs, w13q, w13s, w2q, w2s, out, h_out, out_exact, 0);
}

/* ------------------------------------------------------------------------------------------
 * Combine  [SMoE "Expert Parallelism Mechanics", combine step: the k expert outputs of a token
 * weighted-summed by its gate weights; SMoE "DeepEP": the combine stays in BF16]
 * ------------------------------------------------------------------------------------------ */

/* y[t] = bf16( sum_i topk_w[t][i] * ebuf[row_of[t][i]] + shared[t] ), sum in fp64.
 * ebuf bf16 [*][d] indexed by receive row; shared bf16 [T][d] or NULL. y_exact (nullable): the
 * fp64 sums before their rounding to bf16 [T][d]. */
void oracle_combine(int T, int d, int k, const uint16_t* ebuf, const int32_t* row_of,
                    const float* topk_w, const uint16_t* shared, uint16_t* y, double* y_exact) {
    for (int t = 0; t < T; ++t)
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int i = 0; i < k; ++i) {
                long row = row_of[(size_t)t * k + i];
                acc += (double)topk_w[(size_t)t * k + i] * oracle_bf16_to_f32(ebuf[row * d + c]);
            }
            if (shared) acc += oracle_bf16_to_f32(shared[(size_t)t * d + c]);
            y[(size_t)t * d + c] = oracle_f32_to_bf16((float)acc);
            if (y_exact) y_exact[(size_t)t * d + c] = acc;
        }
}

/* ------------------------------------------------------------------------------------------
 * Redundant experts and their placement  [SMoE "Hot-Expert Skew": replicate the busiest
 * experts on under-loaded GPUs and let the dispatch split their tokens over the replicas;
 * exercise 5: each copy takes an equal share of its expert's load and copies are assigned,
 * largest first, to the least-loaded rank (LPT). Reading R-k.]
 * ------------------------------------------------------------------------------------------ */

/* load [E] (estimated rows per expert), R ranks of S slots. Outputs: slot_expert [R*S] (expert
 * held by each slot), n_copies [E], copy_slot [E][max_copies] (slot of each copy, ascending;
 * unused entries -1). Returns 0, or -1 when R*S < E or some expert would need more than
 * max_copies copies. */
int oracle_place_experts(int E, int R, int S, const double* load, int max_copies,
                         int32_t* slot_expert, int32_t* n_copies, int32_t* copy_slot) {
    int P = R * S;
    if (P < E || max_copies < 1) return -1;
    for (int e = 0; e < E; ++e) n_copies[e] = 1;
    /* the spare slots: one more copy at a time to the largest load per copy */
    for (int extra = 0; extra < P - E; ++extra) {
        int best = 0;
        for (int e = 1; e < E; ++e)
            if (load[e] / n_copies[e] > load[best] / n_copies[best]) best = e;
        n_copies[best] += 1;
        if (n_copies[best] > max_copies) return -1;
    }
    /* the copies, largest share first (ties: lower expert, lower copy) */
    int* ce = (int*)malloc(sizeof(int) * P);
    int* cc = (int*)malloc(sizeof(int) * P);
    double* cl = (double*)malloc(sizeof(double) * P);
    int n = 0;
    for (int e = 0; e < E; ++e)
        for (int c = 0; c < n_copies[e]; ++c) {
            ce[n] = e; cc[n] = c; cl[n] = load[e] / n_copies[e]; ++n;
        }
    for (int a = 1; a < n; ++a) {               /* insertion sort: plain and stable */
        int e = ce[a], c = cc[a];
        double l = cl[a];
        int b = a - 1;
        while (b >= 0 && cl[b] < l) { ce[b + 1] = ce[b]; cc[b + 1] = cc[b]; cl[b + 1] = cl[b]; --b; }
        ce[b + 1] = e; cc[b + 1] = c; cl[b + 1] = l;
    }
    /* LPT onto ranks with a free slot */
    double* rank_load = (double*)calloc((size_t)R, sizeof(double));
    int* rank_used = (int*)calloc((size_t)R, sizeof(int));
    int* copy_rank = (int*)malloc(sizeof(int) * P);   /* rank of copy index (e, c), by list pos */
    for (int a = 0; a < n; ++a) {
        int r_best = -1;
        for (int r = 0; r < R; ++r)
            if (rank_used[r] < S && (r_best < 0 || rank_load[r] < rank_load[r_best])) r_best = r;
        copy_rank[a] = r_best;
        rank_load[r_best] += cl[a];
        rank_used[r_best] += 1;
    }
    /* slots of each rank in (expert, copy) order */
    for (int i = 0; i < E * max_copies; ++i) copy_slot[i] = -1;
    for (int r = 0; r < R; ++r) {
        int j = 0;
        for (int e = 0; e < E; ++e)
            for (int c = 0; c < n_copies[e]; ++c)
                for (int a = 0; a < n; ++a)
                    if (ce[a] == e && cc[a] == c && copy_rank[a] == r) {
                        slot_expert[r * S + j] = e;
                        ++j;
                    }
    }
    /* copies of each expert numbered in slot order */
    for (int e = 0; e < E; ++e) {
        int c = 0;
        for (int p = 0; p < P; ++p)
            if (slot_expert[p] == e) copy_slot[e * max_copies + c++] = p;
    }
    free(ce); free(cc); free(cl); free(rank_load); free(rank_used); free(copy_rank);
    return 0;
}

/* The dispatch index of R-g over the slots of a placement (R-k): counts [R][P] (rows source s
 * sends to slot p), row_of [T][k], src_tok [R*R*cap] (nullable), cap = (T/R) * min(k, S),
 * P = R*S. Returns 0, or -1 on a bad shape. */
int oracle_dispatch_index_placed(int T, int E, int k, int R, int S, const int32_t* topk_idx,
                                 const int32_t* n_copies, const int32_t* copy_slot,
                                 int max_copies, int32_t* counts, int32_t* row_of,
                                 int32_t* src_tok) {
    if (T % R || R * S < E) return -1;
    int Ts = T / R, P = R * S;
    int cap = Ts * (k < S ? k : S);
    int32_t* seen = (int32_t*)calloc((size_t)R * E, sizeof(int32_t));   /* j per (s, e) */
    int32_t* slot_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
    memset(counts, 0, sizeof(int32_t) * (size_t)R * P);
    for (int t = 0; t < T; ++t) {               /* tokens in ascending order */
        int s = t / Ts;
        for (int i = 0; i < k; ++i) {
            int e = topk_idx[(size_t)t * k + i];
            int j = seen[s * E + e]++;
            int c = (j + s) % n_copies[e];
            int p = copy_slot[e * max_copies + c];
            slot_of[(size_t)t * k + i] = p;
            counts[(size_t)s * P + p] += 1;
        }
    }
    if (src_tok)
        for (long r = 0; r < (long)R * R * cap; ++r) src_tok[r] = -1;
    int32_t* run = (int32_t*)calloc((size_t)R * P, sizeof(int32_t));
    for (int t = 0; t < T; ++t) {
        int s = t / Ts;
        for (int i = 0; i < k; ++i) {
            int p = slot_of[(size_t)t * k + i];
            int r = p / S;
            int off = 0;                        /* rows of earlier slots of rank r from s */
            for (int q = r * S; q < p; ++q) off += counts[(size_t)s * P + q];
            int row = (r * R + s) * cap + off + run[(size_t)s * P + p]++;
            row_of[(size_t)t * k + i] = row;
            if (src_tok) src_tok[row] = t;
        }
    }
    free(seen); free(slot_of); free(run);
    return 0;
}

/* ------------------------------------------------------------------------------------------
 * Array forms of the scalar helpers (for the tests)
 * ------------------------------------------------------------------------------------------ */
void oracle_exp_array(long n, const float* z, float* out) {
    for (long i = 0; i < n; ++i) out[i] = oracle_exp(z[i]);
}
void oracle_sigmoid_array(long n, const float* z, float* out) {
    for (long i = 0; i < n; ++i) out[i] = oracle_sigmoid(z[i]);
}
void oracle_f32_to_e4m3_array(long n, const float* v, uint8_t* q) {
    for (long i = 0; i < n; ++i) q[i] = oracle_f32_to_e4m3(v[i]);
}
void oracle_e4m3_to_f32_array(long n, const uint8_t* q, float* v) {
    for (long i = 0; i < n; ++i) v[i] = oracle_e4m3_to_f32(q[i]);
}
void oracle_f32_to_bf16_array(long n, const float* v, uint16_t* h) {
    for (long i = 0; i < n; ++i) h[i] = oracle_f32_to_bf16(v[i]);
}
