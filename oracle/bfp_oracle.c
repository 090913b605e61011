/*
 * ORACLE — test infrastructure only.
 *
 * A plain, slow, single-threaded CPU statement of what the BFP MoE decode
 * path computes. Only the tests, the smoke check and the benchmark's CPU
 * baseline leg may call it; the library never does, and it shares no code,
 * header or table with the library or its kernels.
 *
 * Sources (all on the block_floating_point pages; "P1" = the Qwen3.6-35B-A3B
 * TT-Mixed-BFP4-BFP8-P150 model card, "P3" = the qwen3.6-a3b-blackhole tt-kernel
 * bundle page, "P4"/"P5" = the two Qwen3.8-27B TT-Mixed-BFP4-BFP8-P150 cards):
 *   - blocks of 16 values (P5, "What changed in this release", GPTQ bullet);
 *   - round-to-nearest conversion (P1, "What is in this release" and
 *     "Verification/Checkpoint"; P5, GPTQ bullet);
 *   - one shared exponent byte per 16 values: BFP8 costs 8.5 bits per value
 *     (P3, QWEN36_KV_DTYPE row: 20.0 -> 10.6 KiB/token) and BFP4 4.5 bits per
 *     value (P4, "Changes in s27", bfp8_v4r: 26,624 instead of 34,816 B/token);
 *   - experts BFP4, dense projections and LM head BFP8, router bf16
 *     (P1, "Precision as served");
 *   - 256 experts, top-8 plus a shared expert (P3, opening paragraph).
 * The pages leave the bit-level rules open. This file takes these readings:
 *   exponent  = the fp32 biased exponent (8 bits, bias 127) of the block's
 *               largest-exponent element; 0 for an all-zero block;
 *   mantissa  = sign-magnitude, magnitude of mb bits (mb = 3 for BFP4, 7 for
 *               BFP8) with the leading bit explicit, value = m * 2^(E-127-(mb-1));
 *   rounding  = to nearest, ties to even, on the dropped bits;
 *   overflow  = a magnitude that rounds up to 2^mb saturates to 2^mb - 1
 *               (the block exponent is kept);
 *   zero, -0 and fp32 subnormal inputs encode as +0; NaN/Inf are rejected.
 *
 * Floating point is fp64 throughout, except where the decode step itself
 * fixes fp32: router logits are rounded to fp32 before selection (top-k is
 * taken on the fp32 logits, ties to the lower index), and outputs are fp32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENONFINITE -4

static int mant_bits(int fmt) { return fmt == 4 ? 3 : (fmt == 8 ? 7 : -1); }

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bf16 bit pattern -> its exact value. */
static double bf16_value(uint16_t b) { return (double)bits_f32((uint32_t)b << 16); }

/* fp32 -> bf16, round to nearest, ties to even (NaN stays NaN). */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u = f32_bits(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* Round sig / 2^s to the nearest integer, ties to even. */
static uint32_t rne_shift(uint32_t sig, int s) {
    if (s <= 0) return sig << (-s);
    if (s >= 32) return 0; /* sig < 2^24 <= 2^(s-1): below one half */
    uint32_t q = sig >> s;
    uint32_t r = sig & ((1u << s) - 1u);
    uint32_t half = 1u << (s - 1);
    if (r > half || (r == half && (q & 1u))) q += 1;
    return q;
}

/*
 * Encode one row-major fp32 matrix [n x k] (k % 16 == 0) into logical BFP
 * fields: exps[n][k/16] (u8 shared exponents) and codes[n][k] (one code per
 * value, sign << mb | magnitude, in the low bits of a byte).
 */
int oracle_encode(int fmt, const float *w, int64_t n, int64_t k, uint8_t *exps, uint8_t *codes) {
    int mb = mant_bits(fmt);
    if (mb < 0 || n < 0 || k < 0 || (k % 16) != 0) return ORACLE_EINVAL;
    const uint32_t mmax = (1u << mb) - 1u;
    int64_t kb = k / 16;
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t b = 0; b < kb; ++b) {
            const float *v = w + r * k + b * 16;
            int e[16];
            int E = 0;
            /* 1-2: per-value biased exponent; zero/subnormal count as value 0; E = max. */
            for (int i = 0; i < 16; ++i) {
                uint32_t u = f32_bits(v[i]);
                int ei = (int)((u >> 23) & 0xFF);
                if (ei == 0xFF) return ORACLE_ENONFINITE;
                e[i] = ei;
                if (ei > E) E = ei;
            }
            exps[r * kb + b] = (uint8_t)E;
            /* 3-6: magnitude = RNE(sig / 2^(24 - mb + E - e)), saturate, attach sign. */
            for (int i = 0; i < 16; ++i) {
                uint32_t u = f32_bits(v[i]);
                uint32_t m = 0;
                if (e[i] != 0) {
                    uint32_t sig = (u & 0x007FFFFFu) | 0x00800000u;
                    int s = 24 - mb + (E - e[i]);
                    m = rne_shift(sig, s);
                    if (m > mmax) m = mmax;
                }
                uint32_t sign = (m != 0) ? (u >> 31) : 0u;
                codes[r * k + b * 16 + i] = (uint8_t)((sign << mb) | m);
            }
        }
    }
    return ORACLE_OK;
}

/* Value of one code under block exponent E: (-1)^s * m * 2^(E - 127 - (mb - 1)), exact in fp64. */
static double code_value(int mb, uint8_t E, uint8_t code) {
    uint32_t m = code & ((1u << mb) - 1u);
    int s = (code >> mb) & 1;
    if (m == 0) return 0.0;
    double v = ldexp((double)m, (int)E - 127 - (mb - 1));
    return s ? -v : v;
}

/* Decode logical fields back to fp32 [n x k] (every decoded value is exact in fp32). */
int oracle_decode(int fmt, const uint8_t *exps, const uint8_t *codes, int64_t n, int64_t k, float *out) {
    int mb = mant_bits(fmt);
    if (mb < 0 || (k % 16) != 0) return ORACLE_EINVAL;
    int64_t kb = k / 16;
    for (int64_t r = 0; r < n; ++r)
        for (int64_t j = 0; j < k; ++j)
            out[r * k + j] = (float)code_value(mb, exps[r * kb + j / 16], codes[r * k + j]);
    return ORACLE_OK;
}

/*
 * Dense BFP linear: y[m][n] = sum_k x[m][k] * W[n][k], fp64 accumulation of
 * exact products, rounded once to fp32; y_bf16 (optional) = RNE of that fp32.
 */
int oracle_linear(int fmt, const uint8_t *exps, const uint8_t *codes, int64_t n, int64_t k,
                  const uint16_t *x, int m, float *y, uint16_t *y_bf16) {
    int mb = mant_bits(fmt);
    if (mb < 0 || (k % 16) != 0 || m < 0) return ORACLE_EINVAL;
    int64_t kb = k / 16;
    for (int r = 0; r < m; ++r) {
        for (int64_t o = 0; o < n; ++o) {
            double acc = 0.0;
            for (int64_t j = 0; j < k; ++j)
                acc += bf16_value(x[(int64_t)r * k + j]) * code_value(mb, exps[o * kb + j / 16], codes[o * k + j]);
            float f = (float)acc;
            y[(int64_t)r * n + o] = f;
            if (y_bf16) y_bf16[(int64_t)r * n + o] = f32_to_bf16_rne(f);
        }
    }
    return ORACLE_OK;
}

/*
 * Router logits: logits[r][e] = fp32( sum_h Wr[e][h] * x[r][h] ) (+ bias[e]),
 * bf16 operands, exact products summed in fp64 and rounded to fp32 once; the
 * bias (optional, fp32) is added in fp32 after that rounding.
 */
int oracle_router_logits(const uint16_t *wr, int n_experts, int hidden, const uint16_t *x, int m,
                         const float *bias, float *logits) {
    for (int r = 0; r < m; ++r) {
        for (int e = 0; e < n_experts; ++e) {
            double acc = 0.0;
            for (int h = 0; h < hidden; ++h)
                acc += bf16_value(wr[(int64_t)e * hidden + h]) * bf16_value(x[(int64_t)r * hidden + h]);
            float l = (float)acc;
            if (bias) l = l + bias[e];
            logits[(int64_t)r * n_experts + e] = l;
        }
    }
    return ORACLE_OK;
}

/*
 * Routing of one row: softmax over all experts (fp64, from the fp32 logits,
 * as exp(l - max) / sum), top-k by descending fp32 logit with ties to the
 * lower index, then the selected probabilities renormalised to sum to 1.
 * idx[k] and w[k] come back in slot order (descending logit).
 */
int oracle_route_row(const float *logits, int n_experts, int k, int32_t *idx, double *w) {
    if (k < 1 || k > n_experts) return ORACLE_EINVAL;
    double mx = -INFINITY;
    for (int e = 0; e < n_experts; ++e) if ((double)logits[e] > mx) mx = logits[e];
    double den = 0.0;
    for (int e = 0; e < n_experts; ++e) den += exp((double)logits[e] - mx);
    unsigned char *taken = (unsigned char *)calloc((size_t)n_experts, 1);
    if (!taken) return ORACLE_EINVAL;
    double sel_sum = 0.0;
    for (int s = 0; s < k; ++s) {
        int best = -1;
        for (int e = 0; e < n_experts; ++e) {
            if (taken[e]) continue;
            if (best < 0 || logits[e] > logits[best]) best = e; /* strict: ties keep the lower index */
        }
        taken[best] = 1;
        idx[s] = best;
        w[s] = exp((double)logits[best] - mx) / den;
        sel_sum += w[s];
    }
    for (int s = 0; s < k; ++s) w[s] /= sel_sum;
    free(taken);
    return ORACLE_OK;
}

/*
 * Greedy next token of one row of fp32 logits (the step after the LM head in
 * greedy decoding; Qwen3.6-35B-A3B card, "Fused decode kernels": the greedy
 * argmax over the logits for up to 16 rows): the index of the largest value,
 * ties to the lower index, compared as fp32 numbers (-0 equals +0). NaN is
 * never chosen; a row of NaN alone gives 0.
 */
int64_t oracle_greedy_row(const float *logits, int64_t n) {
    int64_t best = -1;
    for (int64_t i = 0; i < n; ++i) {
        if (isnan(logits[i])) continue;
        if (best < 0 || logits[i] > logits[best]) best = i; /* strict: ties keep the lower index */
    }
    return best < 0 ? 0 : best;
}

static double sigmoid(double a) { return 1.0 / (1.0 + exp(-a)); }

/*
 * One expert's SwiGLU FFN on one bf16 row, all in fp64 with the decoded BFP
 * weights:  o = D (silu(G x) * (U x)),  silu(a) = a * sigmoid(a).
 * G, U: [ffn x hidden]; D: [hidden x ffn]; each given as logical (exps, codes).
 */
int oracle_expert_ffn(int fmt, int hidden, int ffn,
                      const uint8_t *g_exps, const uint8_t *g_codes,
                      const uint8_t *u_exps, const uint8_t *u_codes,
                      const uint8_t *d_exps, const uint8_t *d_codes,
                      const uint16_t *x, double *o) {
    int mb = mant_bits(fmt);
    if (mb < 0 || hidden % 16 || ffn % 16) return ORACLE_EINVAL;
    double *h = (double *)malloc(sizeof(double) * (size_t)ffn);
    if (!h) return ORACLE_EINVAL;
    int hb = hidden / 16, fb = ffn / 16;
    for (int f = 0; f < ffn; ++f) {
        double a = 0.0, b = 0.0;
        for (int j = 0; j < hidden; ++j) {
            double xv = bf16_value(x[j]);
            a += code_value(mb, g_exps[(int64_t)f * hb + j / 16], g_codes[(int64_t)f * hidden + j]) * xv;
            b += code_value(mb, u_exps[(int64_t)f * hb + j / 16], u_codes[(int64_t)f * hidden + j]) * xv;
        }
        h[f] = a * sigmoid(a) * b;
    }
    for (int i = 0; i < hidden; ++i) {
        double acc = 0.0;
        for (int f = 0; f < ffn; ++f)
            acc += code_value(mb, d_exps[(int64_t)i * fb + f / 16], d_codes[(int64_t)i * ffn + f]) * h[f];
        o[i] = acc;
    }
    free(h);
    return ORACLE_OK;
}

/* Shared-expert gate of one row: sigmoid(g . x), bf16 operands, fp64. */
double oracle_shared_gate(const uint16_t *g, const uint16_t *x, int hidden) {
    double acc = 0.0;
    for (int h = 0; h < hidden; ++h) acc += bf16_value(g[h]) * bf16_value(x[h]);
    return sigmoid(acc);
}

/*
 * RMSNorm with unit weight, then bf16: out = bf16( h / sqrt(mean(h^2) + eps) ),
 * the normalisation taken in fp32 (the decode step's precision for norms).
 */
int oracle_rmsnorm_bf16(const uint16_t *h, int m, int hidden, float eps, uint16_t *out) {
    for (int r = 0; r < m; ++r) {
        double ss = 0.0;
        for (int j = 0; j < hidden; ++j) { double v = bf16_value(h[(int64_t)r * hidden + j]); ss += v * v; }
        float mean = (float)(ss / hidden);
        float inv = 1.0f / sqrtf(mean + eps);
        for (int j = 0; j < hidden; ++j) {
            float v = (float)bf16_value(h[(int64_t)r * hidden + j]);
            out[(int64_t)r * hidden + j] = f32_to_bf16_rne(v * inv);
        }
    }
    return ORACLE_OK;
}

/* Residual update of the stack: h <- bf16(h + y), fp32 add of the bf16 value and the fp32 layer output. */
int oracle_residual_bf16(uint16_t *h, const float *y, int64_t count) {
    for (int64_t i = 0; i < count; ++i) h[i] = f32_to_bf16_rne((float)bf16_value(h[i]) + y[i]);
    return ORACLE_OK;
}
