/*
 * ORACLE -- test infrastructure, not part of the product.
 *
 * A plain, slow, single-threaded C definition of the routed MoE FFN layer,
 * used only by the test suite, by the package's smoke check and by the CPU
 * baseline leg of the benchmark.  It shares no code with the CUDA library and
 * includes none of its headers.
 *
 * What the layer is, and where it is stated:
 *  - thewafflehaus/butter PR #69, commit "feat(laguna): Laguna-S-2.1 decode on
 *    the CUDA engine": each token's MoE layer picks ten experts from sigmoid
 *    router scores shifted by a correction bias, and adds a shared expert;
 *    expert weights are 4-bit, re-quantised when the model is loaded; the
 *    gate and up projections run fused (SwiGLU).
 *  - same page, commit "feat(laguna): batched prefill with tensor-core
 *    projections, fused MoE, CTA scheduling": in prefill the experts run as a
 *    grouped GEMM over descriptors built on the device (per-expert counts,
 *    offsets and a token order), with gate and up stacked per expert and the
 *    shared expert also in W4A16.
 *  - thewafflehaus/FFAI PR #72, Nemotron W4A16 Marlin MoE commit: offsets in
 *    CSR form (one per expert plus one), a router-sorted token index, and a
 *    deterministic scatter-add of the expert outputs.
 *  - the layer statement accompanying the pages fixes the rest: the bias is
 *    used for selection only; combine weights are the selected sigmoid scores
 *    normalised to sum 1; int4 symmetric per group along K with
 *    scale = absmax/7 stored as fp16 and q = clamp(round(w/s), -8, 7), two
 *    nibbles per byte; activations bf16, fp32 accumulation, bf16 output.
 *
 * Readings taken where the statement is open (each is listed with its reason
 * in the design notes):
 *  R1 dequantised weight w^ = q * s exactly (fp32 holds it exactly: 4 x 11
 *     significant bits); no intermediate rounding of w^.
 *  R2 round(.) is round-half-to-even (rint); s is absmax/7 in fp32, then
 *     rounded to fp16; an all-zero group has s = 0 and q = 0.
 *  R3 nibble order: byte j of a row holds element 2j in bits 0-3 and element
 *     2j+1 in bits 4-7, each as 4-bit two's complement.
 *  R4 SwiGLU: h = silu(gate) * up with gate rows 0..F-1 and up rows F..2F-1 of
 *     the fused gate+up matrix; silu(z) = z / (1 + e^-z).
 *  R5 rounding points: x (bf16 input), h (bf16), out (bf16).  Router logits
 *     and scores in fp64; expert dot products accumulate in fp32 in ascending
 *     index order; the combine accumulates in fp32 in the order
 *     j = 0..k-1 then the shared expert.
 *  R6 selection: the k largest s + b, ties to the lower expert id, listed in
 *     descending order; combine weights w_j = s_j / sum_j s_j.
 *  R7 shared expert: weight 1, no gate.
 *  R8 descriptors: perm lists slot ids t*k + j sorted by (expert, token);
 *     pos is its inverse; sched orders experts by count, largest first, ties
 *     to the lower id.
 *  R15 GGUF-style Q4 block: 32 weights share one fp16 scale d (2 bytes,
 *      little-endian) followed by 16 bytes of 4-bit codes n, weight i in bits
 *      0-3 of byte i and weight i + 16 in bits 4-7; the weight is (n - 8) * d.
 *      The import keeps the weights exact where the canonical format can:
 *      with a group of at most 32 every group lies inside one block, so
 *      s = d (its fp16 bits) and q = n - 8, which is already in [-8, 7].  A
 *      group of 64 or 128 spans blocks with different scales: those rows are
 *      decoded exactly (fp32 holds every (n - 8) * d) and packed with R1-R3.
 *  R16 W8A8 variant (thewafflehaus/FFAI PR #72, Nemotron-H section: W8A8
 *      grouped MoE, fp8 activations x fp8 weights; the scale recipe of the
 *      same pages' FP8 projection commit: one weight scale per output
 *      channel, one activation scale per token row, both folded in after the
 *      GEMM).  fp8 is E4M3 without infinities: 1 sign, 4 exponent bits (bias
 *      7), 3 fraction bits, subnormals down to 2^-9, largest finite 448;
 *      values round to nearest, ties to even, and saturate to +-448.  A
 *      weight row w gets s_w = absmax / 448 and q = e4m3(w / s_w); an
 *      activation row x (the token's bf16 x for gate+up, the bf16 H row for
 *      down) gets a = absmax / 448 and x_q = e4m3(x / a); both divisions in
 *      fp32; an all-zero row has scale 0 and codes 0.  A projection is
 *      v = (acc * a) * s_w, acc = sum_k q_k * x_q,k in fp32 in ascending k
 *      (every product exact).  SwiGLU, rounding points, combine and shared
 *      expert as R4-R7 (the shared expert is W8A8 too).
 *  R14 residual add (thewafflehaus/FFAI PR #72, Nemotron commit "ffai_add3":
 *      residual + routed + shared in one launch, routed and shared summed
 *      first): with a residual row r (bf16), out = bf16(float(r) + acc), where
 *      acc is the fp32 routed + shared sum of R5, rounded once.
 */
#include "moe_oracle.h"

#include <math.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Number formats (IEEE 754 binary16 and bfloat16), from their definitions. */

typedef struct {
    int p;        /* significant bits, including the implicit one */
    int emin;     /* exponent of the smallest normal */
    int emax;     /* exponent of the largest finite binade */
    int bias;
} orc_fmt;

static const orc_fmt FMT_F16 = {11, -14, 15, 15};
static const orc_fmt FMT_BF16 = {8, -126, 127, 127};

/* Round a >= 0 (finite) to the nearest value of format f, ties to even.
   Returns +INFINITY on overflow. */
static double round_to_fmt(double a, orc_fmt f) {
    if (a == 0.0) return 0.0;
    int ex;
    frexp(a, &ex);
    int e = ex - 1; /* a in [2^e, 2^(e+1)) */
    if (e < f.emin) e = f.emin;
    double quantum = ldexp(1.0, e - (f.p - 1));
    double r = rint(a / quantum) * quantum;
    double maxfin = ldexp(2.0 - ldexp(1.0, 1 - f.p), f.emax);
    if (r > maxfin) return INFINITY;
    return r;
}

static uint16_t encode_fmt(double v, int neg, orc_fmt f) {
    int fbits = f.p - 1;
    uint16_t sign = neg ? (uint16_t)0x8000 : 0;
    if (isnan(v)) return (uint16_t)(sign | (((1u << (15 - fbits)) - 1) << fbits) | (1u << (fbits - 1)));
    if (v == 0.0) return sign;
    if (isinf(v)) return (uint16_t)(sign | (((1u << (15 - fbits)) - 1) << fbits));
    int ex;
    frexp(v, &ex);
    int e = ex - 1;
    if (e < f.emin) {
        double frac = v / ldexp(1.0, f.emin - fbits); /* subnormal: integer < 2^fbits */
        return (uint16_t)(sign | (uint16_t)frac);
    }
    double frac = (v / ldexp(1.0, e) - 1.0) * ldexp(1.0, fbits);
    return (uint16_t)(sign | ((uint16_t)(e + f.bias) << fbits) | (uint16_t)frac);
}

static double decode_fmt(uint16_t h, orc_fmt f) {
    int fbits = f.p - 1;
    int ebits = 15 - fbits;
    int neg = (h >> 15) & 1;
    unsigned ef = (h >> fbits) & ((1u << ebits) - 1);
    unsigned frac = h & ((1u << fbits) - 1);
    double v;
    if (ef == (1u << ebits) - 1) v = frac ? NAN : INFINITY;
    else if (ef == 0) v = (double)frac * ldexp(1.0, f.emin - fbits);
    else v = (1.0 + (double)frac * ldexp(1.0, -fbits)) * ldexp(1.0, (int)ef - f.bias);
    return neg ? -v : v;
}

static uint16_t to_fmt(double x, orc_fmt f) {
    if (isnan(x)) return encode_fmt(x, 0, f);
    int neg = signbit(x) ? 1 : 0;
    return encode_fmt(round_to_fmt(fabs(x), f), neg, f);
}

uint16_t orc_f32_to_f16(float x) { return to_fmt((double)x, FMT_F16); }
float orc_f16_to_f32(uint16_t h) { return (float)decode_fmt(h, FMT_F16); }
uint16_t orc_f32_to_bf16(float x) { return to_fmt((double)x, FMT_BF16); }
uint16_t orc_f64_to_bf16(double x) { return to_fmt(x, FMT_BF16); }
float orc_bf16_to_f32(uint16_t h) { return (float)decode_fmt(h, FMT_BF16); }

/* ------------------------------------------------------------------ */
/* int4 weights: quantise / pack, and the exact dequantised value.      */

static int nibble_value(const uint8_t* q_row, int64_t i) {
    unsigned byte = q_row[i / 2];
    unsigned nib = (i % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
    return (nib >= 8) ? (int)nib - 16 : (int)nib; /* 4-bit two's complement */
}

void orc_pack_w4(const float* w, int64_t rows, int64_t K, int32_t group, uint8_t* q,
                 uint16_t* s) {
    int64_t ngroups = K / group;
    for (int64_t r = 0; r < rows; ++r) {
        const float* wr = w + r * K;
        uint8_t* qr = q + r * (K / 2);
        memset(qr, 0, (size_t)(K / 2));
        for (int64_t gi = 0; gi < ngroups; ++gi) {
            float absmax = 0.0f;
            for (int64_t i = gi * group; i < (gi + 1) * group; ++i) {
                float a = fabsf(wr[i]);
                if (a > absmax) absmax = a;
            }
            uint16_t s16 = orc_f32_to_f16(absmax / 7.0f);
            s[r * ngroups + gi] = s16;
            float sf = orc_f16_to_f32(s16);
            for (int64_t i = gi * group; i < (gi + 1) * group; ++i) {
                int qi = 0;
                if (sf != 0.0f) {
                    float t = wr[i] / sf;
                    float rt = rintf(t);
                    if (rt < -8.0f) rt = -8.0f;
                    if (rt > 7.0f) rt = 7.0f;
                    qi = (int)rt;
                }
                unsigned nib = (unsigned)qi & 0xFu;
                qr[i / 2] |= (uint8_t)((i % 2 == 0) ? nib : (nib << 4));
            }
        }
    }
}

void orc_dequant_w4(const uint8_t* q, const uint16_t* s, int64_t rows, int64_t K, int32_t group,
                    float* w_hat) {
    int64_t ngroups = K / group;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t i = 0; i < K; ++i)
            w_hat[r * K + i] = (float)nibble_value(q + r * (K / 2), i) *
                               orc_f16_to_f32(s[r * ngroups + i / group]);
}

/* ------------------------------------------------------------------ */
/* Load-time import of GGUF-style Q4 blocks (R15).                      */
/* thewafflehaus/butter PR #69, commit "feat(laguna): Laguna-S-2.1       */
/* decode on the CUDA engine": the expert weights are read from GGUF and */
/* re-quantised to the engine's 4-bit format when the model is loaded.   */

void orc_dequant_q4_blocks(const uint8_t* blocks, int64_t rows, int64_t K, float* w) {
    int64_t nb = K / 32;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* blk = blocks + (r * nb + b) * 18;
            uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8)); /* little-endian fp16 */
            float dscale = orc_f16_to_f32(dbits);
            for (int i = 0; i < 32; ++i) {
                int byte = blk[2 + (i & 15)];
                int n = i < 16 ? (byte & 15) : (byte >> 4);
                w[r * K + b * 32 + i] = (float)(n - 8) * dscale;
            }
        }
}

void orc_import_q4_blocks(const uint8_t* blocks, int64_t rows, int64_t K, int32_t group,
                          uint8_t* q, uint16_t* s) {
    if (group <= 32) {  /* every group inside one block: s = d, q = n - 8 */
        int64_t nb = K / 32, ng = K / group;
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* blk = blocks + (r * nb + b) * 18;
                uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
                for (int i = 0; i < 32; i += group) s[r * ng + (b * 32 + i) / group] = dbits;
                for (int j = 0; j < 16; ++j) {
                    int e0 = 2 * j, e1 = 2 * j + 1; /* elements of packed byte j */
                    int n0 = e0 < 16 ? (blk[2 + e0] & 15) : (blk[2 + e0 - 16] >> 4);
                    int n1 = e1 < 16 ? (blk[2 + e1] & 15) : (blk[2 + e1 - 16] >> 4);
                    int q0 = n0 - 8, q1 = n1 - 8; /* two's-complement nibbles */
                    q[r * (K / 2) + b * 16 + j] = (uint8_t)((q0 & 15) | ((q1 & 15) << 4));
                }
            }
        return;
    }
    float* w = (float*)malloc(sizeof(float) * (size_t)(rows * K));
    orc_dequant_q4_blocks(blocks, rows, K, w);
    orc_pack_w4(w, rows, K, group, q, s);
    free(w);
}

/* ------------------------------------------------------------------ */
/* Router: fp64 logits and sigmoid scores, biased top-k selection.      */

void orc_router(const uint16_t* x, const float* W_r, const float* bias, int64_t T, int32_t d,
                int32_t E, int32_t k, int64_t t0, int64_t t1, int32_t* topk_idx, float* topk_w,
                double* margin, double* scores) {
    double* s = (double*)malloc(sizeof(double) * (size_t)E);
    double* key = (double*)malloc(sizeof(double) * (size_t)E);
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    (void)T;
    for (int64_t t = t0; t < t1; ++t) {
        const uint16_t* xt = x + t * d;
        for (int32_t e = 0; e < E; ++e) {
            double l = 0.0;
            for (int32_t i = 0; i < d; ++i)
                l += (double)orc_bf16_to_f32(xt[i]) * (double)W_r[(int64_t)e * d + i];
            s[e] = 1.0 / (1.0 + exp(-l));
            key[e] = s[e] + (double)bias[e];
            taken[e] = 0;
            if (scores) scores[t * E + e] = s[e];
        }
        double kth = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || key[e] > key[best])) best = e;
            taken[best] = 1;
            topk_idx[t * k + j] = best;
            kth = key[best];
        }
        if (margin) {
            if (k < E) {
                int32_t next = -1;
                for (int32_t e = 0; e < E; ++e)
                    if (!taken[e] && (next < 0 || key[e] > key[next])) next = e;
                margin[t] = kth - key[next];
            } else {
                margin[t] = INFINITY;
            }
        }
        double sum = 0.0;
        for (int32_t j = 0; j < k; ++j) sum += s[topk_idx[t * k + j]];
        for (int32_t j = 0; j < k; ++j)
            topk_w[t * k + j] = (float)(s[topk_idx[t * k + j]] / sum);
    }
    free(s);
    free(key);
    free(taken);
}

/* ------------------------------------------------------------------ */
/* Expert descriptors.                                                  */

void orc_descriptors(const int32_t* topk_idx, int64_t T, int32_t E, int32_t k, int32_t* counts,
                     int32_t* offsets, int32_t* perm, int32_t* pos, int32_t* sched) {
    if (E <= 0) return;
    for (int32_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t sl = 0; sl < T * k; ++sl) counts[topk_idx[sl]] += 1;
    offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int64_t cursor = 0;
    for (int32_t e = 0; e < E; ++e)
        for (int64_t t = 0; t < T; ++t)
            for (int32_t j = 0; j < k; ++j)
                if (topk_idx[t * k + j] == e) perm[cursor++] = (int32_t)(t * k + j);
    for (int64_t r = 0; r < T * k; ++r) pos[perm[r]] = (int32_t)r;
    /* experts by count, largest first; equal counts keep ascending ids */
    unsigned char* used = (unsigned char*)calloc((size_t)E, 1);
    for (int32_t i = 0; i < E; ++i) {
        int32_t best = -1;
        for (int32_t e = 0; e < E; ++e)
            if (!used[e] && (best < 0 || counts[e] > counts[best])) best = e;
        used[best] = 1;
        sched[i] = best;
    }
    free(used);
}

/* ------------------------------------------------------------------ */
/* One expert on one token: fused gate+up SwiGLU, then the down projection. */

static float dot_w4_row(const float* xf, const uint8_t* q_row, const uint16_t* s_row, int64_t K,
                        int32_t group) {
    float acc = 0.0f;
    for (int64_t gi = 0; gi < K / group; ++gi) {
        float sc = orc_f16_to_f32(s_row[gi]);
        for (int64_t i = gi * group; i < (gi + 1) * group; ++i) {
            float w_hat = (float)nibble_value(q_row, i) * sc; /* exact */
            acc += xf[i] * w_hat;                             /* product exact; sum rounds */
        }
    }
    return acc;
}

void orc_expert_token(const uint16_t* x, int32_t d, int32_t F, int32_t group,
                      const uint8_t* q_gu, const uint16_t* s_gu, const uint8_t* q_dn,
                      const uint16_t* s_dn, uint16_t* h, float* y) {
    float* xf = (float*)malloc(sizeof(float) * (size_t)d);
    float* hf = (float*)malloc(sizeof(float) * (size_t)F);
    for (int32_t i = 0; i < d; ++i) xf[i] = orc_bf16_to_f32(x[i]);
    int64_t gu_row_bytes = d / 2, gu_row_scales = d / group;
    for (int32_t f = 0; f < F; ++f) {
        float g = dot_w4_row(xf, q_gu + (int64_t)f * gu_row_bytes, s_gu + (int64_t)f * gu_row_scales,
                             d, group);
        float u = dot_w4_row(xf, q_gu + (int64_t)(F + f) * gu_row_bytes,
                             s_gu + (int64_t)(F + f) * gu_row_scales, d, group);
        double silu = (double)g / (1.0 + exp(-(double)g));
        h[f] = orc_f64_to_bf16(silu * (double)u);
        hf[f] = orc_bf16_to_f32(h[f]);
    }
    int64_t dn_row_bytes = F / 2, dn_row_scales = F / group;
    for (int32_t c = 0; c < d; ++c)
        y[c] = dot_w4_row(hf, q_dn + (int64_t)c * dn_row_bytes, s_dn + (int64_t)c * dn_row_scales, F,
                          group);
    free(xf);
    free(hf);
}

/* ------------------------------------------------------------------ */
/* The layer for a list of tokens, given the selection.                 */

void orc_layer_tokens(const uint16_t* x, int32_t d, int32_t E, int32_t k, int32_t F, int32_t Fs,
                      int32_t group, const int32_t* topk_idx, const float* topk_w,
                      const uint8_t* q_gu, const uint16_t* s_gu, const uint8_t* q_dn,
                      const uint16_t* s_dn, const uint8_t* qs_gu, const uint16_t* ss_gu,
                      const uint8_t* qs_dn, const uint16_t* ss_dn, const uint16_t* residual,
                      const int64_t* tokens, int64_t n_tokens, uint16_t* out, uint16_t* h_routed,
                      uint16_t* h_shared) {
    int64_t gu_bytes = (int64_t)2 * F * (d / 2), gu_scales = (int64_t)2 * F * (d / group);
    int64_t dn_bytes = (int64_t)d * (F / 2), dn_scales = (int64_t)d * (F / group);
    float* y = (float*)malloc(sizeof(float) * (size_t)d);
    float* acc = (float*)malloc(sizeof(float) * (size_t)d);
    uint16_t* h = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(F > Fs ? F : Fs));
    (void)E;
    for (int64_t n = 0; n < n_tokens; ++n) {
        int64_t t = tokens[n];
        const uint16_t* xt = x + t * d;
        for (int32_t c = 0; c < d; ++c) acc[c] = 0.0f;
        for (int32_t j = 0; j < k; ++j) {
            int64_t e = topk_idx[t * k + j];
            float wj = topk_w[t * k + j];
            orc_expert_token(xt, d, F, group, q_gu + e * gu_bytes, s_gu + e * gu_scales,
                             q_dn + e * dn_bytes, s_dn + e * dn_scales, h, y);
            if (h_routed) memcpy(h_routed + (n * k + j) * F, h, sizeof(uint16_t) * (size_t)F);
            for (int32_t c = 0; c < d; ++c) {
                float p = wj * y[c];
                acc[c] = acc[c] + p;
            }
        }
        orc_expert_token(xt, d, Fs, group, qs_gu, ss_gu, qs_dn, ss_dn, h, y);
        if (h_shared) memcpy(h_shared + n * Fs, h, sizeof(uint16_t) * (size_t)Fs);
        for (int32_t c = 0; c < d; ++c) {
            acc[c] = acc[c] + y[c];
            if (residual) acc[c] = orc_bf16_to_f32(residual[t * d + c]) + acc[c];
            out[n * d + c] = orc_f32_to_bf16(acc[c]);
        }
    }
    free(y);
    free(acc);
    free(h);
}

/* ------------------------------------------------------------------ */
/* W8A8 (R16): E4M3 codes, per-row scales, scales folded after the sum.  */

/* E4M3 without infinities, from its definition: value of a code. */
float orc_e4m3_to_f32(uint8_t b) {
    int neg = (b >> 7) & 1;
    int ef = (b >> 3) & 15, frac = b & 7;
    double v;
    if (ef == 15 && frac == 7) return NAN;
    if (ef == 0) v = (double)frac * ldexp(1.0, -9);
    else v = (1.0 + frac / 8.0) * ldexp(1.0, ef - 7);
    return (float)(neg ? -v : v);
}

/* Nearest E4M3 value of x, ties to even, saturating to +-448. */
uint8_t orc_f32_to_e4m3(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint8_t)(sign | 0x7E);
    int ex;
    frexp(a, &ex);
    int e = ex - 1;
    if (e < -6) e = -6;                         /* subnormal binade shares 2^-6's quantum */
    double quantum = ldexp(1.0, e - 3);
    double r = rint(a / quantum) * quantum;
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return sign;
    frexp(r, &ex);
    e = ex - 1;
    if (e < -6) return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9)));
    return (uint8_t)(sign | ((e + 7) << 3) | (int)((r / ldexp(1.0, e) - 1.0) * 8.0));
}

/* One row's scale (absmax / 448 in fp32) and codes. */
static void quant_row_fp8(const float* v, int64_t K, uint8_t* q, float* scale) {
    float amax = 0.0f;
    for (int64_t i = 0; i < K; ++i) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    float sc = amax / 448.0f;
    *scale = sc;
    for (int64_t i = 0; i < K; ++i) q[i] = sc == 0.0f ? 0 : orc_f32_to_e4m3(v[i] / sc);
}

void orc_pack_w8(const float* w, int64_t rows, int64_t K, uint8_t* q, float* s) {
    for (int64_t r = 0; r < rows; ++r) quant_row_fp8(w + r * K, K, q + r * K, s + r);
}

void orc_quant_rows_fp8(const float* x, int64_t n, int64_t K, uint8_t* q, float* a) {
    for (int64_t r = 0; r < n; ++r) quant_row_fp8(x + r * K, K, q + r * K, a + r);
}

/* v = (acc * a) * s_w with acc the fp32 ascending sum of exact products. */
static float dot_w8_row(const uint8_t* xq, float a, const uint8_t* q_row, float s_row, int64_t K) {
    float acc = 0.0f;
    for (int64_t i = 0; i < K; ++i) acc += orc_e4m3_to_f32(q_row[i]) * orc_e4m3_to_f32(xq[i]);
    return (acc * a) * s_row;
}

void orc_expert_token_w8a8(const uint16_t* x, int32_t d, int32_t F, const uint8_t* q_gu,
                           const float* s_gu, const uint8_t* q_dn, const float* s_dn, uint16_t* h,
                           float* y) {
    float* xf = (float*)malloc(sizeof(float) * (size_t)d);
    float* hf = (float*)malloc(sizeof(float) * (size_t)F);
    uint8_t* xq = (uint8_t*)malloc((size_t)d);
    uint8_t* hq = (uint8_t*)malloc((size_t)F);
    float a_x, a_h;
    for (int32_t i = 0; i < d; ++i) xf[i] = orc_bf16_to_f32(x[i]);
    quant_row_fp8(xf, d, xq, &a_x);
    for (int32_t f = 0; f < F; ++f) {
        float g = dot_w8_row(xq, a_x, q_gu + (int64_t)f * d, s_gu[f], d);
        float u = dot_w8_row(xq, a_x, q_gu + (int64_t)(F + f) * d, s_gu[F + f], d);
        double silu = (double)g / (1.0 + exp(-(double)g));
        h[f] = orc_f64_to_bf16(silu * (double)u);
        hf[f] = orc_bf16_to_f32(h[f]);
    }
    quant_row_fp8(hf, F, hq, &a_h);
    for (int32_t c = 0; c < d; ++c) y[c] = dot_w8_row(hq, a_h, q_dn + (int64_t)c * F, s_dn[c], F);
    free(xf);
    free(hf);
    free(xq);
    free(hq);
}

void orc_layer_w8a8_tokens(const uint16_t* x, int32_t d, int32_t k, int32_t F, int32_t Fs,
                           const int32_t* topk_idx, const float* topk_w, const uint8_t* q_gu,
                           const float* s_gu, const uint8_t* q_dn, const float* s_dn,
                           const uint8_t* qs_gu, const float* ss_gu, const uint8_t* qs_dn,
                           const float* ss_dn, const int64_t* tokens, int64_t n_tokens,
                           uint16_t* out, uint16_t* h_routed, uint16_t* h_shared) {
    int64_t gu_bytes = (int64_t)2 * F * d, dn_bytes = (int64_t)d * F;
    float* y = (float*)malloc(sizeof(float) * (size_t)d);
    float* acc = (float*)malloc(sizeof(float) * (size_t)d);
    uint16_t* h = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(F > Fs ? F : Fs));
    for (int64_t n = 0; n < n_tokens; ++n) {
        int64_t t = tokens[n];
        const uint16_t* xt = x + t * d;
        for (int32_t c = 0; c < d; ++c) acc[c] = 0.0f;
        for (int32_t j = 0; j < k; ++j) {
            int64_t e = topk_idx[t * k + j];
            float wj = topk_w[t * k + j];
            orc_expert_token_w8a8(xt, d, F, q_gu + e * gu_bytes, s_gu + e * 2 * F,
                                  q_dn + e * dn_bytes, s_dn + e * d, h, y);
            if (h_routed) memcpy(h_routed + (n * k + j) * F, h, sizeof(uint16_t) * (size_t)F);
            for (int32_t c = 0; c < d; ++c) {
                float p = wj * y[c];
                acc[c] = acc[c] + p;
            }
        }
        orc_expert_token_w8a8(xt, d, Fs, qs_gu, ss_gu, qs_dn, ss_dn, h, y);
        if (h_shared) memcpy(h_shared + n * Fs, h, sizeof(uint16_t) * (size_t)Fs);
        for (int32_t c = 0; c < d; ++c) {
            acc[c] = acc[c] + y[c];
            out[n * d + c] = orc_f32_to_bf16(acc[c]);
        }
    }
    free(y);
    free(acc);
    free(h);
}

void orc_f32_to_e4m3_array(const float* x, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_e4m3(x[i]);
}
void orc_e4m3_to_f32_array(const uint8_t* b, int64_t n, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_to_f32(b[i]);
}

/* ------------------------------------------------------------------ */
/* Element-wise helpers over arrays (used by the tests' format pins).   */

void orc_f32_to_f16_array(const float* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(x[i]);
}
void orc_f16_to_f32_array(const uint16_t* h, int64_t n, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f32(h[i]);
}
void orc_f32_to_bf16_array(const float* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(x[i]);
}
void orc_f64_to_bf16_array(const double* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16(x[i]);
}
void orc_bf16_to_f32_array(const uint16_t* h, int64_t n, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f32(h[i]);
}
