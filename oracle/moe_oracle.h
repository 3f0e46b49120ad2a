/*
 * ORACLE -- test infrastructure, not part of the product.  Only the test
 * suite, the package's smoke check and the benchmark's CPU-baseline leg use it.
 *
 * Plain C definition of the routed MoE FFN layer (sigmoid top-k router with
 * score-correction bias, int4 W4A16 experts with fused gate+up SwiGLU, down
 * projection, weighted combine plus an always-on shared expert).  The source
 * passages and the readings taken are listed at the top of moe_oracle.c.
 *
 * Conventions: bf16 and fp16 values travel as their 16-bit patterns
 * (uint16_t).  Packed int4 weights are [rows][K/2] bytes, scales fp16
 * [rows][K/group].  All arrays are row-major and caller-owned.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>
#include <stdlib.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Number formats, round-to-nearest-even, from the IEEE 754 definitions. */
uint16_t orc_f32_to_f16(float x);
float orc_f16_to_f32(uint16_t h);
uint16_t orc_f32_to_bf16(float x);
uint16_t orc_f64_to_bf16(double x);
float orc_bf16_to_f32(uint16_t h);

/* Symmetric int4 quantisation per group of `group` consecutive K elements:
   s = fp16(absmax / 7), q = clamp(rint(w / s), -8, 7); byte j of a row holds
   element 2j (bits 0-3) and 2j+1 (bits 4-7). */
void orc_pack_w4(const float* w, int64_t rows, int64_t K, int32_t group, uint8_t* q, uint16_t* s);
/* w_hat = q * s, exact in fp32. */
void orc_dequant_w4(const uint8_t* q, const uint16_t* s, int64_t rows, int64_t K, int32_t group,
                    float* w_hat);

/* GGUF-style Q4 blocks, 18 bytes per 32 weights of a row (K % 32 == 0):
   an fp16 scale d (little-endian), then 16 bytes whose byte i holds the code
   n of weight i in bits 0-3 and of weight i + 16 in bits 4-7; the weight is
   (n - 8) * d.  orc_dequant_q4_blocks writes w [rows][K] (exact in fp32);
   orc_import_q4_blocks packs it at `group`: for group <= 32 exactly (s = d,
   q = n - 8), for group 64 / 128 by re-quantising w with orc_pack_w4. */
void orc_dequant_q4_blocks(const uint8_t* blocks, int64_t rows, int64_t K, float* w);
void orc_import_q4_blocks(const uint8_t* blocks, int64_t rows, int64_t K, int32_t group,
                          uint8_t* q, uint16_t* s);

/* Router for tokens [t0, t1): fp64 logits x . W_r[e], fp64 sigmoid scores s,
   top-k of s + bias (ties to lower id, descending), weights s_j / sum s_j.
   margin[t] = (k-th largest key) - ((k+1)-th largest key), +inf when k == E.
   scores (nullable) receives s as [T][E]. */
void orc_router(const uint16_t* x, const float* W_r, const float* bias, int64_t T, int32_t d,
                int32_t E, int32_t k, int64_t t0, int64_t t1, int32_t* topk_idx, float* topk_w,
                double* margin, double* scores);

/* counts[E], offsets[E+1] (exclusive scan), perm[T*k] (slot ids sorted by
   (expert, token)), pos[T*k] (inverse of perm), sched[E] (experts by count
   desc, ties to lower id). */
void orc_descriptors(const int32_t* topk_idx, int64_t T, int32_t E, int32_t k, int32_t* counts,
                     int32_t* offsets, int32_t* perm, int32_t* pos, int32_t* sched);

/* One expert on one token: h[F] (bf16) = silu(gate) * up, y[d] (fp32) = down . h. */
void orc_expert_token(const uint16_t* x, int32_t d, int32_t F, int32_t group,
                      const uint8_t* q_gu, const uint16_t* s_gu, const uint8_t* q_dn,
                      const uint16_t* s_dn, uint16_t* h, float* y);

/* Layer output for the listed tokens: out[n][d] bf16 for token tokens[n].
   Routed weights are stacked over experts: q_gu [E][2F][d/2], s_gu
   [E][2F][d/group], q_dn [E][d][F/2], s_dn [E][d][F/group]; the shared expert
   has F = Fs.  residual (nullable) is a bf16 [T][d] row per token, added in
   fp32 after the routed + shared sum and before the one bf16 rounding.
   h_routed (nullable) receives [n][k][F], h_shared (nullable) [n][Fs]. */
void orc_layer_tokens(const uint16_t* x, int32_t d, int32_t E, int32_t k, int32_t F, int32_t Fs,
                      int32_t group, const int32_t* topk_idx, const float* topk_w,
                      const uint8_t* q_gu, const uint16_t* s_gu, const uint8_t* q_dn,
                      const uint16_t* s_dn, const uint8_t* qs_gu, const uint16_t* ss_gu,
                      const uint8_t* qs_dn, const uint16_t* ss_dn, const uint16_t* residual,
                      const int64_t* tokens, int64_t n_tokens, uint16_t* out, uint16_t* h_routed,
                      uint16_t* h_shared);


/* W8A8 (fp8 E4M3 weights and activations, reading R16): per-row scales
   (absmax / 448, fp32), codes E4M3 rounded to nearest even and saturated to
   +-448.  Weights q [rows][K] bytes, s fp32 [rows]; a layer's routed gate+up
   codes are [E][2F][d] with scales [E][2F], down [E][d][F] with [E][d]. */
float orc_e4m3_to_f32(uint8_t b);
uint8_t orc_f32_to_e4m3(float x);
void orc_pack_w8(const float* w, int64_t rows, int64_t K, uint8_t* q, float* s);
void orc_quant_rows_fp8(const float* x, int64_t n, int64_t K, uint8_t* q, float* a);
void orc_expert_token_w8a8(const uint16_t* x, int32_t d, int32_t F, const uint8_t* q_gu,
                           const float* s_gu, const uint8_t* q_dn, const float* s_dn, uint16_t* h,
                           float* y);
void orc_layer_w8a8_tokens(const uint16_t* x, int32_t d, int32_t k, int32_t F, int32_t Fs,
                           const int32_t* topk_idx, const float* topk_w, const uint8_t* q_gu,
                           const float* s_gu, const uint8_t* q_dn, const float* s_dn,
                           const uint8_t* qs_gu, const float* ss_gu, const uint8_t* qs_dn,
                           const float* ss_dn, const int64_t* tokens, int64_t n_tokens,
                           uint16_t* out, uint16_t* h_routed, uint16_t* h_shared);
void orc_f32_to_e4m3_array(const float* x, int64_t n, uint8_t* out);
void orc_e4m3_to_f32_array(const uint8_t* b, int64_t n, float* out);

/* Element-wise array forms of the format conversions. */
void orc_f32_to_f16_array(const float* x, int64_t n, uint16_t* out);
void orc_f16_to_f32_array(const uint16_t* h, int64_t n, float* out);
void orc_f32_to_bf16_array(const float* x, int64_t n, uint16_t* out);
void orc_f64_to_bf16_array(const double* x, int64_t n, uint16_t* out);
void orc_bf16_to_f32_array(const uint16_t* h, int64_t n, float* out);

#ifdef __cplusplus
}
#endif
#endif
