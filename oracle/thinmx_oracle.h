/*
 * thinmx CPU oracle — TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, single-threaded C implementation of everything the
 * weight-only low-bit matvec path computes, in fp64.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it.  It
 * shares no code, header, table or helper with the CUDA library; the two
 * are compared element by element on the same seeded inputs.
 *
 * Sources followed (the pages are informal devlogs of the "ThinTensor"
 * decode runtime):
 *   [DL4]  ThinTensor devlog feed, kerbin.cskartikey.dev/@satvikhardat,
 *          "Dev Log #4 — 91–96 tok/s with Selective MXFP4", sections
 *          "Why this was not just normal quantization" and
 *          "Where Blackwell helps" (store fewer bytes, block scales, BF16
 *          activations, safe accumulation, then the row postscale).
 *   [DL2]  same feed, "Dev Log #2", the execution-tape operator list
 *          (gated_activation, router, expert stages).
 *   [SHIP] ThinTensor project page, stardance.hackclub.com/projects/29750,
 *          "Hitting 100hrs and final ship" (production MXFP4/INT4
 *          quantizers; exact routing), the MoE drift devlog (tl.dot_scaled
 *          over the selected experts), the 97.87 tok/s notes
 *          (dense_int4_layers) and the fixes list ("correct affine INT4
 *          partial-group quantization").
 *   [DL3]  same feed, "Dev Log #3 — SmolLM3-3B Results": the "quality
 *          FP8" profile (gate/up and down projections in FP8, the rest in
 *          BF16) and its FP8 MLP kernel, a scaled matvec whose row sum of
 *          w * x is multiplied by the row's scale.  The element format
 *          (E4M3) and the scale rule (row amax / 448) are not printed.
 *          The same section's attention kernel: single-token GQA, each
 *          query head mapped to kv_head = head // (heads // kv_heads),
 *          scores = sum(key * q) * scale over the cached tokens, with the
 *          KV cache kept in BF16 ("KV cache: full BF16", causal KV).
 *   [SHIP] also: the 97.87 tok/s notes pack the MoE experts of layers
 *          0:24 as 1-bit "Q1" structures (packed_expert_q1_layers), 9.52
 *          GB of MXFP4 experts becoming 2.38 GB, and the final devlog names
 *          Q2 and Q1 quantizers and a low-bit selected-expert SwiGLU
 *          kernel.  The encoding is not printed; the reading taken here is
 *          the one the 4x footprint ratio fixes for an MX-style format: one
 *          bit (Q1) or two (Q2) per weight plus one E8M0 byte per 128
 *          weights (1 + 8/128 = 1.0625 bits against MXFP4's 4.25).
 * The pages never spell out the bit formats; E2M1 (1 sign, 2 exponent bits
 * with bias 1, 1 mantissa bit) and E8M0 (8 exponent bits, bias 127, 0xFF =
 * NaN) are the MXFP4 element and scale formats, and the scale rule
 * X = floor(log2 amax) - 2 maps the block maximum into E2M1's top binade.
 *
 * Parity pins: every function here is pinned by tests/test_oracle_pins.py
 * against closed forms, exhaustive tables, invariants and library routines.
 */
#ifndef THINMX_ORACLE_H
#define THINMX_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status values (own copy; the oracle includes nothing from the library). */
#define ORC_OK 0
#define ORC_ERR_SHAPE 2
#define ORC_ERR_NONFINITE 4

/* ---- scalar formats ---------------------------------------------------- */
double   orc_e2m1_value(unsigned code);          /* code 0..15 -> value      */
double   orc_e8m0_value(unsigned byte);          /* 2^(b-127); 255 -> NaN    */
unsigned orc_e2m1_encode(double t);              /* nearest, ties to even
                                                    mantissa, saturate at 6,
                                                    sign bit kept on zero    */
int      orc_floor_log2(float a);                /* a > 0 finite             */
double   orc_bf16_value(uint16_t b);
uint16_t orc_bf16_round(double v);               /* round-to-nearest-even    */
double   orc_f16_value(uint16_t h);
uint16_t orc_f16_round(double v);                /* round-to-nearest-even    */

/* ---- MXFP4 ------------------------------------------------------------- */
/* w: fp32 [n][k], k % 32 == 0.  codes: [n][k/2] (low nibble = even k).
   scales: E8M0 [n][k/32].  A block holding a NaN/Inf gets scale 0xFF and
   zero codes, and the call returns ORC_ERR_NONFINITE. */
int  orc_mxfp4_quantize(const float* w, int64_t n, int64_t k,
                        uint8_t* codes, uint8_t* scales);
void orc_mxfp4_dequantize(const uint8_t* codes, const uint8_t* scales,
                          int64_t n, int64_t k, double* out /* [n][k] */);
/* y[m][n] = postscale[n] * sum_k deq[n][k] * x[m][k]; postscale may be NULL */
void orc_mxfp4_matvec(const uint8_t* codes, const uint8_t* scales,
                      const float* postscale, int64_t n, int64_t k,
                      const uint16_t* x_bf16, int64_t m, double* y);
void orc_bf16_matvec(const uint16_t* w_bf16, int64_t n, int64_t k,
                     const uint16_t* x_bf16, int64_t m, double* y);
void orc_swiglu(const double* g, const double* u, int64_t len, double* h);
void orc_mxfp4_swiglu_matvec(const uint8_t* g_codes, const uint8_t* g_scales,
                             const float* g_post,
                             const uint8_t* u_codes, const uint8_t* u_scales,
                             const float* u_post, int64_t n, int64_t k,
                             const uint16_t* x_bf16, int64_t m, double* h);
void orc_bf16_swiglu_matvec(const uint16_t* wg, const uint16_t* wu,
                            int64_t n, int64_t k, const uint16_t* x_bf16,
                            int64_t m, double* h);

/* ---- MoE --------------------------------------------------------------- */
void orc_router_logits(const uint16_t* x_bf16, const uint16_t* wr_bf16,
                       int32_t n_experts, int64_t hidden, double* logits);
void orc_topk(const float* logits, int32_t n_experts, int32_t top_k,
              int32_t* idx);
void orc_softmax_selected(const float* logits, const int32_t* idx,
                          int32_t top_k, double* p);
/* Experts are stacked: gate/up [E][2*inter][hidden] (gate rows first),
   down [E][hidden][inter].  out [hidden] fp64, idx/p [top_k].  x is one
   token (M = 1). */
int  orc_moe_mlp(const uint16_t* x_bf16, int64_t hidden, int64_t inter,
                 const uint16_t* wr_bf16, int32_t n_experts, int32_t top_k,
                 const uint8_t* gu_codes, const uint8_t* gu_scales,
                 const uint8_t* dn_codes, const uint8_t* dn_scales,
                 double* out, int32_t* idx, double* p,
                 float* logits32 /* [E], out */);

/* ---- FP8 (E4M3) with one fp32 scale per row ----------------------------- */
/* E4M3 without infinities: bit 7 sign, bits 6..3 exponent (bias 7), bits
   2..0 mantissa; 0x7F / 0xFF are NaN, the largest magnitude is 448.
   Quantise per row: scale = fp32(amax / 448), code = E4M3 round-to-nearest-
   even of w / scale, saturating at 448 (amax = 0: scale 0, zero codes; a
   row holding a NaN/Inf: NaN scale, zero codes, ORC_ERR_NONFINITE).
   codes: [n][k] one byte per weight; scales: fp32 [n]. */
double   orc_e4m3_value(unsigned code);
unsigned orc_e4m3_encode(double t);
int  orc_fp8_quantize(const float* w, int64_t n, int64_t k, uint8_t* codes,
                      float* scales);
void orc_fp8_dequantize(const uint8_t* codes, const float* scales, int64_t n,
                        int64_t k, double* out /* [n][k] */);
/* y[m][n] = scale[n] * sum_k E4M3(code[n][k]) * x[m][k] */
void orc_fp8_matvec(const uint8_t* codes, const float* scales, int64_t n,
                    int64_t k, const uint16_t* x_bf16, int64_t m, double* y);
void orc_fp8_swiglu_matvec(const uint8_t* g_codes, const float* g_scales,
                           const uint8_t* u_codes, const float* u_scales,
                           int64_t n, int64_t k, const uint16_t* x_bf16,
                           int64_t m, double* h);

/* ---- grouped affine INT4 ----------------------------------------------- */
/* groups [g*G, min((g+1)*G, k)); codes [n][k/2] low nibble = even k
   (k even); scales fp16 [n][ceil(k/G)]; zp [n][ceil(ceil(k/G)/2)] low
   nibble = even group. */
int  orc_int4_quantize(const float* w, int64_t n, int64_t k, int32_t group,
                       uint8_t* codes, uint16_t* scales_f16, uint8_t* zp);
void orc_int4_dequantize(const uint8_t* codes, const uint16_t* scales_f16,
                         const uint8_t* zp, int64_t n, int64_t k,
                         int32_t group, double* out);
void orc_int4_matvec(const uint8_t* codes, const uint16_t* scales_f16,
                     const uint8_t* zp, int64_t n, int64_t k, int32_t group,
                     const uint16_t* x_bf16, int64_t m, double* y);

/* ---- single-token GQA attention [DL3] --------------------------------- */
/* o[h][:] = sum_t softmax_t(scale * q[h] . k[kvh][t]) * v[kvh][t], with
   kvh = h / (heads / kv_heads), t < len; k, v [kv_heads][cap][d] bf16. */
int orc_gqa_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                   int32_t heads, int32_t kv_heads, int32_t d, int64_t cap,
                   int64_t len, double scale, double* o);

/* ---- Q1 / Q2 packed low-bit experts [SHIP] ---------------------------- */
/* bits 1 or 2 per weight, one E8M0 step 2^X per block of 128 along k (the
   last block may be partial); X = the power of two nearest the block's
   mean |w|; Q1 code = sign, Q2 code = clamp(floor(w / 2^X) + 2, 0, 3).
   Buffer layout: plane 0 [n][P] (+ plane 1 [n][P] for Q2), scales [n][S],
   P = ceil(k/8) and S = ceil(k/128), each rounded up to 16 bytes. */
int64_t orc_lowbit_plane_bytes(int64_t k);
int64_t orc_lowbit_scale_bytes(int64_t k);
int64_t orc_lowbit_matrix_bytes(int32_t bits, int64_t n, int64_t k);
int  orc_lowbit_quantize(int32_t bits, const float* w, int64_t n, int64_t k,
                         uint8_t* buf);
void orc_lowbit_dequantize(int32_t bits, const uint8_t* buf, int64_t n,
                           int64_t k, double* out);
int  orc_moe_lowbit_mlp(int32_t bits, const uint16_t* x_bf16, int64_t hidden,
                        int64_t inter, const uint16_t* wr_bf16,
                        int32_t n_experts, int32_t top_k, const uint8_t* gu,
                        const uint8_t* dn, double* out, int32_t* idx,
                        double* p, float* logits32, double* h);

#ifdef __cplusplus
}
#endif
#endif
