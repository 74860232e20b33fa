/*
 * CPU oracle of the LatentMoE layer forward pass -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, single-threaded C in fp64.  It exists to check the CUDA path:
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load it.  It shares no code, header, table or constant with the CUDA
 * library, and the library never calls it.
 *
 * Sources followed (page title, section):
 *  [P2-MoE]  "SGLang 0.5.17: Kimi K3 原生 MXFP4 推理架构解析", section
 *            "MoE 稀疏激活：896 专家中选 16" -- router scores = token x router
 *            weights, keep the top 16 of 896 experts, evaluate only those.
 *  [P2-MX]   same page, section "MXFP4 原生支持" -- one shared scale per block
 *            of 32 (or 64) elements; dequantisation fused with the GEMM.
 *  [P1-L1]   "从Kimi K3到MiniMax-H3：国产大模型竞争进入“推理系统战”", section 二,
 *            first layer -- 4-bit weights are combined with higher-precision
 *            activations and higher-precision accumulation.
 *  [P1-A]    same page, section 一 -- experts run in a 3584-wide latent space
 *            (LatentMoE) with a gated FFN (SwiGLU family; K3's "SiTU" is not
 *            defined there, so SiLU gating is the stated assumption).
 *  [P3-EP]   "Kimi K3 Day-0 适配剖析", section 四 -- dispatch tokens to their
 *            experts, expert compute, combine the results back by weight.
 *
 * Formats (one byte per code unless packed):
 *  e2m1  : 4-bit, sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 *  e4m3  : 8-bit, sign bit 7, exponent bits 6..3 (bias 7), mantissa 2..0,
 *          no infinities, S.1111.111 is NaN, max finite 448.
 *  e8m0  : scale byte s encodes 2^(s-127); 255 is NaN.
 *  MXFP4 : codes[r][K/2], element 2i in the low nibble of byte i;
 *          scales[r][K/32], one e8m0 per 32 consecutive elements along K.
 *  MXFP8 : codes[r][K] e4m3, scales[r][K/32] e8m0.
 */
#ifndef LMOE_ORACLE_H
#define LMOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- element codecs ---------------------------------------------------- */
double oracle_e2m1_value(uint8_t code);
double oracle_e4m3_value(uint8_t code);
double oracle_e8m0_value(uint8_t s);
uint8_t oracle_e2m1_encode(double v);
uint8_t oracle_e4m3_encode(double v);
/* Shared block exponent X = floor(log2(amax)) - emax (emax 2 for e2m1,
 * 8 for e4m3), then the scale byte clamp(X + 127, 0, 254); amax == 0 gives
 * byte 0.  Returns the scale byte. */
uint8_t oracle_scale_byte(double amax, int emax);

/* ---- block quantisation ------------------------------------------------ */
void oracle_quant_mxfp4(const float *w, int64_t rows, int K, uint8_t *q, uint8_t *s);
void oracle_quant_mxfp8(const uint16_t *x_bf16, int64_t rows, int K, uint8_t *q, uint8_t *s);
void oracle_quant_mxfp8_f64(const double *x, int64_t rows, int K, uint8_t *q, uint8_t *s);
/* MXFP4 of double values (the gated product h in the FP4-activation mode):
 * the rule of oracle_quant_mxfp4, from exact double inputs. */
void oracle_quant_mxfp4_f64(const double *x, int64_t rows, int K, uint8_t *q, uint8_t *s);
void oracle_dequant_mxfp4(const uint8_t *q, const uint8_t *s, int64_t rows, int K, double *out);
void oracle_dequant_mxfp8(const uint8_t *q, const uint8_t *s, int64_t rows, int K, double *out);

/* ---- routing ----------------------------------------------------------- */
void oracle_router_logits(const uint16_t *x_bf16, const float *Wr, const float *bias, int T, int d, int E,
                          float *logits);
void oracle_topk_softmax(const float *logits, int T, int E, int k, int32_t *idx, float *w);
void oracle_permute(const int32_t *idx, int T, int k, int E, int32_t *counts, int32_t *offsets, int32_t *perm,
                    int32_t *inv);

/* ---- experts and combine ----------------------------------------------- */
typedef struct {
    const uint8_t *gate_q, *gate_s; /* [E][I][d/2], [E][I][d/32] */
    const uint8_t *up_q, *up_s;     /* [E][I][d/2], [E][I][d/32] */
    const uint8_t *down_q, *down_s; /* [E][d][I/2], [E][d][I/32] */
} oracle_experts;

/* y for the listed tokens (all T when tokens == NULL, ntok = T):
 * y_t = sum_j w[t][j] * FFN_{idx[t][j]}(x_t), returned as bf16 bits and,
 * when y_f64 != NULL, before the bf16 rounding. */
void oracle_moe_tokens(const uint16_t *x_bf16, const int32_t *idx, const float *w, const oracle_experts *W, int T,
                       int d, int E, int k, int I, const int32_t *tokens, int ntok, uint16_t *y_bf16, double *y_f64);
/* One expert's FFN on one token: out[d] = Wd * MXFP8(silu(Wg x^) * (Wu x^)), x^ = MXFP8(x). */
void oracle_expert_ffn_token(const uint16_t *x_bf16_row, const oracle_experts *W, int e, int d, int I, double *out);
/* The same layer with a choice of activation format: act 1 rounds x and h
 * to MXFP8 (oracle_moe_tokens), act 2 to MXFP4 (e2m1 + E8M0 per 32, the
 * weights' rule) -- the full-FP4 variant, whose numerics differ from the
 * MXFP8 layer by the coarser activation grid. */
#define ORACLE_ACT_MXFP8 1
#define ORACLE_ACT_MXFP4 2
void oracle_moe_tokens_act(const uint16_t *x_bf16, const int32_t *idx, const float *w, const oracle_experts *W,
                           int T, int d, int E, int k, int I, const int32_t *tokens, int ntok, int act,
                           uint16_t *y_bf16, double *y_f64);
/* Brute force: every expert evaluated for every listed token, unselected gates zero. */
void oracle_moe_dense(const uint16_t *x_bf16, const int32_t *idx, const float *w, const oracle_experts *W, int T,
                      int d, int E, int k, int I, const int32_t *tokens, int ntok, double *y_f64);

/* out[i] = bf16 bits of v[i] rounded to nearest even (ties to the even
 * significand, overflow past the largest finite bf16 to infinity, bf16
 * subnormals below 2^-126), rounded once from the double value. */
void oracle_round_bf16(const double *v, int64_t n, uint16_t *out);

/* out[r][n] = bf16( sum_c x[r][c] * W[n][c] ), all bf16 bits, fp64 accumulation. */
void oracle_linear_bf16(const uint16_t *x, const uint16_t *W, int64_t rows, int K, int N, uint16_t *out);

#ifdef __cplusplus
}
#endif
#endif
