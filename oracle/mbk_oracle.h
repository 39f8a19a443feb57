/*
 * mbk_oracle.h -- plain, slow, CPU reference of batch-1 Llama-shaped decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library or its
 * Python binding) may include, link, load or call this code; only the tests, the
 * package's smoke check and the benchmark's CPU-baseline leg use it.  It shares no
 * code, header, table or constant with the CUDA path.
 *
 * What it computes is the decoder the MegaBake pages describe, op by op:
 *   "MegaBake: a PyTorch model compiled into one CUDA kernel, and what its 5.5x is
 *    measured against" (the "article"), section "What a megakernel is, and why small
 *    models want one": per layer an RMSNorm, the Q/K/V projections, RoPE, attention,
 *    the output projection, a residual add, a second norm, gate and up projections,
 *    SiLU, the down projection and a second residual add; and the megabake/megabake
 *    README ("Current status"): embedding, every layer, final norm, vocabulary
 *    projection and the KV-cache update, with a static contiguous decode KV cache.
 * The pages give the op list but no formulas; the formulas below are the textbook
 * (Hugging Face Llama) definitions of those ops.
 *
 * Precision (the pages are silent; this is the reading taken): weights and the KV
 * cache are bf16; every activation is stored as fp32; every reduction (dot product,
 * sum of squares, softmax sum) is accumulated in double and each op's result is
 * rounded once to fp32.  Only K and V are rounded to bf16 (round to nearest even)
 * when they are written into the cache; attention reads the rounded cache, including
 * the row just written.
 *
 * Parity pins for each function are listed beside it.  Whole-decoder parity with the
 * pages' own numbers is unpinned: the pages publish no weights or outputs.
 */
#ifndef MBK_ORACLE_H
#define MBK_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int n_layers, hidden, intermediate, n_heads, n_kv_heads, head_dim, vocab, kv_capacity;
  double rms_eps, rope_theta;
  int qkv_bias;
} orc_config;

/* bf16 tensors are passed as their raw 16-bit patterns; matrices are [out, in] row-major. */
typedef struct {
  const uint16_t *attn_norm, *wq, *wk, *wv, *bq, *bk, *bv, *wo, *mlp_norm, *w_gate, *w_up, *w_down;
} orc_layer;

/* ---- building blocks (exported so that the tests can pin each one) ---- */

/* bf16 <-> fp32.  orc_f32_to_bf16 rounds to nearest, ties to even (NaN kept quiet). */
float orc_bf16_to_f32(uint16_t b);
uint16_t orc_f32_to_bf16(float f);

/* out[i] = x[i] / sqrt(mean(x^2) + eps) * g[i]   (g == NULL means a gain of 1). */
void orc_rmsnorm(const float *x, const uint16_t *g, int n, double eps, float *out);

/* y[r] = sum_k W[r,k] x[k] (+ b[r])  for r < rows.  W bf16 [rows, cols], b bf16 or NULL. */
void orc_gemv(const uint16_t *W, const float *x, const uint16_t *b, int rows, int cols, float *y, int nthreads);

/* Rotary embedding, rotate-half convention: for each of n_heads vectors of length d and
 * each i < d/2, (v[i], v[i+d/2]) is rotated by the angle pos * theta^(-2i/d). */
void orc_rope(float *v, int n_heads, int d, int pos, double theta);

/* Decode attention for one layer.  q: [nq][d] fp32 (post-RoPE).  K, V: bf16 caches of
 * one layer laid out [nkv][cap][d].  Query head h reads kv head h / (nq/nkv), keys
 * j = 0..ctx-1; scores q.K_j / sqrt(d), softmax over j, o_h = sum_j a_j V_j.  o: [nq][d]. */
void orc_attention(const float *q, const uint16_t *K, const uint16_t *V, int nq, int nkv, int d, int cap, int ctx,
                   float *o, int nthreads);

/* h[i] = silu(g[i]) * u[i],  silu(z) = z / (1 + exp(-z)). */
void orc_silu_mul(const float *g, const float *u, int n, float *h);

/* Write cache rows p0..p0+n-1 of one layer from pre-RoPE K and V (fp32, [nkv][n][d]):
 * K is rotated by its position, both are rounded to bf16.  kv_layer points at the
 * layer's [2][nkv][cap][d] block. */
void orc_kv_fill(const orc_config *cfg, uint16_t *kv_layer, const float *k_raw, const float *v_raw, int p0, int n);

/* ---- the whole decode step ----
 * Embeds `token`, runs every layer at position `pos` (writing cache row `pos` of every
 * layer, attending over rows 0..pos), applies the final norm and the tied vocabulary
 * projection.  kv_cache: bf16 [L][2][nkv][cap][d] (K then V per layer).  logits: fp32 [V].
 * taps (optional, may be NULL): fp32 [(2L+1)][H], the residual stream after the embedding
 * and after each attention and MLP sublayer.  nthreads <= 0 uses every core OpenMP offers.
 * Returns 0, or -1 for an invalid argument (nothing is written then). */
int orc_decode_step(const orc_config *cfg, const uint16_t *embed, const uint16_t *final_norm, const orc_layer *layers,
                    uint16_t *kv_cache, int token, int pos, float *logits, float *taps, int nthreads);

/* ---- FP8 weights (opt-in weight format; the MegaBake website lists FP8 under "Next") ----
 * The pages name FP8 weight streaming but fix no format; the reading taken here: OCP FP8 E4M3
 * (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN;
 * largest finite 448, smallest normal 2^-6, subnormals m * 2^-9) with one fp32 scale per output
 * row.  Row r of a bf16 matrix W: amax = max_k |W[r,k]|; s = amax / 448 in fp32 (1 for an all-zero
 * row); q[r,k] = E4M3(W[r,k] / s), the fp32 quotient rounded to the nearest code, ties to the even
 * code, magnitudes above 448 saturating to 448.  A projection over such a row is
 * y[r] = s * sum_k E4M3value(q[r,k]) x[k] (+ bias): the scale applies to the exact sum.
 * Which weights: every layer's Wq, Wk, Wv, Wo, Wgate, Wup, Wdown and the LM head's copy of E; the
 * embedding lookup, norm gains and biases stay bf16.  Parity pins: exact codes of hand-computed
 * values, ties, saturation, the round trip of every finite code, and the row maximum mapping to 448. */
uint8_t orc_fp8_from_f32(float f);
float orc_fp8_to_f32(uint8_t c);
/* q: [rows][cols] codes, s: [rows] scales. */
void orc_quantize_fp8(const uint16_t *W, int rows, int cols, uint8_t *q, float *s);
/* y[r] = s[r] * sum_k value(Q[r,k]) x[k] (+ b[r]), accumulated in double, stored as fp32. */
void orc_gemv_fp8(const uint8_t *Q, const float *s, const float *x, const uint16_t *b, int rows, int cols, float *y,
                  int nthreads);

/* The FP8 copies of one layer's projections, in the order Wq, Wk, Wv, Wo, Wgate, Wup, Wdown. */
typedef struct {
  const uint8_t *q[7];
  const float *s[7];
} orc_fp8_layer;
typedef struct {
  const orc_fp8_layer *layers;  /* [L] */
  const uint8_t *lm_q;          /* [V][H]: the LM head's copy of E */
  const float *lm_s;            /* [V] */
} orc_fp8_weights;

/* orc_decode_step with every projection and the LM head on FP8 weights (the embedding row, the
 * norms and the biases still come from the bf16 tensors). */
int orc_decode_step_fp8(const orc_config *cfg, const uint16_t *embed, const uint16_t *final_norm, const orc_layer *layers,
                        const orc_fp8_weights *fp8, uint16_t *kv_cache, int token, int pos, float *logits, float *taps,
                        int nthreads);

/* ---- prefill: n given tokens at positions p0 .. p0 + n - 1 (its plain definition) ----
 * The pages give prefill no computation of its own (the article, "Where it loses", only measures the
 * megakernel's prefill path), so this is the teacher-forced decode of the n tokens written
 * layer-major: each layer takes all n tokens, appends all their K/V rows, then token t attends over
 * the cache rows 0 .. p0 + t through an explicit causal mask on the scores of every key up to
 * p0 + n - 1 (masked scores are -inf, so they add exact zeros).  Every other op is the decode step's.
 * logits: fp32 [n][V], or NULL (cache only).  Returns 0, or -1 for an invalid argument.
 * Pin: equals n calls of orc_decode_step bit for bit (logits and cache). */
int orc_prefill(const orc_config *cfg, const uint16_t *embed, const uint16_t *final_norm, const orc_layer *layers,
                uint16_t *kv_cache, const int32_t *tokens, int n, int p0, float *logits, int nthreads);

/* Number of OpenMP threads the oracle would use for nthreads <= 0 (1 without OpenMP). */
int orc_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif
