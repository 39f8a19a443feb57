/*
 * mbk_oracle.c -- plain CPU reference of batch-1 Llama-shaped decode.
 * TEST INFRASTRUCTURE ONLY (see mbk_oracle.h): the product path never links or calls it.
 *
 * Written for readability, not speed: one output element per loop iteration, double
 * accumulation, no blocking or fusion beyond what each op's definition states.  OpenMP
 * (when compiled in) only splits independent output rows or heads across threads, so the
 * result does not depend on the thread count.
 */
#include "mbk_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

static int threads_for(int nthreads) { return nthreads > 0 ? nthreads : orc_max_threads(); }

/* bf16 is the upper half of an IEEE binary32. */
float orc_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

uint16_t orc_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0) /* NaN: keep it a quiet NaN */
    return (uint16_t)((u >> 16) | 0x0040u);
  /* round to nearest, ties to even: add 0x7fff plus the lowest kept bit, then truncate */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

/* RMSNorm (article, "How a model gets in": the rms_norm region; Hugging Face Llama
 * definition): x / sqrt(mean(x^2) + eps) * gain. */
void orc_rmsnorm(const float *x, const uint16_t *g, int n, double eps, float *out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += (double)x[i] * (double)x[i];
  double inv = 1.0 / sqrt(ss / (double)n + eps);
  for (int i = 0; i < n; ++i) {
    double gi = g ? (double)orc_bf16_to_f32(g[i]) : 1.0;
    out[i] = (float)((double)x[i] * inv * gi);
  }
}

/* A projection at batch 1 is a matrix-vector product over the [out, in] weight; the
 * q/k/v bias (README, "Current status": addmm biases) is added to the exact sum. */
void orc_gemv(const uint16_t *W, const float *x, const uint16_t *b, int rows, int cols, float *y, int nthreads) {
  int nt = threads_for(nthreads);
  (void)nt;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nt) schedule(static)
#endif
  for (int r = 0; r < rows; ++r) {
    const uint16_t *w = W + (size_t)r * cols;
    double acc = 0.0;
    for (int k = 0; k < cols; ++k) acc += (double)orc_bf16_to_f32(w[k]) * (double)x[k];
    if (b) acc += (double)orc_bf16_to_f32(b[r]);
    y[r] = (float)acc;
  }
}

/* E4M3 value of a code, from the format's definition. */
float orc_fp8_to_f32(uint8_t c) {
  const int e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);           /* subnormal: m/8 * 2^-6 */
  else
    v = ldexp(1.0 + m / 8.0, e - 7);    /* normal */
  return (float)((c & 0x80) ? -v : v);
}

/* Nearest code to f (ties to the even code), saturating at 448: the non-negative finite codes
 * 0x00..0x7E are increasing in value, so the nearest is found between the two codes that
 * bracket |f|. */
static double fp8_value[0x7F]; /* the non-negative finite codes' values (filled once) */
static int fp8_value_ready = 0;

uint8_t orc_fp8_from_f32(float f) {
  if (!fp8_value_ready) {
    for (int c = 0; c < 0x7F; ++c) fp8_value[c] = orc_fp8_to_f32((uint8_t)c);
    fp8_value_ready = 1;
  }
  if (isnan(f)) return 0x7F;
  const uint8_t sign = signbit(f) ? 0x80 : 0x00;
  const double a = fabs((double)f);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  int lo = 0, hi = 0x7E; /* largest code with value <= a */
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (fp8_value[mid] <= a) lo = mid; else hi = mid - 1;
  }
  const double vlo = fp8_value[lo], vhi = fp8_value[lo + 1];
  int c;
  if (a - vlo < vhi - a) c = lo;
  else if (a - vlo > vhi - a) c = lo + 1;
  else c = (lo % 2 == 0) ? lo : lo + 1;
  return (uint8_t)(sign | c);
}

void orc_quantize_fp8(const uint16_t *W, int rows, int cols, uint8_t *q, float *s) {
  for (int r = 0; r < rows; ++r) {
    const uint16_t *w = W + (size_t)r * cols;
    float amax = 0.0f;
    for (int k = 0; k < cols; ++k) {
      const float a = fabsf(orc_bf16_to_f32(w[k]));
      if (a > amax) amax = a;
    }
    const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
    s[r] = sc;
    for (int k = 0; k < cols; ++k) q[(size_t)r * cols + k] = orc_fp8_from_f32(orc_bf16_to_f32(w[k]) / sc);
  }
}

void orc_gemv_fp8(const uint8_t *Q, const float *s, const float *x, const uint16_t *b, int rows, int cols, float *y,
                  int nthreads) {
  int nt = threads_for(nthreads);
  (void)nt;
  float lut[256];
  for (int c = 0; c < 256; ++c) lut[c] = orc_fp8_to_f32((uint8_t)c);
#ifdef _OPENMP
#pragma omp parallel for num_threads(nt) schedule(static)
#endif
  for (int r = 0; r < rows; ++r) {
    const uint8_t *w = Q + (size_t)r * cols;
    double acc = 0.0;
    for (int k = 0; k < cols; ++k) acc += (double)lut[w[k]] * (double)x[k];
    acc *= (double)s[r];
    if (b != NULL) acc += (double)orc_bf16_to_f32(b[r]);  /* the bias is not quantized */
    y[r] = (float)acc;
  }
}

/* RoPE (article, "How a model gets in": the rope region).  Rotate-half pairing as in
 * Hugging Face Llama: element i pairs with element i + d/2, frequency theta^(-2i/d). */
void orc_rope(float *v, int n_heads, int d, int pos, double theta) {
  int half = d / 2;
  for (int h = 0; h < n_heads; ++h) {
    float *x = v + (size_t)h * d;
    for (int i = 0; i < half; ++i) {
      double inv_freq = pow(theta, -(2.0 * (double)i) / (double)d);
      double ang = (double)pos * inv_freq;
      double c = cos(ang), s = sin(ang);
      double a = x[i], b = x[i + half];
      x[i] = (float)(a * c - b * s);
      x[i + half] = (float)(b * c + a * s);
    }
  }
}

/* Decode attention over the static cache (README, "Current status": decode attention with
 * the query heads that share a KV head reading the same cached keys and values).
 * Plain softmax(q K^T / sqrt(d)) V per query head, with the maximum subtracted. */
void orc_attention(const float *q, const uint16_t *K, const uint16_t *V, int nq, int nkv, int d, int cap, int ctx,
                   float *o, int nthreads) {
  int group = nq / nkv;
  int nt = threads_for(nthreads);
  (void)nt;
  double scale = 1.0 / sqrt((double)d);
#ifdef _OPENMP
#pragma omp parallel for num_threads(nt) schedule(static)
#endif
  for (int h = 0; h < nq; ++h) {
    int kv = h / group;
    const float *qh = q + (size_t)h * d;
    const uint16_t *Kh = K + (size_t)kv * cap * d;
    const uint16_t *Vh = V + (size_t)kv * cap * d;
    double *s = (double *)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1));
    double m = -INFINITY;
    for (int j = 0; j < ctx; ++j) {
      double acc = 0.0;
      for (int t = 0; t < d; ++t) acc += (double)qh[t] * (double)orc_bf16_to_f32(Kh[(size_t)j * d + t]);
      s[j] = acc * scale;
      if (s[j] > m) m = s[j];
    }
    double z = 0.0;
    for (int j = 0; j < ctx; ++j) {
      s[j] = exp(s[j] - m);
      z += s[j];
    }
    for (int t = 0; t < d; ++t) {
      double acc = 0.0;
      for (int j = 0; j < ctx; ++j) acc += s[j] * (double)orc_bf16_to_f32(Vh[(size_t)j * d + t]);
      o[(size_t)h * d + t] = ctx > 0 ? (float)(acc / z) : 0.0f;
    }
    free(s);
  }
}

/* Gated activation (article, "How a model gets in": the fused SiLU-mul region). */
void orc_silu_mul(const float *g, const float *u, int n, float *h) {
  for (int i = 0; i < n; ++i) {
    double z = g[i];
    double silu = z / (1.0 + exp(-z));
    h[i] = (float)(silu * (double)u[i]);
  }
}

void orc_kv_fill(const orc_config *cfg, uint16_t *kv_layer, const float *k_raw, const float *v_raw, int p0, int n) {
  int nkv = cfg->n_kv_heads, d = cfg->head_dim, cap = cfg->kv_capacity;
  uint16_t *Kc = kv_layer;
  uint16_t *Vc = kv_layer + (size_t)nkv * cap * d;
  float *tmp = (float *)malloc(sizeof(float) * (size_t)d);
  for (int h = 0; h < nkv; ++h) {
    for (int i = 0; i < n; ++i) {
      int p = p0 + i;
      const float *kr = k_raw + ((size_t)h * n + i) * d;
      const float *vr = v_raw + ((size_t)h * n + i) * d;
      memcpy(tmp, kr, sizeof(float) * (size_t)d);
      orc_rope(tmp, 1, d, p, cfg->rope_theta);
      for (int t = 0; t < d; ++t) {
        Kc[((size_t)h * cap + p) * d + t] = orc_f32_to_bf16(tmp[t]);
        Vc[((size_t)h * cap + p) * d + t] = orc_f32_to_bf16(vr[t]);
      }
    }
  }
  free(tmp);
}

static int config_ok(const orc_config *c) {
  if (c->n_layers <= 0 || c->hidden <= 0 || c->intermediate <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0) return 0;
  if (c->head_dim <= 0 || (c->head_dim % 2) != 0 || c->vocab <= 0 || c->kv_capacity <= 0) return 0;
  if (c->n_heads % c->n_kv_heads != 0) return 0;
  return 1;
}

/* One decode step, in the order the article's section "What a megakernel is, and why small
 * models want one" lists the ops, with the embedding at the start and the final norm and
 * tied vocabulary projection at the end (README, "Current status"). */
/* A projection of the step: on the bf16 weight, or on its FP8 copy when there is one. */
static void project(const uint16_t *W, const orc_fp8_layer *f8, int slot, const float *x, const uint16_t *b, int rows,
                    int cols, float *y, int nthreads) {
  if (f8)
    orc_gemv_fp8(f8->q[slot], f8->s[slot], x, b, rows, cols, y, nthreads);
  else
    orc_gemv(W, x, b, rows, cols, y, nthreads);
}

static int decode_step(const orc_config *cfg, const uint16_t *embed, const uint16_t *final_norm, const orc_layer *layers,
                       const orc_fp8_weights *fp8, uint16_t *kv_cache, int token, int pos, float *logits, float *taps,
                       int nthreads);

int orc_decode_step(const orc_config *cfg, const uint16_t *embed, const uint16_t *final_norm, const orc_layer *layers,
                    uint16_t *kv_cache, int token, int pos, float *logits, float *taps, int nthreads) {
  return decode_step(cfg, embed, final_norm, layers, NULL, kv_cache, token, pos, logits, taps, nthreads);
}

int orc_decode_step_fp8(const orc_config *cfg, const uint16_t *embed, const uint16_t *final_norm, const orc_layer *layers,
                        const orc_fp8_weights *fp8, uint16_t *kv_cache, int token, int pos, float *logits, float *taps,
                        int nthreads) {
  if (!fp8 || !fp8->layers || !fp8->lm_q || !fp8->lm_s) return -1;
  return decode_step(cfg, embed, final_norm, layers, fp8, kv_cache, token, pos, logits, taps, nthreads);
}

static int decode_step(const orc_config *cfg, const uint16_t *embed, const uint16_t *final_norm, const orc_layer *layers,
                       const orc_fp8_weights *fp8, uint16_t *kv_cache, int token, int pos, float *logits, float *taps,
                       int nthreads) {
  if (!cfg || !embed || !layers || !kv_cache || !logits || !config_ok(cfg)) return -1;
  if (token < 0 || token >= cfg->vocab || pos < 0 || pos >= cfg->kv_capacity) return -1;
  const int L = cfg->n_layers, H = cfg->hidden, I = cfg->intermediate;
  const int nq = cfg->n_heads, nkv = cfg->n_kv_heads, d = cfg->head_dim, cap = cfg->kv_capacity;
  const size_t qdim = (size_t)nq * d, kvdim = (size_t)nkv * d;

  float *x = (float *)malloc(sizeof(float) * H);
  float *xn = (float *)malloc(sizeof(float) * H);
  float *y = (float *)malloc(sizeof(float) * H);
  float *q = (float *)malloc(sizeof(float) * qdim);
  float *k = (float *)malloc(sizeof(float) * kvdim);
  float *v = (float *)malloc(sizeof(float) * kvdim);
  float *o = (float *)malloc(sizeof(float) * qdim);
  float *g = (float *)malloc(sizeof(float) * I);
  float *u = (float *)malloc(sizeof(float) * I);
  float *hbuf = (float *)malloc(sizeof(float) * I);

  /* embedding: the token's row of E, widened to fp32 */
  for (int i = 0; i < H; ++i) x[i] = orc_bf16_to_f32(embed[(size_t)token * H + i]);
  if (taps) memcpy(taps, x, sizeof(float) * H);

  for (int l = 0; l < L; ++l) {
    const orc_layer *w = &layers[l];
    const orc_fp8_layer *f8 = fp8 ? &fp8->layers[l] : NULL;
    uint16_t *Kc = kv_cache + (size_t)l * 2 * nkv * cap * d;
    uint16_t *Vc = Kc + (size_t)nkv * cap * d;

    /* attention sublayer */
    orc_rmsnorm(x, w->attn_norm, H, cfg->rms_eps, xn);
    project(w->wq, f8, 0, xn, cfg->qkv_bias ? w->bq : NULL, nq * d, H, q, nthreads);
    project(w->wk, f8, 1, xn, cfg->qkv_bias ? w->bk : NULL, nkv * d, H, k, nthreads);
    project(w->wv, f8, 2, xn, cfg->qkv_bias ? w->bv : NULL, nkv * d, H, v, nthreads);
    orc_rope(q, nq, d, pos, cfg->rope_theta);
    orc_rope(k, nkv, d, pos, cfg->rope_theta);
    for (int h = 0; h < nkv; ++h)
      for (int t = 0; t < d; ++t) {
        Kc[((size_t)h * cap + pos) * d + t] = orc_f32_to_bf16(k[(size_t)h * d + t]);
        Vc[((size_t)h * cap + pos) * d + t] = orc_f32_to_bf16(v[(size_t)h * d + t]);
      }
    orc_attention(q, Kc, Vc, nq, nkv, d, cap, pos + 1, o, nthreads);
    project(w->wo, f8, 3, o, NULL, H, nq * d, y, nthreads);
    for (int i = 0; i < H; ++i) x[i] = (float)((double)x[i] + (double)y[i]);
    if (taps) memcpy(taps + (size_t)(2 * l + 1) * H, x, sizeof(float) * H);

    /* MLP sublayer */
    orc_rmsnorm(x, w->mlp_norm, H, cfg->rms_eps, xn);
    project(w->w_gate, f8, 4, xn, NULL, I, H, g, nthreads);
    project(w->w_up, f8, 5, xn, NULL, I, H, u, nthreads);
    orc_silu_mul(g, u, I, hbuf);
    project(w->w_down, f8, 6, hbuf, NULL, H, I, y, nthreads);
    for (int i = 0; i < H; ++i) x[i] = (float)((double)x[i] + (double)y[i]);
    if (taps) memcpy(taps + (size_t)(2 * l + 2) * H, x, sizeof(float) * H);
  }

  /* final norm, then the tied vocabulary projection (the embedding matrix) */
  orc_rmsnorm(x, final_norm, H, cfg->rms_eps, xn);
  if (fp8)
    orc_gemv_fp8(fp8->lm_q, fp8->lm_s, xn, NULL, cfg->vocab, H, logits, nthreads);
  else
    orc_gemv(embed, xn, NULL, cfg->vocab, H, logits, nthreads);

  free(x); free(xn); free(y); free(q); free(k); free(v); free(o); free(g); free(u); free(hbuf);
  return 0;
}

/* Causal attention of the n tokens of a prefill at one layer: token t (position p0 + t) scores every
 * key 0 .. p0 + n - 1 and masks keys above its own position with -inf before the softmax. */
static void causal_attention(const float *q, const uint16_t *K, const uint16_t *V, int nq, int nkv, int d, int cap,
                             int n, int p0, float *o) {
  const int group = nq / nkv, nkeys = p0 + n;
  const double scale = 1.0 / sqrt((double)d);
  double *sc = (double *)malloc(sizeof(double) * (size_t)nkeys);
  for (int t = 0; t < n; ++t)
    for (int h = 0; h < nq; ++h) {
      const float *qh = q + ((size_t)t * nq + h) * d;
      const uint16_t *Kh = K + (size_t)(h / group) * cap * d;
      const uint16_t *Vh = V + (size_t)(h / group) * cap * d;
      double m = -INFINITY;
      for (int j = 0; j < nkeys; ++j) {
        if (j > p0 + t) {
          sc[j] = -INFINITY; /* the causal mask */
          continue;
        }
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += (double)qh[i] * (double)orc_bf16_to_f32(Kh[(size_t)j * d + i]);
        sc[j] = acc * scale;
        if (sc[j] > m) m = sc[j];
      }
      double z = 0.0;
      for (int j = 0; j < nkeys; ++j) {
        sc[j] = exp(sc[j] - m); /* exp(-inf) = 0 for masked keys */
        z += sc[j];
      }
      for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int j = 0; j < nkeys; ++j) acc += sc[j] * (double)orc_bf16_to_f32(Vh[(size_t)j * d + i]);
        o[((size_t)t * nq + h) * d + i] = (float)(acc / z);
      }
    }
  free(sc);
}

int orc_prefill(const orc_config *cfg, const uint16_t *embed, const uint16_t *final_norm, const orc_layer *layers,
                uint16_t *kv_cache, const int32_t *tokens, int n, int p0, float *logits, int nthreads) {
  if (!cfg || !embed || !layers || !kv_cache || !tokens || !config_ok(cfg) || n < 1 || p0 < 0 ||
      p0 > cfg->kv_capacity - n)
    return -1;
  for (int t = 0; t < n; ++t)
    if (tokens[t] < 0 || tokens[t] >= cfg->vocab) return -1;
  const int L = cfg->n_layers, H = cfg->hidden, I = cfg->intermediate;
  const int nq = cfg->n_heads, nkv = cfg->n_kv_heads, d = cfg->head_dim, cap = cfg->kv_capacity;
  const size_t qdim = (size_t)nq * d, kvdim = (size_t)nkv * d;
  float *x = (float *)malloc(sizeof(float) * (size_t)n * H);
  float *q = (float *)malloc(sizeof(float) * (size_t)n * qdim);
  float *o = (float *)malloc(sizeof(float) * (size_t)n * qdim);
  float *xn = (float *)malloc(sizeof(float) * H);
  float *y = (float *)malloc(sizeof(float) * H);
  float *kr = (float *)malloc(sizeof(float) * kvdim);
  float *vr = (float *)malloc(sizeof(float) * kvdim);
  float *gt = (float *)malloc(sizeof(float) * I);
  float *ut = (float *)malloc(sizeof(float) * I);
  float *ht = (float *)malloc(sizeof(float) * I);

  for (int t = 0; t < n; ++t)
    for (int i = 0; i < H; ++i) x[(size_t)t * H + i] = orc_bf16_to_f32(embed[(size_t)tokens[t] * H + i]);
  for (int l = 0; l < L; ++l) {
    const orc_layer *w = &layers[l];
    uint16_t *Kc = kv_cache + (size_t)l * 2 * nkv * cap * d;
    uint16_t *Vc = Kc + (size_t)nkv * cap * d;
    /* every token's projections and cache rows first */
    for (int t = 0; t < n; ++t) {
      const int pos = p0 + t;
      float *qt = q + (size_t)t * qdim;
      orc_rmsnorm(x + (size_t)t * H, w->attn_norm, H, cfg->rms_eps, xn);
      orc_gemv(w->wq, xn, cfg->qkv_bias ? w->bq : NULL, nq * d, H, qt, nthreads);
      orc_gemv(w->wk, xn, cfg->qkv_bias ? w->bk : NULL, nkv * d, H, kr, nthreads);
      orc_gemv(w->wv, xn, cfg->qkv_bias ? w->bv : NULL, nkv * d, H, vr, nthreads);
      orc_rope(qt, nq, d, pos, cfg->rope_theta);
      orc_rope(kr, nkv, d, pos, cfg->rope_theta);
      for (int h = 0; h < nkv; ++h)
        for (int i = 0; i < d; ++i) {
          Kc[((size_t)h * cap + pos) * d + i] = orc_f32_to_bf16(kr[(size_t)h * d + i]);
          Vc[((size_t)h * cap + pos) * d + i] = orc_f32_to_bf16(vr[(size_t)h * d + i]);
        }
    }
    causal_attention(q, Kc, Vc, nq, nkv, d, cap, n, p0, o);
    for (int t = 0; t < n; ++t) {
      float *xt = x + (size_t)t * H;
      orc_gemv(w->wo, o + (size_t)t * qdim, NULL, H, nq * d, y, nthreads);
      for (int i = 0; i < H; ++i) xt[i] = (float)((double)xt[i] + (double)y[i]);
      orc_rmsnorm(xt, w->mlp_norm, H, cfg->rms_eps, xn);
      orc_gemv(w->w_gate, xn, NULL, I, H, gt, nthreads);
      orc_gemv(w->w_up, xn, NULL, I, H, ut, nthreads);
      orc_silu_mul(gt, ut, I, ht);
      orc_gemv(w->w_down, ht, NULL, H, I, y, nthreads);
      for (int i = 0; i < H; ++i) xt[i] = (float)((double)xt[i] + (double)y[i]);
    }
  }
  if (logits)
    for (int t = 0; t < n; ++t) {
      orc_rmsnorm(x + (size_t)t * H, final_norm, H, cfg->rms_eps, xn);
      orc_gemv(embed, xn, NULL, cfg->vocab, H, logits + (size_t)t * cfg->vocab, nthreads);
    }
  free(x); free(q); free(o); free(xn); free(y); free(kr); free(vr); free(gt); free(ut); free(ht);
  return 0;
}
