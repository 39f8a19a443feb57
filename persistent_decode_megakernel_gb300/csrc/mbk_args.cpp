// mbk_args.cpp -- argument checks shared by the C ABI's entry points (see mbk_args.h).
#include "mbk_args.h"

#include <cmath>
#include <cstdlib>

namespace mbk {

namespace {
bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
}  // namespace

PlanShape shape_of(const mbk_config& c) {
  PlanShape s;
  s.L = c.n_layers;
  s.H = c.hidden;
  s.I = c.intermediate;
  s.nq = c.n_heads;
  s.nkv = c.n_kv_heads;
  s.d = c.head_dim;
  s.V = c.vocab;
  s.C = c.kv_capacity;
  s.qkv_bias = c.qkv_bias ? 1 : 0;
  s.wb = c.weight_format == MBK_WEIGHTS_FP8 ? 1 : 2;
  return s;
}

int config_check(const mbk_config* cfg) {
  if (!cfg) return MBK_ERR_INVALID_ARG;
  if (!(cfg->rms_eps >= 0.0) || !std::isfinite(cfg->rms_eps)) return MBK_ERR_INVALID_ARG;
  if (!(cfg->rope_theta > 0.0) || !std::isfinite(cfg->rope_theta)) return MBK_ERR_INVALID_ARG;
  if (cfg->weight_format != MBK_WEIGHTS_BF16 && cfg->weight_format != MBK_WEIGHTS_FP8) return MBK_ERR_INVALID_ARG;
  if (!validate_shape(shape_of(*cfg)).empty()) return MBK_ERR_INVALID_ARG;
  return MBK_OK;
}

int gather_weights(const mbk_config* cfg, const mbk_weights* weights, const void* kv_cache, WeightAddrs* out) {
  if (config_check(cfg) != MBK_OK || !weights || !weights->embed || !weights->final_norm || !weights->layers || !kv_cache ||
      !out)
    return MBK_ERR_INVALID_ARG;
  if (!aligned16(weights->embed) || !aligned16(weights->final_norm) || !aligned16(kv_cache)) return MBK_ERR_INVALID_ARG;
  const PlanShape s = shape_of(*cfg);
  WeightAddrs& wa = *out;
  wa = WeightAddrs();
  wa.embed = (uint64_t)(uintptr_t)weights->embed;
  wa.final_norm = (uint64_t)(uintptr_t)weights->final_norm;
  wa.layers.resize(s.L);
  for (int l = 0; l < s.L; ++l) {
    const mbk_layer_weights& lw = weights->layers[l];
    const void* ptrs[W_NSLOTS] = {lw.attn_norm, lw.wq, lw.wk, lw.wv, lw.bq, lw.bk, lw.bv, lw.wo, lw.mlp_norm, lw.w_gate, lw.w_up, lw.w_down};
    for (int k = 0; k < W_NSLOTS; ++k) {
      const bool is_bias = (k == W_BQ || k == W_BK || k == W_BV);
      if (is_bias && !s.qkv_bias) {
        wa.layers[l][k] = 0;
        continue;
      }
      if (!ptrs[k]) return MBK_ERR_INVALID_ARG;
      if (!is_bias && k != W_ATTN_NORM && k != W_MLP_NORM && !aligned16(ptrs[k])) return MBK_ERR_INVALID_ARG;
      wa.layers[l][k] = (uint64_t)(uintptr_t)ptrs[k];
    }
  }
  return MBK_OK;
}

int env_int(const char* name, int dflt) {
  const char* v = getenv(name);
  if (!v || !*v) return dflt;
  return atoi(v);
}

}  // namespace mbk
