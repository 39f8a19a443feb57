// mbk_args.h -- argument checks shared by every entry point that takes a config and weights
// (mbk_create, mbk_create_paged, mbk_plan_check, mbk_decode_step_static).  Host code only.
#pragma once
#include <stdint.h>

#include "../../include/mbk.h"
#include "mbk_sched.h"

namespace mbk {

// The scheduler's view of a config.
PlanShape shape_of(const mbk_config& c);

// MBK_OK, or MBK_ERR_INVALID_ARG for a null config, a non-finite or non-positive RoPE theta, a
// negative or non-finite RMSNorm epsilon, an unknown weight format, or a shape the scheduler
// rejects (validate_shape).
int config_check(const mbk_config* cfg);

// Checks the config (config_check), then every tensor pointer: the embedding, the final norm gain,
// the KV cache and every projection weight present and 16-byte aligned (they are streamed with
// 16-byte bulk copies and 128-bit loads), the norm gains and (qkv_bias) the q/k/v biases present.
// Fills `out` with the addresses (biases 0 when the config has none).  MBK_OK or
// MBK_ERR_INVALID_ARG; touches no GPU.
int gather_weights(const mbk_config* cfg, const mbk_weights* weights, const void* kv_cache, WeightAddrs* out);

// An integer environment knob, or `dflt` when unset or empty.
int env_int(const char* name, int dflt);

}  // namespace mbk
