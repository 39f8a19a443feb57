// mbk_sched.h -- host-side static scheduler: turns a decoder shape into per-CTA task lists.
#pragma once
#include <stdint.h>

#include <array>
#include <string>
#include <vector>

#include "mbk_plan.h"

namespace mbk {

// Device addresses of the weights (as integers, so the scheduler can also run on fake addresses).
enum WeightSlot { W_ATTN_NORM, W_Q, W_K, W_V, W_BQ, W_BK, W_BV, W_O, W_MLP_NORM, W_GATE, W_UP, W_DOWN, W_NSLOTS };
struct WeightAddrs {
  uint64_t embed = 0, final_norm = 0;
  uint64_t lm_head = 0;  // rows the LM head streams: the embedding (bf16) or its FP8 copy; 0 = embed
  std::vector<std::array<uint64_t, W_NSLOTS>> layers;
};

struct PlanOptions {
  int max_tasks_per_op = 0;    // split each projection into at most this many tasks (0: one per CTA)
  int fuse_attention = -1;     // fold the O projection into the attention tasks: -1 where it applies, 0 never
  int smem_limit = 232448;     // dynamic shared memory available per CTA
  int attn_mma = 1;            // attention on the tensor cores where the shape allows (0: never)
  int attn_split = 0;          // longest attention split in positions (0: kAttnSplitMax; else a multiple of 64)
  int combine_tasks = 0;       // O-projection tasks of a split context (each polls every split's outputs);
                               // 0: one per kCombineRows output rows
};

struct Plan {
  int num_ctas = 0;
  std::vector<Task> tasks;           // every CTA's tasks, CTA-major
  std::vector<uint32_t> task_off;    // [num_ctas + 1] offsets into tasks
  std::vector<Chunk> chunks;         // weight chunks and attention placeholders (Task::chunk0), CTA-major
  std::vector<uint32_t> chunk_off;   // [num_ctas + 1] offsets into chunks
  ActLayout act{};
  uint64_t act_words = 0;            // words per step (one parity)
  bool fused_attn = false;           // attention tasks also apply Wo (TF_WO); no O-projection tasks
  bool attn_mma = false;             // attention on the tensor cores (head_dim 64, g <= 8; ring 1024-aligned)
  int nsplit = 1;                    // context splits per KV head
  int split_len = 0;                 // positions per split
  int combine_group = 1;             // splits whose o words one poll of the split combine brings
  int attn_rows_per_stage = 0;       // cached positions per ring stage
  int num_stages = 0;
  int smem_bytes = 0;
  int sv_floats = 0;                 // floats in the input-vector region
  int max_cta_tasks = 0;             // tasks of the busiest CTA (records staged in shared memory, kTaskWindow at a time)
  uint32_t off_sv = 0, off_res = 0, off_resid = 0, off_tasks = 0, off_ring = 0;  // shared-memory layout (bytes)
  int64_t weight_bytes = 0;          // static chunk bytes per step
  int64_t max_cta_bytes = 0;
};

// Returns an empty string on success, otherwise the reason the shape is unsupported.
std::string validate_shape(const PlanShape& s);

// Builds the plan.  Returns "" or an error message.
std::string build_plan(const PlanShape& s, const WeightAddrs& w, int num_ctas, const PlanOptions& opt, Plan* out);

// Independent consistency checks of a built plan (coverage of every weight row exactly once,
// per-CTA task order, copy alignment and bounds, stage and result capacities).
std::string check_plan(const PlanShape& s, const WeightAddrs& w, const Plan& p);

// Fake, well-separated weight addresses for planning without device memory.
WeightAddrs fake_weight_addrs(const PlanShape& s);

}  // namespace mbk
