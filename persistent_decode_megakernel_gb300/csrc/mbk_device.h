// mbk_device.h -- parameters of the persistent decode kernel (shared by mbk_kernel.cu and mbk_api.cu).
#pragma once
#include <stdint.h>

#include "mbk_plan.h"

namespace mbk {

// Device status word values (host maps them to the negative MBK_ERR_* codes).
enum DeviceStatus : unsigned { DS_OK = 0, DS_TIMEOUT = 4 };

// Per-layer weight pointers, in the order of WeightSlot (mbk_sched.h); bf16 bit patterns.
enum LayerSlot { LW_ATTN_NORM, LW_Q, LW_K, LW_V, LW_BQ, LW_BK, LW_BV, LW_O, LW_MLP_NORM, LW_GATE, LW_UP, LW_DOWN };
struct LayerW {
  const uint16_t* w[12];
};

// Constant for the lifetime of a handle (4-byte multiple, copied word by word into shared memory).
struct KernelParams {
  int L, H, I, nq, nkv, d, V, C, g;
  float eps, attn_scale, inv_H;  // inv_H = 1/H rounded to fp32
  int qkv_bias;
  // schedule
  const Task* tasks;
  const uint32_t* task_off;     // [grid + 1]
  const Chunk* chunks;
  const uint32_t* chunk_off;    // [grid + 1]
  ActLayout act;
  int nsplit, split_len, rows_per_stage, num_stages;
  int combine_group;            // split combine: splits whose o words one poll brings (<= nsplit)
  uint32_t off_sv, off_res, off_resid, off_tasks, off_ring;
  // tensors
  const uint16_t* embed;
  const uint16_t* final_norm;
  const LayerW* layers;
  uint16_t* kv;                 // the KV cache (layout below)
  const float2* rope;           // [C][d/2] (cos, sin)
  unsigned long long* words;    // activation exchange words [L * act.per_layer]
  unsigned* status;             // device status [4]: code, cta, task, detail
  unsigned* host_status;        // the same, in mapped pinned host memory (may be null)
  unsigned long long timeout_ns;
  unsigned long long* trace;    // null, or 4 globaltimer stamps per task (begin, ready, end, first stage)
  const unsigned long long* inject;  // null, or words [L][H]: row l replaces the input of layer l >= 1
  unsigned poll_backoff_ns;     // sleep between polls of a word that is not ready yet (0: none)
  int lm_tasks;                 // LM-head tasks of a step (greedy decoding: contributions to its argmax)
  // KV-cache layout.  Contiguous (page_table null): [L][2][nkv][C][d], page_size = C.  Paged: a pool
  // of pages, each [L][2][nkv][page_size][d]; page_table[q] is the page that holds positions
  // q * page_size ..; page_size is a power of two (page_shift its log2) and the table has at most
  // kMaxPages entries (copied into shared memory at kernel start).
  const int32_t* page_table;
  int page_size, page_shift;
  unsigned long long page_elems;  // bf16 elements of one page: L * 2 * nkv * page_size * d
  // Attention on the tensor cores (head_dim 64, at most 8 query heads per KV head): the producer
  // copies K/V stages as 2-D tiles of attn_box_rows rows (min(64, page_size)) through the tensor map
  // passed beside these parameters -- the whole cache (or page pool) as rows of 64 bf16, 128-byte
  // swizzle.  0: rows are bulk-copied and the attention runs on the CUDA cores.
  int attn_mma, attn_box_rows;
  // Streamed projection weights: bf16 (wbytes 2, wscale null) or FP8 E4M3 copies (wbytes 1) with one
  // fp32 scale per output row: per layer [q|k|v rows][Wo rows][gate rows][up rows][Wd rows]
  // (wscale_layer floats), then the LM head's V rows.
  int wbytes;
  int wscale_layer;
  const float* wscale;
};

// Changes every step.
// One launch decodes n consecutive positions pos, pos+1, ... (teacher-forced tokens).
struct StepParams {
  int token;                 // the token when tokens is null (n == 1)
  int pos;                   // position of the launch's first step
  unsigned tag;              // tag of the first step (never 0); step i writes its words with tag + i
  float* logits;             // device fp32 [n][V] (or one [V] buffer every step overwrites)
  int logits_step;           // floats between the logits of consecutive steps: V, or 0
  const int* tokens;         // device [n], or null
  int n;                     // steps in this launch
  unsigned long long* sync;  // step counter: every CTA adds 1 after each step (null when n == 1)
  unsigned long long sync_base;  // its value when the launch starts
  // greedy decoding (greedy != 0): the token of step i + 1 is the argmax of step i's logits (lowest
  // index among equal values); tokens[] is unused.  amax[i] collects the packed (value, index) key of
  // step i by atomic max, amax_done[i] counts the LM-head tasks that contributed (both zeroed by the
  // host), and out_tokens[i] receives the argmax of step i (written by the CTA that completes it).
  int greedy;
  unsigned long long* amax;
  unsigned* amax_done;
  int* out_tokens;
  unsigned long long* tokword;  // the argmax of step i as a word tagged tag + i + 1 (read by step i + 1)
};

}  // namespace mbk
