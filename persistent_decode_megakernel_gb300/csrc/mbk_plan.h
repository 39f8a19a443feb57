// mbk_plan.h -- the static schedule shared by the host scheduler (mbk_plan.cpp) and the persistent
// kernel (mbk_kernel.cu).  Plain structs only; no CUDA types, so the scheduler builds and is
// checked without a GPU.
//
// The schedule is the GB300 form of the pages' phase table (MegaBake article, "How a model gets in",
// step 4 "Schedule" and the table-driven kernel loop described after it): depth lives in data, not
// code.  Instead of phases closed by grid barriers, every CTA walks its OWN ordered task list; a
// task waits only for the activation words it reads (per-element dependency tags), and its weights
// are input-independent, so a producer warp streams them into shared memory ahead of the waits.
#pragma once
#include <stdint.h>

namespace mbk {

enum TaskType : uint16_t {
  T_QKV = 1,     // rmsnorm(x) -> rows of [Wq;Wk;Wv] (+bias) -> raw q|k|v words
  T_ATTN = 2,    // one KV head, one context split: RoPE, KV append (owner split), softmax partial
  T_OPROJ = 3,   // combine attention splits -> rows of Wo -> x_attn = x + Wo.o
  T_GATEUP = 4,  // rmsnorm(x_attn) -> rows of Wg and Wu -> h = silu(g) * u
  T_DOWN = 5,    // rows of Wd -> x_mlp = x_attn + Wd.h
  T_LMHEAD = 6,  // final rmsnorm(x) -> rows of E -> logits
};

// One task of one CTA.  GEMV tasks: output rows [row0, row0 + nrows) of the op's output space
// (QKV: the concatenation q|k|v; GATEUP: rows of I, results g then u), weights in static chunks
// [chunk0, chunk0 + nchunks).  ATTN tasks: row0 = KV head, nrows = context split index; their
// chunks (cached K/V rows) are derived on the device from the step's position.
struct Task {
  uint16_t type;
  uint16_t layer;
  uint32_t row0;
  uint32_t nrows;
  uint32_t chunk0;
  uint32_t nchunks;
  uint32_t gpr;     // GEMV: 0 = one warp per row (small tasks); else warps sharing one weight row
                    // (a power of two; each keeps its K slice of the input in registers)
  uint32_t lpr;     // GEMV: lanes per warp working on a row (always 32)
  uint32_t pad;
};
static_assert(sizeof(Task) == 32, "Task layout");

// One bulk copy into one ring stage: `rows` whole weight rows starting at `src` (bytes = rows *
// row bytes; a multiple of 16, src 16-byte aligned).  An attention task owns one placeholder chunk
// (rows == kAttnChunk) whose stages -- cached K/V rows, their number set by the step's position --
// the producer derives on the device; its src packs {layer:16 | kv head:16 | split:32}.
struct Chunk {
  uint64_t src;
  uint32_t bytes;
  uint32_t rows;
};
constexpr uint32_t kAttnChunk = 0xFFFFFFFFu;
static_assert(sizeof(Chunk) == 16, "Chunk layout");

// Offsets (in 8-byte words) of one layer's activation exchange words.
struct ActLayout {
  uint32_t qkv;       // (nq + 2 nkv) * d   raw projections, pre-RoPE
  uint32_t att;       // nkv * nsplit * g * (d + 2)   per split: o (normalised), m, l per head
  uint32_t xa;        // H   residual stream after the attention sublayer
  uint32_t hh;        // I   silu(g) * u
  uint32_t xm;        // H   residual stream after the MLP sublayer (input of the next layer)
  uint32_t per_layer; // words per layer
};

constexpr int kStageBytes = 16384;     // one ring stage
constexpr int kMaxTaskRows = 2048;     // output rows per task
constexpr int kResSlots = 4096;        // per-task partial results (rows x warps per row)
constexpr int kComputeWarps = 16;
constexpr int kThreads = 32 * (kComputeWarps + 1);  // warp 0 streams weights, warps 1..16 compute
constexpr int kAttnSplitMax = 512;     // context positions per attention split (long contexts)
constexpr int kAttnSplitStages = 8;    // ring stages per attention split
constexpr int kMaxRingStages = 32;
constexpr int kMaxTaskChunks = 256;
constexpr int kGemvBatch = 4;          // ring stages a GEMV consumes together
constexpr int kGemvXVec = 4;           // 16-byte input vectors a GEMV lane keeps in registers
constexpr int kCtlBytes = 4096;        // shared-memory control block (barriers, flags, tables)
constexpr int kMaxLayers = 64;

struct PlanShape {
  int L, H, I, nq, nkv, d, V, C;
  int qkv_bias;
};

}  // namespace mbk
