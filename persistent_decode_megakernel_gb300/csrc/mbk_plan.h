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

// What a task reads and writes, decided by the scheduler so that the kernel does no per-type
// address arithmetic: activation words are indices into the step's word array.
enum TaskFlags : uint16_t {
  TF_NORM = 1,        // the input is RMS-normalised with gain table entry `gain`
  TF_PAIRS = 2,       // gate/up: rows r and nrows + r of the task pair up (silu(gate) * up)
  TF_BIAS = 4,        // q/k/v bias added to the rows
  TF_IN_EMB = 8,      // the input is the token's embedding row (layer 0)
  TF_IN_LAYER = 16,   // the input is the layer's input stream (replaceable by injected words)
  TF_RES = 32,        // the rows add a residual
  TF_RES_EMB = 64,    // ... taken from the token's embedding row (layer 0)
  TF_RES_LAYER = 128, // ... taken from the layer's input stream (replaceable by injected words)
  TF_COMBINE = 256,   // the input is the attention output of several context splits
  TF_LOGITS = 512,    // the rows are logits (written to the caller's buffer, not as words)
  TF_WO = 1024,       // attention task that also applies its KV head's columns of Wo to output rows
                      // [row0, row0 + nrows) (KV head in aux), writing that head's partial sums
  TF_KV_APPEND = 2048,// this attention task appends the step's K/V row to the cache
  TF_IN_SUM = 4096,   // the input adds the per-KV-head attention partials (words aux + s*H + e)
  TF_RES_SUM = 8192,  // the residual rows add the per-KV-head attention partials (words aux + s*H + r)
};

// One task of one CTA.  GEMV tasks: output rows [row0, row0 + nrows) of the op's output space
// (QKV: the concatenation q|k|v; GATEUP: rows of I, results g then u), weights in static chunks
// [chunk0, chunk0 + nchunks).  ATTN tasks: row0 = KV head, nrows = context split index; their
// chunks (cached K/V rows) are derived on the device from the step's position; in_off/out_off
// are the layer's q|k|v and attention-output words.  With TF_WO (one context split, few KV heads)
// the attention task of KV head aux also owns output rows [row0, row0 + nrows) of the O projection
// restricted to that head's columns: the O projection needs no task and no exchange of its own, and
// its consumers sum the heads' partials.
struct Task {
  uint16_t type;
  uint16_t layer;
  uint16_t gpr;     // GEMV: 0 = one warp per row (small tasks); else warps sharing one weight row
                    // (a power of two; each keeps its K slice of the input in registers)
  uint16_t flags;   // TaskFlags
  uint32_t row0;
  uint32_t nrows;
  uint32_t chunk0;
  uint32_t nchunks;
  uint32_t in_off;  // first input word
  uint32_t in_n;    // input length
  uint32_t res_off; // first residual word (TF_RES, from words)
  uint32_t out_off; // first output word
  uint32_t gain;    // gain table entry (TF_NORM): attn_norm of layer l at 2l, mlp_norm at 2l+1, final at 2L
  uint32_t aux;     // TF_WO: the KV head; TF_IN_SUM / TF_RES_SUM: first word of the attention partials
};
static_assert(sizeof(Task) == 48, "Task layout");

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
// A strided chunk (rows has this bit): rows & ~kStridedRows segments of bytes / rows bytes each,
// the first at src, the next one O-projection row (n_heads * head_dim bf16) further on, packed
// back to back in the stage.  Used for a KV head's columns of Wo.
constexpr uint32_t kStridedRows = 1u << 30;
static_assert(sizeof(Chunk) == 16, "Chunk layout");

// Offsets (in 8-byte words) of one layer's activation exchange words.
struct ActLayout {
  uint32_t qkv;       // (nq + 2 nkv) * d   raw projections, pre-RoPE
  uint32_t att;       // nsplit * nq * (d + 2): o [split][head][d] (normalised per split), then
                      // (m, l) [split][head][2] -- the active splits of a step are a prefix of each
  uint32_t xa;        // H   residual stream after the attention sublayer (unused with TF_WO)
  uint32_t hh;        // I   silu(g) * u
  uint32_t xm;        // H   residual stream after the MLP sublayer (input of the next layer)
  uint32_t ap;        // nkv * H  per-KV-head partial O projections (TF_WO plans; else empty)
  uint32_t per_layer; // words per layer
};

constexpr int kStageBytes = 16384;     // one ring stage
constexpr int kMaxTaskRows = 2048;     // output rows per task
constexpr int kResSlots = 4096;        // per-task partial results (rows x warps per row)
// 11 compute warps + the producer = 12 warps, three per SM sub-partition, so every thread may use up
// to 168 registers.  Measured against 15 (16 warps, 128 registers): +0.4% on the 135M shape, +1% on
// Qwen2-0.5B, +5% on SmolLM-1.7B; 7 compute warps lose 9-16%.
constexpr int kComputeWarps = 11;
constexpr int kThreads = 32 * (kComputeWarps + 1);  // warp 0 streams weights, warps 1..11 compute
constexpr int kMaxHidden = 2048;       // largest hidden size
constexpr int kVecPerThread = (kMaxHidden + kComputeWarps * 32 - 1) / (kComputeWarps * 32);  // H or task rows / thread
constexpr int kAttnSplitMax = 512;     // context positions per attention split (long contexts)
constexpr int kAttnSplitStages = 8;    // ring stages per attention split
constexpr int kMaxRingStages = 32;
constexpr int kMaxTaskChunks = 256;
constexpr int kGemvBatch = 4;          // ring stages a GEMV consumes together
constexpr int kGemvXVec = 4;           // 16-byte input vectors a GEMV lane keeps in registers
static_assert(kGemvXVec % 2 == 0, "the GEMV loads its weights in pairs of vectors");
constexpr int kCtlBytes = 5376;        // shared-memory control block (barriers, flags, tables, parameters)
constexpr int kMaxPages = 256;         // logical pages of a paged KV cache (its table lives in the control block)
constexpr int kMaxLayers = 64;
constexpr int kTaskWindow = 160;      // task records staged in shared memory at a time
constexpr int kMaxFusedKvHeads = 4;   // the O projection is fused into attention for at most this many KV heads
constexpr int kMaxFusedGroupWidth = 512;  // ... and query-head groups of at most this many elements (g * head_dim)
// Trace stamps per task: begin, inputs ready, end, first weight stage, then up to four phase marks of
// the task (0 where a task type has fewer phases).
constexpr int kTraceStamps = 8;

struct PlanShape {
  int L, H, I, nq, nkv, d, V, C;
  int qkv_bias;
  int wb = 2;  // bytes of a streamed projection weight: 2 (bf16) or 1 (FP8 E4M3 with per-row scales)
};

}  // namespace mbk
