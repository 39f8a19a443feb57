// mbk_prefill.h -- host interface of the prefill path (mbk_prefill.cu), used by the C ABI (mbk_api.cu).
//
// Prefill runs n tokens whose ids are known in advance (a prompt) through the decoder at positions
// p0 .. p0 + n - 1 and appends their K/V rows to the cache.  Its plain definition is n teacher-forced
// decode steps; with all n tokens at hand the projections become dense [n, K] x [K, N] contractions,
// which run on the tensor cores (tcgen05) instead of the decode kernel's GEMVs.
#pragma once
#include <cuda.h>  // CUtensorMap and its enums (types only: the encoder is looked up at run time)
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "mbk_device.h"

namespace mbk {

// The decoder as the prefill reads it.  All pointers are device pointers; weights are bf16 bit
// patterns in the Hugging Face [out, in] layout, 16-byte aligned.
struct PrefillModel {
  int L, H, I, nq, nkv, d, V;
  float eps, inv_H;             // RMSNorm epsilon; 1 / hidden rounded to fp32
  float attn_scale;             // 1 / sqrt(head_dim)
  int qkv_bias;
  const uint16_t* embed;        // [V][H]: embedding rows and the tied LM head
  const uint16_t* final_norm;   // [H]
  std::vector<LayerW> layers;   // per layer, in LayerSlot order
  const float2* rope;           // [C][d/2] (cos, sin) of position p and frequency i
  // the KV cache: contiguous [L][2][nkv][C][d] (page_table null, page_size = C) or a pool of pages
  // [num_pages][L][2][nkv][page_size][d] found through page_table (page_size = 1 << page_shift)
  uint16_t* kv;
  const int32_t* page_table;
  int page_size, page_shift;
  unsigned long long page_elems;
  unsigned* status;             // device status word [4] shared with the decode kernel
  unsigned* host_status;        // its mapped host copy (may be null)
  unsigned long long timeout_ns;
};

// Workspace and tensor maps, owned by a handle.  The workspace grows on demand (a call with more
// tokens than it holds reallocates it); the weight maps are encoded on the first call.
struct PrefillState {
  int cap = 0;                  // tokens the workspace holds
  void* ws = nullptr;           // one device allocation holding the buffers below
  float* x = nullptr;           // [cap][H]       residual stream
  float* qkv = nullptr;         // [cap][qd+2kvd] projections (q and k rotated in place)
  float* gu = nullptr;          // [cap][2I]      gate | up
  uint16_t* a_hi = nullptr;     // [cap][max(H, qd, I)] GEMM input, bf16 high part
  uint16_t* a_lo = nullptr;     // ... and the bf16 remainder
  int32_t* tokens = nullptr;    // [cap]
  int32_t* pos = nullptr;       // [cap] position of each token
  int32_t* seq = nullptr;       // [cap] its sequence
  int32_t* rows = nullptr;      // [cap] the last token of each sequence (logits of the last tokens)
  int2* tiles = nullptr;        // [cap] attention tiles: (first token, tokens) of one sequence
  int32_t* tables = nullptr;    // page tables of a batch of sequences (grown on demand)
  size_t tables_cap = 0;        // int32 entries allocated there
  std::vector<CUtensorMap> wmaps;  // per layer Wq, Wk, Wv, Wo, Wgate, Wup, Wdown; then E
  bool smem_set = false;
};

// The tokens of one call: n_seq sequences, sequence s contributing counts[s] consecutive tokens at
// positions starts[s] .. starts[s] + counts[s] - 1; the token array holds them grouped by sequence,
// in sequence order.  tables: HOST [n_seq][max_pages] page tables of a paged pool, or null to address
// the cache as the model does (one sequence: contiguous, or the handle's own page table).
struct PrefillBatch {
  int n_seq = 1;
  const int32_t* counts = nullptr;
  const int32_t* starts = nullptr;
  const int32_t* tables = nullptr;
  int max_pages = 0;
};

// Logits the caller asks for (values of the C ABI's MBK_PREFILL_LOGITS_*).
enum PrefillLogits { PL_NONE = 0, PL_LAST = 1, PL_ALL = 2 };

// Runs the tokens of `batch` on `stream` (asynchronous after the host-to-device copies).  tokens_host:
// n = sum of counts ids, grouped by sequence; everything already validated by the caller (positions
// inside each sequence's cache, page tables inside the pool, no page shared between sequences).
// logits: device fp32, [n][V] (PL_ALL), [n_seq][V] (PL_LAST: the last token of each sequence) or
// unused (PL_NONE).  Returns an MBK_* code.  inject (diagnostics; may be null): device fp32 [L][n][H];
// block l >= 1 replaces the residual stream entering layer l.
int prefill_run(const PrefillModel& m, PrefillState& st, const int32_t* tokens_host, int n, const PrefillBatch& batch,
                float* logits, int mode, cudaStream_t stream, const float* inject = nullptr);

// Frees the workspace (the tensor maps are host memory).
void prefill_free(PrefillState& st);

// Tensor map of a KV cache (or page pool) of head_dim 64 for the decode kernel's tensor-core
// attention: `rows` rows of 64 bf16 (128 bytes) from `kv` (16-byte aligned), tiles of 64 columns by
// box_rows rows with the 128-byte swizzle; reads past the last row return zeros.  False if the
// encoder is unavailable or refuses the arguments.
bool make_kv_tile_map(CUtensorMap* map, const void* kv, uint64_t rows, uint32_t box_rows);

}  // namespace mbk
