/*
 * mbk.h -- C ABI of the persistent batch-1 decode megakernel for GB300 (sm_103a).
 *
 * One call to mbk_decode_step runs a whole decode step of a Llama-shaped bf16 decoder as ONE
 * persistent cooperative kernel (one CTA per SM): token embedding, for every layer RMSNorm,
 * Q/K/V projection (+ bias), RoPE, KV-cache append, GQA decode attention, output projection,
 * residual add, RMSNorm, gate/up projection, SiLU*up, down projection, residual add, then the
 * final norm and the tied vocabulary projection, with no return to the host in between.
 *
 * Where the operation is defined (the MegaBake pages; they give the op list, not formulas):
 *  - "MegaBake: a PyTorch model compiled into one CUDA kernel, and what its 5.5x is measured
 *    against", section "What a megakernel is, and why small models want one": the per-layer op
 *    sequence of a Llama-style decode step and the one-CTA-per-SM persistent execution model.
 *  - megabake/megabake README, section "Current status": embedding, every layer, final norm,
 *    vocabulary projection and KV-cache updates inside one cooperative kernel; q/k/v biases in
 *    the projection epilogue; flash-decoding attention that splits long contexts across CTAs and
 *    packs the query heads sharing a KV head so each cached key/value is read once.
 *  - MegaBake project website, "Integration & evaluation": bf16, static contiguous decode KV state.
 * The formulas are the Hugging Face Llama definitions: RMSNorm x/sqrt(mean(x^2)+eps)*g; RoPE in
 * the rotate-half convention (element i pairs with i+d/2, angle pos*theta^(-2i/d)), applied to q
 * and k after the bias, with K cached after rotation; softmax(q.K/sqrt(d)) V with query head h
 * reading KV head h/(n_heads/n_kv_heads); silu(z) = z/(1+exp(-z)); tied LM head (logits = E.xn).
 *
 * Numerics: weights and KV cache bf16 (or, with MBK_WEIGHTS_FP8, the library's E4M3 copies of the
 * projections with one fp32 scale per row); all activations fp32 (accumulation in fp32); K and V
 * are rounded to bf16 (round to nearest even) when appended, and attention reads the rounded values.
 *
 * Memory layouts (all row-major, C order):
 *  - weight matrices: bf16 [out][in] (Hugging Face nn.Linear layout), read in place;
 *  - embedding / LM head: bf16 [vocab][hidden];
 *  - KV cache: bf16 [n_layers][2][n_kv_heads][kv_capacity][head_dim] (index 0 = K, 1 = V), or a
 *    pool of pages [num_pages][n_layers][2][n_kv_heads][page_size][head_dim] (mbk_create_paged);
 *  - logits: fp32 [vocab].
 *
 * Ownership: the caller owns the weights, the KV cache and every logits buffer; they must stay
 * valid (and the weights unchanged) for the handle's lifetime.  The library copies no weights,
 * except the FP8 copies it makes for MBK_WEIGHTS_FP8.  It owns those, its task tables, activation
 * exchange buffers, RoPE table, page table and status word, all freed by mbk_destroy.
 *
 * Threading / streams: a handle is not thread-safe.  Steps on one handle must be issued in order
 * on one stream (or on streams ordered by the caller); two steps of one handle must never run
 * concurrently.  Different handles are independent.
 *
 * Beside the decode step, mbk_prefill runs a prompt's tokens as dense contractions on the tensor
 * cores (tcgen05) and mbk_batch_step runs several sequences of a paged pool in one step through the
 * same kernels; both are compiled but have not yet been run on a GPU.
 *
 * Errors: every function returning int returns MBK_OK (0) or a negative MBK_ERR_* code.  Host
 * checks run before any launch and leave device state unchanged.  A device-side failure (a wait
 * that ran out of time) is recorded in a device status word; it is returned by the next
 * decode, prefill, batch or mbk_kv_fill call on the handle and by mbk_get_status, and is sticky
 * until mbk_destroy.
 */
#ifndef MBK_H
#define MBK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MBK_OK 0
#define MBK_ERR_INVALID_ARG (-1)  /* null pointer, out-of-range token/position, bad shape     */
#define MBK_ERR_UNSUPPORTED (-2)  /* not an sm_10x GPU, or the cooperative grid does not fit */
#define MBK_ERR_CUDA (-3)         /* a CUDA runtime call failed                              */
#define MBK_ERR_TIMEOUT (-4)      /* a device-side wait gave up (sticky)                     */
#define MBK_ERR_NOMEM (-5)        /* device or host allocation failed                        */
#define MBK_ERR_STATE (-6)        /* not possible in the present state: an armed injection, or no
                                     schedule for the shape (mbk_plan_check)                    */

typedef struct mbk_handle mbk_handle;

/* Decoder shape.  head_dim must be 64 or 128; n_heads % n_kv_heads == 0; hidden, intermediate
 * and n_heads*head_dim must be multiples of 8 (16-byte rows for bulk copies). */
typedef struct {
  int n_layers;
  int hidden;        /* H */
  int intermediate;  /* I */
  int n_heads;       /* query heads */
  int n_kv_heads;    /* key/value heads */
  int head_dim;      /* d */
  int vocab;         /* V */
  int kv_capacity;   /* C: cache rows per (layer, K|V, kv head) */
  double rms_eps;
  double rope_theta;
  int qkv_bias;      /* 1: bq, bk, bv are used (Qwen2); 0: ignored */
  int weight_format; /* MBK_WEIGHTS_BF16 (0): stream the bf16 weights as given.  MBK_WEIGHTS_FP8 (1): at
                      * create the library quantizes every projection (Wq, Wk, Wv, Wo, Wgate, Wup, Wdown)
                      * and the LM head's copy of the embedding to FP8 E4M3 with one fp32 scale per
                      * output row (scale = row max |w| / 448; codes = w / scale rounded to nearest
                      * even, saturating), owns those copies and streams them: about half the bytes
                      * per token.  The embedding lookup, norm gains and biases stay bf16.  The MegaBake
                      * website lists FP8 under "Next"; the format is this library's reading.  Needs
                      * hidden and intermediate to be multiples of 16. */
} mbk_config;

enum { MBK_WEIGHTS_BF16 = 0, MBK_WEIGHTS_FP8 = 1 };

/* Device pointers of one layer's bf16 tensors ([out][in] for matrices, [n] for vectors).
 * bq/bk/bv may be NULL when qkv_bias == 0. */
typedef struct {
  const void *attn_norm, *wq, *wk, *wv, *bq, *bk, *bv, *wo, *mlp_norm, *w_gate, *w_up, *w_down;
} mbk_layer_weights;

typedef struct {
  const void *embed;                /* device bf16 [V][H]; also the tied LM head */
  const void *final_norm;           /* device bf16 [H] */
  const mbk_layer_weights *layers;  /* HOST array of n_layers entries (copied at create) */
} mbk_weights;

/* Builds the static schedule for this shape on `device`, allocates the library's buffers and
 * computes the RoPE table.  kv_cache: device bf16 buffer of
 * n_layers*2*n_kv_heads*kv_capacity*head_dim elements (contents are not touched at create).
 * Every device pointer must be 16-byte aligned.  On success *out receives the handle. */
int mbk_create(const mbk_config *cfg, const mbk_weights *weights, void *kv_cache, int device, mbk_handle **out);

/* As mbk_create, with a PAGED KV cache: kv_pool is a device bf16 pool of num_pages pages, each
 * [n_layers][2][n_kv_heads][page_size][head_dim] (a page holds page_size consecutive positions of
 * every layer and head).  Which page holds positions q*page_size .. (q+1)*page_size - 1 is set with
 * mbk_set_page_table; until then no position is mapped.  The decode step itself is unchanged: the
 * weight producer copies cached rows page by page and the appended row goes to its page.  The pages
 * list a paged KV cache under "Next" (megabake/megabake README, "Current status"); the layout is
 * this library's.  Errors: as mbk_create, and MBK_ERR_INVALID_ARG unless page_size is a power of
 * two in [32, kv_capacity], num_pages >= 1 and kv_capacity / page_size (rounded up) <= 256. */
int mbk_create_paged(const mbk_config *cfg, const mbk_weights *weights, void *kv_pool, int32_t num_pages,
                     int32_t page_size, int device, mbk_handle **out);

/* FP8 copies of a bf16 matrix, exactly as mbk_create makes them for MBK_WEIGHTS_FP8: w (device bf16
 * [rows][cols], cols even) -> q (device [rows][cols] E4M3 codes) and s (device fp32 [rows] scales).
 * Asynchronous on `stream`.  Errors: MBK_ERR_INVALID_ARG for a NULL pointer, rows < 1 or an odd
 * or non-positive cols. */
int mbk_quantize_fp8(const void *w, int32_t rows, int32_t cols, void *q, float *s, void *stream);

/* Paged handles: pages[q] (HOST array of n_pages distinct entries in [0, num_pages)) is the pool
 * page of logical page q; positions [0, min(kv_capacity, n_pages * page_size)) are then mapped and
 * may be decoded or filled.  The table is copied on `stream` before the call returns; a call that
 * changes it must be ordered after the steps that use the old one.  Errors: MBK_ERR_INVALID_ARG for
 * a contiguous handle, n_pages < 1 or above kv_capacity / page_size (rounded up), an entry out of
 * range or repeated. */
int mbk_set_page_table(mbk_handle *h, const int32_t *pages, int32_t n_pages, void *stream);

/* One decode step: embeds token_id, writes K/V at `position` for every layer, attends over
 * cache rows [0, position] and writes fp32 logits[vocab] to the DEVICE buffer logits_out.
 * Cache rows below `position` are the caller's responsibility (earlier steps or mbk_kv_fill).
 * stream: a cudaStream_t (NULL = legacy default stream).  Asynchronous: returns after the launch.
 * Errors: MBK_ERR_INVALID_ARG if token_id is not in [0, vocab) or position not in
 * [0, kv_capacity) (for a paged cache: not mapped) or logits_out is NULL; a sticky device error
 * from an earlier step. */
int mbk_decode_step(mbk_handle *h, int32_t token_id, int32_t position, float *logits_out, void *stream);

/* n_steps consecutive decode steps in ONE launch: token tokens[i] (a HOST array of n_steps ids,
 * copied before the call returns) at position position + i, logits of step i written to the
 * DEVICE buffer logits_out + i * vocab (n_steps * vocab floats).  The results are those of n_steps
 * calls of mbk_decode_step (teacher-forced decoding: the tokens are given, e.g. a prompt or a draft
 * to verify); one launch saves the per-launch gap, the kernel prologue and the cold start of the
 * weight stream at every step but the first.  Inside the launch each step's K/V copies wait until
 * every CTA has finished the step before (the cache rows it appended).  The pages have no
 * multi-step call; the MegaBake website lists multi-step decoding under "Next".
 * Errors: MBK_ERR_INVALID_ARG if n_steps < 1, a token is not in [0, vocab), or
 * [position, position + n_steps) is not inside [0, kv_capacity); MBK_ERR_STATE if a diagnostic
 * injection is armed (it applies to single steps only); a sticky device error. */
int mbk_decode_steps(mbk_handle *h, const int32_t *tokens, int32_t n_steps, int32_t position, float *logits_out,
                     void *stream);

/* Greedy decoding of n_steps tokens in ONE launch: step 0 decodes first_token at `position`, and
 * step i >= 1 decodes, at position + i, the argmax of step i - 1's logits (the lowest index among
 * equal values).  tokens_out: DEVICE int32[n_steps]; tokens_out[i] is the argmax of step i's logits,
 * so tokens_out[n_steps - 1] is the token that would come next.  logits_out: DEVICE buffer of
 * n_steps * vocab floats, or NULL when only the tokens are wanted.  The argmax is taken on the
 * device at the end of each step (every LM-head task adds its largest logit by a 64-bit atomic
 * max), and the next step's embedding waits for it, so no host round trip separates the steps.
 * The pages list multi-step decoding under "Next" (MegaBake website); the feedback of the argmax
 * is the plain greedy reading.  Errors: MBK_ERR_INVALID_ARG if tokens_out is NULL, n_steps < 1,
 * first_token is not in [0, vocab) or [position, position + n_steps) is not inside
 * [0, kv_capacity); MBK_ERR_STATE if a diagnostic injection is armed; a sticky device error. */
int mbk_decode_greedy(mbk_handle *h, int32_t first_token, int32_t n_steps, int32_t position, int32_t *tokens_out,
                      float *logits_out, void *stream);

/* Prefill: n_tokens given tokens (a prompt) at positions position .. position + n_tokens - 1,
 * computed as dense contractions over all of them on the tensor cores instead of one decode step
 * per token.  The MegaBake article ("Where it loses") names prefill as the megakernel's weakest
 * path; its plain definition is n_tokens teacher-forced decode steps, and that is what this computes
 * (each token attends to the cache rows up to its own position), layer by layer: RMSNorm, the
 * Q/K/V projection (+ bias), RoPE, the KV append, causal attention, the O projection and residual,
 * RMSNorm, gate/up, SiLU * up, the down projection and residual; then the final norm and the tied
 * LM head.  The cache rows of every layer at those positions are written, exactly as the decode
 * steps would write them (bf16, nearest even).
 *   tokens: HOST array of n_tokens ids, copied before the call returns.
 *   logits_mode: MBK_PREFILL_LOGITS_NONE (cache only; logits_out unused and may be NULL),
 *     MBK_PREFILL_LOGITS_LAST (the last token's logits: DEVICE fp32[vocab]) or
 *     MBK_PREFILL_LOGITS_ALL (every token's: DEVICE fp32[n_tokens][vocab]).
 * Numerics: projections multiply the bf16 weights by fp32 activations carried as a bf16 pair
 * (hi = bf16(x), lo = bf16(x - hi); fp32 accumulation), so results match the fp32-activation decode
 * within its tolerances.  Memory: the handle keeps a device workspace of about
 * n_tokens * (4 * (2 * hidden + (n_heads + 2 * n_kv_heads) * head_dim + 2 * intermediate) +
 * 4 * max(hidden, intermediate, n_heads * head_dim)) bytes; a call with more tokens than any
 * before it reallocates it (a synchronising cudaFree/cudaMalloc).  Asynchronous on `stream`
 * otherwise.  Not a counterpart of a MegaBake entry point (the pages have none for prefill).
 * Errors: MBK_ERR_INVALID_ARG if n_tokens < 1, a token is not in [0, vocab), the positions are not
 * inside [0, kv_capacity) (for a paged cache: mapped), logits_mode is unknown, or logits_out is NULL
 * while logits are asked for; MBK_ERR_UNSUPPORTED for an FP8 handle (prefill reads the bf16
 * weights) or when the driver has no tensor-map encoder; MBK_ERR_NOMEM if the workspace cannot be
 * allocated; MBK_ERR_STATE if a decode step's diagnostic injection is armed, MBK_ERR_INVALID_ARG if a
 * prefill injection (mbk_debug_prefill_inject) is armed for another n_tokens; a sticky device error.  A device
 * wait that runs out of time is reported like a decode step's (mbk_get_status). */
#define MBK_PREFILL_LOGITS_NONE 0
#define MBK_PREFILL_LOGITS_LAST 1
#define MBK_PREFILL_LOGITS_ALL 2
int mbk_prefill(mbk_handle *h, const int32_t *tokens, int32_t n_tokens, int32_t position, float *logits_out,
                int32_t logits_mode, void *stream);

/* Small-batch decode, and prompts of several sequences, in one step: n_seq sequences share a PAGED
 * handle's pool (mbk_create_paged), each with its own page table, and sequence s contributes counts[s]
 * tokens at positions starts[s] .. starts[s] + counts[s] - 1 -- one token for a decode step, or a
 * chunk of a prompt.  The MegaBake README ("Current status") lists small-batch decode under "Next";
 * the reading here: the step is, for every sequence, its counts[s] teacher-forced decode steps on its
 * own cache (each token attends to its sequence's rows up to its own position), and the sequences do
 * not interact.  All tokens of the step go through the prefill's tensor-core contractions together,
 * so every weight is read once per step for up to 128 tokens, whatever the mix of decode tokens and
 * prompt chunks.
 *   tokens: HOST int32 array of sum(counts) ids, grouped by sequence in sequence order.
 *   page_tables: HOST int32 [n_seq][ceil(kv_capacity / page_size)]: entry q of table s is the pool page
 *     holding positions q * page_size .. of sequence s (entries past the last position used are not read).
 *   logits_mode: MBK_PREFILL_LOGITS_NONE, _LAST (the last token of each sequence: DEVICE fp32
 *     [n_seq][vocab]) or _ALL (every token, in token order: DEVICE fp32 [sum(counts)][vocab]).
 * The handle's own page table (mbk_set_page_table) is neither used nor changed.
 * Errors: MBK_ERR_INVALID_ARG for a NULL array, n_seq < 1, a contiguous handle, counts[s] < 1, a
 * position outside [0, kv_capacity), a token outside [0, vocab), a table entry outside the pool, a
 * page used twice (within or across the sequences' used ranges), an unknown logits_mode or NULL
 * logits_out while logits are asked for; as mbk_prefill otherwise.  Not yet run on a GPU. */
int mbk_batch_step(mbk_handle *h, int32_t n_seq, const int32_t *counts, const int32_t *starts, const int32_t *tokens,
                   const int32_t *page_tables, float *logits_out, int32_t logits_mode, void *stream);

/* As mbk_decode_step, then copies the logits into the HOST buffer logits_host (vocab floats;
 * pinned memory makes the copy asynchronous) and synchronises `stream` before returning. */
int mbk_decode_step_host(mbk_handle *h, int32_t token_id, int32_t position, float *logits_host, void *stream);

/* Loads cache rows [p0, p0+n) of `layer` from pre-RoPE keys and values (device fp32
 * [n_kv_heads][n][head_dim] each): K is rotated by its position with the same RoPE as a decode
 * step, then both are rounded to bf16 and stored.  Asynchronous on `stream`. */
int mbk_kv_fill(mbk_handle *h, int layer, const float *k_raw, const float *v_raw, int32_t p0, int32_t n,
                void *stream);

/* Device status of the most recently COMPLETED step (synchronise the stream first):
 * MBK_OK or MBK_ERR_TIMEOUT.  Reading it does not clear it. */
int mbk_get_status(mbk_handle *h);

/* Human-readable text of an error code (static storage). */
const char *mbk_error_string(int code);

/* Frees everything the library allocated for the handle.  Waits for the handle's work to finish.
 * NULL is ignored. */
void mbk_destroy(mbk_handle *h);

/* ---- decoding without device allocation ----
 * (Not a counterpart of anything in the MegaBake pages: it exists for callers of this library.)
 *
 * mbk_decode_step_static is one decode step, computed exactly like mbk_decode_step, for callers
 * that cannot allocate device memory when they decode: code running under a caller-owned memory
 * pool or budget that forbids new device allocations, or inside a runtime whose allocator must not
 * be re-entered.  It calls no cudaMalloc, cudaFree or other allocating routine and needs no handle.
 * Everything the library keeps for a step (static schedule, activation exchange words, RoPE table,
 * status word) lives in one device array of MBK_STATIC_SCRATCH_BYTES that is part of the library:
 * every GPU that loads the library holds it until the process exits.
 *  - The caller passes the config, the weights, the KV cache, the token, the position and the
 *    DEVICE logits buffer, as for mbk_create + mbk_decode_step; the current device is used.
 *  - The first call on a device looks up the array's device address (and sets the kernel's shared
 *    memory limit) with that device current; make that first call before any stream capture.
 *  - All calls on a device share the array, which keeps the last call's contents: the schedule is
 *    rebuilt and uploaded (then the stream is synchronised once) only when the config or any
 *    pointer differs from the previous call; the exchange words and the status word are cleared
 *    on every call.  A call that needs a rebuild must therefore be made outside stream capture:
 *    inside a capture it returns MBK_ERR_STATE and leaves the capture untouched.  Calls whose GPU
 *    work overlaps (two streams, two threads) race on the array: order them on one stream.
 *  - Device-side waits are bounded by MBK_WAIT_TIMEOUT_MS (default 1000), as for a handle.
 *  - Returns MBK_ERR_INVALID_ARG for the same argument errors as mbk_create / mbk_decode_step and
 *    when the shape needs more than MBK_STATIC_SCRATCH_BYTES (nothing is launched then);
 *    MBK_ERR_UNSUPPORTED or MBK_ERR_CUDA as mbk_create.  A device-side wait that times out is not
 *    reported by this entry point (the launch still ends; its logits are then invalid). */
#define MBK_STATIC_SCRATCH_BYTES (16u << 20)
int mbk_decode_step_static(const mbk_config *cfg, const mbk_weights *weights, void *kv_cache, int32_t token_id,
                           int32_t position, float *logits_out, void *stream);

/* ---- diagnostics (for tests and profiling; not needed to decode) ---- */

/* Residual stream of the most recently COMPLETED step (synchronise its stream first), copied to the
 * HOST buffer taps_out as fp32 [(2*n_layers+1)][hidden]: the embedding row, then the stream after
 * each layer's attention and MLP sublayers.  Returns MBK_OK or MBK_ERR_INVALID_ARG / MBK_ERR_CUDA. */
int mbk_debug_taps(mbk_handle *h, float *taps_out);

/* Region-by-region checking: makes the NEXT step read, as the residual stream entering each layer
 * l >= 1, row l of the HOST buffer x_in ([n_layers][hidden] fp32; row 0 is ignored -- layer 0 reads
 * the embedding) instead of layer l-1's output, so every layer can be compared with a reference
 * from identical inputs.  It applies to one step; passing NULL cancels it.  Not for decoding. */
int mbk_debug_inject(mbk_handle *h, const float *x_in);

/* The same for prefill: makes the NEXT mbk_prefill call, which must have n_tokens tokens, read as
 * the residual stream entering each layer l >= 1 block l of the HOST buffer x_in
 * ([n_layers][n_tokens][hidden] fp32, copied before this call returns; block 0 is ignored) instead of
 * layer l-1's output.  Every layer's K/V rows then come from identical inputs on both sides of a
 * comparison.  Passing NULL cancels it.  Errors: MBK_ERR_INVALID_ARG for n_tokens outside
 * [1, kv_capacity]; MBK_ERR_NOMEM / MBK_ERR_CUDA.  Not for decoding. */
int mbk_debug_prefill_inject(mbk_handle *h, const float *x_in, int32_t n_tokens);

/* Static schedule of the handle: writes up to `capacity` rows of 6 int32
 * {cta, type (1 QKV, 2 ATTN, 3 OPROJ, 4 GATEUP, 5 DOWN, 6 LMHEAD), layer, row0, nrows, nchunks}
 * in global task order to the HOST buffer `out` and returns the number of tasks (or a negative code). */
int64_t mbk_debug_plan(mbk_handle *h, int32_t *out, int64_t capacity);

/* Per-task timing: when enabled, every later step records for each task eight globaltimer stamps
 * (ns): {begin, inputs ready, end, first weight stage ready (0 if none), then four phase marks of the
 * task, 0 where unused}.  Attention tasks mark: 4 the query rotation and the K/V rows staged, 5 the
 * (position block, head) items done, 6 the output merged (before the fused O rows).  Projection
 * tasks put the SM clock count (clock64) at their end in slot 7, so that a trace also shows the
 * clock the step ran at.
 * Enabling allocates a device buffer of 64 bytes per task; disabling frees it.  mbk_trace_read
 * copies the stamps of the most recently completed traced step (synchronise first) into the HOST
 * buffer `out` (8 uint64 per task, global task order) and returns the number of tasks (or a
 * negative code). */
int mbk_trace_enable(mbk_handle *h, int enable);
int64_t mbk_trace_read(mbk_handle *h, uint64_t *out, int64_t capacity_tasks);

/* ---- introspection of the static schedule (host only; no GPU needed) ---- */

typedef struct {
  int num_ctas;            /* CTAs the plan was built for (one per SM) */
  int num_tasks;           /* tasks over all CTAs */
  int num_chunks;          /* static weight chunks over all CTAs */
  int stage_bytes;         /* bytes of one shared-memory ring stage */
  int num_stages;          /* stages in each CTA's ring */
  int attn_splits;         /* context splits per KV head */
  int64_t weight_bytes;    /* weight bytes streamed per step by the static chunks */
  int64_t max_cta_bytes;   /* largest per-CTA share of those bytes */
  int64_t act_words;       /* 8-byte activation exchange words per step */
  int smem_bytes;          /* dynamic shared memory per CTA */
  int combine_group;       /* splits whose outputs one poll of the split combine brings (<= attn_splits) */
  int attn_mma;            /* 1: attention runs on the tensor cores (head_dim 64, <= 8 query heads per KV head) */
} mbk_plan_info;

/* Builds the schedule for `cfg` as if on a GPU with `num_sms` SMs, checks it (every weight row
 * covered exactly once, every task's inputs produced by an earlier task in every CTA's order,
 * every bulk copy 16-byte aligned and within its tensor) and fills *info.  Returns MBK_OK,
 * MBK_ERR_INVALID_ARG for a shape the kernel does not support, or MBK_ERR_STATE when a check
 * fails.  Weight addresses are taken from a fake base so no device memory is needed.
 *
 * Environment knobs read wherever a schedule is built (mbk_create, mbk_create_paged,
 * mbk_decode_step_static, mbk_plan_check, mbk_plan_simulate), all for experiments, defaults best
 * measured: MBK_MAX_TASKS_PER_OP (at most this many CTAs per projection), MBK_FUSE_ATTENTION (0: the
 * O projection as tasks of its own), MBK_ATTN_MMA (0: attention on the CUDA cores instead of the
 * tensor cores), MBK_ATTN_SPLIT (context split length, a multiple of 64; default 512) and
 * MBK_COMBINE_TASKS (O-projection tasks of a split context; default one per 24 output rows).  At
 * launch: MBK_WAIT_TIMEOUT_MS (bounded waits, default 1000) and MBK_POLL_BACKOFF_NS (sleep between
 * polls, default 0). */
int mbk_plan_check(const mbk_config *cfg, int num_sms, mbk_plan_info *info);

/* Execution model of the schedule's exchange protocol (host only; no GPU needed).  Builds the plan as
 * mbk_plan_check does and runs one step at `position` through a model of the kernel's waits: every CTA
 * runs its task list in order, and a task runs once every activation word it reads (its input vector,
 * residual rows, per-KV-head partials, the active context splits' outputs, or for attention its KV
 * head's q/k/v words) has been written in this step; it then writes its output words.  Readiness only
 * grows within a step, so if tasks remain when no task is ready the plan can deadlock on the GPU
 * whatever the timing (the kernel's bounded waits would then report MBK_ERR_TIMEOUT).  The depths
 * count exchange rounds: the longest chain of tasks each reading a word its predecessor wrote.  The
 * same environment knobs as mbk_plan_check apply, and the fault-injection knob MBK_DEBUG_DROP_TASK.  Returns MBK_OK when every task ran and no word was
 * written twice, MBK_ERR_STATE otherwise (details in *info), MBK_ERR_INVALID_ARG for a bad argument
 * or an unsupported shape. */
typedef struct {
  int tasks_total;              /* tasks in the plan */
  int tasks_run;                /* tasks that could run: all of them unless the plan can deadlock */
  int exchange_depth;           /* longest chain of tasks each reading a word written by the one before */
  int schedule_depth;           /* the same, with each CTA's task order counted as a dependency too */
  int64_t words_written_twice;  /* output words written by more than one task (0 in a valid plan) */
  int stuck_cta;                /* -1, or the first CTA whose next task never becomes ready */
  int stuck_task_type;          /* that task's type (1 QKV, 2 ATTN, 3 OPROJ, 4 GATEUP, 5 DOWN, 6 LMHEAD) */
  int stuck_layer;              /* ... and layer */
  int64_t stuck_word;           /* a word it waits for that no task writes before it (-1 if none) */
} mbk_sim_info;
int mbk_plan_simulate(const mbk_config *cfg, int num_sms, int position, mbk_sim_info *info);

#ifdef __cplusplus
}
#endif
#endif /* MBK_H */
