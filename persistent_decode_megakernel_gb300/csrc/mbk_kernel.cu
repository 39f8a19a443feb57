// mbk_kernel.cu -- the persistent batch-1 decode kernel for sm_103a (GB300).
//
// One cooperative launch per decode step, one CTA per SM (MegaBake article, "What a megakernel is,
// and why small models want one": resident CTAs working through a task list and synchronising
// through global memory).  Every CTA runs 12 warps:
//   warp 0      streams the weights of its upcoming tasks into a ring of shared-memory stages with
//               TMA bulk copies (cp.async.bulk + mbarrier transaction counts), and an attention
//               task's cached K/V rows as 2-D TMA tiles with the 128-byte swizzle the tensor-core
//               attention reads.  Weights do not depend on the token, so the stream runs ahead of the
//               data dependencies by up to the ring's depth -- the "cross-phase prefetch of the next
//               GEMM's weights while a CTA waits" the article lists as future work ("Checking the 5.5x").
//   warps 1-11  execute the CTA's tasks in order.  Activations move between CTAs as 64-bit words
//               {tag:32 | fp32 value:32}, each written once per step by exactly one thread; a reader
//               polls the word until its tag equals this step's tag.  A value and its readiness
//               travel in one single-copy-atomic store, so no fence, counter or grid barrier is
//               needed (the pages' counting grid barrier is the thing this replaces).
// The step is a long chain of small dependent tasks, so the kernel is built for latency: one code
// path serves every projection type and one serves attention (its blocks on the tensor cores, or on
// the CUDA cores in a separate instantiation), keeping the instructions of a task hot in the
// instruction cache; a projection row's output word is written by the warp that
// computed it the moment its dot product is done; token-independent loads (norm gains, biases,
// descriptors) are issued before a task waits for its inputs and consumed after.
// Every wait is bounded by a globaltimer budget; on expiry the CTA records timeout status and
// finishes its task list without waiting or writing, so the launch always terminates.
#include <cuda.h>  // CUtensorMap (the type only)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mbk_device.h"

namespace mbk {

// ------------------------------------------------------------------ small device helpers
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ unsigned long long ld_word(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_word(unsigned long long* p, unsigned tag, float v) {
  unsigned long long w = ((unsigned long long)tag << 32) | (unsigned long long)__float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* b, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* b, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// 1-D TMA bulk copy global -> this CTA's shared memory, completing `bytes` on mbarrier `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, unsigned bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
// 2-D TMA tile copy global -> shared memory (box and 128-byte swizzle from the tensor map), completing
// on mbarrier `bar`; x is the innermost coordinate (elements), y the row.
__device__ __forceinline__ void tile_load(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(
          smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kComputeWarps * 32) : "memory"); }
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

constexpr int kCT = kComputeWarps * 32;  // compute threads

// Input vectors of a GEMV live in shared memory in a split layout: element i of n sits at
// (i/8)*4 + i%4 in the lower half (i%8 < 4) or at n/2 + (i/8)*4 + i%4 - 4 in the upper half, so the
// two float4 a lane multiplies with one 16-byte weight vector are contiguous across lanes.
__device__ __forceinline__ int xpos(int i, int n) { return ((i >> 3) << 2) + (i & 3) + ((i & 4) ? (n >> 1) : 0); }


// Shared-memory control block (the first kCtlBytes of dynamic shared memory).
struct Ctl {
  uint64_t full[kMaxRingStages];
  uint64_t empty[kMaxRingStages];
  uint32_t stage_rows[kMaxRingStages];  // weight rows held by each stage (written by the producer)
  unsigned abort;       // set once this CTA gave up a wait: later activation waits return at once
  unsigned prod_quit;   // the producer stopped early (its consumers stopped taking stages)
  unsigned skip;        // an earlier step failed: this launch does nothing
  int gtoken;           // greedy decoding: this step's token (polled by thread 0)
  float red[32];        // block reduction scratch
  unsigned long long amax[kComputeWarps + 1];  // greedy decoding: per-warp argmax keys of the LM head
  float2 rope[64];      // cos/sin of this step's position, i < head_dim / 2
  const uint16_t* gain[2 * kMaxLayers + 1];  // attn_norm[l] at 2l, mlp_norm[l] at 2l+1, final at 2L
  const uint16_t* bias[3 * kMaxLayers];      // bq, bk, bv of layer l at 3l..3l+2
  KernelParams params;  // the launch parameters, copied here: reads through a pointer into the
                        // parameter window are slow, shared-memory reads are not
  int32_t pages[kMaxPages];  // paged KV cache: the page table
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block too large");

// ------------------------------------------------------------------ out-of-line slow paths
__device__ __noinline__ void record_failure(unsigned* status, unsigned* host_status, unsigned* abort_flag,
                                            unsigned task, unsigned detail) {
  if (atomicCAS(&status[0], 0u, (unsigned)DS_TIMEOUT) == 0u) {
    status[1] = blockIdx.x;
    status[2] = task;
    status[3] = detail;
    if (host_status) {
      volatile unsigned* hs = host_status;
      hs[1] = blockIdx.x;
      hs[2] = task;
      hs[3] = detail;
      __threadfence_system();
      hs[0] = (unsigned)DS_TIMEOUT;
    }
  }
  *(volatile unsigned*)abort_flag = 1u;
}

// Element offset of KV-cache row `p` of (layer, kv = 0 for K / 1 for V, KV head h), contiguous or paged.
__device__ __forceinline__ size_t kv_off(const KernelParams& P, const Ctl* ctl, int layer, int kv, int h, int p) {
  size_t page = 0;
  int r = p;
  if (P.page_table != nullptr) {
    page = (size_t)(unsigned)ctl->pages[p >> P.page_shift];
    r = p & (P.page_size - 1);
  }
  return page * P.page_elems + ((((size_t)layer * 2 + kv) * P.nkv + h) * P.page_size + r) * P.d;
}

// ------------------------------------------------------------------ per-CTA context (registers)
struct Ctx {
  const KernelParams* P;
  Ctl* ctl;
  unsigned char* ring;
  float* logits;
  unsigned tag;
  int pos, token;
  unsigned ns;          // ring stages
  unsigned stage;       // ring slot of the next stage to consume
  unsigned phase;       // its parity
  int ctid;             // 0..kCT-1 among compute threads
  int warp, lane;       // compute warp 0..kComputeWarps-1
  unsigned task_index;
  bool first_stage;     // tracing: the task has not yet received a weight stage
  bool mma;             // attention on the tensor cores: K/V stages arrive as 128-byte-swizzled tiles
};

__device__ __forceinline__ void trace_mark(Ctx& c, int k) {
  if (c.P->trace != nullptr && c.ctid == 0) c.P->trace[(size_t)c.task_index * kTraceStamps + k] = global_ns();
}
__device__ __forceinline__ bool aborted(const Ctx& c) { return *(volatile unsigned*)&c.ctl->abort != 0u; }
__device__ __forceinline__ void put_word(Ctx& c, unsigned long long* p, float v) {
  if (!aborted(c)) st_word(p, c.tag, v);
}

// Called every 32 unsuccessful polls with the wait's start time (0 on the first call).  Returns the
// start time to keep waiting with, or 0 once the wait must end: this CTA aborted, another CTA
// recorded a failure, or the wait ran past the timeout (which this call then records).  Out of line
// so that the polling loops stay small; it runs once per 32 polls.
__device__ __noinline__ unsigned long long wait_check(const KernelParams* P, Ctl* ctl, unsigned long long t0,
                                                      unsigned task, unsigned detail) {
  if (*(volatile unsigned*)&ctl->abort) return 0ull;
  const unsigned long long now = global_ns();
  if (t0 == 0ull) return now;
  if (*(volatile unsigned*)P->status != 0u || now - t0 > P->timeout_ns) {
    record_failure(P->status, P->host_status, &ctl->abort, task, detail);
    return 0ull;
  }
  return t0;
}

// ------------------------------------------------------------------ activation input of a task
// A vector a task reads: element e (0 <= e < n) is the word src[e], or -- with src == nullptr --
// the bf16 value emb[e] (the token's embedding row).  Values land in dst, in the split GEMV layout
// when xlayout.  With a gain the values stored are x * gain[e] and the sum of squares of x is
// returned: RMSNorm's 1/sqrt(mean(x^2) + eps) is applied to the GEMV results instead, so the norm
// costs no pass of its own (the pages' "folding" of small producers into their consumer).
struct InVec {
  const unsigned long long* src;
  const uint16_t* emb;
  const uint16_t* gain;
  float* dst;
  int n, xlayout;
  // up to three segments: elements [0, n1) from src, [n1, n1 + n2) from src2, the rest from src3
  // (one poll for a KV head's queries, key and value); n1 = n for a plain vector
  const unsigned long long* src2;
  const unsigned long long* src3;
  int n1, n2;
  // with nterm > 0 every element also adds nterm words terms[t * tstride + e] (the per-KV-head
  // partial O projections), summed in t order after the base value (poll_sum)
  const unsigned long long* terms;
  int nterm, tstride;
};
// Where element e of a polled vector lands: in order (xlayout 0), in the split GEMV layout (1), or
// (2, an attention task's queries | K | V, n1 = g * d query elements, n2 = d) with every query head in
// a row of d + d/8 floats in which each run of 32 elements sits 16 bytes after the previous one
// (attn_qpos), the K and V rows after the heads.
__device__ __forceinline__ int attn_qpos(int i) { return i + ((i >> 5) << 2); }  // i < d: element of one head
__device__ __forceinline__ int dst_index(const InVec& v, int e) {
  if (v.xlayout == 1) return xpos(e, v.n);
  if (v.xlayout == 2) {
    const int dsh = 31 - __clz(v.n2);
    if (e < v.n1) return (e >> dsh) * (v.n2 + (v.n2 >> 3)) + attn_qpos(e & (v.n2 - 1));
    return v.n1 + (v.n1 >> 3) + (e - v.n1);
  }
  return e;
}
__device__ __forceinline__ const unsigned long long* word_addr(const InVec& v, int e) {
  return e < v.n1 ? v.src + e : (e < v.n1 + v.n2 ? v.src2 + (e - v.n1) : v.src3 + (e - v.n1 - v.n2));
}

// Threads tid = 0..nth-1 poll elements tid + k*nth, kPollWords at a time; all loads of a group are in
// flight together and every retry re-loads all words still pending, so a late group costs one round
// trip per retry, not one per word (the hidden and intermediate vectors of the decoder shapes fit one
// group).  The gains are loaded with the words and used only after the group arrived, so their
// latency hides behind the wait.  Values are consumed in element order whatever their arrival order,
// which keeps the sum of squares deterministic.  After a failed wait the remaining words read as 0.
constexpr int kPollWords = 8;
__device__ __forceinline__ float poll_vec(Ctx& c, const InVec& v, unsigned detail, int tid = -1, int nth = kCT) {
  if (tid < 0) tid = c.ctid;
  float ss = 0.f;
#pragma unroll 1
  for (int e0 = tid; e0 < v.n; e0 += kPollWords * nth) {
    unsigned long long w[kPollWords];
    uint32_t graw[kPollWords];
    unsigned pend = 0u;
#pragma unroll
    for (int k = 0; k < kPollWords; ++k) {
      const int e = e0 + k * nth;
      w[k] = 0ull;
      graw[k] = 0x3f80u;  // bf16 1.0
      if (e < v.n) {
        if (v.src != nullptr) {
          w[k] = ld_word(word_addr(v, e));
          pend |= 1u << k;
        } else {
          w[k] = (unsigned long long)((uint32_t)v.emb[e] << 16);
        }
        if (v.gain != nullptr) graw[k] = v.gain[e];
      }
    }
    unsigned spins = 0u;
    unsigned long long t0 = 0ull;
    while (pend != 0u) {
#pragma unroll
      for (int k = 0; k < kPollWords; ++k)
        if (((pend >> k) & 1u) && (unsigned)(w[k] >> 32) == c.tag) pend &= ~(1u << k);
      if (pend == 0u) break;
      if ((++spins & 31u) == 0u && (t0 = wait_check(c.P, c.ctl, t0, c.task_index, detail | (unsigned)e0)) == 0ull) {
#pragma unroll
        for (int k = 0; k < kPollWords; ++k)
          if ((pend >> k) & 1u) w[k] = 0ull;
        break;
      }
      if (c.P->poll_backoff_ns) __nanosleep(c.P->poll_backoff_ns);
#pragma unroll
      for (int k = 0; k < kPollWords; ++k) {
        const int e = e0 + k * nth;
        if ((pend >> k) & 1u) w[k] = ld_word(word_addr(v, e));
      }
    }
#pragma unroll
    for (int k = 0; k < kPollWords; ++k) {
      const int e = e0 + k * nth;
      if (e < v.n) {
        float x = __uint_as_float((uint32_t)w[k]);
        if (v.gain != nullptr) {
          ss = fmaf(x, x, ss);
          x *= __uint_as_float(graw[k] << 16);
        }
        v.dst[dst_index(v, e)] = x;
      }
    }
  }
  return ss;
}

// poll_vec for vectors that are sums: element e = base word (or embedding value) + the nterm
// partial words of e, two elements per thread at a time with every word of both in flight together.
// The sum is taken in a fixed order (base, then heads in order), so it is deterministic.
__device__ __forceinline__ float poll_sum(Ctx& c, const InVec& v, unsigned detail, int tid = -1, int nth = kCT) {
  if (tid < 0) tid = c.ctid;
  constexpr int T = 1 + kMaxFusedKvHeads;
  const int nt = 1 + v.nterm;
  float ss = 0.f;
#pragma unroll 1
  for (int e0 = tid; e0 < v.n; e0 += 2 * nth) {
    unsigned long long w[2][T];
    uint32_t graw[2];
    unsigned pend = 0u;  // bit k * T + t
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int e = e0 + k * nth;
      graw[k] = 0x3f80u;
#pragma unroll
      for (int t = 0; t < T; ++t) w[k][t] = 0ull;
      if (e < v.n) {
        if (v.src != nullptr) {
          w[k][0] = ld_word(v.src + e);
          pend |= 1u << (k * T);
        } else {
          w[k][0] = (unsigned long long)((uint32_t)v.emb[e] << 16);
        }
#pragma unroll
        for (int t = 1; t < T; ++t)
          if (t < nt) {
            w[k][t] = ld_word(v.terms + (size_t)(t - 1) * v.tstride + e);
            pend |= 1u << (k * T + t);
          }
        if (v.gain != nullptr) graw[k] = v.gain[e];
      }
    }
    unsigned spins = 0u;
    unsigned long long t0 = 0ull;
    while (pend != 0u) {
#pragma unroll
      for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int t = 0; t < T; ++t)
          if (((pend >> (k * T + t)) & 1u) && (unsigned)(w[k][t] >> 32) == c.tag) pend &= ~(1u << (k * T + t));
      if (pend == 0u) break;
      if ((++spins & 31u) == 0u && (t0 = wait_check(c.P, c.ctl, t0, c.task_index, detail | (unsigned)e0)) == 0ull) {
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
          for (int t = 0; t < T; ++t)
            if ((pend >> (k * T + t)) & 1u) w[k][t] = 0ull;
        break;
      }
      if (c.P->poll_backoff_ns) __nanosleep(c.P->poll_backoff_ns);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int e = e0 + k * nth;
        if ((pend >> (k * T)) & 1u) w[k][0] = ld_word(v.src + e);
#pragma unroll
        for (int t = 1; t < T; ++t)
          if ((pend >> (k * T + t)) & 1u) w[k][t] = ld_word(v.terms + (size_t)(t - 1) * v.tstride + e);
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int e = e0 + k * nth;
      if (e < v.n) {
        float x = __uint_as_float((uint32_t)w[k][0]);
#pragma unroll
        for (int t = 1; t < T; ++t)
          if (t < nt) x += __uint_as_float((uint32_t)w[k][t]);
        if (v.gain != nullptr) {
          ss = fmaf(x, x, ss);
          x *= __uint_as_float(graw[k] << 16);
        }
        v.dst[v.xlayout ? xpos(e, v.n) : e] = x;
      }
    }
  }
  return ss;
}

// ------------------------------------------------------------------ weight ring (consumer side)
// Keeps testing a ring stage whose first test failed; records a failure after the timeout.
__device__ __noinline__ void spin_stage(uint64_t* full, unsigned parity, const KernelParams* P, Ctl* ctl, unsigned task,
                                        unsigned detail) {
  const unsigned long long t0 = global_ns();
  while (!mbar_test(full, parity)) {
    if (*(volatile unsigned*)&ctl->prod_quit) return;  // nothing more will arrive
    if (global_ns() - t0 > P->timeout_ns) {
      record_failure(P->status, P->host_status, &ctl->abort, task, detail);
      return;
    }
  }
}
// Ring slot `k` stages after the current one (k < ns): its slot index and parity.
__device__ __forceinline__ void slot_after(const Ctx& c, unsigned k, unsigned& s, unsigned& ph) {
  s = c.stage + k;
  ph = c.phase;
  if (s >= c.ns) {
    s -= c.ns;
    ph ^= 1u;
  }
}
// The stage k after the current one, once its data has landed.
__device__ __forceinline__ unsigned char* stage_wait(Ctx& c, unsigned k) {
  unsigned s, ph;
  slot_after(c, k, s, ph);
  if (!mbar_test(&c.ctl->full[s], ph)) spin_stage(&c.ctl->full[s], ph, c.P, c.ctl, c.task_index, 0xF000u | s);
  if (c.first_stage) {
    trace_mark(c, 3);
    c.first_stage = false;
  }
  return c.ring + (size_t)s * kStageBytes;
}
__device__ __forceinline__ unsigned stage_rows_at(const Ctx& c, unsigned k) {
  unsigned s, ph;
  slot_after(c, k, s, ph);
  return c.ctl->stage_rows[s];
}
// Hand `n` stages back to the producer (every compute warp arrives once per stage).
__device__ __forceinline__ void stages_release(Ctx& c, unsigned n) {
  __syncwarp();
#pragma unroll 1
  for (unsigned k = 0; k < n; ++k) {
    if (c.lane == 0) mbar_arrive(&c.ctl->empty[c.stage]);
    if (++c.stage == c.ns) {
      c.stage = 0;
      c.phase ^= 1u;
    }
  }
}

__device__ __forceinline__ unsigned long long* layer_words(const KernelParams& P, int l) {
  return P.words + (size_t)l * P.act.per_layer;
}
// Words of the residual stream entering layer l >= 1: the previous layer's output, or -- in the
// diagnostic mode that checks every layer from the same inputs as a reference -- injected words.
__device__ __forceinline__ const unsigned long long* x_in_words(const KernelParams& P, int l) {
  if (l == 0) return nullptr;  // the embedding row
  return P.inject != nullptr ? P.inject + (size_t)l * P.H : layer_words(P, l - 1) + P.act.xm;
}

__device__ __forceinline__ unsigned long long pack2(uint32_t lo, uint32_t hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b, unsigned long long acc) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(acc));
  return d;
}
__device__ __forceinline__ float sum2(unsigned long long v) {
  return __uint_as_float((uint32_t)v) + __uint_as_float((uint32_t)(v >> 32));
}
// bf16 pair in one 32-bit word -> fp32x2 {element 2i, element 2i+1}
__device__ __forceinline__ unsigned long long bf2(uint32_t w) { return pack2(w << 16, w & 0xffff0000u); }
// Two FP8 E4M3 weights (low byte first) as a packed fp32 pair: E4M3 -> f16 is exact (one
// instruction for both), then f16 -> f32.  (Re-basing the f16 bits as fp32 with integer operations
// instead of the two conversions measured slower.)
__device__ __forceinline__ unsigned long long f8x2(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)(two & 0xffffu)));
  float lo, hi;
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi) : "r"(h2));
  return pack2(__float_as_uint(lo), __float_as_uint(hi));
}
// A weight "vector": 8 consecutive weights of a row, 16 bytes of bf16 or (F8) 8 bytes of E4M3 codes
// (held in .x and .y).  wpair<F8>(w, j) gives weights 2j and 2j + 1 as a packed fp32 pair.
template <bool F8>
__device__ __forceinline__ uint4 wload(const unsigned char* row, int v) {
  if constexpr (F8) {
    const uint2 w = reinterpret_cast<const uint2*>(row)[v];
    return make_uint4(w.x, w.y, 0u, 0u);
  } else {
    return reinterpret_cast<const uint4*>(row)[v];
  }
}
template <bool F8>
__device__ __forceinline__ unsigned long long wpair(const uint4& w, int j) {
  if constexpr (F8)
    return f8x2(j == 0 ? w.x : j == 1 ? (w.x >> 16) : j == 2 ? w.y : (w.y >> 16));
  else
    return bf2(j == 0 ? w.x : j == 1 ? w.y : j == 2 ? w.z : w.w);
}

template <bool F8>
__device__ __forceinline__ void gemv_xreg(Ctx& c, const Task& t, int in, const float* x, float* res, float scale) {
  const int nvec = in >> 3;  // 8-weight vectors per row
  const int gpr = (int)t.gpr, gshift = 31 - __clz(gpr);
  // warp = rw * gpr + slice; warps beyond the last whole group (rw >= rpp) take no rows
  const int slice = c.warp & (gpr - 1), rw = c.warp >> gshift, rpp = kComputeWarps >> gshift;
  const int rstart = rw < rpp ? rw : 1 << 30;
  const int vps = (nvec + gpr - 1) >> gshift;  // vectors per slice
  const int v0 = slice * vps, v1 = min(nvec, v0 + vps);
  // this lane's x: vectors v0 + lane + 32k, as packed pairs
  unsigned long long xp[kGemvXVec][4];
  const float* xhi = x + (in >> 1);
#pragma unroll
  for (int k = 0; k < kGemvXVec; ++k) {
    const int v = v0 + c.lane + 32 * k;
    float4 p = make_float4(0.f, 0.f, 0.f, 0.f), q = p;
    if (v < v1) {
      p = reinterpret_cast<const float4*>(x)[v];
      q = reinterpret_cast<const float4*>(xhi)[v];
    }
    xp[k][0] = pack2(__float_as_uint(p.x), __float_as_uint(p.y));
    xp[k][1] = pack2(__float_as_uint(p.z), __float_as_uint(p.w));
    xp[k][2] = pack2(__float_as_uint(q.x), __float_as_uint(q.y));
    xp[k][3] = pack2(__float_as_uint(q.z), __float_as_uint(q.w));
  }
  const size_t row_bytes = (size_t)in * (F8 ? 1 : 2);
  int rbase = 0;
  for (uint32_t k0 = 0; k0 < t.nchunks; k0 += kGemvBatch) {
    const int nb = (int)min((uint32_t)kGemvBatch, t.nchunks - k0);
    const unsigned char* s0 = stage_wait(c, 0);
    const unsigned char* s1 = nb > 1 ? stage_wait(c, 1) : s0;
    const unsigned char* s2 = nb > 2 ? stage_wait(c, 2) : s0;
    const unsigned char* s3 = nb > 3 ? stage_wait(c, 3) : s0;
    const int n0 = (int)stage_rows_at(c, 0);
    const int n1 = nb > 1 ? (int)stage_rows_at(c, 1) : 0;
    const int n2 = nb > 2 ? (int)stage_rows_at(c, 2) : 0;
    const int n3 = nb > 3 ? (int)stage_rows_at(c, 3) : 0;
    const int total = n0 + n1 + n2 + n3;
    auto row_of = [&](int r) -> const unsigned char* {
      const unsigned char* base = s0;
      if (r >= n0) {
        r -= n0;
        base = s1;
        if (r >= n1) {
          r -= n1;
          base = s2;
          if (r >= n2) {
            r -= n2;
            base = s3;
          }
        }
      }
      return base + (size_t)r * row_bytes;
    };
    // four rows per iteration (independent accumulator chains); the loop bound is uniform across
    // the warp (shuffles below)
    for (int ra = rstart; ra < total; ra += 4 * rpp) {
      const unsigned char* R[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) R[i] = row_of(ra + i * rpp < total ? ra + i * rpp : ra);
      unsigned long long acc[4][2];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = 0ull;
#pragma unroll
      for (int k = 0; k < kGemvXVec; ++k) {
        const int v = v0 + c.lane + 32 * k;
        const int vi = v < v1 ? v : 0;  // clamped index; its x registers are zero
        uint4 w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = wload<F8>(R[i], vi);
        if (v >= v1) {
#pragma unroll
          for (int i = 0; i < 4; ++i) w[i] = make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[i][0] = ffma2(wpair<F8>(w[i], 0), xp[k][0], acc[i][0]);
          acc[i][1] = ffma2(wpair<F8>(w[i], 1), xp[k][1], acc[i][1]);
          acc[i][0] = ffma2(wpair<F8>(w[i], 2), xp[k][2], acc[i][0]);
          acc[i][1] = ffma2(wpair<F8>(w[i], 3), xp[k][3], acc[i][1]);
        }
      }
      float sm[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sm[i] = sum2(acc[i][0]) + sum2(acc[i][1]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) sm[i] += __shfl_xor_sync(0xffffffffu, sm[i], o);
      }
      if (c.lane == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (ra + i * rpp < total) res[((rbase + ra + i * rpp) << gshift) + slice] = sm[i] * scale;
      }
    }
    stages_release(c, (unsigned)nb);
    rbase += total;
  }
  compute_sync();
}

constexpr int kDotRound = 2;  // 16-byte vectors per lane per round of a row dot product
// Loads of one round are issued unconditionally (an index past the row end is clamped to the row
// start and its weights zeroed), so they are all in flight before the first FMA.
template <bool F8>
__device__ __forceinline__ float dot_row(const Ctx& c, const unsigned char* row, const float4* xlo, const float4* xhi, int nvec) {
  unsigned long long a0 = 0ull, a1 = 0ull;
#pragma unroll 1
  for (int v0 = c.lane; v0 < nvec; v0 += 32 * kDotRound) {
    uint4 w[kDotRound];
    float4 p[kDotRound], q[kDotRound];
#pragma unroll
    for (int it = 0; it < kDotRound; ++it) {
      const int v = v0 + 32 * it;
      const int vi = v < nvec ? v : v0;
      w[it] = wload<F8>(row, vi);
      p[it] = xlo[vi];
      q[it] = xhi[vi];
      if (v >= nvec) w[it] = make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int it = 0; it < kDotRound; ++it) {
      a0 = ffma2(wpair<F8>(w[it], 0), pack2(__float_as_uint(p[it].x), __float_as_uint(p[it].y)), a0);
      a1 = ffma2(wpair<F8>(w[it], 1), pack2(__float_as_uint(p[it].z), __float_as_uint(p[it].w)), a1);
      a0 = ffma2(wpair<F8>(w[it], 2), pack2(__float_as_uint(q[it].x), __float_as_uint(q[it].y)), a0);
      a1 = ffma2(wpair<F8>(w[it], 3), pack2(__float_as_uint(q[it].z), __float_as_uint(q[it].w)), a1);
    }
  }
  return sum2(a0) + sum2(a1);
}
// Two rows against the same x (gate and up rows): the x vectors are loaded once for both.
template <bool F8>
__device__ __forceinline__ void dot_row2(const Ctx& c, const unsigned char* ra, const unsigned char* rb, const float4* xlo,
                                         const float4* xhi, int nvec, float& sa, float& sb) {
  unsigned long long a0 = 0ull, a1 = 0ull, b0 = 0ull, b1 = 0ull;
#pragma unroll 1
  for (int v0 = c.lane; v0 < nvec; v0 += 64) {
    uint4 wa[2], wb[2];
    float4 p[2], q[2];
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int v = v0 + 32 * it;
      const int vi = v < nvec ? v : v0;
      wa[it] = wload<F8>(ra, vi);
      wb[it] = wload<F8>(rb, vi);
      p[it] = xlo[vi];
      q[it] = xhi[vi];
      if (v >= nvec) wa[it] = wb[it] = make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const unsigned long long x0 = pack2(__float_as_uint(p[it].x), __float_as_uint(p[it].y));
      const unsigned long long x1 = pack2(__float_as_uint(p[it].z), __float_as_uint(p[it].w));
      const unsigned long long x2 = pack2(__float_as_uint(q[it].x), __float_as_uint(q[it].y));
      const unsigned long long x3 = pack2(__float_as_uint(q[it].z), __float_as_uint(q[it].w));
      a0 = ffma2(wpair<F8>(wa[it], 0), x0, a0);
      a1 = ffma2(wpair<F8>(wa[it], 1), x1, a1);
      a0 = ffma2(wpair<F8>(wa[it], 2), x2, a0);
      a1 = ffma2(wpair<F8>(wa[it], 3), x3, a1);
      b0 = ffma2(wpair<F8>(wb[it], 0), x0, b0);
      b1 = ffma2(wpair<F8>(wb[it], 1), x1, b1);
      b0 = ffma2(wpair<F8>(wb[it], 2), x2, b0);
      b1 = ffma2(wpair<F8>(wb[it], 3), x3, b1);
    }
  }
  sa = sum2(a0) + sum2(a1);
  sb = sum2(b0) + sum2(b1);
}
// Rows of the stages of one batch, in chunk order: row r of the batch.
struct BatchRows {
  const unsigned char* s[kGemvBatch];
  int n[kGemvBatch];
  int total;
  __device__ __forceinline__ const unsigned char* row(int r, size_t row_bytes) const {
    const unsigned char* base = s[0];
    if (r >= n[0]) {
      r -= n[0];
      base = s[1];
      if (r >= n[1]) {
        r -= n[1];
        base = s[2];
        if (r >= n[2]) {
          r -= n[2];
          base = s[3];
        }
      }
    }
    return base + (size_t)r * row_bytes;
  }
};
__device__ __forceinline__ BatchRows batch_wait(Ctx& c, int nb) {
  BatchRows b;
  b.s[0] = stage_wait(c, 0);
  b.s[1] = nb > 1 ? stage_wait(c, 1) : b.s[0];
  b.s[2] = nb > 2 ? stage_wait(c, 2) : b.s[0];
  b.s[3] = nb > 3 ? stage_wait(c, 3) : b.s[0];
  b.n[0] = (int)stage_rows_at(c, 0);
  b.n[1] = nb > 1 ? (int)stage_rows_at(c, 1) : 0;
  b.n[2] = nb > 2 ? (int)stage_rows_at(c, 2) : 0;
  b.n[3] = nb > 3 ? (int)stage_rows_at(c, 3) : 0;
  b.total = b.n[0] + b.n[1] + b.n[2] + b.n[3];
  return b;
}

__device__ __forceinline__ float res_row(const float* res, int i, int gpr) {
  if (gpr <= 1) return res[i];
  float v = 0.f;
  for (int s = 0; s < gpr; ++s) v += res[i * gpr + s];
  return v;
}

// One rotate-half RoPE pair: (x0, x1) at (i, i + d/2) turned by the angle whose cosine and sine are
// r.x and r.y.  Products and sums are rounded one at a time (no contraction), so every site that
// rotates the same values gets the same bits -- the K row appended to the cache and the score this
// step takes with it.
__device__ __forceinline__ float2 rope_rot(float x0, float x1, float2 r) {
  return make_float2(__fsub_rn(__fmul_rn(x0, r.x), __fmul_rn(x1, r.y)), __fadd_rn(__fmul_rn(x1, r.x), __fmul_rn(x0, r.y)));
}

// ------------------------------------------------------------------ attention on the tensor cores
// Head dimension 64, at most 8 query heads per KV head.  The producer brings each stage's K rows
// (64 of them, 128 bytes each) and then its V rows as 2-D TMA tiles with the 128-byte swizzle: the
// 16-byte chunk c of row r sits at chunk c ^ (r & 7), so the 8 rows a fragment load touches fall in
// different banks.  Both products run transposed on mma.sync m16n8k16 (bf16 operands, fp32
// accumulation), so that the 16-row side of the tile holds positions or dimensions and the 8-column
// side the (at most 8) query heads:
//   S^T = K Q^T   A = 16 K rows (ldmatrix), B = the queries, rows = positions, cols = heads;
//   O^T += V^T P^T  A = V rows loaded transposed (ldmatrix.trans), rows = 16 of the 64 dimensions;
//                   B = the probabilities: S^T's accumulator fragments as bf16, transposed 8x8 in
//                   registers (movmatrix).
// fp32 operands reach the bf16 MMAs as high/low pairs (x = hi + lo, hi = bf16(x), lo = bf16(x - hi)):
// two MMAs per product, with the relative error of the pair (about 2^-17) instead of bf16's 2^-9.
// K and V are bf16 in the cache, so they go in exactly.
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const float h0 = __bfloat162float(__float2bfloat16_rn(x0)), h1 = __bfloat162float(__float2bfloat16_rn(x1));
  hi = bf16x2(h0, h1);
  lo = bf16x2(x0 - h0, x1 - h1);
}
// D += A B for one m16n8k16 tile
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                          uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
constexpr int kMmaRows = kStageBytes / (2 * 64 * 2);  // K (then V) rows of one stage at head_dim 64
// byte offset of 16-byte chunk `ch` of row r inside a swizzled tile of 128-byte rows (1024-byte aligned)
__device__ __forceinline__ uint32_t swz128(int r, int ch) { return (uint32_t)r * 128u + (uint32_t)((ch ^ (r & 7)) << 4); }

// The (block, head) work of one attention task on the tensor cores.  16-position blocks of the nh
// cached rows go round-robin over the compute warps; each warp keeps a running softmax (max m, sum l,
// unnormalised o) per query head over its blocks and writes it as one partial; the current row
// (owner split) is a partial of its own (m = its score, l = 1, o = its V row).  Partial p of head h
// goes to pw + (p * g + h) * (d + 4) as o[d], m, l -- the item layout the merge reads.  Returns the
// number of partials.  sq holds the raw (not yet rotated) fp32 queries (attn_qpos layout, QS floats
// a head), kv the raw current K and V rows (fp32), s_first the ring slot of the task's first stage.
__device__ __forceinline__ int attn_items_mma(Ctx& c, const float* sq, int QS, int g, int nh, bool owner,
                                              const float* kv, unsigned s_first, float scale, float* pw) {
  constexpr int D = 64;
  const int gid = c.lane >> 2, tig = c.lane & 3, mi = c.lane >> 3, rr = c.lane & 7;
  const int nkb = (nh + 15) >> 4;
  const int nwp = min(kComputeWarps, nkb);
  const float2* cs = c.ctl->rope;  // this step's cos/sin
  if (c.warp < nkb) {
    // B = Q^T: b0 = Q[head gid][16 ks + 2 tig, +1], b1 = the same 8 columns on (zero for heads >= g).
    // The lane holds both halves of each rotate-half pair it needs (columns i and i + 32 sit in
    // k-steps ks and ks + 2), so it applies RoPE to the raw queries itself.
    float qv[4][2][2];
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float2 x = make_float2(0.f, 0.f);
        if (gid < g) x = *reinterpret_cast<const float2*>(sq + gid * QS + attn_qpos(16 * ks + 8 * hf + 2 * tig));
        qv[ks][hf][0] = x.x;
        qv[ks][hf][1] = x.y;
      }
    }
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float2 y = rope_rot(qv[ks][hf][e], qv[ks + 2][hf][e], cs[16 * ks + 8 * hf + 2 * tig + e]);
          qv[ks][hf][e] = y.x;
          qv[ks + 2][hf][e] = y.y;
        }
      }
    }
    uint32_t qh[4][2], ql[4][2];
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) split_pair(qv[ks][hf][0], qv[ks][hf][1], qh[ks][hf], ql[ks][hf]);
    }
    float ot[4][4];  // O^T tile mt: dims 16 mt + gid (+ 8) by heads 2 tig, 2 tig + 1
#pragma unroll
    for (int i = 0; i < 4; ++i) ot[i][0] = ot[i][1] = ot[i][2] = ot[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2 tig and 2 tig + 1 (l: this lane's rows)
#pragma unroll 1
    for (int kb = c.warp; kb < nkb; kb += kComputeWarps) {
      const int j0 = kb << 4, r0 = j0 & (kMmaRows - 1);
      unsigned slot = s_first + (unsigned)(j0 / kMmaRows);
      slot = slot >= c.ns ? slot - c.ns : slot;
      const uint32_t kaddr = smem_addr(c.ring + (size_t)slot * kStageBytes), vaddr = kaddr + kMmaRows * 128u;
      // S^T: A = K rows r0 .. r0 + 15 by dims 16 ks .. 16 ks + 15 (one ldmatrix.x4 per k-step)
      const int arow = r0 + rr + ((mi & 1) ? 8 : 0);
      float sh[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kaddr + swz128(arow, 2 * ks + (mi >> 1)), a0, a1, a2, a3);
        mma_16816(sh, a0, a1, a2, a3, qh[ks][0], qh[ks][1]);
        mma_16816(sl, a0, a1, a2, a3, ql[ks][0], ql[ks][1]);
      }
      // sc[0], sc[1]: position j0 + gid, heads 2 tig, 2 tig + 1; sc[2], sc[3]: position j0 + gid + 8
      float sc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = j0 + gid + ((k & 2) ? 8 : 0);
        sc[k] = j < nh ? (sh[k] + sl[k]) * scale : -INFINITY;
      }
      float bm0 = fmaxf(sc[0], sc[2]), bm1 = fmaxf(sc[1], sc[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {  // over the 8 lanes holding the block's other positions
        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
      }
      const float nm0 = fmaxf(m0, bm0), nm1 = fmaxf(m1, bm1);  // finite: position j0 < nh is valid
      const float cr0 = exp2f(m0 - nm0), cr1 = exp2f(m1 - nm1);  // rescale of the running sums (0 at first)
      m0 = nm0;
      m1 = nm1;
      const float p0 = exp2f(sc[0] - m0), p1 = exp2f(sc[1] - m1), p2 = exp2f(sc[2] - m0), p3 = exp2f(sc[3] - m1);
      l0 = fmaf(l0, cr0, p0 + p2);
      l1 = fmaf(l1, cr1, p1 + p3);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        ot[i][0] *= cr0;
        ot[i][1] *= cr1;
        ot[i][2] *= cr0;
        ot[i][3] *= cr1;
      }
      // B = P^T (k = positions, n = heads)
      uint32_t h01, l01, h23, l23;
      split_pair(p0, p1, h01, l01);
      split_pair(p2, p3, h23, l23);
      const uint32_t bh0 = transpose8x8(h01), bh1 = transpose8x8(h23), bl0 = transpose8x8(l01), bl1 = transpose8x8(l23);
      // O^T: A = V^T, dims 16 mt .. 16 mt + 15 by the block's 16 positions
      const int vrow = r0 + rr + ((mi & 2) ? 8 : 0);
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(vaddr + swz128(vrow, 2 * mt + (mi & 1)), a0, a1, a2, a3);
        mma_16816(ot[mt], a0, a1, a2, a3, bh0, bh1);
        mma_16816(ot[mt], a0, a1, a2, a3, bl0, bl1);
      }
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = 2 * tig + hh;
      if (h < g) {
        float* pp = pw + (size_t)(c.warp * g + h) * (D + 4);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          pp[16 * mt + gid] = ot[mt][hh];
          pp[16 * mt + gid + 8] = ot[mt][2 + hh];
        }
        if (gid == 0) {
          pp[D] = hh ? m1 : m0;
          pp[D + 1] = hh ? l1 : l0;
        }
      }
    }
  }
  if (owner) {  // the current row: head h on warp kComputeWarps - 1 - h (the warps with the fewest blocks)
    const int h = kComputeWarps - 1 - c.warp;
    if (h >= 0 && h < g) {
      // lane: elements 2 lane, 2 lane + 1 of the raw query and of the raw K and V rows (kv); the
      // rotate-half partner of element i < 32 is i + 32, in lane (lane + 16) mod 32.  K is rotated
      // and rounded exactly as the row appended to the cache.
      const int e = 2 * c.lane;
      const bool lo = c.lane < 16;
      const float2 q = *reinterpret_cast<const float2*>(sq + h * QS + attn_qpos(e));
      const float2 k = *reinterpret_cast<const float2*>(kv + e);
      const float2 v = *reinterpret_cast<const float2*>(kv + D + e);
      const float q0p = __shfl_xor_sync(0xffffffffu, q.x, 16), q1p = __shfl_xor_sync(0xffffffffu, q.y, 16);
      const float k0p = __shfl_xor_sync(0xffffffffu, k.x, 16), k1p = __shfl_xor_sync(0xffffffffu, k.y, 16);
      const float2 r0 = cs[e & 31], r1 = cs[(e + 1) & 31];
      const float2 qa = lo ? rope_rot(q.x, q0p, r0) : rope_rot(q0p, q.x, r0);
      const float2 qb = lo ? rope_rot(q.y, q1p, r1) : rope_rot(q1p, q.y, r1);
      const float2 ka = lo ? rope_rot(k.x, k0p, r0) : rope_rot(k0p, k.x, r0);
      const float2 kb = lo ? rope_rot(k.y, k1p, r1) : rope_rot(k1p, k.y, r1);
      const float q0 = lo ? qa.x : qa.y, q1 = lo ? qb.x : qb.y;
      const float k0 = __bfloat162float(__float2bfloat16_rn(lo ? ka.x : ka.y));
      const float k1 = __bfloat162float(__float2bfloat16_rn(lo ? kb.x : kb.y));
      const float sdot = warp_sum(fmaf(q0, k0, q1 * k1));
      float* pp = pw + (size_t)(nwp * g + h) * (D + 4);
      *reinterpret_cast<float2*>(pp + e) =
          make_float2(__bfloat162float(__float2bfloat16_rn(v.x)), __bfloat162float(__float2bfloat16_rn(v.y)));
      if (c.lane == 0) {
        pp[D] = sdot * scale;
        pp[D + 1] = 1.f;
      }
    }
  }
  return nwp + (owner ? 1 : 0);
}

// ------------------------------------------------------------------ attention task
// One KV head, one context split: the g query heads sharing the KV head are packed into the task,
// so each K/V row is read once from HBM (README, "Current status", decode attention).  Cached
// positions [a, min(a + split_len, pos)) arrive through the ring (all of the task's stages are
// held at once); the owner split (the one holding `pos`) also takes the current row from the QKV
// words, rotates and rounds it, appends it to the cache and attends to it.
// Work items are (32-position block, query head) pairs, spread over the warps; in an item every
// lane owns one position: it computes that position's score alone (no cross-lane reduction), the
// warp takes the block's max and sum, and the lanes then accumulate the block's output with each
// lane owning output elements.  One barrier later the blocks of each head are merged by their
// log-sum-exp weights.  Writes per query head o (normalised over this split) and (m, l); scores
// are kept in base-2 units (scaled by log2 e), so m is too.
template <bool F8>
__device__ __forceinline__ void task_attn(Ctx& c, const Task& t, float* sv, float* res) {
  const KernelParams& P = *c.P;
  const bool wo = (t.flags & TF_WO) != 0;  // fused O projection: KV head in aux, output rows row0..
  const int l = t.layer, kvh = wo ? (int)t.aux : (int)t.row0, sp = wo ? 0 : (int)t.nrows;
  const int d = P.d, g = P.g, R = P.rows_per_stage, half = d / 2;
  const int dshift = 31 - __clz(d), hshift = dshift - 1;
  const int pos = c.pos;
  const int a = sp * P.split_len;
  if (a > pos) return;  // inactive split (the producer streamed nothing for it either)
  const int b = min(a + P.split_len, pos);
  const bool owner = (pos / P.split_len) == sp;
  const int nh = b - a;                       // cached positions
  const int np = nh + (owner ? 1 : 0);        // positions attended
  const int nst = (nh + R - 1) / R;           // ring stages of this task
  const int O = g * d;
  const int nblk = (np + 31) >> 5;            // 32-position blocks
  const int items = nblk * g;

  const int QS = d + (d >> 3);                // floats per query head (attn_qpos: each run of 32 elements
                                              // 16 bytes after the previous one, so that lane-rotated
                                              // 16-byte chunk reads of a head touch distinct banks)
  float* sq = sv;                             // [g][QS]  queries (rotated in place)
  float* kc = sq + g * QS;                    // [d]     current K (raw)
  float* vc = kc + d;                         // [d]     current V (raw)
  uint16_t* cur = reinterpret_cast<uint16_t*>(vc + d);  // [2][d] bf16: the rotated K, V row appended
  float* pw = vc + 2 * d;                     // [items][d + 4]  per-item o, m, l (16-byte aligned items)
  float* pbw = pw + items * (d + 4) + c.warp * 32;  // [warp][32]  this warp's item probabilities
  const float2* cs = c.ctl->rope;             // this step's cos/sin (loaded at kernel start)

  // 1. the packed queries and (owner) the current K/V row, in one poll: they land in sq|kc|vc
  {
    const unsigned long long* w = layer_words(P, l) + P.act.qkv;
    const int qd = P.nq * d, kvd = P.nkv * d;
    InVec v;
    v.src = w + (size_t)kvh * O;
    v.src2 = w + qd + kvh * d;
    v.src3 = w + qd + kvd + kvh * d;
    v.n1 = O;
    v.n2 = d;
    v.n = owner ? O + 2 * d : O;
    v.emb = nullptr;
    v.gain = nullptr;
    v.dst = sq;
    v.xlayout = 2;
    v.terms = nullptr;
    v.nterm = 0;
    v.tstride = 0;
    poll_vec(c, v, 0x200000u);
  }
  compute_sync();
  trace_mark(c, 1);
  // RoPE (rotate-half pairs (i, i + d/2)) of the queries, in place (the tensor-core path rotates
  // them in its fragments instead); the current K/V row is rounded to bf16 and appended
  if (!c.mma) {
#pragma unroll 1
    for (int e = c.ctid; e < g * half; e += kCT) {
      const int h = e >> hshift, i = e & (half - 1);
      float* q = sq + h * QS;
      const int i0 = attn_qpos(i), i1 = attn_qpos(i + half);
      const float2 y = rope_rot(q[i0], q[i1], cs[i]);
      q[i0] = y.x;
      q[i1] = y.y;
    }
  }
  if (owner && c.ctid >= kCT - half) {
    const int i = c.ctid - (kCT - half);
    const float2 y = rope_rot(kc[i], kc[i + half], cs[i]);
    const __nv_bfloat16 k0 = __float2bfloat16_rn(y.x);
    const __nv_bfloat16 k1 = __float2bfloat16_rn(y.y);
    const __nv_bfloat16 v0 = __float2bfloat16_rn(vc[i]);
    const __nv_bfloat16 v1 = __float2bfloat16_rn(vc[i + half]);
    cur[i] = __bfloat16_as_ushort(k0);
    cur[i + half] = __bfloat16_as_ushort(k1);
    cur[d + i] = __bfloat16_as_ushort(v0);
    cur[d + i + half] = __bfloat16_as_ushort(v1);
    if (!aborted(c) && (!wo || (t.flags & TF_KV_APPEND))) {  // one task per head appends the row
      __nv_bfloat16* Kc = reinterpret_cast<__nv_bfloat16*>(P.kv) + kv_off(P, c.ctl, l, 0, kvh, pos);
      __nv_bfloat16* Vc = reinterpret_cast<__nv_bfloat16*>(P.kv) + kv_off(P, c.ctl, l, 1, kvh, pos);
      Kc[i] = k0;
      Kc[i + half] = k1;
      Vc[i] = v0;
      Vc[i + half] = v1;
    }
  }
  // the task's K/V rows: stage st holds positions a + st*R .. (K rows, then V rows); R is a power of
  // two and the stages are consecutive ring slots, so no division is needed; position nh (owner)
  // is the row just appended
  unsigned s_first = 0, ph_unused = 0;
  slot_after(c, 0, s_first, ph_unused);
#pragma unroll 1
  for (int st = 0; st < nst; ++st) stage_wait(c, (unsigned)st);
  if (!c.mma) {
    compute_sync();  // the rotated queries and the current row
  } else if ((nh & 15) != 0 && c.warp == ((nh - 1) >> 4) % kComputeWarps) {
    // tensor-core path (no block barrier: each warp reads only the raw queries and its own blocks):
    // V rows nh .. (end of the last 16-row block) hold whatever the tile copy read past the task's
    // rows; the warp that takes that block zeroes them, so that their zero weights cannot meet a NaN.
    // The fence orders these writes before the producer's next tile copy into the slot.
    for (int i = c.lane; i < (16 - (nh & 15)) * 8; i += 32) {
      const int row = nh + (i >> 3);
      unsigned slot = s_first + (unsigned)(row / kMmaRows);
      slot = slot >= c.ns ? slot - c.ns : slot;
      *reinterpret_cast<uint4*>(c.ring + (size_t)slot * kStageBytes + kMmaRows * 128 + (row & (kMmaRows - 1)) * 128 +
                                (i & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
  }
  trace_mark(c, 4);
  const int rshift = 31 - __clz(R);
  const unsigned ns = c.ns;
  auto krow = [&](int j) -> const uint16_t* {
    if (j >= nh) return cur;
    unsigned s = s_first + (unsigned)(j >> rshift);
    s = s >= ns ? s - ns : s;
    return reinterpret_cast<const uint16_t*>(c.ring + (size_t)s * kStageBytes) + ((size_t)(j & (R - 1)) << dshift);
  };
  auto vrow = [&](int j) -> const uint16_t* { return krow(j) + (j >= nh ? d : R * d); };

  // 2. work items: (block, head) -> per-item o (unnormalised), m, l
  const float scale = P.attn_scale * 1.4426950408889634f;
  const int nchunk = d >> 3;  // 16-byte K chunks per row
  int nparts = nblk;          // partials per query head for the merge
  if (c.mma) nparts = attn_items_mma(c, sq, QS, g, nh, owner, kc, s_first, scale, pw);
#pragma unroll 1
  for (int it = c.mma ? items : c.warp; it < items; it += kComputeWarps) {  // (CUDA-core items)
    const int blk = it / g, h = it - blk * g;
    const int j = (blk << 5) + c.lane;
    const bool valid = j < np;
    // this lane's score: the full dot product of its K row with the query, chunk order rotated
    // by lane so that the 32 rows are read without bank conflicts
    const int j0b = blk << 5;
    const int nj = min(32, np - j0b);
    float s = -INFINITY;
    if (valid) {
      const uint4* kr = reinterpret_cast<const uint4*>(krow(j));
      const float4* qh = reinterpret_cast<const float4*>(sq + h * QS);
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll 4
      for (int k = 0; k < nchunk; ++k) {
        const int cch = (k + c.lane) & (nchunk - 1);
        const uint4 kw = kr[cch];
        const int qc = 2 * cch + (cch >> 2);  // the chunk's first float4 (attn_qpos)
        const float4 q0 = qh[qc], q1 = qh[qc + 1];
        s0 = fmaf(bf16_lo(kw.x), q0.x, s0);
        s1 = fmaf(bf16_hi(kw.x), q0.y, s1);
        s2 = fmaf(bf16_lo(kw.y), q0.z, s2);
        s3 = fmaf(bf16_hi(kw.y), q0.w, s3);
        s0 = fmaf(bf16_lo(kw.z), q1.x, s0);
        s1 = fmaf(bf16_hi(kw.z), q1.y, s1);
        s2 = fmaf(bf16_lo(kw.w), q1.z, s2);
        s3 = fmaf(bf16_hi(kw.w), q1.w, s3);
      }
      s = ((s0 + s1) + (s2 + s3)) * scale;
    }
    const float m = warp_max(s);
    const float p = valid ? exp2f(s - m) : 0.f;
    const float lsum = warp_sum(p);
    // the block's output: lane owns element pairs 2*lane (+64); the 32 positions' weights go through
    // the warp's buffer and come back four at a time as broadcast loads (fewer shared-memory and
    // shuffle operations than one shuffle per position).  A block's cached rows are consecutive rows
    // of one stage (32 divides R); the appended row, if the block holds it, comes last.
    pbw[c.lane] = p;
    __syncwarp();
    const int ncache = max(0, min(nj, nh - j0b));
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f, b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f;
    if (ncache > 0) {
      const uint16_t* vb = vrow(j0b) + 2 * c.lane;
      const float4* pb4 = reinterpret_cast<const float4*>(pbw);
      int jj = 0;
#pragma unroll 2
      for (; jj + 4 <= ncache; jj += 4) {
        const float4 p4 = pb4[jj >> 2];
        const uint32_t v0 = *reinterpret_cast<const uint32_t*>(vb + jj * d);
        const uint32_t v1 = *reinterpret_cast<const uint32_t*>(vb + (jj + 1) * d);
        const uint32_t v2 = *reinterpret_cast<const uint32_t*>(vb + (jj + 2) * d);
        const uint32_t v3 = *reinterpret_cast<const uint32_t*>(vb + (jj + 3) * d);
        a0 = fmaf(p4.x, bf16_lo(v0), a0);
        a1 = fmaf(p4.x, bf16_hi(v0), a1);
        b0 = fmaf(p4.y, bf16_lo(v1), b0);
        b1 = fmaf(p4.y, bf16_hi(v1), b1);
        a0 = fmaf(p4.z, bf16_lo(v2), a0);
        a1 = fmaf(p4.z, bf16_hi(v2), a1);
        b0 = fmaf(p4.w, bf16_lo(v3), b0);
        b1 = fmaf(p4.w, bf16_hi(v3), b1);
        if (d > 64) {
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(vb + jj * d + 64);
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(vb + (jj + 1) * d + 64);
          const uint32_t w2 = *reinterpret_cast<const uint32_t*>(vb + (jj + 2) * d + 64);
          const uint32_t w3 = *reinterpret_cast<const uint32_t*>(vb + (jj + 3) * d + 64);
          a2 = fmaf(p4.x, bf16_lo(w0), a2);
          a3 = fmaf(p4.x, bf16_hi(w0), a3);
          b2 = fmaf(p4.y, bf16_lo(w1), b2);
          b3 = fmaf(p4.y, bf16_hi(w1), b3);
          a2 = fmaf(p4.z, bf16_lo(w2), a2);
          a3 = fmaf(p4.z, bf16_hi(w2), a3);
          b2 = fmaf(p4.w, bf16_lo(w3), b2);
          b3 = fmaf(p4.w, bf16_hi(w3), b3);
        }
      }
      for (; jj < ncache; ++jj) {
        const float pj = pbw[jj];
        const uint32_t v01 = *reinterpret_cast<const uint32_t*>(vb + jj * d);
        a0 = fmaf(pj, bf16_lo(v01), a0);
        a1 = fmaf(pj, bf16_hi(v01), a1);
        if (d > 64) {
          const uint32_t v23 = *reinterpret_cast<const uint32_t*>(vb + jj * d + 64);
          a2 = fmaf(pj, bf16_lo(v23), a2);
          a3 = fmaf(pj, bf16_hi(v23), a3);
        }
      }
    }
    a0 += b0;
    a1 += b1;
    a2 += b2;
    a3 += b3;
    if (nj > ncache) {  // the appended row
      const float pj = pbw[ncache];
      const uint16_t* vr = cur + d + 2 * c.lane;
      const uint32_t v01 = *reinterpret_cast<const uint32_t*>(vr);
      a0 = fmaf(pj, bf16_lo(v01), a0);
      a1 = fmaf(pj, bf16_hi(v01), a1);
      if (d > 64) {
        const uint32_t v23 = *reinterpret_cast<const uint32_t*>(vr + 64);
        a2 = fmaf(pj, bf16_lo(v23), a2);
        a3 = fmaf(pj, bf16_hi(v23), a3);
      }
    }
    float* pi = pw + it * (d + 4);
    pi[2 * c.lane] = a0;
    pi[2 * c.lane + 1] = a1;
    if (d > 64) {
      pi[64 + 2 * c.lane] = a2;
      pi[64 + 2 * c.lane + 1] = a3;
    }
    if (c.lane == 0) {
      pi[d] = m;
      pi[d + 1] = lsum;
    }
    __syncwarp();  // every lane has read the warp's weights before the next item writes them
  }
  stages_release(c, (unsigned)nst);
  compute_sync();
  trace_mark(c, 5);

  const int istride = g * (d + 4);  // items of one head are g apart
  if (wo) {
    // 3'. (fused) output rows of this KV head's columns of Wo.  The partials are merged once
    // (o = sum_p o_p 2^(m_p - M) / sum_p l_p 2^(m_p - M), M = max_p m_p), each thread of the first
    // O/4 taking four elements, into the query area (free now); after the barrier every warp reads
    // the merged o for its dot products.  (Merging in every warp instead saves the barrier but
    // multiplies the shared-memory reads by the warp count.)
    float* om = sq;
#pragma unroll 1
    for (int i = c.ctid; i < (O >> 2); i += kCT) {
      const int e0 = i << 2, h = e0 >> dshift, tt = e0 & (d - 1);
      const float* ph = pw + h * (d + 4);
      float M = -INFINITY;
#pragma unroll 4
      for (int q = 0; q < nparts; ++q) M = fmaxf(M, ph[q * istride + d]);
      float den = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int q = 0; q < nparts; ++q) {
        const float* pq = ph + q * istride;
        const float f = exp2f(pq[d] - M);
        den = fmaf(pq[d + 1], f, den);
        const float4 o4 = *reinterpret_cast<const float4*>(pq + tt);
        acc.x = fmaf(o4.x, f, acc.x);
        acc.y = fmaf(o4.y, f, acc.y);
        acc.z = fmaf(o4.z, f, acc.z);
        acc.w = fmaf(o4.w, f, acc.w);
      }
      const float inv = 1.f / den;
      *reinterpret_cast<float4*>(om + e0) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
    compute_sync();
    const int nvec = O >> 3;  // <= 64 for fused plans
    float ov[2][8];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int v = c.lane + 32 * k;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
      if (v < nvec) {
        a = *reinterpret_cast<const float4*>(om + 8 * v);
        b = *reinterpret_cast<const float4*>(om + 8 * v + 4);
      }
      ov[k][0] = a.x;
      ov[k][1] = a.y;
      ov[k][2] = a.z;
      ov[k][3] = a.w;
      ov[k][4] = b.x;
      ov[k][5] = b.y;
      ov[k][6] = b.z;
      ov[k][7] = b.w;
    }
    trace_mark(c, 6);
    const size_t row_bytes = (size_t)O * (F8 ? 1 : 2);
    unsigned long long* out = P.words + t.out_off;
    // FP8: the scales of Wo's rows (one per full row, shared by every KV head's segment)
    const float* rsc = F8 ? P.wscale + (size_t)l * P.wscale_layer + (P.nq + 2 * P.nkv) * d + t.row0 : nullptr;
    int rbase = 0;
#pragma unroll 1
    for (uint32_t k0 = 1; k0 < t.nchunks; k0 += kGemvBatch) {
      const int nb = (int)min((uint32_t)kGemvBatch, t.nchunks - k0);
      const BatchRows b = batch_wait(c, nb);
#pragma unroll 1
      for (int q = c.warp; q < b.total; q += kComputeWarps) {
        const unsigned char* row = b.row(q, row_bytes);
        float a = 0.f;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int v = c.lane + 32 * k;
          if (v < nvec) {
            if constexpr (F8) {
              const uint4 w = wload<true>(row, v);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const unsigned long long wp = wpair<true>(w, j);
                a = fmaf(__uint_as_float((uint32_t)wp), ov[k][2 * j], a);
                a = fmaf(__uint_as_float((uint32_t)(wp >> 32)), ov[k][2 * j + 1], a);
              }
            } else {
              const uint4 w = reinterpret_cast<const uint4*>(row)[v];
              a = fmaf(bf16_lo(w.x), ov[k][0], a);
              a = fmaf(bf16_hi(w.x), ov[k][1], a);
              a = fmaf(bf16_lo(w.y), ov[k][2], a);
              a = fmaf(bf16_hi(w.y), ov[k][3], a);
              a = fmaf(bf16_lo(w.z), ov[k][4], a);
              a = fmaf(bf16_hi(w.z), ov[k][5], a);
              a = fmaf(bf16_lo(w.w), ov[k][6], a);
              a = fmaf(bf16_hi(w.w), ov[k][7], a);
            }
          }
        }
        a = warp_sum(a);
        if constexpr (F8) a *= rsc[rbase + q];
        if (c.lane == 0) st_word(out + rbase + q, c.tag, a);
      }
      stages_release(c, (unsigned)nb);
      rbase += b.total;
    }
    return;
  }

  // 3. merge the blocks of each head: o = sum_b o_b 2^(m_b - M) / sum_b l_b 2^(m_b - M)
  const int hq0 = kvh * g;  // first query head of the task
  unsigned long long* out_o = layer_words(P, l) + P.act.att + ((size_t)sp * P.nq + hq0) * d;
  unsigned long long* out_ml = layer_words(P, l) + P.act.att + (size_t)P.nsplit * P.nq * d + ((size_t)sp * P.nq + hq0) * 2;
#pragma unroll 1
  for (int e = c.ctid; e < O; e += kCT) {
    const int h = e >> dshift, tt = e & (d - 1);
    const float* ph = pw + h * (d + 4);
    float M = -INFINITY;
    for (int q = 0; q < nparts; ++q) M = fmaxf(M, ph[q * istride + d]);
    float num = 0.f, den = 0.f;
#pragma unroll 4
    for (int q = 0; q < nparts; ++q) {
      const float f = exp2f(ph[q * istride + d] - M);
      num = fmaf(ph[q * istride + tt], f, num);
      den = fmaf(ph[q * istride + d + 1], f, den);
    }
    st_word(out_o + e, c.tag, num / den);
    if (tt == 0) {
      st_word(out_ml + 2 * h, c.tag, M);
      st_word(out_ml + 2 * h + 1, c.tag, den);
    }
  }
}

// The split combine when the active splits' o words do not fit one poll: combine_group splits per
// poll into `scratch` ([group][nq*d] floats), the first poll also bringing the (m, l) words of every
// active split (after the first group's o words).  The sums run on in `o` in split order, so the
// result is the one a single poll gives.  Each group costs a poll and two block barriers.  Kept out
// of line (Ctx by value): only caches longer than the shared memory's combine area take it.
__device__ __noinline__ void combine_splits_grouped(Ctx c, int l, float* o, float* scratch, int tid, int nth) {
  const KernelParams& P = *c.P;
  const int d = P.d, nqd = P.nq * d, dshift = 31 - __clz(d);
  const int nact = c.pos / P.split_len + 1;
  const int cg = P.combine_group, ng0 = min(cg, nact);
  const unsigned long long* ob = layer_words(P, l) + P.act.att;  // o words [split][head][d], then (m, l)
  const float* ml = scratch + ng0 * nqd;  // (m, l) of the active splits, [split][head][2]
#pragma unroll 1
  for (int g0 = 0; g0 < nact; g0 += cg) {
    const int ng = min(cg, nact - g0);
    if (tid >= 0) {
      InVec v;
      v.src = ob + (size_t)g0 * nqd;
      v.src2 = ob + (size_t)P.nsplit * nqd;  // (m, l) of the active splits: a prefix of [split][head][2]
      v.src3 = nullptr;
      v.n1 = ng * nqd;
      v.n2 = g0 == 0 ? nact * P.nq * 2 : 0;
      v.n = v.n1 + v.n2;
      v.emb = nullptr;
      v.gain = nullptr;
      v.dst = scratch;
      v.xlayout = 0;
      v.terms = nullptr;
      v.nterm = 0;
      v.tstride = 0;
      poll_vec(c, v, 0x310000u, tid, nth);
    }
    compute_sync();
    const bool last = g0 + ng == nact;
#pragma unroll 1
    for (int e = c.ctid; e < nqd; e += kCT) {
      const int h = e >> dshift;
      float M = -INFINITY;
      for (int s = 0; s < nact; ++s) M = fmaxf(M, ml[(s * P.nq + h) * 2]);
      float num = g0 == 0 ? 0.f : o[xpos(e, nqd)], den = 0.f;
#pragma unroll 4
      for (int s = 0; s < (last ? nact : g0 + ng); ++s) {  // den (kept by the last group) needs every split
        const float* m = ml + (s * P.nq + h) * 2;
        const float wgt = m[1] * exp2f(m[0] - M);
        if (s >= g0) num = fmaf(wgt, scratch[(s - g0) * nqd + e], num);
        den += wgt;
      }
      o[xpos(e, nqd)] = last ? num / den : num;
    }
    if (!last) compute_sync();  // the next group's words overwrite the scratch
  }
}

// Attention output of every query head into o[nq*d] (split GEMV layout) when the context has
// several splits: the active splits of each head are combined by their log-sum-exp weights
// (split-context "flash decoding", README "Current status").  One poll brings every active split's o
// words and (m, l) words into `scratch` (nsplit * (nq*d + nq*2) floats) -- threads tid of nth take
// part, up to eight words each in flight -- and, after the block barrier, each output is the
// weighted mean of the splits' normalised outputs, weights l_s 2^(m_s - max m), summed in split order.
// (combine_splits_grouped takes over when they do not fit one poll.)  The caller's other threads may
// poll other words meanwhile; every compute thread reaches the barrier.
__device__ __forceinline__ void combine_splits(Ctx& c, int l, float* o, float* scratch, int tid, int nth) {
  const KernelParams& P = *c.P;
  const int d = P.d, nqd = P.nq * d, dshift = 31 - __clz(d);
  const int nact = c.pos / P.split_len + 1;
  if (nact > P.combine_group) {
    combine_splits_grouped(c, l, o, scratch, tid, nth);
    return;
  }
  const unsigned long long* ob = layer_words(P, l) + P.act.att;  // o words [split][head][d], then (m, l)
  const int no = nact * nqd;              // o words of the active splits (a prefix of [split][head][d])
  if (tid >= 0) {
    InVec v;
    v.src = ob;
    v.src2 = ob + (size_t)P.nsplit * nqd;  // (m, l) of the active splits: a prefix of [split][head][2]
    v.src3 = nullptr;
    v.n1 = no;
    v.n2 = nact * P.nq * 2;
    v.n = v.n1 + v.n2;
    v.emb = nullptr;
    v.gain = nullptr;
    v.dst = scratch;
    v.xlayout = 0;
    v.terms = nullptr;
    v.nterm = 0;
    v.tstride = 0;
    poll_vec(c, v, 0x310000u, tid, nth);
  }
  compute_sync();
  const float* ml = scratch + no;
#pragma unroll 1
  for (int e = c.ctid; e < nqd; e += kCT) {
    const int h = e >> dshift;
    float M = -INFINITY;
    for (int s = 0; s < nact; ++s) M = fmaxf(M, ml[(s * P.nq + h) * 2]);
    float num = 0.f, den = 0.f;
#pragma unroll 4
    for (int s = 0; s < nact; ++s) {
      const float* m = ml + (s * P.nq + h) * 2;
      const float wgt = m[1] * exp2f(m[0] - M);
      num = fmaf(wgt, scratch[s * nqd + e], num);
      den += wgt;
    }
    o[xpos(e, nqd)] = num / den;
  }
}

// One output row of a projection, written by lane 0 of the warp that computed it (or by the
// thread that summed its slices): QKV adds the q/k/v bias and O/down add the residual (both staged
// in `add`), gate/up writes silu(gate) * up, the LM head writes a logit.  Words are written even
// after a failed wait (the step is reported failed; consumers then finish instead of waiting).
__device__ __forceinline__ void emit_row(Ctx& c, int type, unsigned long long* out, int r, float a, float u,
                                         const float* add, float* logits) {
  if (type == T_LMHEAD) {
    if (!aborted(c)) logits[r] = a;
    return;
  }
  const float v = type == T_GATEUP ? a / (1.0f + __expf(-a)) * u : add[r] + a;
  st_word(out + r, c.tag, v);
}

// Greedy decoding, end of step `step` (every compute thread, after the block barrier that ends the
// step's last task).  The largest logit of the CTA's LM-head tasks (the lowest row among equal
// values) joins the step's argmax by one 64-bit atomic max of its key (ordered value bits, then
// ~row: keys of different values order like the values), and the tasks are counted.  The CTA whose
// count completes the step reads the argmax, reports it and publishes it as a tagged word with the
// next step's tag; every CTA polls that word like any other input at the start of the next step.
// Nothing here waits.
__device__ __noinline__ void greedy_boundary(const KernelParams* P, const StepParams* S, Ctl* ctl, int step,
                                            uint32_t t0, uint32_t t1) {
  const int ctid = (int)threadIdx.x - 32, lane = (int)threadIdx.x & 31;
  const float* logits = S->logits + (size_t)step * S->logits_step;
  unsigned long long key = 0ull;
  unsigned ntask = 0;
  for (uint32_t ti = t1; ti > t0; --ti) {  // the LM-head tasks close the CTA's list
    const Task* t = P->tasks + (ti - 1);
    if (t->type != T_LMHEAD) break;
    ++ntask;
    const unsigned row0 = t->row0, nrows = t->nrows;
    for (unsigned i = (unsigned)ctid; i < nrows; i += kCT) {
      const unsigned u = __float_as_uint(logits[row0 + i]);
      const unsigned ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
      const unsigned long long k = ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (row0 + i));
      key = k > key ? k : key;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long k2 = __shfl_xor_sync(0xffffffffu, key, o);
    key = k2 > key ? k2 : key;
  }
  if (lane == 0) ctl->amax[ctid >> 5] = key;
  compute_sync();
  if (ctid == 0 && ntask > 0) {
    unsigned long long best = 0ull;
    for (int w = 0; w < kComputeWarps; ++w) best = ctl->amax[w] > best ? ctl->amax[w] : best;
    atomicMax(S->amax + step, best);
    __threadfence();
    const unsigned before = atomicAdd(S->amax_done + step, ntask);
    if (before + ntask == (unsigned)P->lm_tasks) {  // the last contribution of the step
      __threadfence();
      const unsigned long long k = atomicOr(S->amax + step, 0ull);
      const unsigned idx = 0xFFFFFFFFu - (unsigned)(k & 0xFFFFFFFFull);
      const int tok = k != 0ull && idx < (unsigned)P->V ? (int)idx : 0;
      S->out_tokens[step] = tok;
      st_word(S->tokword, S->tag + (unsigned)step + 1u, __int_as_float(tok));
    }
  }
}

// A projection task (QKV, O, gate/up, down, LM head): one code path for every type.  The critical
// path after the inputs arrive is one block barrier, the row's dot products and the output store:
// weight stages are checked before the inputs are polled, and the norm scale (a reduction of the
// per-warp sums of squares) is computed by every warp alongside its dot products.
template <bool F8>
__device__ __forceinline__ void task_gemv(Ctx& c, const Task& t, float* sv, float* res, float* add) {
  const KernelParams& P = *c.P;
  const int l = t.layer, type = t.type, n = (int)t.nrows;
  // 1. what the task reads and writes (word offsets and flags set by the scheduler)
  const unsigned f = t.flags;
  const uint16_t* emb_row = P.embed + (size_t)c.token * P.H;
  const unsigned long long* layer_in = P.inject != nullptr ? P.inject + (size_t)l * P.H : nullptr;
  InVec x, r;
  x.src = (f & TF_IN_EMB) ? nullptr : ((f & TF_IN_LAYER) && layer_in ? layer_in : P.words + t.in_off);
  x.emb = emb_row;
  x.gain = (f & TF_NORM) ? c.ctl->gain[t.gain] : nullptr;
  x.dst = sv;
  x.n = (int)t.in_n;
  x.xlayout = 1;
  x.src2 = x.src3 = nullptr;
  x.n1 = x.n;
  x.n2 = 0;
  x.terms = P.words + t.aux;
  x.nterm = (f & TF_IN_SUM) ? P.nkv : 0;
  x.tstride = P.H;
  r.src = (f & TF_RES_EMB) ? nullptr : ((f & TF_RES_LAYER) && layer_in ? layer_in + t.row0 : P.words + t.res_off);
  r.emb = emb_row + t.row0;
  r.gain = nullptr;
  r.dst = add;
  r.n = (f & TF_RES) ? n : 0;
  r.xlayout = 0;
  r.src2 = r.src3 = nullptr;
  r.n1 = r.n;
  r.n2 = 0;
  r.terms = P.words + t.aux;
  r.nterm = (f & TF_RES_SUM) ? P.nkv : 0;
  r.tstride = P.H;
  unsigned long long* out = P.words + t.out_off;
  const int in = (int)t.in_n;
  const bool combine = (f & TF_COMBINE) != 0;  // O projection over several context splits
  // the q/k/v bias of the task's rows: loads issued before the inputs are polled
  uint32_t braw[kVecPerThread];
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) braw[k] = 0u;
  if (f & TF_BIAS) {
    const int qd = P.nq * P.d, kvd = P.nkv * P.d;
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
      const int i = c.ctid + k * kCT;
      if (i < n) {
        const int o = (int)t.row0 + i;
        const uint16_t* b = o < qd ? c.ctl->bias[3 * l] + o
                                   : (o < qd + kvd ? c.ctl->bias[3 * l + 1] + (o - qd) : c.ctl->bias[3 * l + 2] + (o - qd - kvd));
        braw[k] = *b;
      }
    }
  }
  // a single-batch task's weights (almost always in shared memory by now) are checked first
  const bool direct = t.gpr == 0;
  const bool one_batch = direct && t.nchunks <= (uint32_t)kGemvBatch;
  BatchRows b0;
  if (one_batch) b0 = batch_wait(c, (int)t.nchunks);
  // 2. inputs: the vector, then (O, down) the residual rows -- one polling loop for both
  float ss = 0.f;
  if (combine) {
    // the splits' words and (O projection) the residual rows in one pass: the last warp polls the
    // residual rows while the others poll the splits
    const int nsp = r.n > 0 ? kCT - 32 : kCT;
    if (c.ctid >= nsp) {
      if (r.nterm > 0) poll_sum(c, r, 0x400000u, c.ctid - nsp, 32);
      else poll_vec(c, r, 0x400000u, c.ctid - nsp, 32);
    }
    combine_splits(c, l, sv, sv + P.nq * P.d, c.ctid < nsp ? c.ctid : -1, nsp);
  } else {
    // one pass for both vectors: with residual rows (O, down) the last warp polls them while the
    // other warps poll the input vector, so neither waits behind the other's round trips
    const int nx = r.n > 0 ? kCT - 32 : kCT;
    if (c.ctid < nx) {
      ss = x.nterm > 0 ? poll_sum(c, x, 0x100000u, c.ctid, nx) : poll_vec(c, x, 0x100000u, c.ctid, nx);
    } else if (r.nterm > 0) {
      poll_sum(c, r, 0x400000u, c.ctid - nx, 32);
    } else {
      poll_vec(c, r, 0x400000u, c.ctid - nx, 32);
    }
  }
  if (type == T_QKV) {
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
      const int i = c.ctid + k * kCT;
      if (i < n) add[i] = __uint_as_float(braw[k] << 16);
    }
  }
  const bool norm = (f & TF_NORM) != 0;
  if (norm) {
    ss = warp_sum(ss);
    if (c.lane == 0) c.ctl->red[c.warp] = ss;
  }
  compute_sync();
  trace_mark(c, 1);
  // the norm scale (every warp sums the per-warp partials with broadcast reads, fixed order); taken
  // after the warp's first dot product so its latency overlaps the GEMV.  1/sqrt(mean + eps) is the
  // hardware estimate refined by one Newton step, y' = y (3 - a y^2) / 2, to within about an ulp.
  auto norm_scale = [&]() -> float {
    if (!norm) return 1.f;
    const float4* r4 = reinterpret_cast<const float4*>(c.ctl->red);
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < (kComputeWarps + 3) / 4; ++w) {
      const float4 v = r4[w];
      tot += (v.x + v.y) + (v.z + (4 * w + 3 < kComputeWarps ? v.w : 0.f));
    }
    const float arg = fmaf(tot, P.inv_H, P.eps);
    const float y = rsqrtf(arg);
    return y * fmaf(-0.5f * arg * y, y, 1.5f);
  };
  float scale = 0.f;
  // 3. the projection and its outputs
  float* logits = c.logits + t.row0;
  const bool pairs = (f & TF_PAIRS) != 0;
  // FP8: the per-row weight scales of the task's rows (gate/up: gate rows, then up rows I further on)
  const float* rsc = nullptr;
  if constexpr (F8) {
    const int qkv = (P.nq + 2 * P.nkv) * P.d;
    const size_t base = type == T_LMHEAD ? (size_t)P.L * P.wscale_layer
                                         : (size_t)l * P.wscale_layer + (type == T_QKV ? 0
                                                                         : type == T_OPROJ ? qkv
                                                                         : type == T_GATEUP ? qkv + P.H
                                                                                            : qkv + P.H + 2 * P.I);
    rsc = P.wscale + base + t.row0;
  }
  if (direct) {
    // one warp per row (gate/up: per row pair); lane 0 writes the output as soon as its row is done
    const int nvec = in >> 3;
    const float4* xlo = reinterpret_cast<const float4*>(sv);
    const float4* xhi = reinterpret_cast<const float4*>(sv + (in >> 1));
    const size_t row_bytes = (size_t)in * (F8 ? 1 : 2);
    int rbase = 0;
#pragma unroll 1
    for (uint32_t k0 = 0; k0 < t.nchunks; k0 += kGemvBatch) {
      const int nb = (int)min((uint32_t)kGemvBatch, t.nchunks - k0);
      const BatchRows b = one_batch ? b0 : batch_wait(c, nb);
      const int rows = pairs ? n : b.total;  // gate/up: one batch holds gate rows, then up rows
#pragma unroll 1
      for (int q = c.warp; q < rows; q += kComputeWarps) {
        float a, u = 0.f;
        if (pairs) {
          dot_row2<F8>(c, b.row(q, row_bytes), b.row(n + q, row_bytes), xlo, xhi, nvec, a, u);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, o);
            u += __shfl_xor_sync(0xffffffffu, u, o);
          }
        } else {
          a = warp_sum(dot_row<F8>(c, b.row(q, row_bytes), xlo, xhi, nvec));
        }
        if (scale == 0.f) scale = norm_scale();
        if constexpr (F8) {
          a *= rsc[rbase + q];
          if (pairs) u *= rsc[P.I + q];
        }
        if (c.lane == 0) emit_row(c, type, out, rbase + q, a * scale, u * scale, add, logits);
      }
      stages_release(c, (unsigned)nb);
      rbase += b.total;
    }
  } else {
    // warps share rows: partial sums in res, summed in a fixed order after the barrier
    gemv_xreg<F8>(c, t, in, sv, res, norm_scale());
    const int gpr = (int)t.gpr;
#pragma unroll 1
    for (int i = c.ctid; i < n; i += kCT) {
      float a = res_row(res, i, gpr), u = pairs ? res_row(res, n + i, gpr) : 0.f;
      if constexpr (F8) {
        a *= rsc[i];
        if (pairs) u *= rsc[P.I + i];
      }
      emit_row(c, type, out, i, a, u, add, logits);
    }
  }
}

// ------------------------------------------------------------------ producer warp
// Walks the CTA's chunk list (32 descriptors per coalesced load, the next batch loaded while the
// current one is issued) and fills the ring.  Lane 0 issues; the other lanes only help load.
// Producer of a multi-step launch, before the first K/V copy of step `step` >= 1: waits until every CTA
// has finished the previous step (so the cache rows it appended are visible), then orders those
// generic-proxy writes before this warp's bulk copies.  Bounded; false if the wait gave up.
__device__ __noinline__ bool wait_prev_step(const unsigned long long* sync, unsigned long long target, int step,
                                            const KernelParams* P, Ctl* ctl) {
  const unsigned long long t0 = global_ns();
  for (;;) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(sync) : "memory");
    if (v >= target) break;
    if (*(volatile unsigned*)P->status != 0u || global_ns() - t0 > 4 * P->timeout_ns) {
      if (atomicCAS(&P->status[0], 0u, (unsigned)DS_TIMEOUT) == 0u) {
        P->status[1] = blockIdx.x;
        P->status[3] = 0xD000u | (unsigned)step;
      }
      *(volatile unsigned*)&ctl->prod_quit = 1u;
      return false;
    }
    __nanosleep(64);
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

__device__ __forceinline__ void produce(const KernelParams& P, const StepParams& S, Ctl* ctl, unsigned char* ring,
                                        uint32_t c0, uint32_t c1, int lane, const CUtensorMap* kvmap, bool mma) {
  const uint64_t policy = evict_first_policy();
  const unsigned ns = (unsigned)P.num_stages;
  unsigned stage = 0, uses = 0;  // ring slot and how many times the ring has wrapped
  bool quit = false;
  // lane 0: wait for a free stage, record its rows, arm its barrier; returns null if consumers stall
  auto acquire = [&](unsigned bytes, uint32_t rows) -> unsigned char* {
    if (uses > 0) {
      const unsigned ph = (uses - 1) & 1u;
      if (!mbar_test(&ctl->empty[stage], ph)) {
        const unsigned long long tstart = global_ns();
        while (!mbar_test(&ctl->empty[stage], ph)) {
          // The ring is full and the stream is far ahead of the consumers: sleep between tests so
          // that this warp leaves its sub-partition's issue slots to the compute warps.
          __nanosleep(128);
          // Consumers keep taking stages even after a failed activation wait (they stop waiting
          // for activations instead), so this only expires if a consumer is wedged: stop streaming.
          if (global_ns() - tstart > 4 * P.timeout_ns) {
            if (atomicCAS(&P.status[0], 0u, (unsigned)DS_TIMEOUT) == 0u) {
              P.status[1] = blockIdx.x;
              P.status[3] = 0xE000u | stage;
            }
            *(volatile unsigned*)&ctl->prod_quit = 1u;
            return nullptr;
          }
        }
      }
    }
    ctl->stage_rows[stage] = rows;
    mbar_expect_tx(&ctl->full[stage], bytes);
    return ring + (size_t)stage * kStageBytes;
  };
  auto advance = [&]() {
    if (++stage == ns) {
      stage = 0;
      ++uses;
    }
  };
  for (int step = 0; step < S.n && !quit; ++step) {
  const int pos = S.pos + step;
  bool synced = step == 0;  // the cache rows of earlier steps are visible to this step's copies
  Chunk next{};
  if (c0 + lane < c1) next = P.chunks[c0 + lane];
  for (uint32_t base = c0; base < c1 && !quit; base += 32) {
    const Chunk mine = next;
    if (base + 32 + lane < c1) next = P.chunks[base + 32 + lane];
    const int cnt = (int)min(32u, c1 - base);
    for (int j = 0; j < cnt && !quit; ++j) {
      const uint64_t src = ((uint64_t)__shfl_sync(0xffffffffu, (unsigned)(mine.src >> 32), j) << 32) |
                           (uint64_t)__shfl_sync(0xffffffffu, (unsigned)mine.src, j);
      const unsigned bytes = __shfl_sync(0xffffffffu, mine.bytes, j);
      const unsigned rows = __shfl_sync(0xffffffffu, mine.rows, j);
      int q = 0;
      if (lane == 0) {
        if (rows == kAttnChunk && !synced) {
          synced = true;
          if (!wait_prev_step(S.sync, S.sync_base + (unsigned long long)step * gridDim.x, step, &P, ctl)) q = 1;
        }
        if (q) {
        } else if (rows == kAttnChunk) {
          const int layer = (int)(src >> 48), kvh = (int)((src >> 32) & 0xFFFF), sp = (int)(unsigned)src;
          const int a = sp * P.split_len;
          if (a <= pos) {
            const int b = min(a + P.split_len, pos);
            for (int jj = a; jj < b; jj += P.rows_per_stage) {
              const int n = min(P.rows_per_stage, b - jj);
              if (mma) {
                // tensor-core path: K then V as swizzled tiles of box rows (a whole stage, or one
                // page's share of it); rows past b come along and are masked by the consumers
                const int br = P.attn_box_rows, nbox = (n + br - 1) / br;
                unsigned char* dst = acquire((unsigned)(2 * nbox * br * 128), (unsigned)n);
                if (!dst) {
                  q = 1;
                  break;
                }
                for (int bx = 0; bx < nbox; ++bx) {
                  const int p = jj + bx * br;
                  const int yk = (int)(kv_off(P, ctl, layer, 0, kvh, p) >> 6), yv = (int)(kv_off(P, ctl, layer, 1, kvh, p) >> 6);
                  tile_load(dst + bx * br * 128, kvmap, 0, yk, &ctl->full[stage], policy);
                  tile_load(dst + kMmaRows * 128 + bx * br * 128, kvmap, 0, yv, &ctl->full[stage], policy);
                }
                advance();
                continue;
              }
              const unsigned nb = (unsigned)(n * P.d * 2);
              unsigned char* dst = acquire(2 * nb, (unsigned)n);
              if (!dst) {
                q = 1;
                break;
              }
              // K rows then V rows; a paged cache gives one copy pair per run of rows inside a page
              for (int r0 = 0; r0 < n;) {
                const int p = jj + r0;
                const int run = P.page_table != nullptr ? min(n - r0, P.page_size - (p & (P.page_size - 1))) : n - r0;
                const unsigned rb = (unsigned)(run * P.d * 2);
                unsigned char* dk = dst + (size_t)r0 * P.d * 2;
                bulk_load(dk, P.kv + kv_off(P, ctl, layer, 0, kvh, p), rb, &ctl->full[stage], policy);
                bulk_load(dk + (size_t)P.rows_per_stage * P.d * 2, P.kv + kv_off(P, ctl, layer, 1, kvh, p), rb,
                          &ctl->full[stage], policy);
                r0 += run;
              }
              advance();
            }
          }
        } else if (rows & kStridedRows) {
          // one KV head's columns of Wo: a segment per output row, packed back to back
          const unsigned n = rows & ~kStridedRows, seg = bytes / n;
          const size_t stride = (size_t)P.nq * P.d * P.wbytes;
          unsigned char* dst = acquire(bytes, n);
          if (!dst) {
            q = 1;
          } else {
            for (unsigned r = 0; r < n; ++r)
              bulk_load(dst + (size_t)r * seg, reinterpret_cast<const unsigned char*>(src) + r * stride, seg,
                        &ctl->full[stage], policy);
            advance();
          }
        } else {
          unsigned char* dst = acquire(bytes, rows);
          if (!dst) {
            q = 1;
          } else {
            bulk_load(dst, reinterpret_cast<const void*>(src), bytes, &ctl->full[stage], policy);
            advance();
          }
        }
      }
      quit = __shfl_sync(0xffffffffu, q, 0) != 0;
    }
  }
  }
}

// ------------------------------------------------------------------ the kernel
// Copies n task records to shared memory (threads `tid` of `nt`).
__device__ __forceinline__ void stage_tasks(const Task* src, Task* dst, int n, int tid, int nt) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  const int n16 = n * (int)(sizeof(Task) / 16);
  for (int i = tid; i < n16; i += nt) d4[i] = s4[i];
}

// kGreedy: greedy decoding (the argmax of each step's logits is the next step's token).  A separate
// instantiation, so that the teacher-forced kernel carries none of its state in registers.
// kMma: attention on the tensor cores (K/V stages as swizzled tiles) or on the CUDA cores; separate
// instantiations, so that each carries only the attention path it runs -- code that is never executed
// still costs instruction-cache capacity in a kernel that walks its whole body every layer.
template <bool kGreedy, bool kF8, bool kMma>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ KernelParams P, const __grid_constant__ StepParams S,
                                                             const __grid_constant__ CUtensorMap kvmap) {
  extern __shared__ __align__(128) unsigned char smem[];
  Ctl* ctl = reinterpret_cast<Ctl*>(smem);
  if (threadIdx.x == 0) {
    ctl->skip = *(volatile unsigned*)P.status;  // sticky error from an earlier step: do nothing
    // the swizzled tiles need 1024-byte aligned ring stages: the host aligns the ring's offset and
    // dynamic shared memory starts on a 1 KB boundary; should it not, the step fails (status) rather
    // than read misplaced rows
    if (kMma && ctl->skip == 0u && (smem_addr(smem + P.off_ring) & 1023u) != 0u) {
      record_failure(P.status, P.host_status, &ctl->abort, 0u, 0xA1160000u);
      ctl->skip = 1u;
    }
    ctl->abort = 0;
    ctl->prod_quit = 0;
    for (int s = 0; s < P.num_stages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], kComputeWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // token-independent tables: this step's RoPE row, the norm-gain and bias pointers
  for (int i = threadIdx.x; i < P.d / 2; i += blockDim.x) ctl->rope[i] = P.rope[(size_t)S.pos * (P.d / 2) + i];
  for (int i = threadIdx.x; i < P.L; i += blockDim.x) {
    ctl->gain[2 * i] = P.layers[i].w[LW_ATTN_NORM];
    ctl->gain[2 * i + 1] = P.layers[i].w[LW_MLP_NORM];
    ctl->bias[3 * i] = P.layers[i].w[LW_BQ];
    ctl->bias[3 * i + 1] = P.layers[i].w[LW_BK];
    ctl->bias[3 * i + 2] = P.layers[i].w[LW_BV];
  }
  if (threadIdx.x == 0) ctl->gain[2 * P.L] = P.final_norm;
  if (P.page_table != nullptr)  // the page table (at most kMaxPages entries: checked by the host)
    for (int i = threadIdx.x; i < (P.C + P.page_size - 1) / P.page_size; i += blockDim.x) ctl->pages[i] = P.page_table[i];
  // this CTA's task records, staged in shared memory kTaskWindow at a time (one window covers a
  // CTA's whole step for the usual shapes)
  const uint32_t t0 = P.task_off[blockIdx.x], t1 = P.task_off[blockIdx.x + 1];
  Task* tasks = reinterpret_cast<Task*>(smem + P.off_tasks);
  stage_tasks(P.tasks + t0, tasks, (int)min(t1 - t0, (uint32_t)kTaskWindow), threadIdx.x, blockDim.x);
  {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&P);
    uint32_t* dst = reinterpret_cast<uint32_t*>(&ctl->params);
    for (int i = threadIdx.x; i < (int)(sizeof(KernelParams) / 4); i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  if (ctl->skip) return;
  unsigned char* ring = smem + P.off_ring;
  constexpr bool mma = kMma;
  const int warp = threadIdx.x / 32;
  if (warp == 0) {
    produce(ctl->params, S, ctl, ring, P.chunk_off[blockIdx.x], P.chunk_off[blockIdx.x + 1], threadIdx.x & 31, &kvmap, mma);
    return;
  }
  Ctx c;
  c.P = &ctl->params;
  c.ctl = ctl;
  c.ring = ring;
  c.mma = mma;

  c.ns = (unsigned)P.num_stages;
  c.stage = 0;
  c.phase = 0;
  c.ctid = threadIdx.x - 32;
  c.warp = warp - 1;
  c.lane = threadIdx.x & 31;
  float* sv = reinterpret_cast<float*>(smem + P.off_sv);
  float* res = reinterpret_cast<float*>(smem + P.off_res);
  float* add = reinterpret_cast<float*>(smem + P.off_resid);
  constexpr bool greedy = kGreedy;
  c.task_index = t0;
#pragma unroll 1
  for (int step = 0; step < S.n; ++step) {
  c.tag = S.tag + (unsigned)step;
  c.pos = S.pos + step;
  c.token = (S.tokens != nullptr && !greedy) ? S.tokens[step] : S.token;
  c.logits = S.logits + (size_t)step * S.logits_step;
  if (step > 0) {
    // every compute warp is past the previous step's last task: this step's RoPE row, and the first
    // window of task records again if the CTA has more than one; greedy: the previous step's argmax
    for (int i = c.ctid; i < P.d / 2; i += kCT) ctl->rope[i] = P.rope[(size_t)c.pos * (P.d / 2) + i];
    if (t1 - t0 > (uint32_t)kTaskWindow) stage_tasks(P.tasks + t0, tasks, kTaskWindow, c.ctid, kCT);
    if constexpr (greedy) {
      // the previous step's argmax: this CTA's part (the call sits here rather than at the end of
      // the step's loop, where it made the compiler spill registers of the task loop), then the
      // token itself, published with this step's tag
      greedy_boundary(c.P, &S, ctl, step - 1, t0, t1);
      InVec v{};
      v.src = S.tokword;
      v.n = v.n1 = 1;
      v.dst = reinterpret_cast<float*>(&ctl->gtoken);
      poll_vec(c, v, 0xA00000u);
    }
    compute_sync();
    if constexpr (greedy) c.token = ctl->gtoken;
  }
#pragma unroll 1
  for (uint32_t ti = t0; ti < t1; ++ti) {
    const uint32_t k = ti - t0;
    if (k != 0 && k % kTaskWindow == 0) {  // the next window (every thread is past the last task)
      stage_tasks(P.tasks + ti, tasks, (int)min(t1 - ti, (uint32_t)kTaskWindow), c.ctid, kCT);
      compute_sync();
    }
    const Task t = tasks[k % kTaskWindow];
    c.task_index = ti;
    c.first_stage = true;
    if (P.trace != nullptr && c.ctid == 0)
      for (int k = 3; k < kTraceStamps; ++k) P.trace[(size_t)ti * kTraceStamps + k] = 0;
    trace_mark(c, 0);
    if (t.type == T_ATTN)
      task_attn<kF8>(c, t, sv, res);
    else
      task_gemv<kF8>(c, t, sv, res, add);
    compute_sync();  // the next task reuses the shared vectors
    trace_mark(c, 2);
    // tracing: the SM clock count at the end of a projection task (slot 7; attention tasks use it
    // for a phase mark), so a trace also gives the clock the tasks ran at
    if (P.trace != nullptr && c.ctid == 0 && t.type != T_ATTN) P.trace[(size_t)ti * kTraceStamps + 7] = clock64();
  }
  // this CTA is done with the step: publish it (with the cache rows its tasks appended) to the
  // producers that copy those rows in the next step
  if (S.sync != nullptr && c.ctid == 0) {
    __threadfence();
    atomicAdd(S.sync, 1ull);
  }
  }
  if constexpr (greedy) greedy_boundary(c.P, &S, ctl, S.n - 1, t0, t1);  // the last step's argmax

}

// ------------------------------------------------------------------ RoPE table and cache fill
// cos/sin of pos * theta^(-2i/d) for every cache position, computed in double precision.
__global__ void rope_table_kernel(float2* out, int C, int d, double theta) {
  const int half = d / 2;
  const size_t n = (size_t)C * half;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n; e += (size_t)gridDim.x * blockDim.x) {
    const int p = (int)(e / half), i = (int)(e % half);
    const double inv_freq = pow(theta, -(2.0 * i) / (double)d);
    double s, co;
    sincos((double)p * inv_freq, &s, &co);
    out[e] = make_float2((float)co, (float)s);
  }
}

// Rows [p0, p0+n) of one layer from pre-RoPE K and V: K rotated like a decode step, both -> bf16.
__global__ void kv_fill_kernel(uint16_t* kv, int layer, const float* k_raw, const float* v_raw, const float2* rope, int nkv,
                               int d, int p0, int n, const int32_t* table, int page_size, int page_shift,
                               unsigned long long page_elems) {
  const int half = d / 2;
  const size_t total = (size_t)nkv * n * half;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int i = (int)(e % half);
    const size_t hj = e / half;
    const int j = (int)(hj % n), h = (int)(hj / n);
    const int p = p0 + j;
    const float* kr = k_raw + ((size_t)h * n + j) * d;
    const float* vr = v_raw + ((size_t)h * n + j) * d;
    const float2 r = rope[(size_t)p * half + i];
    const float x0 = kr[i], x1 = kr[i + half];
    const size_t page = table != nullptr ? (size_t)(unsigned)table[p >> page_shift] : 0;
    const int row = table != nullptr ? (p & (page_size - 1)) : p;
    const size_t kbase = page * page_elems + ((((size_t)layer * 2) * nkv + h) * page_size + row) * d;
    __nv_bfloat16* K = reinterpret_cast<__nv_bfloat16*>(kv) + kbase;
    __nv_bfloat16* V = reinterpret_cast<__nv_bfloat16*>(kv) + kbase + (size_t)nkv * page_size * d;
    K[i] = __float2bfloat16_rn(x0 * r.x - x1 * r.y);
    K[i + half] = __float2bfloat16_rn(x1 * r.x + x0 * r.y);
    V[i] = __float2bfloat16_rn(vr[i]);
    V[i + half] = __float2bfloat16_rn(vr[i + half]);
  }
}

}  // namespace mbk

// Launch helpers used by the C ABI (mbk_api.cu).
namespace mbk {
const void* decode_kernel_ptr(bool greedy, bool fp8, bool mma) {
  if (mma) {
    if (fp8)
      return greedy ? reinterpret_cast<const void*>(&decode_kernel<true, true, true>)
                    : reinterpret_cast<const void*>(&decode_kernel<false, true, true>);
    return greedy ? reinterpret_cast<const void*>(&decode_kernel<true, false, true>)
                  : reinterpret_cast<const void*>(&decode_kernel<false, false, true>);
  }
  if (fp8)
    return greedy ? reinterpret_cast<const void*>(&decode_kernel<true, true, false>)
                  : reinterpret_cast<const void*>(&decode_kernel<false, true, false>);
  return greedy ? reinterpret_cast<const void*>(&decode_kernel<true, false, false>)
                : reinterpret_cast<const void*>(&decode_kernel<false, false, false>);
}

// FP8 copies of a bf16 matrix [rows][cols] (cols even): per row the scale amax / 448 (1 for an
// all-zero row) and the E4M3 codes of w / scale (nearest, ties to even, saturating at 448).  One
// block per row at a time.
__global__ void quantize_fp8_kernel(const uint16_t* w, int rows, int cols, uint8_t* q, float* s) {
  __shared__ float red[32];
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint16_t* wr = w + (size_t)r * cols;
    float amax = 0.f;
    for (int k = threadIdx.x; k < cols; k += blockDim.x) amax = fmaxf(amax, fabsf(bf16_to_f32(wr[k])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
    const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    if (threadIdx.x == 0) s[r] = sc;
    for (int k = 2 * threadIdx.x; k < cols; k += 2 * blockDim.x) {
      const float lo = __fdiv_rn(bf16_to_f32(wr[k]), sc), hi = __fdiv_rn(bf16_to_f32(wr[k + 1]), sc);
      unsigned short two;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(two) : "f"(hi), "f"(lo));  // lo -> the low byte
      *reinterpret_cast<unsigned short*>(q + (size_t)r * cols + k) = two;
    }
    __syncthreads();  // red[] is reused by the next row
  }
}
cudaError_t launch_quantize_fp8(const uint16_t* w, int rows, int cols, uint8_t* q, float* s, cudaStream_t st) {
  quantize_fp8_kernel<<<rows < 2048 ? rows : 2048, 256, 0, st>>>(w, rows, cols, q, s);
  return cudaGetLastError();
}
cudaError_t launch_rope_table(float2* out, int C, int d, double theta, cudaStream_t st) {
  rope_table_kernel<<<264, 256, 0, st>>>(out, C, d, theta);
  return cudaGetLastError();
}
cudaError_t launch_kv_fill(const KernelParams& kp, int layer, const float* k_raw, const float* v_raw, int p0, int n,
                           cudaStream_t st) {
  kv_fill_kernel<<<264, 256, 0, st>>>(kp.kv, layer, k_raw, v_raw, kp.rope, kp.nkv, kp.d, p0, n, kp.page_table, kp.page_size,
                                      kp.page_shift, kp.page_elems);
  return cudaGetLastError();
}
}  // namespace mbk

