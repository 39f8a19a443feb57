// mbk_kernel.cu -- the persistent batch-1 decode kernel for sm_103a (GB300).
//
// One cooperative launch per decode step, one CTA per SM (MegaBake article, "What a megakernel is,
// and why small models want one": resident CTAs working through a task list and synchronising
// through global memory).  Every CTA runs 17 warps:
//   warp 0      streams the weights of its upcoming tasks into a ring of shared-memory stages with
//               TMA bulk copies (cp.async.bulk + mbarrier transaction counts).  Weights do not depend
//               on the token, so the stream runs ahead of the data dependencies by up to the ring's
//               depth -- the "cross-phase prefetch of the next GEMM's weights while a CTA waits" the
//               article lists as future work ("Checking the 5.5x").
//   warps 1-16  execute the CTA's tasks in order.  Activations move between CTAs as 64-bit words
//               {tag:32 | fp32 value:32}, each written once per step by exactly one thread; a reader
//               spins on the word until its tag equals this step's tag.  A value and its readiness
//               travel in one single-copy-atomic store, so no fence, counter or grid barrier is
//               needed (the pages' counting grid barrier is the thing this replaces).
// Everything a task needs that does not depend on the token (norm gains, biases, RoPE cos/sin,
// descriptors) is loaded before the task waits for its inputs -- gains one task ahead -- so the
// critical path of a task is: inputs arrive -> one block barrier -> GEMV on shared-memory weights
// -> words out.  All task code is inlined into the kernel so its context stays in registers; only
// the rare slow paths (a word that is not ready yet, a failure) are out of line.
// Every spin is bounded by a globaltimer budget; on expiry the CTA records timeout status and
// finishes its task list without waiting or writing, so the launch always terminates.
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
  unsigned pad;
  float red[32];        // block reduction scratch
  float2 rope[64];      // cos/sin of this step's position, i < head_dim / 2
  const uint16_t* gain[2 * kMaxLayers + 1];  // attn_norm[l] at 2l, mlp_norm[l] at 2l+1, final at 2L
  const uint16_t* bias[3 * kMaxLayers];      // bq, bk, bv of layer l at 3l..3l+2
  KernelParams params;  // the launch parameters, copied here: reads through a pointer into the
                        // parameter window are slow, shared-memory reads are not
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

// Keeps polling a word that was not ready at the first load; returns its value (0 on abort).
__device__ __noinline__ float spin_word(const unsigned long long* p, unsigned tag, unsigned* abort_flag, unsigned* status,
                                        unsigned* host_status, unsigned long long timeout, unsigned task,
                                        unsigned detail, unsigned backoff_ns) {
  if (*(volatile unsigned*)abort_flag) return 0.f;
  const unsigned long long t0 = global_ns();
  for (unsigned n = 1;; ++n) {
    if (backoff_ns) __nanosleep(backoff_ns);
    const unsigned long long w = ld_word(p);
    if ((unsigned)(w >> 32) == tag) return __uint_as_float((unsigned)w);
    if ((n & 63u) == 0u) {
      if (*(volatile unsigned*)abort_flag) return 0.f;
      if (*(volatile unsigned*)status != 0u || global_ns() - t0 > timeout) {
        record_failure(status, host_status, abort_flag, task, detail);
        return 0.f;
      }
    }
  }
}

// Waits for a ring stage whose first test failed; records a failure after the timeout.
__device__ __noinline__ void spin_stage(uint64_t* full, unsigned parity, unsigned* prod_quit, unsigned* status,
                                        unsigned* host_status, unsigned* abort_flag, unsigned long long timeout,
                                        unsigned task, unsigned detail) {
  const unsigned long long t0 = global_ns();
  while (!mbar_test(full, parity)) {
    if (*(volatile unsigned*)prod_quit) return;  // nothing more will arrive
    if (global_ns() - t0 > timeout) {
      record_failure(status, host_status, abort_flag, task, detail);
      return;
    }
  }
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
  int ctid;             // 0..511 among compute threads
  int warp, lane;       // compute warp 0..15
  unsigned task_index;
  bool first_stage;     // tracing: the task has not yet received a weight stage
};

__device__ __forceinline__ void trace_mark(Ctx& c, int k) {
  if (c.P->trace != nullptr && c.ctid == 0) c.P->trace[(size_t)c.task_index * 4 + k] = global_ns();
}
__device__ __forceinline__ bool aborted(const Ctx& c) { return *(volatile unsigned*)&c.ctl->abort != 0u; }
__device__ __forceinline__ float word_value(Ctx& c, unsigned long long w, const unsigned long long* p, unsigned detail) {
  if ((unsigned)(w >> 32) == c.tag) return __uint_as_float((unsigned)w);
  return spin_word(p, c.tag, &c.ctl->abort, c.P->status, c.P->host_status, c.P->timeout_ns, c.task_index, detail,
                   c.P->poll_backoff_ns);
}
__device__ __forceinline__ void put_word(Ctx& c, unsigned long long* p, float v) {
  if (!aborted(c)) st_word(p, c.tag, v);
}

// Batched polling: this thread's words src[i], i = ctid + k*kCT < n, with up to 4 loads in flight.
template <typename F>
__device__ __forceinline__ void poll_words(Ctx& c, const unsigned long long* src, int n, unsigned detail, F&& sink) {
  for (int k0 = 0; k0 * kCT < n; k0 += 4) {
    unsigned long long w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = c.ctid + (k0 + k) * kCT;
      w[k] = i < n ? ld_word(src + i) : 0ull;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = c.ctid + (k0 + k) * kCT;
      if (i < n) sink(i, k0 + k, word_value(c, w[k], src + i, detail | (unsigned)i));
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
  if (!mbar_test(&c.ctl->full[s], ph))
    spin_stage(&c.ctl->full[s], ph, &c.ctl->prod_quit, c.P->status, c.P->host_status, &c.ctl->abort, c.P->timeout_ns,
               c.task_index, 0xF000u | s);
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

// Norm gain a task applies to its input (null for tasks without a norm).
__device__ __forceinline__ const uint16_t* task_gain(const Ctl* ctl, const Task& t, int L) {
  if (t.type == T_QKV) return ctl->gain[2 * t.layer];
  if (t.type == T_GATEUP) return ctl->gain[2 * t.layer + 1];
  if (t.type == T_LMHEAD) return ctl->gain[2 * L];
  return nullptr;
}
// This thread's gain values (elements ctid + k*kCT) of a task, loaded ahead of the task.
__device__ __forceinline__ void load_gains(const Ctx& c, const Task& t, float g[4]) {
  const uint16_t* gp = task_gain(c.ctl, t, c.P->L);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = c.ctid + k * kCT;
    g[k] = (gp != nullptr && i < c.P->H) ? bf16_to_f32(gp[i]) : 0.f;
  }
}

// ------------------------------------------------------------------ input vector of a GEMV task
// Loads n activations (words, or the token's embedding row when src is null) into sv in the split
// layout.  With a norm (gr != null, n == H), it stores gain * x and leaves this thread's share of
// sum(x^2) in *ss: RMSNorm's scalar 1/sqrt(mean(x^2)+eps) is applied to the GEMV results instead,
// so the norm costs no barrier of its own (the pages' "folding" of small producers into their
// consumer).  No barrier here.
__device__ __forceinline__ void fetch_input(Ctx& c, const unsigned long long* src, int n, const float* gr, float* sv,
                                            float* ss) {
  float acc = 0.f;
  if (src == nullptr) {
    const uint16_t* e = c.P->embed + (size_t)c.token * n;
    for (int k = 0; k * kCT < n; ++k) {
      const int i = c.ctid + k * kCT;
      if (i < n) {
        float x = bf16_to_f32(e[i]);
        if (gr != nullptr) {
          acc = fmaf(x, x, acc);
          x *= gr[k & 3];
        }
        sv[xpos(i, n)] = x;
      }
    }
  } else {
    poll_words(c, src, n, 0x100000u, [&](int i, int k, float x) {
      if (gr != nullptr) {
        acc = fmaf(x, x, acc);
        x *= gr[k & 3];
      }
      sv[xpos(i, n)] = x;
    });
  }
  *ss = acc;
}

// ------------------------------------------------------------------ GEMV on ring stages
// Dot products of the task's weight rows (in chunk order) with x, consuming up to kGemvBatch ring
// stages at a time.  Warps split K into t.gpr slices; each warp keeps its slice of x in registers
// (loaded once) and streams rows past it, so shared-memory traffic is the weight bytes alone.  Two
// bf16 weights multiply two x values per packed fp32x2 FMA (each an ordinary fp32 FMA).
// res[row * gpr + slice] = scale * partial; res_row() sums the slices in a fixed order, so results
// are deterministic.  Ends with a compute barrier.
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

__device__ __forceinline__ void gemv_xreg(Ctx& c, const Task& t, int in, const float* x, float* res, float scale) {
  const int nvec = in >> 3;  // 16-byte vectors per row
  const int gpr = (int)t.gpr, gshift = 31 - __clz(gpr);
  const int slice = c.warp & (gpr - 1), rw = c.warp >> gshift, rpp = kComputeWarps >> gshift;
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
  const size_t row_bytes = (size_t)in * 2;
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
    auto row_of = [&](int r) -> const uint4* {
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
      return reinterpret_cast<const uint4*>(base + (size_t)r * row_bytes);
    };
    // two rows per iteration; the loop bound is uniform across the warp (shuffles below)
    for (int ra = rw; ra < total; ra += 2 * rpp) {
      const int rb = ra + rpp;
      const bool two = rb < total;
      const uint4* A = row_of(ra);
      const uint4* B = row_of(two ? rb : ra);
      unsigned long long a0 = 0ull, a1 = 0ull, b0 = 0ull, b1 = 0ull;
#pragma unroll
      for (int k = 0; k < kGemvXVec; ++k) {
        const int v = v0 + c.lane + 32 * k;
        if (v < v1) {
          const uint4 wa = A[v];
          const uint4 wb = B[v];
          a0 = ffma2(bf2(wa.x), xp[k][0], a0);
          a1 = ffma2(bf2(wa.y), xp[k][1], a1);
          a0 = ffma2(bf2(wa.z), xp[k][2], a0);
          a1 = ffma2(bf2(wa.w), xp[k][3], a1);
          b0 = ffma2(bf2(wb.x), xp[k][0], b0);
          b1 = ffma2(bf2(wb.y), xp[k][1], b1);
          b0 = ffma2(bf2(wb.z), xp[k][2], b0);
          b1 = ffma2(bf2(wb.w), xp[k][3], b1);
        }
      }
      float sa = sum2(a0) + sum2(a1), sb = sum2(b0) + sum2(b1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sa += __shfl_xor_sync(0xffffffffu, sa, o);
        sb += __shfl_xor_sync(0xffffffffu, sb, o);
      }
      if (c.lane == 0) {
        res[((rbase + ra) << gshift) + slice] = sa * scale;
        if (two) res[((rbase + rb) << gshift) + slice] = sb * scale;
      }
    }
    stages_release(c, (unsigned)nb);
    rbase += total;
  }
  compute_sync();
}
// Small tasks (at most 16 rows per batch, t.gpr == 0): one warp per row over the full K, x read
// from shared memory -- the fewest instructions when each warp has a row or two.
__device__ __forceinline__ void gemv_rows(Ctx& c, const Task& t, int in, const float* x, float* res, float scale) {
  const int nvec = in >> 3;
  const float4* xlo = reinterpret_cast<const float4*>(x);
  const float4* xhi = reinterpret_cast<const float4*>(x + (in >> 1));
  const size_t row_bytes = (size_t)in * 2;
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
    for (int r = c.warp; r < total; r += kComputeWarps) {
      int rr = r;
      const unsigned char* base = s0;
      if (rr >= n0) {
        rr -= n0;
        base = s1;
        if (rr >= n1) {
          rr -= n1;
          base = s2;
          if (rr >= n2) {
            rr -= n2;
            base = s3;
          }
        }
      }
      const uint4* row = reinterpret_cast<const uint4*>(base + (size_t)rr * row_bytes);
      unsigned long long a0 = 0ull, a1 = 0ull;
      for (int v = c.lane; v < nvec; v += 32) {
        const uint4 w = row[v];
        const float4 p = xlo[v], q = xhi[v];
        a0 = ffma2(bf2(w.x), pack2(__float_as_uint(p.x), __float_as_uint(p.y)), a0);
        a1 = ffma2(bf2(w.y), pack2(__float_as_uint(p.z), __float_as_uint(p.w)), a1);
        a0 = ffma2(bf2(w.z), pack2(__float_as_uint(q.x), __float_as_uint(q.y)), a0);
        a1 = ffma2(bf2(w.w), pack2(__float_as_uint(q.z), __float_as_uint(q.w)), a1);
      }
      const float acc = warp_sum(sum2(a0) + sum2(a1));
      if (c.lane == 0) res[rbase + r] = acc * scale;
    }
    stages_release(c, (unsigned)nb);
    rbase += total;
  }
  compute_sync();
}
__device__ __forceinline__ void gemv(Ctx& c, const Task& t, int in, const float* x, float* res, float scale) {
  if (t.gpr == 0) gemv_rows(c, t, in, x, res, scale);
  else gemv_xreg(c, t, in, x, res, scale);
}
__device__ __forceinline__ float res_row(const float* res, int i, int gpr) {
  if (gpr <= 1) return res[i];
  float v = 0.f;
  for (int s = 0; s < gpr; ++s) v += res[i * gpr + s];
  return v;
}

// ------------------------------------------------------------------ attention task
// One KV head, one context split.  Cached positions [a, min(a + split_len, pos)) arrive through the
// ring (all of the task's stages are held at once); the owner split (the one holding `pos`) also
// takes the current row from the QKV words, rotates and rounds it, appends it to the cache, and
// attends to it.  Writes per query head o (normalised over this split), m and l.
// Query heads sharing the KV head are packed into the task, so each K/V row is read once (README,
// "Current status", decode attention).
__device__ __forceinline__ void task_attn(Ctx& c, const Task& t, float* sv) {
  const KernelParams& P = *c.P;
  const int l = t.layer, kvh = (int)t.row0, sp = (int)t.nrows;
  const int d = P.d, g = P.g, R = P.rows_per_stage, half = d / 2;
  const int pos = c.pos;
  const int a = sp * P.split_len;
  if (a > pos) return;  // inactive split (the producer streamed nothing for it either)
  const int b = min(a + P.split_len, pos);
  const bool owner = (pos / P.split_len) == sp;
  const int nh = b - a;                       // cached positions
  const int np = nh + (owner ? 1 : 0);        // positions attended
  const int nst = (nh + R - 1) / R;           // ring stages of this task
  const int SL = P.split_len + 1;             // score row stride
  const int O = g * d;                        // outputs of the task

  float* sq = sv;                 // [g][d]     rotated queries
  float* ss = sq + O;             // [g][SL]    scores, then probabilities
  float* part = ss + g * SL;          // [max(2 kCT, O)] partial outputs
  float* kc = part + max(2 * kCT, O); // [d]        current K (rotated, bf16-rounded)
  float* vc = kc + d;             // [d]        current V (bf16-rounded)
  float* sm = vc + d;             // [g]        max
  float* sl = sm + g;             // [g]        sum
  const float2* cs = c.ctl->rope;  // this step's cos/sin (loaded at kernel start)

  const unsigned long long* w = layer_words(P, l) + P.act.qkv;
  const int qd = P.nq * d, kvd = P.nkv * d;
  poll_words(c, w + (size_t)kvh * O, O, 0x200000u, [&](int i, int, float x) { sq[i] = x; });
  if (owner) {
    poll_words(c, w + qd + kvh * d, d, 0x210000u, [&](int i, int, float x) { kc[i] = x; });
    poll_words(c, w + qd + kvd + kvh * d, d, 0x220000u, [&](int i, int, float x) { vc[i] = x; });
  }
  compute_sync();
  trace_mark(c, 1);
  // RoPE (rotate-half pairs (i, i + d/2)); the current K/V row is rounded to bf16 and appended.
  for (int e = c.ctid; e < g * half; e += kCT) {
    const int h = e / half, i = e - h * half;
    const float2 r = cs[i];
    const float x0 = sq[h * d + i], x1 = sq[h * d + i + half];
    sq[h * d + i] = x0 * r.x - x1 * r.y;
    sq[h * d + i + half] = x1 * r.x + x0 * r.y;
  }
  if (owner && c.ctid < half) {
    const int i = c.ctid;
    const float2 r = cs[i];
    const float x0 = kc[i], x1 = kc[i + half];
    const __nv_bfloat16 k0 = __float2bfloat16_rn(x0 * r.x - x1 * r.y);
    const __nv_bfloat16 k1 = __float2bfloat16_rn(x1 * r.x + x0 * r.y);
    const __nv_bfloat16 v0 = __float2bfloat16_rn(vc[i]);
    const __nv_bfloat16 v1 = __float2bfloat16_rn(vc[i + half]);
    kc[i] = __bfloat162float(k0);
    kc[i + half] = __bfloat162float(k1);
    vc[i] = __bfloat162float(v0);
    vc[i + half] = __bfloat162float(v1);
    if (!aborted(c)) {
      __nv_bfloat16* Kc = reinterpret_cast<__nv_bfloat16*>(P.kv) + ((((size_t)l * 2 + 0) * P.nkv + kvh) * P.C + pos) * d;
      __nv_bfloat16* Vc = reinterpret_cast<__nv_bfloat16*>(P.kv) + ((((size_t)l * 2 + 1) * P.nkv + kvh) * P.C + pos) * d;
      Kc[i] = k0;
      Kc[i + half] = k1;
      Vc[i] = v0;
      Vc[i + half] = v1;
    }
  }
  compute_sync();

  // the task's cached K/V: stage st holds positions a + st*R .. (K rows, then V rows); R is a power
  // of two and the stages are consecutive ring slots, so no division is needed in the loops below
  unsigned s_first = 0, ph_unused = 0;
  slot_after(c, 0, s_first, ph_unused);
  for (int st = 0; st < nst; ++st) stage_wait(c, (unsigned)st);
  const int rshift = 31 - __clz(R);
  const unsigned ns = c.ns;
  auto kstage = [&](int j) -> const uint16_t* {
    unsigned s = s_first + (unsigned)(j >> rshift);
    s = s >= ns ? s - ns : s;
    return reinterpret_cast<const uint16_t*>(c.ring + (size_t)s * kStageBytes) + (size_t)(j & (R - 1)) * d;
  };

  // scores: 8 lanes per position; the K row is loaded once and dotted with every packed query head
  const float scale = P.attn_scale;
  const int elems = d / 8;  // 8 or 16 per lane
  for (int jb = c.warp * 4; jb < np; jb += kComputeWarps * 4) {
    const int j = jb + c.lane / 8, sub = c.lane % 8;
    const bool valid = j < np;
    float kf[16];
    if (valid && j < nh) {
      const uint16_t* kr = kstage(j) + sub * elems;
#pragma unroll
      for (int e = 0; e < 16; e += 8) {
        if (e < elems) {
          const uint4 kw = *reinterpret_cast<const uint4*>(kr + e);
          kf[e + 0] = bf16_lo(kw.x);
          kf[e + 1] = bf16_hi(kw.x);
          kf[e + 2] = bf16_lo(kw.y);
          kf[e + 3] = bf16_hi(kw.y);
          kf[e + 4] = bf16_lo(kw.z);
          kf[e + 5] = bf16_hi(kw.z);
          kf[e + 6] = bf16_lo(kw.w);
          kf[e + 7] = bf16_hi(kw.w);
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) kf[e + q] = 0.f;
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) kf[e] = (valid && e < elems) ? kc[sub * elems + e] : 0.f;
    }
    for (int h = 0; h < g; ++h) {
      const float* qr = sq + h * d + sub * elems;
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 16; e += 4) {
        if (e < elems) {
          const float4 q = *reinterpret_cast<const float4*>(qr + e);
          acc = fmaf(kf[e + 0], q.x, acc);
          acc = fmaf(kf[e + 1], q.y, acc);
          acc = fmaf(kf[e + 2], q.z, acc);
          acc = fmaf(kf[e + 3], q.w, acc);
        }
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      if (valid && sub == 0) ss[h * SL + j] = acc * scale;
    }
  }
  compute_sync();
  // softmax over this split: warp h handles head h
  if (c.warp < g) {
    const int h = c.warp;
    float mx = -INFINITY;
    for (int j = c.lane; j < np; j += 32) mx = fmaxf(mx, ss[h * SL + j]);
    mx = warp_max(mx);
    float psum = 0.f;
    for (int j = c.lane; j < np; j += 32) {
      const float p = expf(ss[h * SL + j] - mx);
      ss[h * SL + j] = p;
      psum += p;
    }
    psum = warp_sum(psum);
    if (c.lane == 0) {
      sm[h] = mx;
      sl[h] = psum;
    }
  }
  compute_sync();
  // o = sum_j p_j V_j, two adjacent outputs per thread (one bf16 pair of V per position).  With
  // O/2 <= 512 output pairs, the threads form kCT / (O/2) groups that split the positions.
  const int O2 = O >> 1;
  const int ngroups = O2 <= kCT ? kCT / O2 : 1;
  auto vsum = [&](int o2, int grp) {
    const int o = o2 * 2, h = o / d, tt = o - h * d;
    const float* pr = ss + h * SL;
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
    int j = grp;
    for (; j + ngroups < nh; j += 2 * ngroups) {
      const uint32_t v0 = *reinterpret_cast<const uint32_t*>(kstage(j) + (size_t)R * d + tt);
      const uint32_t v1 = *reinterpret_cast<const uint32_t*>(kstage(j + ngroups) + (size_t)R * d + tt);
      const float p0 = pr[j], p1 = pr[j + ngroups];
      a0 = fmaf(p0, bf16_lo(v0), a0);
      a1 = fmaf(p0, bf16_hi(v0), a1);
      b0 = fmaf(p1, bf16_lo(v1), b0);
      b1 = fmaf(p1, bf16_hi(v1), b1);
    }
    for (; j < np; j += ngroups) {
      const float p0 = pr[j];
      if (j < nh) {
        const uint32_t v0 = *reinterpret_cast<const uint32_t*>(kstage(j) + (size_t)R * d + tt);
        a0 = fmaf(p0, bf16_lo(v0), a0);
        a1 = fmaf(p0, bf16_hi(v0), a1);
      } else {
        a0 = fmaf(p0, vc[tt], a0);
        a1 = fmaf(p0, vc[tt + 1], a1);
      }
    }
    part[grp * O + o] = a0 + b0;
    part[grp * O + o + 1] = a1 + b1;
  };
  if (O2 <= kCT) {
    if (c.ctid / O2 < ngroups) vsum(c.ctid % O2, c.ctid / O2);
  } else {
    for (int o2 = c.ctid; o2 < O2; o2 += kCT) vsum(o2, 0);
  }
  stages_release(c, (unsigned)nst);
  compute_sync();
  unsigned long long* out = layer_words(P, l) + P.act.att + (size_t)(kvh * P.nsplit + sp) * g * (d + 2);
  for (int e = c.ctid; e < g * (d + 2); e += kCT) {
    const int h = e / (d + 2), tt = e - h * (d + 2);
    float v;
    if (tt < d) {
      float acc = 0.f;
      for (int q = 0; q < ngroups; ++q) acc += part[q * O + h * d + tt];
      v = acc / sl[h];
    } else {
      v = tt == d ? sm[h] : sl[h];
    }
    put_word(c, out + e, v);
  }
}

// Attention output of every query head into o[nq*d], combining the active context splits of each
// KV head by their log-sum-exp weights (split-context "flash decoding", README "Current status").
__device__ __forceinline__ void fetch_attention(Ctx& c, int l, float* o) {
  const KernelParams& P = *c.P;
  const int d = P.d, g = P.g;
  const int nact = c.pos / P.split_len + 1;
  const unsigned long long* base = layer_words(P, l) + P.act.att;
  const int blk = g * (d + 2);  // words per (KV head, split)
  if (nact == 1) {
    // one split: o is the split's normalised output
    for (int e0 = 0; e0 * kCT < P.nq * d; e0 += 4) {
      unsigned long long w[4];
      const unsigned long long* ptr[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = c.ctid + (e0 + k) * kCT;
        const int h = e / d, tt = e - h * d;
        ptr[k] = base + (size_t)(h / g) * P.nsplit * blk + (h % g) * (d + 2) + tt;
        w[k] = e < P.nq * d ? ld_word(ptr[k]) : 0ull;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = c.ctid + (e0 + k) * kCT;
        if (e < P.nq * d) o[xpos(e, P.nq * d)] = word_value(c, w[k], ptr[k], 0x300000u | e);
      }
    }
    return;
  }
  for (int e = c.ctid; e < P.nq * d; e += kCT) {
    const int h = e / d, tt = e - h * d, kvh = h / g, hh = h - kvh * g;
    float M = -INFINITY;
    for (int s = 0; s < nact; ++s) {
      const unsigned long long* p = base + (size_t)(kvh * P.nsplit + s) * blk + hh * (d + 2) + d;
      M = fmaxf(M, word_value(c, ld_word(p), p, 0x310000u | s));
    }
    float num = 0.f, den = 0.f;
    for (int s = 0; s < nact; ++s) {
      const unsigned long long* bp = base + (size_t)(kvh * P.nsplit + s) * blk + hh * (d + 2);
      const float m = word_value(c, ld_word(bp + d), bp + d, 0x320000u | s);
      const float lsum = word_value(c, ld_word(bp + d + 1), bp + d + 1, 0x330000u | s);
      const float wgt = lsum * expf(m - M);
      num = fmaf(wgt, word_value(c, ld_word(bp + tt), bp + tt, 0x340000u | s), num);
      den += wgt;
    }
    o[xpos(e, P.nq * d)] = num / den;
  }
}

// ------------------------------------------------------------------ producer warp
// Walks the CTA's chunk list (32 descriptors per coalesced load, the next batch loaded while the
// current one is issued) and fills the ring.  Lane 0 issues; the other lanes only help load.
__device__ __forceinline__ void produce(const KernelParams& P, int pos, Ctl* ctl, unsigned char* ring, uint32_t c0,
                                        uint32_t c1, int lane) {
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
        if (rows == kAttnChunk) {
          const int layer = (int)(src >> 48), kvh = (int)((src >> 32) & 0xFFFF), sp = (int)(unsigned)src;
          const int a = sp * P.split_len;
          if (a <= pos) {
            const int b = min(a + P.split_len, pos);
            const size_t head_off = (((size_t)layer * 2) * P.nkv + kvh) * P.C * P.d;
            const uint16_t* K = P.kv + head_off;
            const uint16_t* V = P.kv + head_off + (size_t)P.nkv * P.C * P.d;
            for (int jj = a; jj < b; jj += P.rows_per_stage) {
              const int n = min(P.rows_per_stage, b - jj);
              const unsigned nb = (unsigned)(n * P.d * 2);
              unsigned char* dst = acquire(2 * nb, (unsigned)n);
              if (!dst) {
                q = 1;
                break;
              }
              bulk_load(dst, K + (size_t)jj * P.d, nb, &ctl->full[stage], policy);
              bulk_load(dst + (size_t)P.rows_per_stage * P.d * 2, V + (size_t)jj * P.d, nb, &ctl->full[stage], policy);
              advance();
            }
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

// ------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ KernelParams P, const StepParams S) {
  extern __shared__ __align__(128) unsigned char smem[];
  Ctl* ctl = reinterpret_cast<Ctl*>(smem);
  if (threadIdx.x == 0) {
    ctl->skip = *(volatile unsigned*)P.status;  // sticky error from an earlier step: do nothing
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
  {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&P);
    uint32_t* dst = reinterpret_cast<uint32_t*>(&ctl->params);
    for (int i = threadIdx.x; i < (int)(sizeof(KernelParams) / 4); i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  if (ctl->skip) return;
  unsigned char* ring = smem + P.off_ring;
  const int warp = threadIdx.x / 32;
  if (warp == 0) {
    produce(ctl->params, S.pos, ctl, ring, P.chunk_off[blockIdx.x], P.chunk_off[blockIdx.x + 1], threadIdx.x & 31);
    return;
  }
  const uint32_t t0 = P.task_off[blockIdx.x], t1 = P.task_off[blockIdx.x + 1];
  Ctx c;
  c.P = &ctl->params;
  c.ctl = ctl;
  c.ring = ring;
  c.logits = S.logits;
  c.tag = S.tag;
  c.pos = S.pos;
  c.token = S.token;
  c.ns = (unsigned)P.num_stages;
  c.stage = 0;
  c.phase = 0;
  c.ctid = threadIdx.x - 32;
  c.warp = warp - 1;
  c.lane = threadIdx.x & 31;
  float* sv = reinterpret_cast<float*>(smem + P.off_sv);
  float* res = reinterpret_cast<float*>(smem + P.off_res);
  float* resid = reinterpret_cast<float*>(smem + P.off_resid);
  // two-deep descriptor pipeline; the gains of the next task load while the current one runs
  Task cur{}, nxt{};
  if (t0 < t1) cur = P.tasks[t0];
  if (t0 + 1 < t1) nxt = P.tasks[t0 + 1];
  float gcur[4], gnext[4];
  load_gains(c, cur, gcur);
  for (uint32_t ti = t0; ti < t1; ++ti) {
    const Task t = cur;
    cur = nxt;
    if (ti + 2 < t1) nxt = P.tasks[ti + 2];
    if (ti + 1 < t1) load_gains(c, cur, gnext);
    c.task_index = ti;
    c.first_stage = true;
    if (P.trace != nullptr && c.ctid == 0) P.trace[(size_t)ti * 4 + 3] = 0;
    trace_mark(c, 0);
    if (t.type == T_ATTN) {
      task_attn(c, t, sv);
    } else {
      // 1. inputs: one fetch path for every projection type
      const int l = t.layer;
      int in = P.H;
      float ss = 0.f;
      float bias[4] = {0.f, 0.f, 0.f, 0.f};
      if (t.type == T_QKV && P.qkv_bias) {
        const int qd = P.nq * P.d, kvd = P.nkv * P.d;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = c.ctid + k * kCT;
          if (i < (int)t.nrows) {
            const int o = (int)t.row0 + i;
            const uint16_t* b = o < qd ? ctl->bias[3 * l] + o
                                       : (o < qd + kvd ? ctl->bias[3 * l + 1] + (o - qd) : ctl->bias[3 * l + 2] + (o - qd - kvd));
            bias[k] = bf16_to_f32(*b);
          }
        }
      }
      if (t.type == T_OPROJ) {
        in = P.nq * P.d;
        fetch_attention(c, l, sv);
      } else {
        const unsigned long long* src;
        if (t.type == T_QKV) src = x_in_words(P, l);
        else if (t.type == T_GATEUP) src = layer_words(P, l) + P.act.xa;
        else if (t.type == T_DOWN) src = layer_words(P, l) + P.act.hh;
        else src = layer_words(P, P.L - 1) + P.act.xm;  // LM head
        if (t.type == T_DOWN) in = P.I;
        fetch_input(c, src, in, t.type == T_DOWN ? nullptr : gcur, sv, &ss);
      }
      if (t.type == T_OPROJ || t.type == T_DOWN) {
        const unsigned long long* rsrc = t.type == T_OPROJ ? x_in_words(P, l) : layer_words(P, l) + P.act.xa;
        if (rsrc == nullptr) {
          const uint16_t* e = P.embed + (size_t)c.token * P.H + t.row0;
          for (int i = c.ctid; i < (int)t.nrows; i += kCT) resid[i] = bf16_to_f32(e[i]);
        } else {
          poll_words(c, rsrc + t.row0, (int)t.nrows, 0x400000u, [&](int i, int, float x) { resid[i] = x; });
        }
      }
      const bool norm = t.type == T_QKV || t.type == T_GATEUP || t.type == T_LMHEAD;
      if (norm) {
        ss = warp_sum(ss);
        if (c.lane == 0) ctl->red[c.warp] = ss;
      }
      compute_sync();
      float scale = 1.f;
      if (norm) {
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kComputeWarps; ++w) tot += ctl->red[w];
        scale = 1.0f / sqrtf(tot / (float)P.H + P.eps);
      }
      trace_mark(c, 1);
      // 2. the projection
      gemv(c, t, in, sv, res, scale);
      // 3. epilogue
      const int gpr = (int)t.gpr, n = (int)t.nrows;
      if (t.type == T_QKV) {
        unsigned long long* out = layer_words(P, l) + P.act.qkv + t.row0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = c.ctid + k * kCT;
          if (i < n) put_word(c, out + i, res_row(res, i, gpr) + bias[k]);
        }
      } else if (t.type == T_GATEUP) {
        unsigned long long* out = layer_words(P, l) + P.act.hh + t.row0;
        for (int i = c.ctid; i < n; i += kCT) {
          const float gt = res_row(res, i, gpr), up = res_row(res, n + i, gpr);
          put_word(c, out + i, gt / (1.0f + expf(-gt)) * up);
        }
      } else if (t.type == T_LMHEAD) {
        if (!aborted(c))
          for (int i = c.ctid; i < n; i += kCT) c.logits[t.row0 + i] = res_row(res, i, gpr);
      } else {
        unsigned long long* out = layer_words(P, l) + (t.type == T_OPROJ ? P.act.xa : P.act.xm) + t.row0;
        for (int i = c.ctid; i < n; i += kCT) put_word(c, out + i, resid[i] + res_row(res, i, gpr));
      }
    }
    compute_sync();  // the next task reuses the shared vectors
    trace_mark(c, 2);
#pragma unroll
    for (int k = 0; k < 4; ++k) gcur[k] = gnext[k];
  }
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
__global__ void kv_fill_kernel(uint16_t* kv_layer, const float* k_raw, const float* v_raw, const float2* rope, int nkv,
                               int C, int d, int p0, int n) {
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
    __nv_bfloat16* K = reinterpret_cast<__nv_bfloat16*>(kv_layer) + ((size_t)h * C + p) * d;
    __nv_bfloat16* V = reinterpret_cast<__nv_bfloat16*>(kv_layer) + ((size_t)(nkv + h) * C + p) * d;
    K[i] = __float2bfloat16_rn(x0 * r.x - x1 * r.y);
    K[i + half] = __float2bfloat16_rn(x1 * r.x + x0 * r.y);
    V[i] = __float2bfloat16_rn(vr[i]);
    V[i + half] = __float2bfloat16_rn(vr[i + half]);
  }
}

}  // namespace mbk

// Launch helpers used by the C ABI (mbk_api.cu).
namespace mbk {
const void* decode_kernel_ptr() { return reinterpret_cast<const void*>(&decode_kernel); }
cudaError_t launch_rope_table(float2* out, int C, int d, double theta, cudaStream_t st) {
  rope_table_kernel<<<264, 256, 0, st>>>(out, C, d, theta);
  return cudaGetLastError();
}
cudaError_t launch_kv_fill(uint16_t* kv_layer, const float* k_raw, const float* v_raw, const float2* rope, int nkv, int C,
                           int d, int p0, int n, cudaStream_t st) {
  kv_fill_kernel<<<264, 256, 0, st>>>(kv_layer, k_raw, v_raw, rope, nkv, C, d, p0, n);
  return cudaGetLastError();
}
}  // namespace mbk
