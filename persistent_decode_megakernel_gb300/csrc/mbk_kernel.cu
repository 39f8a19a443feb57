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
// the next task's descriptor) is loaded before the task waits for its inputs, so the critical path
// of a task is: inputs arrive -> one block barrier -> GEMV on shared-memory weights -> words out.
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

// Shared-memory control block (first KB of dynamic shared memory).
struct Ctl {
  uint64_t full[kMaxRingStages];
  uint64_t empty[kMaxRingStages];
  uint32_t stage_rows[kMaxRingStages];  // weight rows held by each stage (written by the producer)
  unsigned abort;       // set once this CTA gave up a wait: later activation waits return at once
  unsigned prod_quit;   // the producer stopped early (its consumers stopped taking stages)
  unsigned skip;        // an earlier step failed: this launch does nothing
  unsigned pad;
  float red[32];        // block reduction scratch
};
static_assert(sizeof(Ctl) <= 1024, "control block must fit the first KB");

struct Ctx {
  const KernelParams* P;
  StepParams S;
  Ctl* ctl;
  unsigned char* ring;
  unsigned it;          // ring position (same sequence as the producer's)
  int ctid;             // 0..511 among compute threads
  int warp, lane;       // compute warp 0..15
  unsigned task_index;
  bool first_stage;     // tracing: the task has not yet received a weight stage
};

// Tracing (off unless P.trace is set): stamp slot k of the current task.
__device__ __forceinline__ void trace_mark(Ctx& c, int k) {
  if (c.P->trace != nullptr && c.ctid == 0) c.P->trace[(size_t)c.task_index * 4 + k] = global_ns();
}

__device__ void record_failure(Ctx& c, unsigned detail) {
  const KernelParams& P = *c.P;
  if (atomicCAS(&P.status[0], 0u, (unsigned)DS_TIMEOUT) == 0u) {
    P.status[1] = blockIdx.x;
    P.status[2] = c.task_index;
    P.status[3] = detail;
    if (P.host_status) {
      volatile unsigned* hs = P.host_status;
      hs[1] = blockIdx.x;
      hs[2] = c.task_index;
      hs[3] = detail;
      __threadfence_system();
      hs[0] = (unsigned)DS_TIMEOUT;
    }
  }
  *(volatile unsigned*)&c.ctl->abort = 1u;
}

__device__ __forceinline__ bool aborted(const Ctx& c) { return *(volatile unsigned*)&c.ctl->abort != 0u; }

// Finish waiting for a word that was not ready at the first load; returns its value (0 on abort).
__device__ __noinline__ float spin_word(Ctx& c, const unsigned long long* p, unsigned detail) {
  if (aborted(c)) return 0.f;
  unsigned long long t0 = global_ns();
  for (unsigned n = 1;; ++n) {
    const unsigned long long w = ld_word(p);
    if ((unsigned)(w >> 32) == c.S.tag) return __uint_as_float((unsigned)w);
    if ((n & 63u) == 0u) {
      if (aborted(c)) return 0.f;
      if (*(volatile unsigned*)c.P->status != 0u || global_ns() - t0 > c.P->timeout_ns) {
        record_failure(c, detail);
        return 0.f;
      }
    }
  }
}
__device__ __forceinline__ float word_value(Ctx& c, unsigned long long w, const unsigned long long* p, unsigned detail) {
  return (unsigned)(w >> 32) == c.S.tag ? __uint_as_float((unsigned)w) : spin_word(c, p, detail);
}

__device__ __forceinline__ void put_word(Ctx& c, unsigned long long* p, float v) {
  if (!aborted(c)) st_word(p, c.S.tag, v);
}

// Batched polling: this thread's words src[i], i = ctid + k*kCT < n, with up to 8 loads in flight.
template <typename F>
__device__ __forceinline__ void poll_words(Ctx& c, const unsigned long long* src, int n, unsigned detail, F&& sink) {
  for (int k0 = 0; k0 * kCT < n; k0 += 8) {
    unsigned long long w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = c.ctid + (k0 + k) * kCT;
      w[k] = i < n ? ld_word(src + i) : 0ull;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = c.ctid + (k0 + k) * kCT;
      if (i < n) sink(i, word_value(c, w[k], src + i, detail | (unsigned)i));
    }
  }
}

// Ring stage `idx` (absolute ring position) once its data has landed.
__device__ __forceinline__ unsigned char* stage_wait(Ctx& c, unsigned idx) {
  const unsigned ns = (unsigned)c.P->num_stages;
  const unsigned s = idx % ns, ph = (idx / ns) & 1u;
  if (!mbar_test(&c.ctl->full[s], ph)) {
    unsigned long long t0 = global_ns();
    while (!mbar_test(&c.ctl->full[s], ph)) {
      if (*(volatile unsigned*)&c.ctl->prod_quit) break;  // nothing more will arrive
      if (global_ns() - t0 > c.P->timeout_ns) {
        record_failure(c, 0xF000u | s);
        break;
      }
    }
  }
  if (c.first_stage) {
    trace_mark(c, 3);
    c.first_stage = false;
  }
  return c.ring + (size_t)s * kStageBytes;
}
// Hand `n` stages back to the producer (every compute warp arrives once per stage).
__device__ __forceinline__ void stages_release(Ctx& c, unsigned n) {
  const unsigned ns = (unsigned)c.P->num_stages;
  __syncwarp();
  if (c.lane == 0)
    for (unsigned k = 0; k < n; ++k) mbar_arrive(&c.ctl->empty[(c.it + k) % ns]);
  c.it += n;
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

// ------------------------------------------------------------------ fused input fetch + RMSNorm
// Loads the residual stream entering this task (words, or the embedding row for layer 0) as
// gain * x into sv and returns 1 / sqrt(mean(x^2) + eps): the norm's scalar is applied to the GEMV
// results, so RMSNorm costs no barrier of its own (the pages' "folding" of small producers into
// their consumer).  Gains are loaded before the wait.  Ends with a compute barrier.
__device__ float fetch_normed(Ctx& c, const unsigned long long* src, const uint16_t* gain, float* sv) {
  const KernelParams& P = *c.P;
  const int n = P.H;  // <= kMaxTaskRows = 4 * kCT
  float gr[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = c.ctid + k * kCT;
    gr[k] = i < n ? bf16_to_f32(gain[i]) : 0.f;
  }
  float ss = 0.f;
  if (src == nullptr) {
    const uint16_t* e = P.embed + (size_t)c.S.token * n;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = c.ctid + k * kCT;
      if (i < n) {
        const float x = bf16_to_f32(e[i]);
        ss = fmaf(x, x, ss);
        sv[i] = x * gr[k];
      }
    }
  } else {
    poll_words(c, src, n, 0x100000u, [&](int i, float x) {
      ss = fmaf(x, x, ss);
      sv[i] = x * gr[(i - c.ctid) / kCT];
    });
  }
  ss = warp_sum(ss);
  if (c.lane == 0) c.ctl->red[c.warp] = ss;
  compute_sync();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kComputeWarps; ++w) tot += c.ctl->red[w];
  return 1.0f / sqrtf(tot / (float)n + P.eps);
}

// ------------------------------------------------------------------ GEMV on ring stages
// Partial dot products of the task's rows in chunk order: t.wpr warps share each weight row (each
// takes a K slice), so small chunks still keep all 16 warps busy.  res[row * wpr + slice] =
// scale * partial; res_row() sums the slices in a fixed order (results are deterministic).
// Rows per stage come from the producer.  Ends with a compute barrier.
__device__ void gemv(Ctx& c, const Task& t, int in, const float* x, float* res, float scale) {
  const int nvec = in >> 3;  // 16-byte vectors per row
  const float4* x4 = reinterpret_cast<const float4*>(x);
  const unsigned ns = (unsigned)c.P->num_stages;
  const int wpr = (int)t.wpr, rpp = kComputeWarps / wpr;
  const int r_in = c.warp / wpr, slice = c.warp % wpr;
  int rbase = 0;
  for (uint32_t k = 0; k < t.nchunks; ++k) {
    const unsigned char* stage = stage_wait(c, c.it);
    const int rows = (int)c.ctl->stage_rows[c.it % ns];
    for (int r = r_in; r < rows; r += rpp) {
      const uint4* row = reinterpret_cast<const uint4*>(stage + (size_t)r * in * 2);
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
      for (int v = slice * 32 + c.lane; v < nvec; v += wpr * 32) {
        const uint4 w = row[v];
        const float4 p = x4[2 * v], q = x4[2 * v + 1];
        a0 = fmaf(bf16_lo(w.x), p.x, a0);
        a1 = fmaf(bf16_hi(w.x), p.y, a1);
        a2 = fmaf(bf16_lo(w.y), p.z, a2);
        a3 = fmaf(bf16_hi(w.y), p.w, a3);
        a0 = fmaf(bf16_lo(w.z), q.x, a0);
        a1 = fmaf(bf16_hi(w.z), q.y, a1);
        a2 = fmaf(bf16_lo(w.w), q.z, a2);
        a3 = fmaf(bf16_hi(w.w), q.w, a3);
      }
      const float acc = warp_sum((a0 + a1) + (a2 + a3));
      if (c.lane == 0) res[(rbase + r) * wpr + slice] = acc * scale;
    }
    stages_release(c, 1);
    rbase += rows;
  }
  compute_sync();
}
__device__ __forceinline__ float res_row(const float* res, int i, int wpr) {
  float v = 0.f;
  for (int s = 0; s < wpr; ++s) v += res[i * wpr + s];
  return v;
}

// ------------------------------------------------------------------ task bodies
__device__ void task_qkv(Ctx& c, const Task& t, float* sv, float* res) {
  const KernelParams& P = *c.P;
  const int l = t.layer;
  const int qd = P.nq * P.d, kvd = P.nkv * P.d;
  float bias[4] = {0.f, 0.f, 0.f, 0.f};
  if (P.qkv_bias) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = c.ctid + k * kCT;
      if (i < (int)t.nrows) {
        const int o = (int)t.row0 + i;
        const uint16_t* b = o < qd ? P.layers[l].w[LW_BQ] + o
                                   : (o < qd + kvd ? P.layers[l].w[LW_BK] + (o - qd) : P.layers[l].w[LW_BV] + (o - qd - kvd));
        bias[k] = bf16_to_f32(*b);
      }
    }
  }
  const float r = fetch_normed(c, x_in_words(P, l), P.layers[l].w[LW_ATTN_NORM], sv);
  trace_mark(c, 1);
  gemv(c, t, P.H, sv, res, r);
  unsigned long long* out = layer_words(P, l) + P.act.qkv;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = c.ctid + k * kCT;
    if (i < (int)t.nrows) put_word(c, out + t.row0 + i, res_row(res, i, (int)t.wpr) + bias[k]);
  }
}

// One KV head, one context split.  Cached positions [a, min(a + split_len, pos)) arrive through the
// ring (all of the task's stages are held at once); the owner split (the one holding `pos`) also
// takes the current row from the QKV words, rotates and rounds it, appends it to the cache, and
// attends to it.  Writes per query head o (normalised over this split), m and l.
// Query heads sharing the KV head are packed into the task, so each K/V row is read once (README,
// "Current status", decode attention).
__device__ void task_attn(Ctx& c, const Task& t, float* sv) {
  const KernelParams& P = *c.P;
  const int l = t.layer, kvh = (int)t.row0, sp = (int)t.nrows;
  const int d = P.d, g = P.g, R = P.rows_per_stage, half = d / 2;
  const int pos = c.S.pos;
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
  float* part = ss + g * SL;      // [max(kCT, O)] partial outputs
  float* kc = part + max(kCT, O); // [d]        current K (rotated, bf16-rounded)
  float* vc = kc + d;             // [d]        current V (bf16-rounded)
  float* sm = vc + d;             // [g]        max
  float* sl = sm + g;             // [g]        sum

  // token-independent loads first: this position's cos/sin
  float2 cs_q[2] = {make_float2(1.f, 0.f), make_float2(1.f, 0.f)};
  const float2* cs = P.rope + (size_t)pos * half;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int e = c.ctid + k * kCT;
    if (e < g * half) cs_q[k] = cs[e % half];
  }
  const float2 cs_k = c.ctid < half ? cs[c.ctid] : make_float2(1.f, 0.f);

  const unsigned long long* w = layer_words(P, l) + P.act.qkv;
  const int qd = P.nq * d, kvd = P.nkv * d;
  poll_words(c, w + (size_t)kvh * O, O, 0x200000u, [&](int i, float x) { sq[i] = x; });
  if (owner) {
    poll_words(c, w + qd + kvh * d, d, 0x210000u, [&](int i, float x) { kc[i] = x; });
    poll_words(c, w + qd + kvd + kvh * d, d, 0x220000u, [&](int i, float x) { vc[i] = x; });
  }
  compute_sync();
  trace_mark(c, 1);
  // RoPE (rotate-half pairs (i, i + d/2)); the current K/V row is rounded to bf16 and appended.
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int e = c.ctid + k * kCT;
    if (e < g * half) {
      const int h = e / half, i = e % half;
      const float x0 = sq[h * d + i], x1 = sq[h * d + i + half];
      sq[h * d + i] = x0 * cs_q[k].x - x1 * cs_q[k].y;
      sq[h * d + i + half] = x1 * cs_q[k].x + x0 * cs_q[k].y;
    }
  }
  if (owner && c.ctid < half) {
    const int i = c.ctid;
    const float x0 = kc[i], x1 = kc[i + half];
    const __nv_bfloat16 k0 = __float2bfloat16_rn(x0 * cs_k.x - x1 * cs_k.y);
    const __nv_bfloat16 k1 = __float2bfloat16_rn(x1 * cs_k.x + x0 * cs_k.y);
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
  const unsigned ns = (unsigned)P.num_stages;
  for (int st = 0; st < nst; ++st) stage_wait(c, c.it + st);
  const int rshift = 31 - __clz(R);
  const unsigned s0 = c.it % ns;
  auto kstage = [&](int j) -> const uint16_t* {
    unsigned s = s0 + (unsigned)(j >> rshift);
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
  // o = sum_j p_j V_j.  With O <= 512 outputs, the threads form kCT / O groups that split the
  // positions (one output per thread); otherwise each thread owns outputs o, o + 512, ...
  const int ngroups = O <= kCT ? kCT / O : 1;
  auto vsum = [&](int o, int grp) {
    const int h = o / d, tt = o % d;
    const float* pr = ss + h * SL;
    float a0 = 0.f, a1 = 0.f;
    int j = grp;
    for (; j + ngroups < nh; j += 2 * ngroups) {
      a0 = fmaf(pr[j], bf16_to_f32(kstage(j)[(size_t)R * d + tt]), a0);
      a1 = fmaf(pr[j + ngroups], bf16_to_f32(kstage(j + ngroups)[(size_t)R * d + tt]), a1);
    }
    for (; j < np; j += ngroups) a0 = fmaf(pr[j], j < nh ? bf16_to_f32(kstage(j)[(size_t)R * d + tt]) : vc[tt], a0);
    part[grp * O + o] = a0 + a1;
  };
  if (O <= kCT) {
    if (c.ctid / O < ngroups) vsum(c.ctid % O, c.ctid / O);
  } else {
    for (int o = c.ctid; o < O; o += kCT) vsum(o, 0);
  }
  stages_release(c, (unsigned)nst);
  compute_sync();
  unsigned long long* out = layer_words(P, l) + P.act.att + (size_t)(kvh * P.nsplit + sp) * g * (d + 2);
  for (int e = c.ctid; e < g * (d + 2); e += kCT) {
    const int h = e / (d + 2), tt = e % (d + 2);
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
__device__ void fetch_attention(Ctx& c, int l, float* o) {
  const KernelParams& P = *c.P;
  const int d = P.d, g = P.g;
  const int nact = c.S.pos / P.split_len + 1;
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
        const int h = e / d, tt = e % d;
        ptr[k] = base + (size_t)(h / g) * P.nsplit * blk + (h % g) * (d + 2) + tt;
        w[k] = e < P.nq * d ? ld_word(ptr[k]) : 0ull;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = c.ctid + (e0 + k) * kCT;
        if (e < P.nq * d) o[e] = word_value(c, w[k], ptr[k], 0x300000u | e);
      }
    }
    return;
  }
  for (int e = c.ctid; e < P.nq * d; e += kCT) {
    const int h = e / d, tt = e % d, kvh = h / g, hh = h % g;
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
    o[e] = num / den;
  }
}

// Residual rows [row0, row0 + n) of a word vector (or the embedding row) into resid.
__device__ void fetch_rows(Ctx& c, const unsigned long long* src, int row0, int n, float* resid) {
  if (src == nullptr) {
    const uint16_t* e = c.P->embed + (size_t)c.S.token * c.P->H + row0;
    for (int i = c.ctid; i < n; i += kCT) resid[i] = bf16_to_f32(e[i]);
  } else {
    poll_words(c, src + row0, n, 0x400000u, [&](int i, float x) { resid[i] = x; });
  }
}

__device__ void task_oproj(Ctx& c, const Task& t, float* sv, float* res, float* resid) {
  const KernelParams& P = *c.P;
  const int l = t.layer;
  fetch_attention(c, l, sv);
  fetch_rows(c, x_in_words(P, l), (int)t.row0, (int)t.nrows, resid);
  compute_sync();
  trace_mark(c, 1);
  gemv(c, t, P.nq * P.d, sv, res, 1.0f);
  unsigned long long* out = layer_words(P, l) + P.act.xa;
  for (int i = c.ctid; i < (int)t.nrows; i += kCT) put_word(c, out + t.row0 + i, resid[i] + res_row(res, i, (int)t.wpr));
}

__device__ void task_gateup(Ctx& c, const Task& t, float* sv, float* res) {
  const KernelParams& P = *c.P;
  const int l = t.layer;
  const float r = fetch_normed(c, layer_words(P, l) + P.act.xa, P.layers[l].w[LW_MLP_NORM], sv);
  trace_mark(c, 1);
  gemv(c, t, P.H, sv, res, r);
  unsigned long long* out = layer_words(P, l) + P.act.hh;
  const int n = (int)t.nrows;
  for (int i = c.ctid; i < n; i += kCT) {
    const float gt = res_row(res, i, (int)t.wpr), up = res_row(res, n + i, (int)t.wpr);
    const float silu = gt / (1.0f + expf(-gt));
    put_word(c, out + t.row0 + i, silu * up);
  }
}

__device__ void task_down(Ctx& c, const Task& t, float* sv, float* res, float* resid) {
  const KernelParams& P = *c.P;
  const int l = t.layer;
  poll_words(c, layer_words(P, l) + P.act.hh, P.I, 0x500000u, [&](int i, float x) { sv[i] = x; });
  fetch_rows(c, layer_words(P, l) + P.act.xa, (int)t.row0, (int)t.nrows, resid);
  compute_sync();
  trace_mark(c, 1);
  gemv(c, t, P.I, sv, res, 1.0f);
  unsigned long long* out = layer_words(P, l) + P.act.xm;
  for (int i = c.ctid; i < (int)t.nrows; i += kCT) put_word(c, out + t.row0 + i, resid[i] + res_row(res, i, (int)t.wpr));
}

__device__ void task_lmhead(Ctx& c, const Task& t, float* sv, float* res) {
  const KernelParams& P = *c.P;
  const float r = fetch_normed(c, layer_words(P, P.L - 1) + P.act.xm, P.final_norm, sv);
  trace_mark(c, 1);
  gemv(c, t, P.H, sv, res, r);
  if (!aborted(c))
    for (int i = c.ctid; i < (int)t.nrows; i += kCT) c.S.logits[t.row0 + i] = res_row(res, i, (int)t.wpr);
}

// ------------------------------------------------------------------ producer warp
// Walks the CTA's chunk list (32 descriptors per coalesced load, the next batch loaded while the
// current one is issued) and fills the ring.  Lane 0 issues; the other lanes only help load.
__device__ void produce(const KernelParams& P, const StepParams& S, Ctl* ctl, unsigned char* ring, uint32_t c0,
                        uint32_t c1, int lane) {
  const uint64_t policy = evict_first_policy();
  const unsigned ns = (unsigned)P.num_stages;
  unsigned it = 0;
  bool quit = false;
  // lane 0: wait for a free stage, record its rows, arm its barrier; returns null if consumers stall
  auto acquire = [&](unsigned bytes, uint32_t rows) -> unsigned char* {
    const unsigned s = it % ns, k = it / ns;
    if (k > 0) {
      const unsigned ph = (k - 1) & 1u;
      if (!mbar_test(&ctl->empty[s], ph)) {
        unsigned long long tstart = global_ns();
        while (!mbar_test(&ctl->empty[s], ph)) {
          // Consumers keep taking stages even after a failed activation wait (they stop waiting
          // for activations instead), so this only expires if a consumer is wedged: stop streaming.
          if (global_ns() - tstart > 4 * P.timeout_ns) {
            if (atomicCAS(&P.status[0], 0u, (unsigned)DS_TIMEOUT) == 0u) {
              P.status[1] = blockIdx.x;
              P.status[3] = 0xE000u | s;
            }
            *(volatile unsigned*)&ctl->prod_quit = 1u;
            return nullptr;
          }
        }
      }
    }
    ctl->stage_rows[s] = rows;
    mbar_expect_tx(&ctl->full[s], bytes);
    return ring + (size_t)s * kStageBytes;
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
          if (a <= S.pos) {
            const int b = min(a + P.split_len, S.pos);
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
              const unsigned s = it % ns;
              bulk_load(dst, K + (size_t)jj * P.d, nb, &ctl->full[s], policy);
              bulk_load(dst + (size_t)P.rows_per_stage * P.d * 2, V + (size_t)jj * P.d, nb, &ctl->full[s], policy);
              ++it;
            }
          }
        } else {
          unsigned char* dst = acquire(bytes, rows);
          if (!dst) {
            q = 1;
          } else {
            bulk_load(dst, reinterpret_cast<const void*>(src), bytes, &ctl->full[it % ns], policy);
            ++it;
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
  __syncthreads();
  if (ctl->skip) return;
  unsigned char* ring = smem + P.off_ring;
  const int warp = threadIdx.x / 32;
  if (warp == 0) {
    produce(P, S, ctl, ring, P.chunk_off[blockIdx.x], P.chunk_off[blockIdx.x + 1], threadIdx.x & 31);
    return;
  }
  const uint32_t t0 = P.task_off[blockIdx.x], t1 = P.task_off[blockIdx.x + 1];
  Ctx c;
  c.P = &P;
  c.S = S;
  c.ctl = ctl;
  c.ring = ring;
  c.it = 0;
  c.ctid = threadIdx.x - 32;
  c.warp = warp - 1;
  c.lane = threadIdx.x & 31;
  float* sv = reinterpret_cast<float*>(smem + P.off_sv);
  float* res = reinterpret_cast<float*>(smem + P.off_res);
  float* resid = reinterpret_cast<float*>(smem + P.off_resid);
  Task next{};
  if (t0 < t1) next = P.tasks[t0];
  for (uint32_t ti = t0; ti < t1; ++ti) {
    const Task t = next;
    if (ti + 1 < t1) next = P.tasks[ti + 1];  // the next descriptor loads while this task runs
    c.task_index = ti;
    c.first_stage = true;
    if (P.trace != nullptr && c.ctid == 0) P.trace[(size_t)ti * 4 + 3] = 0;
    trace_mark(c, 0);
    switch (t.type) {
      case T_QKV: task_qkv(c, t, sv, res); break;
      case T_ATTN: task_attn(c, t, sv); break;
      case T_OPROJ: task_oproj(c, t, sv, res, resid); break;
      case T_GATEUP: task_gateup(c, t, sv, res); break;
      case T_DOWN: task_down(c, t, sv, res, resid); break;
      case T_LMHEAD: task_lmhead(c, t, sv, res); break;
      default: break;
    }
    compute_sync();  // the next task reuses the shared vectors
    trace_mark(c, 2);
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
