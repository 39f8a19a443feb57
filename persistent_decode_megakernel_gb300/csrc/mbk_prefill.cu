// mbk_prefill.cu -- prefill: n tokens known in advance (a prompt) through the decoder in one pass per
// layer, appending their K/V rows to the cache.
//
// The MegaBake article ("Where it loses") measures its prefill path 3-21x slower than eager PyTorch:
// the megakernel is built for one token, and a prompt pushed through it re-reads every weight per
// token.  Here a prompt takes the dense road instead.  Its plain definition is n teacher-forced
// decode steps at positions p0 .. p0 + n - 1 (each token attends to the cache rows up to its own
// position), and the kernels below compute exactly that, layer by layer for all n tokens at once:
//
//   embed -> per layer: RMSNorm | Q/K/V GEMM (+bias) | RoPE + KV append | causal attention
//            | O GEMM (+= residual) | RMSNorm | gate/up GEMM | SiLU * up | down GEMM (+= residual)
//         -> final RMSNorm | LM-head GEMM (every token, or the last one only)
//
// GEMMs run on the 5th-generation tensor cores: one CTA per 128 x 128 output tile, a single thread
// issues tcgen05.mma (kind::f16, bf16 operands, fp32 accumulator in tensor memory), a second
// thread feeds a 2-stage ring of shared-memory tiles with TMA (two CTAs per SM) (cp.async.bulk.tensor, 128-byte
// swizzle), and the four warps read the accumulator back with tcgen05.ld for the epilogue.
//
// Precision.  The decoder keeps activations in fp32 (only the KV cache is bf16), so a GEMM input x
// is passed as two bf16 tensors hi = bf16(x) and lo = bf16(x - hi): W.x = W.hi + W.lo with exact
// products and fp32 accumulation, leaving a representation error of about 2^-17 |x| -- far below
// the one-bf16-ulp bar of the cache rows -- for twice the tensor work of a plain bf16 GEMM.
//
// Every wait on an mbarrier is bounded by the handle's timeout; on expiry the kernel records
// DS_TIMEOUT in the status word shared with the decode kernel, waits (again bounded) for its copies
// and tensor-core operations in flight, frees its tensor memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "mbk.h"
#include "mbk_prefill.h"

namespace mbk {
namespace {

// ------------------------------------------------------------------ GEMM tiling
constexpr int kBM = 128;                        // tokens per tile (tensor-memory lanes)
constexpr int kBN = 128;                        // outputs per tile (tensor-memory columns)
constexpr int kBK = 64;                         // K per stage: one 128-byte swizzle row of bf16
constexpr int kUK = 16;                         // K of one tcgen05.mma (kind::f16)
constexpr int kGemmStages = 2;                  // two CTAs per SM: one's epilogue overlaps the other's
                                                // loads and MMAs (4 stages and one CTA measured 3% slower)
constexpr int kTileBytes = kBM * kBK * 2;       // one operand tile: 16 KB (kBM == kBN)
constexpr int kStageBytesP = 3 * kTileBytes;    // A high part, A low part, B
constexpr int kGemmSmem = kGemmStages * kStageBytesP + 1024;  // + slack: swizzled tiles sit on 1 KB
constexpr int kGemmThreads = 128;
constexpr int kMaxSeg = 3;
static_assert(kBM == kBN, "one tile size for both operands");

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, bits 10-12 = 1), both K-major (bits 15, 16 = 0), N / 8 in bits 17-22, M / 16 in
// bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);

// One output segment of a GEMM: the rows of one weight matrix, written to columns col0.. of `out`.
struct GemmSeg {
  int n;                   // outputs (rows of the weight)
  int col0;                // first column in `out`
  int tile0;               // first tile (blockIdx.x) of the segment
  const uint16_t* bias;    // bf16 [n], or null
};

struct GemmArgs {
  CUtensorMap a_hi, a_lo;       // activations [M][K] bf16 (box 64 x 128, 128-byte swizzle, zero fill)
  CUtensorMap b[kMaxSeg];       // weights [n_s][K] bf16 (same box and swizzle)
  GemmSeg seg[kMaxSeg];
  int nseg;
  int M, K;
  float* out;                   // fp32 [M][ldo]
  int ldo;
  int accumulate;               // 0: out = acc (+ bias); 1: out += acc (residual stream)
  unsigned* status;
  unsigned* host_status;
  unsigned long long timeout_ns;
};

// ------------------------------------------------------------------ device helpers
__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint16_t to_bf16(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
// x as a pair of bf16 values: hi = bf16(x), lo = bf16(x - hi) (the difference is exact in fp32)
__device__ __forceinline__ void split_store(float v, uint16_t* hi, uint16_t* lo, size_t i) {
  const uint16_t h = to_bf16(v);
  hi[i] = h;
  lo[i] = to_bf16(v - bf16f(h));
}
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

__device__ __forceinline__ void mbar_init(uint64_t* b, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* b, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(saddr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

void __device__ record_timeout(unsigned* status, unsigned* host_status, unsigned detail) {
  if (atomicCAS(&status[0], 0u, (unsigned)DS_TIMEOUT) == 0u) {
    status[1] = blockIdx.x;
    status[2] = 0xFFFFFFFFu;  // not a task of the decode schedule
    status[3] = detail;
    if (host_status) {
      volatile unsigned* hs = host_status;
      hs[1] = blockIdx.x;
      hs[2] = 0xFFFFFFFFu;
      hs[3] = detail;
      __threadfence_system();
      hs[0] = (unsigned)DS_TIMEOUT;
    }
  }
}

// Waits until the phase of parity `parity` of barrier b has completed.  Gives up (false) after
// timeout_ns, or earlier once `abort` (if given) is set or the status word (if given) shows a failure.
__device__ __noinline__ bool mbar_wait(uint64_t* b, unsigned parity, const volatile unsigned* abort,
                                       const unsigned* status, unsigned long long timeout_ns) {
  unsigned long long t0 = 0ull;
  for (unsigned spins = 0;; ++spins) {
    if (mbar_test(b, parity)) return true;
    if ((spins & 63u) == 63u) {
      if ((abort != nullptr && *abort != 0u) || (status != nullptr && *(const volatile unsigned*)status != 0u))
        return false;
      const unsigned long long t = now_ns();
      if (t0 == 0ull)
        t0 = t;
      else if (t - t0 > timeout_ns)
        return false;
    }
  }
}

// 2-D TMA tile load (x = element column, y = row) into this CTA's shared memory.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          saddr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(saddr(bar))
      : "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with 128-byte swizzle:
// rows of 64 elements (128 bytes), groups of 8 rows 1024 bytes apart.  Fields: start address >> 4
// (bits 0-13), leading byte offset >> 4 (bits 16-29; unused by this layout, set to 1), stride byte
// offset >> 4 (bits 32-45), descriptor version 1 (bits 46-47), base offset 0 (the tile starts on
// a 1024-byte boundary), layout type 2 = 128-byte swizzle (bits 61-63).  A step of kUK elements
// along K inside the 128-byte row moves the start address by 32 bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t d = (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          tmem_d),
      "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}
// Arrives on `bar` once every tcgen05.mma this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's tensor-memory lane (warp w reads lanes 32w .. 32w+31).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------ the GEMM
// out[m][col0 + j] (=|+=) sum_k (A_hi + A_lo)[m][k] * W[j][k] (+ bias[j]) for one 128 x 128 tile.
// Warp 0 lane 0 issues the TMA loads, warp 1 lane 0 the MMAs, warp 2 owns the tensor memory, and all
// four warps run the epilogue (thread i holds output row m0 + i).
__global__ void __launch_bounds__(kGemmThreads, 2) prefill_gemm_kernel(const __grid_constant__ GemmArgs g) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full[kGemmStages];
  __shared__ __align__(8) uint64_t empty[kGemmStages];
  __shared__ __align__(8) uint64_t accum;
  __shared__ uint32_t tmem_slot;
  __shared__ unsigned failed;
  const uint32_t raw = saddr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);  // first 1024-byte boundary
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int s = 0;
  while (s + 1 < g.nseg && (int)blockIdx.x >= g.seg[s + 1].tile0) ++s;
  const int n0 = ((int)blockIdx.x - g.seg[s].tile0) * kBN;  // first weight row of the tile
  const int m0 = (int)blockIdx.y * kBM;
  const int kblocks = (g.K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGemmStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&accum, 1);
    failed = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&tmem_slot)),
                 "r"(kBN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile unsigned* abort = &failed;

  int issued = 0;  // k blocks whose loads were issued (thread 0)
  if (warp == 0 && lane == 0) {
    for (int kb = 0; kb < kblocks; ++kb) {
      const int st = kb % kGemmStages;
      if (kb >= kGemmStages && !mbar_wait(&empty[st], ((kb / kGemmStages) - 1) & 1, abort, g.status, g.timeout_ns)) {
        failed = 1u;
        break;
      }
      unsigned char* sa = smem + st * kStageBytesP;
      mbar_expect_tx(&full[st], kStageBytesP);
      tma_load_2d(sa, &g.a_hi, kb * kBK, m0, &full[st]);
      tma_load_2d(sa + kTileBytes, &g.a_lo, kb * kBK, m0, &full[st]);
      tma_load_2d(sa + 2 * kTileBytes, &g.b[s], kb * kBK, n0, &full[st]);
      issued = kb + 1;
    }
  } else if (warp == 1 && lane == 0) {
    for (int kb = 0; kb < kblocks; ++kb) {
      const int st = kb % kGemmStages;
      if (!mbar_wait(&full[st], (kb / kGemmStages) & 1, abort, g.status, g.timeout_ns)) {
        failed = 1u;
        break;
      }
      tc_fence_after();
      const uint32_t sa = saddr(smem + st * kStageBytesP);
#pragma unroll
      for (int k = 0; k < kBK / kUK; ++k) {
        const uint64_t bd = sw128_desc(sa + 2 * kTileBytes + k * kUK * 2);
        umma_bf16(tmem, sw128_desc(sa + k * kUK * 2), bd, (kb | k) != 0 ? 1u : 0u);
        umma_bf16(tmem, sw128_desc(sa + kTileBytes + k * kUK * 2), bd, 1u);
      }
      umma_commit(&empty[st]);  // the stage is free once these MMAs have read it
    }
    umma_commit(&accum);  // always: completes once every MMA issued above has finished
  }
  __syncwarp();
  __syncthreads();
  if (threadIdx.x == 0) {
    // every MMA issued above has finished (waited for even after a failure, so that no MMA still
    // writes the tensor memory when it is freed; bounded by time alone)
    if (!mbar_wait(&accum, 0, nullptr, nullptr, g.timeout_ns)) failed = 1u;
  }
  __syncthreads();
  tc_fence_after();
  const bool ok = failed == 0u;  // uniform: read after the barrier

  if (ok) {
    const int row = m0 + warp * 32 + lane;
    const GemmSeg& sg = g.seg[s];
#pragma unroll 1
    for (int c = 0; c < kBN; c += 32) {
      float v[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, v);  // every lane: .sync.aligned
      const int j0 = n0 + c;  // weight row of v[0]
      if (row < g.M && j0 < sg.n) {
        const int nv = min(32, sg.n - j0);
        float* o = g.out + (size_t)row * g.ldo + sg.col0 + j0;
        if (sg.bias != nullptr) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nv) v[j] += bf16f(sg.bias[j0 + j]);
        }
        if (nv == 32 && ((uintptr_t)o & 15u) == 0u) {
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            float4* p = reinterpret_cast<float4*>(o + j);
            float4 w = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            if (g.accumulate) {
              const float4 a = *p;
              w.x += a.x;
              w.y += a.y;
              w.z += a.z;
              w.w += a.w;
            }
            *p = w;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nv) o[j] = g.accumulate ? o[j] + v[j] : v[j];
        }
      }
    }
  } else if (threadIdx.x == 0) {
    record_timeout(g.status, g.host_status, 0xF0000000u | (unsigned)blockIdx.y);
    // copies still in flight land before the CTA leaves: the last stages this thread issued
    for (int kb = max(0, issued - kGemmStages); kb < issued; ++kb)
      mbar_wait(&full[kb % kGemmStages], (unsigned)(kb / kGemmStages) & 1u, nullptr, nullptr, g.timeout_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kBN) : "memory");
  }
}


// ------------------------------------------------------------------ elementwise kernels
// Sum of v over the block, returned to every thread (red: one float per warp).
__device__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red is free again after an earlier call
  if (lane == 0) red[warp] = v;
  __syncthreads();
  return warp_sum(lane < (int)(blockDim.x >> 5) ? red[lane] : 0.f);
}

// x[t][:] = E[tokens[t]][:] widened to fp32.
__global__ void embed_kernel(const uint16_t* E, const int32_t* tokens, int n, int H, float* x) {
  for (int t = blockIdx.x; t < n; t += gridDim.x) {
    const uint16_t* e = E + (size_t)tokens[t] * H;
    for (int i = threadIdx.x; i < H; i += blockDim.x) x[(size_t)t * H + i] = bf16f(e[i]);
  }
}

// Rows rows[r] (or r, when rows is null), r < n, of x [.][H]: xn = x / sqrt(mean(x^2) + eps) * gain,
// written to rows 0 .. n - 1 of the GEMM input pair (hi, lo) [.][H].
__global__ void norm_split_kernel(const float* x, int H, const uint16_t* gain, float eps, float inv_H,
                                  const int32_t* rows, int n, uint16_t* hi, uint16_t* lo) {
  __shared__ float red[32];
  for (int r = blockIdx.x; r < n; r += gridDim.x) {
    const float* xr = x + (size_t)(rows != nullptr ? rows[r] : r) * H;
    float ss = 0.f;
    for (int i = threadIdx.x; i < H; i += blockDim.x) ss = fmaf(xr[i], xr[i], ss);
    const float inv = rsqrtf(block_sum(ss, red) * inv_H + eps);
    for (int i = threadIdx.x; i < H; i += blockDim.x) split_store(xr[i] * inv * bf16f(gain[i]), hi, lo, (size_t)r * H + i);
  }
}

// The cache: contiguous (tables null, page_size = capacity) or a pool of pages found through one page
// table per sequence, tables[seq * max_pages + q] holding positions q * page_size ...
struct KvGeom {
  uint16_t* kv;
  const int32_t* tables;
  int max_pages;
  int page_size, page_shift, nkv, d;
  unsigned long long page_elems;
};
__device__ __forceinline__ const int32_t* table_of(const KvGeom& g, int seq) {
  return g.tables != nullptr ? g.tables + (size_t)seq * g.max_pages : nullptr;
}
// Element offset of cache row p of (layer, kv = 0 for K / 1 for V, KV head h) of the sequence whose
// page table is `table` (null: contiguous).
__device__ __forceinline__ size_t kv_index(const KvGeom& g, const int32_t* table, int layer, int kv, int h, int p) {
  size_t page = 0;
  int r = p;
  if (table != nullptr) {
    page = (size_t)(unsigned)table[p >> g.page_shift];
    r = p & (g.page_size - 1);
  }
  return page * g.page_elems + ((((size_t)layer * 2 + kv) * g.nkv + h) * g.page_size + r) * g.d;
}

// Token t (position pos[t] of sequence seq[t]): rotate its q and k heads in place (rotate-half pairs
// (i, i + d/2) by the angle of table row p), then store its K and V rows in its sequence's cache as
// bf16 (nearest even).
__global__ void rope_kv_kernel(float* qkv, int ld, int n, const int32_t* pos, const int32_t* seq, int nq,
                               const float2* rope, KvGeom g, int layer) {
  const int d = g.d, half = d / 2, nkv = g.nkv;
  for (int t = blockIdx.x; t < n; t += gridDim.x) {
    const int p = pos[t];
    const int32_t* table = table_of(g, seq[t]);
    float* row = qkv + (size_t)t * ld;
    for (int e = threadIdx.x; e < (nq + nkv) * half; e += blockDim.x) {
      const int hh = e / half, i = e - hh * half;  // heads: q heads, then k heads (contiguous)
      float* v = row + (size_t)hh * d;
      const float2 cs = rope[(size_t)p * half + i];
      const float a = v[i], b = v[i + half];
      v[i] = a * cs.x - b * cs.y;
      v[i + half] = b * cs.x + a * cs.y;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < 2 * nkv * d; e += blockDim.x) {
      const int sel = e / (nkv * d), rem = e - sel * nkv * d, h = rem / d, j = rem - h * d;
      g.kv[kv_index(g, table, layer, sel, h, p) + j] = to_bf16(row[(size_t)(nq + sel * nkv) * d + rem]);
    }
    __syncthreads();
  }
}

// h = silu(gate) * up for gu [n][2I] (gate columns 0..I-1, up columns I..2I-1), split into (hi, lo).
__global__ void silu_split_kernel(const float* gu, int n, int I, uint16_t* hi, uint16_t* lo) {
  const size_t total = (size_t)n * I;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const size_t t = e / I, c = e - t * I;
    const float gv = gu[t * 2 * I + c], uv = gu[t * 2 * I + I + c];
    split_store(gv / (1.0f + __expf(-gv)) * uv, hi, lo, e);
  }
}

// ------------------------------------------------------------------ causal attention
// One CTA: a tile of at most kAttnWarps tokens of one sequence at consecutive positions (one per warp;
// tiles are built on the host) and one KV head with its g query heads.
// Keys are staged 32 at a time in shared memory (one per lane for the scores; K rows padded to an
// odd number of words so that the lanes' rows fall in different banks), each warp keeps an online
// softmax per query head (running max, sum and output), and a token stops at its own position.
constexpr int kAttnWarps = 8;
constexpr int kAttnKeys = 32;
constexpr int kMaxGroup = 16;  // query heads per KV head (the schedule's limit too)

struct AttnArgs {
  const float* qkv;             // rotated q at columns [0, nq * d) of row t
  int ld;
  KvGeom kv;
  const int32_t* pos;           // [n] position of each token
  const int32_t* seq;           // [n] its sequence
  const int2* tiles;            // [blocks] (first token, tokens) of each tile
  int layer, nq, g;
  float scale_log2;             // 1/sqrt(d) * log2(e): scores in base 2
  uint16_t* o_hi;               // [n][nq * d] attention output, split for the O GEMM
  uint16_t* o_lo;
};

template <int D>
constexpr int attn_smem(int g) {
  return (kAttnKeys * (D / 2 + 1) + kAttnKeys * (D / 2)) * 4 + kAttnWarps * g * D * 4;
}

template <int D>
__global__ void __launch_bounds__(kAttnWarps * 32) prefill_attn_kernel(const AttnArgs a) {
  constexpr int KW = D / 2 + 1;   // K row stride in words (odd)
  constexpr int VW = D / 2;       // V row stride in words
  constexpr int DPL = D / 32;     // output elements per lane
  extern __shared__ __align__(16) uint32_t asm_words[];
  uint32_t* ks = asm_words;                                   // [32][KW]
  uint32_t* vs = ks + kAttnKeys * KW;                         // [32][VW] (16-byte aligned: KW*32 words is a multiple of 4)
  float* qs = reinterpret_cast<float*>(vs + kAttnKeys * VW);  // [warps][g][D]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.y, g = a.g;
  const int2 tile = a.tiles[blockIdx.x];
  const int t0 = tile.x, t = t0 + warp;
  const bool active = warp < tile.y;
  const int pos = active ? a.pos[t] : -1;
  const int last = a.pos[t0 + tile.y - 1];  // the tile's largest position (positions increase in a tile)
  const int32_t* table = table_of(a.kv, a.seq[t0]);
  float* q = qs + (size_t)warp * g * D;
  if (active)
    for (int e = lane; e < g * D; e += 32) q[e] = a.qkv[(size_t)t * a.ld + (size_t)kvh * g * D + e];
  __syncwarp();

  float m[kMaxGroup], l[kMaxGroup], o[kMaxGroup][DPL];
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int k = 0; k < DPL; ++k) o[h][k] = 0.f;
  }

  for (int c0 = 0; c0 <= last; c0 += kAttnKeys) {
    __syncthreads();  // the previous block of keys is no longer read
    for (int e = threadIdx.x; e < kAttnKeys * (D / 8); e += blockDim.x) {  // 16-byte pieces
      const int r = e / (D / 8), piece = e - r * (D / 8), p = c0 + r;
      uint4 kk = make_uint4(0u, 0u, 0u, 0u), vv = kk;
      if (p <= last) {
        kk = *reinterpret_cast<const uint4*>(a.kv.kv + kv_index(a.kv, table, a.layer, 0, kvh, p) + piece * 8);
        vv = *reinterpret_cast<const uint4*>(a.kv.kv + kv_index(a.kv, table, a.layer, 1, kvh, p) + piece * 8);
      }
      uint32_t* kd = ks + r * KW + piece * 4;
      kd[0] = kk.x;
      kd[1] = kk.y;
      kd[2] = kk.z;
      kd[3] = kk.w;
      *reinterpret_cast<uint4*>(vs + r * VW + piece * 4) = vv;
    }
    __syncthreads();
    if (!active || c0 > pos) continue;  // warp-uniform
    const bool valid = c0 + lane <= pos;
    const uint32_t* kr = ks + lane * KW;
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      if (h >= g) break;  // warp-uniform
      const float* qh = q + h * D;
      float sc = 0.f;
#pragma unroll 8
      for (int w = 0; w < D / 2; ++w) {
        const uint32_t kw = kr[w];
        sc = fmaf(qh[2 * w], bf16_lo(kw), sc);
        sc = fmaf(qh[2 * w + 1], bf16_hi(kw), sc);
      }
      sc = valid ? sc * a.scale_log2 : -INFINITY;
      const float mn = fmaxf(m[h], warp_max(sc));  // finite: key c0 <= pos is valid
      const float alpha = exp2f(m[h] - mn);        // 0 on the first block (m = -inf)
      const float pj = valid ? exp2f(sc - mn) : 0.f;
      l[h] = l[h] * alpha + warp_sum(pj);
      m[h] = mn;
#pragma unroll
      for (int k = 0; k < DPL; ++k) o[h][k] *= alpha;
#pragma unroll 4
      for (int j = 0; j < kAttnKeys; ++j) {
        const float pb = __shfl_sync(0xffffffffu, pj, j);
        const uint32_t* vr = vs + j * VW + lane * (DPL / 2);
#pragma unroll
        for (int k = 0; k < DPL / 2; ++k) {
          const uint32_t vw = vr[k];
          o[h][2 * k] = fmaf(pb, bf16_lo(vw), o[h][2 * k]);
          o[h][2 * k + 1] = fmaf(pb, bf16_hi(vw), o[h][2 * k + 1]);
        }
      }
    }
  }
  if (!active) return;
  const size_t qd = (size_t)a.nq * D;
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    if (h >= g) break;
    const float inv = 1.f / l[h];
#pragma unroll
    for (int k = 0; k < DPL; ++k)
      split_store(o[h][k] * inv, a.o_hi, a.o_lo, (size_t)t * qd + (size_t)(kvh * g + h) * D + lane * DPL + k);
  }
}


// ------------------------------------------------------------------ causal attention on the tensor cores
// Head dim 64, at most 8 query heads per KV head.  One CTA: a tile of at most 32 (g <= 4) or 16 tokens of
// one sequence and one KV head (mma_tile_tokens).  Its query rows are the (token, head) pairs, 16 per warp (row rho of the tile
// is token rho / g, head rho % g), so the g heads of a group share every K/V block.  Keys come 64 at a
// time, three buffers deep (one block barrier per block: a buffer refilled at block b was last read at
// block b - 2), by cp.async into shared tiles of 128-byte rows with the 16-byte chunk c of row r
// at chunk c ^ (r & 7) (the eight rows of a fragment load fall in eight bank groups); rows past the
// tile's last position are zero-filled.  Per warp and block, on mma.sync m16n8k16 (bf16 operands, fp32
// accumulation): S = Q K^T (B = K rows by ldmatrix) and O += P V (B = V rows by ldmatrix.trans), with S's
// accumulator fragments reused as P's A fragments; the fp32 queries and probabilities enter as bf16
// high/low pairs (x = hi + lo, relative error 2^-17 per operand; K and V are bf16 and enter exactly).
// An online softmax per row (running max and sum, scores in base 2); a row stops mattering past its
// token's position (masked to -inf).
constexpr int kMmaKeys = 64;
constexpr int kMmaBufs = 3;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ void hi_lo_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const float h0 = bf16f(to_bf16(x0)), h1 = bf16f(to_bf16(x1));
  hi = pack_bf16x2(h0, h1);
  lo = pack_bf16x2(x0 - h0, x1 - h1);
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// byte offset of 16-byte chunk c of row r in a [rows][128 B] swizzled tile
__device__ __forceinline__ uint32_t swz_off(int r, int c) { return (uint32_t)r * 128u + (uint32_t)((c ^ (r & 7)) << 4); }
// 16-byte asynchronous copy global -> shared; zero-filled when !ok (src is then not read)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(ok ? 16 : 0) : "memory");
}

__global__ void __launch_bounds__(kMaxGroup / 2 * 32) prefill_attn_mma_kernel(const AttnArgs a) {
  constexpr int D = 64;
  __shared__ __align__(1024) unsigned char kvs[kMmaBufs][2][kMmaKeys * 128];  // [buffer][K, V][64 rows of 128 B]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nthr = blockDim.x;
  const int gid = lane >> 2, tig = lane & 3;
  const int kvh = blockIdx.y, g = a.g;
  // a tile's work grows with its position and the tiles are in increasing position order: the
  // blocks take them from the last, so the longest start first and the short ones fill the tail
  const int2 tile = a.tiles[gridDim.x - 1 - blockIdx.x];
  const int t0 = tile.x, ntok = tile.y;
  const int last = a.pos[t0 + ntok - 1];  // the tile's largest position (positions increase in a tile)
  const int32_t* table = table_of(a.kv, a.seq[t0]);
  // this lane's rows gid and gid + 8 of the warp; rows past the tile (ntok * g) run as position `last`
  // with zero queries (finite, never written)
  int rtok[2], rhead[2], rpos[2];
  bool rok[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int rho = 16 * warp + gid + 8 * r;
    rok[r] = rho < ntok * g;
    rtok[r] = rok[r] ? rho / g : 0;
    rhead[r] = rok[r] ? rho - rtok[r] * g : 0;
    rpos[r] = rok[r] ? a.pos[t0 + rtok[r]] : last;
  }
  // A = Q: for k-step ks, a0 = (row gid, columns 16 ks + 2 tig, +1), a1 = (row gid + 8, same),
  // a2 = (row gid, +8), a3 = (row gid + 8, +8); high and low parts
  uint32_t qh[4][4], ql[4][4];
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = i & 1, col = 16 * ks + 2 * tig + ((i & 2) ? 8 : 0);
      float2 x = make_float2(0.f, 0.f);
      if (rok[r])
        x = *reinterpret_cast<const float2*>(a.qkv + (size_t)(t0 + rtok[r]) * a.ld + (size_t)(kvh * g + rhead[r]) * D + col);
      hi_lo_pair(x.x, x.y, qh[ks][i], ql[ks][i]);
    }
  }
  float o[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  const int nblk = last / kMmaKeys + 1;
  auto load = [&](int b) {  // key block b into buffer b % kMmaBufs: K rows, then V rows (16-byte pieces)
    const int p0 = b * kMmaKeys;
    const uint32_t base = saddr(&kvs[b % kMmaBufs][0][0]);
    for (int e = threadIdx.x; e < 2 * kMmaKeys * 8; e += nthr) {
      const int kv = e / (kMmaKeys * 8), r = (e >> 3) & (kMmaKeys - 1), c = e & 7, p = p0 + r;
      const bool ok = p <= last;
      const uint16_t* src = ok ? a.kv.kv + kv_index(a.kv, table, a.layer, kv, kvh, p) + c * 8 : a.kv.kv;
      cp_async16(base + (uint32_t)kv * (kMmaKeys * 128) + swz_off(r, c), src, ok);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  load(0);
  const int mi = lane >> 3, rr = lane & 7;
#pragma unroll 1
  for (int b = 0; b < nblk; ++b) {
    if (b + 1 < nblk) {
      load(b + 1);  // its buffer was last read in block b - 2, before every warp passed block b - 1's barrier
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();  // block b has landed for every thread's copies
    const int p0 = b * kMmaKeys;
    const uint32_t kb = saddr(&kvs[b % kMmaBufs][0][0]), vb = saddr(&kvs[b % kMmaBufs][1][0]);
    // S = Q K^T: n-tile n holds keys p0 + 8 n .. + 7; ldmatrix.x4 brings the B fragments of two n-tiles
    float sc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + swz_off(16 * np + ((mi >> 1) << 3) + rr, 2 * ks + (mi & 1)), b0, b1, b2, b3);
        mma_bf16_16816(sc[2 * np], qh[ks], b0, b1);
        mma_bf16_16816(sc[2 * np], ql[ks], b0, b1);
        mma_bf16_16816(sc[2 * np + 1], qh[ks], b2, b3);
        mma_bf16_16816(sc[2 * np + 1], ql[ks], b2, b3);
      }
    }
    // scale and mask: element k of n-tile n is (row gid + 8 (k >> 1), key p0 + 8 n + 2 tig + (k & 1))
    float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int key = p0 + 8 * n + 2 * tig + (k & 1);
        sc[n][k] = key <= rpos[k >> 1] ? sc[n][k] * a.scale_log2 : -INFINITY;
      }
      bm0 = fmaxf(bm0, fmaxf(sc[n][0], sc[n][1]));
      bm1 = fmaxf(bm1, fmaxf(sc[n][2], sc[n][3]));
    }
    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 1));
    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 2));
    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 1));
    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 2));
    // key 0 <= every row's position, so the first block gives every row a finite max; a later block
    // whose keys are all past a row's position leaves that row's max as it was
    const float nm0 = fmaxf(m0, bm0), nm1 = fmaxf(m1, bm1);
    const float al0 = exp2f(m0 - nm0), al1 = exp2f(m1 - nm1);
    m0 = nm0;
    m1 = nm1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      sc[n][0] = exp2f(sc[n][0] - m0);
      sc[n][1] = exp2f(sc[n][1] - m0);
      sc[n][2] = exp2f(sc[n][2] - m1);
      sc[n][3] = exp2f(sc[n][3] - m1);
      ps0 += sc[n][0] + sc[n][1];
      ps1 += sc[n][2] + sc[n][3];
      o[n][0] *= al0;
      o[n][1] *= al0;
      o[n][2] *= al1;
      o[n][3] *= al1;
    }
    l0 = fmaf(l0, al0, ps0);
    l1 = fmaf(l1, al1, ps1);
    // O += P V: k-step kk covers keys 16 kk .. + 15 (n-tiles 2 kk, 2 kk + 1 of S as P's A fragment)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t ph[4], pl[4];
      hi_lo_pair(sc[2 * kk][0], sc[2 * kk][1], ph[0], pl[0]);
      hi_lo_pair(sc[2 * kk][2], sc[2 * kk][3], ph[1], pl[1]);
      hi_lo_pair(sc[2 * kk + 1][0], sc[2 * kk + 1][1], ph[2], pl[2]);
      hi_lo_pair(sc[2 * kk + 1][2], sc[2 * kk + 1][3], ph[3], pl[3]);
#pragma unroll
      for (int dp = 0; dp < 4; ++dp) {  // dims 16 dp .. + 15: two n-tiles
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz_off(16 * kk + ((mi & 1) << 3) + rr, 2 * dp + (mi >> 1)), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], ph, b0, b1);
        mma_bf16_16816(o[2 * dp], pl, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], ph, b2, b3);
        mma_bf16_16816(o[2 * dp + 1], pl, b2, b3);
      }
    }
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const size_t qd = (size_t)a.nq * D;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (!rok[r]) continue;
    const float inv = 1.f / (r ? l1 : l0);
    const size_t base = (size_t)(t0 + rtok[r]) * qd + (size_t)(kvh * g + rhead[r]) * D + 2 * tig;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      split_store(o[n][2 * r] * inv, a.o_hi, a.o_lo, base + 8 * n);
      split_store(o[n][2 * r + 1] * inv, a.o_hi, a.o_lo, base + 8 * n + 1);
    }
  }
}

// ------------------------------------------------------------------ host side
// cuTensorMapEncodeTiled, looked up through the runtime (no link against the driver library).
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiled encoder() {
  static const EncodeTiled fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

// Tensor map of a bf16 matrix [rows][cols] (row-major, 16-byte aligned, cols a multiple of 8): tiles
// of 64 columns x 128 rows with 128-byte swizzle; reads outside the matrix return zeros.
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols) {
  const EncodeTiled enc = encoder();
  if (enc == nullptr || ((uintptr_t)base & 15u) != 0u || cols % 8 != 0 || rows == 0) return false;
  const cuuint64_t dim[2] = {cols, rows};
  const cuuint64_t stride[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBM};
  const cuuint32_t estride[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dim, stride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

enum WeightMap { WM_Q, WM_K, WM_V, WM_O, WM_GATE, WM_UP, WM_DOWN, WM_PER_LAYER };

struct Seg {
  const CUtensorMap* map;
  int n, col0;
  const uint16_t* bias;
};

cudaError_t gemm(const PrefillModel& m, const CUtensorMap& a_hi, const CUtensorMap& a_lo, const Seg* segs, int nseg,
                 int M, int K, float* out, int ldo, int accumulate, cudaStream_t st) {
  GemmArgs g;
  g.a_hi = a_hi;
  g.a_lo = a_lo;
  int tiles = 0;
  for (int i = 0; i < kMaxSeg; ++i) {
    if (i < nseg) {
      g.b[i] = *segs[i].map;
      g.seg[i] = GemmSeg{segs[i].n, segs[i].col0, tiles, segs[i].bias};
      tiles += (segs[i].n + kBN - 1) / kBN;
    } else {
      g.b[i] = *segs[0].map;
      g.seg[i] = GemmSeg{0, 0, 1 << 30, nullptr};
    }
  }
  g.nseg = nseg;
  g.M = M;
  g.K = K;
  g.out = out;
  g.ldo = ldo;
  g.accumulate = accumulate;
  g.status = m.status;
  g.host_status = m.host_status;
  g.timeout_ns = m.timeout_ns;
  prefill_gemm_kernel<<<dim3((unsigned)tiles, (unsigned)((M + kBM - 1) / kBM)), kGemmThreads, kGemmSmem, st>>>(g);
  return cudaGetLastError();
}

// The tensor-core attention takes head dim 64 with at most 8 query heads per KV head; its tiles hold
// 32 tokens up to 4 query heads per KV head and 16 beyond, so tokens x g heads make at most 8 warps of
// 16 rows.
bool mma_attention(const PrefillModel& m) { return m.d == 64 && m.nq / m.nkv <= kMaxGroup / 2; }
int mma_tile_tokens(const PrefillModel& m) { return m.nq / m.nkv <= 4 ? 32 : 16; }

cudaError_t attention(const PrefillModel& m, const PrefillState& s, const KvGeom& geom, int layer, int ntiles,
                      cudaStream_t st) {
  AttnArgs a;
  a.qkv = s.qkv;
  a.ld = (m.nq + 2 * m.nkv) * m.d;
  a.kv = geom;
  a.pos = s.pos;
  a.seq = s.seq;
  a.tiles = s.tiles;
  a.layer = layer;
  a.nq = m.nq;
  a.g = m.nq / m.nkv;
  a.scale_log2 = m.attn_scale * 1.4426950408889634f;
  a.o_hi = s.a_hi;
  a.o_lo = s.a_lo;
  const dim3 grid((unsigned)ntiles, (unsigned)m.nkv);
  if (mma_attention(m)) {
    // (tile tokens * g) / 16 warps
    prefill_attn_mma_kernel<<<grid, (unsigned)(mma_tile_tokens(m) * a.g / 16 * 32), 0, st>>>(a);
  } else if (m.d == 64)
    prefill_attn_kernel<64><<<grid, kAttnWarps * 32, attn_smem<64>(a.g), st>>>(a);
  else
    prefill_attn_kernel<128><<<grid, kAttnWarps * 32, attn_smem<128>(a.g), st>>>(a);
  return cudaGetLastError();
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

bool ensure_workspace(const PrefillModel& m, PrefillState& s, int n) {
  if (n <= s.cap) return true;
  prefill_free(s);
  const int cap = (n + kBM - 1) / kBM * kBM;
  const size_t qd = (size_t)m.nq * m.d, kvd = (size_t)m.nkv * m.d;
  const size_t kmax = std::max(std::max((size_t)m.H, (size_t)m.I), qd);
  const size_t b_x = round256(sizeof(float) * cap * m.H), b_qkv = round256(sizeof(float) * cap * (qd + 2 * kvd));
  const size_t b_gu = round256(sizeof(float) * cap * 2 * m.I), b_a = round256(2 * cap * kmax);
  const size_t b_int = round256(sizeof(int32_t) * 6 * (size_t)cap);  // tokens, pos, seq, rows, tiles (2 each)
  unsigned char* w = nullptr;
  if (cudaMalloc(reinterpret_cast<void**>(&w), b_x + b_qkv + b_gu + 2 * b_a + b_int) != cudaSuccess) return false;
  s.ws = w;
  s.x = reinterpret_cast<float*>(w);
  s.qkv = reinterpret_cast<float*>(w + b_x);
  s.gu = reinterpret_cast<float*>(w + b_x + b_qkv);
  s.a_hi = reinterpret_cast<uint16_t*>(w + b_x + b_qkv + b_gu);
  s.a_lo = reinterpret_cast<uint16_t*>(w + b_x + b_qkv + b_gu + b_a);
  s.tokens = reinterpret_cast<int32_t*>(w + b_x + b_qkv + b_gu + 2 * b_a);  // the int region: see pack_tokens
  s.pos = s.tokens + cap;
  s.seq = s.pos + cap;
  s.rows = s.seq + cap;
  s.tiles = reinterpret_cast<int2*>(s.rows + cap);
  s.cap = cap;
  return true;
}

// The int region of the workspace as one host image [tokens | pos | seq | rows | tiles] (cap entries
// each, tiles two): the positions and sequence of every token, the last token of every sequence, and
// the attention tiles (at most tile_tokens consecutive tokens of one sequence).  Returns the tile count.
int pack_tokens(const PrefillBatch& b, const int32_t* tokens, int n, int cap, int tile_tokens, std::vector<int32_t>& img) {
  img.assign((size_t)6 * cap, 0);
  int32_t* tok = img.data();
  int32_t* pos = tok + cap;
  int32_t* seq = pos + cap;
  int32_t* rows = seq + cap;
  int32_t* tiles = rows + cap;
  int t = 0, nt = 0;
  for (int q = 0; q < b.n_seq; ++q) {
    for (int i = 0; i < b.counts[q]; ++i, ++t) {
      tok[t] = tokens[t];
      pos[t] = b.starts[q] + i;
      seq[t] = q;
      if (i % tile_tokens == 0) {
        tiles[2 * nt] = t;
        tiles[2 * nt + 1] = std::min(tile_tokens, b.counts[q] - i);
        ++nt;
      }
    }
    rows[q] = t - 1;
  }
  (void)n;
  return nt;
}

}  // namespace

bool make_kv_tile_map(CUtensorMap* map, const void* kv, uint64_t rows, uint32_t box_rows) {
  const EncodeTiled enc = encoder();
  if (enc == nullptr || ((uintptr_t)kv & 15u) != 0u || rows == 0 || rows > 0x7fffffffull || box_rows == 0 || box_rows > 256)
    return false;
  const cuuint64_t dim[2] = {64, rows};
  const cuuint64_t stride[1] = {128};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estride[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kv), dim, stride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void prefill_free(PrefillState& s) {
  if (s.ws != nullptr) cudaFree(s.ws);
  s.ws = nullptr;
  s.x = s.qkv = s.gu = nullptr;
  s.a_hi = s.a_lo = nullptr;
  s.tokens = s.pos = s.seq = s.rows = nullptr;
  s.tiles = nullptr;
  s.cap = 0;
  if (s.tables != nullptr) cudaFree(s.tables);
  s.tables = nullptr;
  s.tables_cap = 0;
}

int prefill_run(const PrefillModel& m, PrefillState& s, const int32_t* tokens_host, int n, const PrefillBatch& batch,
                float* logits, int mode, cudaStream_t st, const float* inject) {
  if (encoder() == nullptr) return MBK_ERR_UNSUPPORTED;
  const int qd = m.nq * m.d, kvd = m.nkv * m.d, qkvd = qd + 2 * kvd;
  if (!s.smem_set) {
    if (cudaFuncSetAttribute(prefill_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem) != cudaSuccess ||
        cudaFuncSetAttribute(prefill_attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             attn_smem<64>(kMaxGroup)) != cudaSuccess ||
        cudaFuncSetAttribute(prefill_attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             attn_smem<128>(kMaxGroup)) != cudaSuccess)
      return MBK_ERR_CUDA;
    s.smem_set = true;
  }
  if (s.wmaps.empty()) {  // the weights do not move for the handle's lifetime
    std::vector<CUtensorMap> maps((size_t)m.L * WM_PER_LAYER + 1);
    for (int l = 0; l < m.L; ++l) {
      const LayerW& w = m.layers[l];
      CUtensorMap* lm = &maps[(size_t)l * WM_PER_LAYER];
      const bool ok = make_map(&lm[WM_Q], w.w[LW_Q], qd, m.H) && make_map(&lm[WM_K], w.w[LW_K], kvd, m.H) &&
                      make_map(&lm[WM_V], w.w[LW_V], kvd, m.H) && make_map(&lm[WM_O], w.w[LW_O], m.H, qd) &&
                      make_map(&lm[WM_GATE], w.w[LW_GATE], m.I, m.H) && make_map(&lm[WM_UP], w.w[LW_UP], m.I, m.H) &&
                      make_map(&lm[WM_DOWN], w.w[LW_DOWN], m.H, m.I);
      if (!ok) return MBK_ERR_UNSUPPORTED;
    }
    if (!make_map(&maps[(size_t)m.L * WM_PER_LAYER], m.embed, m.V, m.H)) return MBK_ERR_UNSUPPORTED;
    s.wmaps.swap(maps);
  }
  if (!ensure_workspace(m, s, n)) return MBK_ERR_NOMEM;
  // the GEMM inputs: one pair of buffers, seen with the row length of each use
  CUtensorMap ah_H, al_H, ah_q, al_q, ah_I, al_I;
  if (!make_map(&ah_H, s.a_hi, n, m.H) || !make_map(&al_H, s.a_lo, n, m.H) || !make_map(&ah_q, s.a_hi, n, qd) ||
      !make_map(&al_q, s.a_lo, n, qd) || !make_map(&ah_I, s.a_hi, n, m.I) || !make_map(&al_I, s.a_lo, n, m.I))
    return MBK_ERR_UNSUPPORTED;
  std::vector<int32_t> img;
  const int ntiles = pack_tokens(batch, tokens_host, n, s.cap, mma_attention(m) ? mma_tile_tokens(m) : kAttnWarps, img);
  if (cudaMemcpyAsync(s.tokens, img.data(), sizeof(int32_t) * img.size(), cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MBK_ERR_CUDA;
  KvGeom geom{m.kv, m.page_table, 0, m.page_size, m.page_shift, m.nkv, m.d, m.page_elems};
  if (batch.tables != nullptr) {  // the batch's own page tables
    const size_t ne = (size_t)batch.n_seq * batch.max_pages;
    if (ne > s.tables_cap) {
      if (s.tables != nullptr) cudaFree(s.tables);
      s.tables = nullptr;
      s.tables_cap = 0;
      if (cudaMalloc(reinterpret_cast<void**>(&s.tables), sizeof(int32_t) * ne) != cudaSuccess) return MBK_ERR_NOMEM;
      s.tables_cap = ne;
    }
    if (cudaMemcpyAsync(s.tables, batch.tables, sizeof(int32_t) * ne, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return MBK_ERR_CUDA;
    geom.tables = s.tables;
    geom.max_pages = batch.max_pages;
  }

  const unsigned rows_grid = (unsigned)std::min(n, 4096);
  bool ok = true;
  auto ck = [&](cudaError_t e) { ok = ok && e == cudaSuccess; };
  embed_kernel<<<rows_grid, 256, 0, st>>>(m.embed, s.tokens, n, m.H, s.x);
  ck(cudaGetLastError());
  for (int l = 0; ok && l < m.L; ++l) {
    const LayerW& w = m.layers[l];
    const CUtensorMap* lm = &s.wmaps[(size_t)l * WM_PER_LAYER];
    if (inject != nullptr && l >= 1)
      ck(cudaMemcpyAsync(s.x, inject + (size_t)l * n * m.H, sizeof(float) * (size_t)n * m.H, cudaMemcpyDeviceToDevice, st));
    // attention sublayer
    norm_split_kernel<<<rows_grid, 256, 0, st>>>(s.x, m.H, w.w[LW_ATTN_NORM], m.eps, m.inv_H, nullptr, n, s.a_hi,
                                                 s.a_lo);
    ck(cudaGetLastError());
    const Seg qkv[3] = {{&lm[WM_Q], qd, 0, m.qkv_bias ? w.w[LW_BQ] : nullptr},
                        {&lm[WM_K], kvd, qd, m.qkv_bias ? w.w[LW_BK] : nullptr},
                        {&lm[WM_V], kvd, qd + kvd, m.qkv_bias ? w.w[LW_BV] : nullptr}};
    ck(gemm(m, ah_H, al_H, qkv, 3, n, m.H, s.qkv, qkvd, 0, st));
    rope_kv_kernel<<<rows_grid, 256, 0, st>>>(s.qkv, qkvd, n, s.pos, s.seq, m.nq, m.rope, geom, l);
    ck(cudaGetLastError());
    ck(attention(m, s, geom, l, ntiles, st));
    const Seg o[1] = {{&lm[WM_O], m.H, 0, nullptr}};
    ck(gemm(m, ah_q, al_q, o, 1, n, qd, s.x, m.H, 1, st));
    // MLP sublayer
    norm_split_kernel<<<rows_grid, 256, 0, st>>>(s.x, m.H, w.w[LW_MLP_NORM], m.eps, m.inv_H, nullptr, n, s.a_hi,
                                                 s.a_lo);
    ck(cudaGetLastError());
    const Seg gu[2] = {{&lm[WM_GATE], m.I, 0, nullptr}, {&lm[WM_UP], m.I, m.I, nullptr}};
    ck(gemm(m, ah_H, al_H, gu, 2, n, m.H, s.gu, 2 * m.I, 0, st));
    silu_split_kernel<<<1216, 256, 0, st>>>(s.gu, n, m.I, s.a_hi, s.a_lo);
    ck(cudaGetLastError());
    const Seg down[1] = {{&lm[WM_DOWN], m.H, 0, nullptr}};
    ck(gemm(m, ah_I, al_I, down, 1, n, m.I, s.x, m.H, 1, st));
  }
  if (ok && mode != PL_NONE) {
    // final norm of every row (or of the last token of each sequence, into rows 0 .., n_seq - 1),
    // then the tied LM head
    const int rows = mode == PL_ALL ? n : batch.n_seq;
    norm_split_kernel<<<std::min(rows, 4096), 256, 0, st>>>(s.x, m.H, m.final_norm, m.eps, m.inv_H,
                                                            mode == PL_ALL ? nullptr : s.rows, rows, s.a_hi, s.a_lo);
    ck(cudaGetLastError());
    const Seg lmh[1] = {{&s.wmaps[(size_t)m.L * WM_PER_LAYER], m.V, 0, nullptr}};
    ck(gemm(m, ah_H, al_H, lmh, 1, rows, m.H, logits, m.V, 0, st));
  }
  return ok ? MBK_OK : MBK_ERR_CUDA;
}

}  // namespace mbk
