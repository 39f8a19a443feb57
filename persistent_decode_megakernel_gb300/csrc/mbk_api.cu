// mbk_api.cu -- the C ABI (include/mbk.h): handle creation, argument checks, the per-step launch.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/mbk.h"
#include "mbk_args.h"
#include "mbk_device.h"
#include "mbk_prefill.h"
#include "mbk_sched.h"

namespace mbk {
const void* decode_kernel_ptr(bool greedy, bool fp8, bool mma);
cudaError_t launch_quantize_fp8(const uint16_t* w, int rows, int cols, uint8_t* q, float* s, cudaStream_t st);
cudaError_t launch_rope_table(float2* out, int C, int d, double theta, cudaStream_t st);
cudaError_t launch_kv_fill(const KernelParams& kp, int layer, const float* k_raw, const float* v_raw, int p0, int n,
                           cudaStream_t st);
}  // namespace mbk

using namespace mbk;

struct mbk_handle {
  int device = 0;
  mbk_config cfg{};
  Plan plan;
  KernelParams kp{};
  unsigned tag = 0;           // last step's tag
  int grid = 0;
  // device allocations
  Task* d_tasks = nullptr;
  uint32_t* d_task_off = nullptr;
  Chunk* d_chunks = nullptr;
  uint32_t* d_chunk_off = nullptr;
  LayerW* d_layers = nullptr;
  float2* d_rope = nullptr;
  unsigned long long* d_words = nullptr;
  unsigned* d_status = nullptr;
  unsigned* h_status = nullptr;  // mapped pinned host memory
  float* d_logits_tmp = nullptr; // for mbk_decode_step_host
  int32_t* d_tokens = nullptr;    // [kv_capacity] token ids of a multi-step call
  unsigned long long* d_sync = nullptr;  // inter-step counter of multi-step launches
  unsigned long long sync_count = 0;     // its value after the last launch
  unsigned long long* d_amax = nullptr;  // [kv_capacity] greedy decoding: argmax key of each step
  unsigned* d_amax_done = nullptr;       // [kv_capacity] ... and the LM-head tasks that contributed
  unsigned long long* d_tokword = nullptr;  // ... and the argmax as a tagged word for the next step
  // paged KV cache (mbk_create_paged): pool size, page size and the device page table
  bool paged = false;
  int num_pages = 0, page_size = 0, max_pages = 0;
  int32_t* d_page_table = nullptr;
  // FP8 weights (MBK_WEIGHTS_FP8): the library's E4M3 copies and their per-row scales
  uint8_t* d_fp8 = nullptr;
  float* d_wscale = nullptr;
  int mapped = 0;  // positions [0, mapped) have cache rows: kv_capacity, or what the page table covers
  // prefill (mbk_prefill): the caller's bf16 weights (an FP8 handle decodes from its copies) and the
  // workspace and tensor maps of the tensor-core path
  std::vector<LayerW> bf16_layers;
  PrefillState prefill;
  float* d_prefill_inject = nullptr;  // mbk_debug_prefill_inject: [L][n][H] layer inputs of the next prefill
  int prefill_inject_n = 0;           // its token count (0: not armed)
  size_t prefill_inject_cap = 0;      // floats allocated
  unsigned long long* d_trace = nullptr;
  unsigned long long* d_inject = nullptr;
  bool inject_armed = false;
  CUtensorMap kvmap{};  // the KV cache as swizzled tiles (tensor-core attention; unused otherwise)
  int last_token = 0;
  int sticky = MBK_OK;
};

namespace {

int lm_task_count(const Plan& p) {
  int n = 0;
  for (const Task& t : p.tasks) n += t.type == T_LMHEAD ? 1 : 0;
  return n;
}

void free_all(mbk_handle* h) {
  cudaFree(h->d_tasks);
  cudaFree(h->d_task_off);
  cudaFree(h->d_chunks);
  cudaFree(h->d_chunk_off);
  cudaFree(h->d_layers);
  cudaFree(h->d_rope);
  cudaFree(h->d_words);
  cudaFree(h->d_status);
  cudaFree(h->d_logits_tmp);
  cudaFree(h->d_tokens);
  cudaFree(h->d_sync);
  cudaFree(h->d_amax);
  cudaFree(h->d_amax_done);
  cudaFree(h->d_tokword);
  cudaFree(h->d_page_table);
  cudaFree(h->d_fp8);
  cudaFree(h->d_wscale);
  prefill_free(h->prefill);
  cudaFree(h->d_prefill_inject);
  cudaFree(h->d_trace);
  cudaFree(h->d_inject);
  if (h->h_status) cudaFreeHost(h->h_status);
}

int sticky_status(mbk_handle* h) {
  if (h->sticky != MBK_OK) return h->sticky;
  if (h->h_status && *(volatile unsigned*)h->h_status != 0u) h->sticky = MBK_ERR_TIMEOUT;
  return h->sticky;
}

}  // namespace

extern "C" {

const char* mbk_error_string(int code) {
  switch (code) {
    case MBK_OK: return "ok";
    case MBK_ERR_INVALID_ARG: return "invalid argument";
    case MBK_ERR_UNSUPPORTED: return "unsupported device or configuration";
    case MBK_ERR_CUDA: return "CUDA runtime error";
    case MBK_ERR_TIMEOUT: return "a device-side wait timed out";
    case MBK_ERR_NOMEM: return "out of memory";
    case MBK_ERR_STATE: return "not possible in the present state";
    default: return "unknown error";
  }
}

int mbk_plan_check(const mbk_config* cfg, int num_sms, mbk_plan_info* info) {
  if (!cfg || !info || num_sms <= 0) return MBK_ERR_INVALID_ARG;
  if (config_check(cfg) != MBK_OK) return MBK_ERR_INVALID_ARG;
  PlanShape s = shape_of(*cfg);
  WeightAddrs w = fake_weight_addrs(s);
  Plan p;
  PlanOptions opt;
  opt.max_tasks_per_op = env_int("MBK_MAX_TASKS_PER_OP", 0);
  opt.fuse_attention = env_int("MBK_FUSE_ATTENTION", -1);
  opt.attn_mma = env_int("MBK_ATTN_MMA", 1);
  opt.attn_split = env_int("MBK_ATTN_SPLIT", 0);
  opt.combine_tasks = env_int("MBK_COMBINE_TASKS", 0);
  std::string err = build_plan(s, w, num_sms, opt, &p);
  if (!err.empty()) return MBK_ERR_STATE;
  info->num_ctas = p.num_ctas;
  info->num_tasks = (int)p.tasks.size();
  info->num_chunks = (int)p.chunks.size();
  info->stage_bytes = kStageBytes;
  info->num_stages = p.num_stages;
  info->attn_splits = p.nsplit;
  info->weight_bytes = p.weight_bytes;
  info->max_cta_bytes = p.max_cta_bytes;
  info->act_words = (int64_t)p.act_words;
  info->smem_bytes = p.smem_bytes;
  info->combine_group = p.combine_group;
  info->attn_mma = p.attn_mma ? 1 : 0;
  return MBK_OK;
}

namespace {
// The KV-cache layout of a handle: contiguous (num_pages == 0) or a pool of num_pages pages.
struct KvLayout {
  int num_pages = 0, page_size = 0;
};
int create_impl(const mbk_config* cfg, const mbk_weights* weights, void* kv_cache, KvLayout kvl, int device,
                mbk_handle** out);
}  // namespace

int mbk_create(const mbk_config* cfg, const mbk_weights* weights, void* kv_cache, int device, mbk_handle** out) {
  return create_impl(cfg, weights, kv_cache, KvLayout{}, device, out);
}

int mbk_create_paged(const mbk_config* cfg, const mbk_weights* weights, void* kv_pool, int32_t num_pages,
                     int32_t page_size, int device, mbk_handle** out) {
  if (!out) return MBK_ERR_INVALID_ARG;
  *out = nullptr;
  if (config_check(cfg) != MBK_OK || num_pages < 1 || page_size < 32 || (page_size & (page_size - 1)) != 0 ||
      page_size > cfg->kv_capacity || (cfg->kv_capacity + page_size - 1) / page_size > kMaxPages)
    return MBK_ERR_INVALID_ARG;
  KvLayout kvl;
  kvl.num_pages = num_pages;
  kvl.page_size = page_size;
  return create_impl(cfg, weights, kv_pool, kvl, device, out);
}

int mbk_quantize_fp8(const void* w, int32_t rows, int32_t cols, void* q, float* s, void* stream) {
  if (!w || !q || !s || rows < 1 || cols < 2 || (cols & 1)) return MBK_ERR_INVALID_ARG;
  return launch_quantize_fp8(reinterpret_cast<const uint16_t*>(w), rows, cols, reinterpret_cast<uint8_t*>(q), s,
                             (cudaStream_t)stream) == cudaSuccess ? MBK_OK : MBK_ERR_CUDA;
}

int mbk_set_page_table(mbk_handle* h, const int32_t* pages, int32_t n_pages, void* stream) {
  if (!h || !pages || !h->paged || n_pages < 1 || n_pages > h->max_pages) return MBK_ERR_INVALID_ARG;
  std::vector<char> used(h->num_pages, 0);
  for (int32_t i = 0; i < n_pages; ++i) {
    if (pages[i] < 0 || pages[i] >= h->num_pages || used[pages[i]]) return MBK_ERR_INVALID_ARG;
    used[pages[i]] = 1;
  }
  if (cudaSetDevice(h->device) != cudaSuccess) return MBK_ERR_CUDA;
  if (cudaMemcpyAsync(h->d_page_table, pages, sizeof(int32_t) * (size_t)n_pages, cudaMemcpyHostToDevice,
                      (cudaStream_t)stream) != cudaSuccess)
    return MBK_ERR_CUDA;
  h->mapped = std::min(h->cfg.kv_capacity, n_pages * h->page_size);
  return MBK_OK;
}

namespace {
int create_impl(const mbk_config* cfg, const mbk_weights* weights, void* kv_cache, KvLayout kvl, int device,
                mbk_handle** out) {
  if (!out) return MBK_ERR_INVALID_ARG;
  *out = nullptr;
  WeightAddrs wa;
  if (gather_weights(cfg, weights, kv_cache, &wa) != MBK_OK) return MBK_ERR_INVALID_ARG;
  const PlanShape s = shape_of(*cfg);

  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return MBK_ERR_UNSUPPORTED;
  if (cudaSetDevice(device) != cudaSuccess) return MBK_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return MBK_ERR_CUDA;
  if (prop.major != 10) return MBK_ERR_UNSUPPORTED;  // built for sm_103a (Blackwell data-center)
  int coop = 0, smem_optin = 0;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device);
  cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  if (!coop) return MBK_ERR_UNSUPPORTED;

  mbk_handle* h = new (std::nothrow) mbk_handle();
  if (!h) return MBK_ERR_NOMEM;
  h->device = device;
  h->cfg = *cfg;
  h->bf16_layers.resize(s.L);
  for (int l = 0; l < s.L; ++l)
    for (int k = 0; k < W_NSLOTS; ++k) h->bf16_layers[l].w[k] = reinterpret_cast<const uint16_t*>(wa.layers[l][k]);
  h->paged = kvl.num_pages > 0;
  h->num_pages = kvl.num_pages;
  h->page_size = kvl.page_size;
  h->max_pages = h->paged ? (cfg->kv_capacity + kvl.page_size - 1) / kvl.page_size : 0;
  h->mapped = h->paged ? 0 : cfg->kv_capacity;
  // FP8 weights: the library's E4M3 copies (each matrix 256-byte aligned) and their row scales, per
  // layer [q|k|v rows][Wo rows][gate rows][up rows][Wd rows], then the LM head's V rows
  int wscale_layer = 0;
  if (s.wb == 1) {
    const int qd = s.nq * s.d, kvd = s.nkv * s.d;
    const int slot_of[7] = {W_Q, W_K, W_V, W_O, W_GATE, W_UP, W_DOWN};
    const int rows_of[7] = {qd, kvd, kvd, s.H, s.I, s.I, s.H};
    const int cols_of[7] = {s.H, s.H, s.H, qd, s.H, s.H, s.I};
    int soff[7];
    for (int m = 0, o = 0; m < 7; ++m) {
      soff[m] = o;
      o += rows_of[m];
      wscale_layer = o;
    }
    auto align = [](size_t b) { return (b + 255) / 256 * 256; };
    size_t bytes = 0;
    std::vector<size_t> off((size_t)s.L * 7);
    for (int l = 0; l < s.L; ++l)
      for (int m = 0; m < 7; ++m) {
        off[(size_t)l * 7 + m] = bytes;
        bytes += align((size_t)rows_of[m] * cols_of[m]);
      }
    const size_t lm_off = bytes;
    bytes += align((size_t)s.V * s.H);
    bool ok = cudaMalloc(&h->d_fp8, bytes) == cudaSuccess &&
              cudaMalloc(&h->d_wscale, sizeof(float) * ((size_t)wscale_layer * s.L + s.V)) == cudaSuccess;
    for (int l = 0; ok && l < s.L; ++l)
      for (int m = 0; ok && m < 7; ++m) {
        uint8_t* q = h->d_fp8 + off[(size_t)l * 7 + m];
        ok = launch_quantize_fp8(reinterpret_cast<const uint16_t*>(wa.layers[l][slot_of[m]]), rows_of[m], cols_of[m], q,
                                 h->d_wscale + (size_t)l * wscale_layer + soff[m], 0) == cudaSuccess;
        wa.layers[l][slot_of[m]] = (uint64_t)(uintptr_t)q;
      }
    if (ok)
      ok = launch_quantize_fp8(reinterpret_cast<const uint16_t*>(wa.embed), s.V, s.H, h->d_fp8 + lm_off,
                               h->d_wscale + (size_t)wscale_layer * s.L, 0) == cudaSuccess;
    wa.lm_head = (uint64_t)(uintptr_t)(h->d_fp8 + lm_off);
    if (!ok || cudaDeviceSynchronize() != cudaSuccess) {
      free_all(h);
      delete h;
      return MBK_ERR_CUDA;
    }
  }
  PlanOptions opt;
  opt.smem_limit = smem_optin;
  opt.max_tasks_per_op = env_int("MBK_MAX_TASKS_PER_OP", 0);
  opt.fuse_attention = env_int("MBK_FUSE_ATTENTION", -1);
  opt.attn_mma = env_int("MBK_ATTN_MMA", 1);
  opt.attn_split = env_int("MBK_ATTN_SPLIT", 0);
  opt.combine_tasks = env_int("MBK_COMBINE_TASKS", 0);
  std::string err = build_plan(s, wa, prop.multiProcessorCount, opt, &h->plan);
  if (!err.empty()) {
    free_all(h);
    delete h;
    return MBK_ERR_UNSUPPORTED;
  }
  // Fault injection for tests (host side only): drop one task, so whoever reads its outputs waits
  // until its bounded timeout and the step reports MBK_ERR_TIMEOUT.
  const int drop = env_int("MBK_DEBUG_DROP_TASK", -1);
  if (drop >= 0 && drop < (int)h->plan.tasks.size()) {
    Plan& pl = h->plan;
    const Task victim = pl.tasks[drop];
    pl.tasks.erase(pl.tasks.begin() + drop);
    for (uint32_t& o : pl.task_off)
      if (o > (uint32_t)drop) --o;
    pl.chunks.erase(pl.chunks.begin() + victim.chunk0, pl.chunks.begin() + victim.chunk0 + victim.nchunks);
    for (uint32_t& o : pl.chunk_off)
      if (o > victim.chunk0) o -= victim.nchunks;
    for (Task& t : pl.tasks)
      if (t.chunk0 > victim.chunk0) t.chunk0 -= victim.nchunks;
  }
  const Plan& p = h->plan;
  h->grid = p.num_ctas;

  for (int k = 0; k < 4; ++k) {  // teacher-forced and greedy, tensor-core and CUDA-core attention
    const bool greedy = (k & 1) != 0, mma = (k & 2) != 0;
    const void* kfn = decode_kernel_ptr(greedy, s.wb == 1, mma);
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin) != cudaSuccess) {
      free_all(h);
      delete h;
      return MBK_ERR_CUDA;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kfn, kThreads, p.smem_bytes) != cudaSuccess || per_sm < 1) {
      free_all(h);
      delete h;
      return MBK_ERR_UNSUPPORTED;
    }
  }

  int rc = MBK_OK;
  auto ck = [&](cudaError_t e) {
    if (e != cudaSuccess && rc == MBK_OK) rc = (e == cudaErrorMemoryAllocation) ? MBK_ERR_NOMEM : MBK_ERR_CUDA;
    return e == cudaSuccess;
  };
  std::vector<LayerW> lw(s.L);
  for (int l = 0; l < s.L; ++l)
    for (int k = 0; k < W_NSLOTS; ++k) lw[l].w[k] = reinterpret_cast<const uint16_t*>(wa.layers[l][k]);
  const size_t rope_n = (size_t)s.C * (s.d / 2);
  if (ck(cudaMalloc(&h->d_tasks, sizeof(Task) * p.tasks.size())) &&
      ck(cudaMalloc(&h->d_task_off, sizeof(uint32_t) * p.task_off.size())) &&
      ck(cudaMalloc(&h->d_chunks, sizeof(Chunk) * std::max<size_t>(1, p.chunks.size()))) &&
      ck(cudaMalloc(&h->d_chunk_off, sizeof(uint32_t) * p.chunk_off.size())) &&
      ck(cudaMalloc(&h->d_layers, sizeof(LayerW) * s.L)) && ck(cudaMalloc(&h->d_rope, sizeof(float2) * rope_n)) &&
      ck(cudaMalloc(&h->d_words, sizeof(unsigned long long) * p.act_words)) &&
      ck(cudaMalloc(&h->d_status, 16)) && ck(cudaMalloc(&h->d_logits_tmp, sizeof(float) * s.V)) &&
      ck(cudaMalloc(&h->d_tokens, sizeof(int32_t) * s.C)) && ck(cudaMalloc(&h->d_sync, 8)) &&
      ck(cudaMalloc(&h->d_amax, sizeof(unsigned long long) * s.C)) && ck(cudaMalloc(&h->d_amax_done, sizeof(unsigned) * s.C)) &&
      ck(cudaMalloc(&h->d_tokword, 8)) && ck(cudaMemset(h->d_tokword, 0, 8)) &&
      (!h->paged || (ck(cudaMalloc(&h->d_page_table, sizeof(int32_t) * h->max_pages)) &&
                     ck(cudaMemset(h->d_page_table, 0, sizeof(int32_t) * h->max_pages)))) &&
      ck(cudaMemset(h->d_sync, 0, 8)) &&
      ck(cudaHostAlloc(&h->h_status, 16, cudaHostAllocMapped))) {
    ck(cudaMemcpy(h->d_tasks, p.tasks.data(), sizeof(Task) * p.tasks.size(), cudaMemcpyHostToDevice));
    ck(cudaMemcpy(h->d_task_off, p.task_off.data(), sizeof(uint32_t) * p.task_off.size(), cudaMemcpyHostToDevice));
    if (!p.chunks.empty()) ck(cudaMemcpy(h->d_chunks, p.chunks.data(), sizeof(Chunk) * p.chunks.size(), cudaMemcpyHostToDevice));
    ck(cudaMemcpy(h->d_chunk_off, p.chunk_off.data(), sizeof(uint32_t) * p.chunk_off.size(), cudaMemcpyHostToDevice));
    ck(cudaMemcpy(h->d_layers, lw.data(), sizeof(LayerW) * s.L, cudaMemcpyHostToDevice));
    ck(cudaMemset(h->d_words, 0, sizeof(unsigned long long) * p.act_words));
    ck(cudaMemset(h->d_status, 0, 16));
    memset(h->h_status, 0, 16);
    ck(launch_rope_table(h->d_rope, s.C, s.d, cfg->rope_theta, 0));
    ck(cudaDeviceSynchronize());
  }
  unsigned* h_status_dev = nullptr;
  if (rc == MBK_OK) ck(cudaHostGetDevicePointer((void**)&h_status_dev, h->h_status, 0));
  if (rc != MBK_OK) {
    free_all(h);
    delete h;
    return rc;
  }

  KernelParams& kp = h->kp;
  kp.L = s.L;
  kp.H = s.H;
  kp.I = s.I;
  kp.nq = s.nq;
  kp.nkv = s.nkv;
  kp.d = s.d;
  kp.V = s.V;
  kp.C = s.C;
  kp.g = s.nq / s.nkv;
  kp.eps = (float)cfg->rms_eps;
  kp.attn_scale = (float)(1.0 / std::sqrt((double)s.d));
  kp.inv_H = (float)(1.0 / (double)kp.H);
  kp.qkv_bias = s.qkv_bias;
  kp.tasks = h->d_tasks;
  kp.task_off = h->d_task_off;
  kp.chunks = h->d_chunks;
  kp.chunk_off = h->d_chunk_off;
  kp.act = p.act;
  kp.nsplit = p.nsplit;
  kp.split_len = p.split_len;
  kp.combine_group = p.combine_group;
  kp.rows_per_stage = p.attn_rows_per_stage;
  kp.num_stages = p.num_stages;
  kp.off_sv = p.off_sv;
  kp.off_res = p.off_res;
  kp.off_resid = p.off_resid;
  kp.off_tasks = p.off_tasks;
  kp.off_ring = p.off_ring;
  kp.embed = reinterpret_cast<const uint16_t*>(weights->embed);
  kp.final_norm = reinterpret_cast<const uint16_t*>(weights->final_norm);
  kp.layers = h->d_layers;
  kp.kv = reinterpret_cast<uint16_t*>(kv_cache);
  kp.rope = h->d_rope;
  kp.words = h->d_words;
  kp.status = h->d_status;
  kp.host_status = h_status_dev;
  kp.timeout_ns = (unsigned long long)env_int("MBK_WAIT_TIMEOUT_MS", 1000) * 1000000ull;
  kp.poll_backoff_ns = (unsigned)std::max(0, env_int("MBK_POLL_BACKOFF_NS", 0));
  kp.lm_tasks = lm_task_count(p);
  kp.page_table = h->paged ? h->d_page_table : nullptr;
  kp.page_size = h->paged ? h->page_size : s.C;
  kp.page_shift = 0;
  while (h->paged && (1 << kp.page_shift) < h->page_size) ++kp.page_shift;
  kp.page_elems = h->paged ? (unsigned long long)s.L * 2 * s.nkv * h->page_size * s.d : 0ull;
  // tensor-core attention: the whole cache (or pool) as rows of 64 bf16; the CUDA-core path if the
  // map cannot be made
  kp.attn_box_rows = std::min(kp.page_size, 64);
  const uint64_t kv_rows = h->paged ? (uint64_t)h->num_pages * (kp.page_elems / 64) : (uint64_t)s.L * 2 * s.nkv * s.C;
  kp.attn_mma = p.attn_mma && make_kv_tile_map(&h->kvmap, kv_cache, kv_rows, (uint32_t)kp.attn_box_rows) ? 1 : 0;
  kp.wbytes = s.wb;
  kp.wscale_layer = wscale_layer;
  kp.wscale = h->d_wscale;
  *out = h;
  return MBK_OK;
}
}  // namespace

namespace {
// One launch of n consecutive steps from pos0 (tokens on the device, or `token` when n == 1).
int launch_steps(mbk_handle* h, int32_t token, const int32_t* d_tokens, int n, int32_t pos0, float* logits, void* stream,
                 int32_t* greedy_out = nullptr) {
  StepParams sp;
  sp.greedy = greedy_out != nullptr;
  sp.amax = h->d_amax;
  sp.amax_done = h->d_amax_done;
  sp.out_tokens = greedy_out;
  sp.tokword = h->d_tokword;
  if (sp.greedy) {
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(h->d_amax, 0, sizeof(unsigned long long) * (size_t)n, st) != cudaSuccess ||
        cudaMemsetAsync(h->d_amax_done, 0, sizeof(unsigned) * (size_t)n, st) != cudaSuccess)
      return MBK_ERR_CUDA;
  }
  sp.token = token;
  sp.pos = pos0;
  // tags tag+1 .. tag+n; tag 0 marks never-written words, so a range that would wrap restarts at 1
  if (h->tag + (unsigned)n < h->tag || h->tag + (unsigned)n == 0u) h->tag = 0;
  sp.tag = h->tag + 1u;
  h->tag += (unsigned)n;
  // greedy decoding without caller logits: every step's logits go to one internal [V] buffer
  sp.logits = logits != nullptr ? logits : h->d_logits_tmp;
  sp.logits_step = logits != nullptr ? h->cfg.vocab : 0;
  sp.tokens = d_tokens;
  sp.n = n;
  sp.sync = n > 1 ? h->d_sync : nullptr;
  sp.sync_base = h->sync_count;
  if (n > 1) h->sync_count += (unsigned long long)n * (unsigned long long)h->grid;
  KernelParams kp = h->kp;
  if (h->inject_armed) {
    kp.inject = h->d_inject;  // one step only
    h->inject_armed = false;
  }
  void* args[] = {&kp, &sp, &h->kvmap};
  cudaError_t e = cudaLaunchCooperativeKernel(decode_kernel_ptr(sp.greedy != 0, h->kp.wbytes == 1, h->kp.attn_mma != 0), dim3(h->grid),
                                              dim3(kThreads), args,
                                              (size_t)h->plan.smem_bytes, (cudaStream_t)stream);
  if (e == cudaErrorCooperativeLaunchTooLarge) return MBK_ERR_UNSUPPORTED;
  return e == cudaSuccess ? MBK_OK : MBK_ERR_CUDA;
}
}  // namespace

int mbk_decode_step(mbk_handle* h, int32_t token_id, int32_t position, float* logits_out, void* stream) {
  if (!h || !logits_out) return MBK_ERR_INVALID_ARG;
  if (token_id < 0 || token_id >= h->cfg.vocab || position < 0 || position >= h->mapped) return MBK_ERR_INVALID_ARG;
  if (int st = sticky_status(h)) return st;
  if (cudaSetDevice(h->device) != cudaSuccess) return MBK_ERR_CUDA;
  h->last_token = token_id;
  return launch_steps(h, token_id, nullptr, 1, position, logits_out, stream);
}

int mbk_decode_steps(mbk_handle* h, const int32_t* tokens, int32_t n_steps, int32_t position, float* logits_out,
                     void* stream) {
  if (!h || !tokens || !logits_out || n_steps < 1) return MBK_ERR_INVALID_ARG;
  if (position < 0 || n_steps > h->mapped || position > h->mapped - n_steps) return MBK_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_steps; ++i)
    if (tokens[i] < 0 || tokens[i] >= h->cfg.vocab) return MBK_ERR_INVALID_ARG;
  if (h->inject_armed) return MBK_ERR_STATE;  // injection is defined for single steps only
  if (int st = sticky_status(h)) return st;
  if (cudaSetDevice(h->device) != cudaSuccess) return MBK_ERR_CUDA;
  if (cudaMemcpyAsync(h->d_tokens, tokens, sizeof(int32_t) * (size_t)n_steps, cudaMemcpyHostToDevice,
                      (cudaStream_t)stream) != cudaSuccess)
    return MBK_ERR_CUDA;
  h->last_token = tokens[n_steps - 1];
  if (n_steps == 1) return launch_steps(h, tokens[0], nullptr, 1, position, logits_out, stream);
  return launch_steps(h, 0, h->d_tokens, n_steps, position, logits_out, stream);
}

int mbk_decode_greedy(mbk_handle* h, int32_t first_token, int32_t n_steps, int32_t position, int32_t* tokens_out,
                      float* logits_out, void* stream) {
  if (!h || !tokens_out || n_steps < 1) return MBK_ERR_INVALID_ARG;
  if (first_token < 0 || first_token >= h->cfg.vocab) return MBK_ERR_INVALID_ARG;
  if (position < 0 || n_steps > h->mapped || position > h->mapped - n_steps) return MBK_ERR_INVALID_ARG;
  if (h->inject_armed) return MBK_ERR_STATE;  // injection is defined for single teacher-forced steps only
  if (int st = sticky_status(h)) return st;
  if (cudaSetDevice(h->device) != cudaSuccess) return MBK_ERR_CUDA;
  h->last_token = first_token;
  return launch_steps(h, first_token, nullptr, n_steps, position, logits_out, stream, tokens_out);
}

namespace {
// The prefill path for n tokens grouped by sequence (mbk_prefill, mbk_batch_step); arguments validated.
int run_tokens(mbk_handle* h, const PrefillBatch& batch, const int32_t* tokens, int32_t n, float* logits_out,
               int32_t logits_mode, void* stream) {
  if (h->cfg.weight_format != MBK_WEIGHTS_BF16) return MBK_ERR_UNSUPPORTED;
  if (h->inject_armed) return MBK_ERR_STATE;
  if (h->prefill_inject_n != 0 && h->prefill_inject_n != n) return MBK_ERR_INVALID_ARG;
  if (int st = sticky_status(h)) return st;
  if (cudaSetDevice(h->device) != cudaSuccess) return MBK_ERR_CUDA;
  const KernelParams& kp = h->kp;
  PrefillModel m;
  m.L = kp.L;
  m.H = kp.H;
  m.I = kp.I;
  m.nq = kp.nq;
  m.nkv = kp.nkv;
  m.d = kp.d;
  m.V = kp.V;
  m.eps = kp.eps;
  m.inv_H = kp.inv_H;
  m.attn_scale = kp.attn_scale;
  m.qkv_bias = kp.qkv_bias;
  m.embed = kp.embed;
  m.final_norm = kp.final_norm;
  m.layers = h->bf16_layers;
  m.rope = kp.rope;
  m.kv = kp.kv;
  m.page_table = kp.page_table;
  m.page_size = kp.page_size;
  m.page_shift = kp.page_shift;
  m.page_elems = kp.page_elems;
  m.status = kp.status;
  m.host_status = kp.host_status;
  m.timeout_ns = kp.timeout_ns;
  const float* inject = h->prefill_inject_n != 0 ? h->d_prefill_inject : nullptr;
  h->prefill_inject_n = 0;  // one call
  return prefill_run(m, h->prefill, tokens, n, batch, logits_out, logits_mode, (cudaStream_t)stream, inject);
}

bool logits_mode_ok(int32_t mode, const float* logits_out) {
  if (mode != MBK_PREFILL_LOGITS_NONE && mode != MBK_PREFILL_LOGITS_LAST && mode != MBK_PREFILL_LOGITS_ALL) return false;
  return mode == MBK_PREFILL_LOGITS_NONE || logits_out != nullptr;
}
}  // namespace

int mbk_prefill(mbk_handle* h, const int32_t* tokens, int32_t n_tokens, int32_t position, float* logits_out,
                int32_t logits_mode, void* stream) {
  if (!h || !tokens || n_tokens < 1 || !logits_mode_ok(logits_mode, logits_out)) return MBK_ERR_INVALID_ARG;
  if (position < 0 || n_tokens > h->mapped || position > h->mapped - n_tokens) return MBK_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_tokens; ++i)
    if (tokens[i] < 0 || tokens[i] >= h->cfg.vocab) return MBK_ERR_INVALID_ARG;
  PrefillBatch b;
  b.n_seq = 1;
  b.counts = &n_tokens;
  b.starts = &position;
  return run_tokens(h, b, tokens, n_tokens, logits_out, logits_mode, stream);
}

int mbk_batch_step(mbk_handle* h, int32_t n_seq, const int32_t* counts, const int32_t* starts, const int32_t* tokens,
                   const int32_t* page_tables, float* logits_out, int32_t logits_mode, void* stream) {
  if (!h || n_seq < 1 || !counts || !starts || !tokens || !page_tables) return MBK_ERR_INVALID_ARG;
  if (!h->paged || !logits_mode_ok(logits_mode, logits_out)) return MBK_ERR_INVALID_ARG;
  const int C = h->cfg.kv_capacity, ps = h->page_size;
  std::vector<char> used(h->num_pages, 0);
  int64_t n = 0;
  for (int32_t q = 0; q < n_seq; ++q) {
    if (counts[q] < 1 || starts[q] < 0 || counts[q] > C || starts[q] > C - counts[q]) return MBK_ERR_INVALID_ARG;
    const int32_t* t = page_tables + (size_t)q * h->max_pages;
    const int need = (starts[q] + counts[q] + ps - 1) / ps;  // pages the sequence's positions reach
    for (int i = 0; i < need; ++i) {
      if (t[i] < 0 || t[i] >= h->num_pages || used[t[i]]) return MBK_ERR_INVALID_ARG;  // in the pool, not shared
      used[t[i]] = 1;
    }
    n += counts[q];
  }
  if (n > (int64_t)1 << 24) return MBK_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= h->cfg.vocab) return MBK_ERR_INVALID_ARG;
  PrefillBatch b;
  b.n_seq = n_seq;
  b.counts = counts;
  b.starts = starts;
  b.tables = page_tables;
  b.max_pages = h->max_pages;
  return run_tokens(h, b, tokens, (int32_t)n, logits_out, logits_mode, stream);
}

int mbk_debug_prefill_inject(mbk_handle* h, const float* x_in, int32_t n_tokens) {
  if (!h) return MBK_ERR_INVALID_ARG;
  if (!x_in) {
    h->prefill_inject_n = 0;
    return MBK_OK;
  }
  if (n_tokens < 1 || n_tokens > h->cfg.kv_capacity) return MBK_ERR_INVALID_ARG;
  if (cudaSetDevice(h->device) != cudaSuccess) return MBK_ERR_CUDA;
  const size_t n = (size_t)h->cfg.n_layers * n_tokens * h->cfg.hidden;
  if (n > h->prefill_inject_cap) {
    cudaFree(h->d_prefill_inject);
    h->d_prefill_inject = nullptr;
    h->prefill_inject_cap = 0;
    if (cudaMalloc(&h->d_prefill_inject, n * sizeof(float)) != cudaSuccess) return MBK_ERR_NOMEM;
    h->prefill_inject_cap = n;
  }
  if (cudaMemcpy(h->d_prefill_inject, x_in, n * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess)
    return MBK_ERR_CUDA;
  h->prefill_inject_n = n_tokens;
  return MBK_OK;
}

int mbk_decode_step_host(mbk_handle* h, int32_t token_id, int32_t position, float* logits_host, void* stream) {
  if (!h || !logits_host) return MBK_ERR_INVALID_ARG;
  int rc = mbk_decode_step(h, token_id, position, h->d_logits_tmp, stream);
  if (rc != MBK_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(logits_host, h->d_logits_tmp, sizeof(float) * h->cfg.vocab, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MBK_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MBK_ERR_CUDA;
  return sticky_status(h);
}

int mbk_kv_fill(mbk_handle* h, int layer, const float* k_raw, const float* v_raw, int32_t p0, int32_t n, void* stream) {
  if (!h || !k_raw || !v_raw) return MBK_ERR_INVALID_ARG;
  const mbk_config& c = h->cfg;
  if (layer < 0 || layer >= c.n_layers || p0 < 0 || n < 0 || (int64_t)p0 + n > h->mapped) return MBK_ERR_INVALID_ARG;
  if (int st = sticky_status(h)) return st;
  if (n == 0) return MBK_OK;
  if (cudaSetDevice(h->device) != cudaSuccess) return MBK_ERR_CUDA;
  cudaError_t e = launch_kv_fill(h->kp, layer, k_raw, v_raw, p0, n, (cudaStream_t)stream);
  return e == cudaSuccess ? MBK_OK : MBK_ERR_CUDA;
}

int mbk_get_status(mbk_handle* h) {
  if (!h) return MBK_ERR_INVALID_ARG;
  if (h->sticky != MBK_OK) return h->sticky;
  unsigned st[4] = {0, 0, 0, 0};
  if (cudaSetDevice(h->device) != cudaSuccess || cudaMemcpy(st, h->d_status, 16, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MBK_ERR_CUDA;
  if (st[0] != 0u) h->sticky = MBK_ERR_TIMEOUT;
  return h->sticky;
}

int mbk_debug_taps(mbk_handle* h, float* taps_out) {
  if (!h || !taps_out) return MBK_ERR_INVALID_ARG;
  const mbk_config& c = h->cfg;
  if (cudaSetDevice(h->device) != cudaSuccess) return MBK_ERR_CUDA;
  std::vector<unsigned long long> words(h->plan.act_words);
  std::vector<uint16_t> emb(c.hidden);
  if (cudaMemcpy(words.data(), h->d_words, words.size() * 8, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(emb.data(), h->kp.embed + (size_t)h->last_token * c.hidden, c.hidden * 2, cudaMemcpyDeviceToHost) !=
          cudaSuccess)
    return MBK_ERR_CUDA;
  auto val = [](unsigned long long w) {
    uint32_t u = (uint32_t)w;
    float f;
    memcpy(&f, &u, 4);
    return f;
  };
  for (int i = 0; i < c.hidden; ++i) {
    uint32_t u = (uint32_t)emb[i] << 16;
    memcpy(&taps_out[i], &u, 4);
  }
  for (int l = 0; l < c.n_layers; ++l) {
    const unsigned long long* lw = words.data() + (size_t)l * h->plan.act.per_layer;
    for (int i = 0; i < c.hidden; ++i) {
      float xa;
      if (h->plan.fused_attn) {
        // x_attn is not stored: the layer input plus the heads' partials, summed as the kernel does
        xa = taps_out[(size_t)(2 * l) * c.hidden + i];
        for (int s = 0; s < c.n_kv_heads; ++s) xa += val(lw[h->plan.act.ap + (size_t)s * c.hidden + i]);
      } else {
        xa = val(lw[h->plan.act.xa + i]);
      }
      taps_out[(size_t)(2 * l + 1) * c.hidden + i] = xa;
      taps_out[(size_t)(2 * l + 2) * c.hidden + i] = val(lw[h->plan.act.xm + i]);
    }
  }
  return MBK_OK;
}

int mbk_debug_inject(mbk_handle* h, const float* x_in) {
  if (!h) return MBK_ERR_INVALID_ARG;
  if (!x_in) {
    h->inject_armed = false;
    return MBK_OK;
  }
  const mbk_config& c = h->cfg;
  if (cudaSetDevice(h->device) != cudaSuccess) return MBK_ERR_CUDA;
  const size_t n = (size_t)c.n_layers * c.hidden;
  if (!h->d_inject && cudaMalloc(&h->d_inject, n * sizeof(unsigned long long)) != cudaSuccess) return MBK_ERR_NOMEM;
  unsigned next_tag = h->tag + 1;
  if (next_tag == 0) next_tag = 1;
  std::vector<unsigned long long> w(n);
  for (size_t i = 0; i < n; ++i) {
    uint32_t u;
    memcpy(&u, &x_in[i], 4);
    w[i] = ((unsigned long long)next_tag << 32) | u;
  }
  if (cudaMemcpy(h->d_inject, w.data(), n * sizeof(unsigned long long), cudaMemcpyHostToDevice) != cudaSuccess)
    return MBK_ERR_CUDA;
  h->inject_armed = true;
  return MBK_OK;
}

int64_t mbk_debug_plan(mbk_handle* h, int32_t* out, int64_t capacity) {
  if (!h || (!out && capacity > 0)) return MBK_ERR_INVALID_ARG;
  const Plan& p = h->plan;
  for (int c = 0; c < p.num_ctas; ++c)
    for (uint32_t i = p.task_off[c]; i < p.task_off[c + 1]; ++i) {
      if ((int64_t)i >= capacity) continue;
      const Task& t = p.tasks[i];
      int32_t* r = out + (size_t)i * 6;
      r[0] = c;
      r[1] = t.type;
      r[2] = t.layer;
      r[3] = (int32_t)t.row0;
      r[4] = (int32_t)t.nrows;
      r[5] = (int32_t)t.nchunks;
    }
  return (int64_t)p.tasks.size();
}

int mbk_trace_enable(mbk_handle* h, int enable) {
  if (!h) return MBK_ERR_INVALID_ARG;
  if (cudaSetDevice(h->device) != cudaSuccess) return MBK_ERR_CUDA;
  if (enable && !h->d_trace) {
    size_t bytes = sizeof(unsigned long long) * kTraceStamps * std::max<size_t>(1, h->plan.tasks.size());
    if (cudaMalloc(&h->d_trace, bytes) != cudaSuccess) return MBK_ERR_NOMEM;
    if (cudaMemset(h->d_trace, 0, bytes) != cudaSuccess) return MBK_ERR_CUDA;
  } else if (!enable && h->d_trace) {
    cudaDeviceSynchronize();
    cudaFree(h->d_trace);
    h->d_trace = nullptr;
  }
  h->kp.trace = h->d_trace;
  return MBK_OK;
}

int64_t mbk_trace_read(mbk_handle* h, uint64_t* out, int64_t capacity_tasks) {
  if (!h || !out || !h->d_trace) return MBK_ERR_INVALID_ARG;
  int64_t n = std::min<int64_t>(capacity_tasks, (int64_t)h->plan.tasks.size());
  if (cudaSetDevice(h->device) != cudaSuccess ||
      cudaMemcpy(out, h->d_trace, sizeof(uint64_t) * kTraceStamps * n, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MBK_ERR_CUDA;
  return (int64_t)h->plan.tasks.size();
}

void mbk_destroy(mbk_handle* h) {
  if (!h) return;
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  free_all(h);
  delete h;
}

}  // extern "C"
