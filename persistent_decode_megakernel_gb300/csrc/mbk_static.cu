// mbk_static.cu -- mbk_decode_step_static: a decode step that allocates no device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where they decode: code that
// runs under a caller-owned memory pool or budget that forbids new device allocations, code that
// runs where allocation would stall other streams, or code embedded in a runtime whose allocator
// must not be re-entered.  For them, this entry point keeps everything the library needs for a
// step -- the static schedule, the activation exchange words, the RoPE table and the status
// word -- in one file-scope device array of fixed size, compiled into the library.  The caller
// still passes the weights, the KV cache and the logits buffer.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/mbk.h"
#include "mbk_args.h"
#include "mbk_prefill.h"  // make_kv_tile_map
#include "mbk_device.h"
#include "mbk_sched.h"

namespace mbk {
const void* decode_kernel_ptr(bool greedy, bool fp8, bool mma);
cudaError_t launch_rope_table(float2* out, int C, int d, double theta, cudaStream_t st);
}  // namespace mbk

using namespace mbk;

namespace {

// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kStaticScratchBytes = MBK_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;

// Host-side state per device: the array's device address (looked up once, with that device
// current) and which schedule the array currently holds.
struct DeviceState {
  bool ready = false;
  unsigned char* base = nullptr;
  int smem_optin = 0;
  int num_sms = 0;
  std::string resident_key;  // config + pointers of the schedule now in the array
  Plan plan;
  KernelParams kp{};
  CUtensorMap kvmap{};  // the cache as swizzled tiles (tensor-core attention)
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

std::string plan_key(const mbk_config& c, const mbk_weights& w, const void* kv) {
  std::string k(reinterpret_cast<const char*>(&c), sizeof c);
  auto add = [&](const void* p) { k.append(reinterpret_cast<const char*>(&p), sizeof p); };
  add(w.embed);
  add(w.final_norm);
  add(kv);
  for (int l = 0; l < c.n_layers; ++l) {
    const mbk_layer_weights& L = w.layers[l];
    const void* ps[] = {L.attn_norm, L.wq, L.wk, L.wv, L.bq, L.bk, L.bv, L.wo, L.mlp_norm, L.w_gate, L.w_up, L.w_down};
    for (const void* p : ps) add(p);
  }
  return k;
}

}  // namespace

extern "C" int mbk_decode_step_static(const mbk_config* cfg, const mbk_weights* weights, void* kv_cache,
                                      int32_t token_id, int32_t position, float* logits_out, void* stream) {
  // the same argument checks as mbk_create (config, every weight pointer present and 16-byte
  // aligned), then the step's own; all of them before any CUDA call
  WeightAddrs wa;
  if (!logits_out || gather_weights(cfg, weights, kv_cache, &wa) != MBK_OK) return MBK_ERR_INVALID_ARG;
  if (token_id < 0 || token_id >= cfg->vocab || position < 0 || position >= cfg->kv_capacity) return MBK_ERR_INVALID_ARG;
  if (cfg->weight_format != MBK_WEIGHTS_BF16) return MBK_ERR_INVALID_ARG;  // this entry streams the bf16 weights
  const PlanShape s = shape_of(*cfg);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MBK_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& D = g_dev[dev];
  if (!D.ready) {
    // one-time set-up on this device (this device is current)
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return MBK_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MBK_ERR_CUDA;
    if (prop.major != 10) return MBK_ERR_UNSUPPORTED;
    int coop = 0;
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    cudaDeviceGetAttribute(&D.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (!coop) return MBK_ERR_UNSUPPORTED;
    for (bool mma : {false, true})
      if (cudaFuncSetAttribute(decode_kernel_ptr(false, false, mma), cudaFuncAttributeMaxDynamicSharedMemorySize, D.smem_optin) !=
          cudaSuccess)
        return MBK_ERR_CUDA;
    D.base = static_cast<unsigned char*>(p);
    D.num_sms = prop.multiProcessorCount;
    D.ready = true;
  }
  cudaStream_t st = (cudaStream_t)stream;

  const std::string key = plan_key(*cfg, *weights, kv_cache);
  if (key != D.resident_key) {
    // a new schedule is uploaded and the stream synchronised once: not possible inside a capture
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return MBK_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone) return MBK_ERR_STATE;
    // build the schedule (host memory) and lay it out in the array
    PlanOptions opt;
    opt.smem_limit = D.smem_optin;
    opt.attn_mma = env_int("MBK_ATTN_MMA", 1);
    opt.attn_split = env_int("MBK_ATTN_SPLIT", 0);
    opt.combine_tasks = env_int("MBK_COMBINE_TASKS", 0);
    Plan plan;
    if (!build_plan(s, wa, D.num_sms, opt, &plan).empty()) return MBK_ERR_UNSUPPORTED;
    // layout: tasks | task_off | chunks | chunk_off | layer table | rope | words | status
    const size_t o_tasks = 0;
    const size_t o_toff = align256(o_tasks + sizeof(Task) * plan.tasks.size());
    const size_t o_chunks = align256(o_toff + sizeof(uint32_t) * plan.task_off.size());
    const size_t o_coff = align256(o_chunks + sizeof(Chunk) * plan.chunks.size());
    const size_t o_layers = align256(o_coff + sizeof(uint32_t) * plan.chunk_off.size());
    const size_t o_rope = align256(o_layers + sizeof(LayerW) * s.L);
    const size_t o_words = align256(o_rope + sizeof(float2) * (size_t)s.C * (s.d / 2));
    const size_t o_status = align256(o_words + sizeof(unsigned long long) * plan.act_words);
    const size_t total = align256(o_status + 16);
    if (total > kStaticScratchBytes) return MBK_ERR_INVALID_ARG;  // the shape needs more than the array holds

    std::vector<LayerW> lw(s.L);
    for (int l = 0; l < s.L; ++l)
      for (int k = 0; k < W_NSLOTS; ++k) lw[l].w[k] = reinterpret_cast<const uint16_t*>(wa.layers[l][k]);
    unsigned char* b = D.base;
    D.resident_key.clear();  // invalid until every upload below has been queued
    if (cudaMemcpyAsync(b + o_tasks, plan.tasks.data(), sizeof(Task) * plan.tasks.size(), cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(b + o_toff, plan.task_off.data(), sizeof(uint32_t) * plan.task_off.size(), cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(b + o_chunks, plan.chunks.data(), sizeof(Chunk) * plan.chunks.size(), cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(b + o_coff, plan.chunk_off.data(), sizeof(uint32_t) * plan.chunk_off.size(), cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(b + o_layers, lw.data(), sizeof(LayerW) * s.L, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        launch_rope_table(reinterpret_cast<float2*>(b + o_rope), s.C, s.d, cfg->rope_theta, st) != cudaSuccess)
      return MBK_ERR_CUDA;
    // the host copies above read `plan` and `lw`; wait before they go out of scope
    if (cudaStreamSynchronize(st) != cudaSuccess) return MBK_ERR_CUDA;

    KernelParams& kp = D.kp;
    kp = KernelParams{};
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
    kp.tasks = reinterpret_cast<const Task*>(b + o_tasks);
    kp.task_off = reinterpret_cast<const uint32_t*>(b + o_toff);
    kp.chunks = reinterpret_cast<const Chunk*>(b + o_chunks);
    kp.chunk_off = reinterpret_cast<const uint32_t*>(b + o_coff);
    kp.act = plan.act;
    kp.nsplit = plan.nsplit;
    kp.split_len = plan.split_len;
    kp.combine_group = plan.combine_group;
    kp.rows_per_stage = plan.attn_rows_per_stage;
    kp.num_stages = plan.num_stages;
    kp.off_sv = plan.off_sv;
    kp.off_res = plan.off_res;
    kp.off_resid = plan.off_resid;
    kp.off_tasks = plan.off_tasks;
    kp.off_ring = plan.off_ring;
    kp.embed = reinterpret_cast<const uint16_t*>(weights->embed);
    kp.final_norm = reinterpret_cast<const uint16_t*>(weights->final_norm);
    kp.layers = reinterpret_cast<const LayerW*>(b + o_layers);
    kp.kv = reinterpret_cast<uint16_t*>(kv_cache);
    kp.rope = reinterpret_cast<const float2*>(b + o_rope);
    kp.words = reinterpret_cast<unsigned long long*>(b + o_words);
    kp.status = reinterpret_cast<unsigned*>(b + o_status);
    kp.host_status = nullptr;
    kp.timeout_ns = (unsigned long long)std::max(1, env_int("MBK_WAIT_TIMEOUT_MS", 1000)) * 1000000ull;
    kp.trace = nullptr;
    kp.inject = nullptr;
    kp.poll_backoff_ns = 0;
    int lm = 0;
    for (const Task& t : plan.tasks) lm += t.type == T_LMHEAD ? 1 : 0;
    kp.lm_tasks = lm;
    kp.page_table = nullptr;  // contiguous cache
    kp.page_size = s.C;
    kp.page_shift = 0;
    kp.page_elems = 0;
    kp.attn_box_rows = std::min(s.C, 64);
    kp.attn_mma = plan.attn_mma && make_kv_tile_map(&D.kvmap, kv_cache, (uint64_t)s.L * 2 * s.nkv * s.C,
                                                    (uint32_t)kp.attn_box_rows) ? 1 : 0;
    kp.wbytes = 2;  // bf16 weights as given
    kp.wscale_layer = 0;
    kp.wscale = nullptr;
    D.plan = plan;
    D.resident_key = key;
  }

  // every step starts from cleared exchange words and status (the array keeps the previous
  // call's contents), so tag 1 always marks this step's words
  const size_t words_bytes = sizeof(unsigned long long) * D.plan.act_words;
  if (cudaMemsetAsync(D.kp.words, 0, words_bytes, st) != cudaSuccess || cudaMemsetAsync(D.kp.status, 0, 16, st) != cudaSuccess)
    return MBK_ERR_CUDA;
  StepParams sp;
  sp.token = token_id;
  sp.pos = position;
  sp.tag = 1u;
  sp.logits = logits_out;
  sp.logits_step = 0;
  sp.tokens = nullptr;
  sp.n = 1;
  sp.sync = nullptr;
  sp.sync_base = 0;
  sp.greedy = 0;
  sp.amax = nullptr;
  sp.amax_done = nullptr;
  sp.out_tokens = nullptr;
  sp.tokword = nullptr;
  KernelParams kp = D.kp;
  void* args[] = {&kp, &sp, &D.kvmap};
  cudaError_t e = cudaLaunchCooperativeKernel(decode_kernel_ptr(false, false, D.kp.attn_mma != 0), dim3(D.plan.num_ctas), dim3(kThreads), args,
                                              (size_t)D.plan.smem_bytes, st);
  if (e == cudaErrorCooperativeLaunchTooLarge) return MBK_ERR_UNSUPPORTED;
  return e == cudaSuccess ? MBK_OK : MBK_ERR_CUDA;
}
