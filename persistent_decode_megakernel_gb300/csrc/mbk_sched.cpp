// mbk_sched.cpp -- host-side static scheduler for the persistent decode kernel.
//
// The pages' planner (MegaBake article, "How a model gets in", steps 4-5) groups regions into
// phases separated by grid barriers and folds small producers into their consumers.  Here the
// plan is finer grained: every projection is split by output rows into tasks spread over all
// CTAs (so every SM streams weights every layer), norms/RoPE/SiLU/residual adds are fused into the
// tasks that need them, and each task depends only on the activation words it reads.  Tasks are
// appended to CTA lists in one global topological order (layer by layer, op by op), which is what
// makes the spin-waits deadlock-free when all CTAs are co-resident.
#include "mbk_sched.h"

#include <algorithm>
#include <cstdio>
#include <map>

namespace mbk {

namespace {

struct Seg {          // a run of rows of one weight matrix
  uint64_t base;      // matrix base address
  int row_bytes;
  int first_row;
  int nrows;
};

void add_chunks(std::vector<Chunk>& out, const Seg& sg) {
  int per = kStageBytes / sg.row_bytes;
  for (int r = 0; r < sg.nrows; r += per) {
    int n = std::min(per, sg.nrows - r);
    Chunk c;
    c.src = sg.base + (uint64_t)(sg.first_row + r) * (uint64_t)sg.row_bytes;
    c.bytes = (uint32_t)(n * sg.row_bytes);
    c.rows = (uint32_t)n;
    out.push_back(c);
  }
}

// GEMV layout of a task: t.gpr warps split each weight row's K range (a warp keeps its slice of
// the input in registers, at most 32 * kGemvXVec vectors), and each warp works on two rows at a
// time.  Among the feasible splits, the largest one that keeps every lane on at least one vector
// and no more warps than the task's largest kGemvBatch-chunk batch can use, within the
// partial-result slots.
constexpr int kCombineRows = 24;  // fewest output rows of a split-context O-projection task (by default)

uint32_t pow2_floor(uint32_t v) {
  uint32_t p = 1;
  while (p * 2 <= v) p *= 2;
  return p;
}
uint32_t pow2_ceil(uint32_t v) {
  uint32_t p = 1;
  while (p < v) p *= 2;
  return p;
}
void gemv_layout(const std::vector<Chunk>& chunks, Task& t, int in, int res_per_row) {
  const uint32_t nvec = (uint32_t)in / 8;
  uint32_t max_rows = 1;
  for (uint32_t k = 0; k < t.nchunks; k += kGemvBatch) {
    uint32_t rows = 0;
    for (uint32_t j = k; j < std::min<uint32_t>(t.nchunks, k + kGemvBatch); ++j) rows += chunks[t.chunk0 + j].rows;
    max_rows = std::max(max_rows, rows);
  }
  if (res_per_row == 2) {
    // gate/up: with one batch and at most one row pair per warp, a warp takes gate row r and up row
    // r together and writes silu(gate) * up itself
    if (t.nchunks <= (uint32_t)kGemvBatch && t.nrows <= (uint32_t)kComputeWarps) {
      t.gpr = 0;
      return;
    }
  } else if (max_rows <= (uint32_t)kComputeWarps) {  // small task: one warp per row, x from shared memory
    t.gpr = 0;
    return;
  }
  const uint32_t need = pow2_ceil((nvec + 32 * kGemvXVec - 1) / (32 * kGemvXVec));  // registers bound
  const uint32_t lanes = pow2_floor(std::max(1u, nvec / 32));                          // a vector per lane
  const uint32_t work = pow2_floor(std::max(1u, (uint32_t)kComputeWarps / ((max_rows + 1) / 2)));
  uint32_t gpr = std::max(need, std::min(lanes, work));
  gpr = std::min<uint32_t>(gpr, pow2_floor(kComputeWarps));
  while (gpr > need && (uint64_t)t.nrows * res_per_row * gpr > (uint64_t)kResSlots) gpr /= 2;
  t.gpr = gpr;
}

}  // namespace

std::string validate_shape(const PlanShape& s) {
  char buf[256];
  if (s.L <= 0 || s.H <= 0 || s.I <= 0 || s.nq <= 0 || s.nkv <= 0 || s.V <= 0 || s.C <= 0) return "non-positive dimension";
  if (s.d != 64 && s.d != 128) return "head_dim must be 64 or 128";
  if (s.nq % s.nkv != 0) return "n_heads must be a multiple of n_kv_heads";
  if (s.nq / s.nkv > 16) return "at most 16 query heads per KV head";
  if (s.H % 8 || s.I % 8) return "hidden and intermediate must be multiples of 8";
  int max_in = std::max(std::max(s.H, s.I), s.nq * s.d);
  if (s.wb != 1 && s.wb != 2) return "weights must be bf16 or FP8";
  if (s.wb == 1 && (s.H % 16 || s.I % 16)) return "FP8 weights need hidden and intermediate sizes that are multiples of 16";
  if (max_in * s.wb > kStageBytes) {
    snprintf(buf, sizeof buf, "a weight row of %d elements exceeds one %d-byte stage", max_in, kStageBytes);
    return buf;
  }
  if (s.H > kMaxTaskRows) return "hidden larger than the per-task result capacity";
  if (s.L > kMaxLayers) return "more layers than the kernel's pointer tables hold";
  return "";
}

WeightAddrs fake_weight_addrs(const PlanShape& s) {
  WeightAddrs w;
  uint64_t base = 1ull << 40;
  auto next = [&](uint64_t bytes) { uint64_t a = base; base += (bytes + 4095) / 4096 * 4096 + 4096; return a; };
  w.embed = next((uint64_t)s.V * s.H * 2);
  w.final_norm = next((uint64_t)s.H * 2);
  w.layers.resize(s.L);
  uint64_t qd = (uint64_t)s.nq * s.d, kvd = (uint64_t)s.nkv * s.d;
  for (int l = 0; l < s.L; ++l) {
    auto& a = w.layers[l];
    a[W_ATTN_NORM] = next(s.H * 2);
    a[W_Q] = next(qd * s.H * 2);
    a[W_K] = next(kvd * s.H * 2);
    a[W_V] = next(kvd * s.H * 2);
    a[W_BQ] = s.qkv_bias ? next(qd * 2) : 0;
    a[W_BK] = s.qkv_bias ? next(kvd * 2) : 0;
    a[W_BV] = s.qkv_bias ? next(kvd * 2) : 0;
    a[W_O] = next((uint64_t)s.H * qd * 2);
    a[W_MLP_NORM] = next(s.H * 2);
    a[W_GATE] = next((uint64_t)s.I * s.H * 2);
    a[W_UP] = next((uint64_t)s.I * s.H * 2);
    a[W_DOWN] = next((uint64_t)s.H * s.I * 2);
  }
  return w;
}

namespace {
// The words a task reads and writes (indices into the step's word array) and its flags.
void fill_task_io(const PlanShape& s, const Plan& p, Task& t) {
  const ActLayout& a = p.act;
  const uint32_t l = t.layer, pl = a.per_layer;
  const uint32_t lw = l * pl, prev = l > 0 ? (l - 1) * pl + a.xm : 0;  // this layer's words; its input stream
  const uint32_t keep_aux = t.type == T_ATTN ? t.aux : 0;  // an attention task's KV head (TF_WO)
  const uint16_t keep_flags = t.type == T_ATTN ? (uint16_t)(t.flags & (TF_WO | TF_KV_APPEND)) : 0;
  t.flags = keep_flags;
  t.in_off = t.in_n = t.res_off = t.out_off = t.gain = 0;
  t.aux = keep_aux;
  switch (t.type) {
    case T_QKV:
      t.flags = TF_NORM | (l == 0 ? TF_IN_EMB : TF_IN_LAYER) | (s.qkv_bias ? TF_BIAS : 0);
      t.in_off = prev;
      t.in_n = (uint32_t)s.H;
      t.gain = 2 * l;
      t.out_off = lw + a.qkv + t.row0;
      break;
    case T_ATTN:
      t.in_off = lw + a.qkv;
      t.in_n = (uint32_t)((s.nq + 2 * s.nkv) * s.d);
      t.out_off = (t.flags & TF_WO) ? lw + a.ap + t.aux * (uint32_t)s.H + t.row0 : lw + a.att;
      break;
    case T_OPROJ:
      t.flags = TF_RES | (l == 0 ? TF_RES_EMB : TF_RES_LAYER) | (p.nsplit > 1 ? TF_COMBINE : 0);
      t.in_off = lw + a.att;
      t.in_n = (uint32_t)(s.nq * s.d);
      t.res_off = prev + t.row0;
      t.out_off = lw + a.xa + t.row0;
      break;
    case T_GATEUP:
      t.flags = TF_NORM | TF_PAIRS;
      if (p.fused_attn) {  // x_attn = layer input + the heads' partial O projections
        t.flags |= TF_IN_SUM | (l == 0 ? TF_IN_EMB : TF_IN_LAYER);
        t.in_off = prev;
        t.aux = lw + a.ap;
      } else {
        t.in_off = lw + a.xa;
      }
      t.in_n = (uint32_t)s.H;
      t.gain = 2 * l + 1;
      t.out_off = lw + a.hh + t.row0;
      break;
    case T_DOWN:
      t.flags = TF_RES;
      t.in_off = lw + a.hh;
      t.in_n = (uint32_t)s.I;
      if (p.fused_attn) {  // residual rows of x_attn, summed the same way
        t.flags |= TF_RES_SUM | (l == 0 ? TF_RES_EMB : TF_RES_LAYER);
        t.res_off = prev + t.row0;
        t.aux = lw + a.ap + t.row0;
      } else {
        t.res_off = lw + a.xa + t.row0;
      }
      t.out_off = lw + a.xm + t.row0;
      break;
    default:  // LM head
      t.flags = TF_NORM | TF_LOGITS;
      t.in_off = (uint32_t)(s.L - 1) * pl + a.xm;
      t.in_n = (uint32_t)s.H;
      t.gain = 2 * (uint32_t)s.L;
      break;
  }
}
}  // namespace

std::string build_plan(const PlanShape& s, const WeightAddrs& w, int num_ctas, const PlanOptions& opt, Plan* out) {
  std::string err = validate_shape(s);
  if (!err.empty()) return err;
  if (num_ctas <= 0) return "no CTAs";
  if ((int)w.layers.size() != s.L) return "weight table does not match n_layers";
  Plan& p = *out;
  p = Plan();
  p.num_ctas = num_ctas;
  const int g = s.nq / s.nkv;
  const int qd = s.nq * s.d, kvd = s.nkv * s.d;

  // attention context splits: one split for short caches; otherwise splits of at most
  // kAttnSplitMax positions and at most kAttnSplitStages ring stages (a split holds all its stages)
  p.attn_rows_per_stage = kStageBytes / (2 * s.d * 2);
  if (opt.attn_split != 0 && (opt.attn_split < 64 || opt.attn_split % 64 != 0)) return "attention split not a multiple of 64";
  const int split_cap = std::min(opt.attn_split > 0 ? opt.attn_split : kAttnSplitMax, kAttnSplitStages * p.attn_rows_per_stage);
  p.split_len = s.C <= split_cap ? s.C : split_cap;
  p.nsplit = (s.C + p.split_len - 1) / p.split_len;
  // the split combine keeps (m, l) of every query head and split in the results area
  if (s.nq * p.nsplit * 2 > kResSlots) return "KV capacity too long for the attention split combine";

  // the O projection fused into the attention tasks: one context split and few KV heads (its
  // consumers sum n_kv + 1 vectors)
  p.fused_attn = p.nsplit == 1 && s.nkv <= kMaxFusedKvHeads && (s.nq / s.nkv) * s.d <= kMaxFusedGroupWidth &&
                 opt.fuse_attention != 0;

  // activation words
  ActLayout a{};
  a.qkv = 0;
  a.att = a.qkv + (uint32_t)(qd + 2 * kvd);
  a.xa = a.att + (uint32_t)(s.nkv * p.nsplit * g * (s.d + 2));
  a.hh = a.xa + (uint32_t)s.H;
  a.xm = a.hh + (uint32_t)s.I;
  a.ap = a.xm + (uint32_t)s.H;
  a.per_layer = a.ap + (p.fused_attn ? (uint32_t)(s.nkv * s.H) : 0u);
  p.act = a;
  p.act_words = (uint64_t)a.per_layer * s.L;

  // shared memory layout: [barriers + flags 1 KB][input vector][results][residuals][ring]
  // attention: rotated queries (d + d/8 floats a head), current K/V (raw, then the bf16 row appended),
  // the partial output (o, m, l) of every (32-position block, query head) item of a split, and each
  // compute warp's 32 item weights
  // tensor-core attention: one partial per compute warp that holds a 16-position block, plus the
  // current row's (in place of the 32-position items)
  p.attn_mma = opt.attn_mma != 0 && s.d == 64 && g <= 8;
  const int attn_parts = p.attn_mma ? std::max((p.split_len + 31) / 32, std::min(kComputeWarps, (p.split_len + 15) / 16) + 1)
                                    : (p.split_len + 31) / 32;
  const int attn_items = attn_parts * g;
  const int attn_floats = g * (s.d + s.d / 8) + 3 * s.d + attn_items * (s.d + 4) + kComputeWarps * 32;
  const int sv_base = std::max(std::max(std::max(s.H, s.I), qd), attn_floats);
  // the O projection of a split context combines the splits from the (m, l) words of every active
  // split and their o words, combine_group splits per poll, polled into the vector area after the
  // combined output; every split in one poll where the shared memory allows (set with the layout)
  auto sv_for = [&](int cg) {
    int v = sv_base;
    if (p.nsplit > 1) v = std::max(v, qd + p.nsplit * 2 * s.nq + cg * qd);
    return (v + 31) / 32 * 32;
  };
  p.combine_group = p.nsplit;
  p.sv_floats = sv_for(p.combine_group);

  // tasks
  std::vector<std::vector<Task>> cta_tasks(num_ctas);
  std::vector<std::vector<Chunk>> cta_chunks(num_ctas);
  std::vector<int64_t> cta_bytes(num_ctas, 0);
  int cursor = 0;
  const int max_tasks = opt.max_tasks_per_op > 0 ? std::min(opt.max_tasks_per_op, num_ctas) : num_ctas;

  // row-split GEMV op: `segs_for(r0, r1)` lists the weight segments of output rows [r0, r1)
  // CTAs that ran this layer's attention tasks: the O projection that follows skips them, since
  // they finish their attention last (when other CTAs are left)
  std::vector<char> busy(num_ctas, 0);
  int n_busy = 0;
  auto gemv_op = [&](TaskType type, int layer, int rows, int res_per_row, int row_bytes, auto segs_for) {
    int n = std::min(max_tasks, rows);
    if (type == T_OPROJ && n_busy < num_ctas) n = std::min(n, num_ctas - n_busy);  // one task per free CTA
    // A split context's O-projection tasks each poll every active split's outputs before their rows;
    // many such tasks flood L2 with polls and slow every exchange of the layer, so they get at least
    // kCombineRows rows each (24 tasks at hidden 576 measured fastest, between 8 and 104)
    if (type == T_OPROJ && p.nsplit > 1)
      n = std::min(n, opt.combine_tasks > 0 ? opt.combine_tasks : std::max(1, rows / kCombineRows));
    // results per task must fit the result slots, and its chunks the per-task chunk bound
    const int rpc = kStageBytes / row_bytes;
    auto chunks_for = [&](int task_rows) { return res_per_row * ((task_rows + rpc - 1) / rpc) + 2; };
    while ((rows + n - 1) / n * res_per_row > kMaxTaskRows || chunks_for((rows + n - 1) / n) > kMaxTaskChunks) ++n;
    for (int i = 0; i < n; ++i) {
      int r0 = (int)((int64_t)rows * i / n), r1 = (int)((int64_t)rows * (i + 1) / n);
      if (r1 <= r0) continue;
      int cta = cursor % num_ctas;
      ++cursor;
      if (type == T_OPROJ && n_busy < num_ctas) {
        while (busy[cta]) {
          cta = cursor % num_ctas;
          ++cursor;
        }
      }
      Task t{};
      t.type = type;
      t.layer = (uint16_t)layer;
      t.row0 = (uint32_t)r0;
      t.nrows = (uint32_t)(r1 - r0);
      t.chunk0 = (uint32_t)cta_chunks[cta].size();
      for (const Seg& sg : segs_for(r0, r1)) add_chunks(cta_chunks[cta], sg);
      t.nchunks = (uint32_t)(cta_chunks[cta].size() - t.chunk0);
      for (uint32_t c = t.chunk0; c < t.chunk0 + t.nchunks; ++c) cta_bytes[cta] += cta_chunks[cta][c].bytes;
      gemv_layout(cta_chunks[cta], t, row_bytes / s.wb, res_per_row);
      cta_tasks[cta].push_back(t);
    }
  };

  const int hb = s.H * s.wb;  // bytes of a weight row over the hidden size
  const uint64_t lm_base = w.lm_head ? w.lm_head : w.embed;
  for (int l = 0; l < s.L; ++l) {
    const auto& W = w.layers[l];
    gemv_op(T_QKV, l, qd + 2 * kvd, 1, hb, [&](int r0, int r1) {
      std::vector<Seg> v;
      int bounds[4] = {0, qd, qd + kvd, qd + 2 * kvd};
      uint64_t bases[3] = {W[W_Q], W[W_K], W[W_V]};
      for (int m = 0; m < 3; ++m) {
        int a0 = std::max(r0, bounds[m]), a1 = std::min(r1, bounds[m + 1]);
        if (a1 > a0) v.push_back(Seg{bases[m], hb, a0 - bounds[m], a1 - a0});
      }
      return v;
    });
    if (p.fused_attn) {
      // attention with the O projection: per KV head, its columns of Wo split by output rows over
      // the CTAs; each task recomputes the head's attention (every task of a head rounds the
      // appended K/V row identically; the first one writes it to the cache)
      const int seg = g * s.d * s.wb;                     // bytes of one row's segment
      const int rpc = kStageBytes / seg;                  // segments per stage
      const int per_head = std::max(1, std::min(s.H, std::min(max_tasks, num_ctas) / s.nkv));
      for (int kvh = 0; kvh < s.nkv; ++kvh) {
        for (int i = 0; i < per_head; ++i) {
          const int r0 = (int)((int64_t)s.H * i / per_head), r1 = (int)((int64_t)s.H * (i + 1) / per_head);
          if (r1 <= r0) continue;
          int cta = cursor % num_ctas;
          ++cursor;
          Task t{};
          t.type = T_ATTN;
          t.layer = (uint16_t)l;
          t.row0 = (uint32_t)r0;
          t.nrows = (uint32_t)(r1 - r0);
          t.aux = (uint32_t)kvh;
          t.flags = (uint16_t)(TF_WO | (i == 0 ? TF_KV_APPEND : 0));
          t.chunk0 = (uint32_t)cta_chunks[cta].size();
          Chunk ph;
          ph.src = ((uint64_t)l << 48) | ((uint64_t)kvh << 32);
          ph.bytes = 0;
          ph.rows = kAttnChunk;
          cta_chunks[cta].push_back(ph);
          for (int r = r0; r < r1; r += rpc) {
            const int n = std::min(rpc, r1 - r);
            Chunk ch;
            ch.src = W[W_O] + (uint64_t)r * qd * s.wb + (uint64_t)kvh * seg;
            ch.bytes = (uint32_t)(n * seg);
            ch.rows = (uint32_t)n | kStridedRows;
            cta_chunks[cta].push_back(ch);
            cta_bytes[cta] += ch.bytes;
          }
          t.nchunks = (uint32_t)(cta_chunks[cta].size() - t.chunk0);
          t.gpr = 0;
          cta_tasks[cta].push_back(t);
        }
      }
    }
    std::fill(busy.begin(), busy.end(), 0);
    n_busy = 0;
    for (int kvh = 0; kvh < s.nkv && !p.fused_attn; ++kvh) {
      for (int sp = 0; sp < p.nsplit; ++sp) {
        int cta = cursor % num_ctas;
        ++cursor;
        if (!busy[cta]) ++n_busy;
        busy[cta] = 1;
        Task t{};
        t.type = T_ATTN;
        t.layer = (uint16_t)l;
        t.row0 = (uint32_t)kvh;
        t.nrows = (uint32_t)sp;
        t.chunk0 = (uint32_t)cta_chunks[cta].size();
        t.nchunks = 1;
        Chunk ph;
        ph.src = ((uint64_t)l << 48) | ((uint64_t)kvh << 32) | (uint64_t)sp;
        ph.bytes = 0;
        ph.rows = kAttnChunk;
        cta_chunks[cta].push_back(ph);
        cta_tasks[cta].push_back(t);
      }
    }
    if (!p.fused_attn)
      gemv_op(T_OPROJ, l, s.H, 1, qd * s.wb, [&](int r0, int r1) {
        return std::vector<Seg>{Seg{W[W_O], qd * s.wb, r0, r1 - r0}};
      });
    gemv_op(T_GATEUP, l, s.I, 2, hb, [&](int r0, int r1) {
      return std::vector<Seg>{Seg{W[W_GATE], hb, r0, r1 - r0}, Seg{W[W_UP], hb, r0, r1 - r0}};
    });
    gemv_op(T_DOWN, l, s.H, 1, s.I * s.wb, [&](int r0, int r1) {
      return std::vector<Seg>{Seg{W[W_DOWN], s.I * s.wb, r0, r1 - r0}};
    });
  }
  {
    // the LM head is split over every CTA regardless of max_tasks (it is bandwidth bound)
    int n = num_ctas;
    const int rows_per_chunk = kStageBytes / hb;
    while ((s.V + n - 1) / n > kMaxTaskRows || ((s.V + n - 1) / n + rows_per_chunk - 1) / rows_per_chunk > kMaxTaskChunks)
      n += num_ctas;
    for (int i = 0; i < n; ++i) {
      int r0 = (int)((int64_t)s.V * i / n), r1 = (int)((int64_t)s.V * (i + 1) / n);
      if (r1 <= r0) continue;
      int cta = cursor % num_ctas;
      ++cursor;
      Task t{};
      t.type = T_LMHEAD;
      t.layer = (uint16_t)(s.L - 1);
      t.row0 = (uint32_t)r0;
      t.nrows = (uint32_t)(r1 - r0);
      t.chunk0 = (uint32_t)cta_chunks[cta].size();
      add_chunks(cta_chunks[cta], Seg{lm_base, hb, r0, r1 - r0});
      t.nchunks = (uint32_t)(cta_chunks[cta].size() - t.chunk0);
      for (uint32_t c = t.chunk0; c < t.chunk0 + t.nchunks; ++c) cta_bytes[cta] += cta_chunks[cta][c].bytes;
      gemv_layout(cta_chunks[cta], t, s.H, 1);
      cta_tasks[cta].push_back(t);
    }
  }

  // shared memory layout: [control block][input vector][results][residuals][task records][ring]
  p.max_cta_tasks = 0;
  for (const auto& v : cta_tasks) p.max_cta_tasks = std::max(p.max_cta_tasks, (int)v.size());
  const int need_stages = std::max(std::max(2, kGemvBatch), (p.split_len + p.attn_rows_per_stage - 1) / p.attn_rows_per_stage + 1);
  for (;;) {
    p.off_sv = kCtlBytes;
    p.off_res = p.off_sv + (uint32_t)p.sv_floats * 4;
    p.off_resid = p.off_res + kResSlots * 4;
    p.off_tasks = p.off_resid + kMaxTaskRows * 4;
    const uint32_t ring_align = p.attn_mma ? 1024u : 128u;  // swizzled tiles: 1024-byte aligned stages
    p.off_ring = (p.off_tasks + (uint32_t)std::min(p.max_cta_tasks, kTaskWindow) * (uint32_t)sizeof(Task) + ring_align - 1) /
                 ring_align * ring_align;
    const int avail = opt.smem_limit - (int)p.off_ring;
    p.num_stages = std::min(kMaxRingStages, std::max(0, avail) / kStageBytes);
    if (p.num_stages >= need_stages) break;
    // the ring must hold one attention split and one GEMV batch: poll the splits in smaller groups
    if (p.nsplit > 1 && p.combine_group > 1) {
      p.combine_group = (p.combine_group + 1) / 2;
      p.sv_floats = sv_for(p.combine_group);
      continue;
    }
    return p.num_stages < 2 ? "not enough shared memory for the weight ring"
                            : "weight ring too small to hold one attention split or one GEMV batch";
  }
  p.smem_bytes = (int)p.off_ring + p.num_stages * kStageBytes;

  // flatten (chunk indices become global); every task gets its word offsets and flags
  p.task_off.assign(num_ctas + 1, 0);
  p.chunk_off.assign(num_ctas + 1, 0);
  for (int c = 0; c < num_ctas; ++c) {
    uint32_t base = (uint32_t)p.chunks.size();
    for (Task t : cta_tasks[c]) {
      t.chunk0 += base;
      fill_task_io(s, p, t);
      p.tasks.push_back(t);
    }
    p.chunks.insert(p.chunks.end(), cta_chunks[c].begin(), cta_chunks[c].end());
    p.task_off[c + 1] = (uint32_t)p.tasks.size();
    p.chunk_off[c + 1] = (uint32_t)p.chunks.size();
  }
  p.weight_bytes = 0;
  for (const Chunk& c : p.chunks)
    if (c.rows != kAttnChunk) p.weight_bytes += c.bytes;
  p.max_cta_bytes = *std::max_element(cta_bytes.begin(), cta_bytes.end());
  return check_plan(s, w, p);
}

namespace {
int op_rank(const Task& t) { return t.type == T_LMHEAD ? 1 << 30 : t.layer * 8 + t.type; }
}  // namespace

std::string check_plan(const PlanShape& s, const WeightAddrs& w, const Plan& p) {
  char buf[256];
  const int qd = s.nq * s.d, kvd = s.nkv * s.d;
  // tensor extents (base -> bytes) for bounds checks
  std::map<uint64_t, uint64_t> extent;
  const uint64_t wb = (uint64_t)s.wb;
  const uint64_t lm_base = w.lm_head ? w.lm_head : w.embed;
  extent[lm_base] = (uint64_t)s.V * s.H * wb;
  for (int l = 0; l < s.L; ++l) {
    const auto& W = w.layers[l];
    extent[W[W_Q]] = (uint64_t)qd * s.H * wb;
    extent[W[W_K]] = (uint64_t)kvd * s.H * wb;
    extent[W[W_V]] = (uint64_t)kvd * s.H * wb;
    extent[W[W_O]] = (uint64_t)s.H * qd * wb;
    extent[W[W_GATE]] = (uint64_t)s.I * s.H * wb;
    extent[W[W_UP]] = (uint64_t)s.I * s.H * wb;
    extent[W[W_DOWN]] = (uint64_t)s.H * s.I * wb;
  }
  std::map<uint64_t, std::vector<int>> covered;  // tensor base -> per-row count
  auto row_bytes_of = [&](uint64_t base) -> int {
    if (base == lm_base) return s.H * s.wb;
    for (int l = 0; l < s.L; ++l) {
      const auto& W = w.layers[l];
      if (base == W[W_O]) return qd * s.wb;
      if (base == W[W_DOWN]) return s.I * s.wb;
    }
    return s.H * s.wb;
  };
  for (auto& e : extent) covered[e.first].assign(e.second / row_bytes_of(e.first), 0);
  // fused plans stream Wo as per-KV-head segments of each row: (row, head) -> count
  std::map<uint64_t, std::vector<int>> covered_wo;
  if (p.fused_attn)
    for (int l = 0; l < s.L; ++l) {
      covered.erase(w.layers[l][W_O]);
      covered_wo[w.layers[l][W_O]].assign((size_t)s.H * s.nkv, 0);
    }

  if ((int)p.task_off.size() != p.num_ctas + 1 || (int)p.chunk_off.size() != p.num_ctas + 1) return "offsets size";
  // every CTA's tasks use exactly its chunk range, in order
  for (int c = 0; c < p.num_ctas; ++c) {
    uint32_t next = p.chunk_off[c];
    for (uint32_t i = p.task_off[c]; i < p.task_off[c + 1]; ++i) {
      if (p.tasks[i].chunk0 != next) return "task chunks not contiguous in CTA order";
      next += p.tasks[i].nchunks;
    }
    if (next != p.chunk_off[c + 1]) return "CTA chunk range not covered by its tasks";
  }
  int attn_tasks = 0;
  for (int c = 0; c < p.num_ctas; ++c) {
    int last_rank = -1;
    for (uint32_t i = p.task_off[c]; i < p.task_off[c + 1]; ++i) {
      const Task& t = p.tasks[i];
      int rk = op_rank(t);
      if (rk < last_rank) {
        snprintf(buf, sizeof buf, "CTA %d: task %u out of topological order", c, i);
        return buf;
      }
      last_rank = rk;
      if (t.chunk0 < p.chunk_off[c] || t.chunk0 + t.nchunks > p.chunk_off[c + 1]) return "task chunks outside its CTA";
      if (t.type == T_ATTN) {
        const Chunk& ph = p.chunks[t.chunk0];
        if (!(t.flags & TF_WO)) {
          ++attn_tasks;
          if (p.fused_attn || t.nchunks != 1 || (int)t.row0 >= s.nkv || (int)t.nrows >= p.nsplit) return "bad attention task";
          if (ph.rows != kAttnChunk || (int)(ph.src >> 48) != t.layer || (int)((ph.src >> 32) & 0xFFFF) != (int)t.row0 ||
              (uint32_t)ph.src != t.nrows)
            return "bad attention placeholder";
          continue;
        }
        // attention with its KV head's columns of Wo for output rows [row0, row0 + nrows)
        if (!p.fused_attn || p.nsplit != 1 || (int)t.aux >= s.nkv || t.nrows == 0 || t.row0 + t.nrows > (uint32_t)s.H)
          return "bad fused attention task";
        if (t.flags & TF_KV_APPEND) ++attn_tasks;
        if (ph.rows != kAttnChunk || (int)(ph.src >> 48) != t.layer || (int)((ph.src >> 32) & 0xFFFF) != (int)t.aux ||
            (uint32_t)ph.src != 0u)
          return "bad attention placeholder";
        const uint64_t wo = w.layers[t.layer][W_O];
        const uint32_t seg = (uint32_t)((s.nq / s.nkv) * s.d * s.wb);
        uint32_t r = t.row0;
        for (uint32_t k = t.chunk0 + 1; k < t.chunk0 + t.nchunks; ++k) {
          const Chunk& ch = p.chunks[k];
          const uint32_t n = ch.rows & ~kStridedRows;
          if (!(ch.rows & kStridedRows) || n == 0 || ch.bytes != n * seg || ch.bytes > (uint32_t)kStageBytes || ch.src % 16 ||
              seg % 16 || ch.src != wo + (uint64_t)r * qd * s.wb + (uint64_t)t.aux * seg)
            return "bad Wo segment chunk";
          for (uint32_t q = 0; q < n; ++q) covered_wo[wo][(size_t)(r + q) * s.nkv + t.aux] += 1;
          r += n;
        }
        if (r != t.row0 + t.nrows) return "Wo segments do not match the task's rows";
        continue;
      }
      int res = t.type == T_GATEUP ? 2 * (int)t.nrows : (int)t.nrows;
      if (res > kMaxTaskRows || t.nrows == 0) return "task result slots exceeded";
      {
        const int in = t.type == T_OPROJ ? qd : (t.type == T_DOWN ? s.I : s.H);
        const uint32_t nvec = (uint32_t)in / 8;
        if (t.gpr == 0 && t.type == T_GATEUP && (t.nchunks > (uint32_t)kGemvBatch || t.nrows > (uint32_t)kComputeWarps))
          return "gate/up row pairs do not fit one batch";
        if (t.gpr != 0 && ((t.gpr & (t.gpr - 1)) || t.gpr > (uint32_t)kComputeWarps ||
                           (uint64_t)res * t.gpr > (uint64_t)kResSlots || (nvec + t.gpr - 1) / t.gpr > 32u * kGemvXVec))
          return "bad GEMV layout";
      }
      int rows_seen = 0;
      for (uint32_t k = t.chunk0; k < t.chunk0 + t.nchunks; ++k) {
        if (k >= p.chunks.size()) return "chunk index out of range";
        const Chunk& ch = p.chunks[k];
        if (ch.bytes == 0 || ch.bytes % 16 || ch.src % 16 || ch.bytes > (uint32_t)kStageBytes) {
          snprintf(buf, sizeof buf, "chunk %u: bad size/alignment (%u bytes at %llx)", k, ch.bytes, (unsigned long long)ch.src);
          return buf;
        }
        auto it = extent.upper_bound(ch.src);
        if (it == extent.begin()) return "chunk outside every tensor";
        --it;
        if (ch.src + ch.bytes > it->first + it->second) return "chunk runs past its tensor";
        int rb = row_bytes_of(it->first);
        if ((ch.src - it->first) % rb || ch.bytes != ch.rows * (uint32_t)rb) return "chunk not whole rows";
        int r0 = (int)((ch.src - it->first) / rb);
        for (uint32_t r = 0; r < ch.rows; ++r) covered[it->first][r0 + r] += 1;
        rows_seen += (int)ch.rows;
      }
      if (t.nchunks > (uint32_t)kMaxTaskChunks) return "too many chunks in one task";
      if (rows_seen != res) {
        snprintf(buf, sizeof buf, "task %u: %d chunk rows for %d results", i, rows_seen, res);
        return buf;
      }
    }
  }
  for (auto& cv : covered)
    for (size_t r = 0; r < cv.second.size(); ++r)
      if (cv.second[r] != 1) {
        snprintf(buf, sizeof buf, "weight row %zu of tensor %llx streamed %d times", r, (unsigned long long)cv.first, cv.second[r]);
        return buf;
      }
  for (auto& cv : covered_wo)
    for (size_t i = 0; i < cv.second.size(); ++i)
      if (cv.second[i] != 1) return "a Wo row segment is not streamed exactly once";
  if (attn_tasks != s.L * s.nkv * p.nsplit) return "attention task count";
  if (p.smem_bytes > 232448) return "shared memory over the sm_10x limit";
  // every GEMV output word of every layer is written by exactly one task; all word ranges in bounds
  {
    std::vector<uint8_t> cov(p.act_words, 0);
    for (const Task& t : p.tasks) {
      if (t.type == T_ATTN) {
        if ((uint64_t)t.in_off + t.in_n > p.act_words) return "attention input words out of range";
        if (t.flags & TF_WO) {
          if ((uint64_t)t.out_off + t.nrows > p.act_words) return "attention partial words out of range";
          for (uint32_t r = 0; r < t.nrows; ++r) ++cov[t.out_off + r];
        }
        continue;
      }
      if ((t.flags & (TF_IN_SUM | TF_RES_SUM)) &&
          (uint64_t)t.aux + (uint64_t)(s.nkv - 1) * s.H + ((t.flags & TF_IN_SUM) ? (uint64_t)s.H : t.nrows) > p.act_words)
        return "attention partial words out of range";
      if ((uint64_t)t.in_off + t.in_n > p.act_words) return "task input words out of range";
      if ((t.flags & TF_RES) && !(t.flags & TF_RES_EMB) && (uint64_t)t.res_off + t.nrows > p.act_words)
        return "task residual words out of range";
      if (t.type == T_LMHEAD) continue;
      if ((uint64_t)t.out_off + t.nrows > p.act_words) return "task output words out of range";
      for (uint32_t r = 0; r < t.nrows; ++r) ++cov[t.out_off + r];
    }
    const ActLayout& a = p.act;
    for (int l = 0; l < s.L; ++l) {
      const uint64_t b = (uint64_t)l * a.per_layer;
      auto once = [&](uint32_t off, int n) {
        for (int i = 0; i < n; ++i)
          if (cov[b + off + i] != 1) return false;
        return true;
      };
      if (!once(a.qkv, qd + 2 * kvd) || !once(a.hh, s.I) || !once(a.xm, s.H))
        return "an output word is not written exactly once";
      if (p.fused_attn ? !once(a.ap, s.nkv * s.H) : !once(a.xa, s.H)) return "an attention output word is not written exactly once";
    }
  }
  return "";
}

}  // namespace mbk
