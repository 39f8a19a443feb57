// mbk_simulate.cpp -- a host-side execution model of the decode kernel's exchange protocol, so that a
// schedule can be checked for deadlocks and measured in exchange rounds without a GPU.
//
// The model follows what the kernel reads and writes (mbk_kernel.cu): every CTA runs its task list in
// order; a task may run once every activation word it reads has been written in this step, and running
// it writes all of its output words.
//   projection task  reads  its input vector [in_off, in_off + in_n) unless it is the token's embedding,
//                           plus the per-KV-head partials aux + s*H + e (s < n_kv) with TF_IN_SUM;
//                           with TF_RES its residual rows [res_off, res_off + nrows) unless they come from
//                           the embedding, plus aux + s*H + e (e < nrows) with TF_RES_SUM; with
//                           TF_COMBINE, instead of its input vector, the (m, l) pairs and the outputs of
//                           every context split active at the step's position;
//                   writes  [out_off, out_off + nrows) (the LM head writes logits, not words)
//   attention task  reads   the packed queries of its KV head, and on the split that owns the step's
//                           position also that head's current K and V words; a split that starts past
//                           the position does nothing;
//                   writes  its split's outputs and (m, l) pairs, or with TF_WO its partial O-projection
//                           rows [out_off, out_off + nrows)
// Readiness only grows within a step (a word once written stays written), so running any ready task
// until none is left decides whether the plan can deadlock: if tasks remain, some CTA's next task waits
// for a word that no task will write before it, whatever the timing on the GPU.
#include <stdint.h>

#include <algorithm>
#include <cstdlib>
#include <string>
#include <vector>

#include "mbk.h"
#include "mbk_sched.h"

namespace mbk {
namespace {

struct Access {
  std::vector<uint64_t> reads, writes;
};

void add_range(std::vector<uint64_t>& v, uint64_t a, uint64_t n) {
  for (uint64_t i = 0; i < n; ++i) v.push_back(a + i);
}

Access access_of(const PlanShape& s, const Plan& p, const Task& t, int pos) {
  Access x;
  const uint64_t qd = (uint64_t)s.nq * s.d, kvd = (uint64_t)s.nkv * s.d, g = (uint64_t)(s.nq / s.nkv);
  const uint64_t lw = (uint64_t)t.layer * p.act.per_layer;
  if (t.type == T_ATTN) {
    const bool wo = (t.flags & TF_WO) != 0;
    const uint64_t kvh = wo ? t.aux : t.row0;
    const int sp = wo ? 0 : (int)t.nrows;
    if ((int64_t)sp * p.split_len > pos) return x;  // inactive split
    const bool owner = pos / p.split_len == sp;
    add_range(x.reads, lw + p.act.qkv + kvh * g * s.d, g * s.d);
    if (owner) {
      add_range(x.reads, lw + p.act.qkv + qd + kvh * s.d, s.d);
      add_range(x.reads, lw + p.act.qkv + qd + kvd + kvh * s.d, s.d);
    }
    if (wo) {
      add_range(x.writes, t.out_off, t.nrows);
    } else {
      add_range(x.writes, lw + p.act.att + ((uint64_t)sp * s.nq + kvh * g) * s.d, g * s.d);
      add_range(x.writes, lw + p.act.att + (uint64_t)p.nsplit * qd + ((uint64_t)sp * s.nq + kvh * g) * 2, 2 * g);
    }
    return x;
  }
  const unsigned f = t.flags;
  if (f & TF_COMBINE) {
    const uint64_t nact = (uint64_t)(pos / p.split_len + 1);
    add_range(x.reads, lw + p.act.att + (uint64_t)p.nsplit * qd, nact * s.nq * 2);
    for (uint64_t sp = 0; sp < nact; ++sp) add_range(x.reads, lw + p.act.att + sp * qd, qd);
  } else {
    if (!(f & TF_IN_EMB)) add_range(x.reads, t.in_off, t.in_n);
    if (f & TF_IN_SUM)
      for (int sh = 0; sh < s.nkv; ++sh) add_range(x.reads, t.aux + (uint64_t)sh * s.H, t.in_n);
  }
  if (f & TF_RES) {
    if (!(f & TF_RES_EMB)) add_range(x.reads, t.res_off, t.nrows);
    if (f & TF_RES_SUM)
      for (int sh = 0; sh < s.nkv; ++sh) add_range(x.reads, t.aux + (uint64_t)sh * s.H, t.nrows);
  }
  if (t.type != T_LMHEAD) add_range(x.writes, t.out_off, t.nrows);
  return x;
}

}  // namespace
}  // namespace mbk

using namespace mbk;

extern "C" int mbk_plan_simulate(const mbk_config* cfg, int num_sms, int position, mbk_sim_info* info) {
  if (!cfg || !info || num_sms <= 0 || position < 0 || position >= cfg->kv_capacity) return MBK_ERR_INVALID_ARG;
  PlanShape s;
  s.L = cfg->n_layers;
  s.H = cfg->hidden;
  s.I = cfg->intermediate;
  s.nq = cfg->n_heads;
  s.nkv = cfg->n_kv_heads;
  s.d = cfg->head_dim;
  s.V = cfg->vocab;
  s.C = cfg->kv_capacity;
  s.qkv_bias = cfg->qkv_bias ? 1 : 0;
  s.wb = cfg->weight_format == MBK_WEIGHTS_FP8 ? 1 : 2;
  if (!validate_shape(s).empty()) return MBK_ERR_INVALID_ARG;
  PlanOptions opt;
  if (const char* e = std::getenv("MBK_MAX_TASKS_PER_OP")) opt.max_tasks_per_op = std::atoi(e);
  if (const char* e = std::getenv("MBK_FUSE_ATTENTION")) opt.fuse_attention = std::atoi(e);
  if (const char* e = std::getenv("MBK_ATTN_MMA")) opt.attn_mma = std::atoi(e);
  if (const char* e = std::getenv("MBK_ATTN_SPLIT")) opt.attn_split = std::atoi(e);
  if (const char* e = std::getenv("MBK_COMBINE_TASKS")) opt.combine_tasks = std::atoi(e);
  Plan p;
  if (!build_plan(s, fake_weight_addrs(s), num_sms, opt, &p).empty()) return MBK_ERR_STATE;
  // the same host-side fault injection as a handle: one task dropped from its CTA's list
  if (const char* e = std::getenv("MBK_DEBUG_DROP_TASK")) {
    const int drop = std::atoi(e);
    if (drop >= 0 && drop < (int)p.tasks.size()) {
      p.tasks.erase(p.tasks.begin() + drop);
      for (uint32_t& o : p.task_off)
        if (o > (uint32_t)drop) --o;
    }
  }

  const size_t nt = p.tasks.size();
  std::vector<Access> acc(nt);
  for (size_t i = 0; i < nt; ++i) acc[i] = access_of(s, p, p.tasks[i], position);
  // writer and depth of every word; depths of tasks
  std::vector<int32_t> writer(p.act_words, -1);
  std::vector<int> xdepth(nt, 0), sdepth(nt, 0);
  std::vector<uint32_t> next(p.task_off.begin(), p.task_off.end() - 1);  // per CTA: next task
  int64_t run = 0, multiply_written = 0;
  int xmax = 0, smax = 0;
  for (bool progress = true; progress;) {
    progress = false;
    for (int c = 0; c < p.num_ctas; ++c) {
      while (next[c] < p.task_off[c + 1]) {
        const uint32_t i = next[c];
        bool ready = true;
        int xd = 0, sd = i > p.task_off[c] ? sdepth[i - 1] : 0;
        for (uint64_t w : acc[i].reads) {
          if (w >= p.act_words || writer[w] < 0) {
            ready = false;
            break;
          }
          xd = std::max(xd, xdepth[writer[w]]);
          sd = std::max(sd, sdepth[writer[w]]);
        }
        if (!ready) break;
        xdepth[i] = xd + 1;
        sdepth[i] = sd + 1;
        xmax = std::max(xmax, xdepth[i]);
        smax = std::max(smax, sdepth[i]);
        for (uint64_t w : acc[i].writes) {
          if (w >= p.act_words) return MBK_ERR_STATE;
          if (writer[w] >= 0) ++multiply_written;
          writer[w] = (int32_t)i;
        }
        ++next[c];
        ++run;
        progress = true;
      }
    }
  }
  info->tasks_total = (int)nt;
  info->tasks_run = (int)run;
  info->exchange_depth = xmax;
  info->schedule_depth = smax;
  info->words_written_twice = multiply_written;
  info->stuck_cta = -1;
  info->stuck_task_type = 0;
  info->stuck_layer = -1;
  info->stuck_word = -1;
  for (int c = 0; c < p.num_ctas && info->stuck_cta < 0; ++c)
    if (next[c] < p.task_off[c + 1]) {
      const uint32_t i = next[c];
      info->stuck_cta = c;
      info->stuck_task_type = p.tasks[i].type;
      info->stuck_layer = p.tasks[i].layer;
      for (uint64_t w : acc[i].reads)
        if (w >= p.act_words || writer[w] < 0) {
          info->stuck_word = (int64_t)w;
          break;
        }
    }
  return (run == (int64_t)nt && multiply_written == 0) ? MBK_OK : MBK_ERR_STATE;
}
