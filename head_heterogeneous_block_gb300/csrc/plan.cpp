// Host-side planning: per-head budgets and the persistent workers' schedule.
//
// Budgets follow S-HPLB's Max-Min budget shifting and the schedule its greedy
// longest-first multiway partition ("S-HPLB: Efficient LLM Attention Serving
// via Sparsity-Aware Head Parallelism Load Balance", Italian summary,
// "Metodologia" A and B; Chinese summary 2.1 and 2.2).  S-HPLB places heads
// on GPUs; here the workers are persistent CTAs on one GPU and the items are
// (head, query-block) pairs, each costing the blocks it attends.
// Everything in this file is integer host code with no CUDA call.

#include <algorithm>
#include <cstring>
#include <functional>
#include <new>
#include <queue>
#include <utility>

#include "plan_impl.h"

namespace sa_host {

sa_status check_shape(const sa_shape* shp) {
  if (!shp) return SA_ERR_INVALID_ARG;
  if (shp->mode != SA_MODE_PREFILL && shp->mode != SA_MODE_DECODE) return SA_ERR_INVALID_ARG;
  if (shp->seq_len <= 0 || shp->block <= 0 || shp->num_q_heads <= 0 ||
      shp->num_kv_heads <= 0 || shp->head_dim <= 0 || shp->batch <= 0)
    return SA_ERR_SHAPE;
  if (shp->seq_len % shp->block != 0) return SA_ERR_SHAPE;
  if (shp->num_q_heads % shp->num_kv_heads != 0) return SA_ERR_SHAPE;
  if (shp->mode == SA_MODE_PREFILL && shp->batch != 1) return SA_ERR_SHAPE;
  const int64_t nb = shp->seq_len / shp->block;
  const int64_t rows = (shp->mode == SA_MODE_PREFILL) ? int64_t(shp->num_q_heads) * nb
                                                      : int64_t(shp->batch) * shp->num_q_heads;
  if (nb > (int64_t(1) << 30) || rows >= (int64_t(1) << 31) ||
      int64_t(shp->num_q_heads) * shp->seq_len >= (int64_t(1) << 31))
    return SA_ERR_SHAPE;
  return SA_OK;
}

sa_status check_supported(const sa_shape* shp) {
  sa_status st = check_shape(shp);
  if (st != SA_OK) return st;
  if (shp->head_dim != 64 && shp->head_dim != 128) return SA_ERR_UNSUPPORTED;
  if (shp->mode == SA_MODE_PREFILL) {
    if (shp->block != 64 && shp->block != 128) return SA_ERR_UNSUPPORTED;
    // B = 64 blocks run on 128-row query tiles; keep d = 64 there.
    if (shp->block == 64 && shp->head_dim != 64) return SA_ERR_UNSUPPORTED;
    if (shp->block == 128 && shp->head_dim != 128) return SA_ERR_UNSUPPORTED;
  } else {
    if (shp->block != 32) return SA_ERR_UNSUPPORTED;
    if (shp->head_dim != 128) return SA_ERR_UNSUPPORTED;
  }
  return SA_OK;
}

std::vector<int32_t> maxmin_shift(int32_t k_uniform, const int32_t* demand, int32_t heads,
                                  int32_t k_min, int32_t nb) {
  std::vector<int32_t> k(heads, k_uniform);
  if (!demand) return k;
  // One block moves per step, from the head with the most budget to spare
  // relative to its demand to the head that is shortest of it.  Surpluses are
  // tracked incrementally; a step changes only two of them.
  std::vector<int64_t> surplus(heads);
  for (int32_t h = 0; h < heads; ++h) surplus[h] = int64_t(k_uniform) - demand[h];
  for (;;) {
    int32_t donor = -1, receiver = -1;
    for (int32_t h = 0; h < heads; ++h) {
      if (k[h] > k_min && (donor < 0 || surplus[h] > surplus[donor])) donor = h;
      if (k[h] < nb && (receiver < 0 || surplus[h] < surplus[receiver])) receiver = h;
    }
    if (donor < 0 || receiver < 0) break;
    if (surplus[donor] - surplus[receiver] <= 1) break;
    --k[donor];
    --surplus[donor];
    ++k[receiver];
    ++surplus[receiver];
  }
  return k;
}

void build_schedule(const std::vector<int32_t>& budgets, int32_t nb, int32_t group,
                    int32_t workers, int32_t policy, std::vector<int32_t>& wptr,
                    std::vector<int32_t>& items, std::vector<int64_t>& loads) {
  const int32_t heads = int32_t(budgets.size());
  const int64_t n = int64_t(heads) * nb;
  auto cost = [&](int32_t id) -> int32_t {
    const int32_t h = id / nb, i = id % nb;
    return std::min(budgets[h], i + 1);
  };
  wptr.assign(workers + 1, 0);
  items.resize(n);
  loads.assign(workers, 0);

  if (policy == SA_SCHED_HEAD_ORDER) {
    for (int32_t w = 0; w < workers; ++w) {
      const int64_t lo = int64_t(w) * n / workers, hi = int64_t(w + 1) * n / workers;
      wptr[w + 1] = int32_t(hi);
      for (int64_t id = lo; id < hi; ++id) {
        items[id] = int32_t(id);
        loads[w] += cost(int32_t(id));
      }
    }
    return;
  }

  // Walk order: cost descending, ties by id; LPT_GROUPED first by KV group.
  std::vector<int32_t> order(n);
  for (int64_t id = 0; id < n; ++id) order[id] = int32_t(id);
  if (policy == SA_SCHED_LPT_GROUPED) {
    std::sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
      const int32_t ga = (a / nb) / group, gb = (b / nb) / group;
      if (ga != gb) return ga < gb;
      const int32_t ca = cost(a), cb = cost(b);
      if (ca != cb) return ca > cb;
      return a < b;
    });
  } else {
    std::sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
      const int32_t ca = cost(a), cb = cost(b);
      if (ca != cb) return ca > cb;
      return a < b;
    });
  }

  // Least-loaded worker first; equal loads go to the lower worker id.
  using Slot = std::pair<int64_t, int32_t>;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int32_t w = 0; w < workers; ++w) heap.push({0, w});
  std::vector<int32_t> owner(n);
  std::vector<int32_t> count(workers, 0);
  for (int64_t r = 0; r < n; ++r) {
    Slot s = heap.top();
    heap.pop();
    owner[r] = s.second;
    ++count[s.second];
    s.first += cost(order[r]);
    loads[s.second] = s.first;
    heap.push(s);
  }
  // CSR by worker, each list in assignment order.
  for (int32_t w = 0; w < workers; ++w) wptr[w + 1] = wptr[w] + count[w];
  std::vector<int32_t> fill(wptr.begin(), wptr.end() - 1);
  for (int64_t r = 0; r < n; ++r) items[fill[owner[r]]++] = order[r];
}

}  // namespace sa_host

extern "C" {

const char* sa_status_string(sa_status status) {
  switch (status) {
    case SA_OK: return "ok";
    case SA_ERR_INVALID_ARG: return "invalid argument";
    case SA_ERR_SHAPE: return "inconsistent shape";
    case SA_ERR_UNSUPPORTED: return "unsupported shape or mode";
    case SA_ERR_CUDA: return "CUDA error";
    case SA_ERR_DEVICE_CHECK: return "device-side check failed";
    case SA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case SA_ERR_NO_MEMORY: return "out of memory";
    case SA_ERR_NOT_UPLOADED: return "plan not uploaded to the device";
  }
  return "unknown status";
}

sa_status sparse_attn_plan(const sa_shape* shp, const sa_plan_params* p, sa_plan** out) {
  if (!shp || !p || !out) return SA_ERR_INVALID_ARG;
  sa_status st = sa_host::check_shape(shp);
  if (st != SA_OK) return st;
  const int32_t nb = int32_t(shp->seq_len / shp->block);
  const int32_t H = shp->num_q_heads;
  if (p->k_min < 2) return SA_ERR_INVALID_ARG;
  // (a single-block sequence keeps its one block under any budget >= k_min)
  if (p->k_uniform < p->k_min || p->k_uniform > std::max(nb, p->k_min)) return SA_ERR_INVALID_ARG;
  if (p->schedule != SA_SCHED_LPT && p->schedule != SA_SCHED_LPT_GROUPED &&
      p->schedule != SA_SCHED_HEAD_ORDER)
    return SA_ERR_INVALID_ARG;
  if (p->demand)
    for (int32_t h = 0; h < H; ++h)
      if (p->demand[h] < 0) return SA_ERR_INVALID_ARG;

  sa_plan* plan = new (std::nothrow) sa_plan();
  if (!plan) return SA_ERR_NO_MEMORY;
  try {
    plan->shape = *shp;
    plan->nb = nb;
    plan->group = H / shp->num_kv_heads;
    plan->schedule = p->schedule;
    plan->k_uniform = p->k_uniform;
    plan->kinds.assign(H, SA_HEAD_RETRIEVAL);
    if (shp->mode == SA_MODE_PREFILL) {
      if (p->head_kind || p->granularity || p->head_budget) { delete plan; return SA_ERR_INVALID_ARG; }
      if (p->num_workers < 1) { delete plan; return SA_ERR_INVALID_ARG; }
      if (p->group_shared != 0 && p->group_shared != 1) { delete plan; return SA_ERR_INVALID_ARG; }
      plan->budgets = sa_host::maxmin_shift(p->k_uniform, p->demand, H, p->k_min, nb);
      plan->group_shared = p->group_shared;
      if (p->group_shared) {
        // a shared list gets the largest of its heads' budgets
        for (int32_t g = 0; g < shp->num_kv_heads; ++g) {
          int32_t k = 0;
          for (int32_t x = 0; x < plan->group; ++x) k = std::max(k, plan->budgets[g * plan->group + x]);
          for (int32_t x = 0; x < plan->group; ++x) plan->budgets[g * plan->group + x] = k;
        }
      }
      plan->num_workers = p->num_workers;
      sa_host::build_schedule(plan->budgets, nb, plan->group, p->num_workers, p->schedule,
                              plan->wptr, plan->items, plan->loads);
      plan->kmax = 0;
      for (int32_t k : plan->budgets) plan->kmax = std::max(plan->kmax, std::min(k, nb));
      plan->total_blocks = 0;
      plan->makespan = 0;
      for (int64_t l : plan->loads) {
        plan->total_blocks += l;
        plan->makespan = std::max(plan->makespan, l);
      }
    } else {
      if (p->demand || p->group_shared) { delete plan; return SA_ERR_INVALID_ARG; }
      bool any_streaming = false;
      if (p->head_kind) {
        for (int32_t h = 0; h < H; ++h) {
          if (p->head_kind[h] != SA_HEAD_RETRIEVAL && p->head_kind[h] != SA_HEAD_STREAMING) {
            delete plan;
            return SA_ERR_INVALID_ARG;
          }
          plan->kinds[h] = p->head_kind[h];
          any_streaming |= p->head_kind[h] == SA_HEAD_STREAMING;
        }
      }
      if (any_streaming && (p->window_blocks < 1 || p->window_blocks > nb)) {
        delete plan;
        return SA_ERR_INVALID_ARG;
      }
      plan->window_blocks = p->window_blocks;
      plan->budgets.resize(H);
      plan->gran.assign(H, shp->block);
      // per-head selection block sizes and budgets of the retrieval heads
      for (int32_t h = 0; h < H; ++h) {
        if (plan->kinds[h] == SA_HEAD_STREAMING) continue;
        if (p->granularity) {
          const int32_t g = p->granularity[h];
          if (g < 16 || g % 16 != 0 || shp->seq_len % g != 0 || shp->seq_len / g > 4096) {
            delete plan;
            return SA_ERR_INVALID_ARG;
          }
          plan->gran[h] = g;
        }
        if (p->head_budget && p->head_budget[h] < p->k_min) {
          delete plan;
          return SA_ERR_INVALID_ARG;
        }
      }
      // streaming: block 0 plus the last window_blocks blocks
      const int32_t stream_count = (nb - p->window_blocks > 0) ? p->window_blocks + 1 : nb;
      plan->kmax = 0;
      plan->total_blocks = 0;
      for (int32_t h = 0; h < H; ++h) {
        if (plan->kinds[h] == SA_HEAD_STREAMING) {
          plan->budgets[h] = stream_count;
        } else if (p->granularity || p->head_budget) {
          const int32_t nbh = int32_t(shp->seq_len / plan->gran[h]);
          plan->budgets[h] = std::min(p->head_budget ? p->head_budget[h] : p->k_uniform, nbh);
        } else {
          plan->budgets[h] = p->k_uniform;
        }
        plan->kmax = std::max(plan->kmax, plan->budgets[h]);
        plan->total_blocks += int64_t(plan->budgets[h]) * shp->batch;
      }
      for (int32_t h = 0; h < H; ++h)
        if (plan->kinds[h] != SA_HEAD_STREAMING) plan->sizes.push_back(plan->gran[h]);
      std::sort(plan->sizes.begin(), plan->sizes.end());
      plan->sizes.erase(std::unique(plan->sizes.begin(), plan->sizes.end()), plan->sizes.end());
      if (plan->sizes.size() > 8) {
        delete plan;
        return SA_ERR_INVALID_ARG;
      }
      plan->score_stride = plan->sizes.empty() ? nb : int32_t(shp->seq_len / plan->sizes[0]);
      plan->num_workers = 0;
      plan->wptr.assign(1, 0);
      plan->makespan = 0;
    }
  } catch (const std::bad_alloc&) {
    delete plan;
    return SA_ERR_NO_MEMORY;
  }
  *out = plan;
  return SA_OK;
}

sa_status sparse_attn_plan_info(const sa_plan* plan, int32_t* num_workers, int32_t* num_items,
                                int32_t* kmax, int64_t* total_blocks, int64_t* makespan) {
  if (!plan) return SA_ERR_INVALID_ARG;
  if (num_workers) *num_workers = plan->num_workers;
  if (num_items)
    *num_items = plan->shape.mode == SA_MODE_PREFILL
                     ? plan->shape.num_q_heads * plan->nb
                     : plan->shape.batch * plan->shape.num_q_heads;
  if (kmax) *kmax = plan->kmax;
  if (total_blocks) *total_blocks = plan->total_blocks;
  if (makespan) *makespan = plan->makespan;
  return SA_OK;
}

sa_status sparse_attn_plan_decode_layout(const sa_plan* plan, int32_t* num_sizes,
                                         int32_t* sizes, int64_t* kcache_floats,
                                         int32_t* score_stride) {
  if (!plan || plan->shape.mode != SA_MODE_DECODE) return SA_ERR_INVALID_ARG;
  const sa_shape& s = plan->shape;
  int64_t floats = 0;
  for (int32_t g : plan->sizes)
    floats += int64_t(s.batch) * s.num_kv_heads * (s.seq_len / g) * s.head_dim;
  if (num_sizes) *num_sizes = int32_t(plan->sizes.size());
  if (sizes)
    for (size_t i = 0; i < plan->sizes.size() && i < 8; ++i) sizes[i] = plan->sizes[i];
  if (kcache_floats) *kcache_floats = floats;
  if (score_stride) *score_stride = plan->score_stride;
  return SA_OK;
}

sa_status sparse_attn_plan_get(const sa_plan* plan, int32_t* budgets, int32_t* wptr,
                               int32_t* items, int64_t* loads) {
  if (!plan) return SA_ERR_INVALID_ARG;
  if (budgets) std::memcpy(budgets, plan->budgets.data(), plan->budgets.size() * sizeof(int32_t));
  if (wptr) std::memcpy(wptr, plan->wptr.data(), plan->wptr.size() * sizeof(int32_t));
  if (items && !plan->items.empty())
    std::memcpy(items, plan->items.data(), plan->items.size() * sizeof(int32_t));
  if (loads && !plan->loads.empty())
    std::memcpy(loads, plan->loads.data(), plan->loads.size() * sizeof(int64_t));
  return SA_OK;
}

}  // extern "C"
