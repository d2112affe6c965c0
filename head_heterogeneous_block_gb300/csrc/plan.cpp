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
  // item (h, i) has id h*nb + i and costs min(k_h, i+1) blocks
  std::vector<int32_t> item_cost(n);
  for (int32_t h = 0; h < heads; ++h)
    for (int32_t i = 0; i < nb; ++i) item_cost[int64_t(h) * nb + i] = std::min(budgets[h], i + 1);
  auto cost = [&](int32_t id) -> int32_t { return item_cost[id]; };
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

  // Walk order: cost descending, ties by id; LPT_GROUPED first by KV group,
  // and its ties by query block, then head (so a group's heads with equal
  // budgets reach each query block together and share its K/V in L2).
  // Costs are integers in [0, nb], so a stable counting sort over the key
  // (group, nb - cost) -- the group part only for LPT_GROUPED -- walking the
  // ids in the tie order gives exactly that order in linear time.
  std::vector<int32_t> order(n);
  {
    const int32_t ngroups = policy == SA_SCHED_LPT_GROUPED ? (heads + group - 1) / group : 1;
    const int64_t nkeys = int64_t(ngroups) * (nb + 1);
    std::vector<int64_t> start(nkeys + 1, 0);
    std::vector<int64_t> keys(n);
    for (int32_t h = 0; h < heads; ++h) {
      const int64_t base = policy == SA_SCHED_LPT_GROUPED ? int64_t(h / group) * (nb + 1) : 0;
      for (int32_t i = 0; i < nb; ++i) {
        const int64_t id = int64_t(h) * nb + i;
        keys[id] = base + (nb - std::max(0, std::min(item_cost[id], nb)));
      }
    }
    for (int64_t id = 0; id < n; ++id) ++start[keys[id] + 1];
    for (int64_t k = 0; k < nkeys; ++k) start[k + 1] += start[k];
    if (policy == SA_SCHED_LPT_GROUPED) {
      for (int32_t i = 0; i < nb; ++i)
        for (int32_t h = 0; h < heads; ++h) {
          const int64_t id = int64_t(h) * nb + i;
          order[start[keys[id]]++] = int32_t(id);
        }
    } else {
      for (int64_t id = 0; id < n; ++id) order[start[keys[id]]++] = int32_t(id);
    }
  }

  // Least-loaded worker first; equal loads go to the lower worker id.  The
  // walk is a sequence of runs of equal cost c, and a run of r items is
  // placed at once: its choices are the r smallest pairs (value, worker)
  // among the sequences L_w + m*c (m >= 0) -- every step takes the smallest
  // head of those sequences and moves that worker's head up by c.  A binary
  // search finds the value V of the r-th pair; worker w takes its pairs below
  // V, plus one at V if it is among the first workers (by id) with a pair
  // there.  A pair's value is q*c + (L_w mod c) at level q = L_w / c + m, so
  // the pairs in (value, worker) order are the levels in turn, each over the
  // workers ordered by (L_w mod c, w): the k-th item of the run goes to the
  // worker of the k-th pair.
  std::vector<int32_t> owner(n);
  std::vector<int32_t> count(workers, 0);
  std::vector<int64_t> L(workers, 0), take(workers, 0), Lq(workers), Lr(workers);
  std::vector<int32_t> act;
  act.reserve(workers);
  int64_t placed = 0;                         // sum of the loads
  for (int64_t r0 = 0; r0 < n;) {
    const int64_t c = cost(order[r0]);
    int64_t r1 = r0;
    while (r1 < n && cost(order[r1]) == c) ++r1;
    const int64_t r = r1 - r0;
    if (c <= 0) {
      // zero cost: every item goes to the least-loaded worker
      int32_t w0 = 0;
      for (int32_t w = 1; w < workers; ++w)
        if (L[w] < L[w0]) w0 = w;
      for (int64_t k = r0; k < r1; ++k) owner[k] = w0;
      count[w0] += int32_t(r);
      r0 = r1;
      continue;
    }
    // L_w = Lq_w * c + Lr_w; worker w has max(0, Vq - Lq_w + [Vr > Lr_w]) pairs
    // below V = Vq * c + Vr
    for (int32_t w = 0; w < workers; ++w) {
      Lq[w] = L[w] / c;
      Lr[w] = L[w] - Lq[w] * c;
    }
    auto below = [&](int64_t V) {
      const int64_t Vq = V / c, Vr = V - Vq * c;
      int64_t t = 0;
      for (int32_t w = 0; w < workers; ++w)
        t += std::max<int64_t>(0, Vq - Lq[w] + (Vr > Lr[w] ? 1 : 0));
      return t;
    };
    int64_t mn = L[0];
    for (int32_t w = 1; w < workers; ++w) mn = std::min(mn, L[w]);
    // below(lo) = 0 < r <= below(hi), since below(V) >= sum_w (V - L_w) / c
    int64_t lo = mn, hi = std::min(mn + r * c, (placed + r * c + workers - 1) / workers);
    while (hi - lo > 1) {
      const int64_t mid = lo + (hi - lo) / 2;
      if (below(mid) < r) lo = mid;
      else hi = mid;
    }
    const int64_t V = lo;                     // the value of the r-th pair
    int64_t extra = r - below(V);             // pairs taken at exactly V
    act.clear();
    const int64_t Vq = V / c, Vr = V - Vq * c;
    for (int32_t w = 0; w < workers; ++w) {
      int64_t t = std::max<int64_t>(0, Vq - Lq[w] + (Vr > Lr[w] ? 1 : 0));
      if (extra > 0 && Vr == Lr[w] && Vq >= Lq[w]) {
        ++t;
        --extra;
      }
      take[w] = t;
      if (t) act.push_back(w);
    }
    std::stable_sort(act.begin(), act.end(),
                     [&](int32_t x, int32_t y) { return Lr[x] < Lr[y]; });
    int64_t qlo = INT64_MAX, qhi = 0;
    for (int32_t w : act) {
      qlo = std::min(qlo, Lq[w]);
      qhi = std::max(qhi, Lq[w] + take[w] - 1);
    }
    int64_t pos = r0;
    for (int64_t q = qlo; q <= qhi && pos < r1; ++q)
      for (int32_t w : act)
        if (Lq[w] <= q && q < Lq[w] + take[w] && pos < r1) owner[pos++] = w;
    for (int32_t w : act) {
      L[w] += take[w] * c;
      count[w] += int32_t(take[w]);
    }
    placed += r * c;
    r0 = r1;
  }
  for (int32_t w = 0; w < workers; ++w) loads[w] = L[w];
  // CSR by worker, each list in assignment order.
  for (int32_t w = 0; w < workers; ++w) wptr[w + 1] = wptr[w] + count[w];
  std::vector<int32_t> fill(wptr.begin(), wptr.end() - 1);
  for (int64_t r = 0; r < n; ++r) items[fill[owner[r]]++] = order[r];
  if (policy == SA_SCHED_LPT_GROUPED) {
    // Each worker runs its items by KV group, query block, then head: the
    // assignment (and every load) is the greedy's, but all workers now sweep
    // a group's query blocks together, so the blocks each sweep reads are
    // still in L2 when the group's other heads need them.
    for (int32_t w = 0; w < workers; ++w)
      std::sort(items.begin() + wptr[w], items.begin() + wptr[w + 1],
                [&](int32_t a, int32_t b) {
                  const int32_t ha = a / nb, hb = b / nb;
                  if (ha / group != hb / group) return ha / group < hb / group;
                  if (a - ha * nb != b - hb * nb) return a - ha * nb < b - hb * nb;
                  return ha < hb;
                });
  }
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
      plan->group_shared = p->group_shared;
      if (!p->group_shared) {
        plan->budgets = sa_host::maxmin_shift(p->k_uniform, p->demand, H, p->k_min, nb);
      } else {
        // one list per KV group: the budget is shifted between groups, each
        // demanding what its most demanding head demands (the totals stay
        // Hkv * k_uniform per group and Hq * k_uniform per head)
        const int32_t Hkv = shp->num_kv_heads, G = plan->group;
        std::vector<int32_t> g_demand;
        if (p->demand) {
          g_demand.assign(Hkv, 0);
          for (int32_t h = 0; h < H; ++h) g_demand[h / G] = std::max(g_demand[h / G], p->demand[h]);
        }
        const std::vector<int32_t> k_g = sa_host::maxmin_shift(
            p->k_uniform, p->demand ? g_demand.data() : nullptr, Hkv, p->k_min, nb);
        plan->budgets.resize(H);
        for (int32_t h = 0; h < H; ++h) plan->budgets[h] = k_g[h / G];
      }
      plan->num_workers = p->num_workers;
      if (p->share_kv != 0 && (p->share_kv != 1 || !p->group_shared || plan->group % 2 != 0)) {
        delete plan;
        return SA_ERR_INVALID_ARG;
      }
      if (p->share_kv) {
        // the two heads of a pair share their list: the work item is (pair,
        // query block), costing both heads' blocks; the greedy runs on the
        // pairs' budgets, G/2 pairs per KV group
        plan->paired = 1;
        std::vector<int32_t> pair_budgets(H / 2);
        for (int32_t x = 0; x < H / 2; ++x) pair_budgets[x] = plan->budgets[2 * x];
        sa_host::build_schedule(pair_budgets, nb, plan->group / 2, p->num_workers, p->schedule,
                                plan->wptr, plan->items, plan->loads);
        for (int64_t& l : plan->loads) l *= 2;
      } else {
        sa_host::build_schedule(plan->budgets, nb, plan->group, p->num_workers, p->schedule,
                                plan->wptr, plan->items, plan->loads);
      }
      plan->kmax = 0;
      for (int32_t k : plan->budgets) plan->kmax = std::max(plan->kmax, std::min(k, nb));
      plan->total_blocks = 0;
      plan->makespan = 0;
      for (int64_t l : plan->loads) {
        plan->total_blocks += l;
        plan->makespan = std::max(plan->makespan, l);
      }
    } else {
      if (p->demand || p->group_shared || p->share_kv) { delete plan; return SA_ERR_INVALID_ARG; }
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
                     ? int32_t(plan->items.size())   // Hq*nb, or Hq/2*nb head pairs
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
