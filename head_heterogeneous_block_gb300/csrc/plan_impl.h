// Internal: the sa_plan object and the host-side planning routines.
#pragma once

#include <cstdint>
#include <vector>

#include "sparse_attn.h"

struct sa_plan {
  sa_shape shape{};
  int32_t nb = 0;
  int32_t group = 1;              // G = Hq / Hkv
  int32_t num_workers = 0;        // 0 for decode plans
  int32_t schedule = SA_SCHED_LPT;
  int32_t kmax = 0;
  int32_t k_uniform = 0;
  int32_t window_blocks = 0;
  int32_t group_shared = 0;       // one block list per KV group
  int32_t paired = 0;             // group-shared, even G: items are head pairs
  int64_t total_blocks = 0;
  int64_t makespan = 0;
  std::vector<int32_t> budgets;   // [Hq]
  std::vector<uint8_t> kinds;     // [Hq]
  // decode: tokens per selection block of each head (streaming heads: B), the
  // distinct sizes of the retrieval heads (ascending) and the score row stride
  std::vector<int32_t> gran;      // [Hq]
  std::vector<int32_t> sizes;
  int32_t score_stride = 0;
  std::vector<int32_t> wptr;      // [W+1]
  std::vector<int32_t> items;     // [N]
  std::vector<int64_t> loads;     // [W]
  // device copy (sparse_attn_plan_upload)
  int device = -1;
  int32_t* d_budgets = nullptr;
  uint8_t* d_kinds = nullptr;
  int32_t* d_gran = nullptr;      // decode: [Hq]
  int32_t* d_wptr = nullptr;
  int32_t* d_items = nullptr;
  int32_t* d_scratch = nullptr;   // sparse_attn_plan_rebuild: 3N int32
  // decode: head indices by kind, streaming heads first ([Hq]), and how many
  // are streaming (sparse_attn_select_kind / sparse_attn_forward_kind)
  int32_t* d_kind_heads = nullptr;
  int32_t n_streaming = 0;
};

namespace sa_host {

// Max-Min budget shifting; returns the per-head budgets.
std::vector<int32_t> maxmin_shift(int32_t k_uniform, const int32_t* demand, int32_t heads,
                                  int32_t k_min, int32_t nb);

// Work lists for the persistent workers (see sparse_attn_plan in the header).
void build_schedule(const std::vector<int32_t>& budgets, int32_t nb, int32_t group,
                    int32_t workers, int32_t policy, std::vector<int32_t>& wptr,
                    std::vector<int32_t>& items, std::vector<int64_t>& loads);

// Validation shared by the entry points.  Returns SA_OK or the error.
sa_status check_shape(const sa_shape* shp);
sa_status check_supported(const sa_shape* shp);

}  // namespace sa_host
