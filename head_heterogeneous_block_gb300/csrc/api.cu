// C ABI entry points that touch the device: plan upload, score, select,
// forward and the decode key-cache pooling.  Arguments are validated on the
// host before anything is launched; the kernels live in score.cu, select.cu,
// prefill.cu and decode.cu.

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <vector>

#include "kernels.h"
#include "plan_impl.h"
#include "sparse_attn.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool same_shape(const sa_shape* a, const sa_shape& b) {
  return a->seq_len == b.seq_len && a->block == b.block && a->num_q_heads == b.num_q_heads &&
         a->num_kv_heads == b.num_kv_heads && a->head_dim == b.head_dim &&
         a->batch == b.batch && a->mode == b.mode;
}

void free_device(sa_plan* p) {
  if (p->device >= 0) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != p->device) cudaSetDevice(p->device);
    cudaFree(p->d_budgets);
    cudaFree(p->d_kinds);
    cudaFree(p->d_gran);
    cudaFree(p->d_wptr);
    cudaFree(p->d_items);
    cudaFree(p->d_scratch);
    cudaFree(p->d_kind_heads);
    if (cur >= 0 && cur != p->device) cudaSetDevice(cur);
  }
  p->d_scratch = nullptr;
  p->d_kind_heads = nullptr;
  p->d_budgets = nullptr;
  p->d_kinds = nullptr;
  p->d_gran = nullptr;
  p->d_wptr = nullptr;
  p->d_items = nullptr;
  p->device = -1;
}

using sa_k::cuda_status;

// Operational wait limit of the prefill forward, in ns (0: the kernel default).
std::atomic<uint64_t> g_wait_ns{0};

int64_t nblocks(const sa_shape* s) { return s->seq_len / s->block; }

// Decode: the largest row a plan's selection handles, in blocks.
int32_t decode_max_row(const sa_plan* p) {
  int32_t row = p->nb;
  for (size_t h = 0; h < p->gran.size(); ++h)
    if (p->kinds[h] != SA_HEAD_STREAMING)
      row = std::max(row, int32_t(p->shape.seq_len / p->gran[h]));
  return row;
}

// Decode: whether any head selects at a size other than B.
bool has_granularity(const sa_plan* p) {
  for (int32_t g : p->gran)
    if (g != p->shape.block) return true;
  return false;
}

}  // namespace

namespace {

// Selection over every row, or (decode) over the rows of the heads in
// `heads` (nh of them); scores may then be NULL when all of them stream.
sa_status select_rows(const sa_shape* shp, const sa_plan* plan, const float* scores,
                      int32_t* idx, int32_t* cnt, int32_t kmax, const int32_t* heads,
                      int32_t nh, bool need_scores, sa_stream_t stream) {
  sa_status s = sa_host::check_supported(shp);
  if (s != SA_OK) return s;
  if (!plan || (need_scores && !scores) || !idx || !cnt) return SA_ERR_INVALID_ARG;
  if (!same_shape(shp, plan->shape)) return SA_ERR_SHAPE;
  if (kmax < plan->kmax) return SA_ERR_SHAPE;
  const bool decode = shp->mode == SA_MODE_DECODE;
  const int32_t max_row = decode ? decode_max_row(plan) : plan->nb;
  if (max_row > (decode ? 4096 : 2048)) return SA_ERR_UNSUPPORTED;
  if (plan->device < 0) return SA_ERR_NOT_UPLOADED;
  sa_k::SelectArgs a;
  a.scores = scores;
  a.budgets = plan->d_budgets;
  a.kinds = plan->d_kinds;
  a.idx = idx;
  a.cnt = cnt;
  a.kmax = kmax;
  a.nb = plan->nb;
  a.Hq = shp->num_q_heads;
  a.decode = shp->mode == SA_MODE_DECODE;
  a.group = plan->group;
  a.group_shared = plan->group_shared;
  a.rows = a.decode ? shp->batch * shp->num_q_heads
                    : (plan->group_shared ? shp->num_kv_heads : shp->num_q_heads) * plan->nb;
  a.window_blocks = plan->window_blocks;
  a.gran = decode ? plan->d_gran : nullptr;
  a.L = int32_t(shp->seq_len);
  a.stride = decode ? plan->score_stride : 0;
  a.max_row = max_row;
  a.heads = heads;
  a.nh = nh;
  if (heads) a.rows = shp->batch * nh;
  return cuda_status(sa_k::launch_select(a, reinterpret_cast<cudaStream_t>(stream)));
}

// Attention over every row, or (decode) over the rows of the heads in `heads`.
sa_status forward_rows(const sa_shape* shp, const sa_plan* plan, const void* q, const void* k,
                       const void* v, const int32_t* idx, const int32_t* cnt, int32_t kmax,
                       void* o, int32_t o_dtype, float* lse, int32_t* dev_status,
                       const int32_t* heads, int32_t nh, sa_stream_t stream) {
  sa_status s = sa_host::check_supported(shp);
  if (s != SA_OK) return s;
  if (!q || !k || !v || !idx || !cnt || !o || !dev_status || kmax < 1) return SA_ERR_INVALID_ARG;
  if (o_dtype != SA_DTYPE_BF16 && o_dtype != SA_DTYPE_F32) return SA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return SA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (shp->mode == SA_MODE_DECODE) {
    if (plan && !same_shape(shp, plan->shape)) return SA_ERR_SHAPE;
    const bool sized = plan && has_granularity(plan);
    if (sized && plan->device < 0) return SA_ERR_NOT_UPLOADED;
    sa_k::DecodeArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.idx = idx;
    a.cnt = cnt;
    a.kmax = kmax;
    a.Bt = shp->batch;
    a.Hq = shp->num_q_heads;
    a.Hkv = shp->num_kv_heads;
    a.L = int(shp->seq_len);
    a.B = shp->block;
    a.d = shp->head_dim;
    a.o = o;
    a.out_f32 = o_dtype == SA_DTYPE_F32;
    a.lse = lse;
    a.dev_status = dev_status;
    a.gran = sized ? plan->d_gran : nullptr;
    a.heads = heads;
    a.nh = nh;
    a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    return cuda_status(sa_k::launch_decode_attention(a, st));
  }
  if (!plan) return SA_ERR_INVALID_ARG;
  if (!same_shape(shp, plan->shape)) return SA_ERR_SHAPE;
  if (plan->device < 0) return SA_ERR_NOT_UPLOADED;
  sa_k::PrefillArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.idx = idx;
  a.cnt = cnt;
  a.kmax = kmax;
  a.wptr = plan->d_wptr;
  a.items = plan->d_items;
  a.num_workers = plan->num_workers;
  a.num_items = (plan->paired ? shp->num_q_heads / 2 : shp->num_q_heads) * plan->nb;
  a.S = int(shp->seq_len);
  a.B = shp->block;
  a.d = shp->head_dim;
  a.Hq = shp->num_q_heads;
  a.Hkv = shp->num_kv_heads;
  a.o = o;
  a.out_f32 = o_dtype == SA_DTYPE_F32;
  a.lse = lse;
  a.dev_status = dev_status;
  a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  bool encode_failed = false;
  cudaError_t e = plan->paired ? sa_k::launch_prefill_attention_pairs(a, st, &encode_failed)
                               : sa_k::launch_prefill_attention(a, st, &encode_failed);
  if (encode_failed) return SA_ERR_CUDA;
  return cuda_status(e);
}

}  // namespace

extern "C" {

sa_status sparse_attn_plan_upload(sa_plan* plan, sa_stream_t stream) {
  if (!plan) return SA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  free_device(plan);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SA_ERR_CUDA;
  const size_t nh = plan->budgets.size();
  const size_t nw = plan->wptr.size();
  const size_t ni = plan->items.size();
  const size_t ng = plan->gran.size();
  // decode: head indices by kind, streaming heads first
  std::vector<int32_t> kind_heads;
  if (plan->shape.mode == SA_MODE_DECODE) {
    for (size_t h = 0; h < plan->kinds.size(); ++h)
      if (plan->kinds[h] == SA_HEAD_STREAMING) kind_heads.push_back(int32_t(h));
    plan->n_streaming = int32_t(kind_heads.size());
    for (size_t h = 0; h < plan->kinds.size(); ++h)
      if (plan->kinds[h] != SA_HEAD_STREAMING) kind_heads.push_back(int32_t(h));
  }
  cudaError_t e = cudaMalloc(&plan->d_budgets, nh * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMalloc(&plan->d_kinds, nh);
  if (e == cudaSuccess && ng) e = cudaMalloc(&plan->d_gran, ng * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMalloc(&plan->d_wptr, nw * sizeof(int32_t));
  if (e == cudaSuccess && ni) e = cudaMalloc(&plan->d_items, ni * sizeof(int32_t));
  if (e == cudaSuccess && !kind_heads.empty())
    e = cudaMalloc(&plan->d_kind_heads, kind_heads.size() * sizeof(int32_t));
  plan->device = dev;
  if (e != cudaSuccess) {
    free_device(plan);
    return cuda_status(e);
  }
  e = cudaMemcpyAsync(plan->d_budgets, plan->budgets.data(), nh * sizeof(int32_t),
                      cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(plan->d_kinds, plan->kinds.data(), nh, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess && ng)
    e = cudaMemcpyAsync(plan->d_gran, plan->gran.data(), ng * sizeof(int32_t),
                        cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(plan->d_wptr, plan->wptr.data(), nw * sizeof(int32_t),
                        cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess && ni)
    e = cudaMemcpyAsync(plan->d_items, plan->items.data(), ni * sizeof(int32_t),
                        cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess && !kind_heads.empty())
    e = cudaMemcpyAsync(plan->d_kind_heads, kind_heads.data(),
                        kind_heads.size() * sizeof(int32_t), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    free_device(plan);
    return cuda_status(e);
  }
  return SA_OK;
}

void sparse_attn_plan_destroy(sa_plan* plan) {
  if (!plan) return;
  free_device(plan);
  delete plan;
}

sa_status sparse_attn_score_workspace_size(const sa_shape* shp, size_t* bytes) {
  if (!bytes) return SA_ERR_INVALID_ARG;
  sa_status st = sa_host::check_shape(shp);
  if (st != SA_OK) return st;
  if (shp->mode == SA_MODE_DECODE) {
    *bytes = 0;
    return SA_OK;
  }
  const size_t n = size_t(shp->num_q_heads + shp->num_kv_heads) * size_t(nblocks(shp)) *
                   size_t(shp->head_dim) * sizeof(float);
  *bytes = (n + 255) & ~size_t(255);
  return SA_OK;
}

sa_status sparse_attn_score(const sa_shape* shp, const void* q, const void* k, float* scores,
                            void* ws, size_t ws_bytes, sa_stream_t stream) {
  sa_status s = sa_host::check_supported(shp);
  if (s != SA_OK) return s;
  if (!q || !k || !scores) return SA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(scores)) return SA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int nb = int(nblocks(shp));
  const int d = shp->head_dim;
  const int G = shp->num_q_heads / shp->num_kv_heads;
  const float scale = float(1.0 / std::sqrt(double(d)));
  if (shp->mode == SA_MODE_DECODE) {
    return cuda_status(sa_k::launch_decode_scores(q, static_cast<const float*>(k), scores,
                                                  shp->batch, shp->num_q_heads, G, nb, d, scale,
                                                  st));
  }
  size_t need = 0;
  sparse_attn_score_workspace_size(shp, &need);
  if (!ws || ws_bytes < need || !aligned16(ws)) return SA_ERR_INVALID_ARG;
  return cuda_status(sa_k::launch_prefill_index(q, k, scores, static_cast<float*>(ws),
                                                shp->num_q_heads, shp->num_kv_heads, nb,
                                                shp->block, d, st));
}

sa_status sparse_attn_select(const sa_shape* shp, const sa_plan* plan, const float* scores,
                             int32_t* idx, int32_t* cnt, int32_t kmax, sa_stream_t stream) {
  return select_rows(shp, plan, scores, idx, cnt, kmax, nullptr, 0, true, stream);
}

sa_status sparse_attn_select_kind(const sa_shape* shp, const sa_plan* plan, const float* scores,
                                  int32_t* idx, int32_t* cnt, int32_t kmax, int32_t head_kind,
                                  sa_stream_t stream) {
  if (!shp || !plan || shp->mode != SA_MODE_DECODE) return SA_ERR_INVALID_ARG;
  if (head_kind != SA_HEAD_STREAMING && head_kind != SA_HEAD_RETRIEVAL) return SA_ERR_INVALID_ARG;
  if (plan->device < 0) return SA_ERR_NOT_UPLOADED;
  const bool streaming = head_kind == SA_HEAD_STREAMING;
  const int32_t nh = streaming ? plan->n_streaming
                               : int32_t(plan->kinds.size()) - plan->n_streaming;
  if (nh == 0) return SA_OK;
  const int32_t* heads = plan->d_kind_heads + (streaming ? 0 : plan->n_streaming);
  return select_rows(shp, plan, scores, idx, cnt, kmax, heads, nh, !streaming, stream);
}

sa_status sparse_attn_select_topp(const sa_shape* shp, const sa_plan* plan, const float* scores,
                                  float p, int32_t* idx, int32_t* cnt, int32_t kmax,
                                  sa_stream_t stream) {
  sa_status s = sa_host::check_supported(shp);
  if (s != SA_OK) return s;
  if (!plan || !scores || !idx || !cnt || !(p == p)) return SA_ERR_INVALID_ARG;
  if (shp->mode != SA_MODE_PREFILL) return SA_ERR_INVALID_ARG;
  if (!same_shape(shp, plan->shape)) return SA_ERR_SHAPE;
  if (kmax < plan->nb) return SA_ERR_SHAPE;
  if (plan->nb > 2048) return SA_ERR_UNSUPPORTED;
  if (plan->device < 0) return SA_ERR_NOT_UPLOADED;
  sa_k::TopPArgs a;
  a.scores = scores;
  a.idx = idx;
  a.cnt = cnt;
  a.kmax = kmax;
  a.nb = plan->nb;
  a.rows = shp->num_q_heads * plan->nb;
  a.p = p;
  return cuda_status(sa_k::launch_select_topp(a, reinterpret_cast<cudaStream_t>(stream)));
}

sa_status sparse_attn_plan_rebuild(sa_plan* plan, const int32_t* cnt, sa_stream_t stream) {
  if (!plan || !cnt) return SA_ERR_INVALID_ARG;
  if (plan->shape.mode != SA_MODE_PREFILL || plan->group_shared) return SA_ERR_INVALID_ARG;
  if (plan->device < 0) return SA_ERR_NOT_UPLOADED;
  if (plan->num_workers > 256 || plan->nb > 2048) return SA_ERR_UNSUPPORTED;
  if (plan->items.size() > (size_t(1) << 19)) return SA_ERR_UNSUPPORTED;
  const int32_t n = int32_t(plan->items.size());
  if (!plan->d_scratch) {
    cudaError_t e = cudaMalloc(&plan->d_scratch, size_t(3) * std::max(n, 1) * sizeof(int32_t));
    if (e != cudaSuccess) return cuda_status(e);
  }
  sa_k::RebuildArgs a;
  a.cnt = cnt;
  a.wptr = plan->d_wptr;
  a.items = plan->d_items;
  a.scratch = plan->d_scratch;
  a.num_items = n;
  a.num_workers = plan->num_workers;
  return cuda_status(sa_k::launch_lpt_rebuild(a, reinterpret_cast<cudaStream_t>(stream)));
}

sa_status sparse_attn_plan_device_schedule(const sa_plan* plan, int32_t* wptr, int32_t* items,
                                           sa_stream_t stream) {
  if (!plan || !wptr || !items) return SA_ERR_INVALID_ARG;
  if (plan->device < 0) return SA_ERR_NOT_UPLOADED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(wptr, plan->d_wptr, plan->wptr.size() * sizeof(int32_t),
                                  cudaMemcpyDefault, st);
  if (e == cudaSuccess && !plan->items.empty())
    e = cudaMemcpyAsync(items, plan->d_items, plan->items.size() * sizeof(int32_t),
                        cudaMemcpyDefault, st);
  return cuda_status(e);
}

sa_status sparse_attn_forward(const sa_shape* shp, const sa_plan* plan, const void* q,
                              const void* k, const void* v, const int32_t* idx,
                              const int32_t* cnt, int32_t kmax, void* o, int32_t o_dtype,
                              float* lse, int32_t* dev_status, sa_stream_t stream) {
  return forward_rows(shp, plan, q, k, v, idx, cnt, kmax, o, o_dtype, lse, dev_status, nullptr, 0,
                      stream);
}

sa_status sparse_attn_forward_kind(const sa_shape* shp, const sa_plan* plan, const void* q,
                                   const void* k, const void* v, const int32_t* idx,
                                   const int32_t* cnt, int32_t kmax, void* o, int32_t o_dtype,
                                   float* lse, int32_t* dev_status, int32_t head_kind,
                                   sa_stream_t stream) {
  if (!shp || !plan || shp->mode != SA_MODE_DECODE) return SA_ERR_INVALID_ARG;
  if (head_kind != SA_HEAD_STREAMING && head_kind != SA_HEAD_RETRIEVAL) return SA_ERR_INVALID_ARG;
  if (plan->device < 0) return SA_ERR_NOT_UPLOADED;
  const bool streaming = head_kind == SA_HEAD_STREAMING;
  const int32_t nh = streaming ? plan->n_streaming
                               : int32_t(plan->kinds.size()) - plan->n_streaming;
  if (nh == 0) return SA_OK;
  const int32_t* heads = plan->d_kind_heads + (streaming ? 0 : plan->n_streaming);
  return forward_rows(shp, plan, q, k, v, idx, cnt, kmax, o, o_dtype, lse, dev_status, heads, nh,
                      stream);
}

sa_status sparse_attn_set_wait_limit(uint64_t ns) {
  g_wait_ns.store(ns, std::memory_order_relaxed);
  return SA_OK;
}

sa_status sparse_attn_pool_kcache(const sa_shape* shp, const void* k, float* kbar,
                                  sa_stream_t stream) {
  sa_status s = sa_host::check_supported(shp);
  if (s != SA_OK) return s;
  if (shp->mode != SA_MODE_DECODE) return SA_ERR_INVALID_ARG;
  if (!k || !kbar || !aligned16(k) || !aligned16(kbar)) return SA_ERR_INVALID_ARG;
  const int64_t rows = int64_t(shp->batch) * shp->num_kv_heads * nblocks(shp);
  return cuda_status(sa_k::launch_pool(k, kbar, rows, shp->block, shp->head_dim,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

sa_status sparse_attn_pool_kcache_plan(const sa_shape* shp, const sa_plan* plan, const void* k,
                                       float* kbar_all, sa_stream_t stream) {
  sa_status s = sa_host::check_supported(shp);
  if (s != SA_OK) return s;
  if (!plan || shp->mode != SA_MODE_DECODE) return SA_ERR_INVALID_ARG;
  if (!same_shape(shp, plan->shape)) return SA_ERR_SHAPE;
  if (!k || !kbar_all || !aligned16(k) || !aligned16(kbar_all)) return SA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  float* dst = kbar_all;
  for (int32_t g : plan->sizes) {
    const int64_t rows = int64_t(shp->batch) * shp->num_kv_heads * (shp->seq_len / g);
    cudaError_t e = sa_k::launch_pool(k, dst, rows, g, shp->head_dim, st);
    if (e != cudaSuccess) return cuda_status(e);
    dst += rows * shp->head_dim;
  }
  return SA_OK;
}

sa_status sparse_attn_score_plan(const sa_shape* shp, const sa_plan* plan, const void* q,
                                 const float* kbar_all, float* scores, sa_stream_t stream) {
  sa_status s = sa_host::check_supported(shp);
  if (s != SA_OK) return s;
  if (!plan || shp->mode != SA_MODE_DECODE) return SA_ERR_INVALID_ARG;
  if (!same_shape(shp, plan->shape)) return SA_ERR_SHAPE;
  if (!q || !kbar_all || !scores || !aligned16(q) || !aligned16(kbar_all) || !aligned16(scores))
    return SA_ERR_INVALID_ARG;
  if (plan->device < 0) return SA_ERR_NOT_UPLOADED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int d = shp->head_dim;
  const int G = shp->num_q_heads / shp->num_kv_heads;
  const float scale = float(1.0 / std::sqrt(double(d)));
  const float* src = kbar_all;
  for (int32_t g : plan->sizes) {
    const int nbg = int(shp->seq_len / g);
    cudaError_t e = sa_k::launch_decode_scores(q, src, scores, shp->batch, shp->num_q_heads, G,
                                               nbg, d, scale, st, plan->score_stride,
                                               plan->d_kinds, plan->d_gran, g);
    if (e != cudaSuccess) return cuda_status(e);
    src += int64_t(shp->batch) * shp->num_kv_heads * nbg * d;
  }
  return SA_OK;
}

sa_status sparse_attn_score_select(const sa_shape* shp, const sa_plan* plan, const void* q,
                                   const float* kbar, float* scores, int32_t* idx, int32_t* cnt,
                                   int32_t kmax, sa_stream_t stream) {
  sa_status s = sa_host::check_supported(shp);
  if (s != SA_OK) return s;
  if (!plan || shp->mode != SA_MODE_DECODE) return SA_ERR_INVALID_ARG;
  if (!same_shape(shp, plan->shape)) return SA_ERR_SHAPE;
  if (!q || !kbar || !idx || !cnt) return SA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kbar) || (scores && !aligned16(scores)))
    return SA_ERR_INVALID_ARG;
  if (kmax < plan->kmax) return SA_ERR_SHAPE;
  if (has_granularity(plan) || shp->head_dim != 128 || plan->group > 16 || plan->nb > 4096)
    return SA_ERR_UNSUPPORTED;
  if (plan->device < 0) return SA_ERR_NOT_UPLOADED;
  if (int32_t(plan->kinds.size()) == plan->n_streaming) return SA_OK;
  sa_k::IndexSelectArgs a = {};
  a.q = q;
  a.kbar = kbar;
  a.scores = scores;
  a.budgets = plan->d_budgets;
  a.kinds = plan->d_kinds;
  a.idx = idx;
  a.cnt = cnt;
  a.kmax = kmax;
  a.Bt = shp->batch;
  a.Hq = shp->num_q_heads;
  a.Hkv = shp->num_kv_heads;
  a.group = plan->group;
  a.nb = plan->nb;
  a.scale = float(1.0 / std::sqrt(double(shp->head_dim)));
  a.max_retrieval = 0;
  for (int32_t g = 0; g < shp->num_kv_heads; ++g) {
    int32_t n = 0;
    for (int32_t x = 0; x < plan->group; ++x)
      n += plan->kinds[size_t(g) * plan->group + x] != SA_HEAD_STREAMING;
    a.max_retrieval = std::max(a.max_retrieval, n);
  }
  a.rows_per_cta = 0;
  return cuda_status(sa_k::launch_decode_index_select(a, reinterpret_cast<cudaStream_t>(stream)));
}

sa_status sparse_attn_decode_step(const sa_shape* shp, const sa_plan* plan, const void* q,
                                  const float* kbar, const void* k, const void* v, float* scores,
                                  int32_t* idx, int32_t* cnt, int32_t kmax, void* o,
                                  int32_t o_dtype, float* lse, int32_t* dev_status,
                                  sa_stream_t stream) {
  sa_status s = sa_host::check_supported(shp);
  if (s != SA_OK) return s;
  if (!plan || shp->mode != SA_MODE_DECODE) return SA_ERR_INVALID_ARG;
  if (!same_shape(shp, plan->shape)) return SA_ERR_SHAPE;
  if (!q || !kbar || !k || !v || !idx || !cnt || !o || !dev_status) return SA_ERR_INVALID_ARG;
  if (o_dtype != SA_DTYPE_BF16 && o_dtype != SA_DTYPE_F32) return SA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kbar) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (scores && !aligned16(scores)))
    return SA_ERR_INVALID_ARG;
  if (kmax < plan->kmax) return SA_ERR_SHAPE;
  if (has_granularity(plan) || shp->head_dim != 128 || shp->block != 32 || plan->group > 16 ||
      plan->nb > 4096)
    return SA_ERR_UNSUPPORTED;
  if (plan->device < 0) return SA_ERR_NOT_UPLOADED;
  sa_k::IndexSelectArgs a = {};
  a.q = q;
  a.kbar = kbar;
  a.scores = scores;
  a.budgets = plan->d_budgets;
  a.kinds = plan->d_kinds;
  a.idx = idx;
  a.cnt = cnt;
  a.kmax = kmax;
  a.Bt = shp->batch;
  a.Hq = shp->num_q_heads;
  a.Hkv = shp->num_kv_heads;
  a.group = plan->group;
  a.nb = plan->nb;
  a.scale = float(1.0 / std::sqrt(double(shp->head_dim)));
  a.max_retrieval = 0;
  for (int32_t g = 0; g < shp->num_kv_heads; ++g) {
    int32_t n = 0;
    for (int32_t x = 0; x < plan->group; ++x)
      n += plan->kinds[size_t(g) * plan->group + x] != SA_HEAD_STREAMING;
    a.max_retrieval = std::max(a.max_retrieval, n);
  }
  a.rows_per_cta = 0;
  a.k = k;
  a.v = v;
  a.o = o;
  a.out_f32 = o_dtype == SA_DTYPE_F32;
  a.lse = lse;
  a.dev_status = dev_status;
  a.window_blocks = plan->window_blocks;
  a.L = int32_t(shp->seq_len);
  a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  return cuda_status(sa_k::launch_decode_step(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
