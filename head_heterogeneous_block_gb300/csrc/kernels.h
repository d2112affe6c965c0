// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "sparse_attn.h"

namespace sa_k {

// A CUDA error as the ABI's status: allocation failures keep their own code.
inline sa_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return SA_OK;
  if (e == cudaErrorMemoryAllocation) return SA_ERR_NO_MEMORY;
  return SA_ERR_CUDA;
}

// Mean of each block of `block` rows: x [rows*block][d] bf16 -> out [rows][d] fp32.
cudaError_t launch_pool(const void* x, float* out, int64_t rows, int block, int d,
                        cudaStream_t st);

// Prefill block scores for j <= i (scores [Hq][nb][nb], upper part untouched).
cudaError_t launch_prefill_scores(const float* qbar, const float* kbar, float* scores, int Hq,
                                  int group, int nb, int d, float scale, cudaStream_t st);

// The whole prefill Index step: pool Q into ws, pool K after it, then score
// every block pair j <= i with scale 1/sqrt(d).  ws holds (Hq + Hkv) * nb * d
// floats: the pooled queries first, then the pooled keys.
cudaError_t launch_prefill_index(const void* q, const void* k, float* scores, float* ws, int Hq,
                                 int Hkv, int nb, int block, int d, cudaStream_t st);

// Decode scores [Bt][Hq][nb] from q [Bt][Hq][d] (bf16) and kbar [Bt][Hkv][nb][d].
// nb pooled rows per (sequence, KV head) at this pass's block size; score
// rows of `stride` floats (0: nb).  gran (device [Hq], with kinds) limits the
// pass to the retrieval heads whose block size is `size`; NULL scores all.
cudaError_t launch_decode_scores(const void* q, const float* kbar, float* scores, int Bt,
                                 int Hq, int group, int nb, int d, float scale,
                                 cudaStream_t st, int stride = 0,
                                 const uint8_t* kinds = nullptr,
                                 const int32_t* gran = nullptr, int size = 0);

// Decode Index and Select of the retrieval heads in one launch: one cluster
// per (sequence, KV group) scores the group's pooled keys for its retrieval
// heads (the scores of launch_decode_scores, bit for bit) and selects each
// retrieval row as launch_select does.  Rows of streaming heads are left as
// they are.  d = 128, group <= 16, nb <= 4096; rows_per_cta is set by the
// launcher.
struct IndexSelectArgs {
  const void* q;            // [Bt][Hq][128] bf16
  const float* kbar;        // [Bt][Hkv][nb][128] pooled keys
  float* scores;            // [Bt][Hq][nb] retrieval rows written, or NULL
  const int32_t* budgets;   // [Hq] device
  const uint8_t* kinds;     // [Hq] device
  int32_t* idx;             // [Bt*Hq][kmax]
  int32_t* cnt;             // [Bt*Hq]
  int32_t kmax;
  int32_t Bt, Hq, Hkv, group, nb;
  float scale;
  int32_t max_retrieval;    // most retrieval heads in one KV group (>= 1; 0 with attend)
  int32_t rows_per_cta;
  // launch_decode_step only: the attention of every head of the group
  const void* k;            // [Bt][Hkv][L][128] bf16 keys
  const void* v;
  void* o;                  // [Bt*Hq][128], bf16 or fp32
  int32_t out_f32;
  float* lse;               // [Bt*Hq] or NULL
  int32_t* dev_status;
  int32_t window_blocks, L;
  uint64_t wait_ns;         // limit of each wait for a copy (0: the 4 s default)
};
cudaError_t launch_decode_index_select(const IndexSelectArgs& a, cudaStream_t st);
// The whole decode step of a plan without per-head block sizes in one launch:
// the Index and Select of launch_decode_index_select, the streaming heads'
// lists as launch_select writes them, and the attention of every row as
// launch_decode_attention computes it (block size 32), bit for bit.
cudaError_t launch_decode_step(const IndexSelectArgs& a, cudaStream_t st);

struct SelectArgs {
  const float* scores;
  const int32_t* budgets;   // [Hq] device
  const uint8_t* kinds;     // [Hq] device
  int32_t* idx;
  int32_t* cnt;
  int32_t kmax;
  int32_t nb;
  int32_t Hq;
  int32_t rows;             // Hq*nb (prefill) or Bt*Hq (decode)
  int32_t decode;           // 0 / 1
  int32_t window_blocks;    // decode streaming heads
  int32_t group;            // G = Hq / Hkv
  int32_t group_shared;     // prefill: one row per (KV group, query block)
  const int32_t* gran;      // decode: [Hq] device block size per head, or NULL
  int32_t L;                // decode: cache length (rows of L / gran[h] blocks)
  int32_t stride;           // decode: score row stride (0: nb)
  int32_t max_row;          // largest row in blocks (picks the kernel width)
  const int32_t* heads;     // decode: NULL (every head), or the nh heads to run: the
  int32_t nh;               //   grid is Bt * nh rows, row = b * Hq + heads[x % nh]
};
cudaError_t launch_select(const SelectArgs& a, cudaStream_t st);

struct TopPArgs {           // prefill rows only
  const float* scores;
  int32_t* idx;
  int32_t* cnt;
  int32_t kmax;             // >= nb
  int32_t nb;
  int32_t rows;             // Hq*nb
  float p;
};
cudaError_t launch_select_topp(const TopPArgs& a, cudaStream_t st);

struct RebuildArgs {
  const int32_t* cnt;       // [N] blocks per item (the item's cost)
  int32_t* wptr;            // [W+1] out
  int32_t* items;           // [N] out
  int32_t* scratch;         // [3N]
  int32_t num_items, num_workers;
};
cudaError_t launch_lpt_rebuild(const RebuildArgs& a, cudaStream_t st);

struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* idx;
  const int32_t* cnt;
  int32_t kmax;
  const int32_t* wptr;      // [W+1] device
  const int32_t* items;     // [N] device
  int32_t num_workers;
  int32_t num_items;
  int32_t S, B, d, Hq, Hkv;
  void* o;
  int32_t out_f32;          // 1: o is fp32, 0: bf16
  float* lse;
  int32_t* dev_status;
  uint64_t wait_ns;         // limit of each operational wait (0: the 4 s default)
};
// Returns cudaSuccess, or an error; *encode_failed is set when a TMA
// descriptor could not be built.
cudaError_t launch_prefill_attention(const PrefillArgs& a, cudaStream_t st, bool* encode_failed);
// Group-shared lists, even G: items are head pairs p*nb + i (num_items = Hq/2 * nb),
// each K/V block feeding both heads' tiles.
cudaError_t launch_prefill_attention_pairs(const PrefillArgs& a, cudaStream_t st,
                                           bool* encode_failed);

struct DecodeArgs {
  const void* q;            // [Bt][Hq][d]
  const void* k;            // [Bt][Hkv][L][d]
  const void* v;
  const int32_t* idx;       // [Bt*Hq][kmax]
  const int32_t* cnt;
  int32_t kmax;
  int32_t Bt, Hq, Hkv, L, B, d;
  void* o;
  int32_t out_f32;
  float* lse;
  int32_t* dev_status;
  const int32_t* gran;      // [Hq] device block size per head (multiple of 16), or NULL: B
  const int32_t* heads;     // NULL (every head), or the nh heads to run, as for select
  int32_t nh;
  uint64_t wait_ns;         // limit of each wait for a copy (0: the 4 s default)
};
cudaError_t launch_decode_attention(const DecodeArgs& a, cudaStream_t st);

}  // namespace sa_k
